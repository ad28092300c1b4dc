"""The C-ABI library loads and exports every symbol include/*.h declares; host
argument checks answer without touching a GPU (no GPU needed)."""
import ctypes
import os
import re

import pytest

from paged_kv_cache_214_gb300 import build as B
from paged_kv_cache_214_gb300 import pkv

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "pkv.h")
HEADERS = ("pkv.h", "pkv_blocks.h", "pkv_graphs.h")


def declared_functions(header=HEADER):
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:int|int64_t|size_t|void|const char\s*\*|pkv_block_manager\s*\*)"
                      r"\s*(\w+)\s*\(", text, flags=re.M)


@pytest.fixture(scope="module")
def lib():
    B.build()
    return pkv.load_library()


def test_header_declares_the_hot_path():
    names = declared_functions()
    for n in ("kv_cache_store", "paged_decode_attention", "paged_prefill_attention",
              "paged_decode_workspace_bytes", "pkv_get_device_error", "pkv_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for header in HEADERS:
        names = declared_functions(os.path.join(os.path.dirname(HEADER), header))
        assert names, header
        for name in names:
            assert hasattr(lib, name), name
            assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_host_argument_checks(lib):
    s = None
    # negative T, unsupported head_dim / block size, head counts
    assert lib.kv_cache_store(None, None, 0, 0, None, None, None, -1, 8, 128, 256, 16, s) == pkv.PKV_ERR_ARG
    assert lib.kv_cache_store(None, None, 0, 0, None, None, None, 0, 8, 64, 256, 16, s) == pkv.PKV_ERR_SHAPE
    assert lib.kv_cache_store(None, None, 0, 0, None, None, None, 0, 8, 128, 16, 16, s) == pkv.PKV_ERR_SHAPE
    assert lib.kv_cache_store(None, None, 0, 0, None, None, None, 0, 8, 128, 256, 16, s) == pkv.PKV_OK
    assert lib.kv_cache_store(None, None, 1024, 1024, None, None, None, 4, 8, 128, 256, 16, s) == pkv.PKV_ERR_ARG
    assert lib.paged_decode_attention(None, None, None, None, None, None, 1, None, 2, 12, 8, 128,
                                      256, 16, 1.0, None, 0, 0, s) == pkv.PKV_ERR_SHAPE
    assert lib.paged_decode_attention(None, None, None, None, None, None, 1, None, 0, 16, 8, 128,
                                      256, 16, 1.0, None, 0, 0, s) == pkv.PKV_OK
    assert lib.paged_decode_attention(None, None, None, None, None, None, 1, None, 2, 16, 8, 128,
                                      256, 16, 1.0, None, 0, 0, s) == pkv.PKV_ERR_ARG
    assert lib.paged_prefill_attention(None, None, None, None, None, None, 1, None, None, 2, 8,
                                       8, 16, 8, 64, 256, 16, 1.0, s) == pkv.PKV_ERR_SHAPE
    assert lib.paged_prefill_attention(None, None, None, None, None, None, 1, None, None, 2, 8,
                                       8, 16, 8, 128, 256, 16, 1.0, s) == pkv.PKV_ERR_ARG
    # pools whose slot count does not fit 32-bit TMA coordinates
    assert lib.kv_cache_store(None, None, 0, 0, None, None, None, 0, 8, 128, 256, 1 << 24, s) == pkv.PKV_ERR_SHAPE


def test_multiquery_host_checks(lib):
    s = None
    mq = lib.paged_decode_attention_multiquery
    # q_len outside [1, 64]
    assert mq(None, None, None, None, None, None, 1, None, 2, 0, 16, 8, 128, 256, 16, 1.0,
              None, 0, 0, s) == pkv.PKV_ERR_ARG
    assert mq(None, None, None, None, None, None, 1, None, 2, 65, 16, 8, 128, 256, 16, 1.0,
              None, 0, 0, s) == pkv.PKV_ERR_ARG
    # Hq not a multiple of Hkv, empty batch, missing pointers
    assert mq(None, None, None, None, None, None, 1, None, 2, 4, 12, 8, 128, 256, 16, 1.0,
              None, 0, 0, s) == pkv.PKV_ERR_SHAPE
    assert mq(None, None, None, None, None, None, 1, None, 0, 4, 16, 8, 128, 256, 16, 1.0,
              None, 0, 0, s) == pkv.PKV_OK
    assert mq(None, None, None, None, None, None, 1, None, 2, 4, 16, 8, 128, 256, 16, 1.0,
              None, 0, 0, s) == pkv.PKV_ERR_ARG
    assert lib.paged_decode_multiquery_workspace_bytes(2, 0, 16, 8, 128, 4, 256, 0) == 0


def test_fp8_host_checks(lib):
    s = None
    st8 = lib.kv_cache_store_fp8
    dec8 = lib.paged_decode_attention_fp8
    nan, inf = float("nan"), float("inf")
    # scales must be finite and > 0, checked before anything else
    for bad in (0.0, -1.0, nan, inf):
        assert st8(None, None, 1024, 1024, None, None, None, 4, 8, 128, 256, 4, bad, 1.0,
                   s) == pkv.PKV_ERR_ARG
        assert st8(None, None, 1024, 1024, None, None, None, 4, 8, 128, 256, 4, 1.0, bad,
                   s) == pkv.PKV_ERR_ARG
        assert dec8(None, None, None, None, None, None, 1, None, 2, 16, 8, 128, 256, 4, 1.0,
                    bad, 1.0, None, 0, 0, s) == pkv.PKV_ERR_ARG
        assert dec8(None, None, None, None, None, None, 1, None, 2, 16, 8, 128, 256, 4, 1.0,
                    1.0, bad, None, 0, 0, s) == pkv.PKV_ERR_ARG
    # nothing to store / decode is not an error; shapes as for the bf16 calls
    assert st8(None, None, 1024, 1024, None, None, None, 0, 8, 128, 256, 4, 1.0, 1.0,
               s) == pkv.PKV_OK
    assert st8(None, None, 1024, 1024, None, None, None, 4, 8, 64, 256, 4, 1.0, 1.0,
               s) == pkv.PKV_ERR_SHAPE
    assert st8(None, None, 1000, 1024, None, None, None, 4, 8, 128, 256, 4, 1.0, 1.0,
               s) == pkv.PKV_ERR_ARG
    assert dec8(None, None, None, None, None, None, 1, None, 0, 16, 8, 128, 256, 4, 1.0, 0.5,
                0.5, None, 0, 0, s) == pkv.PKV_OK
    assert dec8(None, None, None, None, None, None, 1, None, 2, 12, 8, 128, 256, 4, 1.0, 0.5,
                0.5, None, 0, 0, s) == pkv.PKV_ERR_SHAPE
    assert dec8(None, None, None, None, None, None, 1, None, 2, 16, 8, 128, 128, 4, 1.0, 0.5,
                0.5, None, 0, 0, s) == pkv.PKV_ERR_SHAPE
    assert dec8(None, None, None, None, None, None, 1, None, 2, 16, 8, 128, 256, 4, 1.0, 0.5,
                0.5, None, 0, 0, s) == pkv.PKV_ERR_ARG


def test_decode_store_host_checks(lib):
    s = None
    ds = lib.paged_decode_attention_store
    P = 16  # a stand-in device address: the checks below fail before any use
    # nothing to do
    assert ds(None, None, None, None, None, 1024, 1024, None, None, None, None, 1, None, 0, 16,
              8, 128, 256, 4, 1.0, None, 0, 0, s) == pkv.PKV_OK
    # shapes, then missing pointers
    assert ds(None, None, None, None, None, 1024, 1024, None, None, None, None, 1, None, 2, 12,
              8, 128, 256, 4, 1.0, None, 0, 0, s) == pkv.PKV_ERR_SHAPE
    assert ds(None, None, None, None, None, 1024, 1024, None, None, None, None, 1, None, 2, 16,
              8, 128, 256, 4, 1.0, None, 0, 0, s) == pkv.PKV_ERR_ARG
    # token strides: at least Hkv * D and a multiple of 8 elements
    for ks in (1000, 1028):
        assert ds(P, None, P, P, P, ks, 1024, P, P, P, P, 1, P, 2, 16, 8, 128, 256, 4, 1.0, None,
                  0, 0, s) == pkv.PKV_ERR_ARG
    # a misaligned new-token row
    assert ds(P, None, P, P + 2, P, 1024, 1024, P, P, P, P, 1, P, 2, 16, 8, 128, 256, 4, 1.0,
              None, 0, 0, s) == pkv.PKV_ERR_ARG


def test_fp8_decode_store_host_checks(lib):
    s = None
    ds = lib.paged_decode_attention_fp8_store
    P = 16  # a stand-in device address: the checks below fail before any use
    nan = float("nan")
    # scales are checked first, then as paged_decode_attention_store
    for ks, vs in ((0.0, 1.0), (1.0, -2.0), (nan, 1.0), (1.0, float("inf"))):
        assert ds(P, None, P, P, P, 1024, 1024, P, P, P, P, 1, P, 2, 16, 8, 128, 256, 4, 1.0,
                  ks, vs, None, 0, 0, s) == pkv.PKV_ERR_ARG
    assert ds(None, None, None, None, None, 1024, 1024, None, None, None, None, 1, None, 0, 16,
              8, 128, 256, 4, 1.0, 0.5, 0.5, None, 0, 0, s) == pkv.PKV_OK
    assert ds(None, None, None, None, None, 1024, 1024, None, None, None, None, 1, None, 2, 16,
              8, 128, 256, 4, 1.0, 0.5, 0.5, None, 0, 0, s) == pkv.PKV_ERR_ARG
    assert ds(P, None, P, P, P, 1020, 1024, P, P, P, P, 1, P, 2, 16, 8, 128, 256, 4, 1.0, 0.5,
              0.5, None, 0, 0, s) == pkv.PKV_ERR_ARG


def test_workspace_query_and_split_plan(lib):
    # one split needs no workspace; several need partials + counters
    assert pkv.paged_decode_workspace_bytes(4, 16, 8, 128, 1, 256, 1) == 0
    ws = pkv.paged_decode_workspace_bytes(8, 32, 8, 128, 512, 256, 16)
    assert ws >= (1 << 20) + 8 * 32 * 16 * (128 * 4 + 4)
    assert pkv.paged_decode_num_splits(8, 32, 8, 128, 512, 256, 16) == 16
    assert pkv.paged_decode_num_splits(8, 32, 8, 128, 64, 256, 7) == 7
    # a requested count is raised so that no split exceeds 32 blocks
    assert pkv.paged_decode_num_splits(8, 32, 8, 128, 512, 256, 7) == 16
    assert pkv.paged_decode_workspace_bytes(8, 32, 8, 64, 512, 256, 16) == 0   # rejected shape
    with pytest.raises(pkv.PkvError):
        pkv.paged_decode_num_splits(8, 32, 8, 64, 512, 256, 0)


def test_decode_flags_reject_unknown_bits(lib):
    # refused on the host, before anything is read or launched
    st = lib.paged_decode_attention_flags(None, None, None, None, None, None, 1, None, 1, 8, 8,
                                          128, 256, 1, 0.1, None, 0, 0, 2, None)
    assert st == pkv.PKV_ERR_ARG
    assert pkv.PKV_DECODE_METADATA_READY == 1


def test_status_strings(lib):
    for code in range(-6, 1):
        assert pkv.status_string(code).startswith("PKV_")
    assert "unknown" in pkv.status_string(42)


def test_bindings_declare_every_signature(lib):
    """ctypes passes undeclared integer arguments as 32-bit ints, which would
    truncate 64-bit device pointers: every exported function must carry
    argtypes / restype from the bindings."""
    from paged_kv_cache_214_gb300 import blocks, graphs
    blocks._lib()
    graphs._lib()
    hdr_dir = os.path.dirname(HEADER)
    for header in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(os.path.join(hdr_dir, header)).read(), flags=re.S)
        names = re.findall(r"^\s*(?:int|int64_t|size_t|void|const char\s*\*|pkv_block_manager\s*\*)"
                           r"\s*(\w+)\s*\(", text, flags=re.M)
        assert names, header
        for name in names:
            fn = getattr(lib, name)
            assert fn.argtypes is not None, f"{name} has no argtypes"
