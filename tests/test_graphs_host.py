"""Host side of the CUDA-graph decode runner, no GPU: the configuration layout
the binding builds matches the library's, the default bucket set is the
pages' list (1, 2, 4, ..., 512, read as powers of two: "Nano-vLLM System
Architecture Analysis", comparison table, "Variable-batch CUDA Graphs"), and
the bucket a batch runs in is the smallest that holds it, checked against
brute force."""
import ctypes

import numpy as np
import pytest

from paged_kv_cache_214_gb300 import build as B
from paged_kv_cache_214_gb300 import graphs, pkv


@pytest.fixture(scope="module", autouse=True)
def lib():
    B.build()
    return graphs._lib()


def test_config_layout_matches_the_library(lib):
    assert lib.pkv_decode_graphs_config_bytes() == ctypes.sizeof(graphs._Config)


def test_default_buckets():
    assert graphs.default_buckets(1) == [1]
    assert graphs.default_buckets(5) == [1, 2, 4]
    full = [1, 2, 4, 8, 16, 32, 64, 128, 256, 512]
    assert graphs.default_buckets(512) == full
    assert graphs.default_buckets(100000) == full
    with pytest.raises(pkv.PkvError):
        graphs.default_buckets(0)


def test_pick_bucket_edges():
    b = [1, 2, 4, 8]
    assert [graphs.pick_bucket(b, n) for n in range(0, 10)] == [0, 1, 2, 4, 4, 8, 8, 8, 8, 0]
    assert graphs.pick_bucket([3, 5], 1) == 3
    for bad_list in ([], [0, 1], [2, 2], [4, 3]):
        with pytest.raises(pkv.PkvError):
            graphs.pick_bucket(bad_list, 1)
    with pytest.raises(pkv.PkvError):
        graphs.pick_bucket(b, -1)


def test_pick_bucket_brute_force():
    g = np.random.default_rng(5)
    for _ in range(200):
        sizes = sorted(set(int(x) for x in g.integers(1, 600, size=g.integers(1, 12))))
        for n in list(g.integers(0, 700, size=20)) + [sizes[0], sizes[-1], sizes[-1] + 1]:
            want = min((s for s in sizes if s >= n), default=0) if n > 0 else 0
            assert graphs.pick_bucket(sizes, int(n)) == want


def _config(**kw):
    """A configuration whose pointers are placeholders that no rejected call
    dereferences; every case below is invalid, so create() returns before any
    CUDA call."""
    fake = 1 << 20
    c = graphs._Config(Hq=16, Hkv=8, D=128, block_size=256, max_blocks_per_seq=4,
                       max_batch=64, num_blocks=1000, kv_fp8=0, scale=0.088,
                       k_scale=1.0, v_scale=1.0, num_buckets=0, buckets=None,
                       k_cache=fake, v_cache=fake, q=fake, k_new=fake, v_new=fake,
                       slot_mapping=fake, block_tables=fake, context_lens=fake, out=fake,
                       lse=fake, workspace=None, workspace_bytes=0)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def _create(lib, cfg):
    h = ctypes.c_void_p(12345)
    st = lib.pkv_decode_graphs_create(ctypes.byref(cfg), ctypes.byref(h))
    assert h.value is None, "a refused create must store NULL"
    return st


def test_create_rejects_bad_configurations(lib):
    assert lib.pkv_decode_graphs_create(None, None) == pkv.PKV_ERR_ARG
    for field in ("q", "k_new", "v_new", "slot_mapping", "block_tables", "context_lens", "out",
                  "k_cache", "v_cache"):
        assert _create(lib, _config(**{field: None})) == pkv.PKV_ERR_ARG, field
    assert _create(lib, _config(max_batch=0)) == pkv.PKV_ERR_ARG
    assert _create(lib, _config(max_blocks_per_seq=0)) == pkv.PKV_ERR_ARG
    assert _create(lib, _config(kv_fp8=2)) == pkv.PKV_ERR_ARG
    bad = (ctypes.c_int32 * 3)(4, 4, 8)
    assert _create(lib, _config(num_buckets=3, buckets=ctypes.cast(bad, graphs._I32P))) == \
        pkv.PKV_ERR_ARG
    big = (ctypes.c_int32 * 2)(4, 65)   # above max_batch
    assert _create(lib, _config(num_buckets=2, buckets=ctypes.cast(big, graphs._I32P))) == \
        pkv.PKV_ERR_ARG
    assert _create(lib, _config(num_buckets=2, buckets=None)) == pkv.PKV_ERR_ARG
    assert _create(lib, _config(num_buckets=65)) == pkv.PKV_ERR_ARG
    assert _create(lib, _config(D=64)) == pkv.PKV_ERR_SHAPE
    assert _create(lib, _config(Hq=12, Hkv=8)) == pkv.PKV_ERR_SHAPE
    assert _create(lib, _config(block_size=128)) == pkv.PKV_ERR_SHAPE
    # a batch of 64 over 4-block tables splits: a workspace is needed
    assert lib.pkv_decode_graphs_workspace_bytes(ctypes.byref(_config())) > 0
    assert _create(lib, _config()) == pkv.PKV_ERR_WORKSPACE
    assert _create(lib, _config(workspace=(1 << 20) + 8, workspace_bytes=1 << 30)) == \
        pkv.PKV_ERR_WORKSPACE   # misaligned
    assert lib.pkv_decode_graphs_workspace_bytes(ctypes.byref(_config(D=64))) == 0


def test_runner_calls_reject_null(lib):
    assert lib.pkv_decode_graphs_run(None, 1, None) == pkv.PKV_ERR_ARG
    assert lib.pkv_decode_graphs_buckets(None, None, 0) == pkv.PKV_ERR_ARG
    lib.pkv_decode_graphs_destroy(None)
