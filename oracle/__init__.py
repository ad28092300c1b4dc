"""CPU oracle for paged KV-cache attention — test infrastructure only.

This package is the slow fp64 definition the GPU library is checked against.
Only the tests, the smoke check and the benchmark's CPU-baseline leg use it;
the GPU library never imports, links or calls it, and it shares no code with
that library.  The arithmetic lives in ``pkv_oracle.cpp`` (plain C++17); this
module builds it with g++ and marshals numpy arrays through ctypes.

Every function cites the passage of the source pages it follows:

* store — "Nano-vLLM System Architecture Analysis", §2 Core Components,
  "Attention with Paged Cache" (K/V written through slot_mapping) and
  "Paged KV Cache" (256-token blocks);
* gather — same section ("gathers all cached K/V from paged blocks");
* decode — same section, decode runs scaled dot-product attention over the
  gathered K/V; GQA from §6 Architecture Support;
* prefill — same section (prefix cache gathered and concatenated with the new
  tokens) and §2 "Scheduler" (chunked prefill), bottom-right causal mask;
* the attention formula softmax(q k^T) v — "Why Understand Inference Engine
  Architecture?", TorchScript Optimization; scale 1/sqrt(D) is an argument.
* e4m3_table / quantize_e4m3 / store_fp8 / decode_fp8 — an FP8 (OCP E4M3)
  KV cache with one scale per tensor; the pages only name quantized KV
  transfers ("Why Understand Inference Engine Architecture?", Tensor
  Parallelism Optimization), so the format is a reading of that line: OCP
  E4M3, nearest code with ties to even, saturated at 448.

bf16 tensors are passed as uint16 bit patterns; outputs are float64.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

STATUS = {
    0: "ok",
    -1: "bad argument",
    -2: "slot out of range",
    -3: "duplicate slot",
    -4: "block id out of range",
    -5: "Lk < Lq",
    -6: "context longer than the block table",
}


class OracleError(RuntimeError):
    pass


def build(src: str = _SRC, out: str = _LIB, extra_flags=()) -> str:
    """Compile the oracle with g++ (-O2, IEEE arithmetic, no fast-math)."""
    cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread",
           *extra_flags, src, "-o", out]
    subprocess.run(cmd, check=True)
    return out


def _stale() -> bool:
    return (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)


def _declare(lib):
    P = ctypes.c_void_p
    i64, i32, f64 = ctypes.c_int64, ctypes.c_int, ctypes.c_double
    lib.oracle_store.argtypes = [P, P, i64, i64, P, P, P, i64, i32, i32, i32, i64]
    lib.oracle_gather.argtypes = [P, P, P, i64, i32, i32, i32, i64, P, P]
    lib.oracle_decode.argtypes = [P, P, P, P, P, P, i32, P, i32, i32, i32, i32,
                                  i32, i64, f64, i32]
    lib.oracle_prefill.argtypes = [P, P, P, P, P, P, i32, P, P, i32, i32, i32,
                                   i32, i32, i64, f64, i32]
    lib.oracle_copy_blocks.argtypes = [P, P, P, P, i64, i32, i32, i32, i64]
    f32 = ctypes.c_float
    lib.oracle_e4m3_table.argtypes = [P]
    lib.oracle_quantize_e4m3.argtypes = [P, i64, f32, P]
    lib.oracle_store_fp8.argtypes = [P, P, i64, i64, P, P, P, i64, i32, i32, i32, i64, f32, f32]
    lib.oracle_decode_fp8.argtypes = [P, P, P, P, P, P, i32, P, i32, i32, i32, i32, i32, i64,
                                      f64, f64, f64, i32]
    for fn in ("oracle_store", "oracle_gather", "oracle_decode", "oracle_prefill",
               "oracle_hardware_threads", "oracle_copy_blocks", "oracle_e4m3_table",
               "oracle_quantize_e4m3", "oracle_store_fp8", "oracle_decode_fp8"):
        getattr(lib, fn).restype = ctypes.c_int
    return lib


def load(path: str | None = None):
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if _stale():
                build()
            _lib = _declare(ctypes.CDLL(_LIB))
    return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _u16(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"bf16 bit patterns must be uint16, got {a.dtype}")
    return np.ascontiguousarray(a)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _check(st: int):
    if st != 0:
        raise OracleError(f"oracle status {st}: {STATUS.get(st, '?')}")


def hardware_threads(lib=None) -> int:
    return (lib or load()).oracle_hardware_threads()


def store(k, v, k_cache, v_cache, slot_mapping, lib=None) -> None:
    """In-place store of k/v [T, Hkv, D] into the caches [NB, bs, Hkv, D]."""
    lib = lib or load()
    k, v = _u16(k), _u16(v)
    if not (k_cache.flags.c_contiguous and v_cache.flags.c_contiguous):
        raise ValueError("caches must be C-contiguous")
    if k_cache.dtype != np.uint16 or v_cache.dtype != np.uint16:
        raise TypeError("caches must be uint16 bf16 bit patterns")
    T, Hkv, D = k.shape
    NB, bs = k_cache.shape[0], k_cache.shape[1]
    sm = _i32(slot_mapping)
    _check(lib.oracle_store(_ptr(k), _ptr(v), Hkv * D, Hkv * D, _ptr(k_cache),
                            _ptr(v_cache), _ptr(sm), T, Hkv, D, bs, NB))


def copy_blocks(k_cache, v_cache, src, dst, lib=None) -> None:
    """In-place: block dst[i] of both caches [NB, bs, Hkv, D] := block src[i]."""
    lib = lib or load()
    if k_cache.dtype != np.uint16 or not k_cache.flags.c_contiguous:
        raise TypeError("caches must be C-contiguous uint16")
    NB, bs, Hkv, D = k_cache.shape
    s, d = _i32(src), _i32(dst)
    _check(lib.oracle_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(s), _ptr(d), len(s), Hkv,
                                  D, bs, NB))


def gather(k_cache, v_cache, table_row, L, lib=None):
    """Contiguous K, V [L, Hkv, D] (uint16) of one sequence."""
    lib = lib or load()
    k_cache, v_cache = _u16(k_cache), _u16(v_cache)
    NB, bs, Hkv, D = k_cache.shape
    row = _i32(table_row)
    K = np.empty((L, Hkv, D), np.uint16)
    V = np.empty((L, Hkv, D), np.uint16)
    _check(lib.oracle_gather(_ptr(k_cache), _ptr(v_cache), _ptr(row), L, Hkv, D,
                             bs, NB, _ptr(K), _ptr(V)))
    return K, V


def decode(q, k_cache, v_cache, block_tables, context_lens, scale, nthreads=0,
           lib=None):
    """out [B, Hq, D] float64, lse [B, Hq] float64."""
    lib = lib or load()
    q, k_cache, v_cache = _u16(q), _u16(k_cache), _u16(v_cache)
    B, Hq, D = q.shape
    NB, bs, Hkv, D2 = k_cache.shape
    assert D == D2
    bt, cl = _i32(block_tables), _i32(context_lens)
    maxblk = bt.shape[1] if bt.ndim == 2 else 0
    out = np.zeros((B, Hq, D), np.float64)
    lse = np.zeros((B, Hq), np.float64)
    _check(lib.oracle_decode(_ptr(out), _ptr(lse), _ptr(q), _ptr(k_cache),
                             _ptr(v_cache), _ptr(bt), maxblk, _ptr(cl), B, Hq, Hkv,
                             D, bs, NB, float(scale), int(nthreads)))
    return out, lse


def prefill(q, k_cache, v_cache, block_tables, cu_seqlens_q, cu_seqlens_k, scale,
            nthreads=0, lib=None):
    """out [sum Lq, Hq, D] float64, lse [sum Lq, Hq] float64."""
    lib = lib or load()
    q, k_cache, v_cache = _u16(q), _u16(k_cache), _u16(v_cache)
    Nq, Hq, D = q.shape
    NB, bs, Hkv, D2 = k_cache.shape
    assert D == D2
    bt, cq, ck = _i32(block_tables), _i32(cu_seqlens_q), _i32(cu_seqlens_k)
    B = cq.shape[0] - 1
    maxblk = bt.shape[1] if bt.ndim == 2 else 0
    out = np.zeros((Nq, Hq, D), np.float64)
    lse = np.zeros((Nq, Hq), np.float64)
    _check(lib.oracle_prefill(_ptr(out), _ptr(lse), _ptr(q), _ptr(k_cache),
                              _ptr(v_cache), _ptr(bt), maxblk, _ptr(cq), _ptr(ck), B,
                              Hq, Hkv, D, bs, NB, float(scale), int(nthreads)))
    return out, lse


def inv_scale(scale: float) -> np.float32:
    """The binary32 reciprocal of a tensor scale, as the quantizer uses it."""
    return np.float32(1.0) / np.float32(scale)


def e4m3_table(lib=None) -> np.ndarray:
    """Value of each of the 256 E4M3 codes (float64, NaN for 0x7F / 0xFF)."""
    lib = lib or load()
    t = np.empty(256, np.float64)
    _check(lib.oracle_e4m3_table(_ptr(t)))
    return t


def quantize_e4m3(x_bits, scale: float, lib=None) -> np.ndarray:
    """E4M3 codes (uint8, same shape) of bf16 values x under tensor scale."""
    lib = lib or load()
    x = _u16(x_bits)
    codes = np.empty(x.shape, np.uint8)
    _check(lib.oracle_quantize_e4m3(_ptr(x), x.size, float(inv_scale(scale)), _ptr(codes)))
    return codes


def store_fp8(k, v, k_cache, v_cache, slot_mapping, k_scale: float, v_scale: float,
              lib=None) -> None:
    """In-place store of bf16 k/v [T, Hkv, D] into uint8 E4M3 caches [NB, bs, Hkv, D]."""
    lib = lib or load()
    k, v = _u16(k), _u16(v)
    for c in (k_cache, v_cache):
        if c.dtype != np.uint8 or not c.flags.c_contiguous:
            raise TypeError("fp8 caches must be C-contiguous uint8")
    T, Hkv, D = k.shape
    NB, bs = k_cache.shape[0], k_cache.shape[1]
    sm = _i32(slot_mapping)
    _check(lib.oracle_store_fp8(_ptr(k), _ptr(v), Hkv * D, Hkv * D, _ptr(k_cache),
                                _ptr(v_cache), _ptr(sm), T, Hkv, D, bs, NB,
                                float(inv_scale(k_scale)), float(inv_scale(v_scale))))


def decode_fp8(q, k_cache, v_cache, block_tables, context_lens, scale, k_scale, v_scale,
               nthreads=0, lib=None):
    """Decode over uint8 E4M3 caches: out [B, Hq, D] float64, lse [B, Hq] float64."""
    lib = lib or load()
    q = _u16(q)
    for c in (k_cache, v_cache):
        if c.dtype != np.uint8 or not c.flags.c_contiguous:
            raise TypeError("fp8 caches must be C-contiguous uint8")
    B, Hq, D = q.shape
    NB, bs, Hkv, D2 = k_cache.shape
    assert D == D2
    bt, cl = _i32(block_tables), _i32(context_lens)
    maxblk = bt.shape[1] if bt.ndim == 2 else 0
    out = np.zeros((B, Hq, D), np.float64)
    lse = np.zeros((B, Hq), np.float64)
    _check(lib.oracle_decode_fp8(_ptr(out), _ptr(lse), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                 _ptr(bt), maxblk, _ptr(cl), B, Hq, Hkv, D, bs, NB, float(scale),
                                 float(k_scale), float(v_scale), int(nthreads)))
    return out, lse
