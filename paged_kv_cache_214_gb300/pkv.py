"""Python binding of libpkv.so (include/pkv.h): argument marshalling only.

Each function takes torch tensors that already live on the GPU, checks their
dtype / layout / device, and passes raw device pointers, sizes and the current
CUDA stream to the C entry point of the same name.  Every step of the
computation runs in the library's CUDA kernels; there is no fallback of any kind:
if the shared library is missing or a call fails, an exception is raised.
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpkv.so")

PKV_OK = 0
PKV_ERR_ARG = -1
PKV_ERR_SHAPE = -2
PKV_ERR_WORKSPACE = -3
PKV_ERR_LAUNCH = -4
PKV_ERR_DEVICE_INDEX = -5
PKV_ERR_TIMEOUT = -6
PKV_DECODE_METADATA_READY = 1

_lock = threading.Lock()
_lib = None
_workspaces = {}


class PkvError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status) if _lib else status}")


def load_library(path: str = LIB_PATH):
    """Load libpkv.so; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build the CUDA library first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(path)
        P, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                                ctypes.c_float, ctypes.c_size_t)
        lib.kv_cache_store.argtypes = [P, P, i64, i64, P, P, P, i64, i32, i32, i32, i64, P]
        lib.kv_cache_store.restype = i32
        lib.kv_cache_copy_blocks.argtypes = [P, P, P, P, i32, i32, i32, i32, i64, P]
        lib.kv_cache_copy_blocks.restype = i32
        lib.paged_decode_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32, i32]
        lib.paged_decode_workspace_bytes.restype = sz
        lib.paged_decode_num_splits.argtypes = [i32, i32, i32, i32, i32, i32, i32]
        lib.paged_decode_num_splits.restype = i32
        lib.paged_decode_attention.argtypes = [P, P, P, P, P, P, i32, P, i32, i32, i32, i32,
                                               i32, i64, f32, P, sz, i32, P]
        lib.paged_decode_attention.restype = i32
        lib.paged_decode_attention_flags.argtypes = [P, P, P, P, P, P, i32, P, i32, i32, i32,
                                                     i32, i32, i64, f32, P, sz, i32,
                                                     ctypes.c_uint32, P]
        lib.paged_decode_attention_flags.restype = i32
        lib.paged_decode_shared_prefix_workspace_bytes.argtypes = [i32] * 8
        lib.paged_decode_shared_prefix_workspace_bytes.restype = sz
        lib.paged_decode_attention_shared_prefix.argtypes = [P, P, P, P, P, P, i32, P, i32, i32,
                                                             i32, i32, i32, i64, f32, i32, P,
                                                             sz, i32, P]
        lib.paged_decode_attention_shared_prefix.restype = i32
        lib.paged_decode_attention_noalloc.argtypes = [P, P, P, P, P, P, i32, P, i32, i32, i32,
                                                       i32, i32, i64, f32, i32, P]
        lib.paged_decode_attention_noalloc.restype = i32
        lib.paged_decode_multiquery_workspace_bytes.argtypes = [i32] * 8
        lib.paged_decode_multiquery_workspace_bytes.restype = sz
        lib.paged_decode_attention_multiquery.argtypes = [P, P, P, P, P, P, i32, P, i32, i32, i32,
                                                          i32, i32, i32, i64, f32, P, sz, i32, P]
        lib.paged_decode_attention_multiquery.restype = i32
        lib.paged_decode_attention_store.argtypes = [P, P, P, P, P, i64, i64, P, P, P, P, i32,
                                                     P, i32, i32, i32, i32, i32, i64, f32, P,
                                                     sz, i32, P]
        lib.paged_decode_attention_store.restype = i32
        lib.paged_decode_attention_fp8_store.argtypes = [P, P, P, P, P, i64, i64, P, P, P, P,
                                                         i32, P, i32, i32, i32, i32, i32, i64,
                                                         f32, f32, f32, P, sz, i32, P]
        lib.paged_decode_attention_fp8_store.restype = i32
        lib.kv_cache_store_fp8.argtypes = [P, P, i64, i64, P, P, P, i64, i32, i32, i32, i64,
                                           f32, f32, P]
        lib.kv_cache_store_fp8.restype = i32
        lib.paged_decode_attention_fp8.argtypes = [P, P, P, P, P, P, i32, P, i32, i32, i32, i32,
                                                   i32, i64, f32, f32, f32, P, sz, i32, P]
        lib.paged_decode_attention_fp8.restype = i32
        lib.paged_prefill_attention.argtypes = [P, P, P, P, P, P, i32, P, P, i32, i32, i32,
                                                i32, i32, i32, i32, i64, f32, P]
        lib.paged_prefill_attention.restype = i32
        lib.pkv_get_device_error.argtypes = [P]
        lib.pkv_get_device_error.restype = i32
        lib.pkv_status_string.argtypes = [i32]
        lib.pkv_status_string.restype = ctypes.c_char_p
        lib.pkv_testing_set_wait_fault.argtypes = [i64, i32]
        lib.pkv_testing_set_wait_fault.restype = i32
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load_library().pkv_status_string(int(status)).decode()


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t: Optional[torch.Tensor]) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _need(t: torch.Tensor, name: str, dtype, ndim: Optional[int] = None,
          contiguous: bool = True):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _pool_dims(k_cache: torch.Tensor, v_cache: torch.Tensor):
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    if k_cache.shape != v_cache.shape:
        raise ValueError("k_cache and v_cache shapes differ")
    NB, bs, Hkv, D = k_cache.shape
    return NB, bs, Hkv, D


def _check(status: int, what: str):
    if status != PKV_OK:
        raise PkvError(status, what)


def kv_cache_store(k: torch.Tensor, v: torch.Tensor, k_cache: torch.Tensor,
                   v_cache: torch.Tensor, slot_mapping: torch.Tensor, stream=None) -> None:
    """k, v: bf16 [T, Hkv, D] (each token's [Hkv, D] contiguous; token stride
    free); caches [NB, bs, Hkv, D]; slot_mapping int32 [T]."""
    lib = load_library()
    NB, bs, Hkv, D = _pool_dims(k_cache, v_cache)
    for name, t in (("k", k), ("v", v)):
        _need(t, name, torch.bfloat16, 3, contiguous=False)
        if tuple(t.shape[1:]) != (Hkv, D) or t.stride(2) != 1 or t.stride(1) != D:
            raise ValueError(f"{name} must be [T, {Hkv}, {D}] with contiguous rows")
    _need(slot_mapping, "slot_mapping", torch.int32, 1)
    T = k.shape[0]
    if v.shape[0] != T or slot_mapping.shape[0] != T:
        raise ValueError("k, v and slot_mapping disagree on T")
    _check(lib.kv_cache_store(_ptr(k), _ptr(v), k.stride(0), v.stride(0), _ptr(k_cache),
                              _ptr(v_cache), _ptr(slot_mapping), T, Hkv, D, bs, NB,
                              _stream(stream)), "kv_cache_store")


def kv_cache_copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor,
                         src_blocks: torch.Tensor, dst_blocks: torch.Tensor,
                         stream=None) -> None:
    """Copy-on-write copies: block dst_blocks[i] of both caches becomes a copy
    of block src_blocks[i] (int32 device tensors of equal length)."""
    lib = load_library()
    NB, bs, Hkv, D = _pool_dims(k_cache, v_cache)
    _need(src_blocks, "src_blocks", torch.int32, 1)
    _need(dst_blocks, "dst_blocks", torch.int32, 1)
    if src_blocks.shape != dst_blocks.shape:
        raise ValueError("src_blocks and dst_blocks differ in length")
    _check(lib.kv_cache_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(src_blocks),
                                    _ptr(dst_blocks), src_blocks.shape[0], Hkv, D, bs, NB,
                                    _stream(stream)), "kv_cache_copy_blocks")


def paged_decode_workspace_bytes(B: int, Hq: int, Hkv: int, D: int, max_blocks_per_seq: int,
                                 block_size: int = 256, num_splits: int = 0) -> int:
    return int(load_library().paged_decode_workspace_bytes(B, Hq, Hkv, D, max_blocks_per_seq,
                                                           block_size, num_splits))


def paged_decode_num_splits(B: int, Hq: int, Hkv: int, D: int, max_blocks_per_seq: int,
                            block_size: int = 256, num_splits: int = 0) -> int:
    n = load_library().paged_decode_num_splits(B, Hq, Hkv, D, max_blocks_per_seq, block_size,
                                               num_splits)
    _check(min(n, 0), "paged_decode_num_splits")
    return int(n)


def decode_workspace(nbytes: int, device) -> torch.Tensor:
    """A zero-initialised, 256-byte aligned workspace of at least nbytes on
    `device`, reused across calls on that device (the library leaves its
    counters zeroed).  Callers running decode concurrently on several streams
    must pass their own workspaces instead."""
    dev = torch.device(device)
    key = (dev.type, dev.index if dev.index is not None else torch.cuda.current_device())
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=dev)
        _workspaces[key] = ws
    return ws


def paged_decode_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                           block_tables: torch.Tensor, context_lens: torch.Tensor,
                           scale: float, out: Optional[torch.Tensor] = None,
                           lse: Optional[torch.Tensor] = None,
                           workspace: Optional[torch.Tensor] = None, num_splits: int = 0,
                           want_lse: bool = True, stream=None, metadata_ready: bool = False
                           ) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """q bf16 [B, Hq, D]; block_tables int32 [B, max_blocks]; context_lens int32
    [B].  Returns (out bf16 [B, Hq, D], lse fp32 [B, Hq] or None).
    metadata_ready: block_tables and context_lens were written before the
    stream's previous kernel started and no running kernel writes them
    (PKV_DECODE_METADATA_READY of paged_decode_attention_flags)."""
    lib = load_library()
    NB, bs, Hkv, D = _pool_dims(k_cache, v_cache)
    _need(q, "q", torch.bfloat16, 3)
    B, Hq, Dq = q.shape
    if Dq != D:
        raise ValueError("q head_dim differs from the cache's")
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(context_lens, "context_lens", torch.int32, 1)
    if block_tables.shape[0] != B or context_lens.shape[0] != B:
        raise ValueError("block_tables / context_lens batch differs from q")
    maxblk = block_tables.shape[1]
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, 3)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if lse is not None:
        _need(lse, "lse", torch.float32, 2)
    need = paged_decode_workspace_bytes(B, Hq, Hkv, D, maxblk, bs, num_splits)
    if workspace is None and need:
        workspace = decode_workspace(need, q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if metadata_ready:
        _check(lib.paged_decode_attention_flags(
            _ptr(out), _ptr(lse), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
            maxblk, _ptr(context_lens), B, Hq, Hkv, D, bs, NB, float(scale), _ptr(workspace),
            ws_bytes, int(num_splits), PKV_DECODE_METADATA_READY, _stream(stream)),
            "paged_decode_attention_flags")
        return out, lse
    _check(lib.paged_decode_attention(_ptr(out), _ptr(lse), _ptr(q), _ptr(k_cache),
                                      _ptr(v_cache), _ptr(block_tables), maxblk,
                                      _ptr(context_lens), B, Hq, Hkv, D, bs, NB, float(scale),
                                      _ptr(workspace), ws_bytes, int(num_splits),
                                      _stream(stream)), "paged_decode_attention")
    return out, lse


def paged_decode_attention_store(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                                 slot_mapping: torch.Tensor, k_cache: torch.Tensor,
                                 v_cache: torch.Tensor, block_tables: torch.Tensor,
                                 context_lens: torch.Tensor, scale: float,
                                 out: Optional[torch.Tensor] = None,
                                 lse: Optional[torch.Tensor] = None,
                                 workspace: Optional[torch.Tensor] = None, num_splits: int = 0,
                                 want_lse: bool = True, stream=None
                                 ) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Store the step's new tokens (k_new / v_new bf16 [B, Hkv, D] at
    slot_mapping[b], which must be -1 or the slot of position
    context_lens[b] - 1) and decode, in one launch.  Returns (out, lse) as
    paged_decode_attention."""
    lib = load_library()
    NB, bs, Hkv, D = _pool_dims(k_cache, v_cache)
    _need(q, "q", torch.bfloat16, 3)
    B, Hq, Dq = q.shape
    if Dq != D:
        raise ValueError("q head_dim differs from the cache's")
    for name, t in (("k_new", k_new), ("v_new", v_new)):
        _need(t, name, torch.bfloat16, 3, contiguous=False)
        if tuple(t.shape) != (B, Hkv, D) or t.stride(2) != 1 or t.stride(1) != D:
            raise ValueError(f"{name} must be [B, {Hkv}, {D}] with contiguous rows")
    _need(slot_mapping, "slot_mapping", torch.int32, 1)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(context_lens, "context_lens", torch.int32, 1)
    maxblk = block_tables.shape[1]
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    need = paged_decode_workspace_bytes(B, Hq, Hkv, D, maxblk, bs, num_splits)
    if workspace is None and need:
        workspace = decode_workspace(need, q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.paged_decode_attention_store(
        _ptr(out), _ptr(lse), _ptr(q), _ptr(k_new), _ptr(v_new), k_new.stride(0),
        v_new.stride(0), _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        maxblk, _ptr(context_lens), B, Hq, Hkv, D, bs, NB, float(scale), _ptr(workspace),
        ws_bytes, int(num_splits), _stream(stream)), "paged_decode_attention_store")
    return out, lse


def _fp8_pool_dims(k_cache: torch.Tensor, v_cache: torch.Tensor):
    for name, t in (("k_cache", k_cache), ("v_cache", v_cache)):
        _need(t, name, torch.uint8, 4)
    if k_cache.shape != v_cache.shape:
        raise ValueError("k_cache and v_cache shapes differ")
    NB, bs, Hkv, D = k_cache.shape
    return NB, bs, Hkv, D


def kv_cache_store_fp8(k: torch.Tensor, v: torch.Tensor, k_cache: torch.Tensor,
                       v_cache: torch.Tensor, slot_mapping: torch.Tensor, k_scale: float,
                       v_scale: float, stream=None) -> None:
    """Store bf16 k/v [T, Hkv, D] into uint8 E4M3 pools [NB, bs, Hkv, D] (one
    scale per tensor)."""
    lib = load_library()
    NB, bs, Hkv, D = _fp8_pool_dims(k_cache, v_cache)
    for name, t in (("k", k), ("v", v)):
        _need(t, name, torch.bfloat16, 3, contiguous=False)
        if t.stride(2) != 1 or t.stride(1) != D:
            raise ValueError(f"{name}: each token's [Hkv, D] rows must be contiguous")
    _need(slot_mapping, "slot_mapping", torch.int32, 1)
    T = k.shape[0]
    _check(lib.kv_cache_store_fp8(_ptr(k), _ptr(v), k.stride(0), v.stride(0), _ptr(k_cache),
                                  _ptr(v_cache), _ptr(slot_mapping), T, Hkv, D, bs, NB,
                                  float(k_scale), float(v_scale), _stream(stream)),
           "kv_cache_store_fp8")


def paged_decode_attention_fp8(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                               block_tables: torch.Tensor, context_lens: torch.Tensor,
                               scale: float, k_scale: float, v_scale: float,
                               out: Optional[torch.Tensor] = None,
                               lse: Optional[torch.Tensor] = None,
                               workspace: Optional[torch.Tensor] = None, num_splits: int = 0,
                               want_lse: bool = True, stream=None
                               ) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Decode over uint8 E4M3 pools; q bf16 [B, Hq, D].  Returns (out bf16
    [B, Hq, D], lse fp32 [B, Hq] or None)."""
    lib = load_library()
    NB, bs, Hkv, D = _fp8_pool_dims(k_cache, v_cache)
    _need(q, "q", torch.bfloat16, 3)
    B, Hq, Dq = q.shape
    if Dq != D:
        raise ValueError("q head_dim differs from the cache's")
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(context_lens, "context_lens", torch.int32, 1)
    maxblk = block_tables.shape[1]
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    need = paged_decode_workspace_bytes(B, Hq, Hkv, D, maxblk, bs, num_splits)
    if workspace is None and need:
        workspace = decode_workspace(need, q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.paged_decode_attention_fp8(
        _ptr(out), _ptr(lse), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), maxblk,
        _ptr(context_lens), B, Hq, Hkv, D, bs, NB, float(scale), float(k_scale), float(v_scale),
        _ptr(workspace), ws_bytes, int(num_splits), _stream(stream)),
        "paged_decode_attention_fp8")
    return out, lse


def paged_decode_attention_fp8_store(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                                     slot_mapping: torch.Tensor, k_cache: torch.Tensor,
                                     v_cache: torch.Tensor, block_tables: torch.Tensor,
                                     context_lens: torch.Tensor, scale: float, k_scale: float,
                                     v_scale: float, out: Optional[torch.Tensor] = None,
                                     lse: Optional[torch.Tensor] = None,
                                     workspace: Optional[torch.Tensor] = None,
                                     num_splits: int = 0, want_lse: bool = True, stream=None
                                     ) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """kv_cache_store_fp8 of the new tokens (bf16 [B, Hkv, D], slot_mapping[b]
    -1 or the slot of position context_lens[b] - 1) and the E4M3 decode, in
    one launch.  Returns (out, lse) as paged_decode_attention_fp8."""
    lib = load_library()
    NB, bs, Hkv, D = _fp8_pool_dims(k_cache, v_cache)
    _need(q, "q", torch.bfloat16, 3)
    B, Hq, Dq = q.shape
    if Dq != D:
        raise ValueError("q head_dim differs from the cache's")
    for name, t in (("k_new", k_new), ("v_new", v_new)):
        _need(t, name, torch.bfloat16, 3, contiguous=False)
        if tuple(t.shape) != (B, Hkv, D) or t.stride(2) != 1 or t.stride(1) != D:
            raise ValueError(f"{name} must be [B, {Hkv}, {D}] with contiguous rows")
    _need(slot_mapping, "slot_mapping", torch.int32, 1)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(context_lens, "context_lens", torch.int32, 1)
    maxblk = block_tables.shape[1]
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    need = paged_decode_workspace_bytes(B, Hq, Hkv, D, maxblk, bs, num_splits)
    if workspace is None and need:
        workspace = decode_workspace(need, q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.paged_decode_attention_fp8_store(
        _ptr(out), _ptr(lse), _ptr(q), _ptr(k_new), _ptr(v_new), k_new.stride(0),
        v_new.stride(0), _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        maxblk, _ptr(context_lens), B, Hq, Hkv, D, bs, NB, float(scale), float(k_scale),
        float(v_scale), _ptr(workspace), ws_bytes, int(num_splits), _stream(stream)),
        "paged_decode_attention_fp8_store")
    return out, lse


def paged_decode_multiquery_workspace_bytes(B: int, q_len: int, Hq: int, Hkv: int, D: int,
                                            max_blocks_per_seq: int, block_size: int = 256,
                                            num_splits: int = 0) -> int:
    return int(load_library().paged_decode_multiquery_workspace_bytes(
        B, q_len, Hq, Hkv, D, max_blocks_per_seq, block_size, num_splits))


def paged_decode_attention_multiquery(q: torch.Tensor, k_cache: torch.Tensor,
                                      v_cache: torch.Tensor, block_tables: torch.Tensor,
                                      context_lens: torch.Tensor, scale: float,
                                      out: Optional[torch.Tensor] = None,
                                      lse: Optional[torch.Tensor] = None,
                                      workspace: Optional[torch.Tensor] = None,
                                      num_splits: int = 0, want_lse: bool = True, stream=None
                                      ) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """q bf16 [B, q_len, Hq, D]: q_len new positions per sequence (already stored
    in the cache, counted in context_lens).  Returns (out bf16 [B, q_len, Hq, D],
    lse fp32 [B, q_len, Hq] or None)."""
    lib = load_library()
    NB, bs, Hkv, D = _pool_dims(k_cache, v_cache)
    _need(q, "q", torch.bfloat16, 4)
    B, q_len, Hq, Dq = q.shape
    if Dq != D:
        raise ValueError("q head_dim differs from the cache's")
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(context_lens, "context_lens", torch.int32, 1)
    if block_tables.shape[0] != B or context_lens.shape[0] != B:
        raise ValueError("block_tables / context_lens batch differs from q")
    maxblk = block_tables.shape[1]
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, 4)
    if lse is None and want_lse:
        lse = torch.empty((B, q_len, Hq), dtype=torch.float32, device=q.device)
    if lse is not None:
        _need(lse, "lse", torch.float32, 3)
    need = paged_decode_multiquery_workspace_bytes(B, q_len, Hq, Hkv, D, maxblk, bs, num_splits)
    if workspace is None and need:
        workspace = decode_workspace(need, q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.paged_decode_attention_multiquery(
        _ptr(out), _ptr(lse), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), maxblk,
        _ptr(context_lens), B, q_len, Hq, Hkv, D, bs, NB, float(scale), _ptr(workspace), ws_bytes,
        int(num_splits), _stream(stream)), "paged_decode_attention_multiquery")
    return out, lse


def paged_decode_shared_prefix_workspace_bytes(B: int, Hq: int, Hkv: int, D: int,
                                               max_blocks_per_seq: int,
                                               shared_prefix_tokens: int,
                                               block_size: int = 256,
                                               num_splits: int = 0) -> int:
    return int(load_library().paged_decode_shared_prefix_workspace_bytes(
        B, Hq, Hkv, D, max_blocks_per_seq, block_size, shared_prefix_tokens, num_splits))


def paged_decode_attention_shared_prefix(q: torch.Tensor, k_cache: torch.Tensor,
                                         v_cache: torch.Tensor, block_tables: torch.Tensor,
                                         context_lens: torch.Tensor, scale: float,
                                         shared_prefix_tokens: int,
                                         out: Optional[torch.Tensor] = None,
                                         lse: Optional[torch.Tensor] = None,
                                         workspace: Optional[torch.Tensor] = None,
                                         num_splits: int = 0, want_lse: bool = True,
                                         stream=None
                                         ) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Decode for a batch whose sequences all start with the same
    `shared_prefix_tokens` tokens (the same physical blocks at the start of every
    table row).  Same results as paged_decode_attention."""
    lib = load_library()
    NB, bs, Hkv, D = _pool_dims(k_cache, v_cache)
    _need(q, "q", torch.bfloat16, 3)
    B, Hq, _ = q.shape
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(context_lens, "context_lens", torch.int32, 1)
    maxblk = block_tables.shape[1]
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, 3)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if lse is not None:
        _need(lse, "lse", torch.float32, 2)
    need = paged_decode_shared_prefix_workspace_bytes(B, Hq, Hkv, D, maxblk,
                                                      shared_prefix_tokens, bs, num_splits)
    if workspace is None and need:
        workspace = decode_workspace(need, q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.paged_decode_attention_shared_prefix(
        _ptr(out), _ptr(lse), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), maxblk,
        _ptr(context_lens), B, Hq, Hkv, D, bs, NB, float(scale), int(shared_prefix_tokens),
        _ptr(workspace), ws_bytes, int(num_splits), _stream(stream)),
        "paged_decode_attention_shared_prefix")
    return out, lse


NOALLOC_SCRATCH_BYTES = 16 << 20


def paged_decode_attention_noalloc(q: torch.Tensor, k_cache: torch.Tensor,
                                   v_cache: torch.Tensor, block_tables: torch.Tensor,
                                   context_lens: torch.Tensor, scale: float,
                                   out: torch.Tensor, lse: Optional[torch.Tensor] = None,
                                   num_splits: int = 0, stream=None) -> None:
    """Decode attention for callers that cannot allocate device memory: the
    split scratch is a fixed 16 MiB array inside the library instead of a
    caller-provided workspace, and the caller passes `out` (and optionally
    `lse`) already allocated.  Calls that overlap on the GPU race on that array."""
    lib = load_library()
    NB, bs, Hkv, D = _pool_dims(k_cache, v_cache)
    _need(q, "q", torch.bfloat16, 3)
    B, Hq, _ = q.shape
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(context_lens, "context_lens", torch.int32, 1)
    _need(out, "out", torch.bfloat16, 3)
    if lse is not None:
        _need(lse, "lse", torch.float32, 2)
    _check(lib.paged_decode_attention_noalloc(
        _ptr(out), _ptr(lse), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        block_tables.shape[1], _ptr(context_lens), B, Hq, Hkv, D, bs, NB, float(scale),
        int(num_splits), _stream(stream)), "paged_decode_attention_noalloc")


def paged_prefill_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                            block_tables: torch.Tensor, cu_seqlens_q: torch.Tensor,
                            cu_seqlens_k: torch.Tensor, max_seqlen_q: int, max_seqlen_k: int,
                            scale: float, out: Optional[torch.Tensor] = None,
                            lse: Optional[torch.Tensor] = None, want_lse: bool = True,
                            stream=None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """q bf16 [sum Lq, Hq, D]; cu_seqlens int32 [B+1].  The new tokens' K/V must
    already be stored in the pool.  Returns (out bf16 [sum Lq, Hq, D], lse fp32
    [sum Lq, Hq] or None)."""
    lib = load_library()
    NB, bs, Hkv, D = _pool_dims(k_cache, v_cache)
    _need(q, "q", torch.bfloat16, 3)
    Nq, Hq, Dq = q.shape
    if Dq != D:
        raise ValueError("q head_dim differs from the cache's")
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    _need(cu_seqlens_k, "cu_seqlens_k", torch.int32, 1)
    B = cu_seqlens_q.shape[0] - 1
    if cu_seqlens_k.shape[0] != B + 1 or block_tables.shape[0] != B:
        raise ValueError("cu_seqlens / block_tables batch sizes differ")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, 3)
    if lse is None and want_lse:
        lse = torch.empty((Nq, Hq), dtype=torch.float32, device=q.device)
    if lse is not None:
        _need(lse, "lse", torch.float32, 2)
    _check(lib.paged_prefill_attention(_ptr(out), _ptr(lse), _ptr(q), _ptr(k_cache),
                                       _ptr(v_cache), _ptr(block_tables),
                                       block_tables.shape[1], _ptr(cu_seqlens_q),
                                       _ptr(cu_seqlens_k), B, int(max_seqlen_q),
                                       int(max_seqlen_k), Hq, Hkv, D, bs, NB, float(scale),
                                       _stream(stream)), "paged_prefill_attention")
    return out, lse


def testing_set_wait_fault(wait_limit_ns: int, withhold_tile: int = -1) -> None:
    """For tests only: lower the kernels' wait limit and make the copy
    producers withhold one tile (see pkv_testing_set_wait_fault in pkv.h);
    testing_set_wait_fault(0, -1) turns it off."""
    _check(load_library().pkv_testing_set_wait_fault(int(wait_limit_ns), int(withhold_tile)),
           "pkv_testing_set_wait_fault")


def get_device_error(stream=None) -> int:
    """Synchronise the stream and read-and-clear the device error word."""
    return int(load_library().pkv_get_device_error(_stream(stream)))
