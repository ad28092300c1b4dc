"""Python binding of the CUDA-graph decode runner (include/pkv_graphs.h).

Argument marshalling only: the runner's static buffers are torch tensors that
this module allocates once (device memory is PyTorch's job here); the padding,
the graph capture and replay, and every kernel run in libpkv.so.  Decode
steps are captured per batch bucket and replayed ("Nano-vLLM System
Architecture Analysis", §2 Core Components, "CUDA Graphs"; comparison table,
"Variable-batch CUDA Graphs").
"""

from __future__ import annotations

import ctypes
from typing import Optional, Sequence, Tuple

import torch

from . import pkv

_I32P = ctypes.POINTER(ctypes.c_int32)


class _Config(ctypes.Structure):
    """pkv_decode_graphs_config, field for field."""
    _fields_ = [("Hq", ctypes.c_int), ("Hkv", ctypes.c_int), ("D", ctypes.c_int),
                ("block_size", ctypes.c_int), ("max_blocks_per_seq", ctypes.c_int),
                ("max_batch", ctypes.c_int), ("num_blocks", ctypes.c_int64),
                ("kv_fp8", ctypes.c_int), ("scale", ctypes.c_float),
                ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float),
                ("num_buckets", ctypes.c_int), ("buckets", _I32P),
                ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
                ("q", ctypes.c_void_p), ("k_new", ctypes.c_void_p), ("v_new", ctypes.c_void_p),
                ("slot_mapping", ctypes.c_void_p), ("block_tables", ctypes.c_void_p),
                ("context_lens", ctypes.c_void_p), ("out", ctypes.c_void_p),
                ("lse", ctypes.c_void_p), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t)]


_declared = False


def _lib():
    """libpkv.so with the runner's signatures declared."""
    global _declared
    lib = pkv.load_library()
    if not _declared:
        P, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        CP = ctypes.POINTER(_Config)
        lib.pkv_decode_graphs_config_bytes.argtypes = []
        lib.pkv_decode_graphs_config_bytes.restype = sz
        lib.pkv_decode_graphs_default_buckets.argtypes = [i32, _I32P, i32]
        lib.pkv_decode_graphs_default_buckets.restype = i32
        lib.pkv_decode_graphs_pick_bucket.argtypes = [_I32P, i32, i32]
        lib.pkv_decode_graphs_pick_bucket.restype = i32
        lib.pkv_decode_graphs_workspace_bytes.argtypes = [CP]
        lib.pkv_decode_graphs_workspace_bytes.restype = sz
        lib.pkv_decode_graphs_create.argtypes = [CP, ctypes.POINTER(P)]
        lib.pkv_decode_graphs_create.restype = i32
        lib.pkv_decode_graphs_buckets.argtypes = [P, _I32P, i32]
        lib.pkv_decode_graphs_buckets.restype = i32
        lib.pkv_decode_graphs_run.argtypes = [P, i32, P]
        lib.pkv_decode_graphs_run.restype = i32
        lib.pkv_decode_graphs_destroy.argtypes = [P]
        lib.pkv_decode_graphs_destroy.restype = None
        if lib.pkv_decode_graphs_config_bytes() != ctypes.sizeof(_Config):
            raise RuntimeError("pkv_decode_graphs_config layout differs from the binding's")
        _declared = True
    return lib


def default_buckets(max_batch: int) -> list:
    """The default bucket sizes kept for max_batch rows (powers of two up to 512)."""
    lib = _lib()
    n = lib.pkv_decode_graphs_default_buckets(int(max_batch), None, 0)
    if n < 0:
        raise pkv.PkvError(n, "pkv_decode_graphs_default_buckets")
    arr = (ctypes.c_int32 * max(n, 1))()
    lib.pkv_decode_graphs_default_buckets(int(max_batch), arr, n)
    return list(arr[:n])


def pick_bucket(buckets: Sequence[int], B: int) -> int:
    """The bucket a batch of B runs in (0: none, the step runs eagerly)."""
    lib = _lib()
    arr = (ctypes.c_int32 * max(len(buckets), 1))(*buckets)
    r = lib.pkv_decode_graphs_pick_bucket(arr, len(buckets), int(B))
    if r < 0:
        raise pkv.PkvError(r, "pkv_decode_graphs_pick_bucket")
    return r


class DecodeGraphs:
    """Decode steps (fused store + decode) replayed from CUDA graphs captured
    for each batch bucket over one pool.

    A step of B sequences: write rows [0, B) of ``q``, ``k_new``, ``v_new``,
    ``slot_mapping``, ``block_tables`` and ``context_lens`` (each allocated
    here for ``max_batch`` rows), call ``run(B)``, read rows [0, B) of ``out``
    and ``lse``.  ``step(...)`` does the writes (device copies on the stream)
    and the run in one call.
    """

    def __init__(self, k_cache: torch.Tensor, v_cache: torch.Tensor, Hq: int,
                 max_blocks_per_seq: int, max_batch: int, scale: float,
                 buckets: Optional[Sequence[int]] = None, k_scale: float = 1.0,
                 v_scale: float = 1.0, want_lse: bool = True):
        lib = _lib()
        if k_cache.dtype == torch.uint8:
            NB, bs, Hkv, D = pkv._fp8_pool_dims(k_cache, v_cache)
            fp8 = 1
        else:
            NB, bs, Hkv, D = pkv._pool_dims(k_cache, v_cache)
            fp8 = 0
        dev = k_cache.device
        bf = torch.bfloat16
        self.k_cache, self.v_cache = k_cache, v_cache
        self.max_batch = int(max_batch)
        self.q = torch.zeros((max_batch, Hq, D), dtype=bf, device=dev)
        self.k_new = torch.zeros((max_batch, Hkv, D), dtype=bf, device=dev)
        self.v_new = torch.zeros((max_batch, Hkv, D), dtype=bf, device=dev)
        self.slot_mapping = torch.full((max_batch,), -1, dtype=torch.int32, device=dev)
        self.block_tables = torch.zeros((max_batch, max_blocks_per_seq), dtype=torch.int32,
                                        device=dev)
        self.context_lens = torch.zeros((max_batch,), dtype=torch.int32, device=dev)
        self.out = torch.zeros((max_batch, Hq, D), dtype=bf, device=dev)
        self.lse = (torch.zeros((max_batch, Hq), dtype=torch.float32, device=dev)
                    if want_lse else None)
        self._buckets = (ctypes.c_int32 * max(len(buckets or ()), 1))(*(buckets or ()))
        cfg = _Config(Hq=Hq, Hkv=Hkv, D=D, block_size=bs,
                      max_blocks_per_seq=int(max_blocks_per_seq), max_batch=self.max_batch,
                      num_blocks=NB, kv_fp8=fp8, scale=float(scale), k_scale=float(k_scale),
                      v_scale=float(v_scale), num_buckets=len(buckets or ()),
                      buckets=ctypes.cast(self._buckets, _I32P),
                      k_cache=k_cache.data_ptr(), v_cache=v_cache.data_ptr(),
                      q=self.q.data_ptr(), k_new=self.k_new.data_ptr(),
                      v_new=self.v_new.data_ptr(), slot_mapping=self.slot_mapping.data_ptr(),
                      block_tables=self.block_tables.data_ptr(),
                      context_lens=self.context_lens.data_ptr(), out=self.out.data_ptr(),
                      lse=0 if self.lse is None else self.lse.data_ptr())
        with torch.cuda.device(dev):   # the split plan reads this device's SM count
            need = lib.pkv_decode_graphs_workspace_bytes(ctypes.byref(cfg))
        self.workspace = torch.zeros(max(need, 256), dtype=torch.uint8, device=dev)
        cfg.workspace = self.workspace.data_ptr()
        cfg.workspace_bytes = self.workspace.numel()
        # the runner's private stream is not ordered after torch's: finish the
        # fills above first; the graphs belong to the pool's device
        torch.cuda.current_stream(dev).synchronize()
        handle = ctypes.c_void_p()
        with torch.cuda.device(dev):
            st = lib.pkv_decode_graphs_create(ctypes.byref(cfg), ctypes.byref(handle))
        pkv._check(st, "pkv_decode_graphs_create")
        self._h = handle
        n = lib.pkv_decode_graphs_buckets(self._h, None, 0)
        arr = (ctypes.c_int32 * max(n, 1))()
        lib.pkv_decode_graphs_buckets(self._h, arr, n)
        self.buckets = list(arr[:n])

    def bucket_for(self, B: int) -> int:
        """The bucket run(B) replays (0: eager, above the largest bucket)."""
        return pick_bucket(self.buckets, B)

    def run(self, B: int, stream=None) -> None:
        """One step over rows [0, B) of the static buffers, on `stream` (default:
        the current stream of the pool's device)."""
        if self._h is None:
            raise RuntimeError("DecodeGraphs has been closed")
        if stream is None:
            stream = torch.cuda.current_stream(self.q.device)
        pkv._check(_lib().pkv_decode_graphs_run(self._h, int(B), pkv._stream(stream)),
                   "pkv_decode_graphs_run")

    def step(self, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
             slot_mapping: torch.Tensor, block_tables: torch.Tensor,
             context_lens: torch.Tensor, stream=None
             ) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
        """Copy one step's inputs into rows [0, B) and run it; returns views of
        rows [0, B) of out and lse."""
        B = q.shape[0]
        if B > self.max_batch:
            raise ValueError(f"batch {B} exceeds max_batch {self.max_batch}")
        W = self.block_tables.shape[1]
        if block_tables.shape[0] != B or block_tables.shape[1] > W:
            raise ValueError("block_tables must be [B, <= max_blocks_per_seq]")
        s = torch.cuda.current_stream(self.q.device) if stream is None else stream
        with torch.cuda.stream(s):
            self.q[:B].copy_(q)
            self.k_new[:B].copy_(k_new)
            self.v_new[:B].copy_(v_new)
            self.slot_mapping[:B].copy_(slot_mapping)
            self.block_tables[:B, :block_tables.shape[1]].copy_(block_tables)
            self.context_lens[:B].copy_(context_lens)
        self.run(B, stream=s)
        return self.out[:B], None if self.lse is None else self.lse[:B]

    def close(self) -> None:
        if getattr(self, "_h", None) is not None:
            torch.cuda.synchronize(self.q.device)
            _lib().pkv_decode_graphs_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
