"""Python binding of the host block manager (include/pkv_blocks.h), argument
marshalling only; the manager itself is C++ inside libpkv.so."""

from __future__ import annotations

import ctypes
from typing import List, Optional, Sequence, Tuple

import numpy as np

from . import pkv

BM_OK = 0
BM_ERR_ARG = -1
BM_ERR_NO_BLOCKS = -2
BM_ERR_NO_SEQ = -3
BM_ERR_EXISTS = -4
BM_ERR_SMALL = -5
_NAMES = {BM_ERR_ARG: "bad argument", BM_ERR_NO_BLOCKS: "not enough free blocks",
          BM_ERR_NO_SEQ: "unknown sequence", BM_ERR_EXISTS: "sequence exists",
          BM_ERR_SMALL: "output too small"}


class BlockManagerError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {_NAMES.get(status, status)}")


_declared = False


def _lib():
    global _declared
    lib = pkv.load_library()
    if not _declared:
        P, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        lib.pkv_bm_create.argtypes = [i64, i32]
        lib.pkv_bm_create.restype = P
        lib.pkv_bm_destroy.argtypes = [P]
        lib.pkv_bm_destroy.restype = None
        lib.pkv_bm_num_free_blocks.argtypes = [P]
        lib.pkv_bm_num_free_blocks.restype = i64
        lib.pkv_bm_add_sequence.argtypes = [P, i64, P, i64, P]
        lib.pkv_bm_append_token.argtypes = [P, i64, i32, P, P, P]
        lib.pkv_bm_fork.argtypes = [P, i64, i64]
        lib.pkv_bm_free_sequence.argtypes = [P, i64]
        lib.pkv_bm_num_tokens.argtypes = [P, i64]
        lib.pkv_bm_num_tokens.restype = i64
        lib.pkv_bm_num_blocks.argtypes = [P, i64]
        lib.pkv_bm_num_blocks.restype = i64
        lib.pkv_bm_block_table.argtypes = [P, i64, P, i64]
        lib.pkv_bm_slot_mapping.argtypes = [P, i64, i64, i64, P]
        lib.pkv_bm_ref_count.argtypes = [P, i64]
        lib.pkv_bm_ref_count.restype = i64
        for f in ("pkv_bm_add_sequence", "pkv_bm_append_token", "pkv_bm_fork",
                  "pkv_bm_free_sequence", "pkv_bm_block_table", "pkv_bm_slot_mapping"):
            getattr(lib, f).restype = i32
        _declared = True
    return lib


def _check(st: int, what: str):
    if st != BM_OK:
        raise BlockManagerError(st, what)


class BlockManager:
    """Free list, content hash -> block id prefix cache, reference counts and
    copy-on-write for a pool of `num_blocks` blocks of `block_size` tokens."""

    def __init__(self, num_blocks: int, block_size: int = 256):
        self._lib = _lib()
        self._h = self._lib.pkv_bm_create(int(num_blocks), int(block_size))
        if not self._h:
            raise BlockManagerError(BM_ERR_ARG, "pkv_bm_create")
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)

    def __del__(self):
        h, self._h = getattr(self, "_h", None), None
        if h:
            self._lib.pkv_bm_destroy(h)

    @property
    def num_free_blocks(self) -> int:
        return int(self._lib.pkv_bm_num_free_blocks(self._h))

    def add_sequence(self, seq_id: int, tokens: Sequence[int]) -> int:
        """Admit a sequence with its prompt; returns how many leading prompt
        tokens already have K/V in the pool (prefix-cache hits)."""
        t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        cached = ctypes.c_int64(0)
        _check(self._lib.pkv_bm_add_sequence(self._h, int(seq_id), t.ctypes.data, t.size,
                                             ctypes.byref(cached)), "add_sequence")
        return int(cached.value)

    def append_token(self, seq_id: int, token: int) -> Tuple[int, Optional[Tuple[int, int]]]:
        """Returns (slot of the new token, (copy_src, copy_dst) or None)."""
        slot = ctypes.c_int64(0)
        src, dst = ctypes.c_int32(-1), ctypes.c_int32(-1)
        _check(self._lib.pkv_bm_append_token(self._h, int(seq_id), int(token),
                                             ctypes.byref(slot), ctypes.byref(src),
                                             ctypes.byref(dst)), "append_token")
        copy = (int(src.value), int(dst.value)) if src.value >= 0 else None
        return int(slot.value), copy

    def fork(self, parent_id: int, child_id: int) -> None:
        _check(self._lib.pkv_bm_fork(self._h, int(parent_id), int(child_id)), "fork")

    def free_sequence(self, seq_id: int) -> None:
        _check(self._lib.pkv_bm_free_sequence(self._h, int(seq_id)), "free_sequence")

    def num_tokens(self, seq_id: int) -> int:
        n = int(self._lib.pkv_bm_num_tokens(self._h, int(seq_id)))
        _check(min(n, 0), "num_tokens")
        return n

    def num_blocks_of(self, seq_id: int) -> int:
        n = int(self._lib.pkv_bm_num_blocks(self._h, int(seq_id)))
        _check(min(n, 0), "num_blocks")
        return n

    def block_table(self, seq_id: int, max_blocks: int) -> np.ndarray:
        out = np.empty(int(max_blocks), np.int32)
        _check(self._lib.pkv_bm_block_table(self._h, int(seq_id), out.ctypes.data,
                                            out.size), "block_table")
        return out

    def block_tables(self, seq_ids: Sequence[int], max_blocks: int) -> np.ndarray:
        return np.stack([self.block_table(s, max_blocks) for s in seq_ids])

    def slot_mapping(self, seq_id: int, begin: int, end: int) -> np.ndarray:
        out = np.empty(max(int(end) - int(begin), 0), np.int32)
        _check(self._lib.pkv_bm_slot_mapping(self._h, int(seq_id), int(begin), int(end),
                                             out.ctypes.data), "slot_mapping")
        return out

    def ref_count(self, block_id: int) -> int:
        n = int(self._lib.pkv_bm_ref_count(self._h, int(block_id)))
        _check(min(n, 0), "ref_count")
        return n
