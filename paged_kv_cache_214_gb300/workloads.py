"""Seeded synthetic inputs for paged KV-cache attention.

This module only draws random numbers and hands out physical blocks the way a
host block manager would; it contains none of the attention or store
arithmetic.  Both the GPU path and the CPU oracle are fed from the tensors it
returns.

Shapes follow Qwen3-style attention (head_dim 128, GQA) with 256-token blocks
("Nano-vLLM System Architecture Analysis", §2 Core Components, "Paged KV Cache";
§6 Architecture Support).  Every workload is synthetic: bf16 values are i.i.d.
N(0, 1); physical block ids come from a seeded permutation of the pool, so a
sequence's blocks are scattered; blocks that no sequence uses also hold N(0, 1)
data, so a stray read shows up as a wrong answer.

The five named workloads:

1. ``tiny-decode``: 4 sequences, context lengths {17, 256, 300, 513}, 16 query /
   8 kv heads, 16-block pool, plus a store of the 4 new tokens.
2. ``decode-b64``: 64 sequences, 16 q / 8 kv heads, context U{512..4096},
   2048-block pool, one new token stored per sequence before attention.
3. ``prefix-shared-decode-b256``: 256 sequences, 32 q / 8 kv heads; every
   sequence starts with the same 2048-token prefix (8 shared blocks), then a
   private suffix of U{0..6144} cached tokens, then the new token (so the
   context is 2049..8193 and the new token never lands in a shared block);
   8192-block pool.
4. ``chunked-prefill-b16``: 16 sequences, 32 q / 8 kv heads, 1024 cached prefix
   tokens + 512 new tokens each (cu_seqlens varlen), 2048-block pool.
5. ``long-decode-b8``: 8 sequences, 32 q / 8 kv heads, context
   U{32768..131072}, 4096-block pool.

Seeds: workload n uses seed 214000 + n.
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import torch

HEAD_DIM = 128
BLOCK_SIZE = 256


def seed_for(config_id: int) -> int:
    return 214000 + int(config_id)


def _cdiv(a: int, b: int) -> int:
    return -(-a // b)


def _randn_bf16(shape, gen: torch.Generator, device) -> torch.Tensor:
    return torch.randn(shape, generator=gen, dtype=torch.bfloat16, device=device)


def _pool(num_blocks: int, Hkv: int, D: int, bs: int, seed: int, device):
    """K and V pools [num_blocks, bs, Hkv, D], bf16 N(0,1), on ``device``."""
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(seed * 7 + 1)
    k_cache = _randn_bf16((num_blocks, bs, Hkv, D), g, dev)
    v_cache = _randn_bf16((num_blocks, bs, Hkv, D), g, dev)
    return k_cache, v_cache


class _BlockAllocator:
    """Hands out physical block ids in the order of a seeded permutation."""

    def __init__(self, num_blocks: int, gen: torch.Generator):
        self.order = torch.randperm(num_blocks, generator=gen).tolist()
        self.next = 0

    def take(self, n: int) -> List[int]:
        if self.next + n > len(self.order):
            raise ValueError("pool too small for this workload")
        out = self.order[self.next:self.next + n]
        self.next += n
        return out


def _slot(table_row: Sequence[int], pos: int, bs: int) -> int:
    # What a host block manager emits for logical position ``pos``: the physical
    # block holding it and the offset inside that block.
    return table_row[pos // bs] * bs + pos % bs


@dataclass
class DecodeWorkload:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    block_size: int
    num_blocks: int
    scale: float
    q: torch.Tensor              # bf16 [B, Hq, D]
    k_new: torch.Tensor          # bf16 [B, Hkv, D]   token stored this step
    v_new: torch.Tensor          # bf16 [B, Hkv, D]
    slot_mapping: torch.Tensor   # int32 [B]          slot of the new token (-1 = none)
    block_tables: torch.Tensor   # int32 [B, max_blocks_per_seq], padded with -1
    context_lens: torch.Tensor   # int32 [B]          includes the new token
    k_cache: torch.Tensor        # bf16 [NB, bs, Hkv, D]
    v_cache: torch.Tensor
    shared_prefix_blocks: int = 0
    extra_tables: List[torch.Tensor] = field(default_factory=list)
    extra_slots: List[torch.Tensor] = field(default_factory=list)

    @property
    def kv_tokens(self) -> int:
        return int(self.context_lens.sum())

    @property
    def unique_kv_tokens(self) -> int:
        """Context tokens counting each physical block's tokens once."""
        shared = self.shared_prefix_blocks * self.block_size
        if self.B == 0:
            return 0
        return int(self.context_lens.sum()) - (self.B - 1) * shared if shared else self.kv_tokens


@dataclass
class PrefillWorkload:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    block_size: int
    num_blocks: int
    scale: float
    q: torch.Tensor              # bf16 [sum Lq, Hq, D]
    k_new: torch.Tensor          # bf16 [sum Lq, Hkv, D]
    v_new: torch.Tensor
    slot_mapping: torch.Tensor   # int32 [sum Lq]
    block_tables: torch.Tensor   # int32 [B, max_blocks_per_seq]
    cu_seqlens_q: torch.Tensor   # int32 [B+1]
    cu_seqlens_k: torch.Tensor   # int32 [B+1]
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    q_lens: List[int] = field(default_factory=list)
    k_lens: List[int] = field(default_factory=list)

    @property
    def max_seqlen_q(self) -> int:
        return max(self.q_lens) if self.q_lens else 0

    @property
    def max_seqlen_k(self) -> int:
        return max(self.k_lens) if self.k_lens else 0


def make_decode(context_lens: Sequence[int], Hq: int, Hkv: int, num_blocks: int,
                seed: int, *, name: str = "decode", D: int = HEAD_DIM,
                block_size: int = BLOCK_SIZE, shared_prefix_tokens: int = 0,
                store_new_token: bool = True, pool_device="cpu",
                max_blocks_per_seq: Optional[int] = None,
                rotations: int = 1) -> DecodeWorkload:
    """Decode batch: one query row per sequence and head.

    ``context_lens`` count the new token.  With ``shared_prefix_tokens`` (a
    multiple of ``block_size``) every sequence's table starts with the same
    physical blocks.  ``rotations`` > 1 also allocates that many further,
    disjoint sets of blocks for the same lengths (``extra_tables`` /
    ``extra_slots``), so that a benchmark can cycle through batches that share no
    memory.
    """
    B = len(context_lens)
    lens = [int(x) for x in context_lens]
    if shared_prefix_tokens % block_size:
        raise ValueError("shared prefix must be whole blocks")
    n_shared = shared_prefix_tokens // block_size
    for L in lens:
        if shared_prefix_tokens and (L < shared_prefix_tokens or
                                     (store_new_token and L == shared_prefix_tokens)):
            raise ValueError("with a shared prefix every context must cover it, and a new "
                             "token must land past it")
    gen = torch.Generator().manual_seed(seed)
    nblk = [_cdiv(L, block_size) for L in lens]
    maxblk = max_blocks_per_seq or max([1] + nblk)
    if max(nblk + [0]) > maxblk:
        raise ValueError("max_blocks_per_seq too small")
    alloc = _BlockAllocator(num_blocks, gen)
    tables, slots = [], []
    for rot in range(rotations):
        shared = alloc.take(n_shared)
        table = torch.full((B, maxblk), -1, dtype=torch.int32)
        slot = torch.full((B,), -1, dtype=torch.int32)
        for b in range(B):
            row = shared + alloc.take(nblk[b] - n_shared)
            table[b, :len(row)] = torch.tensor(row, dtype=torch.int32)
            if store_new_token and lens[b] > 0:
                slot[b] = _slot(row, lens[b] - 1, block_size)
        tables.append(table)
        slots.append(slot)
    q = _randn_bf16((B, Hq, D), gen, "cpu")
    k_new = _randn_bf16((B, Hkv, D), gen, "cpu")
    v_new = _randn_bf16((B, Hkv, D), gen, "cpu")
    k_cache, v_cache = _pool(num_blocks, Hkv, D, block_size, seed, pool_device)
    return DecodeWorkload(
        name=name, B=B, Hq=Hq, Hkv=Hkv, D=D, block_size=block_size,
        num_blocks=num_blocks, scale=D ** -0.5, q=q, k_new=k_new, v_new=v_new,
        slot_mapping=slots[0], block_tables=tables[0],
        context_lens=torch.tensor(lens, dtype=torch.int32), k_cache=k_cache,
        v_cache=v_cache, shared_prefix_blocks=n_shared,
        extra_tables=tables[1:], extra_slots=slots[1:])


def make_prefill(prefix_lens: Sequence[int], new_lens: Sequence[int], Hq: int,
                 Hkv: int, num_blocks: int, seed: int, *, name: str = "prefill",
                 D: int = HEAD_DIM, block_size: int = BLOCK_SIZE,
                 pool_device="cpu",
                 max_blocks_per_seq: Optional[int] = None) -> PrefillWorkload:
    """Chunked prefill batch: sequence i has prefix_lens[i] tokens already in the
    pool and new_lens[i] new tokens (queries, and K/V to store)."""
    B = len(prefix_lens)
    P = [int(x) for x in prefix_lens]
    N = [int(x) for x in new_lens]
    gen = torch.Generator().manual_seed(seed)
    k_lens = [p + n for p, n in zip(P, N)]
    nblk = [_cdiv(L, block_size) for L in k_lens]
    maxblk = max_blocks_per_seq or max([1] + nblk)
    alloc = _BlockAllocator(num_blocks, gen)
    table = torch.full((B, maxblk), -1, dtype=torch.int32)
    slots = []
    for i in range(B):
        row = alloc.take(nblk[i])
        if row:
            table[i, :len(row)] = torch.tensor(row, dtype=torch.int32)
        slots += [_slot(row, P[i] + r, block_size) for r in range(N[i])]
    total_q = sum(N)
    q = _randn_bf16((total_q, Hq, D), gen, "cpu")
    k_new = _randn_bf16((total_q, Hkv, D), gen, "cpu")
    v_new = _randn_bf16((total_q, Hkv, D), gen, "cpu")
    cu_q = [0]
    cu_k = [0]
    for n, L in zip(N, k_lens):
        cu_q.append(cu_q[-1] + n)
        cu_k.append(cu_k[-1] + L)
    k_cache, v_cache = _pool(num_blocks, Hkv, D, block_size, seed, pool_device)
    return PrefillWorkload(
        name=name, B=B, Hq=Hq, Hkv=Hkv, D=D, block_size=block_size,
        num_blocks=num_blocks, scale=D ** -0.5, q=q, k_new=k_new, v_new=v_new,
        slot_mapping=torch.tensor(slots, dtype=torch.int32), block_tables=table,
        cu_seqlens_q=torch.tensor(cu_q, dtype=torch.int32),
        cu_seqlens_k=torch.tensor(cu_k, dtype=torch.int32), k_cache=k_cache,
        v_cache=v_cache, q_lens=N, k_lens=k_lens)


def _uniform_ints(lo: int, hi: int, n: int, seed: int) -> List[int]:
    g = torch.Generator().manual_seed(seed ^ 0x5EED)
    return torch.randint(lo, hi + 1, (n,), generator=g).tolist()


CONFIG_NAMES = {
    1: "tiny-decode",
    2: "decode-b64",
    3: "prefix-shared-decode-b256",
    4: "chunked-prefill-b16",
    5: "long-decode-b8",
}


def config_workload(config_id: int, pool_device="cpu", rotations: int = 1):
    """The named workload ``config_id`` (1..5)."""
    s = seed_for(config_id)
    name = CONFIG_NAMES[config_id]
    if config_id == 1:
        return make_decode([17, 256, 300, 513], 16, 8, 16, s, name=name,
                           pool_device=pool_device, rotations=rotations)
    if config_id == 2:
        lens = _uniform_ints(512, 4096, 64, s)
        return make_decode(lens, 16, 8, 2048, s, name=name,
                           pool_device=pool_device, rotations=rotations)
    if config_id == 3:
        suffix = _uniform_ints(0, 6144, 256, s)
        lens = [2048 + x + 1 for x in suffix]
        return make_decode(lens, 32, 8, 8192, s, name=name,
                           shared_prefix_tokens=2048, pool_device=pool_device,
                           rotations=rotations)
    if config_id == 4:
        return make_prefill([1024] * 16, [512] * 16, 32, 8, 2048, s, name=name,
                            pool_device=pool_device)
    if config_id == 5:
        lens = _uniform_ints(32768, 131072, 8, s)
        return make_decode(lens, 32, 8, 4096, s, name=name,
                           pool_device=pool_device, rotations=rotations)
    raise ValueError(f"unknown workload {config_id}")
