"""The host block manager driving the GPU kernels through a small serving loop:
admit prompts (prefix-cache hits skip their prefill), prefill the rest, decode
steps, fork a sequence (copy-on-write on its next append), free and re-admit.
Every step's store, copies, prefill and decode are checked against the oracle
run on a host copy of the pool."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_close, bits
from paged_kv_cache_214_gb300 import pkv
from paged_kv_cache_214_gb300.blocks import BlockManager

pytestmark = pytest.mark.gpu

NB, BS, HKV, HQ, D = 40, 256, 8, 16, 128
MAXBLK = 8


class KV:
    """K/V of a token depends on the whole prefix: identical prefixes give
    identical K/V (what makes prefix caching valid)."""

    def __init__(self, seed):
        self.seed = seed

    def rows(self, tokens, begin, end):
        out_k, out_v = [], []
        for p in range(begin, end):
            key = hash((self.seed, tuple(tokens[:p + 1]))) & 0x7FFFFFFF
            g = torch.Generator().manual_seed(key)
            out_k.append(torch.randn((HKV, D), generator=g).to(torch.bfloat16))
            out_v.append(torch.randn((HKV, D), generator=g).to(torch.bfloat16))
        return torch.stack(out_k), torch.stack(out_v)


def test_block_manager_drives_store_prefill_decode_and_cow():
    dev = "cuda"
    g = torch.Generator().manual_seed(11)
    kc = torch.randn((NB, BS, HKV, D), generator=g).to(torch.bfloat16)
    vc = torch.randn((NB, BS, HKV, D), generator=g).to(torch.bfloat16)
    kh, vh = bits(kc).copy(), bits(vc).copy()          # oracle's pool
    kc, vc = kc.to(dev), vc.to(dev)                     # library's pool
    bm = BlockManager(NB, BS)
    kvgen = KV(5)
    scale = D ** -0.5
    rng = np.random.RandomState(3)
    tokens = {}

    def store(seq_rows):
        """seq_rows: list of (seq, begin, end) whose K/V go into the pool."""
        ks, vs, slots = [], [], []
        for s, b, e in seq_rows:
            k, v = kvgen.rows(tokens[s], b, e)
            ks.append(k)
            vs.append(v)
            slots.append(bm.slot_mapping(s, b, e))
        k, v = torch.cat(ks), torch.cat(vs)
        sl = np.concatenate(slots).astype(np.int32)
        pkv.kv_cache_store(k.to(dev), v.to(dev), kc, vc, torch.from_numpy(sl).to(dev))
        oracle.store(bits(k), bits(v), kh, vh, sl)

    def prefill(seqs, cached):
        tables = bm.block_tables(seqs, MAXBLK)
        new = [len(tokens[s]) - cached[s] for s in seqs]
        total = [len(tokens[s]) for s in seqs]
        store([(s, cached[s], len(tokens[s])) for s in seqs])
        q = torch.randn((sum(new), HQ, D), generator=g).to(torch.bfloat16)
        cq = np.concatenate([[0], np.cumsum(new)]).astype(np.int32)
        ck = np.concatenate([[0], np.cumsum(total)]).astype(np.int32)
        out, lse = pkv.paged_prefill_attention(
            q.to(dev), kc, vc, torch.from_numpy(tables).to(dev), torch.from_numpy(cq).to(dev),
            torch.from_numpy(ck).to(dev), max(new), max(total), scale)
        ro, rl = oracle.prefill(bits(q), kh, vh, tables, cq, ck, scale)
        assert_close(out, lse, ro, rl, "prefill")

    def decode_step(seqs):
        copies = []
        for s in seqs:
            tok = int(rng.randint(50))
            tokens[s].append(tok)
            slot, cp = bm.append_token(s, tok)
            assert slot == bm.slot_mapping(s, len(tokens[s]) - 1, len(tokens[s]))[0]
            if cp:
                copies.append(cp)
        if copies:
            src = np.array([c[0] for c in copies], np.int32)
            dst = np.array([c[1] for c in copies], np.int32)
            pkv_copy(src, dst)
            oracle.copy_blocks(kh, vh, src, dst)
        store([(s, len(tokens[s]) - 1, len(tokens[s])) for s in seqs])
        tables = bm.block_tables(seqs, MAXBLK)
        lens = np.array([len(tokens[s]) for s in seqs], np.int32)
        q = torch.randn((len(seqs), HQ, D), generator=g).to(torch.bfloat16)
        out, lse = pkv.paged_decode_attention(q.to(dev), kc, vc, torch.from_numpy(tables).to(dev),
                                              torch.from_numpy(lens).to(dev), scale)
        ro, rl = oracle.decode(bits(q), kh, vh, tables, lens, scale)
        assert_close(out, lse, ro, rl, "decode")
        return len(copies)

    def pkv_copy(src, dst):
        pkv.kv_cache_copy_blocks(kc, vc, torch.from_numpy(src).to(dev),
                                 torch.from_numpy(dst).to(dev))

    # admit: A and B share a 512-token prefix (two full blocks), C is unrelated
    stem = list(rng.randint(50, size=512))
    tokens[0] = stem + list(rng.randint(50, size=100))
    tokens[1] = stem + list(rng.randint(50, size=37))
    tokens[2] = list(rng.randint(50, size=300))
    cached = {s: bm.add_sequence(s, tokens[s]) for s in (0, 1, 2)}
    assert cached == {0: 0, 1: 512, 2: 0}
    # A prefills first; B's shared part is then already in the pool
    prefill([0], cached)
    prefill([1, 2], cached)
    for _ in range(3):
        decode_step([0, 1, 2])
    # fork A: both share its partial last block; the next appends copy it once
    bm.fork(0, 3)
    tokens[3] = list(tokens[0])
    n_copies = decode_step([0, 1, 2, 3])
    assert n_copies == 1
    for _ in range(2):
        assert decode_step([0, 1, 2, 3]) == 0
    # free A and B; a new prompt with the same stem hits the cached prefix blocks
    bm.free_sequence(0)
    bm.free_sequence(1)
    tokens[4] = stem + list(rng.randint(50, size=20))
    cached = {4: bm.add_sequence(4, tokens[4])}
    assert cached[4] == 512
    prefill([4], cached)
    decode_step([2, 3, 4])
    torch.cuda.synchronize()
    assert pkv.get_device_error() == pkv.PKV_OK


def test_copy_blocks_matches_oracle():
    dev = "cuda"
    g = torch.Generator().manual_seed(12)
    kc = torch.randn((12, BS, HKV, D), generator=g).to(torch.bfloat16)
    vc = torch.randn((12, BS, HKV, D), generator=g).to(torch.bfloat16)
    kh, vh = bits(kc).copy(), bits(vc).copy()
    kc, vc = kc.to(dev), vc.to(dev)
    src = np.array([3, 0, 7], np.int32)
    dst = np.array([5, 11, 1], np.int32)
    s, d = torch.from_numpy(src).to(dev), torch.from_numpy(dst).to(dev)
    pkv.kv_cache_copy_blocks(kc, vc, s, d)
    oracle.copy_blocks(kh, vh, src, dst)
    torch.cuda.synchronize()
    assert np.array_equal(bits(kc), kh) and np.array_equal(bits(vc), vh)
    # a bad block id is skipped and reported
    bad = torch.tensor([99], dtype=torch.int32, device=dev)
    pkv.kv_cache_copy_blocks(kc, vc, bad, d[:1])
    assert pkv.get_device_error() == pkv.PKV_ERR_DEVICE_INDEX
    assert np.array_equal(bits(kc), kh)
