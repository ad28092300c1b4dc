"""paged_decode_attention_store (the step's store and the decode in one launch)
on the GPU against the oracle's store followed by its decode (max|dout| <=
1e-2, max|dlse| <= 1e-3), and bit for bit against the two separate calls."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_close, bits, compact_pool
from paged_kv_cache_214_gb300 import pkv
from paged_kv_cache_214_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def compact_slots(w, seqs):
    used = w.block_tables[seqs][w.block_tables[seqs] >= 0].unique()
    remap = {int(b): i for i, b in enumerate(used)}
    bs = w.block_size
    return np.array([remap[int(s) // bs] * bs + int(s) % bs if s >= 0 else -1
                     for s in w.slot_mapping[seqs]], np.int32)


def run_and_check(w, num_splits=0, sample=None, what=""):
    dev = "cuda"
    kc, vc = w.k_cache.to(dev), w.v_cache.to(dev)
    seqs = list(range(w.B)) if sample is None else list(sample)
    kh, vh, th = compact_pool(kc, vc, w.block_tables[seqs])   # before any library kernel
    out, lse = pkv.paged_decode_attention_store(
        w.q.to(dev), w.k_new.to(dev), w.v_new.to(dev), w.slot_mapping.to(dev), kc, vc,
        w.block_tables.to(dev), w.context_lens.to(dev), w.scale, num_splits=num_splits)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == pkv.PKV_OK
    oracle.store(bits(w.k_new[seqs]), bits(w.v_new[seqs]), kh, vh, compact_slots(w, seqs))
    ref_o, ref_l = oracle.decode(bits(w.q[seqs]), kh, vh, th, w.context_lens[seqs].numpy(),
                                 w.scale)
    # the pools hold the new tokens afterwards, as after kv_cache_store
    kh2, vh2, _ = compact_pool(kc, vc, w.block_tables[seqs])
    assert np.array_equal(kh2, kh) and np.array_equal(vh2, vh), f"{what}: pool contents"
    return assert_close(out[seqs], lse[seqs], ref_o, ref_l, what)


def test_tiny_decode_workload():
    run_and_check(W.config_workload(1), what="tiny-decode")


@pytest.mark.parametrize("num_splits", [1, 2, 3, 7, 0])
def test_forced_splits(num_splits):
    # new tokens at block starts and ends, in the last and in a middle split
    lens = [1, 17, 255, 256, 257, 600, 1000, 4095, 4096, 4097]
    w = W.make_decode(lens, 16, 8, 96, 1600 + num_splits)
    run_and_check(w, num_splits=num_splits, what=f"S={num_splits}")


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (16, 8), (32, 8), (64, 8), (14, 2), (16, 1)])
def test_head_groupings(Hq, Hkv):
    # several query-head groups per kv head write the same new row
    w = W.make_decode([5, 64, 130, 700, 2000], Hq, Hkv, 24, 1700 + Hq * 10 + Hkv)
    run_and_check(w, what=f"Hq={Hq},Hkv={Hkv}")


def test_empty_contexts_store_nothing():
    w = W.make_decode([0, 300, 0, 1], 16, 8, 8, 1800)
    assert int(w.slot_mapping[0]) == -1 and int(w.slot_mapping[2]) == -1
    run_and_check(w, what="empty contexts")


def test_decode_b64_workload():
    run_and_check(W.config_workload(2, pool_device="cuda"), sample=[0, 17, 40, 63],
                  what="decode-b64")


def test_same_bits_as_store_then_decode():
    dev = "cuda"
    w = W.make_decode([3, 256, 257, 1000, 3000, 6000], 32, 8, 64, 1900)
    args = (w.block_tables.to(dev), w.context_lens.to(dev), w.scale)
    kc1, vc1 = w.k_cache.to(dev), w.v_cache.to(dev)
    kc2, vc2 = kc1.clone(), vc1.clone()
    q, kn, vn, slots = w.q.to(dev), w.k_new.to(dev), w.v_new.to(dev), w.slot_mapping.to(dev)
    pkv.kv_cache_store(kn, vn, kc1, vc1, slots)
    o1, l1 = pkv.paged_decode_attention(q, kc1, vc1, *args)
    o2, l2 = pkv.paged_decode_attention_store(q, kn, vn, slots, kc2, vc2, *args)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(kc1, kc2) and torch.equal(vc1, vc2)


def test_slot_other_than_last_position_is_reported_and_not_written():
    dev = "cuda"
    w = W.make_decode([300, 700], 16, 8, 8, 2000)
    kc, vc = w.k_cache.to(dev), w.v_cache.to(dev)
    before = kc.clone()
    slots = w.slot_mapping.clone()
    slots[1] = int(w.block_tables[1, 0]) * 256 + 5     # position 5, not 699
    pkv.paged_decode_attention_store(w.q.to(dev), w.k_new.to(dev), w.v_new.to(dev),
                                     slots.to(dev), kc, vc, w.block_tables.to(dev),
                                     w.context_lens.to(dev), w.scale)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == pkv.PKV_ERR_DEVICE_INDEX
    assert pkv.get_device_error() == pkv.PKV_OK
    flat_after = kc.view(-1, w.Hkv, w.D)
    flat_before = before.view(-1, w.Hkv, w.D)
    assert torch.equal(flat_after[int(slots[1])], flat_before[int(slots[1])])
    # sequence 0's token was stored
    assert torch.equal(flat_after[int(slots[0])], w.k_new[0].to(dev))
