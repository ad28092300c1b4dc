"""paged_decode_attention_shared_prefix on the GPU against the oracle (which
simply reads every sequence's blocks, shared or not), and against the plain
decode entry point."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import ATOL_LSE, ATOL_OUT, assert_close, bits, compact_pool
from paged_kv_cache_214_gb300 import pkv
from paged_kv_cache_214_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def run_and_check(w, P, num_splits=0, sample=None, store=True, what=""):
    dev = "cuda"
    kc, vc = w.k_cache.to(dev), w.v_cache.to(dev)
    seqs = list(range(w.B)) if sample is None else list(sample)
    tables = w.block_tables[seqs]
    kh, vh, th = compact_pool(kc, vc, tables)
    used = tables[tables >= 0].unique()
    remap = {int(b): i for i, b in enumerate(used)}
    bs = w.block_size
    if store:
        slot_host = np.array([remap[int(s) // bs] * bs + int(s) % bs if s >= 0 else -1
                              for s in w.slot_mapping[seqs]], np.int32)
        pkv.kv_cache_store(w.k_new.to(dev), w.v_new.to(dev), kc, vc, w.slot_mapping.to(dev))
        oracle.store(bits(w.k_new[seqs]), bits(w.v_new[seqs]), kh, vh, slot_host)
    out, lse = pkv.paged_decode_attention_shared_prefix(
        w.q.to(dev), kc, vc, w.block_tables.to(dev), w.context_lens.to(dev), w.scale, P,
        num_splits=num_splits)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == pkv.PKV_OK
    ref_o, ref_l = oracle.decode(bits(w.q[seqs]), kh, vh, th, w.context_lens[seqs].numpy(),
                                 w.scale)
    return assert_close(out[seqs], lse[seqs], ref_o, ref_l, what)


@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (16, 8), (24, 8), (8, 8)])
@pytest.mark.parametrize("P", [256, 1024])
def test_shared_prefix_small(Hq, Hkv, P):
    suffix = [1, 2, 255, 256, 300, 1000, 64, 129]
    w = W.make_decode([P + s for s in suffix], Hq, Hkv, 64, 8000 + P + Hq,
                      shared_prefix_tokens=P, pool_device="cuda")
    run_and_check(w, P, what=f"P={P} Hq={Hq}")
    run_and_check(w, P, num_splits=3, store=False, what=f"P={P} Hq={Hq} S=3")


def test_context_equal_to_prefix():
    w = W.make_decode([512, 512, 700], 32, 8, 16, 8100, shared_prefix_tokens=512,
                      store_new_token=False, pool_device="cuda")
    run_and_check(w, 512, store=False, what="ctx == P")


def test_many_sequences_more_than_one_row_tile():
    # B*g = 300*4 rows per kv head: several 128-row tiles, the last one ragged
    suffix = list(np.random.RandomState(0).randint(1, 700, size=300))
    w = W.make_decode([512 + int(s) for s in suffix], 32, 8, 2 + 300 * 3, 8200,
                      shared_prefix_tokens=512, pool_device="cuda")
    run_and_check(w, 512, sample=sorted(set(range(0, 300, 23)) | {299}), what="B=300")


def test_prefix_shared_b256_workload_sampled():
    w = W.config_workload(3, pool_device="cuda")
    g = torch.Generator().manual_seed(78)
    sample = sorted(torch.randperm(w.B, generator=g)[:12].tolist())
    run_and_check(w, 2048, sample=sample, what="prefix-shared-b256")


def test_matches_plain_decode():
    w = W.make_decode([2048 + s for s in (5, 900, 3000)], 32, 8, 48, 8300,
                      shared_prefix_tokens=2048, store_new_token=False, pool_device="cuda")
    dev = "cuda"
    args = (w.q.to(dev), w.k_cache, w.v_cache, w.block_tables.to(dev), w.context_lens.to(dev),
            w.scale)
    o1, l1 = pkv.paged_decode_attention(*args)
    o1, l1 = o1.clone(), l1.clone()
    o2, l2 = pkv.paged_decode_attention_shared_prefix(*args, 2048)
    torch.cuda.synchronize()
    assert (o1.float() - o2.float()).abs().max().item() <= ATOL_OUT
    assert (l1 - l2).abs().max().item() <= ATOL_LSE


def test_unshared_prefix_is_reported():
    w = W.make_decode([600, 700], 16, 8, 16, 8400, shared_prefix_tokens=512,
                      store_new_token=False, pool_device="cuda")
    bt = w.block_tables.clone()
    bt[1, 1] = int(bt[1, 2])        # sequence 1's second prefix block differs
    dev = "cuda"
    assert pkv.get_device_error() == pkv.PKV_OK
    pkv.paged_decode_attention_shared_prefix(w.q.to(dev), w.k_cache, w.v_cache, bt.to(dev),
                                             w.context_lens.to(dev), w.scale, 512)
    assert pkv.get_device_error() == pkv.PKV_ERR_DEVICE_INDEX


def test_bad_prefix_length_rejected_on_host():
    w = W.make_decode([600], 16, 8, 8, 8500, store_new_token=False, pool_device="cuda")
    dev = "cuda"
    for P in (100, 256 * 10):
        with pytest.raises(pkv.PkvError) as e:
            pkv.paged_decode_attention_shared_prefix(
                w.q.to(dev), w.k_cache, w.v_cache, w.block_tables.to(dev),
                w.context_lens.to(dev), w.scale, P)
        assert e.value.status == pkv.PKV_ERR_ARG
