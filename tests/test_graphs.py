"""The CUDA-graph decode runner (pkv_decode_graphs_*) against the oracle.

Decode steps are captured once per batch bucket and replayed with the step's
batch padded up to the bucket ("Nano-vLLM System Architecture Analysis", §2
Core Components, "CUDA Graphs"; comparison table, "Variable-batch CUDA
Graphs"), and batches above the largest bucket run eagerly.  Each step here
gets fresh seeded inputs copied into the runner's fixed pool and static rows;
the oracle stores the step's new tokens into a host copy of the same pool and
decodes.  Checked per step: the whole pool bit for bit (so a padding row that
kept a stale slot from a larger earlier batch and stored into it would show),
rows [0, B) of out / lse within the decode tolerance, and padding rows
[B, bucket) as empty rows (out 0, lse -inf).  Batches shrink and grow between
steps so that padding rows hold the previous batch's live inputs."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_close, bits
from paged_kv_cache_214_gb300 import graphs, pkv
from paged_kv_cache_214_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def lens_for(B, max_len, seed):
    g = np.random.default_rng(seed)
    return [int(x) for x in g.integers(1, max_len + 1, size=B)]


def check_padding(runner, B):
    b = runner.bucket_for(B)
    if b > B:
        assert (runner.out[B:b] == 0).all(), "padding rows' out must be 0"
        if runner.lse is not None:
            assert torch.isneginf(runner.lse[B:b]).all(), "padding rows' lse must be -inf"


def run_bf16_steps(Hq, Hkv, W_blocks, NB, max_batch, batches, buckets, seed0):
    dev = "cuda"
    kc = torch.zeros((NB, 256, Hkv, 128), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    runner = graphs.DecodeGraphs(kc, vc, Hq, W_blocks, max_batch, 128 ** -0.5,
                                 buckets=buckets)
    try:
        for i, B in enumerate(batches):
            lens = lens_for(B, W_blocks * 256, seed0 + i)
            w = W.make_decode(lens, Hq, Hkv, NB, seed0 + 100 + i, max_blocks_per_seq=W_blocks)
            kh, vh = bits(w.k_cache).copy(), bits(w.v_cache).copy()
            kc.copy_(w.k_cache)
            vc.copy_(w.v_cache)
            out, lse = runner.step(w.q.to(dev), w.k_new.to(dev), w.v_new.to(dev),
                                   w.slot_mapping.to(dev), w.block_tables.to(dev),
                                   w.context_lens.to(dev))
            torch.cuda.synchronize()
            assert pkv.get_device_error() == pkv.PKV_OK
            oracle.store(bits(w.k_new), bits(w.v_new), kh, vh, w.slot_mapping.numpy())
            assert np.array_equal(bits(kc), kh) and np.array_equal(bits(vc), vh), \
                f"B={B}: the pool differs from the oracle's store"
            ref_o, ref_l = oracle.decode(bits(w.q), kh, vh, w.block_tables.numpy(),
                                         w.context_lens.numpy(), w.scale)
            assert_close(out, lse, ref_o, ref_l, f"graph step B={B}")
            check_padding(runner, B)
    finally:
        runner.close()


def test_buckets_shrink_and_grow_against_oracle():
    """Default buckets clipped to 80 rows (1, 2, 4, ..., 64), eager above 64;
    contexts up to four blocks (small batches take the tile-split plan)."""
    run_bf16_steps(Hq=8, Hkv=2, W_blocks=4, NB=340, max_batch=80,
                   batches=[13, 1, 64, 40, 3, 80, 7, 64], buckets=None, seed0=9100)


def test_largest_bucket_and_eager_above_it():
    """The 512 bucket, a batch that pads up to it, and batches above it (eager)."""
    run_bf16_steps(Hq=8, Hkv=2, W_blocks=1, NB=530, max_batch=520,
                   batches=[512, 300, 520, 513, 2], buckets=None, seed0=9200)


def test_runner_buckets_and_choice():
    dev = "cuda"
    kc = torch.zeros((8, 256, 2, 128), dtype=torch.bfloat16, device=dev)
    r = graphs.DecodeGraphs(kc, kc.clone(), 8, 2, 100, 0.1)
    try:
        assert r.buckets == [1, 2, 4, 8, 16, 32, 64]
        assert [r.bucket_for(B) for B in (1, 3, 9, 64, 65, 100)] == [1, 4, 16, 64, 0, 0]
        with pytest.raises(pkv.PkvError):
            r.run(101)
        r.run(0)   # queues nothing
    finally:
        r.close()
    r = graphs.DecodeGraphs(kc, kc.clone(), 8, 2, 100, 0.1, buckets=[3, 50])
    try:
        assert r.buckets == [3, 50]
    finally:
        r.close()
    with pytest.raises(pkv.PkvError):
        graphs.DecodeGraphs(kc, kc.clone(), 8, 2, 100, 0.1, buckets=[4, 4])
    with pytest.raises(pkv.PkvError):
        graphs.DecodeGraphs(kc, kc.clone(), 8, 2, 100, 0.1, buckets=[4, 101])


def test_graph_replay_equals_fused_call_over_padded_rows():
    """Rows [0, B) of a replay are bit-identical to paged_decode_attention_store
    over the bucket's rows with the padding rows empty."""
    dev = "cuda"
    Hq, Hkv, Wb, NB = 16, 8, 6, 200
    kc = torch.zeros((NB, 256, Hkv, 128), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    r = graphs.DecodeGraphs(kc, vc, Hq, Wb, 32, 128 ** -0.5)
    try:
        B = 11
        w = W.make_decode(lens_for(B, Wb * 256, 9300), Hq, Hkv, NB, 9301, max_blocks_per_seq=Wb)
        kc.copy_(w.k_cache)
        vc.copy_(w.v_cache)
        out, lse = r.step(w.q.to(dev), w.k_new.to(dev), w.v_new.to(dev), w.slot_mapping.to(dev),
                          w.block_tables.to(dev), w.context_lens.to(dev))
        torch.cuda.synchronize()
        b = r.bucket_for(B)
        assert b == 16
        pad = lambda t, fill: torch.cat([t, torch.full((b - B,) + tuple(t.shape[1:]), fill,
                                                       dtype=t.dtype)])
        k2, v2 = w.k_cache.to(dev), w.v_cache.to(dev)
        o2, l2 = pkv.paged_decode_attention_store(
            pad(w.q, 0).to(dev), pad(w.k_new, 0).to(dev), pad(w.v_new, 0).to(dev),
            pad(w.slot_mapping, -1).to(dev), k2, v2, pad(w.block_tables, 0).to(dev),
            pad(w.context_lens, 0).to(dev), w.scale)
        torch.cuda.synchronize()
        assert torch.equal(kc, k2) and torch.equal(vc, v2)
        assert torch.equal(out, o2[:B]) and torch.equal(lse, l2[:B])
        assert pkv.get_device_error() == pkv.PKV_OK
    finally:
        r.close()


def test_fp8_runner_against_oracle():
    """E4M3 pools (the fused FP8 store + decode), custom buckets, eager above."""
    dev = "cuda"
    Hq, Hkv, Wb, NB, ks, vs = 8, 2, 4, 110, 6.0 / 448, 5.0 / 448
    k8 = torch.zeros((NB, 256, Hkv, 128), dtype=torch.uint8, device=dev)
    v8 = torch.zeros_like(k8)
    r = graphs.DecodeGraphs(k8, v8, Hq, Wb, 24, 128 ** -0.5, buckets=[2, 8, 16], k_scale=ks,
                            v_scale=vs)
    try:
        for i, B in enumerate([5, 16, 24, 1]):
            w = W.make_decode(lens_for(B, Wb * 256, 9400 + i), Hq, Hkv, NB, 9500 + i,
                              max_blocks_per_seq=Wb)
            k8h = np.zeros((NB, 256, Hkv, 128), np.uint8)
            v8h = np.zeros_like(k8h)
            all_slots = np.arange(NB * 256, dtype=np.int32)
            oracle.store_fp8(bits(w.k_cache).reshape(-1, Hkv, 128),
                             bits(w.v_cache).reshape(-1, Hkv, 128), k8h, v8h, all_slots, ks, vs)
            k8.copy_(torch.from_numpy(k8h))
            v8.copy_(torch.from_numpy(v8h))
            out, lse = r.step(w.q.to(dev), w.k_new.to(dev), w.v_new.to(dev),
                              w.slot_mapping.to(dev), w.block_tables.to(dev),
                              w.context_lens.to(dev))
            torch.cuda.synchronize()
            assert pkv.get_device_error() == pkv.PKV_OK
            oracle.store_fp8(bits(w.k_new), bits(w.v_new), k8h, v8h, w.slot_mapping.numpy(),
                             ks, vs)
            assert np.array_equal(k8.cpu().numpy(), k8h) and np.array_equal(v8.cpu().numpy(), v8h)
            ref_o, ref_l = oracle.decode_fp8(bits(w.q), k8h, v8h, w.block_tables.numpy(),
                                             w.context_lens.numpy(), w.scale, ks, vs)
            assert_close(out, lse, ref_o, ref_l, f"fp8 graph step B={B}")
            check_padding(r, B)
    finally:
        r.close()
