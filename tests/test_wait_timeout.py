"""The bounded-wait failure path on the GPU, made to run out without faulting
or hanging anything: the test hook (pkv_testing_set_wait_fault) lowers the
kernels' wait limit to 1 ms and makes the copy producers withhold one tile, so
a consumer's wait on that tile's barrier runs out while no copy is outstanding
on it.  The call must come back, report PKV_ERR_TIMEOUT through the device
error word, and leave the library usable: the next normal call returns PKV_OK
and matches the oracle (for the tensor-core kernel this also shows that the
timed-out blocks released their tensor memory, which every block allocates in
full)."""
import time

import pytest
import torch

import oracle
from gpu_helpers import assert_close, bits
from paged_kv_cache_214_gb300 import pkv
from paged_kv_cache_214_gb300 import workloads as W

pytestmark = pytest.mark.gpu

LIMIT_NS = 1_000_000   # 1 ms


@pytest.fixture
def wait_fault():
    """Arms the hook for one test and always turns it off afterwards."""
    yield lambda tile: pkv.testing_set_wait_fault(LIMIT_NS, tile)
    pkv.testing_set_wait_fault(0, -1)


def test_hook_rejects_bad_settings():
    for args in ((-1, -1), (0, 3), (3_000_000_000, -1), (LIMIT_NS, -2)):
        with pytest.raises(pkv.PkvError) as e:
            pkv.testing_set_wait_fault(*args)
        assert e.value.status == pkv.PKV_ERR_ARG
    pkv.testing_set_wait_fault(0, -1)


@pytest.mark.parametrize("num_splits", [1, 4])
def test_decode_wait_runs_out_then_recovers(wait_fault, num_splits):
    # every block's key range has more than three 64-token tiles
    w = W.make_decode([3000, 1500, 3500], 16, 8, 48, 8100, store_new_token=False)
    dev = "cuda"
    args = (w.q.to(dev), w.k_cache.to(dev), w.v_cache.to(dev), w.block_tables.to(dev),
            w.context_lens.to(dev), w.scale)
    assert pkv.get_device_error() == pkv.PKV_OK
    wait_fault(2)
    t0 = time.perf_counter()
    pkv.paged_decode_attention(*args, num_splits=num_splits)
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 10.0
    assert pkv.get_device_error() == pkv.PKV_ERR_TIMEOUT
    pkv.testing_set_wait_fault(0, -1)
    out, lse = pkv.paged_decode_attention(*args, num_splits=num_splits)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == pkv.PKV_OK
    ref_o, ref_l = oracle.decode(bits(w.q), bits(w.k_cache), bits(w.v_cache),
                                 w.block_tables.numpy(), w.context_lens.numpy(), w.scale)
    assert_close(out, lse, ref_o, ref_l, f"decode after a timeout, S={num_splits}")


def test_small_batch_decode_wait_runs_out_then_recovers(wait_fault):
    # a batch too small to fill the GPU, one context of four blocks: 64-token
    # tile splits, the 2-stage consumer-issued form; every block's first tile
    # is withheld
    w = W.make_decode([300, 900, 40], 16, 8, 8, 8120, store_new_token=False)
    dev = "cuda"
    maxblk = w.block_tables.shape[1]
    assert pkv.paged_decode_num_splits(w.B, w.Hq, w.Hkv, w.D, maxblk, w.block_size, 0) > maxblk
    args = (w.q.to(dev), w.k_cache.to(dev), w.v_cache.to(dev), w.block_tables.to(dev),
            w.context_lens.to(dev), w.scale)
    assert pkv.get_device_error() == pkv.PKV_OK
    wait_fault(0)
    t0 = time.perf_counter()
    pkv.paged_decode_attention(*args)
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 10.0
    assert pkv.get_device_error() == pkv.PKV_ERR_TIMEOUT
    pkv.testing_set_wait_fault(0, -1)
    out, lse = pkv.paged_decode_attention(*args)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == pkv.PKV_OK
    ref_o, ref_l = oracle.decode(bits(w.q), bits(w.k_cache), bits(w.v_cache),
                                 w.block_tables.numpy(), w.context_lens.numpy(), w.scale)
    assert_close(out, lse, ref_o, ref_l, "small-batch decode after a timeout")


def test_one_split_two_group_decode_wait_runs_out_then_recovers(wait_fault):
    # a small batch of contexts of at most three blocks: one split per
    # sequence, two consumer groups taking alternate tiles; every block's first
    # tile is withheld, so both groups' waits and the producer's run out
    w = W.make_decode([300, 513, 40], 16, 8, 8, 8130, store_new_token=False)
    dev = "cuda"
    maxblk = w.block_tables.shape[1]
    assert maxblk == 3
    assert pkv.paged_decode_num_splits(w.B, w.Hq, w.Hkv, w.D, maxblk, w.block_size, 0) == 1
    args = (w.q.to(dev), w.k_cache.to(dev), w.v_cache.to(dev), w.block_tables.to(dev),
            w.context_lens.to(dev), w.scale)
    assert pkv.get_device_error() == pkv.PKV_OK
    wait_fault(0)
    t0 = time.perf_counter()
    pkv.paged_decode_attention(*args)
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 10.0
    assert pkv.get_device_error() == pkv.PKV_ERR_TIMEOUT
    pkv.testing_set_wait_fault(0, -1)
    out, lse = pkv.paged_decode_attention(*args)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == pkv.PKV_OK
    ref_o, ref_l = oracle.decode(bits(w.q), bits(w.k_cache), bits(w.v_cache),
                                 w.block_tables.numpy(), w.context_lens.numpy(), w.scale)
    assert_close(out, lse, ref_o, ref_l, "one-split decode after a timeout")


@pytest.mark.parametrize("num_splits", [0, 2])
def test_fp8_decode_wait_runs_out_then_recovers(wait_fault, num_splits):
    # E4M3 pools: the consumer-issued form (automatic splits of this batch) and
    # the producer-warp form (num_splits = 2: splits of 8 blocks or more).  After
    # the timeout the next call must return PKV_OK with the bits of a call made
    # before the fault (the E4M3 decode is checked against the oracle in
    # test_fp8.py).
    w = W.make_decode([3000, 1500, 3500, 4000], 32, 8, 64, 8150 + num_splits,
                      store_new_token=False)
    dev = "cuda"
    NB, bs = w.num_blocks, w.block_size
    k8 = torch.empty((NB, bs, w.Hkv, w.D), dtype=torch.uint8, device=dev)
    v8 = torch.empty_like(k8)
    every = torch.arange(NB * bs, dtype=torch.int32, device=dev)
    ks = vs = 6.0 / 448
    pkv.kv_cache_store_fp8(w.k_cache.to(dev).view(-1, w.Hkv, w.D),
                           w.v_cache.to(dev).view(-1, w.Hkv, w.D), k8, v8, every, ks, vs)
    args = (w.q.to(dev), k8, v8, w.block_tables.to(dev), w.context_lens.to(dev), w.scale, ks, vs)
    ref_o, ref_l = pkv.paged_decode_attention_fp8(*args, num_splits=num_splits)
    ref_o, ref_l = ref_o.clone(), ref_l.clone()
    torch.cuda.synchronize()
    assert pkv.get_device_error() == pkv.PKV_OK
    wait_fault(2)
    t0 = time.perf_counter()
    pkv.paged_decode_attention_fp8(*args, num_splits=num_splits)
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 10.0
    assert pkv.get_device_error() == pkv.PKV_ERR_TIMEOUT
    pkv.testing_set_wait_fault(0, -1)
    out, lse = pkv.paged_decode_attention_fp8(*args, num_splits=num_splits)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == pkv.PKV_OK
    assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)


@pytest.mark.parametrize("Hq,Hkv", [(16, 8), (8, 8)])
def test_prefill_wait_runs_out_then_recovers(wait_fault, Hq, Hkv):
    w = W.make_prefill([512, 300, 0], [256, 300, 640], Hq, Hkv, 32, 8200 + Hq)
    dev = "cuda"
    kc, vc = w.k_cache.to(dev), w.v_cache.to(dev)
    kh, vh = bits(w.k_cache).copy(), bits(w.v_cache).copy()
    pkv.kv_cache_store(w.k_new.to(dev), w.v_new.to(dev), kc, vc, w.slot_mapping.to(dev))
    args = (w.q.to(dev), kc, vc, w.block_tables.to(dev), w.cu_seqlens_q.to(dev),
            w.cu_seqlens_k.to(dev), w.max_seqlen_q, w.max_seqlen_k, w.scale)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == pkv.PKV_OK
    wait_fault(3)
    t0 = time.perf_counter()
    pkv.paged_prefill_attention(*args)
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 10.0
    assert pkv.get_device_error() == pkv.PKV_ERR_TIMEOUT
    pkv.testing_set_wait_fault(0, -1)
    out, lse = pkv.paged_prefill_attention(*args)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == pkv.PKV_OK
    oracle.store(bits(w.k_new), bits(w.v_new), kh, vh, w.slot_mapping.numpy())
    ref_o, ref_l = oracle.prefill(bits(w.q), kh, vh, w.block_tables.numpy(),
                                  w.cu_seqlens_q.numpy(), w.cu_seqlens_k.numpy(), w.scale)
    assert_close(out, lse, ref_o, ref_l, f"prefill after a timeout, Hq={Hq}")
