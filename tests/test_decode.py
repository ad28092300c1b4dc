"""paged_decode_attention on the GPU against the oracle (max|dout| <= 1e-2,
max|dlse| <= 1e-3), including the store of the step's new token."""
import time

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_close, bits, compact_pool
from paged_kv_cache_214_gb300 import pkv
from paged_kv_cache_214_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def run_and_check(w, num_splits=0, sample=None, what=""):
    """Store the new tokens then decode on the GPU; the oracle repeats the store
    and decode on host copies of the original inputs.  `sample`: indices of the
    sequences the oracle checks (all by default)."""
    dev = "cuda"
    kc, vc = w.k_cache.to(dev), w.v_cache.to(dev)
    seqs = list(range(w.B)) if sample is None else list(sample)
    tables = w.block_tables[seqs]
    kh, vh, th = compact_pool(kc, vc, tables)      # before any library kernel runs
    slot_host = w.slot_mapping[seqs].clone()
    # slots of the sampled sequences, renumbered to the compact copy
    used = tables[tables >= 0].unique()
    remap = {int(b): i for i, b in enumerate(used)}
    bs = w.block_size
    slot_host = torch.tensor([remap[int(s) // bs] * bs + int(s) % bs if s >= 0 else -1
                              for s in slot_host], dtype=torch.int32)
    pkv.kv_cache_store(w.k_new.to(dev), w.v_new.to(dev), kc, vc, w.slot_mapping.to(dev))
    out, lse = pkv.paged_decode_attention(w.q.to(dev), kc, vc, w.block_tables.to(dev),
                                          w.context_lens.to(dev), w.scale,
                                          num_splits=num_splits)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == pkv.PKV_OK
    oracle.store(bits(w.k_new[seqs]), bits(w.v_new[seqs]), kh, vh, slot_host.numpy())
    ref_o, ref_l = oracle.decode(bits(w.q[seqs]), kh, vh, th, w.context_lens[seqs].numpy(),
                                 w.scale)
    return assert_close(out[seqs], lse[seqs], ref_o, ref_l, what)


def test_tiny_decode_workload():
    run_and_check(W.config_workload(1), what="tiny-decode")


@pytest.mark.parametrize("num_splits", [1, 2, 3, 7, 0, 64])
def test_forced_splits(num_splits):
    lens = [1, 17, 255, 256, 257, 600, 1000, 4095, 4096, 4097]
    w = W.make_decode(lens, 16, 8, 96, 1000 + num_splits)
    run_and_check(w, num_splits=num_splits, what=f"S={num_splits}")


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (16, 8), (32, 8), (24, 8), (64, 8), (4, 1), (14, 2), (16, 1)])
def test_head_groupings(Hq, Hkv):
    lens = [5, 64, 130, 700, 2000]
    w = W.make_decode(lens, Hq, Hkv, 24, 2000 + Hq * 10 + Hkv)
    run_and_check(w, what=f"Hq={Hq},Hkv={Hkv}")


def test_ragged_tile_tails():
    # every residue of the 64-token tile and of the 256-token block
    lens = [1, 2, 63, 64, 65, 127, 128, 129, 191, 192, 193, 255, 256, 257, 511, 512, 513]
    w = W.make_decode(lens, 32, 8, 64, 3000)
    run_and_check(w, num_splits=0, what="tails")
    run_and_check(w, num_splits=2, what="tails S=2")


@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (16, 4), (32, 4)])
def test_small_batch_tile_splits(Hq, Hkv):
    """Batches too small to fill the GPU with one-block splits split into
    64-token tiles (ranges that start inside a block) once a context spans four
    blocks or more; every tile and block residue of the context length."""
    lens = [1, 63, 64, 65, 200, 256, 257, 700, 1000]
    w = W.make_decode(lens, Hq, Hkv, 32, 3050 + Hq)
    maxblk = w.block_tables.shape[1]
    assert maxblk == 4
    assert pkv.paged_decode_num_splits(w.B, Hq, Hkv, 128, maxblk) == 4 * maxblk
    run_and_check(w, what=f"tile splits Hq={Hq},Hkv={Hkv}")


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 4), (8, 2), (16, 4), (32, 4)])
def test_small_batch_short_contexts_one_split(Hq, Hkv):
    """A small batch whose contexts span at most three blocks runs one split per
    sequence (no partials, no merge, no workspace), on the form with two
    consumer groups taking alternate tiles (1, 2, 4 and 8 query heads per
    block)."""
    lens = [1, 63, 64, 65, 200, 256, 257, 700]
    w = W.make_decode(lens, Hq, Hkv, 24, 3070 + Hq)
    maxblk = w.block_tables.shape[1]
    assert maxblk == 3
    assert pkv.paged_decode_num_splits(w.B, Hq, Hkv, 128, maxblk) == 1
    run_and_check(w, what=f"one split Hq={Hq},Hkv={Hkv}")


@pytest.mark.parametrize("lens,Hq,Hkv", [([17, 256, 300, 513], 16, 8),
                                          ([3000, 900, 5000, 257, 64, 1], 32, 8)])
def test_metadata_ready_flag(lens, Hq, Hkv):
    """PKV_DECODE_METADATA_READY (tables and lengths read before the wait for
    the previous kernel): the one-split two-group form and a split batch match
    the oracle and equal the plain call bit for bit, also as two calls in a
    replayed CUDA graph whose inputs change between replays."""
    dev = "cuda"
    w = W.make_decode(lens, Hq, Hkv, 64, 3600 + Hq, store_new_token=False)
    q, kc, vc = w.q.to(dev), w.k_cache.to(dev), w.v_cache.to(dev)
    tables, ctx = w.block_tables.to(dev), w.context_lens.to(dev)
    o1, l1 = pkv.paged_decode_attention(q, kc, vc, tables, ctx, w.scale)
    torch.cuda.synchronize()
    o2, l2 = pkv.paged_decode_attention(q, kc, vc, tables, ctx, w.scale, metadata_ready=True)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == pkv.PKV_OK
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    ref_o, ref_l = oracle.decode(bits(w.q), bits(w.k_cache), bits(w.v_cache),
                                 w.block_tables.numpy(), w.context_lens.numpy(), w.scale)
    assert_close(o2, l2, ref_o, ref_l, "metadata ready")

    # two flagged calls in one graph; tables and lengths rewritten between
    # replays by host copies, finished before the replay starts
    w2 = W.make_decode([max(1, L // 2) for L in lens], Hq, Hkv, 64, 3700 + Hq,
                       store_new_token=False, max_blocks_per_seq=w.block_tables.shape[1])
    out = torch.empty_like(q)
    lse = torch.empty((w.B, Hq), dtype=torch.float32, device=dev)
    need = pkv.paged_decode_workspace_bytes(w.B, Hq, Hkv, 128, tables.shape[1])
    ws = torch.zeros(max(need, 256), dtype=torch.uint8, device=dev)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    torch.cuda.synchronize()
    call = lambda: pkv.paged_decode_attention(q, kc, vc, tables, ctx, w.scale, out=out,  # noqa: E731
                                              lse=lse, workspace=ws, stream=s,
                                              metadata_ready=True)
    with torch.cuda.stream(s):
        call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
        call()
    for ww in (w2, w):
        tables.copy_(ww.block_tables)
        ctx.copy_(ww.context_lens)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert pkv.get_device_error() == pkv.PKV_OK
        ref_o, ref_l = oracle.decode(bits(w.q), bits(w.k_cache), bits(w.v_cache),
                                     ww.block_tables.numpy(), ww.context_lens.numpy(), w.scale)
        assert_close(out, lse, ref_o, ref_l, "metadata ready in a graph")


def test_empty_context_gives_zero_and_neg_inf():
    w = W.make_decode([0, 300, 0], 16, 8, 8, 3100, store_new_token=False)
    dev = "cuda"
    out, lse = pkv.paged_decode_attention(w.q.to(dev), w.k_cache.to(dev), w.v_cache.to(dev),
                                          w.block_tables.to(dev), w.context_lens.to(dev),
                                          w.scale, num_splits=2)
    torch.cuda.synchronize()
    assert (out[0] == 0).all() and (out[2] == 0).all()
    assert torch.isneginf(lse[0]).all() and torch.isneginf(lse[2]).all()
    assert torch.isfinite(lse[1]).all()


def test_repeated_calls_share_workspace():
    """The arrival counters are reset by every call: the same inputs give the
    same bits call after call."""
    w = W.make_decode([3000, 5000, 100], 32, 8, 64, 3200, store_new_token=False)
    dev = "cuda"
    args = (w.q.to(dev), w.k_cache.to(dev), w.v_cache.to(dev), w.block_tables.to(dev),
            w.context_lens.to(dev), w.scale)
    o1, l1 = pkv.paged_decode_attention(*args, num_splits=5)
    o1, l1 = o1.clone(), l1.clone()
    for _ in range(3):
        o2, l2 = pkv.paged_decode_attention(*args, num_splits=5)
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_one_workspace_serves_every_shape():
    """Calls of different shapes share one workspace: each call's partials never
    overwrite the counters of another shape."""
    dev = "cuda"
    ws = torch.zeros(64 << 20, dtype=torch.uint8, device=dev)
    cases = [W.make_decode([3000, 900, 5000], 32, 8, 64, 3500, store_new_token=False),
             W.make_decode([700, 4000], 24, 8, 64, 3501, store_new_token=False),
             W.make_decode([2500, 2600, 100, 4100], 16, 8, 64, 3502, store_new_token=False)]
    for rep in range(2):
        for w in cases:
            out, lse = pkv.paged_decode_attention(
                w.q.to(dev), w.k_cache.to(dev), w.v_cache.to(dev), w.block_tables.to(dev),
                w.context_lens.to(dev), w.scale, workspace=ws, num_splits=3 + rep)
            torch.cuda.synchronize()
            ref_o, ref_l = oracle.decode(bits(w.q), bits(w.k_cache), bits(w.v_cache),
                                         w.block_tables.numpy(), w.context_lens.numpy(), w.scale)
            assert_close(out, lse, ref_o, ref_l, f"shared workspace rep {rep}")


def test_decode_b64_full():
    run_and_check(W.config_workload(2, pool_device="cuda"), what="decode-b64")


def test_prefix_shared_b256_full():
    """Every sequence and head of the prefix-shared workload (256 sequences)."""
    w = W.config_workload(3, pool_device="cuda")
    t0 = time.perf_counter()
    run_and_check(w, what="prefix-shared-b256")
    print(f"prefix-shared-b256: GPU + oracle check of all {w.B} sequences "
          f"{time.perf_counter() - t0:.1f} s")


def test_long_decode_b8_full():
    """Every sequence and head of the long-context workload (split-K path)."""
    w = W.config_workload(5, pool_device="cuda")
    t0 = time.perf_counter()
    run_and_check(w, what="long-decode-b8")
    print(f"long-decode-b8: GPU + oracle check of all {w.B} sequences "
          f"{time.perf_counter() - t0:.1f} s")


def test_bad_block_id_and_long_context_are_reported():
    w = W.make_decode([300, 40], 16, 8, 8, 3300, store_new_token=False)
    dev = "cuda"
    bt = w.block_tables.clone()
    bt[0, 1] = 1 << 20                   # outside the pool
    lens = w.context_lens.clone()
    args = (w.q.to(dev), w.k_cache.to(dev), w.v_cache.to(dev))
    assert pkv.get_device_error() == pkv.PKV_OK
    pkv.paged_decode_attention(*args, bt.to(dev), lens.to(dev), w.scale)
    assert pkv.get_device_error() == pkv.PKV_ERR_DEVICE_INDEX
    lens[1] = 10_000                     # longer than its table can address
    pkv.paged_decode_attention(*args, w.block_tables.to(dev), lens.to(dev), w.scale)
    assert pkv.get_device_error() == pkv.PKV_ERR_DEVICE_INDEX
    assert pkv.get_device_error() == pkv.PKV_OK


def test_workspace_too_small_is_rejected():
    w = W.make_decode([3000, 5000], 32, 8, 64, 3400, store_new_token=False)
    dev = "cuda"
    small = torch.zeros(256, dtype=torch.uint8, device=dev)
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_decode_attention(w.q.to(dev), w.k_cache.to(dev), w.v_cache.to(dev),
                                   w.block_tables.to(dev), w.context_lens.to(dev), w.scale,
                                   workspace=small, num_splits=4)
    assert e.value.status == pkv.PKV_ERR_WORKSPACE
