"""paged_decode_attention_multiquery (q_len new positions per sequence, the
verify step of speculative decoding) on the GPU against the oracle's prefill
with Lq = q_len (max|dout| <= 1e-2, max|dlse| <= 1e-3), after the store of the
new tokens."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_close, bits, compact_pool
from paged_kv_cache_214_gb300 import pkv
from paged_kv_cache_214_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def verify_batch(cached, q_len, Hq, Hkv, num_blocks, seed):
    """Sequences with `cached` tokens each plus q_len new ones to check."""
    return W.make_prefill(cached, [q_len] * len(cached), Hq, Hkv, num_blocks, seed,
                          name="verify")


def run_and_check(w, q_len, num_splits=0, what=""):
    """GPU: store the new tokens, then the multi-query decode.  Oracle: the same
    store and a prefill with Lq = q_len on host copies of the original inputs."""
    dev = "cuda"
    kc, vc = w.k_cache.to(dev), w.v_cache.to(dev)
    kh, vh, th = compact_pool(kc, vc, w.block_tables)
    used = w.block_tables[w.block_tables >= 0].unique()
    remap = {int(b): i for i, b in enumerate(used)}
    bs = w.block_size
    slot_host = np.array([remap[int(s) // bs] * bs + int(s) % bs for s in w.slot_mapping],
                         np.int32)
    pkv.kv_cache_store(w.k_new.to(dev), w.v_new.to(dev), kc, vc, w.slot_mapping.to(dev))
    q = w.q.to(dev).view(w.B, q_len, w.Hq, w.D)
    ctx = torch.tensor(w.k_lens, dtype=torch.int32, device=dev)
    out, lse = pkv.paged_decode_attention_multiquery(q, kc, vc, w.block_tables.to(dev), ctx,
                                                     w.scale, num_splits=num_splits)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == pkv.PKV_OK
    oracle.store(bits(w.k_new), bits(w.v_new), kh, vh, slot_host)
    ref_o, ref_l = oracle.prefill(bits(w.q), kh, vh, th, w.cu_seqlens_q.numpy(),
                                  w.cu_seqlens_k.numpy(), w.scale)
    return assert_close(out.view(-1, w.Hq, w.D), lse.view(-1, w.Hq), ref_o, ref_l, what)


def tensor_core_path(w, q_len):
    """True when the call runs on the tensor-core verify kernel (which needs
    no workspace) rather than the split-K decode kernel."""
    return pkv.paged_decode_multiquery_workspace_bytes(
        w.B, q_len, w.Hq, w.Hkv, w.D, w.block_tables.shape[1]) == 0


def expect_tensor_core(w, q_len):
    """The routing rule: the tensor-core kernel takes batches of at least one
    (sequence, kv head) item per SM with more than 8 (position, head) rows per
    kv head; up to 8 rows fit one split-K decode block, which reads K/V once."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return w.B * w.Hkv >= sms and (w.Hq // w.Hkv) * q_len > 8


# 24 ragged sequences (across block and tile boundaries, some holding nothing
# but the new tokens): 24 x 8 kv heads = 192 items, the tensor-core path
CACHED_24 = [0, 1, 63, 64, 127, 128, 255, 256, 300, 511, 512, 700,
             999, 1024, 1100, 1500, 1777, 2000, 2047, 2048, 2300, 2600, 3000, 3500]


@pytest.mark.parametrize("q_len", [2, 4, 8])
@pytest.mark.parametrize("Hq,Hkv", [(16, 8), (32, 8), (8, 8), (24, 8)])
def test_verify_large_batch(q_len, Hq, Hkv):
    # 192 items: the tensor-core kernel for more than 8 rows per kv head,
    # the split-K decode kernel (all rows in one block) otherwise
    w = verify_batch(CACHED_24, q_len, Hq, Hkv, 512, 7000 + 10 * q_len + Hq)
    assert tensor_core_path(w, q_len) == expect_tensor_core(w, q_len)
    run_and_check(w, q_len, what=f"q_len={q_len} Hq={Hq} Hkv={Hkv}")


@pytest.mark.parametrize("q_len", [2, 4, 8])
@pytest.mark.parametrize("Hq,Hkv", [(16, 8), (32, 8), (8, 8), (24, 8)])
def test_verify_split_decode_path(q_len, Hq, Hkv):
    # 9 sequences x 8 kv heads: too few items for the tensor-core path
    cached = [0, 1, 63, 64, 255, 256, 700, 1500, 2047]
    w = verify_batch(cached, q_len, Hq, Hkv, 96, 7050 + 10 * q_len + Hq)
    assert not tensor_core_path(w, q_len)
    run_and_check(w, q_len, what=f"split decode q_len={q_len} Hq={Hq} Hkv={Hkv}")


def test_rows_beyond_one_tile_use_split_decode():
    # g * q_len = 16 * 16 = 256 rows per kv head: more than one 128-row tile
    w = verify_batch(CACHED_24[:12], 16, 32, 2, 256, 7060)
    assert not tensor_core_path(w, 16)
    run_and_check(w, 16, what="g*q_len > 128")


@pytest.mark.parametrize("num_splits", [1, 2, 5, 16])
def test_forced_splits_leave_early_positions_empty(num_splits):
    # with many splits the last one can hold only keys that the earlier query
    # positions must not see: their partial there is empty and must not spoil
    # the merge
    q_len = 8
    # contexts of 256k + 3 and 256k + 2: the last block holds only keys that
    # position 0 cannot see
    cached = [256 * 5 - 5, 256 * 3 - 6, 100, 256 * 7 - 2, 2]
    w = verify_batch(cached, q_len, 16, 8, 96, 7100 + num_splits)
    run_and_check(w, q_len, num_splits=num_splits, what=f"splits={num_splits}")


def test_q_len_one_is_plain_decode():
    # q_len = 1 gives bit-identical results to paged_decode_attention
    dev = "cuda"
    w = W.make_decode([5, 256, 257, 1000, 3000], 16, 8, 64, 7200)
    kc, vc = w.k_cache.to(dev), w.v_cache.to(dev)
    tables, ctx = w.block_tables.to(dev), w.context_lens.to(dev)
    q = w.q.to(dev)
    o1, l1 = pkv.paged_decode_attention(q, kc, vc, tables, ctx, w.scale)
    o2, l2 = pkv.paged_decode_attention_multiquery(q.unsqueeze(1), kc, vc, tables, ctx, w.scale)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2.squeeze(1))
    assert torch.equal(l1, l2.squeeze(1))


def test_context_shorter_than_q_len_is_reported():
    dev = "cuda"
    w = verify_batch([10, 20], 4, 16, 8, 8, 7300)
    kc, vc = w.k_cache.to(dev), w.v_cache.to(dev)
    q = w.q.to(dev).view(2, 4, 16, 128)
    ctx = torch.tensor([14, 3], dtype=torch.int32, device=dev)   # 3 < q_len
    pkv.paged_decode_attention_multiquery(q, kc, vc, w.block_tables.to(dev), ctx, w.scale)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == pkv.PKV_ERR_DEVICE_INDEX
    assert pkv.get_device_error() == pkv.PKV_OK   # reading clears it


@pytest.mark.parametrize("q_len", [4, 8])
def test_verify_batch_of_decode_size(q_len):
    # batch-64 verify of q_len proposed tokens over contexts like the decode
    # bench: 8 rows per kv head on the split-K decode kernel, 16 on tcgen05
    lens = W._uniform_ints(512, 4096, 64, W.seed_for(2))
    w = verify_batch([L - q_len for L in lens], q_len, 16, 8, 1200, 7400 + q_len)
    assert tensor_core_path(w, q_len) == (q_len == 8)
    run_and_check(w, q_len, what=f"b64 verify q_len={q_len}")
