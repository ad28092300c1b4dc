"""paged_prefill_attention (tcgen05) on the GPU against the oracle, after the
store of the chunk's new tokens (max|dout| <= 1e-2, max|dlse| <= 1e-3)."""
import time

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_close, bits, compact_pool
from paged_kv_cache_214_gb300 import pkv
from paged_kv_cache_214_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def run_and_check(w, sample=None, what=""):
    """GPU: store the new tokens, then prefill.  Oracle: the same two steps on
    host copies of the inputs taken before any library kernel ran.  `sample`:
    the sequences the oracle checks (all by default)."""
    dev = "cuda"
    kc, vc = w.k_cache.to(dev), w.v_cache.to(dev)
    seqs = list(range(w.B)) if sample is None else list(sample)
    tables = w.block_tables[seqs]
    kh, vh, th = compact_pool(kc, vc, tables)
    used = tables[tables >= 0].unique()
    remap = {int(b): i for i, b in enumerate(used)}
    bs = w.block_size
    cq = w.cu_seqlens_q.tolist()
    rows = [r for s in seqs for r in range(cq[s], cq[s + 1])]
    slots = [int(x) for x in w.slot_mapping[rows]]
    slot_host = np.array([remap[s // bs] * bs + s % bs for s in slots], np.int32)
    pkv.kv_cache_store(w.k_new.to(dev), w.v_new.to(dev), kc, vc, w.slot_mapping.to(dev))
    out, lse = pkv.paged_prefill_attention(
        w.q.to(dev), kc, vc, w.block_tables.to(dev), w.cu_seqlens_q.to(dev),
        w.cu_seqlens_k.to(dev), w.max_seqlen_q, w.max_seqlen_k, w.scale)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == pkv.PKV_OK
    oracle.store(bits(w.k_new[rows]), bits(w.v_new[rows]), kh, vh, slot_host)
    lq = [w.q_lens[s] for s in seqs]
    lk = [w.k_lens[s] for s in seqs]
    cu_q = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    ref_o, ref_l = oracle.prefill(bits(w.q[rows]), kh, vh, th, cu_q, cu_k, w.scale)
    return assert_close(out[rows], lse[rows], ref_o, ref_l, what)


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 2), (32, 8), (12, 4)])
def test_ragged_chunks(Hq, Hkv):
    prefix = [0, 0, 256, 1000, 37, 511]
    new = [1, 130, 129, 300, 5, 256]
    w = W.make_prefill(prefix, new, Hq, Hkv, 64, 5000 + Hq + Hkv)
    run_and_check(w, what=f"ragged Hq={Hq} Hkv={Hkv}")


def test_tile_and_block_edges():
    # q and k lengths at every tile / block boundary residue
    new = [127, 128, 129, 255, 256, 257, 384]
    prefix = [1, 127, 128, 129, 0, 255, 256]
    w = W.make_prefill(prefix, new, 8, 2, 96, 5100)
    run_and_check(w, what="edges")


def test_one_row_chunks_match_decode_semantics():
    w = W.make_prefill([17, 256, 999], [1, 1, 1], 16, 8, 16, 5200)
    run_and_check(w, what="Lq=1")


def test_no_prefix_long_prompt():
    w = W.make_prefill([0, 0], [1536, 700], 8, 8, 32, 5300)
    run_and_check(w, what="no prefix")


def test_chunked_prefill_b16_full():
    """Every row and head of the chunked-prefill workload (16 sequences)."""
    w = W.config_workload(4, pool_device="cuda")
    t0 = time.perf_counter()
    run_and_check(w, what="chunked-prefill-b16")
    print(f"chunked-prefill-b16: GPU + oracle check of all {w.B} sequences "
          f"{time.perf_counter() - t0:.1f} s")


@pytest.mark.parametrize("Hq,Hkv", [(2, 1), (16, 8), (6, 1)])
def test_no_prefix_even_groups(Hq, Hkv):
    # two query heads per item (even group sizes), prompts with no cached prefix
    w = W.make_prefill([0, 0, 0], [1000, 128, 77], Hq, Hkv, 32, 5310 + Hq)
    run_and_check(w, what=f"no prefix Hq={Hq} Hkv={Hkv}")


@pytest.mark.parametrize("Hq", [8, 16])
def test_lk_less_than_lq_is_reported(Hq):
    w = W.make_prefill([0, 100], [64, 64], Hq, 8, 8, 5400)
    dev = "cuda"
    cu_k = w.cu_seqlens_k.clone()
    cu_k[2] = cu_k[1] + 10            # sequence 1: Lk = 10 < Lq = 64
    assert pkv.get_device_error() == pkv.PKV_OK
    pkv.paged_prefill_attention(w.q.to(dev), w.k_cache.to(dev), w.v_cache.to(dev),
                                w.block_tables.to(dev), w.cu_seqlens_q.to(dev), cu_k.to(dev),
                                w.max_seqlen_q, w.max_seqlen_k, w.scale)
    assert pkv.get_device_error() == pkv.PKV_ERR_DEVICE_INDEX
    assert pkv.get_device_error() == pkv.PKV_OK


@pytest.mark.parametrize("Hq", [8, 16])
def test_bad_block_id_is_reported(Hq):
    w = W.make_prefill([300], [64], Hq, 8, 8, 5500)
    dev = "cuda"
    bt = w.block_tables.clone()
    bt[0, 0] = -3
    pkv.paged_prefill_attention(w.q.to(dev), w.k_cache.to(dev), w.v_cache.to(dev), bt.to(dev),
                                w.cu_seqlens_q.to(dev), w.cu_seqlens_k.to(dev), w.max_seqlen_q,
                                w.max_seqlen_k, w.scale)
    assert pkv.get_device_error() == pkv.PKV_ERR_DEVICE_INDEX
