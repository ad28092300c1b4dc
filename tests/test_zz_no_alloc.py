"""paged_decode_attention_noalloc: decode for callers that cannot allocate
device memory (e.g. a plugin whose host framework owns every allocation), with
its split scratch in a fixed array inside the library.

Checked through the C ABI against the oracle and against paged_decode_attention
(which takes a caller-provided workspace), on two calls in a row, within the
tolerances the other decode tests use; then a large call followed by a smaller
one with another head grouping, which must not see the large call's leftover
counters or partials.  This file is collected last on purpose."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import ATOL_LSE, ATOL_OUT, assert_close, bits
from paged_kv_cache_214_gb300 import pkv
from paged_kv_cache_214_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _inputs(w, dev="cuda"):
    return (w.q.to(dev), w.k_cache.to(dev), w.v_cache.to(dev), w.block_tables.to(dev),
            w.context_lens.to(dev))


def _oracle(w):
    return oracle.decode(bits(w.q), bits(w.k_cache), bits(w.v_cache), w.block_tables.numpy(),
                         w.context_lens.numpy(), w.scale)


def _noalloc(w, args, num_splits):
    q = args[0]
    out = torch.full_like(q, float("nan"))
    lse = torch.full((w.B, w.Hq), float("nan"), dtype=torch.float32, device=q.device)
    pkv.paged_decode_attention_noalloc(*args, w.scale, out, lse, num_splits=num_splits)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == pkv.PKV_OK
    return out, lse


@pytest.mark.parametrize("num_splits", [0, 5])
def test_noalloc_matches_oracle_and_workspace_path_twice(num_splits):
    w = W.make_decode([3000, 900, 8000, 257, 4100, 1], 32, 8, 96, 7100,
                      store_new_token=False)
    args = _inputs(w)
    need = pkv.paged_decode_workspace_bytes(w.B, w.Hq, w.Hkv, w.D, args[3].shape[1],
                                            num_splits=num_splits)
    assert 0 < need <= pkv.NOALLOC_SCRATCH_BYTES
    ref_o, ref_l = pkv.paged_decode_attention(*args, w.scale, num_splits=num_splits)
    ref_o, ref_l = ref_o.clone(), ref_l.clone()
    orc_o, orc_l = _oracle(w)
    for _ in range(2):
        out, lse = _noalloc(w, args, num_splits)
        assert_close(out, lse, orc_o, orc_l, f"noalloc vs oracle, S={num_splits}")
        assert (out.float() - ref_o.float()).abs().max().item() <= ATOL_OUT
        assert (lse - ref_l).abs().max().item() <= ATOL_LSE


def test_noalloc_large_call_then_smaller_call():
    """A large call leaves counters and partials in the shared array; a smaller
    call with another head grouping (fewer counters, another partial layout)
    must still match the oracle and the workspace path, twice."""
    big = W.make_decode([6000, 7000, 5000, 6500, 4000, 7100, 3000, 6900], 64, 8, 240, 7200,
                        store_new_token=False)
    small = W.make_decode([2000, 300, 4500], 12, 2, 48, 7201, store_new_token=False)
    big_args, small_args = _inputs(big), _inputs(small)
    assert (pkv.paged_decode_workspace_bytes(big.B, big.Hq, big.Hkv, big.D,
                                             big_args[3].shape[1], num_splits=7)
            <= pkv.NOALLOC_SCRATCH_BYTES)
    orc_big, orc_small = _oracle(big), _oracle(small)
    ref_o, ref_l = pkv.paged_decode_attention(*small_args, small.scale, num_splits=3)
    ref_o, ref_l = ref_o.clone(), ref_l.clone()
    for rep in range(2):
        out, lse = _noalloc(big, big_args, 7)
        assert_close(out, lse, *orc_big, f"large call {rep}")
        out, lse = _noalloc(small, small_args, 3)
        assert_close(out, lse, *orc_small, f"smaller call {rep}")
        assert (out.float() - ref_o.float()).abs().max().item() <= ATOL_OUT
        assert (lse - ref_l).abs().max().item() <= ATOL_LSE


def test_noalloc_rejects_work_beyond_its_scratch():
    # 64 sequences x 32 heads x 64 splits of partials: far beyond 16 MiB.  The
    # call is refused on the host, so the inputs' contents do not matter.
    dev = "cuda"
    B, Hq, Hkv, maxblk = 64, 32, 8, 64
    q = torch.zeros((B, Hq, 128), dtype=torch.bfloat16, device=dev)
    kc = torch.zeros((4, 256, Hkv, 128), dtype=torch.bfloat16, device=dev)
    bt = torch.zeros((B, maxblk), dtype=torch.int32, device=dev)
    lens = torch.full((B,), maxblk * 256, dtype=torch.int32, device=dev)
    need = pkv.paged_decode_workspace_bytes(B, Hq, Hkv, 128, maxblk, num_splits=64)
    assert need > pkv.NOALLOC_SCRATCH_BYTES
    out = torch.zeros_like(q)
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_decode_attention_noalloc(q, kc, kc, bt, lens, 128 ** -0.5, out, num_splits=64)
    assert e.value.status == pkv.PKV_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert not out.any()


def test_noalloc_refuses_a_bad_argument_before_queueing_anything():
    # a misaligned output pointer: refused by the argument checks, which now
    # run before the counter clear is queued
    w = W.make_decode([700, 300], 16, 8, 8, 7300, store_new_token=False)
    args = _inputs(w)
    buf = torch.zeros(w.B * w.Hq * w.D + 8, dtype=torch.bfloat16, device="cuda")
    out = buf[1:1 + w.B * w.Hq * w.D].view(w.B, w.Hq, w.D)   # 2-byte offset
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_decode_attention_noalloc(*args, w.scale, out, num_splits=2)
    assert e.value.status == pkv.PKV_ERR_ARG
    torch.cuda.synchronize()
    assert not buf.any()
    # and the next good call still matches the oracle
    out, lse = _noalloc(w, args, 2)
    assert_close(out, lse, *_oracle(w), "after a refused call")
    assert np.isfinite(lse.cpu().numpy()).all()


def test_noalloc_after_a_timed_out_call():
    """A no-allocation call whose wait runs out (the test hook lowers the wait
    limit and withholds a tile; nothing faults or hangs) reports
    PKV_ERR_TIMEOUT, and the next call, on the same shared scratch, returns
    PKV_OK and matches the oracle."""
    w = W.make_decode([3000, 1500, 3500], 16, 8, 48, 7400, store_new_token=False)
    args = _inputs(w)
    out = torch.zeros_like(args[0])
    assert pkv.get_device_error() == pkv.PKV_OK
    try:
        pkv.testing_set_wait_fault(1_000_000, 2)
        pkv.paged_decode_attention_noalloc(*args, w.scale, out, num_splits=4)
        torch.cuda.synchronize()
        assert pkv.get_device_error() == pkv.PKV_ERR_TIMEOUT
    finally:
        pkv.testing_set_wait_fault(0, -1)
    o, lse = _noalloc(w, args, 4)
    assert_close(o, lse, *_oracle(w), "no-allocation call after a timed-out one")
