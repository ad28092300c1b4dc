"""paged_decode_attention_noalloc: decode for callers that cannot allocate
device memory (e.g. a plugin whose host framework owns every allocation), with
its split scratch in a fixed array inside the library.

Checked through the C ABI against paged_decode_attention (which takes a
caller-provided workspace), on two calls in a row, within the tolerances the
other decode tests use.  This file is collected last on purpose."""
import pytest
import torch

from gpu_helpers import ATOL_LSE, ATOL_OUT
from paged_kv_cache_214_gb300 import pkv
from paged_kv_cache_214_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _inputs(w, dev="cuda"):
    return (w.q.to(dev), w.k_cache.to(dev), w.v_cache.to(dev), w.block_tables.to(dev),
            w.context_lens.to(dev))


@pytest.mark.parametrize("num_splits", [0, 5])
def test_noalloc_matches_workspace_path_twice(num_splits):
    w = W.make_decode([3000, 900, 8000, 257, 4100, 1], 32, 8, 96, 7100,
                      store_new_token=False, pool_device="cuda")
    q, kc, vc, bt, lens = _inputs(w)
    need = pkv.paged_decode_workspace_bytes(w.B, w.Hq, w.Hkv, w.D, bt.shape[1],
                                            num_splits=num_splits)
    assert 0 < need <= pkv.NOALLOC_SCRATCH_BYTES
    ref_o, ref_l = pkv.paged_decode_attention(q, kc, vc, bt, lens, w.scale,
                                              num_splits=num_splits)
    ref_o, ref_l = ref_o.clone(), ref_l.clone()
    for _ in range(2):
        out = torch.full_like(q, float("nan"))
        lse = torch.full((w.B, w.Hq), float("nan"), dtype=torch.float32, device=q.device)
        pkv.paged_decode_attention_noalloc(q, kc, vc, bt, lens, w.scale, out, lse,
                                           num_splits=num_splits)
        torch.cuda.synchronize()
        assert pkv.get_device_error() == pkv.PKV_OK
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
