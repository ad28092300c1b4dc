"""Helpers shared by the GPU parity tests: move a workload to the device, and
hand the oracle host copies of exactly the inputs the GPU saw (taken before
any library kernel ran)."""
from __future__ import annotations

import numpy as np
import torch

ATOL_OUT = 1e-2   # max |out_gpu - out_oracle| (bf16 output, fp32 accumulation)
ATOL_LSE = 1e-3   # max |lse_gpu - lse_oracle|


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def to_dev(t, dev="cuda"):
    return t.to(dev) if t.device.type != "cuda" else t


def compact_pool(k_cache, v_cache, tables: torch.Tensor):
    """Host copy of only the physical blocks that `tables` references, with the
    tables renumbered to the copy.  Relabelling physical blocks leaves the
    oracle's result bit-identical (pinned by the permutation-invariance pin)."""
    used = tables[tables >= 0].unique()
    remap = torch.full((k_cache.shape[0],), -1, dtype=torch.int64)
    remap[used.long()] = torch.arange(used.numel())
    idx = used.to(k_cache.device).long()
    kc = bits(k_cache.index_select(0, idx))
    vc = bits(v_cache.index_select(0, idx))
    t = tables.clone().long()
    t[t >= 0] = remap[t[t >= 0]]
    return kc.copy(), vc.copy(), t.to(torch.int32).numpy()


def assert_close(out_gpu: torch.Tensor, lse_gpu, ref_o: np.ndarray, ref_l: np.ndarray, what=""):
    o = out_gpu.float().cpu().numpy().astype(np.float64)
    err_o = float(np.abs(o - ref_o).max()) if o.size else 0.0
    assert np.abs(ref_o).max(initial=0) < 4.0, "tolerance assumes |out| < 4 (bf16 half-ulp)"
    assert err_o <= ATOL_OUT, f"{what}: max|dout| = {err_o}"
    if lse_gpu is not None:
        l = lse_gpu.cpu().numpy().astype(np.float64)
        fin = np.isfinite(ref_l)
        assert np.array_equal(np.isfinite(l), fin), f"{what}: lse finiteness differs"
        err_l = float(np.abs(l[fin] - ref_l[fin]).max()) if fin.any() else 0.0
        assert err_l <= ATOL_LSE, f"{what}: max|dlse| = {err_l}"
        return err_o, err_l
    return err_o, None
