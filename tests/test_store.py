"""kv_cache_store on the GPU against the oracle: bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import bits, compact_pool
from paged_kv_cache_214_gb300 import pkv
from paged_kv_cache_214_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _check_store(k, v, kc, vc, slots):
    """Run the GPU store on (kc, vc) in place and compare with the oracle's store
    on host copies of the touched blocks; also check nothing else changed."""
    before_k, before_v = kc.clone(), vc.clone()
    pkv.kv_cache_store(k, v, kc, vc, slots)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == pkv.PKV_OK
    s = slots.cpu().long()
    bs = kc.shape[1]
    valid = s[s >= 0]
    blocks = torch.unique(valid // bs)
    table = blocks.to(torch.int32)[None, :]
    kh, vh, tb = compact_pool(before_k, before_v, table)
    remap = {int(b): int(c) for b, c in zip(blocks, torch.tensor(tb[0]))}
    s_c = s.clone()
    s_c[s >= 0] = torch.tensor([remap[int(x) // bs] * bs + int(x) % bs for x in valid],
                               dtype=torch.int64)
    oracle.store(bits(k), bits(v), kh, vh, s_c.to(torch.int32).numpy())
    ga, gb, _ = compact_pool(kc, vc, table)
    assert np.array_equal(ga, kh) and np.array_equal(gb, vh), "stored rows differ"
    # every slot outside slot_mapping is unchanged
    changed = ((kc != before_k) | (vc != before_v)).flatten(2).any(-1).flatten()
    allowed = torch.zeros_like(changed)
    allowed[valid.to(changed.device)] = True
    assert not (changed & ~allowed).any(), "a slot outside slot_mapping changed"


@pytest.mark.parametrize("cfg", [1, 2, 4])
def test_store_workloads(cfg):
    w = W.config_workload(cfg, pool_device="cuda")
    _check_store(w.k_new.cuda(), w.v_new.cuda(), w.k_cache, w.v_cache, w.slot_mapping.cuda())


def test_store_edge_slots_and_padding():
    g = torch.Generator().manual_seed(5)
    NB, bs, Hkv, D = 8, 256, 8, 128
    kc = torch.randn((NB, bs, Hkv, D), generator=g).to(torch.bfloat16).cuda()
    vc = torch.randn((NB, bs, Hkv, D), generator=g).to(torch.bfloat16).cuda()
    slots = torch.tensor([0, 255, 256, 3 * bs + 128, NB * bs - 1, -1, -7], dtype=torch.int32)
    T = len(slots)
    k = torch.randn((T, Hkv, D), generator=g).to(torch.bfloat16).cuda()
    v = torch.randn((T, Hkv, D), generator=g).to(torch.bfloat16).cuda()
    _check_store(k, v, kc, vc, slots.cuda())


def test_store_strided_and_unaligned_rows():
    """Token stride larger than a row (a slice of a fused QKV buffer), and an odd
    stride that forces the element-wise path."""
    g = torch.Generator().manual_seed(6)
    NB, bs, Hkv, D = 4, 256, 2, 128
    for extra in (3 * Hkv * D, 1):
        kc = torch.randn((NB, bs, Hkv, D), generator=g).to(torch.bfloat16).cuda()
        vc = torch.randn((NB, bs, Hkv, D), generator=g).to(torch.bfloat16).cuda()
        T = 37
        buf = torch.randn((T, Hkv * D + extra), generator=g).to(torch.bfloat16).cuda()
        buf2 = torch.randn((T, Hkv * D + extra), generator=g).to(torch.bfloat16).cuda()
        k = buf[:, :Hkv * D].view(T, Hkv, D) if extra != 1 else \
            torch.as_strided(buf, (T, Hkv, D), (Hkv * D + 1, D, 1))
        v = torch.as_strided(buf2, (T, Hkv, D), (Hkv * D + extra, D, 1))
        slots = torch.randperm(NB * bs, generator=g)[:T].to(torch.int32)
        _check_store(k, v, kc, vc, slots.cuda())


def test_store_empty_is_noop():
    kc = torch.zeros((2, 256, 1, 128), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    e = torch.empty((0, 1, 128), dtype=torch.bfloat16, device="cuda")
    pkv.kv_cache_store(e, e, kc, vc, torch.empty(0, dtype=torch.int32, device="cuda"))
    assert not kc.any() and not vc.any()


def test_store_out_of_range_slot_reported_and_skipped():
    kc = torch.zeros((2, 256, 1, 128), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    k = torch.ones((2, 1, 128), dtype=torch.bfloat16, device="cuda")
    slots = torch.tensor([512, 3], dtype=torch.int32, device="cuda")
    assert pkv.get_device_error() == pkv.PKV_OK
    pkv.kv_cache_store(k, k, kc, vc, slots)
    assert pkv.get_device_error() == pkv.PKV_ERR_DEVICE_INDEX
    assert pkv.get_device_error() == pkv.PKV_OK  # read-and-clear
    assert kc[0, 3].float().eq(1).all() and kc.float().sum() == 128
