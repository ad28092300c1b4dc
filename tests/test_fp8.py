"""FP8 (E4M3) KV cache on the GPU against the oracle: kv_cache_store_fp8 must
produce the oracle's codes bit for bit; paged_decode_attention_fp8 over those
codes must match the oracle's fp64 decode of the same codes (max|dout| <= 1e-2,
max|dlse| <= 1e-3)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_close, bits, compact_pool
from paged_kv_cache_214_gb300 import pkv
from paged_kv_cache_214_gb300 import workloads as W

pytestmark = pytest.mark.gpu

E4M3_MAX = 448.0


def bf16_from_bits(u16: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(u16.astype(np.uint16).view(np.int16)).view(torch.bfloat16)


def spread_values(shape, seed):
    """bf16 values over many binades: subnormal codes, ties, saturation."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(shape, generator=g, dtype=torch.float32)
    e = torch.randint(-14, 10, shape, generator=g).float()
    return (x * torch.pow(2.0, e)).to(torch.bfloat16)


def store_on_gpu(k, v, k_scale, v_scale, slots, num_blocks, Hkv):
    dev = "cuda"
    k8 = torch.zeros((num_blocks, 256, Hkv, 128), dtype=torch.uint8, device=dev)
    v8 = torch.zeros_like(k8)
    pkv.kv_cache_store_fp8(k.to(dev) if k.device.type != "cuda" else k,
                           v.to(dev) if v.device.type != "cuda" else v, k8, v8,
                           torch.as_tensor(slots, dtype=torch.int32).to(dev), k_scale, v_scale)
    torch.cuda.synchronize()
    return k8, v8


def assert_codes_equal(gpu: torch.Tensor, ref: np.ndarray, inputs: np.ndarray = None,
                       what=""):
    """Bit-exact comparison; on a mismatch name the first differing elements
    (with the bf16 input bits when `inputs` gives them in slot order)."""
    g = gpu.cpu().numpy()
    if np.array_equal(g, ref):
        return
    bad = np.flatnonzero(g.reshape(-1) != ref.reshape(-1))[:12]
    rows = []
    for i in bad:
        x = f"x=0x{int(inputs.reshape(-1)[i]):04x} " if inputs is not None else ""
        rows.append(f"[{i}] {x}gpu=0x{int(g.reshape(-1)[i]):02x} "
                    f"oracle=0x{int(ref.reshape(-1)[i]):02x}")
    raise AssertionError(f"{what}: {np.count_nonzero(g != ref)} codes differ: " + "; ".join(rows))


def store_on_oracle(k, v, k_scale, v_scale, slots, num_blocks, Hkv):
    k8 = np.zeros((num_blocks, 256, Hkv, 128), np.uint8)
    v8 = np.zeros_like(k8)
    oracle.store_fp8(bits(k.contiguous()), bits(v.contiguous()), k8, v8,
                     np.asarray(slots, np.int32), k_scale, v_scale)
    return k8, v8


@pytest.mark.parametrize("k_scale,v_scale", [(1.0, 1.0), (0.75, 3.0), (2.0 ** -5, 1.0 / 7),
                                             (6.0 / E4M3_MAX, 5.5 / E4M3_MAX)])
def test_store_bit_exact(k_scale, v_scale):
    # 600 tokens over 4 blocks: scattered slots, padding (-1) entries skipped
    T, Hkv, NB = 600, 8, 4
    k = spread_values((T, Hkv, 128), 8000)
    v = spread_values((T, Hkv, 128), 8001)
    g = torch.Generator().manual_seed(8002)
    slots = torch.randperm(NB * 256, generator=g)[:T].to(torch.int32)
    slots[::37] = -1
    gk, gv = store_on_gpu(k, v, k_scale, v_scale, slots, NB, Hkv)
    assert pkv.get_device_error() == pkv.PKV_OK
    rk, rv = store_on_oracle(k, v, k_scale, v_scale, slots, NB, Hkv)
    assert_codes_equal(gk, rk, what="K")
    assert_codes_equal(gv, rv, what="V")


def test_store_special_values_and_ties():
    # every finite bf16 magnitude from 2^-12 to 2^10 (round-to-nearest-even
    # ties, subnormal codes, values past 448 that saturate), +-0, +-inf and a
    # positive NaN, under scale 1
    mags = np.arange(0x3980, 0x4480, dtype=np.uint16)      # 2^-12 .. 2^10
    special = np.array([0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC0], np.uint16)
    vals = np.concatenate([mags, mags | 0x8000, special])
    n = -(-vals.size // 1024) * 1024
    vals = np.concatenate([vals, np.zeros(n - vals.size, np.uint16)])
    k = bf16_from_bits(vals).view(-1, 8, 128)
    v = bf16_from_bits(vals[::-1].copy()).view(-1, 8, 128)
    T = k.shape[0]
    slots = np.arange(T, dtype=np.int32)
    gk, gv = store_on_gpu(k, v, 1.0, 1.0, slots, 1, 8)
    rk, rv = store_on_oracle(k, v, 1.0, 1.0, slots, 1, 8)
    pad = np.zeros(256 * 1024 - vals.size, np.uint16)
    assert_codes_equal(gk, rk, np.concatenate([vals, pad]), "K")
    assert_codes_equal(gv, rv, np.concatenate([vals[::-1], pad]), "V")
    # a few fixed codes, as a sanity check on the byte order of the pairs
    flat = gk.cpu().numpy().reshape(-1)[:vals.size]
    pos = {int(u): i for i, u in enumerate(vals)}
    assert flat[pos[0x3F80]] == 0x38          # 1.0
    assert flat[pos[0x43E0]] == 0x7E          # 448
    assert flat[pos[0x4400]] == 0x7E          # 512 saturates
    assert flat[pos[0x7F80]] == 0x7E and flat[pos[0xFF80]] == 0xFE   # +-inf saturate
    assert flat[pos[0x7FC0]] == 0x7F          # NaN


def test_negative_nan_gives_a_nan_code():
    # the sign of a NaN's code is not fixed by the format reading: 0x7F or 0xFF
    vals = np.full(1024, 0xFFC0, np.uint16)
    k = bf16_from_bits(vals).view(1, 8, 128)
    gk, gv = store_on_gpu(k, k, 1.0, 1.0, [0], 1, 8)
    codes = np.unique(gk.cpu().numpy()[0, 0])
    assert set(codes.tolist()) <= {0x7F, 0xFF}


def test_store_unaligned_rows_take_the_scalar_path():
    # token stride of Hkv*D + 1 elements: rows start off 16-byte boundaries
    T, Hkv = 300, 4
    base = spread_values((T, Hkv * 128 + 1), 8100)
    shape, strides = (T, Hkv, 128), (Hkv * 128 + 1, 128, 1)
    k, v = base.as_strided(shape, strides), base.as_strided(shape, strides, 1)
    dbase = base.cuda()
    kd, vd = dbase.as_strided(shape, strides), dbase.as_strided(shape, strides, 1)
    slots = np.arange(T, dtype=np.int32)[::-1].copy()
    gk, gv = store_on_gpu(kd, vd, 0.5, 0.25, slots, 2, Hkv)
    rk, rv = store_on_oracle(k, v, 0.5, 0.25, slots, 2, Hkv)
    assert_codes_equal(gk, rk, what="K")
    assert_codes_equal(gv, rv, what="V")


def test_store_slot_out_of_range_is_reported():
    k = spread_values((4, 8, 128), 8200)
    store_on_gpu(k, k, 1.0, 1.0, [0, 1, 256 * 2, 3], 2, 8)
    assert pkv.get_device_error() == pkv.PKV_ERR_DEVICE_INDEX
    assert pkv.get_device_error() == pkv.PKV_OK


def run_decode_and_check(w, k_scale, v_scale, num_splits=0, what=""):
    """GPU: quantize the whole bf16 pool with the FP8 store, store the step's new
    tokens, decode.  Oracle: the same three steps from host copies of the bf16
    inputs.  The two FP8 pools must agree bit for bit before the decodes are
    compared."""
    dev = "cuda"
    kc, vc = w.k_cache.to(dev), w.v_cache.to(dev)
    NB, bs, Hkv = w.num_blocks, w.block_size, w.Hkv
    k8, v8 = store_on_gpu(kc.view(NB * bs, Hkv, 128), vc.view(NB * bs, Hkv, 128), k_scale,
                          v_scale, np.arange(NB * bs, dtype=np.int32), NB, Hkv)
    pkv.kv_cache_store_fp8(w.k_new.to(dev), w.v_new.to(dev), k8, v8, w.slot_mapping.to(dev),
                           k_scale, v_scale)
    tables, ctx = w.block_tables.to(dev), w.context_lens.to(dev)
    out, lse = pkv.paged_decode_attention_fp8(w.q.to(dev), k8, v8, tables, ctx, w.scale,
                                              k_scale, v_scale, num_splits=num_splits)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == pkv.PKV_OK

    kh, vh, th = compact_pool(kc, vc, w.block_tables)
    n_used = kh.shape[0]
    k8h = np.zeros((n_used, bs, Hkv, 128), np.uint8)
    v8h = np.zeros_like(k8h)
    oracle.store_fp8(kh.reshape(-1, Hkv, 128), vh.reshape(-1, Hkv, 128), k8h, v8h,
                     np.arange(n_used * bs, dtype=np.int32), k_scale, v_scale)
    used = w.block_tables[w.block_tables >= 0].unique()
    remap = {int(b): i for i, b in enumerate(used)}
    slot_host = np.array([remap[int(s) // bs] * bs + int(s) % bs if s >= 0 else -1
                          for s in w.slot_mapping], np.int32)
    oracle.store_fp8(bits(w.k_new), bits(w.v_new), k8h, v8h, slot_host, k_scale, v_scale)
    idx = used.to(dev).long()
    assert_codes_equal(k8.index_select(0, idx), k8h, kh, f"{what}: K")
    assert_codes_equal(v8.index_select(0, idx), v8h, vh, f"{what}: V")
    ref_o, ref_l = oracle.decode_fp8(bits(w.q), k8h, v8h, th, w.context_lens.numpy(), w.scale,
                                     k_scale, v_scale)
    return assert_close(out, lse, ref_o, ref_l, what)


CTX = [1, 17, 255, 256, 257, 1000, 4096, 6000]
SCALES = [(1.0, 1.0), (6.0 / E4M3_MAX, 5.0 / E4M3_MAX), (1.0 / 128, 1.0 / 200)]


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (16, 8), (32, 8), (64, 8), (12, 4)])
@pytest.mark.parametrize("k_scale,v_scale", SCALES)
def test_decode_matches_oracle(Hq, Hkv, k_scale, v_scale):
    w = W.make_decode(CTX, Hq, Hkv, 64, 8300 + Hq + Hkv)
    run_decode_and_check(w, k_scale, v_scale, what=f"Hq={Hq} Hkv={Hkv} ks={k_scale}")


@pytest.mark.parametrize("num_splits", [1, 3, 16])
def test_decode_forced_splits(num_splits):
    w = W.make_decode(CTX, 32, 8, 64, 8400 + num_splits)
    run_decode_and_check(w, *SCALES[1], num_splits=num_splits, what=f"splits={num_splits}")


@pytest.mark.parametrize("num_splits,Hq", [(2, 16), (3, 32), (2, 64)])
def test_decode_long_splits(num_splits, Hq):
    # splits of 8 blocks or more run the E4M3 decode's producer-warp form (a
    # fifth warp copies the stages, 6 stages at two blocks per SM)
    w = W.make_decode(CTX, Hq, 8, 64, 8450 + Hq + num_splits)
    maxblk = w.block_tables.shape[1]
    S = pkv.paged_decode_num_splits(w.B, w.Hq, w.Hkv, w.D, maxblk, w.block_size, num_splits)
    assert S == num_splits and -(-maxblk // S) >= 8
    run_decode_and_check(w, *SCALES[1], num_splits=num_splits, what=f"long splits S={S}")


def test_decode_empty_context_gives_zero_and_minus_inf():
    w = W.make_decode([0, 300, 0], 16, 8, 8, 8500)
    run_decode_and_check(w, *SCALES[1], what="empty contexts")


def test_decode_long_context():
    w = W.make_decode([40000, 70001], 32, 8, 460, 8600, pool_device="cuda")
    run_decode_and_check(w, *SCALES[1], what="long context")


def test_decode_b64_workload():
    # the batch-64 decode workload (16 q heads / 8 kv heads, contexts U[512, 4096])
    w = W.config_workload(2, pool_device="cuda")
    run_decode_and_check(w, *SCALES[1], what="decode-b64 fp8")


@pytest.mark.parametrize("num_splits", [0, 2])
@pytest.mark.parametrize("Hq,Hkv", [(16, 8), (32, 8), (64, 8)])
def test_fused_store_decode_same_bits_as_two_calls(Hq, Hkv, num_splits):
    # paged_decode_attention_fp8_store = kv_cache_store_fp8 + the E4M3 decode
    # (num_splits = 2: 12-block splits, the producer-warp form)
    dev = "cuda"
    ks, vs = SCALES[1]
    w = W.make_decode([0, 3, 256, 257, 1000, 3000, 6000], Hq, Hkv, 64, 8700 + Hq)
    NB, bs = w.num_blocks, w.block_size
    k8, v8 = store_on_gpu(w.k_cache.view(NB * bs, Hkv, 128), w.v_cache.view(NB * bs, Hkv, 128),
                          ks, vs, np.arange(NB * bs, dtype=np.int32), NB, Hkv)
    k8b, v8b = k8.clone(), v8.clone()
    q, kn, vn, slots = w.q.to(dev), w.k_new.to(dev), w.v_new.to(dev), w.slot_mapping.to(dev)
    tables, ctx = w.block_tables.to(dev), w.context_lens.to(dev)
    pkv.kv_cache_store_fp8(kn, vn, k8, v8, slots, ks, vs)
    o1, l1 = pkv.paged_decode_attention_fp8(q, k8, v8, tables, ctx, w.scale, ks, vs,
                                            num_splits=num_splits)
    o2, l2 = pkv.paged_decode_attention_fp8_store(q, kn, vn, slots, k8b, v8b, tables, ctx,
                                                  w.scale, ks, vs, num_splits=num_splits)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == pkv.PKV_OK
    assert torch.equal(k8, k8b) and torch.equal(v8, v8b)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    # and the oracle agrees with the fused result
    run_decode_and_check(w, ks, vs, num_splits=num_splits, what=f"fused fp8 Hq={Hq}")
