"""Pins for the CPU oracle: checks that tie it to something other than itself.

Each ``pin_*`` function takes a loaded oracle library (ctypes handle) and raises
AssertionError on failure.  ``test_oracle_pins.py`` runs them on the real oracle;
``test_oracle_mutants.py`` runs them on deliberately broken builds of the
oracle and requires every broken build to fail at least one pin.

What pins what:
* store/gather addressing — round trip, explicit offsets 0 / 255 / 256, padding
  slots, rejection of out-of-range and repeated slots;
* attention values — brute force: dense softmax(scale q K^T) V written here with
  numpy matrix products on contiguous K/V that the test itself scatters into a
  shuffled pool; torch's CPU scaled_dot_product_attention in float64;
* closed forms — one key (out = v0, lse = s0); equal keys (out = mean of V,
  lse = s + ln L); one dominant key;
* invariances — physical block relabelling and prefix sharing (bit-identical),
  causal perturbation, chunked vs whole prefill, prefill with one query row vs
  decode, GQA vs MHA with repeated K/V.
* FP8 (E4M3) cache — the code table against torch's float8_e4m3fn and fixed
  anchors of the format; the quantizer against a brute-force search for the
  nearest finite code (ties to the even code) and against torch's conversion
  in range; the FP8 store's addressing; the FP8 decode against the bf16 decode
  on a pool holding the same values.
"""

from __future__ import annotations

import math

import numpy as np
import torch

import oracle as O

D = 128


def _bf16(shape, gen, scale=1.0):
    return (torch.randn(shape, generator=gen) * scale).to(torch.bfloat16)


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _f64(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float64).numpy()


def _scatter_pool(seqs_k, seqs_v, Hkv, bs, NB, gen, shared=None):
    """Build a shuffled pool from contiguous per-sequence K/V (torch bf16
    [L, Hkv, D]).  Returns (k_cache, v_cache torch bf16 [NB, bs, Hkv, D],
    tables int32 [B, maxblk]).  Unused blocks hold random data.
    ``shared``: (n_tokens) — the first n_tokens (whole blocks) of every sequence
    are identical and mapped to the same physical blocks."""
    k_cache = _bf16((NB, bs, Hkv, D), gen)
    v_cache = _bf16((NB, bs, Hkv, D), gen)
    perm = torch.randperm(NB, generator=gen).tolist()
    nxt = 0
    B = len(seqs_k)
    nblk = [-(-k.shape[0] // bs) for k in seqs_k]
    maxblk = max(nblk + [1])
    tables = np.full((B, maxblk), -1, np.int32)
    shared_blocks = []
    if shared:
        ns = shared // bs
        shared_blocks = perm[nxt:nxt + ns]
        nxt += ns
    for b in range(B):
        row = list(shared_blocks)
        need = nblk[b] - len(row)
        row += perm[nxt:nxt + need]
        nxt += need
        tables[b, :len(row)] = row
        for j in range(seqs_k[b].shape[0]):
            blk, off = row[j // bs], j % bs
            k_cache[blk, off] = seqs_k[b][j]
            v_cache[blk, off] = seqs_v[b][j]
    return k_cache, v_cache, tables


def dense_attention(q, K, V, scale, mask=None):
    """Textbook attention with numpy matrix products.
    q [M, D], K/V [L, D] float64; mask [M, L] bool (True = visible)."""
    M = q.shape[0]
    if K.shape[0] == 0:
        return np.zeros((M, V.shape[1])), np.full(M, -np.inf)
    S = (q @ K.T) * scale
    if mask is not None:
        S = np.where(mask, S, -np.inf)
    mx = S.max(axis=1, keepdims=True)
    P = np.exp(S - mx)
    l = P.sum(axis=1, keepdims=True)
    return (P @ V) / l, mx[:, 0] + np.log(l[:, 0])


# --------------------------------------------------------------------------
# store / gather addressing


def pin_store_roundtrip(lib):
    gen = torch.Generator().manual_seed(1)
    NB, bs, Hkv = 6, 256, 2
    k_cache = _bits(_bf16((NB, bs, Hkv, D), gen)).copy()
    v_cache = _bits(_bf16((NB, bs, Hkv, D), gen)).copy()
    before_k, before_v = k_cache.copy(), v_cache.copy()
    # offsets 0, 255 of block 3, 0 of block 4 (= flat 256 past block 3's start),
    # block 5's last slot, and one padding token
    slots = np.array([3 * bs + 0, 3 * bs + 255, 3 * bs + 256, NB * bs - 1, -1], np.int32)
    T = len(slots)
    k = _bits(_bf16((T, Hkv, D), gen))
    v = _bits(_bf16((T, Hkv, D), gen))
    O.store(k, v, k_cache, v_cache, slots, lib=lib)
    assert np.array_equal(k_cache[3, 0], k[0]) and np.array_equal(v_cache[3, 0], v[0])
    assert np.array_equal(k_cache[3, 255], k[1]) and np.array_equal(v_cache[3, 255], v[1])
    assert np.array_equal(k_cache[4, 0], k[2]) and np.array_equal(v_cache[4, 0], v[2])
    assert np.array_equal(k_cache[5, 255], k[3]) and np.array_equal(v_cache[5, 255], v[3])
    # nothing else changed (the padding token wrote nothing)
    touched = np.zeros((NB, bs), bool)
    touched[3, 0] = touched[3, 255] = touched[4, 0] = touched[5, 255] = True
    assert np.array_equal(k_cache[~touched], before_k[~touched])
    assert np.array_equal(v_cache[~touched], before_v[~touched])
    # round trip through a table: a sequence whose logical tokens 0..L-1 live in
    # blocks [4, 1, 3]; store then gather returns the stored rows bitwise.
    table = np.array([4, 1, 3], np.int32)
    L = 600
    pos = np.arange(L)
    slot_of = table[pos // bs] * bs + pos % bs
    kk = _bits(_bf16((L, Hkv, D), gen))
    vv = _bits(_bf16((L, Hkv, D), gen))
    O.store(kk, vv, k_cache, v_cache, slot_of.astype(np.int32), lib=lib)
    K, V = O.gather(k_cache, v_cache, table, L, lib=lib)
    assert np.array_equal(K, kk) and np.array_equal(V, vv)


def pin_copy_blocks(lib):
    """Copy-on-write copies: the destination block reads back as the source
    (through a table that points at it), nothing else changes, and an
    out-of-range id is rejected without a change."""
    gen = torch.Generator().manual_seed(16)
    NB, bs, Hkv = 6, 16, 2
    kc = _bits(_bf16((NB, bs, Hkv, D), gen)).copy()
    vc = _bits(_bf16((NB, bs, Hkv, D), gen)).copy()
    k0, v0 = kc.copy(), vc.copy()
    O.copy_blocks(kc, vc, [2, 4], [5, 0], lib=lib)
    K_src, V_src = O.gather(k0, v0, np.array([2, 4], np.int32), 2 * bs, lib=lib)
    K_dst, V_dst = O.gather(kc, vc, np.array([5, 0], np.int32), 2 * bs, lib=lib)
    assert np.array_equal(K_src, K_dst) and np.array_equal(V_src, V_dst)
    for b in (1, 2, 3, 4):
        assert np.array_equal(kc[b], k0[b]) and np.array_equal(vc[b], v0[b])
    try:
        O.copy_blocks(kc, vc, [1], [NB], lib=lib)
    except O.OracleError:
        pass
    else:
        raise AssertionError("an out-of-range block id was accepted")


def pin_store_rejects(lib):
    gen = torch.Generator().manual_seed(2)
    NB, bs, Hkv = 2, 256, 1
    kc = np.zeros((NB, bs, Hkv, D), np.uint16)
    vc = np.zeros((NB, bs, Hkv, D), np.uint16)
    k = _bits(_bf16((2, Hkv, D), gen))
    for bad in ([NB * bs, 0], [5, 5]):
        try:
            O.store(k, k, kc, vc, np.array(bad, np.int32), lib=lib)
        except O.OracleError:
            pass
        else:
            raise AssertionError(f"slots {bad} were accepted")
        assert not kc.any(), "a rejected store modified the cache"


# --------------------------------------------------------------------------
# decode


def _decode_case(gen, lens, Hq, Hkv, bs, NB, shared=None, scale=None):
    seqs_k, seqs_v = [], []
    prefix_k = _bf16((shared, Hkv, D), gen) if shared else None
    prefix_v = _bf16((shared, Hkv, D), gen) if shared else None
    for L in lens:
        k = _bf16((L, Hkv, D), gen)
        v = _bf16((L, Hkv, D), gen)
        if shared:
            k[:shared] = prefix_k
            v[:shared] = prefix_v
        seqs_k.append(k)
        seqs_v.append(v)
    kc, vc, tables = _scatter_pool(seqs_k, seqs_v, Hkv, bs, NB, gen, shared=shared)
    q = _bf16((len(lens), Hq, D), gen)
    return dict(q=q, seqs_k=seqs_k, seqs_v=seqs_v, kc=kc, vc=vc, tables=tables,
                lens=np.array(lens, np.int32), scale=scale or D ** -0.5)


def _run_decode(lib, c, nthreads=2):
    return O.decode(_bits(c["q"]), _bits(c["kc"]), _bits(c["vc"]), c["tables"],
                    c["lens"], c["scale"], nthreads=nthreads, lib=lib)


def pin_decode_bruteforce(lib):
    gen = torch.Generator().manual_seed(3)
    for bs in (16, 256):
        c = _decode_case(gen, [1, 17, 40, 70], Hq=8, Hkv=2, bs=bs, NB=24)
        out, lse = _run_decode(lib, c)
        g = 8 // 2
        for b, L in enumerate(c["lens"]):
            for h in range(8):
                K = _f64(c["seqs_k"][b][:, h // g])
                V = _f64(c["seqs_v"][b][:, h // g])
                o_ref, l_ref = dense_attention(_f64(c["q"][b, h])[None], K, V, c["scale"])
                assert np.max(np.abs(out[b, h] - o_ref[0])) < 1e-12, (bs, b, h)
                assert abs(lse[b, h] - l_ref[0]) < 1e-12, (bs, b, h)


def pin_decode_sdpa(lib):
    """torch's CPU scaled_dot_product_attention in float64 on the contiguous
    (unpaged) K/V; GQA through repeat_interleave."""
    gen = torch.Generator().manual_seed(4)
    Hq, Hkv = 8, 2
    c = _decode_case(gen, [5, 33, 257], Hq=Hq, Hkv=Hkv, bs=16, NB=40)
    out, lse = _run_decode(lib, c)
    for b, L in enumerate(c["lens"]):
        q = c["q"][b].to(torch.float64)[:, None, :]                   # [Hq, 1, D]
        K = c["seqs_k"][b].to(torch.float64).permute(1, 0, 2)          # [Hkv, L, D]
        V = c["seqs_v"][b].to(torch.float64).permute(1, 0, 2)
        K = K.repeat_interleave(Hq // Hkv, dim=0)
        V = V.repeat_interleave(Hq // Hkv, dim=0)
        ref = torch.nn.functional.scaled_dot_product_attention(q, K, V, scale=c["scale"])
        assert np.max(np.abs(out[b] - ref[:, 0].numpy())) < 1e-12
        s = (q @ K.transpose(1, 2))[:, 0] * c["scale"]
        assert np.max(np.abs(lse[b] - torch.logsumexp(s, dim=-1).numpy())) < 1e-12


def pin_decode_closed_forms(lib):
    gen = torch.Generator().manual_seed(5)
    Hq = Hkv = 2
    bs, NB = 16, 12
    # (a) one key: out = v0, lse = scale * q.k0
    c = _decode_case(gen, [1], Hq, Hkv, bs, NB)
    out, lse = _run_decode(lib, c)
    for h in range(Hq):
        assert np.array_equal(out[0, h], _f64(c["seqs_v"][0][0, h]))
        s0 = float(np.dot(_f64(c["q"][0, h]), _f64(c["seqs_k"][0][0, h]))) * c["scale"]
        assert abs(lse[0, h] - s0) < 1e-12
    # (b) all keys equal: out = mean of V, lse = s + ln L
    L = 37
    c = _decode_case(gen, [L], Hq, Hkv, bs, NB)
    k0 = c["seqs_k"][0][0].clone()
    c["seqs_k"][0][:] = k0
    kc, vc, tables = _scatter_pool(c["seqs_k"], c["seqs_v"], Hkv, bs, NB, gen)
    c.update(kc=kc, vc=vc, tables=tables)
    out, lse = _run_decode(lib, c)
    for h in range(Hq):
        mean_v = _f64(c["seqs_v"][0][:, h]).mean(axis=0)
        assert np.max(np.abs(out[0, h] - mean_v)) < 1e-12
        s = float(np.dot(_f64(c["q"][0, h]), _f64(k0[h]))) * c["scale"]
        assert abs(lse[0, h] - (s + math.log(L))) < 1e-12
    # (c) one key scores ~100 above the others: out is that key's v
    c = _decode_case(gen, [20], Hq, Hkv, bs, NB)
    q = c["q"]
    for h in range(Hq):
        c["seqs_k"][0][:, h] = 0
        c["seqs_k"][0][7, h] = (q[0, h].to(torch.float32) * 100.0 / max(
            float((q[0, h].float() ** 2).sum()) * c["scale"], 1e-3)).to(torch.bfloat16)
    kc, vc, tables = _scatter_pool(c["seqs_k"], c["seqs_v"], Hkv, bs, NB, gen)
    c.update(kc=kc, vc=vc, tables=tables)
    out, _ = _run_decode(lib, c)
    for h in range(Hq):
        assert np.max(np.abs(out[0, h] - _f64(c["seqs_v"][0][7, h]))) < 1e-9


def pin_decode_permutation_invariance(lib):
    gen = torch.Generator().manual_seed(6)
    c = _decode_case(gen, [3, 50, 129], Hq=4, Hkv=2, bs=16, NB=30)
    out0, lse0 = _run_decode(lib, c)
    NB = c["kc"].shape[0]
    pi = torch.randperm(NB, generator=gen)
    kc = torch.empty_like(c["kc"])
    vc = torch.empty_like(c["vc"])
    kc[pi] = c["kc"]
    vc[pi] = c["vc"]
    tables = c["tables"].copy()
    used = tables >= 0
    tables[used] = pi.numpy()[tables[used]]
    c2 = dict(c, kc=kc, vc=vc, tables=tables)
    out1, lse1 = _run_decode(lib, c2, nthreads=3)
    assert np.array_equal(out0, out1) and np.array_equal(lse0, lse1)


def pin_decode_sharing_invariance(lib):
    """Sequences whose tables share the prefix blocks give the same bits as the
    same sequences with private copies of the prefix."""
    gen = torch.Generator().manual_seed(7)
    shared = 32
    c = _decode_case(gen, [40, 77, 33], Hq=4, Hkv=2, bs=16, NB=40, shared=shared)
    out_shared, lse_shared = _run_decode(lib, c)
    kc, vc, tables = _scatter_pool(c["seqs_k"], c["seqs_v"], 2, 16, 40, gen)
    assert len(np.unique(tables[tables >= 0])) == (tables >= 0).sum()
    out_priv, lse_priv = _run_decode(lib, dict(c, kc=kc, vc=vc, tables=tables))
    assert np.array_equal(out_shared, out_priv) and np.array_equal(lse_shared, lse_priv)
    # and the shared tables really do share blocks
    assert (c["tables"][:, :2] == c["tables"][0, :2]).all()


def pin_decode_gqa_equals_mha(lib):
    gen = torch.Generator().manual_seed(8)
    Hq, Hkv, bs, NB = 8, 2, 16, 20
    c = _decode_case(gen, [9, 45], Hq, Hkv, bs, NB)
    out_g, lse_g = _run_decode(lib, c)
    rk = [k.repeat_interleave(Hq // Hkv, dim=1) for k in c["seqs_k"]]
    rv = [v.repeat_interleave(Hq // Hkv, dim=1) for v in c["seqs_v"]]
    kc, vc, tables = _scatter_pool(rk, rv, Hq, bs, NB, gen)
    out_m, lse_m = _run_decode(lib, dict(c, kc=kc, vc=vc, tables=tables))
    assert np.array_equal(out_g, out_m) and np.array_equal(lse_g, lse_m)


def pin_decode_empty_context(lib):
    gen = torch.Generator().manual_seed(9)
    c = _decode_case(gen, [0, 5], Hq=2, Hkv=1, bs=16, NB=4)
    out, lse = _run_decode(lib, c)
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(lse[1]))


# --------------------------------------------------------------------------
# prefill


def _prefill_case(gen, prefix, new, Hq, Hkv, bs, NB):
    seqs_k, seqs_v = [], []
    for p, n in zip(prefix, new):
        seqs_k.append(_bf16((p + n, Hkv, D), gen))
        seqs_v.append(_bf16((p + n, Hkv, D), gen))
    kc, vc, tables = _scatter_pool(seqs_k, seqs_v, Hkv, bs, NB, gen)
    q = _bf16((sum(new), Hq, D), gen)
    cu_q = np.concatenate([[0], np.cumsum(new)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum([p + n for p, n in zip(prefix, new)])]).astype(np.int32)
    return dict(q=q, seqs_k=seqs_k, seqs_v=seqs_v, kc=kc, vc=vc, tables=tables,
                cu_q=cu_q, cu_k=cu_k, prefix=list(prefix), new=list(new),
                scale=D ** -0.5)


def _run_prefill(lib, c, nthreads=2):
    return O.prefill(_bits(c["q"]), _bits(c["kc"]), _bits(c["vc"]), c["tables"],
                     c["cu_q"], c["cu_k"], c["scale"], nthreads=nthreads, lib=lib)


def pin_prefill_bruteforce(lib):
    gen = torch.Generator().manual_seed(10)
    Hq, Hkv = 4, 2
    c = _prefill_case(gen, [0, 20, 35], [7, 13, 70], Hq, Hkv, bs=16, NB=20)
    out, lse = _run_prefill(lib, c)
    g = Hq // Hkv
    for i, (p, n) in enumerate(zip(c["prefix"], c["new"])):
        Lk = p + n
        rows = slice(c["cu_q"][i], c["cu_q"][i + 1])
        mask = np.arange(Lk)[None, :] <= (Lk - n + np.arange(n))[:, None]
        for h in range(Hq):
            K = _f64(c["seqs_k"][i][:, h // g])
            V = _f64(c["seqs_v"][i][:, h // g])
            o_ref, l_ref = dense_attention(_f64(c["q"][rows, h]), K, V, c["scale"], mask)
            assert np.max(np.abs(out[rows, h] - o_ref)) < 1e-12, (i, h)
            assert np.max(np.abs(lse[rows, h] - l_ref)) < 1e-12, (i, h)


def pin_prefill_sdpa_causal(lib):
    """No prefix: prefill equals torch's causal SDPA (float64)."""
    gen = torch.Generator().manual_seed(11)
    Hq, Hkv = 4, 4
    c = _prefill_case(gen, [0], [45], Hq, Hkv, bs=16, NB=6)
    out, _ = _run_prefill(lib, c)
    q = c["q"].to(torch.float64).permute(1, 0, 2)
    K = c["seqs_k"][0].to(torch.float64).permute(1, 0, 2)
    V = c["seqs_v"][0].to(torch.float64).permute(1, 0, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(q, K, V, is_causal=True,
                                                           scale=c["scale"])
    assert np.max(np.abs(out - ref.permute(1, 0, 2).numpy())) < 1e-12


def pin_prefill_causal_perturbation(lib):
    gen = torch.Generator().manual_seed(12)
    Hq, Hkv, bs, NB = 2, 1, 16, 10
    c = _prefill_case(gen, [24], [30], Hq, Hkv, bs, NB)
    out0, lse0 = _run_prefill(lib, c)
    Lk, n = 54, 30
    r = 11                       # row r sees keys 0 .. Lk-n+r = 35
    k2 = [c["seqs_k"][0].clone()]
    v2 = [c["seqs_v"][0].clone()]
    k2[0][Lk - n + r + 1:] = _bf16((n - r - 1, Hkv, D), gen) * 3
    v2[0][Lk - n + r + 1:] = _bf16((n - r - 1, Hkv, D), gen) * 3
    kc, vc, tables = _scatter_pool(k2, v2, Hkv, bs, NB, gen)
    out1, lse1 = _run_prefill(lib, dict(c, kc=kc, vc=vc, tables=tables))
    assert np.array_equal(out0[: r + 1], out1[: r + 1])
    assert np.array_equal(lse0[: r + 1], lse1[: r + 1])
    assert not np.array_equal(out0[r + 1:], out1[r + 1:])


def pin_prefill_one_row_equals_decode(lib):
    gen = torch.Generator().manual_seed(13)
    Hq, Hkv, bs, NB = 4, 2, 16, 16
    c = _prefill_case(gen, [30, 64], [1, 1], Hq, Hkv, bs, NB)
    out_p, lse_p = _run_prefill(lib, c)
    lens = np.array([31, 65], np.int32)
    out_d, lse_d = O.decode(_bits(c["q"]), _bits(c["kc"]), _bits(c["vc"]), c["tables"],
                            lens, c["scale"], lib=lib)
    assert np.array_equal(out_p, out_d) and np.array_equal(lse_p, lse_d)


def pin_prefill_chunk_invariance(lib):
    """Prefill of 96 tokens at once equals prefill of 64 then 32 over the pool."""
    gen = torch.Generator().manual_seed(14)
    Hq, Hkv, bs, NB = 4, 2, 16, 12
    c = _prefill_case(gen, [0], [96], Hq, Hkv, bs, NB)
    out_full, lse_full = _run_prefill(lib, c)
    qa, qb = c["q"][:64], c["q"][64:]
    ca = dict(c, q=qa, cu_q=np.array([0, 64], np.int32), cu_k=np.array([0, 64], np.int32))
    cb = dict(c, q=qb, cu_q=np.array([0, 32], np.int32), cu_k=np.array([0, 96], np.int32))
    out_a, lse_a = _run_prefill(lib, ca)
    out_b, lse_b = _run_prefill(lib, cb)
    assert np.array_equal(out_full[:64], out_a) and np.array_equal(out_full[64:], out_b)
    assert np.array_equal(lse_full[:64], lse_a) and np.array_equal(lse_full[64:], lse_b)


def pin_prefill_rejects_lk_lt_lq(lib):
    gen = torch.Generator().manual_seed(15)
    c = _prefill_case(gen, [0], [8], 2, 1, 16, 2)
    c["cu_k"] = np.array([0, 4], np.int32)
    try:
        _run_prefill(lib, c)
    except O.OracleError:
        return
    raise AssertionError("Lk < Lq was accepted")


# ---------------------------------------------------------------- FP8 (E4M3)

def _finite_codes(table):
    codes = np.array([c for c in range(256) if np.isfinite(table[c])], np.int64)
    return codes, table[codes]


def _nearest_code(v: float, codes, vals) -> int:
    """Brute force: the finite code nearest to v, ties to the even code; the
    search runs over magnitudes (codes 0x00..0x7E) and the sign of v is put back
    on the result (so -0 and tiny negatives give 0x80).  Past the largest finite
    magnitude the nearest finite value is that magnitude itself."""
    if math.isnan(v):
        return 0x7F
    a = abs(v)
    pos = codes < 0x80
    pc, pv = codes[pos], vals[pos]
    if a >= pv.max():
        c = int(pc[np.argmax(pv)])
    else:
        d = np.abs(pv - a)
        cand = pc[d == d.min()]
        c = int(cand[0]) if len(cand) == 1 else int([x for x in cand if x % 2 == 0][0])
    return c | 0x80 if math.copysign(1.0, v) < 0 else c


def pin_e4m3_table(lib):
    t = O.e4m3_table(lib=lib)
    # fixed anchors of the format: sign, bias 7, 3 mantissa bits, subnormals
    assert t[0x00] == 0.0 and t[0x01] == 2.0 ** -9 and t[0x07] == 7 * 2.0 ** -9
    assert t[0x08] == 2.0 ** -6 and t[0x38] == 1.0 and t[0x39] == 1.125
    assert t[0x7E] == 448.0 and math.isnan(t[0x7F]) and math.isnan(t[0xFF])
    assert t[0xB8] == -1.0 and t[0xFE] == -448.0 and math.copysign(1.0, t[0x80]) < 0
    assert np.all(np.diff(t[0x00:0x7F]) > 0)           # increasing over the positive codes
    # every code against torch's float8_e4m3fn decoding
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(np.isnan(ref), np.isnan(t))
    fin = ~np.isnan(ref)
    assert np.array_equal(ref[fin], t[fin])


def pin_e4m3_quantizer(lib):
    t = O.e4m3_table(lib=lib)
    codes, vals = _finite_codes(t)
    pos = np.sort(vals[vals > 0])
    mids = (pos[:-1] + pos[1:]) / 2                          # exact ties
    # the largest bf16 values overflow the binary32 product at scale 2^-5, and
    # infinity saturates like any magnitude past 448
    xs = [0.0, -0.0, 2.0 ** -10, 3 * 2.0 ** -10, 2.0 ** -9, 448.0, 460.0, 464.0, 470.0,
          480.0, 1e4, 1e30, 3.3e38, math.inf]
    xs += list(pos) + list(mids) + list(mids * (1 + 2.0 ** -7)) + list(mids * (1 - 2.0 ** -7))
    gen = torch.Generator().manual_seed(81)
    xs += list((torch.randn(2000, generator=gen) * 40).tolist())
    xs += list((torch.randn(500, generator=gen) * 0.01).tolist())
    x = torch.tensor(xs + [-v for v in xs], dtype=torch.float64).to(torch.bfloat16)
    for scale in (1.0, 0.75, 3.0, 2.0 ** -5):
        got = O.quantize_e4m3(_bits(x), scale, lib=lib)
        inv = np.float32(1.0) / np.float32(scale)
        with np.errstate(over="ignore"):                       # binary32 product
            v = (x.float().numpy() * inv).astype(np.float32)
        want = np.array([_nearest_code(float(a), codes, vals) for a in v], np.uint8)
        assert np.array_equal(got, want), f"scale {scale}"
        # torch's conversion agrees wherever no saturation is involved
        inr = np.abs(v) <= 448.0
        tc = torch.from_numpy(v[inr]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(tc, got[inr]), f"torch scale {scale}"


def pin_store_fp8(lib):
    gen = torch.Generator().manual_seed(82)
    NB, bs, Hkv = 3, 256, 2
    T = 5
    k = _bf16((T, Hkv, D), gen, 30.0)
    v = _bf16((T, Hkv, D), gen, 0.2)
    kc = np.zeros((NB, bs, Hkv, D), np.uint8)
    vc = np.zeros((NB, bs, Hkv, D), np.uint8)
    slots = np.array([0, 255, 256, -1, 3 * 256 - 1], np.int32)
    O.store_fp8(_bits(k), _bits(v), kc, vc, slots, 0.5, 0.01, lib=lib)
    kq = O.quantize_e4m3(_bits(k), 0.5, lib=lib)
    vq = O.quantize_e4m3(_bits(v), 0.01, lib=lib)
    flat_k, flat_v = kc.reshape(NB * bs, Hkv, D), vc.reshape(NB * bs, Hkv, D)
    for t, s_ in enumerate(slots):
        if s_ < 0:
            continue
        assert np.array_equal(flat_k[s_], kq[t]) and np.array_equal(flat_v[s_], vq[t])
    written = {int(s_) for s_ in slots if s_ >= 0}
    for s_ in range(NB * bs):
        if s_ not in written:
            assert not flat_k[s_].any() and not flat_v[s_].any()
    bad = np.array([0, 3 * 256], np.int32)
    try:
        O.store_fp8(_bits(k[:2]), _bits(v[:2]), kc, vc, bad, 1.0, 1.0, lib=lib)
        raise AssertionError("out-of-range slot accepted")
    except O.OracleError:
        pass


def pin_decode_fp8_equals_bf16(lib):
    # a pool of random codes; its values times power-of-two scales are exact in
    # bf16, so the bf16 decode of that pool must give the same doubles
    t = O.e4m3_table(lib=lib)
    gen = torch.Generator().manual_seed(83)
    NB, bs, Hkv, Hq = 4, 256, 2, 4
    kc = torch.randint(0, 256, (NB, bs, Hkv, D), generator=gen, dtype=torch.int64).numpy()
    vc = torch.randint(0, 256, (NB, bs, Hkv, D), generator=gen, dtype=torch.int64).numpy()
    for c in (kc, vc):
        c[(c & 0x7F) == 0x7F] = 0x3A                        # no NaN codes
    kc, vc = kc.astype(np.uint8), vc.astype(np.uint8)
    ks, vs = 0.25, 2.0
    kb = torch.from_numpy(t[kc] * ks).to(torch.bfloat16)
    vb = torch.from_numpy(t[vc] * vs).to(torch.bfloat16)
    assert np.array_equal(kb.double().numpy(), t[kc] * ks)   # exact
    q = _bf16((3, Hq, D), gen, 0.05)
    tables = np.array([[2, 0, -1, -1], [1, 3, 0, 2], [3, -1, -1, -1]], np.int32)
    lens = np.array([300, 1000, 17], np.int32)
    o8, l8 = O.decode_fp8(_bits(q), kc, vc, tables, lens, D ** -0.5, ks, vs, lib=lib)
    ob, lb = O.decode(_bits(q), _bits(kb), _bits(vb), tables, lens, D ** -0.5, lib=lib)
    assert np.array_equal(o8, ob) and np.array_equal(l8, lb)


ALL_PINS = [
    pin_store_roundtrip,
    pin_store_rejects,
    pin_copy_blocks,
    pin_decode_bruteforce,
    pin_decode_sdpa,
    pin_decode_closed_forms,
    pin_decode_permutation_invariance,
    pin_decode_sharing_invariance,
    pin_decode_gqa_equals_mha,
    pin_decode_empty_context,
    pin_prefill_bruteforce,
    pin_prefill_sdpa_causal,
    pin_prefill_causal_perturbation,
    pin_prefill_one_row_equals_decode,
    pin_prefill_chunk_invariance,
    pin_prefill_rejects_lk_lt_lq,
    pin_e4m3_table,
    pin_e4m3_quantizer,
    pin_store_fp8,
    pin_decode_fp8_equals_bf16,
]
