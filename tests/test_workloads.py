"""Properties of the seeded synthetic workloads (no GPU)."""
import numpy as np
import torch

import oracle
from paged_kv_cache_214_gb300 import workloads as W


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def test_tiny_decode_shapes_and_tables():
    w = W.config_workload(1)
    assert (w.B, w.Hq, w.Hkv, w.D, w.block_size, w.num_blocks) == (4, 16, 8, 128, 256, 16)
    assert w.context_lens.tolist() == [17, 256, 300, 513]
    used = w.block_tables[w.block_tables >= 0]
    assert len(used) == 7 and len(set(used.tolist())) == 7      # no sharing in workload 1
    # new-token slots: position ctx-1, i.e. offsets 16, 255, 43 and 0 (block 2 of seq 3)
    offs = (w.slot_mapping % 256).tolist()
    assert offs == [16, 255, 43, 0]
    assert int(w.slot_mapping[3]) // 256 == int(w.block_tables[3, 2])


def test_store_then_gather_puts_new_token_last():
    """Slots from the generator land at logical position ctx-1 (oracle round trip)."""
    w = W.config_workload(1)
    kc, vc = _bits(w.k_cache).copy(), _bits(w.v_cache).copy()
    oracle.store(_bits(w.k_new), _bits(w.v_new), kc, vc, w.slot_mapping.numpy())
    for b in range(w.B):
        L = int(w.context_lens[b])
        K, V = oracle.gather(kc, vc, w.block_tables[b].numpy(), L)
        assert np.array_equal(K[L - 1], _bits(w.k_new[b]))
        assert np.array_equal(V[L - 1], _bits(w.v_new[b]))


def test_shared_prefix_tables():
    w = W.make_decode([600, 700, 513], 4, 2, 32, 1, shared_prefix_tokens=512)
    t = w.block_tables
    assert (t[:, :2] == t[0, :2]).all()
    private = t[:, 2:][t[:, 2:] >= 0].tolist()
    assert len(private) == len(set(private)) and not set(private) & set(t[0, :2].tolist())
    assert w.unique_kv_tokens == 600 + 700 + 513 - 2 * 512
    # the new token never goes into a shared block
    assert all(int(s) // 256 not in t[0, :2].tolist() for s in w.slot_mapping)


def test_rotations_are_disjoint():
    w = W.make_decode([300, 1000], 4, 2, 64, 3, rotations=3)
    sets = [set(x[x >= 0].tolist()) for x in [w.block_tables] + w.extra_tables]
    assert all(not (a & b) for i, a in enumerate(sets) for b in sets[i + 1:])


def test_prefill_layout():
    w = W.make_prefill([256, 0], [100, 20], 4, 2, 16, 5)
    assert w.cu_seqlens_q.tolist() == [0, 100, 120]
    assert w.cu_seqlens_k.tolist() == [0, 356, 376]
    assert w.q.shape == (120, 4, 128) and w.slot_mapping.shape == (120,)
    kc, vc = _bits(w.k_cache).copy(), _bits(w.v_cache).copy()
    oracle.store(_bits(w.k_new), _bits(w.v_new), kc, vc, w.slot_mapping.numpy())
    K, _ = oracle.gather(kc, vc, w.block_tables[0].numpy(), 356)
    assert np.array_equal(K[256:], _bits(w.k_new[:100]))


def test_seeded_determinism():
    a = W.config_workload(1)
    b = W.config_workload(1)
    assert torch.equal(a.q, b.q) and torch.equal(a.block_tables, b.block_tables)
    assert torch.equal(a.k_cache, b.k_cache)
