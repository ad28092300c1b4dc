"""Host block manager (include/pkv_blocks.h): free list, prefix-cache hits,
reference counts, fork + copy-on-write.  No GPU needed."""
import numpy as np
import pytest

from paged_kv_cache_214_gb300 import build as B
from paged_kv_cache_214_gb300.blocks import BlockManager, BlockManagerError, BM_ERR_NO_BLOCKS

BS = 4   # small blocks keep the cases readable; the logic is size independent


@pytest.fixture(scope="module", autouse=True)
def _lib():
    B.build()


def check_invariants(bm, seqs):
    """Reference counts equal the number of live sequences holding a block; free
    blocks are exactly those with count 0."""
    counts = np.zeros(bm.num_blocks, np.int64)
    for s in seqs:
        n = bm.num_blocks_of(s)
        t = bm.block_table(s, n)
        assert len(set(t.tolist())) == n          # no block twice in one table
        counts[t] += 1
    for b in range(bm.num_blocks):
        assert bm.ref_count(b) == counts[b], b
    assert bm.num_free_blocks == int((counts == 0).sum())


def test_fresh_allocation_and_slots():
    bm = BlockManager(10, BS)
    assert bm.add_sequence(1, list(range(10))) == 0     # 2 full blocks + partial
    assert bm.num_blocks_of(1) == 3 and bm.num_free_blocks == 7
    t = bm.block_table(1, 5)
    assert (t[3:] == -1).all()
    slots = bm.slot_mapping(1, 0, 10)
    assert slots.tolist() == [t[p // BS] * BS + p % BS for p in range(10)]
    s, copy = bm.append_token(1, 99)
    assert copy is None and s == t[2] * BS + 2
    s, _ = bm.append_token(1, 100)                       # fills block 2
    s, _ = bm.append_token(1, 101)                       # opens a 4th block
    assert bm.num_blocks_of(1) == 4 and s == bm.block_table(1, 4)[3] * BS
    check_invariants(bm, [1])


def test_prefix_cache_hit_shares_blocks():
    bm = BlockManager(12, BS)
    prompt = [7, 7, 1, 2, 3, 4, 5, 6, 9]
    bm.add_sequence(1, prompt)
    cached = bm.add_sequence(2, prompt[:8] + [42, 43])   # same first two blocks
    assert cached == 8
    t1, t2 = bm.block_table(1, 3), bm.block_table(2, 3)
    assert (t1[:2] == t2[:2]).all() and t1[2] != t2[2]
    assert bm.ref_count(t1[0]) == 2
    # a different first block: no sharing at all, even if later blocks match
    cached = bm.add_sequence(3, [0, 0, 0, 0] + prompt[4:8])
    assert cached == 0
    check_invariants(bm, [1, 2, 3])


def test_freed_blocks_keep_their_content_for_later_hits():
    bm = BlockManager(8, BS)
    bm.add_sequence(1, list(range(8)))
    t = bm.block_table(1, 2)
    bm.free_sequence(1)
    assert bm.num_free_blocks == 8
    assert bm.add_sequence(2, list(range(8)) + [9]) == 8   # cached, though freed
    assert (bm.block_table(2, 3)[:2] == t).all()
    check_invariants(bm, [2])


def test_eviction_of_a_cached_free_block():
    bm = BlockManager(3, BS)
    bm.add_sequence(1, [1, 2, 3, 4])
    bm.free_sequence(1)
    bm.add_sequence(2, [5] * 12)        # takes all three blocks, evicting the cache
    bm.free_sequence(2)
    assert bm.add_sequence(3, [1, 2, 3, 4]) == 0
    check_invariants(bm, [3])


def test_blocks_filled_by_decode_become_cacheable():
    bm = BlockManager(8, BS)
    bm.add_sequence(1, [1, 2])
    for tok in (3, 4, 5):
        bm.append_token(1, tok)
    assert bm.add_sequence(2, [1, 2, 3, 4, 8]) == 4
    check_invariants(bm, [1, 2])


def test_out_of_blocks_is_all_or_nothing():
    bm = BlockManager(3, BS)
    bm.add_sequence(1, list(range(8)))
    with pytest.raises(BlockManagerError) as e:
        bm.add_sequence(2, list(range(100, 109)))     # needs 3, 1 free
    assert e.value.status == BM_ERR_NO_BLOCKS
    assert bm.num_free_blocks == 1
    check_invariants(bm, [1])
    bm.add_sequence(3, [5])
    with pytest.raises(BlockManagerError):
        for t in range(10):
            bm.append_token(3, t)
    check_invariants(bm, [1, 3])


def test_fork_and_copy_on_write():
    bm = BlockManager(10, BS)
    bm.add_sequence(1, [1, 2, 3, 4, 5, 6])            # block A full, block B partial
    bm.fork(1, 2)
    tA, tB = bm.block_table(1, 2)
    assert bm.ref_count(tA) == 2 and bm.ref_count(tB) == 2
    slot, copy = bm.append_token(2, 7)                # shared partial block: CoW
    assert copy is not None and copy[0] == tB
    new_b = copy[1]
    assert slot == new_b * BS + 2
    assert bm.block_table(2, 2).tolist() == [tA, new_b]
    assert bm.ref_count(tB) == 1 and bm.ref_count(tA) == 2
    slot, copy = bm.append_token(1, 8)                # parent now owns B alone
    assert copy is None and slot == tB * BS + 2
    check_invariants(bm, [1, 2])
    bm.free_sequence(1)
    bm.free_sequence(2)
    assert bm.num_free_blocks == 10


def test_random_operations_keep_invariants():
    rng = np.random.RandomState(0)
    bm = BlockManager(64, BS)
    live, next_id = [], 0
    vocab = [list(rng.randint(0, 3, size=12)) for _ in range(4)]   # shared prompt stems
    for _ in range(600):
        op = rng.randint(4)
        try:
            if op == 0 or not live:
                stem = vocab[rng.randint(4)]
                bm.add_sequence(next_id, stem[:rng.randint(1, 12)] + list(rng.randint(0, 3, size=rng.randint(0, 6))))
                live.append(next_id)
                next_id += 1
            elif op == 1:
                bm.append_token(live[rng.randint(len(live))], int(rng.randint(3)))
            elif op == 2:
                bm.fork(live[rng.randint(len(live))], next_id)
                live.append(next_id)
                next_id += 1
            else:
                bm.free_sequence(live.pop(rng.randint(len(live))))
        except BlockManagerError as e:
            assert e.status == BM_ERR_NO_BLOCKS
        check_invariants(bm, live)
