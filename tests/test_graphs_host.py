"""Host side of the CUDA-graph decode runner, no GPU: the configuration layout
the binding builds matches the library's, the default bucket set is the
pages' list (1, 2, 4, ..., 512, read as powers of two: "Nano-vLLM System
Architecture Analysis", comparison table, "Variable-batch CUDA Graphs"), and
the bucket a batch runs in is the smallest that holds it, checked against
brute force."""
import ctypes

import numpy as np
import pytest

from paged_kv_cache_214_gb300 import build as B
from paged_kv_cache_214_gb300 import graphs, pkv


@pytest.fixture(scope="module", autouse=True)
def lib():
    B.build()
    return graphs._lib()


def test_config_layout_matches_the_library(lib):
    assert lib.pkv_decode_graphs_config_bytes() == ctypes.sizeof(graphs._Config)


def test_default_buckets():
    assert graphs.default_buckets(1) == [1]
    assert graphs.default_buckets(5) == [1, 2, 4]
    full = [1, 2, 4, 8, 16, 32, 64, 128, 256, 512]
    assert graphs.default_buckets(512) == full
    assert graphs.default_buckets(100000) == full
    with pytest.raises(pkv.PkvError):
        graphs.default_buckets(0)


def test_pick_bucket_edges():
    b = [1, 2, 4, 8]
    assert [graphs.pick_bucket(b, n) for n in range(0, 10)] == [0, 1, 2, 4, 4, 8, 8, 8, 8, 0]
    assert graphs.pick_bucket([3, 5], 1) == 3
    for bad_list in ([], [0, 1], [2, 2], [4, 3]):
        with pytest.raises(pkv.PkvError):
            graphs.pick_bucket(bad_list, 1)
    with pytest.raises(pkv.PkvError):
        graphs.pick_bucket(b, -1)


def test_pick_bucket_brute_force():
    g = np.random.default_rng(5)
    for _ in range(200):
        sizes = sorted(set(int(x) for x in g.integers(1, 600, size=g.integers(1, 12))))
        for n in list(g.integers(0, 700, size=20)) + [sizes[0], sizes[-1], sizes[-1] + 1]:
            want = min((s for s in sizes if s >= n), default=0) if n > 0 else 0
            assert graphs.pick_bucket(sizes, int(n)) == want
