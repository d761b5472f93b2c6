"""Host-side figures the benchmark reports, pinned on CPU: the logical
Vertical-Slash edge count of eq.(5) (closed form in bench.py) against the
oracle's per-row logical sets, and the page's printed vertical count."""
import numpy as np
import pytest

import bench
import oracle


@pytest.mark.parametrize("seed", range(6))
def test_logical_edges_match_the_oracle_sets(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 300))
    C = rng.choice(n, size=int(rng.integers(0, min(n, 40) + 1)), replace=False)
    D = rng.choice(n, size=int(rng.integers(0, min(n, 60) + 1)), replace=False)
    want = sum(len(oracle.vs_logical_set(i, C, D)) for i in range(n))
    assert bench.logical_edges(n, C, D) == want


def test_logical_edges_page_example():
    # n = 1024, verticals {0, 512}, no slashes: 1024 + 512 attended (row, key) pairs
    assert bench.logical_edges(1024, [0, 512], []) == 1536
    # a single slash at offset 0 is the diagonal: n pairs; with column 0 the pair (0, 0) is shared
    assert bench.logical_edges(10, [0], [0]) == 10 + 10 - 1
