"""The end-to-end leg's grouping (bench.e2e_groups): every (row, KV head) cache is
uploaded by exactly one group and downloaded exactly once at its own final length,
into disjoint contiguous stretches of the host buffers."""
import numpy as np
import pytest

import bench


@pytest.mark.parametrize("batch,h_kv,want,outlier", [
    (4, 8, 8, 7),     # 32K x 4: fewer rows than groups, one outlier head per row
    (16, 4, 32, None),
    (32, 8, 32, None),
    (1, 8, 8, None),
    (1, 2, 8, 0),
    (3, 5, 2, 2),     # more rows than groups
    (7, 3, 1, None),
])
def test_every_cache_once_at_its_length(batch, h_kv, want, outlier):
    rng = np.random.default_rng(batch * 100 + h_kv)
    comp = rng.integers(1, 3000, size=batch)
    fin = np.array([[5000 if h == outlier else comp[b] for h in range(h_kv)] for b in range(batch)], np.int64)
    bounds, runs, total = bench.e2e_groups(batch, h_kv, fin, want)
    # groups cover every cache once
    seen = np.zeros((batch, h_kv), int)
    for b0, b1, h0, h1 in bounds:
        assert 0 <= b0 < b1 <= batch and 0 <= h0 < h1 <= h_kv
        assert b1 - b0 == 1 or (h0, h1) == (0, h_kv)  # a head range only within one row
        seen[b0:b1, h0:h1] += 1
    assert (seen == 1).all()
    if batch < want:
        assert len(bounds) == batch * min(h_kv, -(-want // batch))
    else:
        assert len(bounds) == want
    # runs: every unit once, at its length, inside its own group, in disjoint stretches
    got = {}
    stretches = []
    for g, u0, u1, L, off in runs:
        b0, b1, h0, h1 = bounds[g]
        for u in range(u0, u1):
            b, h = divmod(u, h_kv)
            assert b0 <= b < b1 and h0 <= h < h1
            assert u not in got
            got[u] = L
            assert L == fin[b, h]
        assert u1 > u0 and u0 // h_kv == (u1 - 1) // h_kv  # a run stays within one row
        stretches.append((off, off + (u1 - u0) * L))
    assert sorted(got) == list(range(batch * h_kv))
    stretches.sort()
    assert stretches[0][0] == 0 and stretches[-1][1] == total
    for (a0, a1), (c0, c1) in zip(stretches, stretches[1:]):
        assert a1 == c0  # contiguous, no overlap
    assert total == int(fin.sum())
