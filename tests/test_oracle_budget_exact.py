"""Budget-exact compression (merge only the oldest chunks needed to reach the budget)
in the oracle: pinned by the separately written brute force, by what a round must
leave untouched, and by the schedule it produces on the 16K layer (derived by hand
from B = R(n + Gamma), the trigger s >= B + g and k = ceil((s - B) / m))."""
import numpy as np
import pytest

import oracle
from oracle import schedule as S
from tests.csm_bruteforce import csm_round_bruteforce


@pytest.mark.parametrize("seed", range(24))
def test_limited_round_matches_bruteforce(seed):
    rng = np.random.default_rng(500 + seed)
    c = int(rng.choice([4, 8, 16]))
    d = int(rng.integers(1, 6))
    n1, n2 = int(rng.integers(0, 4)), int(rng.integers(0, 6))
    s = n1 + n2 + int(rng.integers(0, 7)) * c + int(rng.integers(0, c))
    m = int(rng.integers(1, c // 2 + 1))
    limit = int(rng.integers(-1, 8))
    K = rng.standard_normal((1, s + 3, d))
    V = rng.standard_normal((1, s + 3, d))
    N = rng.integers(1, 5, (1, s + 3)).astype(np.int32)
    out = oracle.csm_round(K, V, N, [s], n1, n2, c, m, limits=[limit])
    Kb, Vb, Nb, sb, _ = csm_round_bruteforce(K[0], V[0], N[0], s, n1, n2, c, m, limit=max(limit, 0))
    L = int(out["len"][0])
    assert L == sb
    np.testing.assert_allclose(out["K"][0, :L], Kb, rtol=0, atol=1e-12)
    np.testing.assert_allclose(out["V"][0, :L], Vb, rtol=0, atol=1e-12)
    assert out["N"][0, :L].tolist() == Nb


def test_limited_round_is_a_prefix_of_the_full_round_and_moves_the_rest():
    rng = np.random.default_rng(3)
    n1, n2, c, m, d = 4, 9, 16, 8, 5
    s = n1 + n2 + 6 * c + 11
    K = np.cumsum(rng.standard_normal((1, s, d)), axis=1)  # correlated keys: real merges
    V = rng.standard_normal((1, s, d))
    N = rng.integers(1, 4, (1, s)).astype(np.int32)
    full = oracle.csm_round(K, V, N, [s], n1, n2, c, m)
    for k in (1, 2, 5):
        lim = oracle.csm_round(K, V, N, [s], n1, n2, c, m, limits=[k])
        head = n1 + k * (c - m)
        assert int(lim["len"][0]) == s - k * m
        # the oldest k chunks come out exactly as in the full round ...
        assert np.array_equal(lim["K"][0, :head], full["K"][0, :head])
        assert np.array_equal(lim["V"][0, :head], full["V"][0, :head])
        assert np.array_equal(lim["N"][0, :head], full["N"][0, :head])
        # ... and everything after them (unprocessed chunks, remainder, recent) moves down unchanged
        rest = s - (n1 + k * c)
        assert np.array_equal(lim["K"][0, head:head + rest], K[0, n1 + k * c:s])
        assert np.array_equal(lim["N"][0, head:head + rest], N[0, n1 + k * c:s])
        assert int(lim["N"][0, :s - k * m].sum()) == int(N.sum())
    for k in (0, -3, 6, 40):  # no limit, or one at least the full chunk count
        same = oracle.csm_round(K, V, N, [s], n1, n2, c, m, limits=[k])
        assert np.array_equal(same["K"], full["K"]) and np.array_equal(same["len"], full["len"])


def test_budget_exact_schedule_of_the_16k_layer():
    # B = 0.2 * (16384 + 1000) = 3476.8, trigger s >= 3540.8, m = 128 (r = 0.5, c = 256).
    # 16384: ceil(12907.2 / 128) = 101 > 63 full chunks -> 63, s = 8320.
    # 8321: ceil(4844.2 / 128) = 38 > 32 -> 32, s = 4225.  4226: ceil(749.2 / 128) = 6 -> 3458.
    # Then s reaches 3541 after 83 appends (step 85): ceil(64.2 / 128) = 1 -> 3413, and again
    # every 128 steps (213, 341, ..., 981): the "every g steps" regime, with period m.
    got = S.plan_budget_exact(16384, 0.2, 1000, 64, 16, 64, 256, 0.5)
    want = [(0, 16384, 63, 8320), (1, 8321, 32, 4225), (2, 4226, 6, 3458)]
    want += [(85 + 128 * i, 3541, 1, 3413) for i in range(8)]
    assert [(st, s, k, s2) for st, s, r, m, k, s2 in got] == want
    # once a round is not capped by the chunks there are, it ends just under the budget
    assert all(s2 <= 3476.8 for _, _, _, _, _, s2 in got[2:])
    # the unlimited schedule compresses far below the budget instead
    assert [x[-1] for x in S.plan(16384, 0.2, 1000, 64, 16, 64, 256, 0.5)] == [8320, 4225, 2178]


def test_chunks_to_budget_edges():
    assert S.chunks_to_budget(3476, 3476.8, 16, 64, 256, 128) == 0      # already under B
    assert S.chunks_to_budget(3477, 3476.8, 16, 64, 256, 128) == 1      # any excess needs a chunk
    assert S.chunks_to_budget(3477, 3476.8, 16, 64, 256, 0) == 0        # nothing can merge
    assert S.chunks_to_budget(300, 0.0, 16, 64, 256, 128) == 0          # no full chunk
    assert S.chunks_to_budget(3604 + 128, 3476.0, 16, 64, 256, 128) == 2
