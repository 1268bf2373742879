"""The C oracle against the separately written brute force on random tiny caches."""
import numpy as np
import pytest

import oracle
from tests.csm_bruteforce import csm_round_bruteforce


@pytest.mark.parametrize("seed", range(40))
def test_random_round_matches_bruteforce(seed):
    rng = np.random.default_rng(1000 + seed)
    c = int(rng.choice([2, 4, 6, 8, 12, 16]))
    d = int(rng.integers(1, 9))
    n1 = int(rng.integers(0, 4))
    n2 = int(rng.integers(0, 5))
    s = int(rng.integers(0, n1 + n2 + 4 * c + c))
    m = int(rng.integers(0, c // 2 + 1))
    cap = s + int(rng.integers(0, 5))
    K = rng.standard_normal((1, max(cap, 1), d))
    V = rng.standard_normal((1, max(cap, 1), d))
    N = rng.integers(1, 6, (1, max(cap, 1))).astype(np.int32)
    out = oracle.csm_round(K, V, N, [s], n1, n2, c, m)
    Kb, Vb, Nb, sb, mb = csm_round_bruteforce(K[0], V[0], N[0], s, n1, n2, c, m)
    L = int(out["len"][0])
    assert L == sb
    if L:
        np.testing.assert_allclose(out["K"][0, :L], Kb, rtol=0, atol=1e-12)
        np.testing.assert_allclose(out["V"][0, :L], Vb, rtol=0, atol=1e-12)
    assert out["N"][0, :L].tolist() == Nb
    for j, row in enumerate(mb):
        assert out["match"][0, j].tolist() == row


def test_several_rounds_and_units_match_bruteforce():
    rng = np.random.default_rng(7)
    BH, cap, d, n1, n2, c = 3, 80, 3, 2, 5, 8
    K = rng.standard_normal((BH, cap, d))
    V = rng.standard_normal((BH, cap, d))
    N = np.ones((BH, cap), np.int32)
    L = np.array([80, 47, 13], np.int32)
    ref = [(K[u].copy(), V[u].copy(), N[u].tolist(), int(L[u])) for u in range(BH)]
    for m in (4, 3, 2, 4):
        out = oracle.csm_round(K, V, N, L, n1, n2, c, m)
        K, V, N, L = out["K"], out["V"], out["N"], out["len"]
        for u in range(BH):
            kb, vb, nb, sb, _ = csm_round_bruteforce(*ref[u][:3], ref[u][3], n1, n2, c, m)
            ref[u] = (kb, vb, nb, sb)
            assert int(L[u]) == sb
            np.testing.assert_allclose(K[u, :sb], kb, rtol=0, atol=1e-11)
            np.testing.assert_allclose(V[u, :sb], vb, rtol=0, atol=1e-11)
            assert N[u, :sb].tolist() == nb
