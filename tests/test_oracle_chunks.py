"""Pins of oracle.csm_chunks, the chunk-list entry point that the full-size GPU
checks use ([Chelsea §三 分块软匹配算法 steps 2-4]): it must do to every chunk of
its list exactly what one CSM round does to that chunk inside a cache.

* Against the separately written brute force: a chunk on its own is a cache
  with no sinks, no recent window and one full chunk, so csm_chunks' rows,
  degrees and matches equal the brute force's round of that cache.
* Against oracle.csm_round on chunks cut from caches: per chunk (unit u, chunk
  j) the output rows at n1 + j (c - m), the match row, the source offsets
  (origin - n1 - j c) and the merged flags agree, and so do the per-A best
  similarities, argmax margins and the top-m cut.
A strided indexing or marshalling mistake in csm_chunks (a wrong chunk, a
transposed d/c stride, records shifted by one chunk) fails one of these.
"""
import numpy as np
import pytest

import oracle
from tests.csm_bruteforce import csm_round_bruteforce


@pytest.mark.parametrize("seed", range(12))
def test_each_chunk_matches_the_bruteforce(seed):
    rng = np.random.default_rng(500 + seed)
    c = int(rng.choice([2, 4, 8, 12, 16]))
    d = int(rng.integers(1, 7))
    m = int(rng.integers(0, c // 2 + 1))
    n = int(rng.integers(1, 6))
    Kc = rng.standard_normal((n, c, d))
    Vc = rng.standard_normal((n, c, d))
    Nc = rng.integers(1, 7, (n, c)).astype(np.int32)
    if seed % 3 == 0:  # exact ties: duplicated keys and a zero key
        Kc[0, 1::2] = Kc[0, 1]
        Kc[-1, 0] = 0.0
    out = oracle.csm_chunks(Kc, Vc, Nc, m)
    for i in range(n):
        kb, vb, nb, sb, mb = csm_round_bruteforce(Kc[i], Vc[i], Nc[i], c, 0, 0, c, m)
        assert sb == c - m
        np.testing.assert_allclose(out["K"][i], kb, rtol=0, atol=1e-12)
        np.testing.assert_allclose(out["V"][i], vb, rtol=0, atol=1e-12)
        assert out["N"][i].tolist() == nb
        if m:
            assert out["match"][i].tolist() == mb[0]
        assert int(out["N"][i].sum()) == int(Nc[i].sum())


@pytest.mark.parametrize("c,m,d", [(16, 8, 5), (16, 5, 3), (8, 2, 4), (64, 32, 8), (64, 27, 16)])
def test_chunks_cut_from_caches_match_the_round(c, m, d):
    rng = np.random.default_rng(c * 100 + m)
    BH, n1, n2 = 3, 3, 5
    cap = n1 + n2 + 6 * c + 7
    K = np.zeros((BH, cap, d))
    z = rng.standard_normal((BH, d))
    for t in range(cap):  # correlated keys, so similarities are close and ranks matter
        z = 0.9 * z + np.sqrt(0.19) * rng.standard_normal((BH, d))
        K[:, t] = z
    V = rng.standard_normal((BH, cap, d))
    N = rng.integers(1, 5, (BH, cap)).astype(np.int32)
    L = np.array([cap, n1 + n2 + 3 * c + 2, n1 + n2 + c], np.int32)
    rd = oracle.csm_round(K, V, N, L, n1, n2, c, m)
    picks = [(u, j) for u in range(BH) for j in range(oracle.num_chunks(int(L[u]), n1, n2, c))]
    rng.shuffle(picks)  # list order must not matter
    sl = lambda a, u, j: a[u, n1 + j * c:n1 + (j + 1) * c]  # noqa: E731
    ch = oracle.csm_chunks(np.stack([sl(K, u, j) for u, j in picks]), np.stack([sl(V, u, j) for u, j in picks]),
                           np.stack([sl(N, u, j) for u, j in picks]), m)
    for i, (u, j) in enumerate(picks):
        o0, o1 = n1 + j * (c - m), n1 + (j + 1) * (c - m)
        np.testing.assert_array_equal(ch["K"][i], rd["K"][u, o0:o1])
        np.testing.assert_array_equal(ch["V"][i], rd["V"][u, o0:o1])
        np.testing.assert_array_equal(ch["N"][i], rd["N"][u, o0:o1])
        np.testing.assert_array_equal(ch["match"][i], rd["match"][u, j])
        np.testing.assert_array_equal(ch["origin"][i] + n1 + j * c, rd["origin"][u, o0:o1])
        np.testing.assert_array_equal(ch["merged"][i], rd["merged"][u, o0:o1])
        np.testing.assert_array_equal(ch["sim"][i], rd["sim"][u, j])
        np.testing.assert_array_equal(ch["margin"][i], rd["margin"][u, j])
        assert ch["cut"][i] == rd["cut"][u, j]


def test_forced_decisions_are_replayed_as_given():
    rng = np.random.default_rng(9)
    c, m, d, n = 16, 6, 4, 5
    Kc = rng.standard_normal((n, c, d))
    Vc = rng.standard_normal((n, c, d))
    Nc = rng.integers(1, 4, (n, c)).astype(np.int32)
    free = oracle.csm_chunks(Kc, Vc, Nc, m)
    forced = free["match"].copy()
    # a different but valid plan: chunk 2's first selected A row moves to B 0
    a = int(np.nonzero(forced[2] >= 0)[0][0])
    forced[2, a] = 0 if forced[2, a] != 0 else 1
    rep = oracle.csm_chunks(Kc, Vc, Nc, m, forced=forced)
    np.testing.assert_array_equal(rep["match"], forced)
    for i in (0, 1, 3, 4):
        np.testing.assert_array_equal(rep["K"][i], free["K"][i])
    b = int(forced[2, a])
    members = [2 * b + 1] + [2 * x for x in np.nonzero(forced[2] == b)[0]]
    w = Nc[2, members].astype(float)
    want = (w[:, None] * Kc[2, members]).sum(0) / w.sum()
    row = int(np.nonzero(rep["origin"][2] == 2 * b + 1)[0][0])
    np.testing.assert_allclose(rep["K"][2, row], want, rtol=0, atol=1e-12)
    assert int(rep["N"][2, row]) == int(w.sum())
