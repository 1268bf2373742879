"""The oracle against hand-worked CSM rounds (tests/golden/csm_hand_cases.json)."""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "csm_hand_cases.json")
CASES = json.load(open(GOLDEN))["cases"]


def as_float(x):
    return float(Fraction(x)) if isinstance(x, str) else float(x)


def arr(rows):
    return np.array([[as_float(v) for v in r] for r in rows])


@pytest.mark.parametrize("case", CASES, ids=[c["name"] for c in CASES])
def test_hand_case(case):
    K = arr(case["K"])
    s, d = K.shape
    V = np.stack([np.arange(s, dtype=float), -np.arange(s, dtype=float)], axis=1)
    N = np.array(case["N"], np.int32)
    assert oracle.edges_per_chunk(case["r"], case["c"]) == case["m"]
    cap = s + 3  # a little spare capacity, as a real cache has
    Kp = np.zeros((1, cap, d)); Kp[0, :s] = K
    Vp = np.zeros((1, cap, d)); Vp[0, :s] = V
    Np = np.zeros((1, cap), np.int32); Np[0, :s] = N
    out = oracle.csm_round(Kp, Vp, Np, [s], case["n1"], case["n2"], case["c"], case["m"])
    L = int(out["len"][0])
    assert L == case["expect_len"]
    assert L == oracle.len_after(s, case["n1"], case["n2"], case["c"], case["m"])
    np.testing.assert_allclose(out["K"][0, :L], arr(case["expect_K"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(out["V"][0, :L], arr(case["expect_V"]), rtol=0, atol=1e-12)
    assert out["N"][0, :L].tolist() == case["expect_N"]
    ch = oracle.num_chunks(s, case["n1"], case["n2"], case["c"])
    assert out["match"][0, :ch].tolist() == case["expect_match"]
    # degrees are conserved exactly
    assert int(out["N"][0, :L].sum()) == int(N.sum())


def test_skip_leaves_unit_untouched():
    case = CASES[0]
    K = arr(case["K"])[None]
    V = np.zeros_like(K)
    N = np.ones((1, K.shape[1]), np.int32)
    out = oracle.csm_round(K, V, N, [K.shape[1]], 0, 0, 8, 2, skip=[1])
    assert int(out["len"][0]) == K.shape[1]
    np.testing.assert_array_equal(out["K"], K)


def test_forced_replay_applies_given_decisions():
    # K1 with the tie at the top-m cut forced the other way (A3 instead of A1)
    case = CASES[0]
    K = arr(case["K"])[None]
    V = np.stack([np.arange(8.0), -np.arange(8.0)], 1)[None]
    N = np.ones((1, 8), np.int32)
    forced = np.array([[[0, -1, -1, 3]]], np.int32)
    out = oracle.csm_round(K, V, N, [8], 0, 0, 8, 2, forced=forced)
    assert out["match"][0, 0].tolist() == [0, -1, -1, 3]
    np.testing.assert_allclose(out["K"][0, :6], [[1, 0], [0, 1], [1, 1], [-1, 0], [-1, 1], [0.5, -1]])
    assert out["N"][0, :6].tolist() == [2, 1, 1, 1, 1, 2]
    with pytest.raises(ValueError):  # wrong edge count is rejected
        oracle.csm_round(K, V, N, [8], 0, 0, 8, 2, forced=np.array([[[0, 1, 2, -1]]], np.int32))


def test_origin_and_merged_records():
    case = CASES[0]  # K1_r025: rows 0 and 2 merge into rows 1 and 3
    K = arr(case["K"])[None]
    V = np.zeros_like(K)
    N = np.ones((1, 8), np.int32)
    out = oracle.csm_round(K, V, N, [8], 0, 0, 8, 2)
    assert out["origin"][0, :6].tolist() == [1, 3, 4, 5, 6, 7]
    assert out["merged"][0, :6].tolist() == [1, 1, 0, 0, 0, 0]
    skipped = oracle.csm_round(K, V, N, [8], 0, 0, 8, 2, skip=[1])
    assert skipped["origin"][0, :8].tolist() == list(range(8))
    assert skipped["merged"][0, :8].tolist() == [0] * 8
