"""Theorem 6.1 pins the oracle's partition choice.

[Chelsea §三 理论分析, Theorem 6.1]: over balanced partitions (A, B) of [2n],
if f has non-increasing, non-negative successive decrements (convex and
non-increasing), the alternating partition A0 = {1,3,...,2n-1} maximises
sum_{x in A} sum_{y in B} f(|x - y|). The test brute-forces every balanced
partition for 2n <= 12 and checks that the partition the oracle actually uses
(A = even 0-based offsets = odd 1-based positions) attains the maximum.
"""
import itertools
import math

import numpy as np
import pytest

import oracle


def objective(A, B, f):
    return sum(f(abs(x - y)) for x in A for y in B)


def brute_max(two_n, f):
    best = -math.inf
    full = set(range(two_n))
    for A in itertools.combinations(range(two_n), two_n // 2):
        B = full.difference(A)
        best = max(best, objective(A, B, f))
    return best


def families(two_n, rng):
    fams = {
        "exp": lambda k: math.exp(-0.7 * k),
        "inverse": lambda k: 1.0 / k,
        "linear": lambda k: float(2 * two_n - k),
        "constant": lambda k: 3.0,
    }
    # random convex non-increasing: f(k) = f(k-1) - delta_k with delta_1 >= delta_2 >= ... >= 0
    deltas = np.sort(rng.uniform(0.0, 1.0, two_n))[::-1]
    vals = np.concatenate([[5.0], 5.0 - np.cumsum(deltas)])
    fams["random_convex"] = lambda k, v=vals: float(v[k - 1])
    return fams


@pytest.mark.parametrize("two_n", [2, 4, 6, 8, 10, 12])
def test_alternating_partition_is_optimal(two_n):
    rng = np.random.default_rng(two_n)
    a_off, b_off = oracle.partition(two_n)
    A, B = [int(x) for x in a_off], [int(x) for x in b_off]
    assert sorted(A + B) == list(range(two_n)) and len(A) == len(B) == two_n // 2
    for name, f in families(two_n, rng).items():
        got = objective(A, B, f)
        assert got >= brute_max(two_n, f) - 1e-12, (two_n, name)


@pytest.mark.parametrize("two_n", [4, 8, 12])
def test_contiguous_partition_is_not_optimal(two_n):
    # the brute force has teeth: splitting a chunk into halves loses for a
    # strictly convex decreasing similarity profile
    f = lambda k: math.exp(-0.7 * k)  # noqa: E731
    half = list(range(two_n // 2))
    rest = list(range(two_n // 2, two_n))
    assert objective(half, rest, f) < brute_max(two_n, f) - 1e-6
