"""The parity rules themselves (oracle/compare.py), on the CPU.

* The merged-row tolerance is what the arithmetic allows: a degree-weighted mean
  formed as the device forms it (fp32 fused multiply-adds in A order, one fp32
  reciprocal of the degree sum, one rounding to bf16) stays inside it for
  clusters of up to 129 members, while a mean with one member's degree dropped,
  or an error as large as 1e-3 * range plus one whole bf16 ulp (the looser
  bound this replaced), falls outside it.
* A decision that differs from the oracle's only at an exact tie is counted as a
  near-tie deviation and logged with its margin (0); a decision that differs
  where the oracle's margin is large is a failure.
"""
import numpy as np
import torch

import oracle
from oracle import compare


def _bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


def _device_mean(n, x):
    """fp32 fma chain in member order, times fl32(1/sum n), rounded once to bf16."""
    acc = np.float32(0.0) * x[0].astype(np.float32)
    for ni, xi in zip(n, x):
        acc = (acc.astype(np.float64) + float(ni) * xi).astype(np.float32)
    inv = np.float32(1.0) / np.float32(float(np.sum(n)))
    return _bf16(acc * inv)


def test_merged_row_tolerance_covers_device_arithmetic_and_no_more():
    rng = np.random.default_rng(0)
    d = 128
    caught_drop = caught_ulp = total = 0
    for k in (2, 3, 17, 64, 129):
        for _ in range(20):
            x = _bf16(rng.standard_normal((k, d)) * rng.choice([0.3, 1.0, 5.0]))
            n = rng.integers(1, 40, k)
            exact = (n[:, None] * x).sum(0) / n.sum()
            got = _device_mean(n, x)
            tol = compare.value_tol(exact[None], "bf16", x)[0]
            assert np.all(np.abs(got - exact) <= tol), k
            n2 = n.copy()
            n2[-1] = 1 if n[-1] > 1 else 7  # one member's degree dropped / wrong
            wrong = (n2[:, None] * x).sum(0) / n2.sum()
            caught_drop += int(np.any(np.abs(wrong - exact) > tol))
            # an error as large as the looser bound 1e-3 * range + one full ulp
            rngx = float(exact.max() - exact.min())
            off = exact + 1e-3 * rngx + compare.ulp(exact, "bf16")
            frac = float(np.mean(np.abs(off - exact) > tol))
            # the fp32 summation term grows with the cluster size; up to 17
            # members the half-ulp term decides nearly everywhere
            caught_ulp += int(frac > (0.9 if k <= 17 else 0.3))
            total += 1
    assert caught_drop >= 0.9 * total and caught_ulp >= 0.9 * total


def test_near_tie_deviation_is_logged_and_a_real_one_fails():
    rng = np.random.default_rng(1)
    c, d, m = 8, 4, 4
    Kc = rng.standard_normal((1, c, d))
    Kc[0, 3] = Kc[0, 1]  # B rows 0 and 1 identical: A rows tie exactly between them
    Vc = rng.standard_normal((1, c, d))
    Nc = np.ones((1, c), np.int32)
    free = oracle.csm_chunks(Kc, Vc, Nc, m)
    assert free["match"][0].max() < 4
    tied = [a for a in range(4) if free["match"][0, a] == 0]
    assert tied, "some A row should pick B0 (lowest index of the tie)"
    gpu = free["match"].copy()
    gpu[0, tied[0]] = 1  # the other member of the exact tie
    fr = dict(match=free["match"][None], sim=free["sim"][None], margin=free["margin"][None],
              cut=free["cut"][None])
    log = []
    dev, fails = compare.check_round(np.concatenate([Kc, Kc], 1), fr, gpu[None], np.array([1]), m, 0, c, log=log)
    assert dev == 1 and not fails
    assert log == [dict(unit=0, chunk=0, a=tied[0], device=1, oracle=0, kind="argmax", oracle_margin=0.0)]
    # a target far from the best similarity is not a near-tie
    bad = free["match"].copy()
    sims = [compare._cos(Kc[0, 2 * tied[0]], Kc[0, 2 * b + 1]) for b in range(4)]
    bad[0, tied[0]] = int(np.argmin(sims))
    dev, fails = compare.check_round(np.concatenate([Kc, Kc], 1), fr, bad[None], np.array([1]), m, 0, c)
    assert dev == 1 and fails
