"""Host-side schedule of the inference pipeline, written out plainly (fp64).

TEST INFRASTRUCTURE (see the package docstring). Independent of the product's
C-ABI host helpers, which the tests compare against these.

[Chelsea §三 算法流程, Algorithm 1]: budget B = R (n + Gamma); a CSM round runs
whenever the cache length s reaches B + g, checked once after prefill and once
after every decode append (one round per check).
[CentroidKV 技术摘要 / 分块软匹配 (CSM), 渐进式调度]: the ratio decays linearly
over rounds, r_j = r_init - j * delta_r; a floor r_min keeps it positive.
"""
from __future__ import annotations

import math


def budget(n: int, R: float, Gamma: int) -> float:
    return float(R) * (float(n) + float(Gamma))


def should_trigger(s: int, B: float, g: int) -> bool:
    return float(s) >= B + float(g)


def ratio(j: int, r_init: float, dr: float, r_min: float) -> float:
    return max(float(r_init) - float(j) * float(dr), float(r_min))


def edges_per_chunk(r: float, c: int) -> int:
    """m = floor(r c); the 1e-9 nudge keeps r c that is an integer in exact
    arithmetic from flooring one below because of fp64 rounding of r."""
    return int(math.floor(float(r) * float(c) + 1e-9))


def num_chunks(s: int, n1: int, n2: int, c: int) -> int:
    mid = s - n1 - n2
    return mid // c if mid > 0 else 0


def len_after(s: int, n1: int, n2: int, c: int, m: int) -> int:
    """Every merged edge removes exactly one A token, m per full chunk."""
    return s - num_chunks(s, n1, n2, c) * m


def chunks_to_budget(s: int, B: float, n1: int, n2: int, c: int, m: int) -> int:
    """Budget-exact compression (an extension beside the pages' Algorithm 1,
    which merges every full chunk): the fewest oldest chunks whose merge brings
    s to <= B. Each merged chunk removes m rows, so k = ceil((s - B) / m),
    capped by the full chunks there are."""
    if m <= 0 or not (float(s) > float(B)):
        return 0
    return min(int(math.ceil((float(s) - float(B)) / float(m))), num_chunks(s, n1, n2, c))


def plan_budget_exact(n: int, R: float, Gamma: int, g: int, n1: int, n2: int, c: int,
                      r_init: float = 0.5, dr: float = 0.0, r_min: float = 0.0, steps: int | None = None):
    """As plan(), but every round merges only chunks_to_budget(...) chunks.

    Returns a list of (step, s_before, r, m, k, s_after)."""
    B = budget(n, R, Gamma)
    s, j, out = n, 0, []
    total = Gamma if steps is None else steps
    for step in range(0, total + 1):
        if step > 0:
            s += 1
        if should_trigger(s, B, g):
            r = ratio(j, r_init, dr, r_min)
            m = edges_per_chunk(r, c)
            k = chunks_to_budget(s, B, n1, n2, c, m)
            s2 = s - k * m
            out.append((step, s, r, m, k, s2))
            s = s2
            j += 1
    return out


def plan(n: int, R: float, Gamma: int, g: int, n1: int, n2: int, c: int,
         r_init: float = 0.5, dr: float = 0.0, r_min: float = 0.0, steps: int | None = None):
    """Rounds of Algorithm 1 for one sequence of prefill length n.

    Returns a list of (step, s_before, r, m, s_after); step 0 is the check right
    after prefill, step i >= 1 the check after the i-th decode append. The
    decode loop runs ``steps`` appends (default Gamma).
    """
    B = budget(n, R, Gamma)
    s, j, out = n, 0, []
    total = Gamma if steps is None else steps
    for step in range(0, total + 1):
        if step > 0:
            s += 1
        if should_trigger(s, B, g):
            r = ratio(j, r_init, dr, r_min)
            m = edges_per_chunk(r, c)
            s2 = len_after(s, n1, n2, c, m)
            out.append((step, s, r, m, s2))
            s = s2
            j += 1
    return out
