"""Comparison rules between a device result and the oracle (test infrastructure).

Decisions. The device computes similarities in fp32, the oracle in fp64, so an
argmax or a top-m cut whose competitors lie within 1e-5 of each other may go
either way. A device decision is accepted iff
  * every processed chunk has exactly m selected A tokens;
  * every selected A token's device target b has oracle cosine within 1e-5 of the
    oracle's best cosine for that A token (argmax near-tie);
  * the device's selected set is a top-m set of the oracle's per-A best cosines
    up to 1e-5 (cut near-tie).
Chunks whose device decisions differ from the oracle's are counted and logged;
the oracle is then replayed with the device decisions forced, and the state must
match that replay: lengths and degrees exactly, rows that are plain copies
bit-exactly, merged centroids within the value tolerance.

Value tolerance for merged K/V rows (per (sequence, head) unit, range = max - min
of the oracle's rows, amax = max |x| of the rows merged from). bf16 storage:

    1e-3 * range + 1/2 bf16 ulp(oracle value) + 2^-16 * amax.

The device forms sum_i n_i x_i with k <= c/2 + 1 fp32 fused multiply-adds,
multiplies by fl(1 / sum n_i) and rounds once to bf16. The fp32 part is off
the exact mean y by at most (k + 2) 2^-24 sum n_i |x_i| / sum n_i
<= 131 * 2^-24 amax < 2^-16 amax (c <= 256); rounding that to bf16 adds at
most half a bf16 ulp of y (if the fp32 value crosses a power of two the bf16
result is that power, no farther from y than the fp32 value). 1e-3 * range is
the stated bound on top. fp32 storage: 1e-6 * range + 4 fp32 ulps.
Attention outputs: 2e-2 absolute for bf16, 1e-5 for fp32.

Near-ties: check_round can collect one record per deviating decision (unit,
chunk, A index, device and oracle choices, the oracle's margin) for logging.
"""
from __future__ import annotations

import numpy as np

NEAR_TIE = 1e-5
ATTN_TOL = {"bf16": 2e-2, "f32": 1e-5}


def ulp(x, dtype):
    a = np.abs(np.asarray(x, np.float64))
    a = np.where(a > 0, a, 1e-30)
    e = np.floor(np.log2(a))
    mant = 7 if dtype == "bf16" else 23
    return np.exp2(e - mant)


def value_tol(ref_rows, dtype, src_rows=None):
    """Per-element bound for merged rows; src_rows: the pre-round rows they are merged
    from (default: ref_rows), for the fp32 summation term."""
    rng = float(ref_rows.max() - ref_rows.min()) if ref_rows.size else 0.0
    if dtype == "bf16":
        src = ref_rows if src_rows is None else src_rows
        amax = float(np.abs(src).max()) if np.size(src) else 0.0
        return 1e-3 * rng + 0.5 * ulp(ref_rows, dtype) + 2.0 ** -16 * amax
    return 1e-6 * rng + 4 * ulp(ref_rows, dtype)


def _cos(x, y):
    nx, ny = np.linalg.norm(x), np.linalg.norm(y)
    return 0.0 if nx == 0 or ny == 0 else float(x @ y) / (nx * ny)


def check_chunk_decisions(Kc, free_match, free_sim, gpu_match, m, tol=NEAR_TIE):
    """One chunk. Kc [c, d] fp64 pre-round keys. Returns (deviates, failure message or None)."""
    g = np.asarray(gpu_match)
    if np.array_equal(g, free_match):
        return False, None
    sel = g >= 0
    if int(sel.sum()) != m:
        return True, f"{int(sel.sum())} edges selected, expected {m}"
    if np.any(g >= len(g)):
        return True, "target outside B"
    for a in np.nonzero(sel)[0]:
        b = int(g[a])
        cs = _cos(Kc[2 * a], Kc[2 * b + 1])
        if cs < free_sim[a] - tol:
            return True, f"A{a}->B{b}: cos {cs:.9f} below best {free_sim[a]:.9f} by more than {tol}"
    if sel.any() and (~sel).any():
        lo = free_sim[sel].min()
        hi = free_sim[~sel].max()
        if lo < hi - tol:
            return True, f"selection is not a top-{m} set: {lo:.9f} < {hi:.9f} - {tol}"
    return True, None


def deviation_records(free_match, free_sim, free_margin, free_cut, gpu_match):
    """One record per A token whose device decision differs from the oracle's:
    a, device and oracle targets (-1 = not selected), and the oracle margin that
    decided it -- the argmax margin (best minus second-best cosine) when the
    target differs, the chunk's top-m cut margin (m-th minus (m+1)-th largest
    edge similarity) when only its selection differs."""
    out = []
    g = np.asarray(gpu_match)
    for a in np.nonzero(g != free_match)[0]:
        gb, fb = int(g[a]), int(free_match[a])
        if gb >= 0 and fb >= 0:
            kind, margin = "argmax", float(free_margin[a])
        else:
            kind, margin = "cut", float(free_cut)
        out.append(dict(a=int(a), device=gb, oracle=fb, kind=kind, oracle_margin=margin))
    return out


def check_round(pre_K, free, gpu_match, n_chunks, m, n1, c, units=None, log=None):
    """Decision check for a full round. pre_K [BH, cap, d] fp64; free: oracle.csm_round
    output; gpu_match [BH, maxch, c/2]; n_chunks [BH] processed chunks per unit.
    log: optional list; one record per deviating decision is appended to it.
    Returns (deviating chunk count, list of failures)."""
    dev, fails = 0, []
    units = range(pre_K.shape[0]) if units is None else units
    for u in units:
        for j in range(int(n_chunks[u])):
            base = n1 + j * c
            d_, f_ = check_chunk_decisions(pre_K[u, base:base + c], free["match"][u, j], free["sim"][u, j],
                                           gpu_match[u, j], m)
            dev += int(d_)
            if f_:
                fails.append(f"unit {u} chunk {j}: {f_}")
            if d_ and log is not None:
                for r in deviation_records(free["match"][u, j], free["sim"][u, j], free["margin"][u, j],
                                           free["cut"][u, j], gpu_match[u, j]):
                    log.append(dict(unit=int(u), chunk=int(j), **r))
    return dev, fails


def compare_state(replay, pre, gpu, dtype, units=None):
    """Device state vs the forced replay. pre/gpu: dicts K, V [BH, cap, d] fp64, N [BH, cap],
    len [BH]. Returns list of failures (empty = pass) and the max merged-row error ratio."""
    fails = []
    worst = 0.0
    units = range(pre["K"].shape[0]) if units is None else units
    for u in units:
        s = int(replay["len"][u])
        if int(gpu["len"][u]) != s:
            fails.append(f"unit {u}: len {int(gpu['len'][u])} != {s}")
            continue
        if not np.array_equal(gpu["N"][u, :s], replay["N"][u, :s]):
            fails.append(f"unit {u}: degrees differ")
        org = replay["origin"][u, :s]
        mrg = replay["merged"][u, :s].astype(bool)
        for name in ("K", "V"):
            g, r = gpu[name][u, :s], replay[name][u, :s]
            copies = ~mrg
            if not np.array_equal(g[copies], pre[name][u, org[copies]]):
                fails.append(f"unit {u}: {name} copied rows are not bit-exact")
            if mrg.any():
                tol = value_tol(r, dtype, pre[name][u, :int(pre["len"][u])])[mrg]
                err = np.abs(g[mrg] - r[mrg])
                worst = max(worst, float((err / tol).max()))
                if np.any(err > tol):
                    fails.append(f"unit {u}: {name} merged rows off by {float(err.max()):.3e}")
    return fails, worst
