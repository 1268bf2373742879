"""A second, separately written CSM round for tiny inputs (test helper).

Written from the same page steps as the C oracle but in a different shape:
whole-chunk numpy similarity matrices, Python sorting of all candidate edges
and dictionary grouping of merge targets. Used only to cross-check the oracle's
bookkeeping (chunk origins, compaction, remainder and recent window, several
rounds) on inputs small enough for pure Python.
"""
import numpy as np


def csm_round_bruteforce(K, V, N, s, n1, n2, c, m, limit=0):
    """K, V: [s, d] float64; N: [s] ints. Returns (K', V', N', s', matches)."""
    K = np.asarray(K, float)[:s]
    V = np.asarray(V, float)[:s]
    N = [int(x) for x in N[:s]]
    n_chunks = max(0, s - n1 - n2) // c
    if limit > 0:  # budget-exact: only the oldest `limit` chunks are matched
        n_chunks = min(n_chunks, limit)
    if n_chunks == 0 or m == 0:
        return K.copy(), V.copy(), list(N), s, []
    rows_k, rows_v, rows_n, matches = [], [], [], []
    for t in range(n1):
        rows_k.append(K[t]); rows_v.append(V[t]); rows_n.append(N[t])
    for j in range(n_chunks):
        base = n1 + j * c
        idx_a = [base + o for o in range(0, c, 2)]
        idx_b = [base + o for o in range(1, c, 2)]
        KA, KB = K[idx_a], K[idx_b]
        na = np.sqrt((KA * KA).sum(1))
        nb = np.sqrt((KB * KB).sum(1))
        S = np.zeros((len(idx_a), len(idx_b)))
        for i in range(len(idx_a)):
            for k in range(len(idx_b)):
                if na[i] > 0 and nb[k] > 0:
                    S[i, k] = float(KA[i] @ KB[k]) / (na[i] * nb[k])
        best = [int(np.argmax(S[i])) for i in range(len(idx_a))]  # first max = lowest B
        cand = sorted(((-S[i, best[i]], i) for i in range(len(idx_a))))
        chosen = {i for _, i in cand[:m]}
        groups = {}
        for i in sorted(chosen):
            groups.setdefault(best[i], []).append(i)
        matches.append([best[i] if i in chosen else -1 for i in range(len(idx_a))])
        for o in range(c):
            t = base + o
            if o % 2 == 0:
                if o // 2 in chosen:
                    continue
                rows_k.append(K[t]); rows_v.append(V[t]); rows_n.append(N[t])
                continue
            members = [t] + [idx_a[i] for i in groups.get(o // 2, [])]
            if len(members) == 1:
                rows_k.append(K[t]); rows_v.append(V[t]); rows_n.append(N[t])
                continue
            w = np.array([N[x] for x in members], float)
            rows_k.append((w[:, None] * K[members]).sum(0) / w.sum())
            rows_v.append((w[:, None] * V[members]).sum(0) / w.sum())
            rows_n.append(int(w.sum()))
    for t in range(n1 + n_chunks * c, s):
        rows_k.append(K[t]); rows_v.append(V[t]); rows_n.append(N[t])
    return np.array(rows_k), np.array(rows_v), rows_n, len(rows_n), matches
