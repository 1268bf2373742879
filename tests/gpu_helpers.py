"""Helpers for the GPU parity tests: run a CSM round through the C ABI and check it
against the oracle with the rules in oracle/compare.py.

Near-ties: every device decision that differs from the oracle's (allowed only where
the oracle's margin is below 1e-5) is printed with its unit, chunk, A index, both
choices and the oracle margin, and appended as one JSON line per decision to the
file named by the CSMKV_NEAR_TIE_LOG environment variable when it is set."""
import json
import os

import numpy as np
import torch

import oracle
from oracle import compare
from online_kv_cache_chunked_gb300 import binding as B


def to64(t):
    return t.detach().cpu().to(torch.float64).numpy()


def snapshot(K, V, N, L):
    BH = K.shape[0] * K.shape[1]
    cap, d = K.shape[2], K.shape[3]
    return dict(K=to64(K).reshape(BH, cap, d), V=to64(V).reshape(BH, cap, d),
                N=N.cpu().numpy().reshape(BH, cap).copy(), len=L.cpu().numpy().reshape(BH).copy())


def skip_vector(batch, h_kv, head_mask=None, seq_mask=None):
    sk = np.zeros(batch * h_kv, np.uint8)
    for u in range(batch * h_kv):
        b, h = divmod(u, h_kv)
        if head_mask is not None and int(head_mask[h]):
            sk[u] = 1
        if seq_mask is not None and not int(seq_mask[b]):
            sk[u] = 1
    return sk


def log_near_ties(records, context):
    """Prints and (if CSMKV_NEAR_TIE_LOG is set) appends the deviation records."""
    if not records:
        return
    for r in records:
        print(f"near-tie [{context}]: {r}")
    path = os.environ.get("CSMKV_NEAR_TIE_LOG")
    if path:
        os.makedirs(os.path.dirname(os.path.abspath(path)), exist_ok=True)
        with open(path, "a") as f:
            for r in records:
                f.write(json.dumps(dict(context=context, **r)) + "\n")


def gpu_round(K, V, N, L, n1, n2, c, r, head_mask=None, seq_mask=None, kernel=0, ws=None, limits=None):
    cache = B.cache_desc(K)
    maxch = max(1, B.csm_max_chunks(cache, n1, n2, c))
    match = torch.full((K.shape[0] * K.shape[1], maxch, c // 2), -2, dtype=torch.int32, device=K.device)
    if ws is None:
        ws = B.new_workspace(B.csm_workspace_bytes(cache, n1, n2, c), K.device)
    hm = None if head_mask is None else torch.as_tensor(np.asarray(head_mask, np.uint8)).to(K.device)
    sm = None if seq_mask is None else torch.as_tensor(np.asarray(seq_mask, np.uint8)).to(K.device)
    lm = None if limits is None else torch.as_tensor(np.asarray(limits, np.int32)).to(K.device)
    B.csm_compress_ex(K, V, N, L, n1, n2, c, r, head_mask=hm, seq_mask=sm, match_out=match,
                      kernel=kernel, seq_max_chunks=lm, workspace=ws)
    torch.cuda.synchronize()
    st = B.csmkv_device_status(ws)
    assert st == 0, f"device status {st}: {B.status_str(st)}"
    return match.cpu().numpy()


def round_parity(K, V, N, L, n1, n2, c, r, dtype, head_mask=None, seq_mask=None, kernel=0, max_dev_frac=0.01,
                 limits=None):
    """Runs one device round in place and checks it against the oracle. Returns stats.
    limits: optional per-sequence chunk caps (budget-exact rounds)."""
    pre = snapshot(K, V, N, L)
    m = B.csm_edges_per_chunk(r, c)
    gm = gpu_round(K, V, N, L, n1, n2, c, r, head_mask, seq_mask, kernel, limits=limits)
    post = snapshot(K, V, N, L)
    sk = skip_vector(K.shape[0], K.shape[1], head_mask, seq_mask)
    ul = None if limits is None else np.repeat(np.asarray(limits, np.int32), K.shape[1])
    free = oracle.csm_round(pre["K"], pre["V"], pre["N"], pre["len"], n1, n2, c, m, skip=sk, limits=ul)
    n_chunks = np.array([0 if sk[u] else oracle.num_chunks(int(pre["len"][u]), n1, n2, c)
                         for u in range(len(sk))])
    if ul is not None:
        n_chunks = np.where(ul > 0, np.minimum(n_chunks, ul), n_chunks)
    if m == 0:
        n_chunks[:] = 0
    log = []
    dev, fails = compare.check_round(pre["K"], free, gm, n_chunks, m, n1, c, log=log)
    log_near_ties(log, f"round c={c} m={m} kernel={kernel}")
    assert not fails, "\n".join(fails[:10])
    forced = np.where(gm >= -1, gm, -1)
    rep = oracle.csm_round(pre["K"], pre["V"], pre["N"], pre["len"], n1, n2, c, m, skip=sk, forced=forced,
                           limits=ul)
    fails, worst = compare.compare_state(rep, pre, post, dtype)
    assert not fails, "\n".join(fails[:10])
    # unprocessed units stay bit-identical
    for u in np.nonzero(n_chunks == 0)[0]:
        s = int(pre["len"][u])
        assert int(post["len"][u]) == s
        assert np.array_equal(post["K"][u, :s], pre["K"][u, :s])
        assert np.array_equal(post["N"][u, :s], pre["N"][u, :s])
    total = int(n_chunks.sum())
    assert dev <= max(2, max_dev_frac * total), f"{dev} of {total} chunks deviate (near-ties)"
    return dict(chunks=total, deviating=dev, worst_ratio=worst)


def attn_parity(q, K, V, N, L, out, dtype, scale=None):
    """Device attention output vs the oracle's on the same cache (rows past the
    longest unit are not copied to the host)."""
    top = max(1, int(L.max()))
    Ks, Vs, Ns = K[:, :, :top], V[:, :, :top], N[:, :, :top]
    ref = oracle.decode_attn_logn(to64(q), to64(Ks), to64(Vs), Ns.cpu().numpy(), L.cpu().numpy(), q.shape[1],
                                  scale=scale)
    got = to64(out)
    err = float(np.abs(got - ref).max()) if got.size else 0.0
    assert np.isfinite(got).all()
    assert err <= compare.ATTN_TOL[dtype], f"attention max error {err}"
    return err
