"""Invariants and special cases that pin the oracle independently of itself.

* Degree-weighted averaging conserves the token count (sum N) exactly and the
  first moments sum_t n_t k_t, sum_t n_t v_t up to fp64 rounding
  [CentroidKV 聚合; Chelsea §三 分块软匹配算法 step 4].
* "At most half per step" [Chelsea §八 局限性; CentroidKV 局限性]: one round
  removes at most half of the chunked middle.
* Degree-aware attention [Chelsea §三 核心公式]:
  - N = 1 everywhere reduces to textbook softmax attention (checked against
    torch.softmax in float64, a library routine);
  - a cache whose clusters are exact duplicates gives, after merging, the same
    output as full attention over the uncompressed cache;
  - adding a constant to every logit leaves the output unchanged.
"""
import numpy as np
import pytest
import torch

import oracle


def test_conservation_over_rounds():
    rng = np.random.default_rng(3)
    BH, cap, d, n1, n2, c = 4, 600, 16, 4, 16, 32
    K = rng.standard_normal((BH, cap, d))
    V = rng.standard_normal((BH, cap, d))
    N = rng.integers(1, 4, (BH, cap)).astype(np.int32)
    L = np.array([600, 533, 150, 52], np.int32)
    for m in (16, 12, 8):
        mom_k = np.array([(N[u, :L[u], None] * K[u, :L[u]]).sum(0) for u in range(BH)])
        mom_v = np.array([(N[u, :L[u], None] * V[u, :L[u]]).sum(0) for u in range(BH)])
        tok = np.array([int(N[u, :L[u]].sum()) for u in range(BH)])
        mids = np.maximum(L - n1 - n2, 0)
        out = oracle.csm_round(K, V, N, L, n1, n2, c, m)
        K, V, N, L2 = out["K"], out["V"], out["N"], out["len"]
        for u in range(BH):
            s = int(L2[u])
            assert int(N[u, :s].sum()) == tok[u]
            np.testing.assert_allclose((N[u, :s, None] * K[u, :s]).sum(0), mom_k[u], atol=1e-9)
            np.testing.assert_allclose((N[u, :s, None] * V[u, :s]).sum(0), mom_v[u], atol=1e-9)
            assert s >= int(L[u]) - mids[u] // 2
            assert s == oracle.len_after(int(L[u]), n1, n2, c, m)
        L = L2


def full_attention_torch(q, K, V, G):
    """Textbook softmax attention in float64 (torch library ops only)."""
    qt, Kt, Vt = (torch.from_numpy(np.asarray(x, float)) for x in (q, K, V))
    Kt = Kt.repeat_interleave(G, dim=1)  # [B, Hq, s, d]
    Vt = Vt.repeat_interleave(G, dim=1)
    logits = torch.einsum("bhd,bhsd->bhs", qt, Kt) / np.sqrt(q.shape[-1])
    return torch.einsum("bhs,bhsd->bhd", torch.softmax(logits, dim=-1), Vt).numpy()


@pytest.mark.parametrize("G", [1, 4, 7])
def test_unit_degrees_is_textbook_softmax(G):
    rng = np.random.default_rng(G)
    B, Hkv, s, d = 2, 3, 37, 16
    K = rng.standard_normal((B, Hkv, s, d))
    V = rng.standard_normal((B, Hkv, s, d))
    q = rng.standard_normal((B, Hkv * G, d)) * 2.0
    N = np.ones((B, Hkv, s), np.int32)
    o = oracle.decode_attn_logn(q, K, V, N, np.full((B, Hkv), s), Hkv * G)
    np.testing.assert_allclose(o, full_attention_torch(q, K, V, G), rtol=0, atol=1e-12)


def test_ragged_lengths_ignore_rows_past_len():
    rng = np.random.default_rng(11)
    B, Hkv, cap, d = 1, 2, 20, 8
    K = rng.standard_normal((B, Hkv, cap, d))
    V = rng.standard_normal((B, Hkv, cap, d))
    N = np.ones((B, Hkv, cap), np.int32)
    q = rng.standard_normal((B, Hkv, d))
    L = np.array([[7, 0]])
    o = oracle.decode_attn_logn(q, K, V, N, L, Hkv)
    ref = full_attention_torch(q[:, :1], K[:, :1, :7], V[:, :1, :7], 1)
    np.testing.assert_allclose(o[:, :1], ref, atol=1e-12)
    assert np.all(o[:, 1] == 0.0)  # an empty head has a zero output


def test_duplicate_clusters_give_full_attention():
    rng = np.random.default_rng(5)
    B, Hkv, G, d, n1, n2, c = 1, 2, 4, 32, 4, 8, 16
    s = n1 + 5 * c + 3 + n2
    base = rng.standard_normal((B * Hkv, s, d))
    vals = rng.standard_normal((B * Hkv, s, d))
    # every A token is an exact copy of its B partner (the next row)
    for u in range(B * Hkv):
        for j in range(5):
            for o in range(0, c, 2):
                t = n1 + j * c + o
                base[u, t] = base[u, t + 1]
                vals[u, t] = vals[u, t + 1]
    N = np.ones((B * Hkv, s), np.int32)
    q = rng.standard_normal((B, Hkv * G, d))
    full = oracle.decode_attn_logn(q, base.reshape(B, Hkv, s, d), vals.reshape(B, Hkv, s, d),
                                   N.reshape(B, Hkv, s), np.full((B, Hkv), s), Hkv * G)
    out = oracle.csm_round(base, vals, N, np.full(B * Hkv, s), n1, n2, c, c // 2)
    L = out["len"]
    assert np.all(L == s - 5 * (c // 2))
    # every A merged into its own partner, so every centroid equals its members
    assert np.all(out["match"][:, :5] == np.arange(c // 2))
    comp = oracle.decode_attn_logn(q, out["K"].reshape(B, Hkv, s, d), out["V"].reshape(B, Hkv, s, d),
                                   out["N"].reshape(B, Hkv, s), L.reshape(B, Hkv), Hkv * G)
    np.testing.assert_allclose(comp, full, rtol=0, atol=1e-12)


def test_logit_shift_invariance():
    rng = np.random.default_rng(9)
    B, Hkv, s, d = 1, 1, 50, 8
    K = rng.standard_normal((B, Hkv, s, d))
    V = rng.standard_normal((B, Hkv, s, d))
    N = rng.integers(1, 9, (B, Hkv, s)).astype(np.int32)
    q = rng.standard_normal((B, 1, d))
    o1 = oracle.decode_attn_logn(q, K, V, N, [[s]], 1)
    # q -> q + alpha * u with every key having the same component along u shifts all logits equally
    u = np.zeros(d); u[0] = 1.0
    K2 = K.copy(); K2[..., 0] = 0.75
    o2 = oracle.decode_attn_logn(q, K2, V, N, [[s]], 1)
    o3 = oracle.decode_attn_logn(q + 40.0 * u, K2, V, N, [[s]], 1)
    np.testing.assert_allclose(o2, o3, rtol=0, atol=1e-12)
    assert not np.allclose(o1, o2)  # the edit changed the logits, so the check is live


def test_degrees_weight_like_repeated_tokens():
    # n_t copies of a token == one centroid with degree n_t
    rng = np.random.default_rng(13)
    d, s = 8, 12
    K = rng.standard_normal((s, d))
    V = rng.standard_normal((s, d))
    n = rng.integers(1, 5, s)
    q = rng.standard_normal((1, 1, d))
    Kx = np.repeat(K, n, axis=0)
    Vx = np.repeat(V, n, axis=0)
    full = full_attention_torch(q, Kx[None, None], Vx[None, None], 1)
    o = oracle.decode_attn_logn(q, K[None, None], V[None, None], n[None, None].astype(np.int32), [[s]], 1)
    np.testing.assert_allclose(o, full, rtol=0, atol=1e-12)


def test_append_writes_row_len_with_unit_degree():
    K = np.zeros((2, 4, 3)); V = np.zeros((2, 4, 3)); N = np.zeros((2, 4), np.int32)
    L = np.array([1, 4], np.int32)
    kn = np.arange(6.0).reshape(2, 3); vn = -kn
    K2, V2, N2, L2, full = oracle.append(K, V, N, L, kn, vn)
    assert L2.tolist() == [2, 4] and full == 1
    np.testing.assert_array_equal(K2[0, 1], kn[0])
    np.testing.assert_array_equal(V2[0, 1], vn[0])
    assert N2[0, 1] == 1 and np.all(K2[1] == 0)
