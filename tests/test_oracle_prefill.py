"""Pins for the oracle's prefill attention ([Chelsea] §三 算法流程, Algorithm 1: the prompt's
O = FlashAttn(Q, K, V), every degree 1): closed forms, causality, the query-to-KV head
mapping and agreement with the separately pinned decode attention at degree 1."""
import numpy as np
import pytest

import oracle


def _case(seed, B=2, Hkv=2, G=3, n=45, cap=48, d=16):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, Hkv * G, n, d))
    K = rng.standard_normal((B, Hkv, cap, d))
    V = rng.standard_normal((B, Hkv, cap, d))
    return q, K, V, n, Hkv * G


def test_first_row_is_its_own_value():
    q, K, V, n, hq = _case(1)
    o = oracle.prefill_attn(q, K, V, n, hq)
    G = hq // K.shape[1]
    for b in range(q.shape[0]):
        for h in range(hq):
            assert np.array_equal(o[b, h, 0], V[b, h // G, 0])


def test_identical_keys_average_the_values():
    q, K, V, n, hq = _case(2)
    K[:] = K[:, :, :1, :]  # every key the same vector: uniform weights over the visible rows
    o = oracle.prefill_attn(q, K, V, n, hq)
    G = hq // K.shape[1]
    for i in (0, 1, 7, n - 1):
        want = V[:, :, : i + 1].mean(axis=2)  # [B, Hkv, d]
        for h in range(hq):
            np.testing.assert_allclose(o[:, h, i], want[:, h // G], rtol=1e-12, atol=1e-12)


def test_two_tokens_with_known_weights():
    # logits 0 and ln 3 give the weights 1/4 and 3/4
    d = 4
    scale = 0.5
    q = np.zeros((1, 1, 2, d))
    q[0, 0, 1, 0] = 1.0
    K = np.zeros((1, 1, 2, d))
    K[0, 0, 1, 0] = np.log(3.0) / scale
    V = np.zeros((1, 1, 2, d))
    V[0, 0, 0] = [4.0, 0.0, 8.0, -4.0]
    V[0, 0, 1] = [0.0, 4.0, 4.0, 4.0]
    o = oracle.prefill_attn(q, K, V, 2, 1, scale=scale)
    np.testing.assert_allclose(o[0, 0, 1], [1.0, 3.0, 5.0, 2.0], rtol=1e-14, atol=1e-14)


def test_causal_future_rows_do_not_matter():
    q, K, V, n, hq = _case(3)
    i = 20
    o = oracle.prefill_attn(q, K, V, n, hq, rows=[i])
    K2, V2 = K.copy(), V.copy()
    K2[:, :, i + 1:] = 100.0
    V2[:, :, i + 1:] = -7.0
    assert np.array_equal(oracle.prefill_attn(q, K2, V2, n, hq, rows=[i]), o)
    K2[:, :, i] += 0.5  # a visible row does matter
    assert not np.allclose(oracle.prefill_attn(q, K2, V2, n, hq, rows=[i]), o)


def test_query_heads_read_their_group():
    q, K, V, n, hq = _case(4)
    Hkv = K.shape[1]
    G = hq // Hkv
    for k in range(Hkv):
        V[:, k] = float(k + 1)  # constant values per KV head: any weights give that constant
    o = oracle.prefill_attn(q, K, V, n, hq)
    for h in range(hq):
        np.testing.assert_allclose(o[:, h], h // G + 1.0, rtol=0, atol=1e-12)


def test_matches_decode_attention_at_degree_one():
    q, K, V, n, hq = _case(5)
    B, Hkv, cap, d = K.shape
    N = np.ones((B, Hkv, cap), np.int32)
    rows = [0, 1, 13, 31, n - 1]
    o = oracle.prefill_attn(q, K, V, n, hq, rows=rows)
    for r, i in enumerate(rows):
        L = np.full((B, Hkv), i + 1, np.int32)
        want = oracle.decode_attn_logn(q[:, :, i], K, V, N, L, hq)
        np.testing.assert_allclose(o[:, :, r], want, rtol=1e-12, atol=1e-12)


def test_row_subset_equals_full():
    q, K, V, n, hq = _case(6)
    full = oracle.prefill_attn(q, K, V, n, hq)
    rows = [44, 3, 17]
    assert np.array_equal(oracle.prefill_attn(q, K, V, n, hq, rows=rows), full[:, :, rows])


def test_rows_outside_the_prompt_are_rejected():
    q, K, V, n, hq = _case(7)
    with pytest.raises(ValueError):
        oracle.prefill_attn(q, K, V, n, hq, rows=[n])
