"""Degree-aware decode attention and append on the GPU against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from online_kv_cache_chunked_gb300 import binding as B
from online_kv_cache_chunked_gb300 import synth
from tests.gpu_helpers import attn_parity, round_parity, to64

pytestmark = pytest.mark.gpu


def _attn(q, K, V, N, L):
    cache = B.cache_desc(K)
    ws = B.new_workspace(B.decode_attn_workspace_bytes(cache, q.shape[1]))
    out = torch.full((q.shape[0], q.shape[1], K.shape[3]), float("nan"), dtype=K.dtype, device=K.device)
    B.decode_attn_logn(q, K, V, N, L, out, ws)
    torch.cuda.synchronize()
    assert B.csmkv_device_status(ws) == 0
    return out


def _case(rng, batch, h_kv, G, cap, D, lengths, dtype=torch.bfloat16, degrees=True, garbage=True):
    K = torch.randn(batch, h_kv, cap, D, device="cuda").to(dtype)
    V = torch.randn(batch, h_kv, cap, D, device="cuda").to(dtype)
    N = torch.from_numpy(rng.integers(1, 50, (batch, h_kv, cap)).astype(np.int32)).cuda() if degrees else \
        torch.ones(batch, h_kv, cap, dtype=torch.int32, device="cuda")
    L = torch.tensor(lengths, dtype=torch.int32, device="cuda").view(batch, h_kv)
    if garbage:  # rows past len hold anything, NaN included
        for b in range(batch):
            for h in range(h_kv):
                s = int(L[b, h])
                K[b, h, s:] = float("nan")
                V[b, h, s:] = float("nan")
    q = (torch.randn(batch, h_kv * G, D, device="cuda") * 1.5).to(dtype)
    return q, K, V, N, L


@pytest.mark.parametrize("G,D", [(4, 128), (7, 128), (1, 128), (8, 128), (4, 64), (2, 64)])
def test_ragged_lengths_and_degrees(cuda_lib, G, D):
    rng = np.random.default_rng(G * 100 + D)
    lengths = [[0, 1, 63, 64, 65, 1000, 4099, 777], [16, 3000, 2, 129, 5000, 0, 64 * 9, 1]]
    q, K, V, N, L = _case(rng, 2, 8, G, 5120, D, lengths)
    out = _attn(q, K, V, N, L)
    attn_parity(q, K, V, N, L, out, "bf16")


def test_unit_degrees_long_context(cuda_lib):
    rng = np.random.default_rng(1)
    q, K, V, N, L = _case(rng, 1, 8, 4, 33000, 128, [[32768, 32000, 100, 31111, 5, 32999, 16384, 1]],
                          degrees=False, garbage=False)
    out = _attn(q, K, V, N, L)
    attn_parity(q, K, V, N, L, out, "bf16")


def test_fp32_path(cuda_lib):
    rng = np.random.default_rng(2)
    q, K, V, N, L = _case(rng, 2, 3, 3, 600, 64, [[545, 0, 17], [600, 1, 333]], dtype=torch.float32)
    out = _attn(q, K, V, N, L)
    attn_parity(q, K, V, N, L, out, "f32")


def test_unsupported_group_size(cuda_lib):
    rng = np.random.default_rng(3)
    q, K, V, N, L = _case(rng, 1, 2, 9, 64, 128, [[10, 10]])
    with pytest.raises(B.CsmkvError) as e:
        _attn(q, K, V, N, L)
    assert e.value.code == 8


def test_duplicate_clusters_equal_full_attention_on_gpu(cuda_lib):
    # CSM on a cache whose A tokens duplicate their partners, then log-N attention
    # over the compressed cache must equal softmax attention over the original
    rng = np.random.default_rng(4)
    n1, n2, c, D, G = 16, 64, 256, 128, 4
    s = n1 + 6 * c + 40 + n2
    K = torch.randn(1, 2, 2048, D, device="cuda").to(torch.bfloat16)
    V = torch.randn(1, 2, 2048, D, device="cuda").to(torch.bfloat16)
    for j in range(6):
        base = n1 + j * c
        K[:, :, base:base + c:2] = K[:, :, base + 1:base + c:2]
        V[:, :, base:base + c:2] = V[:, :, base + 1:base + c:2]
    N = torch.ones(1, 2, 2048, dtype=torch.int32, device="cuda")
    L = torch.full((1, 2), s, dtype=torch.int32, device="cuda")
    q = torch.randn(1, 2 * G, D, device="cuda").to(torch.bfloat16)
    full = _attn(q, K, V, N, L)
    round_parity(K, V, N, L, n1, n2, c, 0.5, "bf16", max_dev_frac=1.0)
    assert int(L[0, 0]) == s - 6 * 128
    comp = _attn(q, K, V, N, L)
    assert float((comp.float() - full.float()).abs().max()) <= 2e-2


def test_append_and_capacity(cuda_lib):
    K = torch.zeros(2, 3, 16, 64, dtype=torch.bfloat16, device="cuda")
    V = torch.zeros_like(K)
    N = torch.zeros(2, 3, 16, dtype=torch.int32, device="cuda")
    L = torch.tensor([[0, 5, 15], [16, 3, 8]], dtype=torch.int32, device="cuda")
    kn = torch.randn(2, 3, 64, device="cuda").to(torch.bfloat16)
    vn = torch.randn(2, 3, 64, device="cuda").to(torch.bfloat16)
    ws = B.new_workspace(B.csm_append_workspace_bytes())
    pre = [to64(K).reshape(6, 16, 64), to64(V).reshape(6, 16, 64), N.cpu().numpy().reshape(6, 16),
           L.cpu().numpy().reshape(6)]
    B.csm_append(K, V, N, L, kn, vn, workspace=ws)
    torch.cuda.synchronize()
    assert B.csmkv_device_status(ws) == 4  # the full unit reports CSMKV_ERR_CAPACITY
    k2, v2, n2, l2, full = oracle.append(*pre, to64(kn).reshape(6, 64), to64(vn).reshape(6, 64))
    assert full == 1
    assert np.array_equal(L.cpu().numpy().reshape(6), l2)
    assert np.array_equal(to64(K).reshape(6, 16, 64), k2) and np.array_equal(to64(V).reshape(6, 16, 64), v2)
    assert np.array_equal(N.cpu().numpy().reshape(6, 16), n2)
    # seq_mask appends only the selected sequences
    B.csmkv_clear_status(ws)
    B.csm_append(K, V, N, L, kn, vn, seq_mask=torch.tensor([1, 0], dtype=torch.uint8, device="cuda"), workspace=ws)
    torch.cuda.synchronize()
    assert L.cpu().tolist() == [[2, 7, 16], [16, 4, 9]]
    assert B.csmkv_device_status(ws) == 4  # unit (0, 2) filled up on the first append
    B.csmkv_clear_status(ws)
    L.copy_(torch.tensor([[1, 1, 1], [1, 1, 1]], dtype=torch.int32))
    B.csm_append(K, V, N, L, kn, vn, workspace=ws)
    torch.cuda.synchronize()
    assert B.csmkv_device_status(ws) == 0 and L.cpu().tolist() == [[2, 2, 2], [2, 2, 2]]


def test_full_64k_stack_decode_sampled(cuda_lib):
    """Full-size attention after the prefill rounds, sampled units checked by the oracle."""
    w = synth.WORKLOADS["llama_64k_32l"]
    d = synth.make_device(w)
    from online_kv_cache_chunked_gb300.pipeline import Pipeline
    p = Pipeline(w, d)
    p.run(steps=3)
    torch.cuda.synchronize()
    assert d["len"].cpu().unique().tolist() == [8323]
    out = p.out[2]
    rng = np.random.default_rng(0)
    layers = sorted(set(int(x) for x in rng.integers(0, w.batch, 4)))
    for b in layers:
        sl = slice(b, b + 1)
        attn_parity(d["q"][2][sl], d["K"][sl], d["V"][sl], d["N"][sl], d["len"][sl], out[sl], "bf16")


def test_many_units_use_the_prologue_path(cuda_lib):
    # more than 2048 (sequence, KV head) units: offsets come from the one-CTA prologue
    rng = np.random.default_rng(6)
    lengths = rng.integers(0, 300, (260, 8)).tolist()
    q, K, V, N, L = _case(rng, 260, 8, 4, 320, 128, lengths, garbage=False)
    out = _attn(q, K, V, N, L)
    attn_parity(q, K, V, N, L, out, "bf16")


def test_repeated_calls_on_one_workspace(cuda_lib):
    # the per-unit completion counters reset themselves: calls 2..4 equal call 1
    rng = np.random.default_rng(8)
    q, K, V, N, L = _case(rng, 2, 8, 4, 9000, 128, rng.integers(0, 9000, (2, 8)).tolist())
    cache = B.cache_desc(K)
    ws = B.new_workspace(B.decode_attn_workspace_bytes(cache, q.shape[1]))
    outs = []
    for _ in range(4):
        o = torch.empty((2, 32, 128), dtype=torch.bfloat16, device="cuda")
        B.decode_attn_logn(q, K, V, N, L, o, ws)
        outs.append(o)
    torch.cuda.synchronize()
    assert B.csmkv_device_status(ws) == 0
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    attn_parity(q, K, V, N, L, outs[0], "bf16")


@pytest.mark.parametrize("batch,h_kv,G,cap,D,dtype", [(2, 8, 4, 1024, 128, torch.bfloat16),
                                                       (3, 4, 7, 640, 64, torch.bfloat16),
                                                       (300, 8, 4, 72, 128, torch.bfloat16),   # > 2048 units
                                                       (2, 2, 2, 256, 128, torch.float32)])
def test_fused_step_matches_append_then_attention(cuda_lib, batch, h_kv, G, cap, D, dtype):
    """decode_step_logn = csm_append + decode_attn_logn, bit for bit: caches, lengths,
    outputs and the status word (a full unit is attended unchanged, CAPACITY recorded)."""
    rng = np.random.default_rng(batch * 100 + D)
    lengths = rng.integers(0, cap, (batch, h_kv))
    lengths[0, 0] = cap          # full: no append, CAPACITY
    lengths[-1, -1] = 0          # empty before the append
    q, K, V, N, L = _case(rng, batch, h_kv, G, cap, D, lengths.tolist(), dtype=dtype)
    kn = torch.randn(batch, h_kv, D, device="cuda").to(dtype)
    vn = torch.randn(batch, h_kv, D, device="cuda").to(dtype)
    K2, V2, N2, L2 = K.clone(), V.clone(), N.clone(), L.clone()
    cache = B.cache_desc(K)
    ws_a = B.new_workspace(B.csm_append_workspace_bytes())
    ws1 = B.new_workspace(B.decode_attn_workspace_bytes(cache, q.shape[1]))
    ws2 = B.new_workspace(B.decode_attn_workspace_bytes(cache, q.shape[1]))
    o1 = torch.empty(batch, h_kv * G, D, dtype=dtype, device="cuda")
    o2 = torch.empty_like(o1)
    B.csm_append(K, V, N, L, kn, vn, workspace=ws_a)
    B.decode_attn_logn(q, K, V, N, L, o1, ws1)
    for _ in range(2):  # the second call shows the per-call state resets (and appends again)
        B.decode_step_logn(q, kn, vn, K2, V2, N2, L2, o2, ws2)
        if _ == 0:
            torch.cuda.synchronize()
            assert B.csmkv_device_status(ws2) == 4  # CSMKV_ERR_CAPACITY
            for a, b in ((K, K2), (V, V2), (N, N2), (L, L2)):
                # NaN garbage past the lengths compares unequal to itself: compare bytes
                assert torch.equal(a.view(torch.uint8) if a.dtype != torch.int32 else a,
                                   b.view(torch.uint8) if b.dtype != torch.int32 else b)
            assert torch.equal(o1.view(torch.uint8), o2.view(torch.uint8))
            attn_parity(q, K2, V2, N2, L2, o2, "bf16" if dtype == torch.bfloat16 else "f32")
    torch.cuda.synchronize()
    assert B.csmkv_device_status(ws_a) == 4
    exp = np.minimum(lengths + 2, cap)
    assert np.array_equal(L2.cpu().numpy(), exp)
