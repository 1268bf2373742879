"""The paged (block-table) layout on the GPU [CentroidKV 技术摘要, 结果: serving
inside vLLM's paged KV cache]: every entry point gives, on a paged copy of a
cache, exactly what it gives on the dense cache (same decisions, caches and
outputs bit for bit), and the results match the oracle, which stays dense
(pages gathered back on the host)."""
import numpy as np
import pytest
import torch

import oracle
from online_kv_cache_chunked_gb300 import binding as B
from online_kv_cache_chunked_gb300 import paged, synth
from online_kv_cache_chunked_gb300.pipeline import Pipeline, final_lengths
from oracle import compare
from tests.gpu_helpers import attn_parity, gpu_round, log_near_ties, snapshot, skip_vector, to64

pytestmark = pytest.mark.gpu


def _dense_case(seed, batch, h_kv, cap, D, lengths, rho=0.93):
    g = torch.Generator(device="cuda").manual_seed(seed)
    z = torch.randn(batch, h_kv, D, generator=g, device="cuda")
    K = torch.empty(batch, h_kv, cap, D, device="cuda")
    eps = torch.randn(batch, h_kv, cap, D, generator=g, device="cuda")
    for t in range(cap):  # correlated keys: close similarities, real ranking work
        z = rho * z + (1 - rho * rho) ** 0.5 * eps[:, :, t]
        K[:, :, t] = z
    K = K.to(torch.bfloat16)
    V = torch.randn(batch, h_kv, cap, D, generator=g, device="cuda").to(torch.bfloat16)
    N = torch.randint(1, 6, (batch, h_kv, cap), generator=g, device="cuda", dtype=torch.int32)
    L = torch.tensor(lengths, dtype=torch.int32, device="cuda").view(batch, h_kv)
    return K, V, N, L


def _assert_same_cache(kv, K, V, N, L):
    K2, V2, N2 = paged.to_dense(kv)
    for b in range(K.shape[0]):
        for h in range(K.shape[1]):
            s = int(L[b, h])
            assert torch.equal(K2[b, h, :s].view(torch.int16), K[b, h, :s].view(torch.int16)), (b, h)
            assert torch.equal(V2[b, h, :s].view(torch.int16), V[b, h, :s].view(torch.int16)), (b, h)
            assert torch.equal(N2[b, h, :s], N[b, h, :s]), (b, h)


@pytest.mark.parametrize("page_rows,D,n1", [(256, 128, 16), (64, 128, 16), (512, 64, 16), (64, 128, 48),
                                             (256, 128, 10)])
def test_paged_rounds_equal_dense_rounds_and_the_oracle(cuda_lib, page_rows, D, n1):
    """n1 a multiple of 16: chunk rows by TMA in 16-row page groups; n1 = 10: row gathers."""
    n2, c = 64, 256
    lengths = [[80 + 5 * 256 + 17, 80 + 3 * 256, 79, 2040], [80 + 256 + 255, 1800, 80 + 256, 0]]
    K, V, N, L = _dense_case(page_rows + D, 2, 4, 2048, D, lengths)
    kv = paged.to_paged(K, V, N, page_rows, spare_pages=7, seed=page_rows)
    Lp = L.clone()
    cache = kv.cache()
    ws = B.new_workspace(B.csm_workspace_bytes(cache, n1, n2, c))
    maxch = B.csm_max_chunks(cache, n1, n2, c)
    for r, hm, sm in [(0.5, None, None), (0.45, [0, 1, 0, 0], None), (0.4, None, [1, 0]), (0.1, None, None)]:
        K2, V2, N2 = paged.to_dense(kv)
        pre = snapshot(K2, V2, N2, Lp)
        hmd = None if hm is None else torch.tensor(hm, dtype=torch.uint8, device="cuda")
        smd = None if sm is None else torch.tensor(sm, dtype=torch.uint8, device="cuda")
        gm_dense = gpu_round(K, V, N, L, n1, n2, c, r, hm, sm, kernel=B.CSM_KERNEL_TC_SPLIT)
        match = torch.full((8, max(1, maxch), c // 2), -2, dtype=torch.int32, device="cuda")
        B.csm_compress_paged(kv, Lp, n1, n2, c, r, head_mask=hmd, seq_mask=smd, match_out=match, workspace=ws)
        torch.cuda.synchronize()
        assert B.csmkv_device_status(ws) == 0
        gm = match.cpu().numpy()
        assert np.array_equal(gm, gm_dense)  # the same decisions as on the dense layout ...
        assert torch.equal(Lp, L)
        _assert_same_cache(kv, K, V, N, L)   # ... and the same cache, bit for bit
        # and against the oracle on the gathered pre-round state
        m = B.csm_edges_per_chunk(r, c)
        sk = skip_vector(2, 4, hm, sm)
        free = oracle.csm_round(pre["K"], pre["V"], pre["N"], pre["len"], n1, n2, c, m, skip=sk)
        nch = np.array([0 if sk[u] else oracle.num_chunks(int(pre["len"][u]), n1, n2, c) for u in range(8)])
        log = []
        _, fails = compare.check_round(pre["K"], free, gm, nch, m, n1, c, log=log)
        log_near_ties(log, f"paged round P={page_rows}")
        assert not fails, fails[:3]
        rep = oracle.csm_round(pre["K"], pre["V"], pre["N"], pre["len"], n1, n2, c, m, skip=sk,
                               forced=np.where(gm >= -1, gm, -1))
        fails, _ = compare.compare_state(rep, pre, snapshot(*paged.to_dense(kv), Lp), "bf16")
        assert not fails, fails[:3]


@pytest.mark.parametrize("page_rows", [64, 256])
def test_paged_append_attention_and_fused_step_equal_dense(cuda_lib, page_rows):
    batch, h_kv, G, cap, D = 2, 8, 4, 4096, 128
    rng = np.random.default_rng(page_rows)
    lengths = rng.integers(0, cap, (batch, h_kv))
    lengths[0, 0], lengths[1, 7] = cap, 0  # a full unit (CAPACITY) and an empty one
    K, V, N, L = _dense_case(7, batch, h_kv, cap, D, lengths.tolist())
    kv = paged.to_paged(K, V, N, page_rows, spare_pages=3, seed=11)
    Lp = L.clone()
    q = torch.randn(batch, h_kv * G, D, device="cuda").to(torch.bfloat16)
    kn = torch.randn(batch, h_kv, D, device="cuda").to(torch.bfloat16)
    vn = torch.randn(batch, h_kv, D, device="cuda").to(torch.bfloat16)
    cache = kv.cache()
    wsd = B.new_workspace(B.decode_attn_workspace_bytes(cache, batch * 0 + h_kv * G))
    wsp = B.new_workspace(B.decode_attn_workspace_bytes(cache, h_kv * G))
    o1 = torch.empty(batch, h_kv * G, D, dtype=torch.bfloat16, device="cuda")
    o2 = torch.empty_like(o1)
    B.decode_attn_logn(q, K, V, N, L, o1, wsd)
    B.decode_attn_logn_paged(q, kv, Lp, o2, wsp)
    torch.cuda.synchronize()
    assert B.csmkv_device_status(wsp) == 0
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    for _ in range(2):  # fused steps (append + attention), twice
        B.decode_step_logn(q, kn, vn, K, V, N, L, o1, wsd)
        B.decode_step_logn_paged(q, kn, vn, kv, Lp, o2, wsp)
        torch.cuda.synchronize()
        assert B.csmkv_device_status(wsp) == 4  # the full unit: CSMKV_ERR_CAPACITY, as on the dense layout
        B.csmkv_clear_status(wsp)
        assert torch.equal(L, Lp)
        assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
        _assert_same_cache(kv, K, V, N, L)
    attn_parity(q, *paged.to_dense(kv), Lp, o2, "bf16")  # the last fused step's output against the oracle
    wsa = B.new_workspace(B.csm_append_workspace_bytes())
    B.csm_append(K, V, N, L, kn, vn, workspace=wsa)
    B.csm_append_paged(kv, Lp, kn, vn, workspace=wsa)
    torch.cuda.synchronize()
    assert torch.equal(L, Lp)
    _assert_same_cache(kv, K, V, N, L)


def test_ragged_batch_paged_pipeline_equals_dense(cuda_lib):
    """The ragged 16-sequence batch at full size in 256-row pages scattered over the
    pool: prefill round and 40 natively issued fused steps with their rounds give the
    same caches and outputs as the dense layout, and the attention matches the oracle."""
    w = synth.scaled(synth.WORKLOADS["qwen2_ragged"], steps=40)
    d1 = synth.make_device(w)
    d2 = {k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in d1.items()}
    kv = paged.to_paged(d2["K"], d2["V"], d2["N"], 256, spare_pages=100, seed=5)
    d2["K"] = d2["V"] = d2["N"] = None
    torch.cuda.empty_cache()
    p1, p2 = Pipeline(w, d1), Pipeline(w, d2, paged=kv)
    p1.run_native()
    p2.run_native()
    torch.cuda.synchronize()
    for ws in (p2.ws_csm, p2.ws_att):
        assert B.csmkv_device_status(ws) == 0
    assert torch.equal(d1["len"], d2["len"])
    assert np.array_equal(d2["len"].cpu().numpy(), final_lengths(w))
    assert torch.equal(p1.out.view(torch.int16), p2.out.view(torch.int16))
    _assert_same_cache(kv, d1["K"], d1["V"], d1["N"], d1["len"])


def test_block_table_entries_outside_the_pool_are_reported_not_followed(cuda_lib):
    """A table entry beyond the pool is never dereferenced: loads of that page read
    zeros, writes through it are skipped, CSMKV_ERR_ARG is recorded, and the other
    units are unaffected."""
    batch, h_kv, G, cap, D = 1, 4, 4, 1024, 128
    K, V, N, L = _dense_case(3, batch, h_kv, cap, D, [[1000, 700, 512, 300]])
    kv = paged.to_paged(K, V, N, 256, seed=2)
    kv.table[1, 1] = kv.num_pages + 5   # unit 1, rows 256..511
    q = torch.randn(batch, h_kv * G, D, device="cuda").to(torch.bfloat16)
    ws = B.new_workspace(B.decode_attn_workspace_bytes(kv.cache(), h_kv * G))
    out = torch.empty(batch, h_kv * G, D, dtype=torch.bfloat16, device="cuda")
    ref = torch.empty_like(out)
    wsd = B.new_workspace(B.decode_attn_workspace_bytes(B.cache_desc(K), h_kv * G))
    B.decode_attn_logn(q, K, V, N, L, ref, wsd)
    B.decode_attn_logn_paged(q, kv, L, out, ws)
    torch.cuda.synchronize()
    assert B.csmkv_device_status(ws) == 1  # CSMKV_ERR_ARG
    keep = [0, 2, 3]
    o, r = out.view(batch, h_kv, G, D), ref.view(batch, h_kv, G, D)
    assert torch.equal(o[:, keep].view(torch.int16), r[:, keep].view(torch.int16))
    wsa = B.new_workspace(B.csm_append_workspace_bytes())
    L2 = torch.tensor([[1000, 300, 512, 300]], dtype=torch.int32, device="cuda")  # unit 1 appends into the bad page
    kn = torch.randn(batch, h_kv, D, device="cuda").to(torch.bfloat16)
    B.csm_append_paged(kv, L2, kn, kn, workspace=wsa)
    torch.cuda.synchronize()
    assert B.csmkv_device_status(wsa) == 1
    assert L2.tolist() == [[1001, 300, 513, 301]]  # nothing written, length unchanged for unit 1
