"""CSM compression on the GPU against the oracle (decisions, degrees, order, values)."""
import numpy as np
import pytest
import torch

from online_kv_cache_chunked_gb300 import binding as B
from online_kv_cache_chunked_gb300 import synth
from oracle import compare
from tests.gpu_helpers import gpu_round, log_near_ties, round_parity, snapshot, to64

pytestmark = pytest.mark.gpu


def _random_cache(rng, batch, h_kv, cap, d, dtype, lengths, rho=0.9, degrees=False):
    K = np.zeros((batch, h_kv, cap, d), np.float32)
    z = rng.standard_normal((batch, h_kv, d))
    for t in range(cap):
        z = rho * z + np.sqrt(1 - rho * rho) * rng.standard_normal((batch, h_kv, d))
        K[:, :, t] = z
    V = rng.standard_normal((batch, h_kv, cap, d)).astype(np.float32)
    N = rng.integers(1, 5, (batch, h_kv, cap)).astype(np.int32) if degrees else np.ones((batch, h_kv, cap), np.int32)
    L = np.array(lengths, np.int32).reshape(batch, h_kv)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    return (torch.from_numpy(K).to(tdt).cuda(), torch.from_numpy(V).to(tdt).cuda(),
            torch.from_numpy(N).cuda(), torch.from_numpy(L).cuda())


def test_tiny_f32_round(cuda_lib):
    w = synth.WORKLOADS["tiny_f32"]
    d = synth.cache_from_numpy(w, synth.make_numpy(w))
    st = round_parity(d["K"], d["V"], d["N"], d["len"], w.n1, w.n2, w.c, w.r_init, "f32")
    assert st["chunks"] == 2 * 15
    assert d["len"].cpu().tolist() == [[544, 544]]


TC_KERNELS = [B.CSM_KERNEL_TC_SPLIT]


@pytest.mark.parametrize("kernel", TC_KERNELS)
@pytest.mark.parametrize("D", [128, 64])
def test_tensor_core_rounds_lockstep(cuda_lib, D, kernel):
    rng = np.random.default_rng(D)
    n1, n2, c = 16, 64, 256
    lengths = [[80 + 5 * 256 + 17, 80 + 3 * 256, 79], [80 + 256 + 255, 1800, 80 + 256]]
    K, V, N, L = _random_cache(rng, 2, 3, 2048, D, "bf16", lengths, rho=0.93, degrees=True)
    for r, hm, sm in [(0.5, None, None), (0.45, [0, 1, 0], None), (0.4, None, [1, 0]), (0.1, None, None)]:
        round_parity(K, V, N, L, n1, n2, c, r, "bf16", head_mask=hm, seq_mask=sm, kernel=kernel)


@pytest.mark.parametrize("dtype,c,D", [("bf16", 8, 16), ("bf16", 64, 64), ("f32", 16, 32), ("f32", 64, 64),
                                       ("bf16", 256, 128), ("f32", 2, 8), ("bf16", 12, 8), ("f32", 256, 128)])
def test_cuda_core_path_shapes(cuda_lib, dtype, c, D):
    rng = np.random.default_rng(c * 1000 + D)
    n1, n2 = 3, 5
    cap = n1 + n2 + 7 * c + c + 16
    cap = (cap + 7) // 8 * 8
    lengths = [[cap - 3, n1 + n2 + 2 * c, n1 + n2 + c - 1, cap]]
    K, V, N, L = _random_cache(rng, 1, 4, cap, D, dtype, lengths, degrees=True)
    for r in (0.5, 0.25, 0.5):
        round_parity(K, V, N, L, n1, n2, c, r, dtype, kernel=1)


@pytest.mark.parametrize("kernel", TC_KERNELS)
def test_tensor_core_and_cuda_core_agree(cuda_lib, kernel):
    rng = np.random.default_rng(42)
    lengths = [[80 + 8 * 256 + 100] * 4]
    K, V, N, L = _random_cache(rng, 1, 4, 2304, 128, "bf16", lengths, rho=0.95)
    copies = [t.clone() for t in (K, V, N, L)]
    m1 = gpu_round(K, V, N, L, 16, 64, 256, 0.5, kernel=kernel)
    m2 = gpu_round(*copies, 16, 64, 256, 0.5, kernel=1)
    assert (m1 != m2).mean() < 1e-3  # the two fp32 tiles differ only in summation order
    assert torch.equal(L, copies[3])


@pytest.mark.parametrize("kernel", TC_KERNELS)
def test_edge_cases(cuda_lib, kernel):
    rng = np.random.default_rng(3)
    n1, n2, c = 16, 64, 256
    cap = 80 + 4 * 256 + 64
    lengths = [[0, 79, 80 + 255, 80 + 256, 80 + 2 * 256, cap]]  # empty, no middle, short middle, exact fits, full
    K, V, N, L = _random_cache(rng, 1, 6, cap, 128, "bf16", lengths)
    st = round_parity(K, V, N, L, n1, n2, c, 0.5, "bf16", kernel=kernel)
    assert st["chunks"] == 0 + 0 + 0 + 1 + 2 + 4
    # n1 = n2 = 0, and an r too small to merge anything (m = 0 is a no-op)
    K, V, N, L = _random_cache(rng, 1, 2, 1024, 128, "bf16", [[1024, 700]])
    round_parity(K, V, N, L, 0, 0, c, 0.5, "bf16", kernel=kernel)
    before = K.clone()
    round_parity(K, V, N, L, 0, 0, c, 0.001, "bf16", kernel=kernel)
    assert torch.equal(before, K)
    # every head masked
    round_parity(K, V, N, L, 0, 0, c, 0.5, "bf16", head_mask=[1, 1], kernel=kernel)


@pytest.mark.parametrize("kernel", TC_KERNELS)
def test_exact_ties_and_zero_keys(cuda_lib, kernel):
    # duplicated keys produce exact-cosine ties; zero keys have cosine 0 everywhere
    rng = np.random.default_rng(5)
    K, V, N, L = _random_cache(rng, 1, 2, 1088, 128, "bf16", [[1088, 1088]])
    Kc = K.clone()
    Kc[0, 0, 100:400] = Kc[0, 0, 100]
    Kc[0, 1, 300:420] = 0
    K.copy_(Kc)
    round_parity(K, V, N, L, 16, 64, 256, 0.5, "bf16", max_dev_frac=1.0, kernel=kernel)


def test_lockstep_16k_layer(cuda_lib):
    w = synth.WORKLOADS["llama_16k"]
    d = synth.cache_from_numpy(w, synth.make_numpy(w))
    from online_kv_cache_chunked_gb300.pipeline import plan
    rounds = plan(w)
    assert [(r.step, r.s_before[0], r.s_after[0]) for r in rounds] == [(0, 16384, 8320), (1, 8321, 4225),
                                                                      (2, 4226, 2178)]
    ws = B.new_workspace(B.csm_append_workspace_bytes())
    stats = []
    for k, rd in enumerate(rounds):
        if rd.step > 0:
            B.csm_append(d["K"], d["V"], d["N"], d["len"], d["k_dec"][rd.step - 1], d["v_dec"][rd.step - 1],
                         workspace=ws)
        stats.append(round_parity(d["K"], d["V"], d["N"], d["len"], w.n1, w.n2, w.c, rd.r, "bf16"))
    assert d["len"].cpu().unique().tolist() == [2178]
    print("16k lockstep:", stats)


@pytest.mark.parametrize("kernel", TC_KERNELS)
def test_lockstep_32k_batch4_progressive_outliers(cuda_lib, kernel):
    w = synth.WORKLOADS["llama_32k_b4"]
    d = synth.cache_from_numpy(w, synth.make_numpy(w))
    from online_kv_cache_chunked_gb300.pipeline import plan
    rounds = plan(w)
    assert [(r.step, r.m, r.s_before[0], r.s_after[0]) for r in rounds] == [
        (0, 128, 32768, 16512), (1, 115, 16513, 9153), (2, 102, 9154, 5584)]
    hm = d["head_mask"].cpu().numpy()
    assert hm.sum() == 1
    ws = B.new_workspace(B.csm_append_workspace_bytes())
    for rd in rounds:
        if rd.step > 0:
            B.csm_append(d["K"], d["V"], d["N"], d["len"], d["k_dec"][rd.step - 1], d["v_dec"][rd.step - 1],
                         workspace=ws)
        round_parity(d["K"], d["V"], d["N"], d["len"], w.n1, w.n2, w.c, rd.r, "bf16", head_mask=hm, kernel=kernel)
    Lh = d["len"].cpu().numpy()
    assert np.all(Lh[:, hm == 1] == 32768 + 2) and np.all(Lh[:, hm == 0] == 5584)


def _sampled_round(K, V, N, L, w, r, n_samples, rng):
    """Full-size round: decisions and values on sampled chunks, structure on every unit."""
    import oracle
    from oracle import compare

    BHu = K.shape[0] * K.shape[1]
    cap, D = K.shape[2], K.shape[3]
    m = B.csm_edges_per_chunk(r, w.c)
    preK, preV, preN, preL = K.clone(), V.clone(), N.clone(), L.clone()
    gm = gpu_round(K, V, N, L, w.n1, w.n2, w.c, r)
    Lp = preL.cpu().numpy().reshape(BHu)
    Lg = L.cpu().numpy().reshape(BHu)
    ch = np.array([oracle.num_chunks(int(s), w.n1, w.n2, w.c) for s in Lp])
    assert np.array_equal(Lg, Lp - ch * m)
    # every unit: sinks untouched, tail moved bit-exactly, degrees conserved
    Kf, Vf = K.view(BHu, cap, D), V.view(BHu, cap, D)
    pKf, pVf = preK.view(BHu, cap, D), preV.view(BHu, cap, D)
    Nf, pNf = N.view(BHu, cap), preN.view(BHu, cap)
    for u in range(BHu):
        s, s2, t0 = int(Lp[u]), int(Lg[u]), w.n1 + int(ch[u]) * w.c
        assert torch.equal(Kf[u, :w.n1], pKf[u, :w.n1])
        d0 = w.n1 + int(ch[u]) * (w.c - m)
        assert torch.equal(Kf[u, d0:s2], pKf[u, t0:s]) and torch.equal(Vf[u, d0:s2], pVf[u, t0:s])
        assert torch.equal(Nf[u, d0:s2], pNf[u, t0:s])
        assert int(Nf[u, :s2].sum()) == int(pNf[u, :s].sum())
    # sampled chunks: exact decisions (up to near-ties) and values
    picks = [(u, int(rng.integers(0, ch[u]))) for u in rng.integers(0, BHu, n_samples) if ch[u] > 0]
    picks += [(u, 0) for u in range(0, BHu, max(1, BHu // 8))] + [(u, int(ch[u]) - 1) for u in range(0, BHu, max(1, BHu // 8))]
    Kc = np.stack([to64(pKf[u, w.n1 + j * w.c:w.n1 + (j + 1) * w.c]) for u, j in picks])
    Vc = np.stack([to64(pVf[u, w.n1 + j * w.c:w.n1 + (j + 1) * w.c]) for u, j in picks])
    Nc = np.stack([pNf[u, w.n1 + j * w.c:w.n1 + (j + 1) * w.c].cpu().numpy() for u, j in picks])
    free = oracle.csm_chunks(Kc, Vc, Nc, m)
    g = np.stack([gm[u, j] for u, j in picks])
    dev = 0
    log = []
    for i in range(len(picks)):
        d_, f_ = compare.check_chunk_decisions(Kc[i], free["match"][i], free["sim"][i], g[i], m)
        assert f_ is None, f"{picks[i]}: {f_}"
        dev += int(d_)
        if d_:
            log += [dict(unit=int(picks[i][0]), chunk=picks[i][1], **r) for r in compare.deviation_records(
                free["match"][i], free["sim"][i], free["margin"][i], free["cut"][i], g[i])]
    log_near_ties(log, f"{w.name} sampled round r={r}")
    rep = oracle.csm_chunks(Kc, Vc, Nc, m, forced=g)
    for i, (u, j) in enumerate(picks):
        d0 = w.n1 + j * (w.c - m)
        for name, T, pre in (("K", Kf, Kc), ("V", Vf, Vc)):
            got = to64(T[u, d0:d0 + w.c - m])
            ref = rep[name][i]
            mrg = rep["merged"][i].astype(bool)
            assert np.array_equal(got[~mrg], pre[i][rep["origin"][i][~mrg]])
            tol = compare.value_tol(ref, "bf16", pre[i])
            assert np.all(np.abs(got - ref)[mrg] <= tol[mrg])
        assert np.array_equal(Nf[u, d0:d0 + w.c - m].cpu().numpy(), rep["N"][i])
    return dict(sampled=len(picks), deviating=dev)


def test_full_64k_32_layers_sampled(cuda_lib):
    w = synth.WORKLOADS["llama_64k_32l"]
    d = synth.make_device(w)
    rng = np.random.default_rng(0)
    ws = B.new_workspace(B.csm_append_workspace_bytes())
    from online_kv_cache_chunked_gb300.pipeline import plan
    for rd in plan(w):
        if rd.step > 0:
            B.csm_append(d["K"], d["V"], d["N"], d["len"], d["k_dec"][rd.step - 1], d["v_dec"][rd.step - 1],
                         workspace=ws)
        print(_sampled_round(d["K"], d["V"], d["N"], d["len"], w, rd.r, 256, rng))
    assert d["len"].cpu().unique().tolist() == [8322]


def test_full_ragged_batch_sampled(cuda_lib):
    w = synth.WORKLOADS["qwen2_ragged"]
    d = synth.make_device(w)
    print(_sampled_round(d["K"], d["V"], d["N"], d["len"], w, 0.5, 256, np.random.default_rng(1)))


def test_timeout_path_reports_and_recovers(cuda_lib):
    rng = np.random.default_rng(9)
    K, V, N, L = _random_cache(rng, 1, 2, 2304, 128, "bf16", [[2304, 2304]])
    cache = B.cache_desc(K)
    ws = B.new_workspace(B.csm_workspace_bytes(cache, 16, 64, 256))
    B.csm_compress_ex(K, V, N, L, 16, 64, 256, 0.5, wait_timeout_ns=20_000_000, withhold_signals=1, workspace=ws)
    torch.cuda.synchronize()
    assert B.csmkv_device_status(ws) == 6  # CSMKV_ERR_TIMEOUT
    B.csmkv_clear_status(ws)
    assert B.csmkv_device_status(ws) == 0
    # the context is still healthy: a normal round on a fresh cache passes parity
    K, V, N, L = _random_cache(rng, 1, 2, 2304, 128, "bf16", [[2304, 2000]])
    round_parity(K, V, N, L, 16, 64, 256, 0.5, "bf16")


@pytest.mark.parametrize("kernel", [B.CSM_KERNEL_TC_SPLIT, B.CSM_KERNEL_SIMT])
def test_budget_exact_rounds(cuda_lib, kernel):
    """Rounds capped per sequence at the oldest k chunks: the rest of each cache moves
    down unchanged (as tail pieces, possibly many), decisions and values as the oracle."""
    rng = np.random.default_rng(11 + kernel)
    n1, n2, c = 16, 64, 256
    lengths = [[80 + 9 * 256 + 77] * 3, [80 + 4 * 256 + 5] * 3, [80 + 7 * 256] * 3]
    K, V, N, L = _random_cache(rng, 3, 3, 2688, 128, "bf16", lengths, rho=0.93, degrees=True)
    for r, lim in [(0.5, [2, 0, 7]), (0.45, [1, 3, 100]), (0.5, [4, 1, -1])]:
        round_parity(K, V, N, L, n1, n2, c, r, "bf16", kernel=kernel, limits=lim)


@pytest.mark.parametrize("kernel", [B.CSM_KERNEL_TC_SPLIT, B.CSM_KERNEL_SIMT])
def test_many_short_units(cuda_lib, kernel):
    """3000 (sequence, head) units of 0-4 chunks each: the prologue walks more units
    than it has threads, the ticket space is wide and mostly tail pieces. Lengths and
    degree sums on every unit; on sampled units the device's merge sets against
    the free-running oracle, then the state against the oracle replaying the
    device's decisions."""
    import oracle
    rng = np.random.default_rng(17 + kernel)
    batch, h_kv, cap, D, n1, n2, c, m = 750, 4, 1104, 128, 16, 64, 256, 128
    lengths = rng.integers(0, cap + 1, (batch, h_kv))
    K, V, N, L = _random_cache(rng, batch, h_kv, cap, D, "bf16", lengths.tolist(), rho=0.9, degrees=True)
    seq_on = (rng.random(batch) < 0.8).astype(np.uint8)
    K0, V0, N0, L0 = K.clone(), V.clone(), N.clone(), L.clone()
    gm = gpu_round(K, V, N, L, n1, n2, c, 0.5, kernel=kernel, seq_mask=seq_on)
    BH = batch * h_kv
    s_pre = L0.view(BH).cpu().numpy()
    s_post = L.view(BH).cpu().numpy()
    rows = torch.arange(cap, device="cuda")[None, :]
    sum_pre = (N0.view(BH, cap) * (rows < L0.view(BH, 1))).sum(dim=1).cpu().numpy()
    sum_post = (N.view(BH, cap) * (rows < L.view(BH, 1))).sum(dim=1).cpu().numpy()
    for u in range(BH):
        s = int(s_pre[u])
        want = s - oracle.num_chunks(s, n1, n2, c) * m if seq_on[u // h_kv] else s
        assert int(s_post[u]) == want, u
    assert np.array_equal(sum_pre, sum_post)
    Kf, Vf, Nf = K.view(BH, cap, D), V.view(BH, cap, D), N.view(BH, cap)
    K0f, V0f, N0f = K0.view(BH, cap, D), V0.view(BH, cap, D), N0.view(BH, cap)
    log = []
    for u in rng.choice(BH, 48, replace=False):
        s, got = int(s_pre[u]), int(s_post[u])
        if got == s:  # masked out or no full chunk: untouched
            assert torch.equal(Kf[u, :s], K0f[u, :s]) and torch.equal(Vf[u, :s], V0f[u, :s])
            continue
        pK, pV, pN = to64(K0f[u:u + 1]), to64(V0f[u:u + 1]), N0f[u:u + 1].cpu().numpy()
        s_arr = np.array([s], np.int32)
        # the device's merge sets against the free-running oracle first ...
        free = oracle.csm_round(pK, pV, pN, s_arr, n1, n2, c, m)
        nch = np.array([oracle.num_chunks(s, n1, n2, c)])
        dev_log = []
        _, fails = compare.check_round(pK, free, gm[u:u + 1], nch, m, n1, c, log=dev_log)
        assert not fails, f"unit {u}: " + "; ".join(fails[:5])
        log += [dict(r, unit=int(u)) for r in dev_log]
        # ... then the state against the oracle replaying the device's decisions
        forced = np.where(gm[u:u + 1] >= -1, gm[u:u + 1], -1)
        ref = oracle.csm_round(pK, pV, pN, s_arr, n1, n2, c, m, forced=forced)
        assert int(ref["len"][0]) == got
        assert np.array_equal(ref["N"][0, :got], Nf[u, :got].cpu().numpy())
        for name, T, src in (("K", Kf, pK), ("V", Vf, pV)):
            r = ref[name][0, :got]
            assert np.all(np.abs(r - to64(T[u, :got])) <= compare.value_tol(r, "bf16", src[0, :s]))
    log_near_ties(log, f"many short units kernel={kernel}")


@pytest.mark.parametrize("D", [128, 64])
def test_head_slices_match_whole_cache(cuda_lib, D):
    """A range of one sequence row's KV heads, passed as its own cache (a contiguous
    [1, heads, cap, d] view), compresses to the same bytes as one call over the whole
    cache: every (sequence, KV head) cache is a separate unit ([Chelsea] §三 分块软匹配算法)."""
    rng = np.random.default_rng(77 + D)
    n1, n2, c, r = 16, 64, 256, 0.45
    lengths = [[80 + 5 * 256 + 17, 80 + 3 * 256, 1800, 79], [80 + 256 + 255, 1800, 80 + 256, 1500]]
    K, V, N, L = _random_cache(rng, 2, 4, 2048, D, "bf16", lengths, rho=0.93, degrees=True)
    hm = torch.tensor([0, 1, 0, 0], dtype=torch.uint8, device="cuda")
    sm = torch.tensor([1, 1], dtype=torch.uint8, device="cuda")
    whole = [t.clone() for t in (K, V, N, L)]
    ws = B.new_workspace(B.csm_workspace_bytes(B.cache_desc(K), n1, n2, c), "cuda")
    B.csm_compress_ex(*whole, n1, n2, c, r, hm, sm, workspace=ws)
    parts = [t.clone() for t in (K, V, N, L)]
    for b, h0, h1 in [(0, 0, 1), (0, 1, 4), (1, 0, 2), (1, 2, 4)]:
        Kp, Vp, Np, Lp = (t[b:b + 1, h0:h1] for t in parts)
        B.csm_compress_ex(Kp, Vp, Np, Lp, n1, n2, c, r, hm[h0:h1], sm[b:b + 1], workspace=ws)
    torch.cuda.synchronize()
    assert B.csmkv_device_status(ws) == 0
    assert torch.equal(parts[3], whole[3])
    for b in range(2):
        for h in range(4):
            s = int(whole[3][b, h])
            assert torch.equal(parts[0][b, h, :s].view(torch.int16), whole[0][b, h, :s].view(torch.int16)), (b, h)
            assert torch.equal(parts[1][b, h, :s].view(torch.int16), whole[1][b, h, :s].view(torch.int16)), (b, h)
            assert torch.equal(parts[2][b, h, :s], whole[2][b, h, :s]), (b, h)
