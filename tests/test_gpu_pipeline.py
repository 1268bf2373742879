"""The whole inference pipeline on the GPU (Algorithm 1) against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from online_kv_cache_chunked_gb300 import synth
from online_kv_cache_chunked_gb300.pipeline import Pipeline, final_lengths
from online_kv_cache_chunked_gb300 import binding as B
from tests.gpu_helpers import attn_parity, to64

pytestmark = pytest.mark.gpu


def test_tiny_f32_free_running(cuda_lib):
    """One forced round and one decode step, compared with a free-running oracle."""
    w = synth.WORKLOADS["tiny_f32"]
    host = synth.make_numpy(w)
    d = synth.cache_from_numpy(w, host)
    BH = w.batch * w.h_kv
    pre = dict(K=to64(d["K"]).reshape(BH, w.cap, w.d), V=to64(d["V"]).reshape(BH, w.cap, w.d),
               N=d["N"].cpu().numpy().reshape(BH, w.cap), L=d["len"].cpu().numpy().reshape(BH))
    p = Pipeline(w, d)
    p.run()
    torch.cuda.synchronize()
    o = oracle.csm_round(pre["K"], pre["V"], pre["N"], pre["L"], w.n1, w.n2, w.c, 32)
    K, V, N, L, _ = oracle.append(o["K"], o["V"], o["N"], o["len"], to64(d["k_dec"][0]).reshape(BH, w.d),
                                  to64(d["v_dec"][0]).reshape(BH, w.d))
    ref = oracle.decode_attn_logn(to64(d["q"][0]), K.reshape(1, 2, w.cap, w.d), V.reshape(1, 2, w.cap, w.d),
                                  N.reshape(1, 2, w.cap), L.reshape(1, 2), w.h_q)
    assert L.tolist() == [545, 545]
    err = float(np.abs(to64(p.out[0]) - ref).max())
    assert err <= 1e-5, err


def test_16k_layer_1000_steps(cuda_lib):
    w = synth.WORKLOADS["llama_16k"]
    d = synth.cache_from_numpy(w, synth.make_numpy(w))
    p = Pipeline(w, d)
    checks = {1, 2, 3, 100, 500, w.steps}
    errs = {}

    def hook(kind, what, before):
        if kind == "attn" and not before and what in checks:
            i = what
            torch.cuda.synchronize()
            errs[i] = attn_parity(d["q"][i - 1], d["K"], d["V"], d["N"], d["len"], p.out[i - 1], "bf16")

    p.run(hook=hook)
    torch.cuda.synchronize()
    assert np.array_equal(d["len"].cpu().numpy(), final_lengths(w))
    assert int(d["N"][0, 0, :int(d["len"][0, 0])].sum()) == 16384 + w.steps
    print("attention errors at sampled steps:", errs)


def test_ragged_batch_pipeline_lengths(cuda_lib):
    w = synth.scaled(synth.WORKLOADS["qwen2_ragged"], steps=40)
    d = synth.make_device(w)
    p = Pipeline(w, d)
    p.run()
    torch.cuda.synchronize()
    assert np.array_equal(d["len"].cpu().numpy(), final_lengths(w))
    b = 5
    attn_parity(d["q"][-1][b:b + 1], d["K"][b:b + 1], d["V"][b:b + 1], d["N"][b:b + 1], d["len"][b:b + 1],
                p.out[-1][b:b + 1], "bf16")


def _attention_at_steps_against_oracle(w, d, checks):
    """Runs the workload in the configuration the benchmark times (prefill rounds,
    then the natively issued loop of fused append + attention steps with the planned
    rounds) and, at every step i in `checks`, compares all query heads' outputs with
    the oracle: the cache as it stood before step i, plus that step's appended token,
    through oracle.append and oracle.decode_attn_logn. Returns the errors."""
    p = Pipeline(w, d)
    p.compress_at(0)
    done, errs = 0, {}
    for i in sorted(checks):
        if i - 1 > done:
            p.decode_native(done + 1, i - 1 - done)
        torch.cuda.synchronize()
        L = d["len"].cpu().numpy()
        top = int(L.max()) + 1
        BH = w.batch * w.h_kv
        pre = [to64(d["K"][:, :, :top]).reshape(BH, top, w.d), to64(d["V"][:, :, :top]).reshape(BH, top, w.d),
               d["N"][:, :, :top].cpu().numpy().reshape(BH, top), L.reshape(BH)]
        p.decode_native(i, 1)
        done = i
        torch.cuda.synchronize()
        K, V, N, Ln, full = oracle.append(*pre, to64(d["k_dec"][i - 1]).reshape(BH, w.d),
                                          to64(d["v_dec"][i - 1]).reshape(BH, w.d))
        assert full == 0
        ref = oracle.decode_attn_logn(to64(d["q"][i - 1]), K.reshape(w.batch, w.h_kv, top, w.d),
                                      V.reshape(w.batch, w.h_kv, top, w.d), N.reshape(w.batch, w.h_kv, top),
                                      Ln.reshape(w.batch, w.h_kv), w.h_q)
        got = to64(p.out[i - 1])
        assert np.isfinite(got).all()
        errs[i] = float(np.abs(got - ref).max())
        assert errs[i] <= 2e-2, (i, errs[i])
    if done < w.steps:
        p.decode_native(done + 1, w.steps - done)
    torch.cuda.synchronize()
    for ws in (p.ws_csm, p.ws_app, p.ws_att):
        assert B.csmkv_device_status(ws) == 0
    assert np.array_equal(d["len"].cpu().numpy(), final_lengths(w))
    return errs


def test_32k_batch4_attention_against_oracle(cuda_lib):
    """The 32K x batch-4 workload at full size: three progressive rounds (m = 128, 115,
    102) on 7 of 8 KV heads, the outlier head left at ~33K tokens, then 1000 fused decode
    steps; every query head checked against the oracle at steps 1, 2, 3, 100 and 1000
    (steps 1 and 2 also fire rounds after their attention)."""
    w = synth.WORKLOADS["llama_32k_b4"]
    d = synth.make_device(w)
    hm = d["head_mask"].cpu().numpy()
    assert hm.sum() == 1
    errs = _attention_at_steps_against_oracle(w, d, {1, 2, 3, 100, w.steps})
    L = d["len"].cpu().numpy()
    assert np.all(L[:, hm == 1] == 32768 + w.steps) and np.all(L[:, hm == 0] == 5584 + w.steps - 2)
    print("32k x4 attention errors at sampled steps:", errs)


def test_ragged_batch_attention_against_oracle(cuda_lib):
    """The ragged 16-sequence batch at full size, every query head at steps 1, 2, 3, 256
    and 512 (the last)."""
    w = synth.WORKLOADS["qwen2_ragged"]
    d = synth.make_device(w)
    print("ragged attention errors:", _attention_at_steps_against_oracle(w, d, {1, 2, 3, 256, w.steps}))


@pytest.mark.parametrize("name,steps", [("llama_32k_b4", 12), ("qwen2_ragged", 40)])
def test_native_loop_matches_per_call_loop(cuda_lib, name, steps):
    """The library-issued decode loop gives bit-identical caches and outputs to the
    same calls made one by one through the binding (rounds at decode steps included)."""
    from online_kv_cache_chunked_gb300 import binding as B
    w = synth.scaled(synth.WORKLOADS[name], steps=steps)
    d1 = synth.make_device(w)
    d2 = {k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in d1.items()}
    p1, p2 = Pipeline(w, d1), Pipeline(w, d2)
    assert any(rd.step >= 1 for rd in p1.rounds)
    p1.run()
    stream = torch.cuda.current_stream()
    ev_att = [torch.cuda.Event(enable_timing=True) for _ in range(2 * w.steps)]
    ev_csm = [torch.cuda.Event(enable_timing=True) for _ in range(2 * len(p2.decode_plan()))]
    for e in ev_att + ev_csm:
        e.record(stream)
    flush = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    p2.run_native(attn_events=ev_att, csm_events=ev_csm, l2_flush=flush)
    torch.cuda.synchronize()
    for ws in (p2.ws_csm, p2.ws_app, p2.ws_att):
        assert B.csmkv_device_status(ws) == 0
    for k in ("K", "V", "N", "len"):
        assert torch.equal(d1[k], d2[k]), k
    assert torch.equal(p1.out, p2.out)
    assert np.array_equal(d2["len"].cpu().numpy(), final_lengths(w))
    assert all(ev_att[2 * i].elapsed_time(ev_att[2 * i + 1]) > 0 for i in range(w.steps))
    assert all(ev_csm[2 * i].elapsed_time(ev_csm[2 * i + 1]) > 0 for i in range(len(ev_csm) // 2))


def test_decode_loop_replays_from_a_cuda_graph(cuda_lib):
    """The library-issued decode loop (appends, attention, the rounds fired at steps 1
    and 2) only enqueues device work, so it can be captured into one CUDA graph; a
    replay gives the same caches and outputs, bit for bit, as the loop run directly."""
    from online_kv_cache_chunked_gb300 import binding as B
    w = synth.scaled(synth.WORKLOADS["llama_32k_b4"], steps=8)
    d1 = synth.make_device(w)
    d2 = {k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in d1.items()}
    p1, p2 = Pipeline(w, d1), Pipeline(w, d2)
    assert [rd.step for rd in p1.rounds] == [0, 1, 2]
    p1.run_native()
    p2.compress_at(0)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        B.csm_decode_run(d2["K"], d2["V"], d2["N"], d2["len"], d2["q"], d2["k_dec"], d2["v_dec"], p2.out, w.n1,
                         w.n2, w.c, rounds=p2.decode_plan(), head_mask=p2.head_mask, ws_csm=p2.ws_csm,
                         ws_append=p2.ws_app, ws_attn=p2.ws_att, steps=w.steps)
    g.replay()
    torch.cuda.synchronize()
    for ws in (p2.ws_csm, p2.ws_app, p2.ws_att):
        assert B.csmkv_device_status(ws) == 0
    for k in ("K", "V", "N", "len"):
        assert torch.equal(d1[k], d2[k]), k
    assert torch.equal(p1.out, p2.out)
    assert np.array_equal(d2["len"].cpu().numpy(), final_lengths(w))


def test_budget_exact_16k_layer_in_lockstep(cuda_lib):
    """Budget-exact schedule on the 16K layer: every round (k = ceil((s - B) / m) oldest
    chunks) checked against the oracle on the device's own pre-round state, lengths
    against the host plan, attention against the oracle at sampled steps."""
    from online_kv_cache_chunked_gb300 import binding as B
    from oracle import schedule as S
    from tests.gpu_helpers import round_parity
    w = synth.scaled(synth.WORKLOADS["llama_16k"], budget_exact=True, steps=300)
    d = synth.cache_from_numpy(w, synth.make_numpy(w))
    p = Pipeline(w, d)
    want = S.plan_budget_exact(16384, w.R, w.steps, w.g, w.n1, w.n2, w.c, w.r_init)
    assert [(rd.step, rd.limits[0], rd.s_after[0]) for rd in p.rounds] == [(st, k, s2) for st, _, _, _, k, s2 in want]
    ws = B.new_workspace(B.csm_append_workspace_bytes())
    by_step = {rd.step: rd for rd in p.rounds}
    checks = {1, 85, 86, 213, 300}
    for step in range(0, w.steps + 1):
        if step > 0:
            B.csm_append(d["K"], d["V"], d["N"], d["len"], d["k_dec"][step - 1], d["v_dec"][step - 1], workspace=ws)
            if step in checks:
                B.decode_attn_logn(d["q"][step - 1], d["K"], d["V"], d["N"], d["len"], p.out[step - 1], p.ws_att)
                torch.cuda.synchronize()
                attn_parity(d["q"][step - 1], d["K"], d["V"], d["N"], d["len"], p.out[step - 1], "bf16")
        if step in by_step:
            rd = by_step[step]
            round_parity(d["K"], d["V"], d["N"], d["len"], w.n1, w.n2, w.c, rd.r, "bf16", limits=list(rd.limits))
    assert np.array_equal(d["len"].cpu().numpy(), final_lengths(w))
    assert int(d["N"][0, 0, :int(d["len"][0, 0])].sum()) == 16384 + w.steps


def test_budget_exact_native_loop_matches_per_call(cuda_lib):
    w = synth.scaled(synth.WORKLOADS["llama_32k_b4"], budget_exact=True, steps=200)
    d1 = synth.make_device(w)
    d2 = {k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in d1.items()}
    p1, p2 = Pipeline(w, d1), Pipeline(w, d2)
    assert sum(1 for rd in p1.rounds if rd.step >= 1) >= 3
    p1.run()
    p2.run_native()
    torch.cuda.synchronize()
    for k in ("K", "V", "N", "len"):
        assert torch.equal(d1[k], d2[k]), k
    assert torch.equal(p1.out, p2.out)
    assert np.array_equal(d2["len"].cpu().numpy(), final_lengths(w))
