"""The whole inference pipeline on the GPU (Algorithm 1) against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from online_kv_cache_chunked_gb300 import synth
from online_kv_cache_chunked_gb300.pipeline import Pipeline, final_lengths
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
