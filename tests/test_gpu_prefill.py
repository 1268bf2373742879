"""GPU parity of prefill attention and of the first CSM round fused into it
([Chelsea] §三 算法流程, Algorithm 1: prefill O = FlashAttn(Q, K, V), then the first
round). The attention is compared with the oracle's causal attention; the second
cache the fused call writes is compared byte for byte with the standalone round
(csm_compress) on the same prompt, whose own oracle parity is checked here too."""
import numpy as np
import pytest
import torch

import oracle
from oracle import compare
from online_kv_cache_chunked_gb300 import binding as B
from tests.gpu_helpers import round_parity, to64

pytestmark = pytest.mark.gpu

D = 128
SENTINEL = 12352.0  # exact in bf16


def _prompt(seed, batch, h_kv, G, n, cap, seq_len=None, dup=0.0):
    """Seeded bf16 prompt: q [batch, h_kv*G, n, D], cache K, V [batch, h_kv, cap, D]
    whose rows at or past each sequence's prompt length hold NaN (they must never
    be read). dup > 0 makes neighbouring keys similar, so that rounds merge real pairs."""
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(batch, h_kv * G, n, D, generator=g)
    K = torch.randn(batch, h_kv, cap, D, generator=g)
    if dup > 0:
        K[:, :, 1::2] = (1 - dup) * K[:, :, 1::2] + dup * K[:, :, 0::2][:, :, : K[:, :, 1::2].shape[2]]
    V = torch.randn(batch, h_kv, cap, D, generator=g)
    lens = [n] * batch if seq_len is None else list(seq_len)
    for b, s in enumerate(lens):
        K[b, :, s:] = float("nan")
        V[b, :, s:] = float("nan")
    q, K, V = (t.to(torch.bfloat16).cuda() for t in (q, K, V))
    sl = None if seq_len is None else torch.tensor(lens, dtype=torch.int32, device="cuda")
    return q, K.contiguous(), V.contiguous(), lens, sl


def _attention_check(q, K, V, lens, out, n):
    """Every written row against the oracle; rows past a sequence's prompt stay untouched."""
    got = to64(out)
    worst = 0.0
    for b, s in enumerate(lens):
        if s > 0:
            ref = oracle.prefill_attn(to64(q[b:b + 1, :, :s]), to64(K[b:b + 1, :, :s]), to64(V[b:b + 1, :, :s]), s,
                                      q.shape[1])
            err = float(np.abs(got[b, :, :s] - ref[0]).max())
            worst = max(worst, err)
            assert np.isfinite(got[b, :, :s]).all()
            assert err <= compare.ATTN_TOL["bf16"], f"sequence {b}: attention max error {err}"
        assert (got[b, :, s:] == SENTINEL).all(), "rows past the prompt were written"
    return worst


@pytest.mark.parametrize("batch,h_kv,G,n,seq_len", [
    (1, 1, 1, 1, None),
    (1, 1, 4, 128, None),
    (2, 2, 4, 129, None),
    (2, 2, 4, 300, None),
    (2, 1, 7, 513, [513, 200]),
    (3, 2, 1, 700, [0, 700, 255]),
])
def test_prefill_attention_matches_oracle(batch, h_kv, G, n, seq_len):
    q, K, V, lens, sl = _prompt(batch * 100 + n, batch, h_kv, G, n, (n + 47) // 8 * 8, seq_len)
    out = torch.full((batch, h_kv * G, n, D), SENTINEL, dtype=torch.bfloat16, device="cuda")
    ws = B.new_workspace(B.prefill_workspace_bytes(), "cuda")
    B.prefill_attn(q, K, V, n, out, ws, seq_len=sl)
    torch.cuda.synchronize()
    assert B.csmkv_device_status(ws) == 0
    _attention_check(q, K, V, lens, out, n)
    out2 = torch.full_like(out, SENTINEL)
    B.prefill_attn(q, K, V, n, out2, ws, seq_len=sl)
    torch.cuda.synchronize()
    assert torch.equal(out, out2), "repeated calls differ"


@pytest.mark.parametrize("grow", [6.0, 0.1])
def test_prefill_attention_when_scores_grow_or_shrink(grow):
    """Keys past row 200 scaled up (the running row max grows by far more than 2^8, so O
    is rescaled in TMEM mid-row) or down (no rescale)."""
    n = 600
    q, K, V, lens, sl = _prompt(11, 1, 2, 2, n, 608)
    K[:, :, 200:n] = (K[:, :, 200:n].float() * grow).to(torch.bfloat16)
    out = torch.full((1, 4, n, D), SENTINEL, dtype=torch.bfloat16, device="cuda")
    ws = B.new_workspace(B.prefill_workspace_bytes(), "cuda")
    B.prefill_attn(q, K, V, n, out, ws)
    torch.cuda.synchronize()
    assert B.csmkv_device_status(ws) == 0
    _attention_check(q, K, V, lens, out, n)


def _standalone_round(K, V, lens, n1, n2, c, r, head_mask):
    """The prompt as a cache with N = 1 and len = s, compressed in place by csm_compress."""
    Ks, Vs = K.clone(), V.clone()
    for b, s in enumerate(lens):  # the standalone round never reads past len; keep NaN out of its checks
        Ks[b, :, s:] = 0
        Vs[b, :, s:] = 0
    N = torch.ones(K.shape[:3], dtype=torch.int32, device="cuda")
    L = torch.tensor([[s] * K.shape[1] for s in lens], dtype=torch.int32, device="cuda")
    return Ks, Vs, N, L


@pytest.mark.parametrize("n1,n2,r,seq_len,head_mask", [
    (16, 64, 0.5, None, None),
    (16, 64, 0.5, [1000, 700], [0, 1]),
    (16, 64, 0.3, [1000, 611], None),
    (0, 32, 0.5, None, None),
    (128, 16, 0.45, [1000, 999], None),
    (200, 64, 0.5, None, [1, 0]),
    (16, 64, 0.0, [1000, 400], None),
])
def test_fused_round_matches_standalone_round(n1, n2, r, seq_len, head_mask):
    batch, h_kv, G, n, c = 2, 2, 2, 1000, 256
    q, K, V, lens, sl = _prompt(7 + n1, batch, h_kv, G, n, n + 24, seq_len, dup=0.6)
    hm = None if head_mask is None else torch.tensor(head_mask, dtype=torch.uint8, device="cuda")
    out = torch.full((batch, h_kv * G, n, D), SENTINEL, dtype=torch.bfloat16, device="cuda")
    Ko = torch.full((batch, h_kv, n + 8, D), SENTINEL, dtype=torch.bfloat16, device="cuda")
    Vo = torch.full_like(Ko, SENTINEL)
    No = torch.full((batch, h_kv, n + 8), -7, dtype=torch.int32, device="cuda")
    Lo = torch.full((batch, h_kv), -7, dtype=torch.int32, device="cuda")
    ws = B.new_workspace(B.prefill_workspace_bytes(), "cuda")
    B.prefill_attn_csm(q, K, V, n, out, Ko, Vo, No, Lo, n1, n2, c, r, ws, seq_len=sl, head_mask=hm)
    torch.cuda.synchronize()
    assert B.csmkv_device_status(ws) == 0

    # the attention part against the oracle (its key tiles start at n1 mod 128 - 128,
    # so its fp32 sums are grouped differently from the attention-only call's)
    _attention_check(q, K, V, lens, out, n)

    # the second cache equals the standalone round on the same prompt
    Ks, Vs, Ns, Ls = _standalone_round(K, V, lens, n1, n2, c, r, head_mask)
    stats = round_parity(Ks, Vs, Ns, Ls, n1, n2, c, r, "bf16", head_mask=head_mask)
    assert torch.equal(Lo, Ls), (Lo, Ls)
    for b in range(batch):
        for h in range(h_kv):
            s = int(Ls[b, h])
            assert torch.equal(Ko[b, h, :s], Ks[b, h, :s]), (b, h)
            assert torch.equal(Vo[b, h, :s], Vs[b, h, :s]), (b, h)
            assert torch.equal(No[b, h, :s], Ns[b, h, :s]), (b, h)
            assert (No[b, h, s:] == -7).all(), "rows past len_out were written"
    m = B.csm_edges_per_chunk(r, c)
    if m > 0:
        assert stats["chunks"] > 0


def test_empty_prompt_writes_only_lengths():
    q, K, V, lens, sl = _prompt(3, 1, 2, 2, 8, 16)
    out = torch.full((1, 4, 8, D), SENTINEL, dtype=torch.bfloat16, device="cuda")
    Ko = torch.zeros(1, 2, 16, D, dtype=torch.bfloat16, device="cuda")
    Vo, No = torch.zeros_like(Ko), torch.zeros(1, 2, 16, dtype=torch.int32, device="cuda")
    Lo = torch.full((1, 2), 9, dtype=torch.int32, device="cuda")
    ws = B.new_workspace(B.prefill_workspace_bytes(), "cuda")
    B.prefill_attn_csm(q, K, V, 0, out, Ko, Vo, No, Lo, 16, 64, 256, 0.5, ws)
    torch.cuda.synchronize()
    assert (Lo == 0).all()
    assert (out == SENTINEL).all()


def test_full_size_prompt_sampled_rows():
    """One layer of the 64K workload's shape in the bench's launch configuration (one
    65536-row prompt, 32 query / 8 KV heads, fused first round r = 0.5): sampled output rows
    of every query head against the oracle (prompt rows of the sampled positions only), and
    the whole second cache byte-equal to the standalone round."""
    n, h_kv, G = 65536, 8, 4
    g = torch.Generator(device="cuda").manual_seed(2024)
    q = torch.randn(1, h_kv * G, n, D, device="cuda", generator=g).to(torch.bfloat16)
    K = torch.randn(1, h_kv, n + 64, D, device="cuda", generator=g).to(torch.bfloat16)
    V = torch.randn(1, h_kv, n + 64, D, device="cuda", generator=g).to(torch.bfloat16)
    out = torch.empty_like(q)
    Ko, Vo = torch.empty_like(K), torch.empty_like(V)
    No = torch.empty(1, h_kv, n + 64, dtype=torch.int32, device="cuda")
    Lo = torch.empty(1, h_kv, dtype=torch.int32, device="cuda")
    ws = B.new_workspace(B.prefill_workspace_bytes(), "cuda")
    B.prefill_attn_csm(q, K, V, n, out, Ko, Vo, No, Lo, 16, 64, 256, 0.5, ws)
    torch.cuda.synchronize()
    assert B.csmkv_device_status(ws) == 0
    rows = np.array([0, 1, 15, 16, 127, 128, 4095, 32767, 40000, n - 2, n - 1], np.int32)
    Kc, Vc = to64(K[:, :, :n]), to64(V[:, :, :n])
    for h in range(0, h_kv * G, 5):  # a spread of query heads (every KV head is read by one)
        ref = oracle.prefill_attn(to64(q[:, h:h + 1]), Kc[:, h // G:h // G + 1], Vc[:, h // G:h // G + 1], n, 1,
                                  rows=rows)
        got = to64(out[:, h:h + 1, rows])
        err = float(np.abs(got - ref).max())
        assert err <= compare.ATTN_TOL["bf16"], f"head {h}: attention max error {err}"
    Ks, Vs = K.clone(), V.clone()
    Ns = torch.ones(1, h_kv, n + 64, dtype=torch.int32, device="cuda")
    Ls = torch.full((1, h_kv), n, dtype=torch.int32, device="cuda")
    wsc = B.new_workspace(B.csm_workspace_bytes(B.cache_desc(Ks), 16, 64, 256), "cuda")
    B.csm_compress(Ks, Vs, Ns, Ls, 16, 64, 256, 0.5, workspace=wsc)
    torch.cuda.synchronize()
    assert torch.equal(Lo, Ls)
    s = int(Ls[0, 0])
    assert torch.equal(Ko[:, :, :s], Ks[:, :, :s]) and torch.equal(Vo[:, :, :s], Vs[:, :, :s])
    assert torch.equal(No[:, :, :s], Ns[:, :, :s])
