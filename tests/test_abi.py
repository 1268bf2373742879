"""The C-ABI library on the CPU: it builds, loads, exports every declared symbol,
its host helpers agree with the oracle's schedule, and argument errors come back
synchronously without touching a GPU."""
import ctypes
import math
import os
import re

import pytest

import oracle
from oracle import schedule as osched
from online_kv_cache_chunked_gb300 import _build
from online_kv_cache_chunked_gb300 import binding as B
from online_kv_cache_chunked_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "csmkv.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return B.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s+\*?([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "return")))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert names == sorted([
        "csm_workspace_bytes", "csm_compress", "csm_compress_ex", "csm_max_chunks", "csm_append_workspace_bytes",
        "csm_append", "decode_attn_workspace_bytes", "decode_attn_logn", "decode_attn_logn_noalloc", "decode_step_logn",
        "csm_decode_run", "csm_budget", "csm_chunks_to_budget", "csm_should_trigger",
        "csm_ratio", "csm_edges_per_chunk", "csm_num_chunks", "csm_len_after", "csmkv_device_status",
        "csmkv_clear_status", "csmkv_status_str", "csm_append_paged", "csm_compress_paged",
        "decode_attn_logn_paged", "decode_step_logn_paged", "prefill_workspace_bytes", "prefill_attn",
        "prefill_attn_csm"]), names
    raw = ctypes.CDLL(_build.OUT)
    for n in names:
        assert hasattr(raw, n), f"{n} declared in csmkv.h but not exported"


def test_status_strings(lib):
    for code in range(9):
        assert B.status_str(code) not in ("", "unknown status")
    assert B.status_str(99) == "unknown status"


@pytest.mark.parametrize("r,c", [(0.5, 256), (0.45, 256), (0.4, 256), (0.1, 256), (0.25, 8), (0.5, 64),
                                 (0.3, 10), (0.0, 256), (0.2, 256), (0.19999999999999996, 256)])
def test_edges_per_chunk_matches_oracle(lib, r, c):
    assert B.csm_edges_per_chunk(r, c) == oracle.edges_per_chunk(r, c)


def test_host_helpers_match_oracle(lib):
    for n, R, G in [(16384, 0.2, 1000), (32768, 0.2, 1000), (65536, 0.2, 1000), (8192, 0.25, 512)]:
        assert math.isclose(B.csm_budget(n, R, G), oracle.budget(n, R, G), rel_tol=0, abs_tol=1e-9)
    for j in range(12):
        assert B.csm_ratio(j, 0.5, 0.05, 0.1) == oracle.ratio(j, 0.5, 0.05, 0.1)
    for s in [0, 10, 79, 80, 335, 336, 16384, 32897, 65536]:
        for m in (0, 51, 128):
            assert B.csm_len_after(s, 16, 64, 256, m) == oracle.len_after(s, 16, 64, 256, m)
        assert B.csm_num_chunks(s, 16, 64, 256) == osched.num_chunks(s, 16, 64, 256)
    for s in (3540, 3541):
        assert B.csm_should_trigger(s, 3476.8, 64) == oracle.should_trigger(s, 3476.8, 64)
    for s in (0, 3476, 3477, 3541, 3604, 3605, 8321, 16384, 65536):
        for Bud in (3476.8, 13307.2, 6753.6):
            for m in (0, 102, 128):
                assert B.csm_chunks_to_budget(s, Bud, 16, 64, 256, m) == osched.chunks_to_budget(s, Bud, 16, 64, 256, m)


@pytest.mark.parametrize("name", sorted(synth.WORKLOADS))
def test_pipeline_plan_matches_oracle_schedule(lib, name):
    from online_kv_cache_chunked_gb300.pipeline import plan
    w = synth.WORKLOADS[name]
    got = plan(w)
    if w.forced_round:
        assert [(r.step, r.m) for r in got] == [(0, B.csm_edges_per_chunk(w.r_init, w.c))]
        return
    for i, n in enumerate(w.n):
        ref = osched.plan(n, w.R, w.steps, w.g, w.n1, w.n2, w.c, w.r_init, w.dr, w.r_min)
        mine = [(r.step, r.s_before[r.seqs.index(i)], r.m, r.s_after[r.seqs.index(i)]) for r in got if i in r.seqs]
        assert mine == [(st, s, m, s2) for st, s, _, m, s2 in ref]


def _cache(**kw):
    d = dict(batch=1, h_kv=2, head_dim=128, cap=1024, dtype=0)
    d.update(kw)
    return B.Cache(d["batch"], d["h_kv"], d["head_dim"], d["cap"], d["dtype"])


def _compress(lib, cache, n1=16, n2=64, c=256, r=0.5, ptr=4096, ws=1 << 20, wsp=1 << 16):
    P = ctypes.c_void_p
    return lib.csm_compress(P(ptr), P(ptr), P(ptr), P(ptr), ctypes.byref(cache), n1, n2, c, r, None, None,
                            P(wsp), ws, None)


def test_csm_argument_errors_without_gpu(lib):
    c = _cache()
    assert _compress(lib, c, r=0.6) == 1
    assert _compress(lib, c, r=-0.1) == 1
    assert _compress(lib, c, r=float("nan")) == 1
    assert _compress(lib, c, c=7) == 1
    assert _compress(lib, c, c=512) == 1
    assert _compress(lib, c, n1=-1) == 1
    assert _compress(lib, _cache(cap=1020)) == 1          # cap % 8
    assert _compress(lib, _cache(head_dim=100)) == 1      # head_dim % 8
    assert _compress(lib, _cache(head_dim=256)) == 1      # head_dim > 128
    assert _compress(lib, _cache(dtype=5)) == 2
    assert _compress(lib, c, ptr=4100) == 3               # misaligned
    assert _compress(lib, c, ws=16) == 5                  # workspace too small
    assert _compress(lib, c, wsp=4096 + 16) == 5          # workspace misaligned
    opts = B.CsmOptions(kernel=2)  # not a kernel choice
    P = ctypes.c_void_p
    assert lib.csm_compress_ex(P(4096), P(4096), P(4096), P(4096), ctypes.byref(c), 16, 64, 256, 0.5, None, None,
                               None, ctypes.byref(opts), P(1 << 16), 1 << 20, None) == 1
    need = lib.csm_workspace_bytes(ctypes.byref(c), 16, 64, 256)
    assert need > 256
    assert lib.csm_max_chunks(ctypes.byref(c), 16, 64, 256) == (1024 - 80) // 256


def test_attention_argument_errors_without_gpu(lib):
    P = ctypes.c_void_p
    c = _cache()

    def call(h_q=8, scale=0.088, ptr=4096, cache=c):
        return lib.decode_attn_logn(P(ptr), P(ptr), P(ptr), P(ptr), P(ptr), ctypes.byref(cache), h_q, scale,
                                    P(ptr), P(1 << 16), 1 << 24, None)
    assert call(h_q=3) == 1          # not a multiple of h_kv
    assert call(h_q=0) == 1
    assert call(scale=0.0) == 1
    assert call(ptr=4104) == 3
    assert call(h_q=18) == 8         # bf16 group of 9 query heads is not covered
    assert call(cache=_cache(head_dim=96)) == 8
    assert lib.csm_append(None, None, None, None, ctypes.byref(c), None, None, None, None, 0, None) == 1


def test_prefill_argument_errors_without_gpu(lib):
    P = ctypes.c_void_p
    c = _cache()  # bf16, head_dim 128

    def attn(h_q=8, n=100, ptr=4096, cache=c, ws=1 << 16, wsb=256, scale=0.0):
        return lib.prefill_attn(P(ptr), P(ptr), P(ptr), ctypes.byref(cache), n, None, h_q, scale, P(ptr), P(ws), wsb,
                                None)
    assert lib.prefill_workspace_bytes() >= 4
    assert attn(h_q=3) == 1          # not a multiple of h_kv
    assert attn(n=-1) == 1
    assert attn(n=c.cap + 1) == 1    # the prompt must fit in the cache
    assert attn(scale=float("nan")) == 1
    assert attn(cache=_cache(head_dim=64)) == 8
    assert attn(cache=_cache(dtype=1)) == 8
    assert attn(ptr=4104) == 3
    assert attn(wsb=0) == 5
    assert attn(ws=0) == 5

    def fused(n=100, cap_out=None, c_=256, r=0.5, N_out=4096, n1=16):
        co = _cache() if cap_out is None else _cache(cap=cap_out)
        return lib.prefill_attn_csm(P(4096), P(4096), P(4096), ctypes.byref(c), n, None, 8, 0.0, P(4096), P(4096),
                                    P(4096), P(N_out), P(4096), ctypes.byref(co), n1, 64, c_, r, None, P(1 << 16),
                                    256, None)
    assert fused(cap_out=64) == 1    # the second cache must hold the prompt
    assert fused(r=0.6) == 1
    assert fused(n1=-1) == 1
    assert fused(N_out=0) == 1
    assert fused(c_=128) == 8        # the fused round covers c == 256 only


def test_no_workspace_attention_checks_arguments_before_touching_the_gpu(lib):
    """The no-workspace entry point runs every argument check before it looks up or
    clears its shared scratch, so these return at once here, with no GPU at all."""
    P = ctypes.c_void_p
    c = _cache()

    def call(h_q=8, scale=0.088, ptr=4096, cache=c, q=4096):
        return lib.decode_attn_logn_noalloc(P(q), P(ptr), P(ptr), P(ptr), P(ptr), ctypes.byref(cache), h_q,
                                            scale, P(ptr), None)
    assert call(h_q=3) == 1
    assert call(scale=float("inf")) == 1
    assert call(q=0) == 1            # NULL query
    assert call(ptr=4104) == 3
    assert call(h_q=18) == 8
    assert call(cache=_cache(dtype=9)) == 2


def test_decode_run_rejects_bad_arguments_without_a_gpu(lib):
    fn = lib.csm_decode_run
    assert fn(None, 1, 1, None) == 1  # CSMKV_ERR_ARG: no loop description
    loop = B.CsmDecodeLoop()
    assert fn(ctypes.byref(loop), 0, 1, None) == 1  # steps are 1-based
    assert fn(ctypes.byref(loop), 1, -1, None) == 1
    assert fn(ctypes.byref(loop), 1, 0, None) == 0  # nothing to do
    assert fn(ctypes.byref(loop), 1, 3, None) == 1  # no inputs
    rounds = (B.CsmRoundPlan * 2)(B.CsmRoundPlan(5, 0.5, None), B.CsmRoundPlan(2, 0.5, None))
    x = ctypes.c_void_p(16)
    loop = B.CsmDecodeLoop(q=x, k_new=x, v_new=x, out=x, rounds=rounds, n_rounds=2)
    assert fn(ctypes.byref(loop), 1, 3, None) == 1  # rounds out of step order
    rounds[1].step = 7
    assert fn(ctypes.byref(loop), 1, 3, None) == 1  # the zeroed cache descriptor (batch 0)
    loop.cache = B.Cache(1, 2, 128, 1024, 7)
    assert fn(ctypes.byref(loop), 1, 3, None) == 2  # unknown dtype
    loop.cache = B.Cache(1, 2, 128, 1024, 0)
    loop.l2_flush = x
    assert fn(ctypes.byref(loop), 1, 3, None) == 1  # a flush buffer without a size


def test_paged_argument_errors_without_gpu(lib):
    """The paged entry points check the block-table descriptor against the logical
    cache before any launch."""
    P = ctypes.c_void_p
    c = _cache(cap=1024)  # logical: 4 pages of 256

    def compress(pages, cache=c):
        return lib.csm_compress_paged(P(4096), P(4096), P(4096), P(4096), ctypes.byref(cache),
                                      ctypes.byref(pages) if pages is not None else None, 16, 64, 256, 0.5,
                                      None, None, None, None, P(1 << 16), 1 << 20, None)

    def attn(pages, cache=c):
        return lib.decode_attn_logn_paged(P(4096), P(4096), P(4096), P(4096), P(4096), ctypes.byref(cache),
                                          ctypes.byref(pages) if pages is not None else None, 8, 0.088, P(4096),
                                          P(1 << 16), 1 << 24, None)
    ok = B.Pages(4096, 256, 4, 64)
    assert compress(None) == 1
    assert compress(B.Pages(0, 256, 4, 64)) == 1         # no table
    assert compress(B.Pages(4098, 256, 4, 64)) == 3      # misaligned table
    assert compress(B.Pages(4096, 96, 4, 64)) == 1       # page_rows not a multiple of 64
    assert compress(B.Pages(4096, 256, 3, 64)) == 1      # max_pages * page_rows != cap
    assert compress(B.Pages(4096, 256, 4, 0)) == 1       # empty pool
    assert compress(ok, _cache(cap=1024, dtype=1)) == 8  # fp32: the block-table variant is tensor-core only
    assert attn(None) == 1
    assert attn(ok, _cache(cap=1024, dtype=1)) == 8      # fp32 paged attention is not covered
    assert attn(B.Pages(4096, 256, 4, 1 << 24)) == 1     # pool rows beyond int32
    assert lib.csm_append_paged(P(4096), P(4096), P(4096), P(4096), ctypes.byref(c), None, P(4096), P(4096), None,
                                P(1 << 16), 256, None) == 1


def test_paged_layout_round_trip_on_cpu():
    import torch

    from online_kv_cache_chunked_gb300 import paged
    g = torch.Generator().manual_seed(0)
    K = torch.randn(2, 3, 512, 16, generator=g).to(torch.bfloat16)
    V = torch.randn(2, 3, 512, 16, generator=g).to(torch.bfloat16)
    N = torch.randint(1, 9, (2, 3, 512), generator=g, dtype=torch.int32)
    kv = paged.to_paged(K, V, N, 128, spare_pages=5, seed=3)
    assert kv.table.shape == (6, 4) and kv.K.shape == (6 * 4 + 5, 128, 16)
    assert sorted(kv.table.view(-1).tolist()) == sorted(set(kv.table.view(-1).tolist()))  # no page twice
    K2, V2, N2 = paged.to_dense(kv)
    assert torch.equal(K2, K) and torch.equal(V2, V) and torch.equal(N2, N)
    c = kv.cache()
    assert (c.batch, c.h_kv, c.head_dim, c.cap) == (2, 3, 16, 512)
    kv = paged.to_paged(K[:, :, :300], V[:, :, :300], N[:, :, :300], 128)  # cap rounded up to whole pages
    assert kv.cap == 384
    K2, _, N2 = paged.to_dense(kv)
    assert torch.equal(K2[:, :, :300], K[:, :, :300]) and not N2[:, :, 300:].any()
