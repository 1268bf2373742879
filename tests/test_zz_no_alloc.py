"""The attention entry point that needs no workspace (for callers that cannot
allocate device memory) against the regular one that takes a workspace, and
against the oracle.

Kept in a file of its own that pytest collects last, so that a run stopping at
the first failure has run every other test before this one.
"""
import ctypes

import numpy as np
import pytest
import torch

from online_kv_cache_chunked_gb300 import binding as B
from tests.gpu_helpers import attn_parity

pytestmark = pytest.mark.gpu


def _inputs(seed, batch, h_kv, G, cap, D, lengths):
    g = torch.Generator(device="cuda").manual_seed(seed)
    K = torch.randn(batch, h_kv, cap, D, generator=g, device="cuda").to(torch.bfloat16)
    V = torch.randn(batch, h_kv, cap, D, generator=g, device="cuda").to(torch.bfloat16)
    N = torch.randint(1, 9, (batch, h_kv, cap), generator=g, device="cuda", dtype=torch.int32)
    L = torch.tensor(lengths, dtype=torch.int32, device="cuda").view(batch, h_kv)
    q = torch.randn(batch, h_kv * G, D, generator=g, device="cuda").to(torch.bfloat16)
    return q, K, V, N, L


def test_no_workspace_matches_workspace_entry_point_twice(cuda_lib):
    """Two calls in a row (different shapes, so the second finds the first one's
    contents in the shared scratch): each output equals the workspace entry
    point's byte for byte -- both run the same deterministic kernel on zeroed
    scratch -- and the oracle's within the bf16 attention tolerance."""
    cases = [(1, 2, 8, 4, 6000, 128, [[5000, 17, 0, 4096, 3000, 1, 64, 5999], [6000, 2500, 333, 65, 64, 63, 0, 1]]),
             (2, 3, 4, 7, 3000, 128, [[2999, 1, 100, 0], [3000, 1500, 64, 7], [10, 20, 30, 2048]])]
    for seed, batch, h_kv, G, cap, D, lengths in cases:
        q, K, V, N, L = _inputs(seed, batch, h_kv, G, cap, D, lengths)
        ws = B.new_workspace(B.decode_attn_workspace_bytes(B.cache_desc(K), q.shape[1]))
        ref = torch.empty(batch, h_kv * G, D, dtype=torch.bfloat16, device="cuda")
        got = torch.full_like(ref, float("nan"))
        B.decode_attn_logn(q, K, V, N, L, ref, ws)
        B.decode_attn_logn_noalloc(q, K, V, N, L, got)
        torch.cuda.synchronize()
        assert B.csmkv_device_status(ws) == 0
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
        err = attn_parity(q, K, V, N, L, got, "bf16")
        assert np.isfinite(err)


def test_no_workspace_rejects_batches_beyond_its_scratch(cuda_lib):
    # 16384 units need far more than the fixed 16 MiB scratch: refused before any launch
    assert B.decode_attn_workspace_bytes(B.Cache(2048, 8, 128, 1024, B.BF16), 32) > (16 << 20)
    cache = B.Cache(2048, 8, 128, 1024, B.BF16)
    P = ctypes.c_void_p
    rc = B.load().decode_attn_logn_noalloc(P(4096), P(4096), P(4096), P(4096), P(4096), ctypes.byref(cache), 32,
                                           0.088, P(4096), None)
    assert rc == 5  # CSMKV_ERR_WORKSPACE
