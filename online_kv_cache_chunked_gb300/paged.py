"""Building a paged (block-table) cache from a dense one, and back.

Layout plumbing for callers, tests and the benchmark (torch gathers and
scatters, run outside any timed region); the compression and attention on a
paged cache run in the library's kernels (binding.*_paged). See csmkv_pages in
include/csmkv.h: every (sequence, KV head) unit owns max_pages pages of
page_rows rows, listed in its row of the block table, taken from one pool per
array; here the pages are placed at a seeded random permutation of the pool,
so consecutive logical pages are scattered as they are in a serving system.
"""
from __future__ import annotations

import torch

from .binding import PagedKV


def to_paged(K, V, N, page_rows: int, spare_pages: int = 0, seed: int = 0) -> PagedKV:
    """K, V: [batch, h_kv, cap, d]; N: [batch, h_kv, cap]. Returns the same contents in a
    paged layout with `spare_pages` unused pool pages; every unit gets ceil(cap /
    page_rows) pages, so the logical capacity is cap rounded up to whole pages."""
    batch, h_kv, cap, d = K.shape
    maxp = -(-cap // page_rows)
    if maxp * page_rows != cap:  # pad the last page of every unit with empty rows
        pad = maxp * page_rows - cap
        K = torch.nn.functional.pad(K, (0, 0, 0, pad))
        V = torch.nn.functional.pad(V, (0, 0, 0, pad))
        N = torch.nn.functional.pad(N, (0, pad))
    used = batch * h_kv * maxp
    npages = used + int(spare_pages)
    g = torch.Generator(device="cpu").manual_seed(seed)
    perm = torch.randperm(npages, generator=g)[:used].to(torch.int32)
    table = perm.view(batch * h_kv, maxp).to(K.device)
    idx = table.view(-1).long()
    Kp = torch.zeros((npages, page_rows, d), dtype=K.dtype, device=K.device)
    Vp = torch.zeros_like(Kp)
    Np = torch.zeros((npages, page_rows), dtype=N.dtype, device=N.device)
    Kp[idx] = K.reshape(used, page_rows, d)
    Vp[idx] = V.reshape(used, page_rows, d)
    Np[idx] = N.reshape(used, page_rows)
    return PagedKV(Kp, Vp, Np, table, batch, h_kv)


def to_dense(kv: PagedKV):
    """The logical cache [batch, h_kv, cap, d] (K, V) and [batch, h_kv, cap] (N) of a paged one."""
    idx = kv.table.reshape(-1).long()
    shape = (kv.batch, kv.h_kv, kv.cap)
    K = kv.K[idx].reshape(*shape, kv.head_dim)
    V = kv.V[idx].reshape(*shape, kv.head_dim)
    N = kv.N[idx].reshape(*shape)
    return K, V, N
