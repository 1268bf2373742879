"""Host driver of the inference pipeline over the C ABI.

[Chelsea §三 算法流程, Algorithm 1]: after prefill the cache holds s = n rows with
N = 1 and the budget is B = R (n + Gamma); one CSM round runs whenever s >= B + g,
checked once after prefill and once after every decode append (append, then
attend, then check). [CentroidKV 渐进式调度]: round j of a sequence uses
r_j = r_init - j * delta_r (floored at r_min).

Every length follows a closed form (each full chunk loses exactly m rows), so the
whole schedule is planned on the host up front with the library's host helpers and
the device is never read back. With `budget_exact` a round merges only the oldest
chunks needed to bring s to <= B (csm_chunks_to_budget), so after the first rounds
the trigger fires about every m appends instead of compressing far below B. All layers of a sequence share its schedule; outlier
heads are never compressed and simply grow by one row per step.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

from . import binding as B


@dataclasses.dataclass
class Round:
    step: int           # 0 = after prefill, i = after the i-th decode append
    r: float
    m: int
    seqs: tuple         # sequences (of the workload, before layer folding) compressed now
    s_before: tuple     # their compressed-head length before the round
    s_after: tuple
    limits: tuple = ()  # budget-exact: chunks merged per sequence (empty: every full chunk)


def plan(w) -> list:
    """All CSM rounds of a workload (see the module docstring)."""
    n = [int(x) for x in w.n]
    s = list(n)
    j = [0] * w.seqs
    Bud = [B.csm_budget(n[i], w.R, w.steps) for i in range(w.seqs)]
    rounds = []
    for step in range(0, w.steps + 1):
        if step > 0:
            s = [x + 1 for x in s]
        if w.forced_round:
            fire = list(range(w.seqs)) if step == 0 else []
        else:
            fire = [i for i in range(w.seqs) if B.csm_should_trigger(s[i], Bud[i], w.g)]
        groups = {}
        for i in fire:
            r = B.csm_ratio(j[i], w.r_init, w.dr, w.r_min)
            groups.setdefault(r, []).append(i)
        for r, seqs in sorted(groups.items(), key=lambda kv: -kv[0]):
            m = B.csm_edges_per_chunk(r, w.c)
            before = tuple(s[i] for i in seqs)
            limits = ()
            if w.budget_exact:
                limits = tuple(B.csm_chunks_to_budget(s[i], Bud[i], w.n1, w.n2, w.c, m) for i in seqs)
            for k, i in enumerate(seqs):
                if w.budget_exact:
                    s[i] = s[i] - limits[k] * m
                else:
                    s[i] = B.csm_len_after(s[i], w.n1, w.n2, w.c, m)
                j[i] += 1
            rounds.append(Round(step, r, m, tuple(seqs), before, tuple(s[i] for i in seqs), limits))
    return rounds


def final_lengths(w, rounds=None) -> np.ndarray:
    """Expected len[batch, h_kv] after the whole run (host mirror)."""
    rounds = plan(w) if rounds is None else rounds
    _, _, mask = _stats(w)
    grown = np.array(w.n, np.int64) + w.steps  # outlier heads: never compressed
    out = np.zeros((w.batch, w.h_kv), np.int64)
    cur = np.array(w.n, np.int64)  # replay of the compressed heads
    ri = 0
    for step in range(0, w.steps + 1):
        if step > 0:
            cur += 1
        while ri < len(rounds) and rounds[ri].step == step:
            for i, sa in zip(rounds[ri].seqs, rounds[ri].s_after):
                cur[i] = sa
            ri += 1
    for b in range(w.batch):
        i = b % w.seqs
        out[b] = np.where(mask.astype(bool), grown[i], cur[i])
    return out


def _stats(w):
    from .synth import head_stats
    return head_stats(w)


class Pipeline:
    """Runs a planned workload on the device through the C ABI.

    data: dict from synth.make_device / synth.cache_from_numpy (K, V, N, len,
    k_dec, v_dec, q, head_mask). The cache tensors are updated in place; the
    attention output of decode step i lands in self.out[i].
    paged: optional binding.PagedKV holding the same cache in a block-table layout;
    every call then goes to the paged entry points (fused decode steps) and the
    dense K, V, N of `data` are not used.
    """

    def __init__(self, w, data, stream=None, csm_kernel=B.CSM_KERNEL_AUTO, paged=None):
        self.w = w
        self.d = data
        self.stream = stream
        self.csm_kernel = int(csm_kernel)
        self.paged = paged
        self.rounds = plan(w)
        K = paged.K if paged is not None else data["K"]
        dev = K.device
        cache = paged.cache() if paged is not None else B.cache_desc(K)
        self.ws_csm = B.new_workspace(B.csm_workspace_bytes(cache, w.n1, w.n2, w.c), dev)
        self.ws_app = B.new_workspace(B.csm_append_workspace_bytes(), dev)
        self.ws_att = B.new_workspace(B.decode_attn_workspace_bytes(cache, w.h_q), dev)
        self.out = torch.empty((w.steps, w.batch, w.h_q, w.d), dtype=K.dtype, device=dev)
        hm = data.get("head_mask")
        self.head_mask = hm if (hm is not None and int(hm.sum()) > 0) else None
        # one device mask per round that does not cover every sequence
        self.masks = []
        for rd in self.rounds:
            if len(rd.seqs) == w.seqs:
                self.masks.append(None)
            else:
                m = np.zeros(w.batch, np.uint8)
                for b in range(w.batch):
                    if b % w.seqs in rd.seqs:
                        m[b] = 1
                self.masks.append(torch.from_numpy(m).to(dev))
        # budget-exact: per-round chunk caps per cache sequence (layers share a sequence's)
        self.limits = []
        for rd in self.rounds:
            if not rd.limits:
                self.limits.append(None)
                continue
            lim = np.zeros(w.batch, np.int32)
            cap_of = dict(zip(rd.seqs, rd.limits))
            for b in range(w.batch):
                lim[b] = cap_of.get(b % w.seqs, 0)
            self.limits.append(torch.from_numpy(lim).to(dev))
        self.by_step = {}
        for k, rd in enumerate(self.rounds):
            self.by_step.setdefault(rd.step, []).append(k)

    def compress_at(self, step, hook=None):
        d, w = self.d, self.w
        for k in self.by_step.get(step, []):
            rd = self.rounds[k]
            if hook:
                hook("csm", rd, True)
            if self.paged is not None:
                B.csm_compress_paged(self.paged, d["len"], w.n1, w.n2, w.c, rd.r, self.head_mask, self.masks[k],
                                     seq_max_chunks=self.limits[k], workspace=self.ws_csm, stream=self.stream)
            elif self.csm_kernel == B.CSM_KERNEL_AUTO and self.limits[k] is None:
                B.csm_compress(d["K"], d["V"], d["N"], d["len"], w.n1, w.n2, w.c, rd.r, self.head_mask,
                               self.masks[k], self.ws_csm, self.stream)
            else:
                B.csm_compress_ex(d["K"], d["V"], d["N"], d["len"], w.n1, w.n2, w.c, rd.r, self.head_mask,
                                  self.masks[k], kernel=self.csm_kernel, seq_max_chunks=self.limits[k],
                                  workspace=self.ws_csm, stream=self.stream)
            if hook:
                hook("csm", rd, False)

    def decode_step(self, i, hook=None):
        """Decode step i (1-based): append, attend, then the trigger's rounds."""
        d = self.d
        if self.paged is not None:
            raise ValueError("a paged pipeline issues its decode steps natively (decode_native)")
        B.csm_append(d["K"], d["V"], d["N"], d["len"], d["k_dec"][i - 1], d["v_dec"][i - 1], None, self.ws_app,
                     self.stream)
        if hook:
            hook("attn", i, True)
        B.decode_attn_logn(d["q"][i - 1], d["K"], d["V"], d["N"], d["len"], self.out[i - 1], self.ws_att,
                           stream=self.stream)
        if hook:
            hook("attn", i, False)
        self.compress_at(i, hook)

    def run(self, hook=None, steps=None):
        """Prefill round(s), then the decode loop one binding call per kernel."""
        self.compress_at(0, hook)
        for i in range(1, (self.w.steps if steps is None else steps) + 1):
            self.decode_step(i, hook)

    def decode_plan(self):
        """(step, r, seq_mask, seq_max_chunks) of every round after prefill, in issue order."""
        return [(rd.step, rd.r, self.masks[k], self.limits[k]) for k, rd in enumerate(self.rounds) if rd.step >= 1]

    def decode_native(self, first_step, steps, attn_events=None, csm_events=None, l2_flush=None, fused=True):
        """Decode steps first_step .. first_step + steps - 1 issued by the library in one
        call, with the rounds the plan fires at those steps (fused: each step's append
        and attention as one kernel)."""
        d, w = self.d, self.w
        kv = self.paged
        K, V, N = (kv.K, kv.V, kv.N) if kv is not None else (d["K"], d["V"], d["N"])
        B.csm_decode_run(K, V, N, d["len"], d["q"], d["k_dec"], d["v_dec"], self.out, w.n1, w.n2,
                         w.c, rounds=self.decode_plan(), head_mask=self.head_mask, ws_csm=self.ws_csm,
                         ws_append=self.ws_app, ws_attn=self.ws_att, first_step=first_step, steps=steps,
                         csm_kernel=self.csm_kernel, attn_events=attn_events, csm_events=csm_events,
                         l2_flush=l2_flush, stream=self.stream, fused_append=fused or kv is not None, paged=kv)

    def run_native(self, steps=None, hook=None, attn_events=None, csm_events=None, l2_flush=None, fused=True):
        """Prefill round(s), then the whole decode loop issued by the library in one call
        (fused: each step's append and attention as one kernel)."""
        self.compress_at(0, hook)
        n = self.w.steps if steps is None else steps
        self.decode_native(1, n, attn_events, csm_events, l2_flush, fused)
