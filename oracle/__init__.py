"""fp64 CPU oracle for online KV-cache clustering (CSM + degree-aware attention).

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. The product path
never touches it, and it shares no code with the CUDA library.

The arithmetic lives in ``csm_oracle.c`` (plain C, fp64, built here with gcc);
this module only converts numpy arrays and calls it. Page shorthand used in
citations:

* [Chelsea]    "Chelsea: Efficient Long-Context LLM Inference via KV Cache
  Clustering" (xllm-io paper review of arXiv 2506.11418).
* [CentroidKV] "CentroidKV: Efficient Long-Context LLM Inference via KV Cache
  Clustering" (gist.science explainer, section 技术摘要).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .schedule import budget, edges_per_chunk, len_after, ratio, should_trigger  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "csm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (fp contraction off so x86 and Arm agree)."""
    with _lock:
        stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
        if force or stale:
            tmp = _LIB + f".tmp{os.getpid()}"
            cmd = ["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
                   "-o", tmp, _SRC, "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i32 = ctypes.c_int32
        lib.oracle_partition.argtypes = [i32, P, P]
        lib.oracle_num_chunks.argtypes = [i32, i32, i32, i32]
        lib.oracle_num_chunks.restype = i32
        lib.oracle_csm_chunk.argtypes = [P, P, P, i32, i32, i32, P, P, P, P, P, P, P, P, P, P]
        lib.oracle_csm_chunk.restype = ctypes.c_int
        lib.oracle_csm_round.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, i32, i32,
                                         P, P, P, P, P, P, i32, P, P, P, i32]
        lib.oracle_csm_round.restype = ctypes.c_int
        lib.oracle_csm_chunks.argtypes = [P, P, P, i32, i32, i32, i32, P, P, P, P, P, P, P, P, P, P, i32]
        lib.oracle_csm_chunks.restype = ctypes.c_int
        lib.oracle_append.argtypes = [P, P, P, P, i32, i32, i32, P, P, P]
        lib.oracle_append.restype = i32
        lib.oracle_decode_attn_logn.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32,
                                                ctypes.c_double, P, i32]
        lib.oracle_prefill_attn.argtypes = [P, P, P, i32, i32, i32, i32, i32, i32, ctypes.c_double, P, i32,
                                            P, i32]
        lib.oracle_max_threads.restype = i32
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _i32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def _threads(n):
    return max_threads() if n is None else int(n)


def partition(c: int):
    """A and B offsets the oracle uses inside a chunk of c tokens."""
    a = np.zeros(c // 2, np.int32)
    b = np.zeros(c // 2, np.int32)
    _load().oracle_partition(c, _ptr(a), _ptr(b))
    return a, b


def num_chunks(s: int, n1: int, n2: int, c: int) -> int:
    return int(_load().oracle_num_chunks(s, n1, n2, c))


def csm_chunks(Kc, Vc, Nc, m: int, forced=None, nthreads=None):
    """CSM steps 2-7 on a list of independent chunks.

    Kc, Vc: [n, c, d]; Nc: [n, c]. Returns dict with K, V [n, c-m, d], N [n, c-m],
    match/sim/margin [n, c/2], cut [n] and origin/merged [n, c-m] (chunk offset
    each output row comes from, and whether it is a merged centroid).
    """
    Kc, Vc, Nc = _f64(Kc), _f64(Vc), _i32(Nc)
    n, c, d = Kc.shape
    h = c // 2
    out = dict(K=np.zeros((n, c - m, d)), V=np.zeros((n, c - m, d)),
               N=np.zeros((n, c - m), np.int32), match=np.zeros((n, h), np.int32),
               sim=np.zeros((n, h)), margin=np.zeros((n, h)), cut=np.zeros(n),
               origin=np.zeros((n, c - m), np.int32), merged=np.zeros((n, c - m), np.uint8))
    f = None if forced is None else _i32(forced)
    rc = _load().oracle_csm_chunks(_ptr(Kc), _ptr(Vc), _ptr(Nc), n, c, d, m, _ptr(f),
                                   _ptr(out["K"]), _ptr(out["V"]), _ptr(out["N"]),
                                   _ptr(out["match"]), _ptr(out["sim"]), _ptr(out["margin"]),
                                   _ptr(out["cut"]), _ptr(out["origin"]), _ptr(out["merged"]),
                                   _threads(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_csm_chunks failed ({rc})")
    return out


def csm_round(K, V, N, length, n1: int, n2: int, c: int, m: int, skip=None,
              forced=None, nthreads=None, limits=None):
    """One CSM round over BH caches. K, V: [BH, cap, d]; N: [BH, cap]; length: [BH].

    Inputs are not modified. Returns dict with the new K, V, N, len, the
    per-chunk records match/sim/margin [BH, maxch, c/2] and cut [BH, maxch]
    (maxch = chunks that fit in cap), and per output row its pre-round row
    (origin [BH, cap]) and whether it is a merged centroid (merged [BH, cap]).
    limits: optional [BH] ints; limits[u] > 0 processes only unit u's first
    limits[u] chunks (budget-exact compression).
    """
    K, V, N, L = _f64(K).copy(), _f64(V).copy(), _i32(N).copy(), _i32(length).copy()
    BH, cap, d = K.shape
    h = c // 2
    maxch = max(1, (cap - n1 - n2) // c)
    rec = dict(match=np.full((BH, maxch, h), -1, np.int32), sim=np.zeros((BH, maxch, h)),
               margin=np.zeros((BH, maxch, h)), cut=np.zeros((BH, maxch)),
               origin=np.zeros((BH, cap), np.int32), merged=np.zeros((BH, cap), np.uint8))
    sk = None if skip is None else np.ascontiguousarray(np.asarray(skip, dtype=np.uint8))
    f = None if forced is None else _i32(forced)
    lim = None if limits is None else _i32(np.asarray(limits).reshape(BH))
    rc = _load().oracle_csm_round(_ptr(K), _ptr(V), _ptr(N), _ptr(L), BH, cap, d, n1, n2, c, m,
                                  _ptr(sk), _ptr(f), _ptr(rec["match"]), _ptr(rec["sim"]),
                                  _ptr(rec["margin"]), _ptr(rec["cut"]), maxch, _ptr(rec["origin"]),
                                  _ptr(rec["merged"]), _ptr(lim), _threads(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_csm_round failed ({rc})")
    return dict(K=K, V=V, N=N, len=L, **rec)


def append(K, V, N, length, k_new, v_new, skip=None):
    """Decode append. Returns new (K, V, N, len) copies and the count of full units."""
    K, V, N, L = _f64(K).copy(), _f64(V).copy(), _i32(N).copy(), _i32(length).copy()
    BH, cap, d = K.shape
    kn, vn = _f64(k_new).reshape(BH, d), _f64(v_new).reshape(BH, d)
    sk = None if skip is None else np.ascontiguousarray(np.asarray(skip, dtype=np.uint8))
    full = _load().oracle_append(_ptr(K), _ptr(V), _ptr(N), _ptr(L), BH, cap, d,
                                 _ptr(kn), _ptr(vn), _ptr(sk))
    return K, V, N, L, int(full)


def decode_attn_logn(q, K, V, N, length, h_q: int, scale=None, nthreads=None):
    """Degree-aware attention. q: [B, Hq, d]; K, V: [B, Hkv, cap, d]; N: [B, Hkv, cap];
    length: [B, Hkv]. Returns o [B, Hq, d] in fp64."""
    K, V, N, L = _f64(K), _f64(V), _i32(N), _i32(length)
    B, Hkv, cap, d = K.shape
    q = _f64(q).reshape(B, h_q, d)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    out = np.zeros((B, h_q, d))
    _load().oracle_decode_attn_logn(_ptr(q), _ptr(K), _ptr(V), _ptr(N), _ptr(L), B, Hkv, h_q,
                                    cap, d, float(scale), _ptr(out), _threads(nthreads))
    return out


def prefill_attn(q, K, V, n: int, h_q: int, scale=None, rows=None, nthreads=None):
    """Causal prefill attention with every degree 1 ([Chelsea] §三 算法流程, Algorithm 1:
    O = FlashAttn(Q, K, V) on the prompt). q: [B, Hq, n, d]; K, V: [B, Hkv, cap, d]
    (rows 0..n-1 are the prompt). rows: query positions to evaluate (default all).
    Returns o [B, Hq, len(rows), d] in fp64."""
    K, V = _f64(K), _f64(V)
    B, Hkv, cap, d = K.shape
    q = _f64(q).reshape(B, h_q, n, d)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    r = None if rows is None else _i32(rows)
    nrows = n if r is None else int(r.size)
    if r is not None and (r.min(initial=0) < 0 or r.max(initial=0) >= n):
        raise ValueError("query rows outside the prompt")
    out = np.zeros((B, h_q, nrows, d))
    _load().oracle_prefill_attn(_ptr(q), _ptr(K), _ptr(V), B, Hkv, h_q, n, cap, d, float(scale), _ptr(r), nrows,
                                _ptr(out), _threads(nthreads))
    return out
