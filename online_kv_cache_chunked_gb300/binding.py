"""ctypes binding of the C ABI in include/csmkv.h (argument marshalling only).

Every function here has the C name and forwards to libcsmkv.so; all the work
of the path runs in its CUDA kernels. Tensors are torch CUDA tensors (device
memory and streams come from PyTorch); the library itself never allocates.
There is no CPU fallback: if the library is missing, load() raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

BF16, F32 = 0, 1
_DTYPES = {torch.bfloat16: BF16, torch.float32: F32}

STATUS = {0: "CSMKV_OK", 1: "CSMKV_ERR_ARG", 2: "CSMKV_ERR_DTYPE", 3: "CSMKV_ERR_ALIGN",
          4: "CSMKV_ERR_CAPACITY", 5: "CSMKV_ERR_WORKSPACE", 6: "CSMKV_ERR_TIMEOUT",
          7: "CSMKV_ERR_CUDA", 8: "CSMKV_ERR_UNSUPPORTED"}


class CsmkvError(RuntimeError):
    def __init__(self, fn, code):
        self.code = int(code)
        super().__init__(f"{fn}: {STATUS.get(self.code, self.code)} ({status_str(self.code)})")


class Cache(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("h_kv", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("cap", ctypes.c_int32), ("dtype", ctypes.c_int32)]


class CsmOptions(ctypes.Structure):
    _fields_ = [("wait_timeout_ns", ctypes.c_int64), ("withhold_signals", ctypes.c_int32),
                ("kernel", ctypes.c_int32), ("seq_max_chunks", ctypes.c_void_p)]


CSM_KERNEL_AUTO, CSM_KERNEL_SIMT, CSM_KERNEL_TC_SPLIT = 0, 1, 3


class CsmRoundPlan(ctypes.Structure):
    _fields_ = [("step", ctypes.c_int32), ("r", ctypes.c_double), ("seq_mask", ctypes.c_void_p),
                ("seq_max_chunks", ctypes.c_void_p)]


class Pages(ctypes.Structure):
    _fields_ = [("table", ctypes.c_void_p), ("page_rows", ctypes.c_int32), ("max_pages", ctypes.c_int32),
                ("num_pages", ctypes.c_int32)]


class PagedKV:
    """A paged (block-table) cache as the C ABI sees it: pools K, V [num_pages, page_rows,
    head_dim] (cache dtype) and N [num_pages, page_rows] (int32), a block table
    [batch * h_kv, max_pages] (int32, device), and the logical shape it stands for
    (batch, h_kv, cap = max_pages * page_rows)."""

    def __init__(self, K, V, N, table, batch, h_kv):
        self.K, self.V, self.N, self.table = K, V, N, table
        self.batch, self.h_kv = int(batch), int(h_kv)
        self.num_pages, self.page_rows, self.head_dim = (int(x) for x in K.shape)
        self.max_pages = int(table.shape[1])

    @property
    def cap(self):
        return self.max_pages * self.page_rows

    def cache(self) -> "Cache":
        return Cache(self.batch, self.h_kv, self.head_dim, self.cap, _DTYPES[self.K.dtype])

    def pages(self) -> Pages:
        return Pages(self.table.data_ptr(), self.page_rows, self.max_pages, self.num_pages)


class CsmDecodeLoop(ctypes.Structure):
    _fields_ = [("K", ctypes.c_void_p), ("V", ctypes.c_void_p), ("N", ctypes.c_void_p), ("len", ctypes.c_void_p),
                ("cache", Cache), ("h_q", ctypes.c_int32), ("scale", ctypes.c_float),
                ("q", ctypes.c_void_p), ("k_new", ctypes.c_void_p), ("v_new", ctypes.c_void_p),
                ("out", ctypes.c_void_p), ("n1", ctypes.c_int32), ("n2", ctypes.c_int32), ("c", ctypes.c_int32),
                ("head_mask", ctypes.c_void_p), ("csm_kernel", ctypes.c_int32),
                ("rounds", ctypes.POINTER(CsmRoundPlan)), ("n_rounds", ctypes.c_int32),
                ("ws_csm", ctypes.c_void_p), ("ws_csm_bytes", ctypes.c_size_t),
                ("ws_append", ctypes.c_void_p), ("ws_append_bytes", ctypes.c_size_t),
                ("ws_attn", ctypes.c_void_p), ("ws_attn_bytes", ctypes.c_size_t),
                ("attn_events", ctypes.POINTER(ctypes.c_void_p)), ("csm_events", ctypes.POINTER(ctypes.c_void_p)),
                ("l2_flush", ctypes.c_void_p), ("l2_flush_bytes", ctypes.c_size_t),
                ("fused_append", ctypes.c_int32), ("pages", ctypes.POINTER(Pages))]


_lib = None

P = ctypes.c_void_p
I32 = ctypes.c_int32
I64 = ctypes.c_int64
F64 = ctypes.c_double
SZ = ctypes.c_size_t
CP = ctypes.POINTER(Cache)

_SIGS = {
    "csm_workspace_bytes": (SZ, [CP, I32, I32, I32]),
    "csm_compress": (ctypes.c_int, [P, P, P, P, CP, I32, I32, I32, F64, P, P, P, SZ, P]),
    "csm_compress_ex": (ctypes.c_int, [P, P, P, P, CP, I32, I32, I32, F64, P, P, P,
                                       ctypes.POINTER(CsmOptions), P, SZ, P]),
    "csm_max_chunks": (I32, [CP, I32, I32, I32]),
    "csm_append_workspace_bytes": (SZ, []),
    "csm_append": (ctypes.c_int, [P, P, P, P, CP, P, P, P, P, SZ, P]),
    "decode_attn_workspace_bytes": (SZ, [CP, I32]),
    "decode_attn_logn": (ctypes.c_int, [P, P, P, P, P, CP, I32, ctypes.c_float, P, P, SZ, P]),
    "decode_attn_logn_noalloc": (ctypes.c_int, [P, P, P, P, P, CP, I32, ctypes.c_float, P, P]),
    "decode_step_logn": (ctypes.c_int, [P, P, P, P, P, P, P, CP, I32, ctypes.c_float, P, P, SZ, P]),
    "csm_decode_run": (ctypes.c_int, [ctypes.POINTER(CsmDecodeLoop), I32, I32, P]),
    "csm_append_paged": (ctypes.c_int, [P, P, P, P, CP, ctypes.POINTER(Pages), P, P, P, P, SZ, P]),
    "csm_compress_paged": (ctypes.c_int, [P, P, P, P, CP, ctypes.POINTER(Pages), I32, I32, I32, F64, P, P, P,
                                          ctypes.POINTER(CsmOptions), P, SZ, P]),
    "decode_attn_logn_paged": (ctypes.c_int, [P, P, P, P, P, CP, ctypes.POINTER(Pages), I32, ctypes.c_float, P,
                                              P, SZ, P]),
    "decode_step_logn_paged": (ctypes.c_int, [P, P, P, P, P, P, P, CP, ctypes.POINTER(Pages), I32,
                                              ctypes.c_float, P, P, SZ, P]),
    "prefill_workspace_bytes": (SZ, []),
    "prefill_attn": (ctypes.c_int, [P, P, P, CP, I32, P, I32, ctypes.c_float, P, P, SZ, P]),
    "prefill_attn_csm": (ctypes.c_int, [P, P, P, CP, I32, P, I32, ctypes.c_float, P, P, P, P, P, CP, I32, I32,
                                        I32, F64, P, P, SZ, P]),
    "csm_budget": (F64, [I64, F64, I64]),
    "csm_should_trigger": (ctypes.c_int, [I64, F64, I32]),
    "csm_ratio": (F64, [I32, F64, F64, F64]),
    "csm_edges_per_chunk": (I32, [F64, I32]),
    "csm_num_chunks": (I64, [I64, I32, I32, I32]),
    "csm_len_after": (I64, [I64, I32, I32, I32, I32]),
    "csm_chunks_to_budget": (I32, [I64, F64, I32, I32, I32, I32]),
    "csmkv_device_status": (ctypes.c_int, [P, P]),
    "csmkv_clear_status": (ctypes.c_int, [P, P]),
    "csmkv_status_str": (ctypes.c_char_p, [ctypes.c_int]),
}


def library_path() -> str:
    return _build.OUT


def load():
    """Loads libcsmkv.so (built by build()); raises if it is missing."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build() "
                               "(there is no fallback path)")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(fn, rc):
    if rc != 0:
        raise CsmkvError(fn, rc)


def cache_desc(K: torch.Tensor) -> Cache:
    """Descriptor of a [batch, h_kv, cap, head_dim] cache tensor."""
    if K.dim() != 4 or not K.is_contiguous():
        raise ValueError("cache tensors are contiguous [batch, h_kv, cap, head_dim]")
    if K.dtype not in _DTYPES:
        raise ValueError(f"unsupported cache dtype {K.dtype}")
    b, h, cap, d = K.shape
    return Cache(b, h, d, cap, _DTYPES[K.dtype])


def new_workspace(nbytes: int, device=None) -> torch.Tensor:
    """A zero-filled device workspace (allocated by PyTorch, not the library)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device or "cuda")


# ---------------------------------------------------------------- CSM
def csm_workspace_bytes(cache: Cache, n1: int, n2: int, c: int) -> int:
    return int(load().csm_workspace_bytes(ctypes.byref(cache), n1, n2, c))


def csm_max_chunks(cache: Cache, n1: int, n2: int, c: int) -> int:
    return int(load().csm_max_chunks(ctypes.byref(cache), n1, n2, c))


def csm_compress(K, V, N, length, n1, n2, c, r, head_mask=None, seq_mask=None, workspace=None,
                 stream=None):
    cache = cache_desc(K)
    rc = load().csm_compress(_ptr(K), _ptr(V), _ptr(N), _ptr(length), ctypes.byref(cache), n1, n2, c,
                             float(r), _ptr(head_mask), _ptr(seq_mask), _ptr(workspace),
                             workspace.numel() if workspace is not None else 0, _stream(stream))
    _check("csm_compress", rc)


def csm_compress_ex(K, V, N, length, n1, n2, c, r, head_mask=None, seq_mask=None, match_out=None,
                    wait_timeout_ns=0, withhold_signals=0, kernel=0, seq_max_chunks=None, workspace=None,
                    stream=None):
    """seq_max_chunks: optional device int32 [batch]; entry > 0 caps that sequence's
    round at its oldest `entry` chunks (budget-exact compression)."""
    cache = cache_desc(K)
    opts = CsmOptions(int(wait_timeout_ns), int(withhold_signals), int(kernel), _ptr(seq_max_chunks))
    rc = load().csm_compress_ex(_ptr(K), _ptr(V), _ptr(N), _ptr(length), ctypes.byref(cache), n1, n2, c,
                                float(r), _ptr(head_mask), _ptr(seq_mask), _ptr(match_out),
                                ctypes.byref(opts), _ptr(workspace),
                                workspace.numel() if workspace is not None else 0, _stream(stream))
    _check("csm_compress_ex", rc)


# ---------------------------------------------------------------- append
def csm_append_workspace_bytes() -> int:
    return int(load().csm_append_workspace_bytes())


def csm_append(K, V, N, length, k_new, v_new, seq_mask=None, workspace=None, stream=None):
    cache = cache_desc(K)
    rc = load().csm_append(_ptr(K), _ptr(V), _ptr(N), _ptr(length), ctypes.byref(cache), _ptr(k_new),
                           _ptr(v_new), _ptr(seq_mask), _ptr(workspace),
                           workspace.numel() if workspace is not None else 0, _stream(stream))
    _check("csm_append", rc)


# ---------------------------------------------------------------- attention
def decode_attn_workspace_bytes(cache: Cache, h_q: int) -> int:
    return int(load().decode_attn_workspace_bytes(ctypes.byref(cache), h_q))


def decode_attn_logn(q, K, V, N, length, out, workspace, scale=None, stream=None):
    cache = cache_desc(K)
    h_q = q.shape[1]
    if scale is None:
        scale = 1.0 / (K.shape[-1] ** 0.5)
    rc = load().decode_attn_logn(_ptr(q), _ptr(K), _ptr(V), _ptr(N), _ptr(length), ctypes.byref(cache), h_q,
                                 float(scale), _ptr(out), _ptr(workspace), workspace.numel(), _stream(stream))
    _check("decode_attn_logn", rc)


def decode_step_logn(q, k_new, v_new, K, V, N, length, out, workspace, scale=None, stream=None):
    """csm_append(k_new, v_new) then decode_attn_logn, fused into one kernel for bf16."""
    cache = cache_desc(K)
    h_q = q.shape[1]
    if scale is None:
        scale = 1.0 / (K.shape[-1] ** 0.5)
    rc = load().decode_step_logn(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(K), _ptr(V), _ptr(N), _ptr(length),
                                 ctypes.byref(cache), h_q, float(scale), _ptr(out), _ptr(workspace),
                                 workspace.numel(), _stream(stream))
    _check("decode_step_logn", rc)


def decode_attn_logn_noalloc(q, K, V, N, length, out, scale=None, stream=None):
    """decode_attn_logn with the library's own fixed scratch instead of a workspace,
    for callers that cannot allocate device memory."""
    cache = cache_desc(K)
    h_q = q.shape[1]
    if scale is None:
        scale = 1.0 / (K.shape[-1] ** 0.5)
    rc = load().decode_attn_logn_noalloc(_ptr(q), _ptr(K), _ptr(V), _ptr(N), _ptr(length), ctypes.byref(cache),
                                         h_q, float(scale), _ptr(out), _stream(stream))
    _check("decode_attn_logn_noalloc", rc)


# ---------------------------------------------------------------- decode loop
def _event_array(events):
    if events is None:
        return None
    handles = []
    for e in events:
        h = e.cuda_event
        if not h:
            raise ValueError("events must have been recorded once (torch creates them lazily)")
        handles.append(h)
    return (ctypes.c_void_p * len(handles))(*handles)


def csm_decode_run(K, V, N, length, q, k_new, v_new, out, n1, n2, c, rounds=(), head_mask=None,
                   ws_csm=None, ws_append=None, ws_attn=None, first_step=1, steps=None, csm_kernel=0,
                   attn_events=None, csm_events=None, l2_flush=None, scale=None, stream=None, fused_append=False,
                   paged=None):
    """Decode steps first_step .. first_step+steps-1 (1-based) issued natively: per step
    append(k_new[i-1], v_new[i-1]), attention(q[i-1]) -> out[i-1], then the planned
    rounds of that step. rounds: iterable of (step, r, seq_mask or None[, seq_max_chunks or
    None]), sorted by step.
    attn_events / csm_events: torch.cuda.Event lists (2 per call), recorded once before.
    paged: a PagedKV (K, V, N are then its pools; every call uses the paged entry points)."""
    cache = paged.cache() if paged is not None else cache_desc(K)
    if steps is None:
        steps = q.shape[0] - first_step + 1
    if scale is None:
        scale = 1.0 / (K.shape[-1] ** 0.5)
    rl = list(rounds)
    rarr = (CsmRoundPlan * max(1, len(rl)))()
    for k, rd in enumerate(rl):
        st, r, sm = rd[:3]
        lim = rd[3] if len(rd) > 3 else None
        rarr[k] = CsmRoundPlan(int(st), float(r), _ptr(sm), _ptr(lim))
    ae, ce = _event_array(attn_events), _event_array(csm_events)
    nb = lambda t: t.numel() * t.element_size() if t is not None else 0  # noqa: E731
    loop = CsmDecodeLoop(_ptr(K), _ptr(V), _ptr(N), _ptr(length), cache, int(q.shape[2]), float(scale),
                         _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(out), int(n1), int(n2), int(c), _ptr(head_mask),
                         int(csm_kernel), rarr, len(rl), _ptr(ws_csm), nb(ws_csm), _ptr(ws_append), nb(ws_append),
                         _ptr(ws_attn), nb(ws_attn), ae, ce, _ptr(l2_flush), nb(l2_flush), int(bool(fused_append)))
    pg = paged.pages() if paged is not None else None
    if pg is not None:
        loop.pages = ctypes.pointer(pg)
    rc = load().csm_decode_run(ctypes.byref(loop), int(first_step), int(steps), _stream(stream))
    _check("csm_decode_run", rc)


# ---------------------------------------------------------------- paged layout
def csm_append_paged(kv, length, k_new, v_new, seq_mask=None, workspace=None, stream=None):
    cache, pg = kv.cache(), kv.pages()
    rc = load().csm_append_paged(_ptr(kv.K), _ptr(kv.V), _ptr(kv.N), _ptr(length), ctypes.byref(cache),
                                 ctypes.byref(pg), _ptr(k_new), _ptr(v_new), _ptr(seq_mask), _ptr(workspace),
                                 workspace.numel() if workspace is not None else 0, _stream(stream))
    _check("csm_append_paged", rc)


def csm_compress_paged(kv, length, n1, n2, c, r, head_mask=None, seq_mask=None, match_out=None, wait_timeout_ns=0,
                       seq_max_chunks=None, workspace=None, stream=None):
    cache, pg = kv.cache(), kv.pages()
    opts = CsmOptions(int(wait_timeout_ns), 0, 0, _ptr(seq_max_chunks))
    rc = load().csm_compress_paged(_ptr(kv.K), _ptr(kv.V), _ptr(kv.N), _ptr(length), ctypes.byref(cache),
                                   ctypes.byref(pg), n1, n2, c, float(r), _ptr(head_mask), _ptr(seq_mask),
                                   _ptr(match_out), ctypes.byref(opts), _ptr(workspace),
                                   workspace.numel() if workspace is not None else 0, _stream(stream))
    _check("csm_compress_paged", rc)


def decode_attn_logn_paged(q, kv, length, out, workspace, scale=None, stream=None):
    cache, pg = kv.cache(), kv.pages()
    if scale is None:
        scale = 1.0 / (kv.head_dim ** 0.5)
    rc = load().decode_attn_logn_paged(_ptr(q), _ptr(kv.K), _ptr(kv.V), _ptr(kv.N), _ptr(length),
                                       ctypes.byref(cache), ctypes.byref(pg), q.shape[1], float(scale), _ptr(out),
                                       _ptr(workspace), workspace.numel(), _stream(stream))
    _check("decode_attn_logn_paged", rc)


def decode_step_logn_paged(q, k_new, v_new, kv, length, out, workspace, scale=None, stream=None):
    cache, pg = kv.cache(), kv.pages()
    if scale is None:
        scale = 1.0 / (kv.head_dim ** 0.5)
    rc = load().decode_step_logn_paged(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(kv.K), _ptr(kv.V), _ptr(kv.N),
                                       _ptr(length), ctypes.byref(cache), ctypes.byref(pg), q.shape[1], float(scale),
                                       _ptr(out), _ptr(workspace), workspace.numel(), _stream(stream))
    _check("decode_step_logn_paged", rc)


# ---------------------------------------------------------------- host helpers
# ---------------------------------------------------------------- prefill
def prefill_workspace_bytes() -> int:
    return int(load().prefill_workspace_bytes())


def prefill_attn(q, K, V, n, out, workspace, seq_len=None, scale=None, stream=None):
    """Causal prefill attention over the prompt rows [0, n) of the cache (K, V).
    q, out: [batch, h_q, n, 128]; seq_len: optional int32 [batch] prompt lengths."""
    cache = cache_desc(K)
    rc = load().prefill_attn(_ptr(q), _ptr(K), _ptr(V), ctypes.byref(cache), int(n), _ptr(seq_len), q.shape[1],
                             float(scale or 0.0), _ptr(out), _ptr(workspace), workspace.numel(), _stream(stream))
    _check("prefill_attn", rc)


def prefill_attn_csm(q, K, V, n, out, K_out, V_out, N_out, len_out, n1, n2, c, r, workspace, seq_len=None,
                     head_mask=None, scale=None, stream=None):
    """prefill_attn plus the prompt's first CSM round (ratio r) written to a second cache."""
    cache = cache_desc(K)
    cache_out = cache_desc(K_out)
    rc = load().prefill_attn_csm(_ptr(q), _ptr(K), _ptr(V), ctypes.byref(cache), int(n), _ptr(seq_len), q.shape[1],
                                 float(scale or 0.0), _ptr(out), _ptr(K_out), _ptr(V_out), _ptr(N_out),
                                 _ptr(len_out), ctypes.byref(cache_out), n1, n2, c, float(r), _ptr(head_mask),
                                 _ptr(workspace), workspace.numel(), _stream(stream))
    _check("prefill_attn_csm", rc)


def csm_budget(n, R, Gamma) -> float:
    return float(load().csm_budget(int(n), float(R), int(Gamma)))


def csm_should_trigger(s, B, g) -> bool:
    return bool(load().csm_should_trigger(int(s), float(B), int(g)))


def csm_ratio(j, r_init, dr, r_min) -> float:
    return float(load().csm_ratio(int(j), float(r_init), float(dr), float(r_min)))


def csm_edges_per_chunk(r, c) -> int:
    return int(load().csm_edges_per_chunk(float(r), int(c)))


def csm_num_chunks(s, n1, n2, c) -> int:
    return int(load().csm_num_chunks(int(s), int(n1), int(n2), int(c)))


def csm_len_after(s, n1, n2, c, m) -> int:
    return int(load().csm_len_after(int(s), int(n1), int(n2), int(c), int(m)))


def csm_chunks_to_budget(s, B, n1, n2, c, m) -> int:
    return int(load().csm_chunks_to_budget(int(s), float(B), int(n1), int(n2), int(c), int(m)))


def csmkv_device_status(workspace, stream=None) -> int:
    return int(load().csmkv_device_status(_ptr(workspace), _stream(stream)))


def csmkv_clear_status(workspace, stream=None) -> None:
    _check("csmkv_clear_status", load().csmkv_clear_status(_ptr(workspace), _stream(stream)))


def status_str(code: int) -> str:
    try:
        return load().csmkv_status_str(int(code)).decode()
    except Exception:  # the library may be missing while formatting an error
        return "?"
