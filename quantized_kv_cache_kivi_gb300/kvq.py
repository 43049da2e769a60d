"""Thin ctypes binding of libkvq.so (include/kvq.h), same names as the C ABI.

Argument marshalling only: every step of the computation runs in the CUDA
kernels of libkvq.so.  torch tensors are passed as raw device pointers
(``data_ptr()``) and streams as ``cuda_stream`` handles.  There is no CPU
fallback: if the library cannot be built or loaded, ``lib()`` raises.

Also provides ``alloc_cache``, which allocates the device buffers of a cache
with torch (the library itself allocates nothing) and fills the C struct.
"""
import ctypes
import math
import os

from . import build as _build

KVQ_OK = 0
KVQ_FLUSH_DUE = 1
KVQ_ERR_INVALID_ARG = -1
KVQ_ERR_UNSUPPORTED = -2
KVQ_ERR_CAPACITY = -3
KVQ_ERR_CUDA = -4
KVQ_ERR_WORKSPACE = -5
KVQ_POLICY_KIVI = 0
KVQ_POLICY_FP16_TAIL = 1
KVQ_ZERO_MIN, KVQ_ZERO_INT = 0, 1
KVQ_STEP_ATTEND_FIRST, KVQ_STEP_FLUSH_FIRST = 0, 1
KVQ_MAX_SEGMENTS = 8
KVQ_MAX_SPLITS = 128
KVQ_MAX_SEQS = 256


class kvq_segment(ctypes.Structure):
    _fields_ = [("bits", ctypes.c_int32), ("capacity", ctypes.c_int32),
                ("nk", ctypes.c_int32), ("nv", ctypes.c_int32),
                ("k_codes", ctypes.c_void_p), ("k_scale", ctypes.c_void_p),
                ("k_zero", ctypes.c_void_p), ("v_codes", ctypes.c_void_p),
                ("v_scale", ctypes.c_void_p), ("v_zero", ctypes.c_void_p)]


class kvq_cache(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("h_kv", ctypes.c_int32), ("h_q", ctypes.c_int32),
                ("d_h", ctypes.c_int32), ("group", ctypes.c_int32),
                ("resid_cap", ctypes.c_int32), ("policy", ctypes.c_int32),
                ("sm_scale", ctypes.c_float), ("n_seg", ctypes.c_int32),
                ("seg", kvq_segment * KVQ_MAX_SEGMENTS),
                ("k_resid", ctypes.c_void_p), ("v_resid", ctypes.c_void_p),
                ("nkr", ctypes.c_int32), ("nvr", ctypes.c_int32),
                ("k_ring_start", ctypes.c_int32), ("v_ring_start", ctypes.c_int32),
                ("zero_point", ctypes.c_int32), ("group_v", ctypes.c_int32)]


class kvq_window_plan(ctypes.Structure):
    _fields_ = [("window", ctypes.c_int32), ("n_windows", ctypes.c_int32),
                ("bits", ctypes.POINTER(ctypes.c_int8)),
                ("perm", ctypes.POINTER(ctypes.c_int32))]


class kvq_seq_state(ctypes.Structure):
    _fields_ = [("nk", ctypes.c_int32), ("nv", ctypes.c_int32),
                ("nkr", ctypes.c_int32), ("nvr", ctypes.c_int32),
                ("k_ring_start", ctypes.c_int32), ("v_ring_start", ctypes.c_int32)]


class kvq_paged_cache(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("h_kv", ctypes.c_int32), ("h_q", ctypes.c_int32),
                ("d_h", ctypes.c_int32), ("group", ctypes.c_int32), ("group_v", ctypes.c_int32),
                ("resid_cap", ctypes.c_int32), ("bits", ctypes.c_int32),
                ("zero_point", ctypes.c_int32), ("page_tokens", ctypes.c_int32),
                ("n_pages", ctypes.c_int32), ("max_pages", ctypes.c_int32),
                ("sm_scale", ctypes.c_float),
                ("k_codes", ctypes.c_void_p), ("k_scale", ctypes.c_void_p),
                ("k_zero", ctypes.c_void_p), ("v_codes", ctypes.c_void_p),
                ("v_scale", ctypes.c_void_p), ("v_zero", ctypes.c_void_p),
                ("block_table", ctypes.c_void_p),
                ("k_resid", ctypes.c_void_p), ("v_resid", ctypes.c_void_p),
                ("err", ctypes.c_void_p),
                ("seq", kvq_seq_state * KVQ_MAX_SEQS)]


_LIB = None
_P = ctypes.c_void_p


def lib():
    """Build (if stale) and load libkvq.so; raises if that is impossible."""
    global _LIB
    if _LIB is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        cp = ctypes.POINTER(kvq_cache)
        L.kvq_quantize_append.argtypes = [cp, _P, _P, ctypes.c_int32,
                                          ctypes.POINTER(kvq_window_plan), _P]
        L.kvq_flush_residual.argtypes = [cp, _P]
        L.kvq_workspace_bytes.argtypes = [cp, ctypes.c_int32]
        L.kvq_workspace_bytes.restype = ctypes.c_size_t
        L.kvq_workspace_init.argtypes = [_P, ctypes.c_size_t, _P]
        L.kvq_decode_attention.argtypes = [cp, _P, _P, _P, ctypes.c_size_t, _P]
        L.kvq_workspace_error.argtypes = [_P, ctypes.POINTER(ctypes.c_int32), _P]
        L.kvq_decode_step.argtypes = [cp, _P, _P, _P, _P, _P, ctypes.c_size_t, ctypes.c_int32, _P]
        L.kvq_decode_step.restype = ctypes.c_int
        L.kvq_decode_step_host.argtypes = [cp, _P, _P, _P, _P, _P, ctypes.c_size_t, ctypes.c_int32, _P]
        L.kvq_decode_step_host.restype = ctypes.c_int
        L.kvq_decode_attention_noalloc.argtypes = [cp, _P, _P, _P]
        L.kvq_decode_attention_noalloc.restype = ctypes.c_int
        L.kvq_noalloc_error.argtypes = [ctypes.POINTER(ctypes.c_int32), _P]
        L.kvq_noalloc_error.restype = ctypes.c_int
        L.kvq_window_assign_workspace_bytes.argtypes = [ctypes.c_int32] * 5
        L.kvq_window_assign_workspace_bytes.restype = ctypes.c_size_t
        L.kvq_window_assign.argtypes = [_P, _P] + [ctypes.c_int32] * 6 + \
            [ctypes.c_float, ctypes.c_float, ctypes.c_int32, _P, ctypes.c_size_t,
             ctypes.POINTER(ctypes.c_int8), ctypes.POINTER(ctypes.c_int32),
             ctypes.POINTER(ctypes.c_double), _P]
        L.kvq_window_assign_eq8_workspace_bytes.argtypes = [ctypes.c_int32] * 5
        L.kvq_window_assign_eq8_workspace_bytes.restype = ctypes.c_size_t
        L.kvq_window_assign_eq8.argtypes = [_P, _P] + [ctypes.c_int32] * 5 + \
            [ctypes.c_double, ctypes.c_double, ctypes.c_int32, _P, ctypes.c_size_t,
             ctypes.POINTER(ctypes.c_int8), ctypes.POINTER(ctypes.c_int32),
             ctypes.POINTER(ctypes.c_double), _P]
        pp = ctypes.POINTER(kvq_paged_cache)
        L.kvq_paged_append.argtypes = [pp, _P, _P, ctypes.c_int32,
                                       ctypes.POINTER(ctypes.c_int32), _P]
        L.kvq_paged_flush_residual.argtypes = [pp, _P]
        L.kvq_paged_workspace_bytes.argtypes = [pp, ctypes.c_int32]
        L.kvq_paged_workspace_bytes.restype = ctypes.c_size_t
        L.kvq_paged_decode_attention.argtypes = [pp, _P, _P, _P, ctypes.c_size_t, _P]
        L.kvq_status_string.argtypes = [ctypes.c_int]
        L.kvq_status_string.restype = ctypes.c_char_p
        L.kvq_last_error_string.argtypes = []
        L.kvq_last_error_string.restype = ctypes.c_char_p
        for name in ("kvq_quantize_append", "kvq_flush_residual", "kvq_workspace_init",
                     "kvq_decode_attention", "kvq_workspace_error", "kvq_window_assign",
                     "kvq_window_assign_eq8", "kvq_paged_append", "kvq_paged_flush_residual",
                     "kvq_paged_decode_attention"):
            getattr(L, name).restype = ctypes.c_int
        _LIB = L
    return _LIB


class KvqError(RuntimeError):
    def __init__(self, status, where):
        L = lib()
        super().__init__("%s: %s (%s)" % (where, L.kvq_status_string(status).decode(),
                                          L.kvq_last_error_string().decode()))
        self.status = status


def _check(status, where, ok=(KVQ_OK,)):
    if status not in ok:
        raise KvqError(status, where)
    return status


def _stream(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


# ---------------------------------------------------------------------------
# same-named wrappers
# ---------------------------------------------------------------------------
def kvq_quantize_append(cache, k_new, v_new, plan=None, stream=None):
    """Append fp16 [B][H_kv][T][d] tokens; returns KVQ_OK or KVQ_FLUSH_DUE."""
    T = int(k_new.shape[2])
    p = ctypes.byref(plan) if plan is not None else None
    st = lib().kvq_quantize_append(ctypes.byref(cache.c), _ptr(k_new), _ptr(v_new), T, p,
                                   _stream(stream))
    return _check(st, "kvq_quantize_append", ok=(KVQ_OK, KVQ_FLUSH_DUE))


def kvq_flush_residual(cache, stream=None):
    return _check(lib().kvq_flush_residual(ctypes.byref(cache.c), _stream(stream)),
                  "kvq_flush_residual")


def kvq_workspace_bytes(cache, max_splits=KVQ_MAX_SPLITS):
    return int(lib().kvq_workspace_bytes(ctypes.byref(cache.c), int(max_splits)))


def kvq_workspace_init(ws, stream=None):
    return _check(lib().kvq_workspace_init(_ptr(ws), ws.numel() * ws.element_size(),
                                           _stream(stream)), "kvq_workspace_init")


def kvq_decode_attention(cache, q, out, ws, stream=None):
    st = lib().kvq_decode_attention(ctypes.byref(cache.c), _ptr(q), _ptr(out), _ptr(ws),
                                    ws.numel() * ws.element_size(), _stream(stream))
    return _check(st, "kvq_decode_attention")


def kvq_decode_step(cache, k_new, v_new, q, out, ws, stream=None, order=KVQ_STEP_ATTEND_FIRST):
    """Append one token per head, then decode attention and the K flush if
    due, in `order` (KVQ_STEP_FLUSH_FIRST: KIVI Algorithm 1's)."""
    st = lib().kvq_decode_step(ctypes.byref(cache.c), _ptr(k_new), _ptr(v_new), _ptr(q), _ptr(out), _ptr(ws),
                               ws.numel() * ws.element_size(), order, _stream(stream))
    return _check(st, "kvq_decode_step")


def kvq_decode_step_host(cache, host_in, host_out, dev_in, dev_out, ws, stream=None,
                         order=KVQ_STEP_ATTEND_FIRST):
    """kvq_decode_step with its inputs copied from host memory and its output
    copied back (host_in / dev_in: [new K | new V | q] fp16)."""
    st = lib().kvq_decode_step_host(ctypes.byref(cache.c), _ptr(host_in), _ptr(host_out), _ptr(dev_in),
                                    _ptr(dev_out), _ptr(ws), ws.numel() * ws.element_size(), order,
                                    _stream(stream))
    return _check(st, "kvq_decode_step_host")


def kvq_decode_attention_noalloc(cache, q, out, stream=None):
    """kvq_decode_attention with the library's static scratch (no workspace)."""
    st = lib().kvq_decode_attention_noalloc(ctypes.byref(cache.c), _ptr(q), _ptr(out),
                                            _stream(stream))
    return _check(st, "kvq_decode_attention_noalloc")


def kvq_noalloc_error(stream=None):
    """Error word of the static scratch after the last no-workspace call."""
    v = ctypes.c_int32(0)
    _check(lib().kvq_noalloc_error(ctypes.byref(v), _stream(stream)), "kvq_noalloc_error")
    return v.value


def kvq_workspace_error(ws, stream=None):
    v = ctypes.c_int32(0)
    _check(lib().kvq_workspace_error(_ptr(ws), ctypes.byref(v), _stream(stream)),
           "kvq_workspace_error")
    return v.value


def kvq_window_assign_workspace_bytes(batch, h_kv, d_h, M, S):
    return int(lib().kvq_window_assign_workspace_bytes(batch, h_kv, d_h, M, S))


def kvq_window_assign(keys, text_keys, S, frac8, frac4, first_window_fp16=False, ws=None,
                      stream=None):
    """keys fp16 [B][H][M][d], text fp16 [B][H][N][d] -> (bits, perm, sim) numpy arrays."""
    import numpy as np
    import torch
    B, H, M, d = keys.shape
    N = text_keys.shape[2]
    nw = M // S
    need = kvq_window_assign_workspace_bytes(B, H, d, M, S)
    if ws is None:
        ws = torch.empty(max(need, 16), dtype=torch.uint8, device=keys.device)
    bits = np.zeros(nw, np.int8)
    perm = np.zeros(nw, np.int32)
    sim = np.zeros(nw, np.float64)
    st = lib().kvq_window_assign(_ptr(keys), _ptr(text_keys), B, H, d, M, S, N, float(frac8),
                                 float(frac4), int(bool(first_window_fp16)), _ptr(ws),
                                 ws.numel(), bits.ctypes.data_as(ctypes.POINTER(ctypes.c_int8)),
                                 perm.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                 sim.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                                 _stream(stream))
    _check(st, "kvq_window_assign")
    return bits, perm, sim


def kvq_window_assign_eq8_workspace_bytes(batch, dim, M, S, N):
    return int(lib().kvq_window_assign_eq8_workspace_bytes(batch, dim, M, S, N))


def kvq_window_assign_eq8(vision, text, S, layer_sim, alpha, first_window_fp16=False, ws=None,
                          stream=None):
    """vision fp16 [B][M][dim], text fp16 [B][N][dim] -> (bits, perm, sim [B][n_windows])."""
    import numpy as np
    import torch
    B, M, dim = vision.shape
    N = text.shape[1]
    nw = M // S
    need = kvq_window_assign_eq8_workspace_bytes(B, dim, M, S, N)
    if ws is None:
        ws = torch.empty(max(need, 16), dtype=torch.uint8, device=vision.device)
    bits = np.zeros(nw, np.int8)
    perm = np.zeros(nw, np.int32)
    sim = np.zeros((B, nw), np.float64)
    st = lib().kvq_window_assign_eq8(_ptr(vision), _ptr(text), B, dim, M, S, N, float(layer_sim),
                                     float(alpha), int(bool(first_window_fp16)), _ptr(ws), ws.numel(),
                                     bits.ctypes.data_as(ctypes.POINTER(ctypes.c_int8)),
                                     perm.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                     sim.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                                     _stream(stream))
    _check(st, "kvq_window_assign_eq8")
    return bits, perm, sim


def kvq_paged_append(cache, k_new, v_new, t_seq=None, stream=None):
    """fp16 [B][H_kv][T][d] new tokens; sequence b takes its first t_seq[b]
    (all T when None).  Returns KVQ_OK or KVQ_FLUSH_DUE."""
    import numpy as np
    T = int(k_new.shape[2])
    ts = None
    if t_seq is not None:
        arr = np.ascontiguousarray(t_seq, np.int32)
        ts = arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    st = lib().kvq_paged_append(ctypes.byref(cache.c), _ptr(k_new), _ptr(v_new), T, ts,
                                _stream(stream))
    return _check(st, "kvq_paged_append", ok=(KVQ_OK, KVQ_FLUSH_DUE))


def kvq_paged_flush_residual(cache, stream=None):
    return _check(lib().kvq_paged_flush_residual(ctypes.byref(cache.c), _stream(stream)),
                  "kvq_paged_flush_residual")


def kvq_paged_workspace_bytes(cache, max_splits=KVQ_MAX_SPLITS):
    return int(lib().kvq_paged_workspace_bytes(ctypes.byref(cache.c), int(max_splits)))


def kvq_paged_decode_attention(cache, q, out, ws, stream=None):
    st = lib().kvq_paged_decode_attention(ctypes.byref(cache.c), _ptr(q), _ptr(out), _ptr(ws),
                                          ws.numel() * ws.element_size(), _stream(stream))
    return _check(st, "kvq_paged_decode_attention")


def make_plan(window, bits, perm):
    """kvq_window_plan over numpy int8 bits / int32 perm (kept alive by the plan)."""
    import numpy as np
    bits = np.ascontiguousarray(bits, np.int8)
    perm = np.ascontiguousarray(perm, np.int32)
    p = kvq_window_plan(int(window), int(bits.size),
                        bits.ctypes.data_as(ctypes.POINTER(ctypes.c_int8)),
                        perm.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)))
    p._keep = (bits, perm)
    return p


# ---------------------------------------------------------------------------
# device buffers of a cache (torch allocations, library layout of kvq.h)
# ---------------------------------------------------------------------------
class Cache:
    """A kvq_cache struct plus the torch tensors that back it."""

    def __init__(self, c, tensors):
        self.c = c
        self.t = tensors

    def seg(self, s):
        return self.c.seg[s]


def alloc_cache(batch, h_kv, h_q, d_h, group, resid_cap, segments, policy=KVQ_POLICY_KIVI,
                sm_scale=None, device="cuda", zero_point=0, group_v=0):
    """segments: list of (bits, capacity); each capacity is rounded up to a
    multiple of ``group`` (the layout kvq.h requires).  Buffers are zero-filled."""
    import torch
    c = kvq_cache()
    c.batch, c.h_kv, c.h_q, c.d_h, c.group = batch, h_kv, h_q, d_h, group
    c.resid_cap, c.policy = resid_cap, policy
    c.zero_point = zero_point
    c.group_v = group_v
    gv = group_v or group
    c.sm_scale = float(sm_scale if sm_scale is not None else 1.0 / math.sqrt(d_h))
    c.n_seg = len(segments)
    tensors = {}
    P = batch * h_kv
    for i, (bits, cap) in enumerate(segments):
        cap = -(-int(cap) // group) * group
        rb = d_h * bits // 8
        t = dict(
            k_codes=torch.zeros(P * cap * rb, dtype=torch.uint8, device=device),
            k_scale=torch.zeros(P * (cap // group) * d_h, dtype=torch.float16, device=device),
            k_zero=torch.zeros(P * (cap // group) * d_h, dtype=torch.float16, device=device),
            v_codes=torch.zeros(P * cap * rb, dtype=torch.uint8, device=device),
            v_scale=torch.zeros(P * cap * (d_h // gv), dtype=torch.float16, device=device),
            v_zero=torch.zeros(P * cap * (d_h // gv), dtype=torch.float16, device=device))
        tensors["seg%d" % i] = t
        s = c.seg[i]
        s.bits, s.capacity, s.nk, s.nv = bits, cap, 0, 0
        for k, v in t.items():
            setattr(s, k, v.data_ptr())
    tensors["k_resid"] = torch.zeros(P * resid_cap * d_h, dtype=torch.float16, device=device)
    tensors["v_resid"] = torch.zeros(P * resid_cap * d_h, dtype=torch.float16, device=device)
    c.k_resid = tensors["k_resid"].data_ptr()
    c.v_resid = tensors["v_resid"].data_ptr()
    c.nkr = c.nvr = c.k_ring_start = c.v_ring_start = 0
    return Cache(c, tensors)


class PagedCache(Cache):
    """A kvq_paged_cache struct plus the torch tensors that back it."""

    def lengths(self, b):
        s = self.c.seq[b]
        return dict(nk=s.nk, nv=s.nv, nkr=s.nkr, nvr=s.nvr, krs=s.k_ring_start,
                    vrs=s.v_ring_start)


def alloc_paged_cache(batch, h_kv, h_q, d_h, group, resid_cap, bits, page_tokens, n_pages,
                      max_pages, block_table=None, sm_scale=None, device="cuda", zero_point=0,
                      group_v=0):
    """Page pool, per-sequence rings, block table and error word of a paged
    cache (layout of kvq.h).  block_table: int [batch][max_pages] pool page
    ids (any order; -1 where unmapped); None maps sequence b's page j to pool
    page b * max_pages + j.  Buffers are zero-filled."""
    import numpy as np
    import torch
    c = kvq_paged_cache()
    c.batch, c.h_kv, c.h_q, c.d_h, c.group, c.group_v = batch, h_kv, h_q, d_h, group, group_v
    c.resid_cap, c.bits, c.zero_point = resid_cap, bits, zero_point
    c.page_tokens, c.n_pages, c.max_pages = page_tokens, n_pages, max_pages
    c.sm_scale = float(sm_scale if sm_scale is not None else 1.0 / math.sqrt(d_h))
    gv = group_v or group
    rows = n_pages * h_kv * page_tokens
    rb = d_h * bits // 8
    if block_table is None:
        if n_pages < batch * max_pages:
            raise ValueError("n_pages < batch * max_pages: pass a block_table")
        block_table = np.arange(batch * max_pages, dtype=np.int32).reshape(batch, max_pages)
    bt = np.ascontiguousarray(block_table, np.int32).reshape(batch, max_pages)
    t = dict(
        k_codes=torch.zeros(rows * rb, dtype=torch.uint8, device=device),
        k_scale=torch.zeros(rows // group * d_h, dtype=torch.float16, device=device),
        k_zero=torch.zeros(rows // group * d_h, dtype=torch.float16, device=device),
        v_codes=torch.zeros(rows * rb, dtype=torch.uint8, device=device),
        v_scale=torch.zeros(rows * (d_h // gv), dtype=torch.float16, device=device),
        v_zero=torch.zeros(rows * (d_h // gv), dtype=torch.float16, device=device),
        block_table=torch.from_numpy(bt.copy()).to(device),
        k_resid=torch.zeros(batch * h_kv * resid_cap * d_h, dtype=torch.float16, device=device),
        v_resid=torch.zeros(batch * h_kv * resid_cap * d_h, dtype=torch.float16, device=device),
        err=torch.zeros(4, dtype=torch.int32, device=device))
    for k, v in t.items():
        setattr(c, k, v.data_ptr())
    cache = PagedCache(c, t)
    cache.table = bt
    return cache


def header_symbols():
    """Names of the functions include/kvq.h declares."""
    import re
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    with open(os.path.join(root, "include", "kvq.h")) as f:
        src = f.read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_]+\s*\*?\s*(kvq_[a-z0-9_]+)\s*\(", src, re.M)))
