"""CPU oracle of the quantized-KV decode path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  It shares
no code with the CUDA library (``quantized_kv_cache_kivi_gb300``) and never
imports it.

Layers:
  * ``kvq_oracle.c`` (plain C, built by ``oracle/build.py``): the quantizer in
    its fp32 expression order, row packing, fp64 dequantization and fp64
    attention, fp64 window similarity.
  * this module: ctypes wrappers, KIVI Algorithm 1 as a per-head state machine
    (``KiviHead``), the WindowQuant ingest and rank rule, and serialization of
    an oracle cache into the library's documented buffer layout.

Every function cites the passage it follows.  Pages: "KIVI: A Tuning-Free
Asymmetric 2bit Quantization for KV Cache" (papercache.org) and "WindowQuant:
Mixed-Precision KV Cache Quantization Based on Window-Level Similarity for
VLMs" (ebiotrade.com).
"""
import ctypes
import math

import numpy as np

from . import build as _build

_LIB = None

_u16p = ctypes.POINTER(ctypes.c_uint16)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_f64p = ctypes.POINTER(ctypes.c_double)
_i32p = ctypes.POINTER(ctypes.c_int)


def lib():
    """Load (building first if needed) the oracle's C library."""
    global _LIB
    if _LIB is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.orc_quantize_group.argtypes = [_u16p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         _u8p, ctypes.c_int, _u16p, _u16p]
        L.orc_quantize_group_intz.argtypes = L.orc_quantize_group.argtypes
        L.orc_quantize_k_block.argtypes = [_u16p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           _u8p, _u16p, _u16p, ctypes.c_int]
        L.orc_quantize_v_token.argtypes = [_u16p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           _u8p, _u16p, _u16p, ctypes.c_int]
        L.orc_pack_row.argtypes = [_u8p, ctypes.c_int, ctypes.c_int, _u8p]
        L.orc_unpack_row.argtypes = [_u8p, ctypes.c_int, ctypes.c_int, _u8p]
        L.orc_attention_dense.argtypes = [ctypes.c_int, ctypes.c_int, _f64p, _f64p, _f64p,
                                          ctypes.c_double, _f64p, _f64p]
        pp = ctypes.POINTER(ctypes.c_void_p)
        L.orc_dequant_head.argtypes = [ctypes.c_int] * 5 + [_i32p] * 4 + [pp] * 6 + \
            [_u16p, _u16p] + [ctypes.c_int] * 4 + [_f64p, _f64p]
        L.orc_dequant_head.restype = ctypes.c_int
        L.orc_window_sims.argtypes = [_u16p, _u16p] + [ctypes.c_int] * 6 + [_f64p]
        L.orc_h2f.argtypes = [ctypes.c_uint16]
        L.orc_h2f.restype = ctypes.c_float
        L.orc_f2h.argtypes = [ctypes.c_float]
        L.orc_f2h.restype = ctypes.c_uint16
        _LIB = L
    return _LIB


def _p(a, t):
    return a.ctypes.data_as(t)


def _as_u16(x):
    """fp16 array (or its uint16 bit pattern) -> contiguous uint16 bit pattern."""
    x = np.asarray(x)
    if x.dtype == np.float16:
        x = x.view(np.uint16)
    assert x.dtype == np.uint16
    return np.ascontiguousarray(x)


# ---------------------------------------------------------------------------
# codec (KIVI "方法细节" first formula; WindowQuant §3.3.3 Eq.14, Eq.16)
# ---------------------------------------------------------------------------
def quantize_group(x, bits, intz=False):
    """One group of fp16 values -> (codes uint8 [n], s fp16-bits, z 16 bits).
    KIVI: z = the fp16 minimum.  intz: the integer-zero-point quantizer
    (WindowQuant Eq.14-16); z is then the integer zero point as int16 bits
    (``zero_int`` reads it) and X' = s (Q - z) (Eq.15)."""
    x = _as_u16(x).ravel()
    codes = np.zeros(x.size, np.uint8)
    s = np.zeros(1, np.uint16)
    z = np.zeros(1, np.uint16)
    fn = lib().orc_quantize_group_intz if intz else lib().orc_quantize_group
    fn(_p(x, _u16p), x.size, 1, bits, _p(codes, _u8p), 1, _p(s, _u16p), _p(z, _u16p))
    return codes, s[0], z[0]


def quantize_k_block(x, bits, intz=False):
    """K block [G][D] fp16 -> codes [G][D], s [D], z [D] (per channel)."""
    x = _as_u16(x)
    G, D = x.shape
    codes = np.zeros((G, D), np.uint8)
    s = np.zeros(D, np.uint16)
    z = np.zeros(D, np.uint16)
    lib().orc_quantize_k_block(_p(x, _u16p), G, D, bits, _p(codes, _u8p), _p(s, _u16p),
                               _p(z, _u16p), int(bool(intz)))
    return codes, s, z


def quantize_v_token(x, G, bits, intz=False):
    """V token [D] fp16 -> codes [D], s [D/G], z [D/G] (per token)."""
    x = _as_u16(x).ravel()
    D = x.size
    codes = np.zeros(D, np.uint8)
    s = np.zeros(D // G, np.uint16)
    z = np.zeros(D // G, np.uint16)
    lib().orc_quantize_v_token(_p(x, _u16p), D, G, bits, _p(codes, _u8p), _p(s, _u16p),
                               _p(z, _u16p), int(bool(intz)))
    return codes, s, z


def pack_row(codes, bits):
    """Codes [D] -> packed row bytes [D*bits/8] (channel c at bit c*bits)."""
    codes = np.ascontiguousarray(codes, np.uint8)
    row = np.zeros(codes.size * bits // 8, np.uint8)
    lib().orc_pack_row(_p(codes, _u8p), codes.size, bits, _p(row, _u8p))
    return row


def unpack_row(row, D, bits):
    row = np.ascontiguousarray(row, np.uint8)
    codes = np.zeros(D, np.uint8)
    lib().orc_unpack_row(_p(row, _u8p), D, bits, _p(codes, _u8p))
    return codes


def h2f(h):
    return float(lib().orc_h2f(int(h)))


def f2h(f):
    return int(lib().orc_f2h(float(f)))


def zero_int(z):
    """The integer zero point(s) stored in 16-bit zero slots (int16 bits)."""
    return np.asarray(z, np.uint16).view(np.int16).astype(np.int64)


def dequant(codes, s, z, intz=False):
    """fp64 dequantization: X' = Q * s + z (KIVI "方法细节"), or with an
    integer zero point X' = s (Q - z) (WindowQuant Eq.15)."""
    s64 = np.asarray(s, np.uint16).view(np.float16).astype(np.float64)
    if intz:
        return s64 * (codes.astype(np.int64) - zero_int(z)).astype(np.float64)
    z64 = np.asarray(z, np.uint16).view(np.float16).astype(np.float64)
    return codes.astype(np.float64) * s64 + z64


# ---------------------------------------------------------------------------
# attention (KIVI "背景知识与设计原则": A = Softmax(t_Q X_K^T), t_O = A X_V)
# ---------------------------------------------------------------------------
def attention_dense(K, V, q, sm_scale, return_p=False):
    """fp64 attention of one query q [D] over K, V [L][D]."""
    K = np.ascontiguousarray(K, np.float64)
    V = np.ascontiguousarray(V, np.float64)
    q = np.ascontiguousarray(q, np.float64)
    L, D = K.shape if K.ndim == 2 else (0, q.size)
    out = np.zeros(D, np.float64)
    p = np.zeros(max(L, 1), np.float64)
    lib().orc_attention_dense(L, D, _p(K, _f64p), _p(V, _f64p), _p(q, _f64p),
                              float(sm_scale), _p(out, _f64p), _p(p, _f64p))
    return (out, p[:L]) if return_p else out


# ---------------------------------------------------------------------------
# KIVI Algorithm 1 as a per-head state machine
# ---------------------------------------------------------------------------
class KiviHead:
    """One (batch, kv-head) KV cache following KIVI Algorithm 1 literally.

    State (KIVI page, "附录细节" Algorithm 1): ``kg`` = list of quantized K
    groups (codes [G][D], s [D], z [D]) = Q(X_Kg); ``kr`` = fp16 residual K
    tokens X_Kr; ``vg`` = list of quantized V tokens = Q(X_Vg); ``vr`` = fp16
    residual V queue X_Vr.  ``krs``/``vrs`` track the library's ring start
    slots: they advance by the number of tokens leaving each ring, mod R.
    """

    def __init__(self, D, G, R, bits, intz=False, Gv=None):
        assert R % G == 0
        self.D, self.G, self.R, self.bits = D, G, R, bits
        self.Gv = Gv or G  # V channel group (default: the K token group)
        self.intz = bool(intz)  # integer zero point (WindowQuant Eq.14-16)
        self.kg, self.kr, self.vg, self.vr = [], [], [], []
        self.krs = 0
        self.vrs = 0

    # KeyQuant(X_K): quantize the first l - (l % R) tokens per channel in
    # groups of G (Algorithm 1, KeyQuant).  Called with an explicit token
    # count when the caller flushes.
    def _key_quant(self, X):
        for g0 in range(0, len(X), self.G):
            self.kg.append(quantize_k_block(np.stack(X[g0:g0 + self.G]), self.bits, self.intz))

    def prefill(self, XK, XV):
        """Algorithm 1 Prefill: V first l-R tokens per token, last R fp16;
        K via KeyQuant: l - l%R tokens per channel, l%R fp16 [reading R7:
        for l < R nothing of V is quantized]."""
        l = XK.shape[0]
        nvq = max(l - self.R, 0)
        for t in range(nvq):
            self.vg.append(quantize_v_token(XV[t], self.Gv, self.bits, self.intz))
        self.vr = [XV[t].copy() for t in range(nvq, l)]
        self.vrs = nvq % self.R
        r = l % self.R
        self._key_quant([XK[t] for t in range(l - r)])
        self.kr = [XK[t].copy() for t in range(l - r, l)]

    def flush_k(self, count=None):
        """Quantize the oldest ``count`` residual K tokens (default: all, the
        Algorithm 1 branch 'if len(X_Kr) == R')."""
        if count is None:
            count = len(self.kr)
        assert count % self.G == 0
        self._key_quant(self.kr[:count])
        self.kr = self.kr[count:]
        self.krs = (self.krs + count) % self.R

    def decode_update(self, tK, tV, flush_k=True):
        """Algorithm 1 Decoding: append t_K, t_V; if len(X_Kr) == R quantize
        and empty it (unless flush_k=False, which leaves a full ring for a
        later flush_k()); if len(X_Vr) > R quantize the oldest V token."""
        self.kr.append(tK.copy())
        self.vr.append(tV.copy())
        if flush_k and len(self.kr) == self.R:
            self.flush_k()
        if len(self.vr) > self.R:
            self.vg.append(quantize_v_token(self.vr[0], self.Gv, self.bits, self.intz))
            self.vr = self.vr[1:]
            self.vrs = (self.vrs + 1) % self.R

    # lengths in the library's terms
    @property
    def nk(self):
        return len(self.kg) * self.G

    @property
    def nv(self):
        return len(self.vg)


class Segmented:
    """One (batch, kv-head) cache with several packed segments (WindowQuant
    §3.3.1): ``segs`` maps a segment position to its bit width and lists of
    quantized K groups / V tokens; ``kr``/``vr`` hold the fp16 tokens."""

    def __init__(self, D, G, R, seg_bits, intz=False, Gv=None):
        self.D, self.G, self.R = D, G, R
        self.Gv = Gv or G
        self.intz = bool(intz)
        self.seg_bits = list(seg_bits)
        self.kg = [[] for _ in seg_bits]
        self.vg = [[] for _ in seg_bits]
        self.kr, self.vr = [], []
        self.krs = self.vrs = 0

    def ingest_windows(self, XK, XV, S, bits, perm):
        """WindowQuant §3.1 / §3.3.1: windows of S tokens are taken in the
        order perm; a window of width b in {2,4,8} is appended to the first
        segment of that width (K per channel over groups of G inside the
        window, V per token); width-16 windows and the tail M mod S stay fp16."""
        nw = len(bits)
        for w in perm:
            lo = w * S
            if bits[w] == 16:
                for t in range(lo, lo + S):
                    self.kr.append(XK[t].copy())
                    self.vr.append(XV[t].copy())
                continue
            s = self.seg_bits.index(bits[w])
            for g0 in range(lo, lo + S, self.G):
                self.kg[s].append(quantize_k_block(XK[g0:g0 + self.G], bits[w], self.intz))
            for t in range(lo, lo + S):
                self.vg[s].append(quantize_v_token(XV[t], self.Gv, bits[w], self.intz))
        for t in range(nw * S, XK.shape[0]):
            self.kr.append(XK[t].copy())
            self.vr.append(XV[t].copy())

    def append_fp16(self, XK, XV):
        """WindowQuant §3.1: text and output tokens stay fp16."""
        for t in range(XK.shape[0]):
            self.kr.append(XK[t].copy())
            self.vr.append(XV[t].copy())


def _head_buffers(head, seg_bits, seg_caps, kg_lists, vg_lists):
    """Serialize one head's state into the library's buffer layout (kvq.h):
    codes [cap][D*bits/8], k scale/zero [cap/G][D], v scale/zero [cap][D/Gv],
    ring [R][D] with residual token i at slot (start + i) % R."""
    D, G, R, Gv = head.D, head.G, head.R, head.Gv
    out = []
    for s, (b, cap) in enumerate(zip(seg_bits, seg_caps)):
        rb = D * b // 8
        kc = np.zeros((cap, rb), np.uint8)
        ks = np.zeros((cap // G, D), np.uint16)
        kz = np.zeros((cap // G, D), np.uint16)
        vc = np.zeros((cap, rb), np.uint8)
        vs = np.zeros((cap, D // Gv), np.uint16)
        vz = np.zeros((cap, D // Gv), np.uint16)
        for gi, (codes, sc, zc) in enumerate(kg_lists[s]):
            for j in range(G):
                kc[gi * G + j] = pack_row(codes[j], b)
            ks[gi] = sc
            kz[gi] = zc
        for u, (codes, sc, zc) in enumerate(vg_lists[s]):
            vc[u] = pack_row(codes, b)
            vs[u] = sc
            vz[u] = zc
        out.append(dict(bits=b, nk=len(kg_lists[s]) * G, nv=len(vg_lists[s]), intz=bool(head.intz),
                        k_codes=kc, k_scale=ks, k_zero=kz, v_codes=vc, v_scale=vs, v_zero=vz))
    kr = np.zeros((R, D), np.uint16)
    vr = np.zeros((R, D), np.uint16)
    for i, t in enumerate(head.kr):
        kr[(head.krs + i) % R] = _as_u16(t)
    for i, t in enumerate(head.vr):
        vr[(head.vrs + i) % R] = _as_u16(t)
    return out, kr, vr


def head_buffers(head, caps):
    """Buffers of a KiviHead (one segment) or a Segmented head."""
    if isinstance(head, KiviHead):
        return _head_buffers(head, [head.bits], caps, [head.kg], [head.vg])
    return _head_buffers(head, head.seg_bits, caps, head.kg, head.vg)


def dequant_head(segs, kr, vr, nkr, nvr, krs, vrs, D, G, R, Gv=None):
    """Dense fp64 K, V [L][D] of one head from its serialized buffers, in the
    attention token order: segments, then the ring from its start slot."""
    n = len(segs)
    bits = np.array([s["bits"] for s in segs], np.int32)
    nk = np.array([s["nk"] for s in segs], np.int32)
    nv = np.array([s["nv"] for s in segs], np.int32)
    intz = np.array([int(bool(s.get("intz", False))) for s in segs], np.int32)
    L = int(nk.sum()) + nkr
    K = np.zeros((max(L, 1), D), np.float64)
    V = np.zeros((max(L, 1), D), np.float64)
    keep = []

    def arr(name, t):
        a = (ctypes.c_void_p * n)()
        for i, s in enumerate(segs):
            x = np.ascontiguousarray(s[name])
            keep.append(x)
            a[i] = x.ctypes.data
        return a

    kc, ks, kz = arr("k_codes", _u8p), arr("k_scale", _u16p), arr("k_zero", _u16p)
    vc, vs, vz = arr("v_codes", _u8p), arr("v_scale", _u16p), arr("v_zero", _u16p)
    kr = _as_u16(kr)
    vr = _as_u16(vr)
    got = lib().orc_dequant_head(D, G, Gv or G, R, n, _p(bits, _i32p), _p(intz, _i32p), _p(nk, _i32p),
                                 _p(nv, _i32p),
                                 kc, ks, kz, vc, vs, vz, _p(kr, _u16p), _p(vr, _u16p),
                                 nkr, nvr, krs, vrs, _p(K, _f64p), _p(V, _f64p))
    if got < 0:
        raise ValueError("K and V token counts differ")
    return K[:L], V[:L]


def attention_head(K, V, q_heads, sm_scale):
    """fp64 outputs [gq][D] of the query heads that share one kv head."""
    return np.stack([attention_dense(K, V, q, sm_scale) for q in np.asarray(q_heads, np.float64)])


# ---------------------------------------------------------------------------
# WindowQuant window assignment (§3.2.1 Eq.8 similarity, §3.3.1 reorder)
# ---------------------------------------------------------------------------
def window_sims(keys, text, S):
    """keys [B][H][M][D] fp16, text [B][H][N][D] fp16 -> sim [M//S] (fp64)."""
    keys = _as_u16(keys)
    text = _as_u16(text)
    B, H, M, D = keys.shape
    N = text.shape[2]
    sim = np.zeros(M // S, np.float64)
    lib().orc_window_sims(_p(keys, _u16p), _p(text, _u16p), B, H, M, N, D, S, _p(sim, _f64p))
    return sim


def rank_counts(frac8, frac4, n):
    """floor(frac*n) with frac taken as fp32 then widened (the library's rule)."""
    n8 = int(math.floor(float(np.float32(frac8)) * n))
    n4 = int(math.floor(float(np.float32(frac4)) * n))
    n8 = min(n8, n)
    n4 = min(n4, n - n8)
    return n8, n4


def window_assign(sim, frac8, frac4, first_window_fp16=False):
    """Bit width per window and the ingest permutation.

    Rank rule (this library's reading of the workload's "top 10% INT8, next
    30% INT4, rest INT2"): windows sorted by similarity descending, ties to
    the lower index; first_window_fp16 pins window 0 to 16 bits (WindowQuant
    §3.2.2) and leaves it out of the ranking.  The permutation lists windows
    by width descending, index ascending (§3.3.1: equal widths contiguous)."""
    n = len(sim)
    bits = np.full(n, 2, np.int8)
    ranked = list(range(n))
    if first_window_fp16 and n > 0:
        bits[0] = 16
        ranked = ranked[1:]
    order = sorted(ranked, key=lambda w: (-sim[w], w))
    n8, n4 = rank_counts(frac8, frac4, len(order))
    for r, w in enumerate(order):
        bits[w] = 8 if r < n8 else (4 if r < n8 + n4 else 2)
    perm = np.array(sorted(range(n), key=lambda w: (-int(bits[w]), w)), np.int32)
    return bits, perm


# ---------------------------------------------------------------------------
# WindowQuant paper-exact assignment (§3.2.1 Eq.8 with thresholds, §3.2.2
# first window, §3.2.3 Eq.10-11 thresholds and the batch vote)
# ---------------------------------------------------------------------------
def eq8_sims(vision, text, S):
    """Eq.8 for every window of every batch element.

    vision fp16 [B][M][D] (vision tokens), text fp16 [B][N][D] (text tokens);
    window i holds vision tokens [i*S, i*S + S).  sim(T, W_i) = 1/(S N) *
    sum_j sum_k t_j . w_k / (|t_j| |w_k|), written out as the mean of the
    matrix of pairwise cosines (fp64).  A zero-norm token contributes 0.
    Returns [B][M // S] float64."""
    V = np.asarray(vision, np.float16).astype(np.float64)
    T = np.asarray(text, np.float16).astype(np.float64)
    B, M, D = V.shape
    nw = M // S
    out = np.zeros((B, nw), np.float64)
    for b in range(B):
        tn = np.linalg.norm(T[b], axis=1)
        Tu = np.where(tn[:, None] > 0, T[b] / np.where(tn > 0, tn, 1.0)[:, None], 0.0)
        for i in range(nw):
            W = V[b, i * S:(i + 1) * S]
            wn = np.linalg.norm(W, axis=1)
            Wu = np.where(wn[:, None] > 0, W / np.where(wn > 0, wn, 1.0)[:, None], 0.0)
            cos = Tu @ Wu.T  # [N][S] pairwise cosines
            out[b, i] = cos.sum() / (S * T.shape[1])
    return out


def eq10_11_thresholds(layer_sim, alpha):
    """T_low = f1(s) = (e^(alpha s) - 1) / (e^alpha - 1),
    T_high = f2(s) = (e^(-alpha s) - 1) / (e^(-alpha) - 1)   (fp64)."""
    s, a = float(layer_sim), float(alpha)
    t_low = math.expm1(a * s) / math.expm1(a)
    t_high = math.expm1(-a * s) / math.expm1(-a)
    return t_low, t_high


def eq8_configs(sims, t_low, t_high):
    """Width per (batch element, window): above T_high FP16, below T_low
    INT2, otherwise INT4 (§3.2.1)."""
    sims = np.asarray(sims, np.float64)
    return np.where(sims > t_high, 16, np.where(sims < t_low, 2, 4)).astype(np.int8)


def window_assign_eq8(sims, layer_sim, alpha, first_window_fp16=False):
    """Paper-exact window widths for a batch and the ingest permutation.

    Per window the configuration each request picks (eq8_configs) is voted
    over the batch and the most frequent one wins (§3.2.3); a tie goes to
    the wider of the tied widths (this library's reading: the pages leave
    ties open, and the wider width loses no accuracy).  first_window_fp16
    pins window 0 to FP16 (§3.2.2).  The permutation lists windows by width
    descending, index ascending, as window_assign's."""
    t_low, t_high = eq10_11_thresholds(layer_sim, alpha)
    cfg = eq8_configs(sims, t_low, t_high)
    B, nw = cfg.shape
    bits = np.zeros(nw, np.int8)
    for w in range(nw):
        counts = {b: int((cfg[:, w] == b).sum()) for b in (16, 4, 2)}
        best = max(counts.values())
        bits[w] = max(b for b in (16, 4, 2) if counts[b] == best)
    if first_window_fp16 and nw > 0:
        bits[0] = 16
    perm = np.array(sorted(range(nw), key=lambda w: (-int(bits[w]), w)), np.int32)
    return bits, perm
