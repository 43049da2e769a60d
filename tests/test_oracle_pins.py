"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these compare the oracle with a retyped copy of itself: each checks a
closed form, an invariant, a brute-force or exact-rational result, or a
hand-derived trace of the pages' Algorithm 1 (fixtures in tests/golden/).
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _fp16(vals):
    return np.asarray(vals, np.float16)


# ---------------------------------------------------------------------------
# fp16 conversions: the oracle's binary16 rounding vs numpy's own implementation
# ---------------------------------------------------------------------------
def test_fp16_roundtrip_all_patterns(orc):
    pats = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = pats.view(np.float16).astype(np.float32)
    finite = np.isfinite(ref)
    got = np.array([orc.h2f(int(p)) for p in pats[finite][::37]], np.float32)
    assert np.array_equal(got, ref[finite][::37])


def test_fp16_rounding_matches_numpy(orc):
    g = np.random.default_rng(0)
    x = np.concatenate([g.standard_normal(4000).astype(np.float32) * 10,
                        g.standard_normal(1000).astype(np.float32) * 1e-5,
                        # exact ties between two fp16 neighbours: round half to even
                        (np.arange(1024, 1100, dtype=np.float32) + 0.5) * 2.0 ** -10 + 1.0])
    got = np.array([orc.f2h(float(v)) for v in x], np.uint16)
    assert np.array_equal(got, x.astype(np.float16).view(np.uint16))


# ---------------------------------------------------------------------------
# quantizer (KIVI "方法细节" formula; WindowQuant §3.3.3 Eq.14, Eq.16)
# ---------------------------------------------------------------------------
def _exact(h):
    return Fraction(float(np.uint16(h).view(np.float16)))


@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("n", [2, 3, 4, 32])
def test_quantizer_exact_rationals(orc, bits, n):
    """Against exact rational arithmetic: z is the minimum, s is the fp16
    rounding of (max-min)/qmax (to 1 ulp, fp32 then fp16), every code is a
    nearest integer of (x-z)/s, and |x - x'| <= s/2 (+ fp32 rounding slack)."""
    qmax = (1 << bits) - 1
    g = np.random.default_rng(bits * 100 + n)
    for trial in range(60):
        scale = 10.0 ** g.uniform(-3, 2)
        x = _fp16(g.standard_normal(n) * scale)
        codes, s, z = orc.quantize_group(x, bits)
        xs = [_exact(v) for v in x.view(np.uint16)]
        mn, mx = min(xs), max(xs)
        assert _exact(z) == mn
        S = _exact(s)
        true_s = (mx - mn) / qmax
        if true_s == 0:
            assert S == 0 and not codes.any()
            continue
        # one fp16 ulp at true_s (subnormals below 2^-14 have a fixed ulp 2^-24)
        ulp = max(Fraction(2) ** (int(np.floor(np.log2(float(true_s)))) - 10), Fraction(2) ** -24)
        assert abs(S - true_s) <= ulp
        assert codes.max() <= qmax
        # rounding s to fp16 can push (max-min)/s past qmax (by qmax*2^-11
        # for normal s, more for subnormal s); the clamp then takes over
        excess = max(mx - mn - qmax * S, Fraction(0))
        for xi, c in zip(xs, codes):
            t = min((xi - mn) / S, Fraction(qmax))
            assert abs(int(c) - t) <= Fraction(1, 2) + Fraction(1, 1 << 14) * max(1, t)
            err = abs(xi - (int(c) * S + mn))
            assert err <= S / 2 * (1 + Fraction(1, 1 << 12)) + excess
        if S >= Fraction(2) ** -14:
            assert excess <= qmax * S / 2048


def test_quantizer_constant_group_exact(orc):
    for bits in (2, 4, 8):
        x = _fp16([1.375] * 32)
        codes, s, z = orc.quantize_group(x, bits)
        assert not codes.any() and s == 0
        rec = orc.dequant(codes, s, z)
        assert np.array_equal(rec, x.astype(np.float64))


def test_quantizer_extremes_hit_end_codes(orc):
    g = np.random.default_rng(5)
    for bits in (2, 4, 8):
        for _ in range(50):
            x = _fp16(g.standard_normal(32))
            codes, s, z = orc.quantize_group(x, bits)
            assert codes[np.argmin(x)] == 0
            assert codes[np.argmax(x)] == (1 << bits) - 1


def test_quantizer_8bit_grid_reconstructs_exactly(orc):
    """Values on the grid z + k*s (exact fp16) come back exactly at 8 bits."""
    s = 2.0 ** -3
    k = np.random.default_rng(1).permutation(256)[:64]
    k[0], k[1] = 0, 255
    x = _fp16(-10.0 + k * s)
    codes, sh, zh = orc.quantize_group(x, 8)
    assert orc.h2f(sh) == s and orc.h2f(zh) == -10.0
    assert np.array_equal(codes, k.astype(np.uint8))
    assert np.array_equal(orc.dequant(codes, sh, zh), x.astype(np.float64))


def test_k_per_channel_v_per_token_grouping(orc):
    """K groups run along tokens (one scale per channel), V groups along
    channels (one scale per G channels) -- KIVI "方法细节"."""
    g = np.random.default_rng(2)
    X = _fp16(g.standard_normal((32, 128)))
    X[:, 7] *= np.float16(20)  # an outlier channel only widens its own K group
    codes, s, z = orc.quantize_k_block(X, 2)
    for c in range(128):
        cc, sc, zc = orc.quantize_group(X[:, c], 2)
        assert np.array_equal(codes[:, c], cc) and s[c] == sc and z[c] == zc
    assert orc.h2f(s[7]) > 10 * max(orc.h2f(s[c]) for c in range(128) if c != 7)
    vc, vs, vz = orc.quantize_v_token(X[3], 32, 4)
    for gi in range(4):
        cc, sc, zc = orc.quantize_group(X[3, gi * 32:(gi + 1) * 32], 4)
        assert np.array_equal(vc[gi * 32:(gi + 1) * 32], cc) and vs[gi] == sc and vz[gi] == zc


def test_pack_rows_golden(orc):
    with open(os.path.join(GOLDEN, "pack_rows.txt")) as f:
        lines = [ln for ln in f if ln.strip() and not ln.startswith("#")]
    assert lines
    for ln in lines:
        b, codes, row = [p.strip() for p in ln.split("|")]
        b = int(b)
        codes = np.array([int(v) for v in codes.split()], np.uint8)
        row = np.array([int(v, 16) for v in row.split()], np.uint8)
        assert np.array_equal(orc.pack_row(codes, b), row)
        assert np.array_equal(orc.unpack_row(row, codes.size, b), codes)


# ---------------------------------------------------------------------------
# Algorithm 1 state machine (KIVI page, "附录细节")
# ---------------------------------------------------------------------------
def _trace_fixture(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for ln in f:
            if ln.strip() and not ln.startswith("#"):
                ev, *nums = ln.split()
                rows.append((ev, tuple(int(v) for v in nums)))
    return rows


@pytest.mark.parametrize("fixture,l", [("algorithm1_trace_R4_G2.txt", 10),
                                       ("algorithm1_short_prefill_R4_G2.txt", 3)])
def test_algorithm1_length_trace(orc, fixture, l):
    rows = _trace_fixture(fixture)
    g = np.random.default_rng(3)
    D = 16
    head = orc.KiviHead(D, 2, 4, 2)
    head.prefill(_fp16(g.standard_normal((l, D))), _fp16(g.standard_normal((l, D))))
    got = [(head.nk, len(head.kr), head.nv, len(head.vr))]
    for _ in rows[1:]:
        head.decode_update(_fp16(g.standard_normal(D)), _fp16(g.standard_normal(D)))
        got.append((head.nk, len(head.kr), head.nv, len(head.vr)))
    assert got == [r[1] for r in rows]


def test_algorithm1_expected_windows(orc):
    """KIVI page: the fp16 sliding window averages R/2 tokens for K and is R
    for V.  Over one full flush cycle the K residual seen at attention time
    takes each length 0..R-1 once, mean (R-1)/2."""
    R, G, D = 8, 2, 8
    g = np.random.default_rng(4)
    head = orc.KiviHead(D, G, R, 2)
    head.prefill(_fp16(g.standard_normal((3 * R, D))), _fp16(g.standard_normal((3 * R, D))))
    kl, vl = [], []
    for _ in range(4 * R):
        head.decode_update(_fp16(g.standard_normal(D)), _fp16(g.standard_normal(D)))
        kl.append(len(head.kr))
        vl.append(len(head.vr))
    assert sorted(set(kl)) == list(range(R)) and np.mean(kl) == (R - 1) / 2
    assert set(vl) == {R}


def test_algorithm1_contents_and_ring_slots(orc):
    """Serialized buffers hold exactly the tokens Algorithm 1 keeps: packed K
    groups reconstruct their tokens within s/2, the ring slots hold the
    residual tokens verbatim, and the dense sequence is in token order."""
    D, G, R, bits = 32, 4, 8, 4
    g = np.random.default_rng(6)
    l, steps = 21, 17
    XK = _fp16(g.standard_normal((l + steps, D)))
    XV = _fp16(g.standard_normal((l + steps, D)))
    head = orc.KiviHead(D, G, R, bits)
    head.prefill(XK[:l], XV[:l])
    for t in range(l, l + steps):
        head.decode_update(XK[t], XV[t])
    segs, kr, vr = orc.head_buffers(head, [64])
    K, V = orc.dequant_head(segs, kr, vr, len(head.kr), len(head.vr), head.krs, head.vrs, D, G, R)
    n = l + steps
    assert K.shape == (n, D) and V.shape == (n, D)
    # residual tokens come back bit-exact, at the end of the sequence
    assert np.array_equal(K[head.nk:], XK[head.nk:n].astype(np.float64))
    assert np.array_equal(V[head.nv:], XV[head.nv:n].astype(np.float64))
    # packed tokens within half a step of their own group's scale
    for gi, (_, s, _) in enumerate(head.kg):
        sc = s.view(np.float16).astype(np.float64)
        err = np.abs(K[gi * G:(gi + 1) * G] - XK[gi * G:(gi + 1) * G].astype(np.float64))
        assert np.all(err <= sc / 2 * (1 + 1e-3) + 1e-12)
    for u, (_, s, _) in enumerate(head.vg):
        sc = np.repeat(s.view(np.float16).astype(np.float64), G)
        assert np.all(np.abs(V[u] - XV[u].astype(np.float64)) <= sc / 2 * (1 + 1e-3) + 1e-12)
    # a partial K flush (one group) moves the K ring start off slot 0; the
    # remaining residual tokens must still come back verbatim, in order
    assert len(head.kr) >= G
    head.flush_k(G)
    assert head.krs == G
    segs, kr, vr = orc.head_buffers(head, [64])
    K, V = orc.dequant_head(segs, kr, vr, len(head.kr), len(head.vr), head.krs, head.vrs, D, G, R)
    assert np.array_equal(K[head.nk:], XK[head.nk:n].astype(np.float64))


# ---------------------------------------------------------------------------
# attention (KIVI "背景知识与设计原则"; WindowQuant §3.3.2 Eq.12-13)
# ---------------------------------------------------------------------------
def test_attention_single_token_returns_its_value(orc):
    g = np.random.default_rng(7)
    K, V, q = g.standard_normal((1, 64)), g.standard_normal((1, 64)), g.standard_normal(64)
    assert np.array_equal(orc.attention_dense(K, V, q, 0.3), V[0])


def test_attention_zero_query_is_mean(orc):
    g = np.random.default_rng(8)
    K, V = g.standard_normal((37, 64)), g.standard_normal((37, 64))
    out, p = orc.attention_dense(K, V, np.zeros(64), 1.0, return_p=True)
    assert np.allclose(p, 1 / 37, rtol=0, atol=1e-15)
    assert np.allclose(out, V.mean(axis=0), rtol=0, atol=1e-13)


def test_attention_two_tokens_closed_form(orc):
    g = np.random.default_rng(9)
    K, V, q = g.standard_normal((2, 16)), g.standard_normal((2, 16)), g.standard_normal(16)
    a = 0.7 * (K @ q)
    p0 = 1.0 / (1.0 + np.exp(a[1] - a[0]))
    out = orc.attention_dense(K, V, q, 0.7)
    assert np.allclose(out, p0 * V[0] + (1 - p0) * V[1], rtol=0, atol=1e-13)


def test_attention_probabilities_and_one_hot_values(orc):
    """With V = identity the output is the probability vector itself: checks
    the softmax normalisation and the token/channel indexing together."""
    g = np.random.default_rng(10)
    L = 48
    K, q = g.standard_normal((L, L)) * 2, g.standard_normal(L)
    out, p = orc.attention_dense(K, np.eye(L), q, 0.25, return_p=True)
    assert abs(p.sum() - 1.0) < 1e-12
    assert np.allclose(out, p, rtol=0, atol=1e-15)
    a = 0.25 * (K @ q)
    assert np.argmax(p) == np.argmax(a) and np.argmin(p) == np.argmin(a)


def test_attention_permutation_and_shift_invariance(orc):
    """Decode attention has no mask, so reordering tokens (K and V rows
    together) leaves the output unchanged (WindowQuant §3.3.2, Eq.12-13);
    adding to every key a vector u with q.u = c shifts every score by the
    same amount, which softmax ignores."""
    g = np.random.default_rng(11)
    L, D = 300, 128
    K, V, q = g.standard_normal((L, D)), g.standard_normal((L, D)), g.standard_normal(D)
    base = orc.attention_dense(K, V, q, 1 / np.sqrt(D))
    perm = g.permutation(L)
    assert np.allclose(orc.attention_dense(K[perm], V[perm], q, 1 / np.sqrt(D)), base,
                       rtol=0, atol=1e-13)
    u = g.standard_normal(D)
    assert np.allclose(orc.attention_dense(K + u, V, q, 1 / np.sqrt(D)), base, rtol=0, atol=1e-12)


def test_attention_8bit_close_to_unquantized(orc):
    """End to end through Algorithm 1, serialization and dequantization: an
    8-bit cache gives the unquantized fp64 attention (numpy's softmax of
    q K^T) within 1e-2 relative to the output's magnitude."""
    D, G, R = 128, 32, 32
    g = np.random.default_rng(12)
    L = 200
    XK = _fp16(g.standard_normal((L, D)))
    XK[:, [3, 50]] *= np.float16(15)
    XV = _fp16(g.standard_normal((L, D)))
    q = _fp16(g.standard_normal(D))
    head = orc.KiviHead(D, G, R, 8)
    head.prefill(XK, XV)
    segs, kr, vr = orc.head_buffers(head, [256])
    K, V = orc.dequant_head(segs, kr, vr, len(head.kr), len(head.vr), head.krs, head.vrs, D, G, R)
    out = orc.attention_dense(K, V, q.astype(np.float64), 1 / np.sqrt(D))
    a = (XK.astype(np.float64) @ q.astype(np.float64)) / np.sqrt(D)
    p = np.exp(a - a.max())
    p /= p.sum()
    ref = p @ XV.astype(np.float64)
    assert np.max(np.abs(out - ref)) / np.max(np.abs(ref)) < 1e-2
    # 2-bit is much coarser but still tracks the output (sanity, not a bound)
    head2 = orc.KiviHead(D, G, R, 2)
    head2.prefill(XK, XV)
    segs, kr, vr = orc.head_buffers(head2, [256])
    K2, V2 = orc.dequant_head(segs, kr, vr, len(head2.kr), len(head2.vr), head2.krs, head2.vrs,
                              D, G, R)
    out2 = orc.attention_dense(K2, V2, q.astype(np.float64), 1 / np.sqrt(D))
    assert np.max(np.abs(out2 - ref)) / np.max(np.abs(ref)) > np.max(np.abs(out - ref)) / np.max(np.abs(ref))


def test_attention_gqa_head_mapping(orc):
    """Query head j reads kv head j // (h_q / h_kv): with kv head h holding
    the constant value h, every query head returns its kv head's index."""
    D = 32
    g = np.random.default_rng(13)
    outs = []
    for h in range(3):
        K = g.standard_normal((20, D))
        V = np.full((20, D), float(h))
        outs.append(orc.attention_head(K, V, g.standard_normal((4, D)), 0.2))
    got = np.concatenate(outs)
    assert np.allclose(got, np.repeat(np.arange(3.0), 4)[:, None], rtol=0, atol=1e-13)


# ---------------------------------------------------------------------------
# WindowQuant window assignment (§3.2.1 Eq.8, §3.2.2, §3.3.1)
# ---------------------------------------------------------------------------
def test_window_similarity_hand_built(orc):
    """Window 1 repeats the text keys (cos 1), window 2 negates them (cos -1),
    window 3 is orthogonal (cos 0)."""
    B, H, D, S, N = 1, 2, 8, 4, 4
    g = np.random.default_rng(14)
    text = _fp16(np.abs(g.standard_normal((B, H, N, D))))
    text[..., D // 2:] = 0
    keys = _fp16(g.standard_normal((B, H, 4 * S, D)))
    keys[:, :, S:2 * S] = text
    keys[:, :, 2 * S:3 * S] = -text
    ortho = np.zeros((B, H, S, D), np.float16)
    ortho[..., D // 2:] = 1
    keys[:, :, 3 * S:] = ortho
    sim = orc.window_sims(keys, text, S)
    assert abs(sim[1] - 1) < 1e-12 and abs(sim[2] + 1) < 1e-12 and abs(sim[3]) < 1e-15
    bits, perm = orc.window_assign(sim, 0.25, 0.25)
    assert bits[1] == 8 and bits[2] == 2


def test_window_similarity_vs_numpy(orc):
    from quantized_kv_cache_kivi_gb300 import synth
    vis, txt = synth.window_keys(3, 2, 4, 16, 32, 20, 64)
    sim = orc.window_sims(vis, txt, 32)
    ref = np.zeros(16)
    for b in range(2):
        t = txt[b].astype(np.float64).transpose(1, 0, 2).reshape(20, -1).sum(0)
        for w in range(16):
            v = vis[b, :, w * 32:(w + 1) * 32].astype(np.float64).transpose(1, 0, 2) \
                .reshape(32, -1).sum(0)
            ref[w] += v @ t / np.linalg.norm(v) / np.linalg.norm(t) / 2
    assert np.allclose(sim, ref, rtol=0, atol=1e-12)
    assert len(set(np.round(sim, 6))) == 16  # the recipe gives distinct ranks


def test_window_rank_counts_and_perm(orc):
    """64 windows at 10% / 30%: 6 INT8, 19 INT4, 39 INT2 (the workload's
    rule); widths contiguous in the permutation, widest first (§3.3.1)."""
    sim = np.random.default_rng(15).standard_normal(64)
    bits, perm = orc.window_assign(sim, 0.1, 0.3)
    assert [(bits == b).sum() for b in (8, 4, 2)] == [6, 19, 39]
    order = np.argsort(-sim, kind="stable")
    assert set(order[:6]) == set(np.nonzero(bits == 8)[0])
    assert sorted(perm) == list(range(64))
    pb = bits[perm]
    assert list(pb) == sorted(pb, reverse=True)
    for b in (8, 4, 2):
        idx = perm[pb == b]
        assert list(idx) == sorted(idx)
    bits16, perm16 = orc.window_assign(sim, 0.1, 0.3, first_window_fp16=True)
    assert bits16[0] == 16 and perm16[0] == 0
    assert [(bits16 == b).sum() for b in (8, 4, 2)] == [6, 18, 39]


def test_window_ingest_reorder_invariance(orc):
    """Quantizing windows in reordered segments changes nothing in the decode
    output compared with attention over the same dequantized windows in
    their original order (WindowQuant §3.3.2)."""
    D, G, R, S = 64, 16, 64, 32
    g = np.random.default_rng(16)
    nw = 6
    XK = _fp16(g.standard_normal((nw * S + 5, D)))
    XV = _fp16(g.standard_normal((nw * S + 5, D)))
    bits = np.array([4, 2, 8, 2, 16, 4], np.int8)
    perm = np.array(sorted(range(nw), key=lambda w: (-bits[w], w)), np.int32)
    head = orc.Segmented(D, G, R, [8, 4, 2])
    head.ingest_windows(XK, XV, S, bits, perm)
    segs, kr, vr = orc.head_buffers(head, [64, 64, 64])
    K, V = orc.dequant_head(segs, kr, vr, len(head.kr), len(head.vr), 0, 0, D, G, R)
    q = g.standard_normal(D)
    out = orc.attention_dense(K, V, q, 0.125)
    # the same per-window reconstruction, laid out in the original order
    Ko, Vo = [], []
    for w in range(nw):
        blk = slice(w * S, (w + 1) * S)
        if bits[w] == 16:
            Ko.append(XK[blk].astype(np.float64))
            Vo.append(XV[blk].astype(np.float64))
            continue
        for g0 in range(w * S, (w + 1) * S, G):
            c, s, z = orc.quantize_k_block(XK[g0:g0 + G], int(bits[w]))
            Ko.append(orc.dequant(c, s, z))
        for t in range(w * S, (w + 1) * S):
            c, s, z = orc.quantize_v_token(XV[t], G, int(bits[w]))
            Vo.append(orc.dequant(c, np.repeat(s, G), np.repeat(z, G))[None])
    Ko.append(XK[nw * S:].astype(np.float64))
    Vo.append(XV[nw * S:].astype(np.float64))
    ref = orc.attention_dense(np.concatenate(Ko), np.concatenate(Vo), q, 0.125)
    assert np.allclose(out, ref, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# WindowQuant paper-exact assignment (§3.2.1 Eq.8, §3.2.2, §3.2.3 Eq.10-11)
# ---------------------------------------------------------------------------
def test_eq10_11_threshold_closed_forms(orc):
    """f1, f2 at the endpoints are 0 and 1; f1 <= f2 on [0, 1]; the two are
    mirror images, f1(s) = 1 - f2(1 - s); and f1(1/2) = 1 / (e^(a/2) + 1)."""
    for alpha in (0.5, 2.0, 5.0):
        assert orc.eq10_11_thresholds(0.0, alpha) == (0.0, 0.0)
        lo, hi = orc.eq10_11_thresholds(1.0, alpha)
        assert abs(lo - 1.0) < 1e-15 and abs(hi - 1.0) < 1e-15
        for s in np.linspace(0.0, 1.0, 41):
            lo, hi = orc.eq10_11_thresholds(s, alpha)
            assert lo <= hi + 1e-15
            assert abs(lo - (1.0 - orc.eq10_11_thresholds(1.0 - s, alpha)[1])) < 1e-14
        lo, hi = orc.eq10_11_thresholds(0.5, alpha)
        assert abs(lo - 1.0 / (math.exp(alpha / 2) + 1.0)) < 1e-15
        assert abs(hi - (1.0 - lo)) < 1e-15


def test_eq8_hand_built_windows(orc):
    """Text tokens along one direction u (positive multiples): a window of
    multiples of u scores 1, of -u scores -1, of vectors orthogonal to u
    scores 0; positive rescaling of any token changes nothing."""
    D, S, N = 16, 4, 3
    u = np.zeros(D); u[3] = 1.0
    v = np.zeros(D); v[7] = 1.0
    text = np.stack([u * c for c in (0.5, 1.0, 2.0)])[None].astype(np.float16)
    wins = [np.stack([u * c for c in (1, 2, 3, 4)]), np.stack([-u * c for c in (1, 2, 3, 4)]),
            np.stack([v * c for c in (1, 0.5, 2, 3)])]
    vision = np.concatenate(wins)[None].astype(np.float16)
    sims = orc.eq8_sims(vision, text, S)
    assert np.allclose(sims[0], [1.0, -1.0, 0.0], atol=1e-12)
    rng = np.random.default_rng(4)
    vis2 = rng.standard_normal((2, 6 * S, D)).astype(np.float16)
    txt2 = rng.standard_normal((2, N, D)).astype(np.float16)
    s1 = orc.eq8_sims(vis2, txt2, S)
    scale_v = np.float16(2.0) ** rng.integers(-2, 3, size=(2, 6 * S, 1))
    scale_t = np.float16(2.0) ** rng.integers(-2, 3, size=(2, N, 1))
    s2 = orc.eq8_sims((vis2 * scale_v).astype(np.float16), (txt2 * scale_t).astype(np.float16), S)
    assert np.allclose(s1, s2, atol=1e-12)


def test_eq8_double_loop(orc):
    """Eq.8 as the literal double sum of cosines, in plain Python loops."""
    rng = np.random.default_rng(5)
    B, S, nw, N, D = 2, 3, 4, 5, 6
    vis = rng.standard_normal((B, S * nw, D)).astype(np.float16)
    txt = rng.standard_normal((B, N, D)).astype(np.float16)
    got = orc.eq8_sims(vis, txt, S)
    for b in range(B):
        for i in range(nw):
            acc = 0.0
            for j in range(N):
                t = [float(x) for x in txt[b, j]]
                tn = math.sqrt(sum(x * x for x in t))
                for k in range(S):
                    w = [float(x) for x in vis[b, i * S + k]]
                    wn = math.sqrt(sum(x * x for x in w))
                    acc += sum(x * y for x, y in zip(t, w)) / (tn * wn)
            assert abs(got[b, i] - acc / (S * N)) < 1e-12


def test_eq8_vote_and_first_window(orc):
    """Thresholds at s = 1/2, alpha = 2: T_low = 1/(e + 1), T_high = e/(e + 1).
    Per window the batch votes; a three-way tie goes to FP16, a tie between
    INT4 and INT2 to INT4; a score equal to T_high is not above it (INT4)."""
    lo, hi = orc.eq10_11_thresholds(0.5, 2.0)
    sims = np.array([[0.9, 0.1, 0.5, hi, 0.1],
                     [0.1, 0.2, 0.6, hi, 0.5],
                     [0.5, 0.9, 0.1, 0.1, 0.6]])
    cfg = orc.eq8_configs(sims, lo, hi)
    assert cfg.tolist() == [[16, 2, 4, 4, 2], [2, 2, 4, 4, 4], [4, 16, 2, 2, 4]]
    bits, perm = orc.window_assign_eq8(sims, 0.5, 2.0)
    assert bits.tolist() == [16, 2, 4, 4, 4]
    assert perm.tolist() == [0, 2, 3, 4, 1]
    two = np.array([[0.5, 0.2], [0.1, 0.2]])  # window 0: INT4 / INT2 tie
    bits, perm = orc.window_assign_eq8(two, 0.5, 2.0)
    assert bits.tolist() == [4, 2] and perm.tolist() == [0, 1]
    bits, perm = orc.window_assign_eq8(two, 0.5, 2.0, first_window_fp16=True)
    assert bits.tolist() == [16, 2] and perm.tolist() == [0, 1]


# ---------------------------------------------------------------------------
# integer-zero-point quantizer (WindowQuant §3.3.3 Eq.14-16)
# ---------------------------------------------------------------------------
def _h(v):
    return float(np.float16(v))


def test_intz_hand_worked_group(orc):
    """x = (0.5, 1, 1.75, 2), 2 bits: s = 0.5, z = -round(0.5 / 0.5) = -1,
    Q = round(x / s) + z = (0, 1, round(3.5) - 1 = 3, 4 - 1 -> clamp 3); the
    zero slot holds the integer -1 and Eq.15 gives s (Q - z) = (0.5, 1, 2, 2).
    The KIVI quantizer rounds (x - min) / s instead and puts 1.75 at code 2
    (2.5 rounds to even)."""
    x = np.array([0.5, 1.0, 1.75, 2.0], np.float16)
    codes, s, z = orc.quantize_group(x, 2, intz=True)
    assert codes.tolist() == [0, 1, 3, 3]
    assert orc.h2f(s) == 0.5 and orc.zero_int(z) == -1
    assert orc.dequant(codes, s, z, intz=True).tolist() == [0.5, 1.0, 2.0, 2.0]
    kcodes, _, kz = orc.quantize_group(x, 2)
    assert kcodes.tolist() == [0, 1, 2, 3] and orc.h2f(kz) == 0.5


def _intz_groups(rng, bits):
    """Groups near zero and far from it (|offset| 20..800, spread 0.01..1:
    the outlier-channel case of a narrow range at a large magnitude)."""
    for _ in range(150):
        yield (rng.standard_normal(32) * rng.choice([0.01, 1.0, 30.0]) + rng.normal() * 5).astype(np.float16)
    for _ in range(150):
        off = rng.uniform(20.0, 800.0) * rng.choice([-1.0, 1.0])
        yield (off + rng.uniform(0.01, 1.0) * rng.standard_normal(32)).astype(np.float16)


def test_intz_grid_and_error_bounds(orc):
    """Through the stored values: the zero slot holds z = -round(min / s)
    exactly (an integer, not a rounded product), Eq.15 s (Q - z) lies on the
    grid s Z, an unclamped code is within s/2 of its input and the top code
    within 3s/2 (the rounded scale can leave the range one step short), each
    plus the rounding of the fp32 quotient x / s.  A zero stored as the fp16
    of -s z (a float offset) fails this on the far-from-zero groups, where
    that rounding is many steps s."""
    rng = np.random.default_rng(17)
    for bits in (2, 4, 8):
        qmax = (1 << bits) - 1
        for x in _intz_groups(rng, bits):
            codes, sh, zh = orc.quantize_group(x, bits, intz=True)
            s = Fraction(orc.h2f(sh))
            assert s > 0
            zi = int(orc.zero_int(zh))
            # z = -round(min / s) up to the fp32 rounding of the quotient
            ratio = Fraction(float(x.min())) / s
            assert abs(-zi - ratio) <= Fraction(1, 2) + abs(ratio) * Fraction(1, 1 << 22)
            for xi, q in zip(x, codes):
                assert 0 <= q <= qmax
                xq = Fraction(float(xi))
                deq = s * (int(q) - zi)
                assert Fraction(orc.dequant(np.array([q]), [sh], [zh], intz=True)[0]) == deq
                bound = (s / 2 if q < qmax else 3 * s / 2) + abs(xq) * Fraction(1, 1 << 22)
                assert abs(xq - deq) <= bound


def test_intz_exact_grid_and_constant(orc):
    """8 bits, inputs on the grid k s with s a power of two: exact, z = 40 in
    the slot.  A constant group takes s = |x| and z = -sign(x): codes 0 and
    an exact reconstruction; a zero group keeps s = 0, z = 0."""
    s = 0.25
    x = (np.arange(-40, 216, 1.0) * s).astype(np.float16)  # 256 points, range 255 s
    codes, sh, zh = orc.quantize_group(x, 8, intz=True)
    assert orc.h2f(sh) == s and orc.zero_int(zh) == 40  # -round(-10 / 0.25)
    assert np.array_equal(orc.dequant(codes, sh, zh, intz=True), x.astype(np.float64))
    for v, bits in ((-3.5, 4), (1000.0, 2), (0.0078125, 8)):
        c, sh, zh = orc.quantize_group(np.full(8, v, np.float16), bits, intz=True)
        assert c.tolist() == [0] * 8 and orc.h2f(sh) == abs(v)
        assert orc.zero_int(zh) == (1 if v < 0 else -1)
        assert orc.dequant(c, sh, zh, intz=True).tolist() == [v] * 8
    c, sh, zh = orc.quantize_group(np.zeros(8, np.float16), 2, intz=True)
    assert c.tolist() == [0] * 8 and orc.h2f(sh) == 0.0 and orc.zero_int(zh) == 0


def _fp16_next(v):
    with np.errstate(over="ignore"):
        return float(np.nextafter(np.float16(v), np.float16(np.inf)))


def test_intz_zero_fits_sixteen_bits(orc):
    """The narrowest groups (min and the next fp16 above it) over the fp16
    binades.  fp16 inputs give |min| / range < 2^11, and an fp16 s is at
    least 2/3 of (max - min) / qmax (a subnormal s can round down by up to a
    third), so at 2 bits Eq.16's s is always kept, with |z| <= 1.5 * 3 * 2^11;
    at 4 bits it is kept whenever s is a normal fp16 (|z| <= 15 * 2^11).
    Where Eq.16 would need more than 16 bits (8 bits; 4 bits with a
    subnormal s), s is the smallest fp16 for which round(min / s) fits (the
    next smaller one does not).  The reconstruction stays within s/2 (3s/2 at
    the top code, whose step the rounded scale can leave short), and at 8
    bits below an fp16 ulp of the input.  Where Eq.16's s rounds to 0 the
    constant-group reading s = |min| holds."""
    raised = {2: 0, 4: 0, 8: 0}
    for e in range(-10, 16):
        for m in (1.0, 1.5, 1.9990234375):
            for sign in (1.0, -1.0):
                lo = np.float16(sign * m * 2.0 ** e)
                hi = np.float16(_fp16_next(lo))
                if not np.isfinite(hi):
                    continue
                x = np.array([lo, hi] * 4, np.float16)
                for bits in (2, 4, 8):
                    qmax = (1 << bits) - 1
                    codes, sh, zh = orc.quantize_group(x, bits, intz=True)
                    s = orc.h2f(sh)
                    zi = int(orc.zero_int(zh))
                    assert abs(zi) <= 32767
                    eq16 = orc.h2f(orc.f2h(np.float32(float(hi) - float(lo)) / np.float32(qmax)))
                    if eq16 == 0.0:  # the range rounds to s = 0: the constant-group reading
                        assert s == abs(float(lo))
                    elif bits == 2:
                        assert s == eq16 and abs(zi) <= 3 * 3072 + 1
                    elif bits == 4 and eq16 >= 2.0 ** -14:
                        assert s == eq16 and abs(zi) <= 15 * 2048 + 16
                    else:
                        assert s >= eq16
                        if s > eq16:  # raised: the fp16 just below does not fit
                            raised[bits] += 1
                            prev = float(np.nextafter(np.float16(s), np.float16(0)))
                            assert abs(np.rint(np.float32(lo) / np.float32(prev))) > 32767
                    deq = orc.dequant(codes, sh, zh, intz=True)
                    with np.errstate(over="ignore"):
                        ulp = float(np.spacing(np.float16(abs(lo))))
                    err = np.abs(deq - x.astype(np.float64))
                    lim = np.where(codes < qmax, s / 2, 3 * s / 2) + abs(float(lo)) * 2.0 ** -22
                    assert np.all(err <= lim)
                    assert bits < 8 or eq16 == 0.0 or err.max() < ulp
    assert raised[8] > 0  # the 8-bit rule is exercised


def test_intz_block_and_token_use_the_group_quantizer(orc):
    rng = np.random.default_rng(3)
    X = rng.standard_normal((32, 16)).astype(np.float16)
    codes, s, z = orc.quantize_k_block(X, 4, intz=True)
    for c in range(16):
        cc, sc, zc = orc.quantize_group(X[:, c], 4, intz=True)
        assert np.array_equal(codes[:, c], cc) and s[c] == sc and z[c] == zc
    v = rng.standard_normal(64).astype(np.float16)
    codes, s, z = orc.quantize_v_token(v, 16, 2, intz=True)
    for g in range(4):
        cc, sc, zc = orc.quantize_group(v[g * 16:(g + 1) * 16], 2, intz=True)
        assert np.array_equal(codes[g * 16:(g + 1) * 16], cc) and s[g] == sc and z[g] == zc


def test_separate_v_group(orc):
    """K groups of G tokens, V groups of Gv channels (G = 8, Gv = 4 here):
    the serialized buffers carry D / Gv V scales per token, and the dequantized
    V of every token is its per-group codes * scale + zero."""
    D, G, Gv, R = 16, 8, 4, 16
    rng = np.random.default_rng(12)
    XK = rng.standard_normal((40, D)).astype(np.float16)
    XV = rng.standard_normal((40, D)).astype(np.float16)
    head = orc.KiviHead(D, G, R, 4, Gv=Gv)
    head.prefill(XK, XV)
    segs, kr, vr = orc.head_buffers(head, [64])
    assert segs[0]["v_scale"].shape == (64, D // Gv)
    K, V = orc.dequant_head(segs, kr, vr, len(head.kr), len(head.vr), head.krs, head.vrs, D, G, R, Gv)
    for t in range(head.nv):
        codes, s, z = orc.quantize_v_token(XV[t], Gv, 4)
        want = [codes[c] * orc.h2f(s[c // Gv]) + orc.h2f(z[c // Gv]) for c in range(D)]
        assert np.array_equal(V[t], np.array(want))
    for gi in range(head.nk // G):
        codes, s, z = orc.quantize_k_block(XK[gi * G:(gi + 1) * G], 4)
        for j in range(G):
            want = [codes[j, c] * orc.h2f(s[c]) + orc.h2f(z[c]) for c in range(D)]
            assert np.array_equal(K[gi * G + j], np.array(want))
