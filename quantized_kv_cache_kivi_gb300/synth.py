"""Seeded synthetic inputs shaped like the pages' workloads.

This module only draws random numbers; it holds none of the quantization or
attention arithmetic, so the CUDA path and the CPU oracle can both be fed from
it.  Every tensor slice is drawn from its own counter-based stream
(numpy's Philox keyed by (seed, tag, batch, head, step)), so any
(batch, head) slice can be regenerated alone, in any order.

Distributions (KIVI page, "键缓存量化维度的原理分析": keys carry large
outliers in a few fixed channels, values do not):
  * K: N(0, 1) per element, with a fixed set of outlier channels per kv head
    multiplied by a factor (the same channels for every token);
  * V and q: N(0, 1).
All values are rounded to fp16 (the pages' cache precision).
"""
import numpy as np

TAG_K, TAG_V, TAG_Q, TAG_OUTLIER, TAG_TEXT, TAG_DIR, TAG_STEP, TAG_LEN, TAG_OFFSET = 1, 2, 3, 4, 5, 6, 7, 8, 9


def rng(seed, tag, b=0, h=0, step=0):
    """Independent Philox stream for (seed, tag, batch, head, step)."""
    code = (int(tag) << 56) | (int(step) << 32) | (int(b) << 16) | int(h)
    return np.random.Generator(np.random.Philox(key=np.array([seed, code], dtype=np.uint64)))


def normal_fp16(g, shape):
    return g.standard_normal(shape, dtype=np.float32).astype(np.float16)


def outlier_channels(seed, h, d, n_out):
    """Fixed outlier channel set of kv head h (a seeded permutation's head)."""
    if n_out <= 0:
        return np.zeros(0, np.int64)
    return np.sort(rng(seed, TAG_OUTLIER, 0, h).permutation(d)[:n_out])


def keys(seed, b, h, n, d, n_out, factor, step=0):
    """K rows [n][d] fp16 of (batch b, kv head h) with outlier channels."""
    x = rng(seed, TAG_K, b, h, step).standard_normal((n, d), dtype=np.float32)
    ch = outlier_channels(seed, h, d, n_out)
    x[:, ch] *= np.float32(factor)
    return x.astype(np.float16)


def values(seed, b, h, n, d, step=0):
    return normal_fp16(rng(seed, TAG_V, b, h, step), (n, d))


def queries(seed, b, h_q, d, step=0):
    """q [h_q][d] fp16 of batch b."""
    return normal_fp16(rng(seed, TAG_Q, b, 0, step), (h_q, d))


def kv_block(seed, batch, h_kv, n, d, n_out, factor, step=0):
    """K, V [batch][h_kv][n][d] fp16."""
    K = np.empty((batch, h_kv, n, d), np.float16)
    V = np.empty((batch, h_kv, n, d), np.float16)
    for b in range(batch):
        for h in range(h_kv):
            K[b, h] = keys(seed, b, h, n, d, n_out, factor, step)
            V[b, h] = values(seed, b, h, n, d, step)
    return K, V


def offset_block(seed, batch, h_kv, n, d, Gv, step=0):
    """K, V [batch][h_kv][n][d] fp16 far from zero with narrow spreads (the
    large-magnitude, narrow-range groups of an outlier channel): K channel c
    of a head is o_c + w_c N(0,1), V channel group j of token t is
    o_tj + w_tj N(0,1), with |o| uniform in [20, 800] (random sign) and w
    uniform in [0.01, 1]."""
    K = np.empty((batch, h_kv, n, d), np.float16)
    V = np.empty((batch, h_kv, n, d), np.float16)
    for b in range(batch):
        for h in range(h_kv):
            g = rng(seed, TAG_OFFSET, b, h, step)
            ok = g.uniform(20.0, 800.0, d) * g.choice([-1.0, 1.0], d)
            wk = g.uniform(0.01, 1.0, d)
            K[b, h] = (ok + wk * g.standard_normal((n, d))).astype(np.float16)
            ov = np.repeat(g.uniform(20.0, 800.0, (n, d // Gv)) * g.choice([-1.0, 1.0], (n, d // Gv)), Gv, axis=1)
            wv = np.repeat(g.uniform(0.01, 1.0, (n, d // Gv)), Gv, axis=1)
            V[b, h] = (ov + wv * g.standard_normal((n, d))).astype(np.float16)
    return K, V


def q_block(seed, batch, h_q, d, step=0):
    return np.stack([queries(seed, b, h_q, d, step) for b in range(batch)])


def window_keys(seed, batch, h_kv, n_win, S, n_text, d, amp=2.0):
    """Vision keys [batch][h_kv][n_win*S][d] and text keys [batch][h_kv][n_text][d].

    N(0,1) noise plus a mean direction per window: window w's mean is
    amp*(cos(theta_w) t + sin(theta_w) u_w), where t is the text mean
    direction, u_w a random unit vector orthogonal to t and theta_w a seeded
    permutation of evenly spaced angles in [0, pi] -- so window similarities
    to the text are distinct and spread over [-1, 1] (non-degenerate ranks)."""
    g = rng(seed, TAG_DIR)
    hd = h_kv * d
    t = g.standard_normal(hd)
    t /= np.linalg.norm(t)
    theta = g.permutation(np.linspace(0.0, np.pi, n_win))
    dirs = np.empty((n_win, hd))
    for w in range(n_win):
        u = g.standard_normal(hd)
        u -= u.dot(t) * t
        u /= np.linalg.norm(u)
        dirs[w] = np.cos(theta[w]) * t + np.sin(theta[w]) * u
    vis = np.empty((batch, h_kv, n_win * S, d), np.float16)
    txt = np.empty((batch, h_kv, n_text, d), np.float16)
    for b in range(batch):
        noise = rng(seed, TAG_TEXT, b).standard_normal((n_text, hd)).astype(np.float32)
        txt[b] = (noise + amp * t).reshape(n_text, h_kv, d).transpose(1, 0, 2).astype(np.float16)
        for w in range(n_win):
            noise = rng(seed, TAG_K, b, w).standard_normal((S, hd)).astype(np.float32)
            vis[b, :, w * S:(w + 1) * S] = (noise + amp * dirs[w]).reshape(S, h_kv, d) \
                .transpose(1, 0, 2).astype(np.float16)
    return vis, txt


# ---------------------------------------------------------------------------
# The workloads (sizes from the pages' model shapes: Llama-2-7B, Llama-3-8B,
# LLaVA-OneVision-Qwen2-7B; KIVI defaults G=32, R=128).
# ---------------------------------------------------------------------------
WORKLOADS = {
    "tiny": dict(batch=1, h_q=1, h_kv=1, d=128, bits=2, G=32, R=32,
                 n_packed=256, n_resid=16, n_out=4, factor=20.0, seed=0),
    "llama2_7b": dict(batch=8, h_q=32, h_kv=32, d=128, bits=2, G=32, R=128,
                      n_packed=3968, n_resid=128, n_out=3, factor=15.0, seed=1),
    "llama3_8b_gqa": dict(batch=16, h_q=32, h_kv=8, d=128, bits=4, G=64, R=128,
                          n_packed=32640, n_resid=128, n_out=3, factor=15.0, seed=2),
    "windowquant_llava_ov": dict(batch=1, h_q=28, h_kv=4, d=128, G=32, R=128,
                                 n_win=64, S=256, n_text=64, frac8=0.1, frac4=0.3, seed=3),
    "streaming": dict(batch=64, h_q=32, h_kv=32, d=128, bits=2, G=32, R=128,
                      prompt=8192, steps=256, n_out=3, factor=15.0, seed=4),
    # per-sequence lengths in one paged cache: Llama-2-7B heads, prompt
    # lengths drawn uniformly from [min_len, max_len] (ragged_lengths)
    "ragged_paged": dict(batch=16, h_q=32, h_kv=32, d=128, bits=2, G=32, R=128, page=256,
                         min_len=512, max_len=8192, n_out=3, factor=15.0, seed=5),
}


def ragged_lengths(w):
    """Seeded per-sequence prompt lengths of a ragged workload."""
    g = rng(w["seed"], TAG_LEN)
    return g.integers(w["min_len"], w["max_len"] + 1, size=w["batch"]).astype(np.int32)
