"""Benchmark: one KIVI decode step over the Llama-2-7B-shaped 2-bit cache.

Workload (default): batch 8, 32 heads (MHA), d_h 128, K/V 2-bit, G 32,
R 128, context 4096 with 3968 packed + 128 fp16 tokens for K and for V.
A step is the whole hot path: quantize-append of the new token (V eviction
quantized per token, K into the ring), decode attention over the cache, and
the K block flush that the append left due -- all through the C ABI.  The
cache lengths are reset after each step so every step sees the same state.

value    = effective KV GB/s = algorithmic bytes read by the attention
           (packed codes + fp16 scales/zeros + fp16 ring) / device step time
roofline = the decode-attention kernel alone: the same bytes / its own
           CUDA-event duration, against the measured HBM copy bandwidth
e2e      = the same metric through the plain API calls with the step's
           inputs copied from pinned host memory and the output read back
L2 is flushed between timed steps: the cache (114 MB) would otherwise sit in
the 129 MB L2.  The flush writes a 256 MiB buffer and then reads another
256 MiB buffer, so the timed step starts with no cache data in L2 and no
dirty lines from the flush itself left to write back.

--impl reference times the CPU oracle (plain C + Python) on a bounded sample
of the same workload (one (batch, kv-head) slice per step), scaled to the
full step.
"""
import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "decode-attn µs/step and effective KV GB/s (% of GB300 HBM peak), 2-bit"
UNIT = "GB/s"
WORKLOAD = "llama2_7b"


def algorithmic_bytes(w, nk, nkr, nv, nvr):
    """Bytes the attention must read: codes + fp16 scale/zero + fp16 ring."""
    P = w["batch"] * w["h_kv"]
    d, G, b = w["d"], w["G"], w["bits"]
    per = nk * d * b // 8 + (nk // G) * d * 2 * 2 + nkr * d * 2
    per += nv * d * b // 8 + nv * (d // G) * 2 * 2 + nvr * d * 2
    return P * per


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def kernel_source_hash():
    """Hash of the sources the Llama-2 decode kernel is built from."""
    h = hashlib.sha256()
    for rel in ("quantized_kv_cache_kivi_gb300/csrc/kvq_decode_warp.cu",
                "quantized_kv_cache_kivi_gb300/csrc/kvq_mma.cuh",
                "quantized_kv_cache_kivi_gb300/csrc/kvq_internal.h",
                "quantized_kv_cache_kivi_gb300/csrc/kvq_device.cuh", "include/kvq.h"):
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """dram bytes per decode launch from the committed ncu summary, if it
    was taken on the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "decode_warp_kernel_llama2_7b.md")
    try:
        txt = open(p).read()
    except OSError:
        return None
    vals = {}
    for line in txt.splitlines():
        line = line.strip().lstrip("-* ")
        if ":" in line and line.startswith(("traffic_bytes_per_launch", "source_hash")):
            k, v = line.split(":", 1)
            vals[k.strip().strip("`")] = v.strip().strip("`")
    if vals.get("source_hash") != kernel_source_hash():
        return None
    try:
        return int(float(vals["traffic_bytes_per_launch"]))
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": mx,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def setup_workload(w, device):
    import torch
    from quantized_kv_cache_kivi_gb300 import kvq, synth

    B, Hq, H, d, G, R, bits = w["batch"], w["h_q"], w["h_kv"], w["d"], w["G"], w["R"], w["bits"]
    L = w["n_packed"] + w["n_resid"]
    cache = kvq.alloc_cache(B, H, Hq, d, G, R, [(bits, L + R)], device=device)
    K, V = synth.kv_block(w["seed"], B, H, L - 1, d, w["n_out"], w["factor"])
    kd = torch.from_numpy(K).to(device)
    vd = torch.from_numpy(V).to(device)
    st = kvq.kvq_quantize_append(cache, kd, vd)
    if st == kvq.KVQ_FLUSH_DUE:
        kvq.kvq_flush_residual(cache)
    del kd, vd
    torch.cuda.synchronize()
    return cache


def cache_bytes(cache):
    """Bytes one decode attention must read from a cache's current state:
    packed codes + fp16 scales/zeros of every segment + the fp16 rings."""
    c = cache.c
    P, d, G = c.batch * c.h_kv, c.d_h, c.group
    Gv = c.group_v or G
    per = (c.nkr + c.nvr) * d * 2
    for i in range(c.n_seg):
        s = c.seg[i]
        per += s.nk * d * s.bits // 8 + (s.nk // G) * d * 4
        per += s.nv * d * s.bits // 8 + s.nv * (d // Gv) * 4
    return P * per


def paged_bytes(cache):
    """Bytes one decode attention must read from a paged cache: every
    sequence's packed codes, scales/zeros and fp16 ring tokens."""
    c = cache.c
    d, G = c.d_h, c.group
    Gv = c.group_v or G
    rb = d * c.bits // 8
    tot = 0
    for b in range(c.batch):
        s = c.seq[b]
        tot += s.nk * rb + (s.nk // G) * d * 4 + s.nv * rb + s.nv * (d // Gv) * 4
        tot += (s.nkr + s.nvr) * d * 2
    return tot * c.h_kv


def streaming_steps(cache, w, device, flush_l2, peak, to_prompt):
    """The streaming workload as specified: after the prompt, `steps`
    generated tokens, each step one kvq_decode_step call in KIVI Algorithm
    1's order: quantize-append of the new token, the K flush when the ring
    reaches R, decode attention; new K, V and q drawn per step (seed =
    step).  L2 is flushed before every step; each step is timed with CUDA
    events around the call.  The cache given holds the prompt; `to_prompt()`
    puts its lengths back to the state right after the prompt's ingest."""
    import torch
    from quantized_kv_cache_kivi_gb300 import kvq

    B, Hq, H, d = w["batch"], w["h_q"], w["h_kv"], w["d"]
    to_prompt()
    out = torch.empty(B, Hq, d, dtype=torch.float16, device=device)
    ws = torch.zeros(kvq.kvq_workspace_bytes(cache, kvq.KVQ_MAX_SPLITS), dtype=torch.uint8, device=device)
    n = w["steps"]
    toks = []
    for t in range(n):
        g = torch.Generator(device=device).manual_seed(w["seed"] * 100003 + t)
        k = torch.randn(B, H, 1, d, generator=g, device=device)
        k[..., :3] *= w["factor"]
        toks.append((k.half(), torch.randn(B, H, 1, d, generator=g, device=device).half(),
                     torch.randn(B, Hq, d, generator=g, device=device).half()))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
    nbytes, flushes = [], 0
    torch.cuda.synchronize()
    for t, (k, v, q) in enumerate(toks):
        flush_l2(t)
        nkr = cache.c.nkr
        ev[t][0].record()
        kvq.kvq_decode_step(cache, k, v, q, out, ws, order=kvq.KVQ_STEP_FLUSH_FIRST)
        ev[t][1].record()
        flushes += cache.c.nkr <= nkr  # the ring did not grow: it was flushed
        nbytes.append(cache_bytes(cache))  # the state the attention read
    torch.cuda.synchronize()
    if kvq.kvq_workspace_error(ws):
        raise RuntimeError("decode kernel reported a timed-out wait")
    us = np.array([e0.elapsed_time(e1) for e0, e1 in ev]) * 1e3
    gbs = float(np.sum(nbytes)) / (float(np.sum(us)) * 1e-6) / 1e9
    return {"steps": n, "us_per_step_mean": float(us.mean()), "us_per_step_max": float(us.max()),
            "us_per_step_min": float(us.min()), "flushes": flushes, "bytes_per_step_mean": float(np.mean(nbytes)),
            "GB/s": gbs, "frac": gbs / peak,
            "note": "step = one kvq_decode_step (append, flush when due, attention: Algorithm 1's order), "
                    "L2 flushed before each step"}


def per_workload_attention(device, flush_l2, peak, reps=20, only=None):
    """Decode attention alone on each workload the pages name besides the
    timed step's, at the state the workload describes: mean CUDA-event time
    over `reps` calls with L2 flushed before each.  Inputs are seeded
    synthetic data of the workloads' shapes and distributions (K ~ N(0,1)
    with 2% outlier channels x15, V, q ~ N(0,1)), drawn on the device."""
    import torch
    from quantized_kv_cache_kivi_gb300 import kvq, synth

    def dev_kv(seed, B, H, n, d, n_out, factor):
        g = torch.Generator(device=device).manual_seed(seed)
        K = torch.randn(B, H, n, d, generator=g, device=device)
        ch = torch.randperm(d, generator=torch.Generator().manual_seed(seed))[:n_out].to(device)
        K[:, :, :, ch] *= factor
        V = torch.randn(B, H, n, d, generator=g, device=device)
        return K.half(), V.half()

    def timed(cache, B, Hq, d, seed):
        q = torch.randn(B, Hq, d, generator=torch.Generator(device=device).manual_seed(seed + 7),
                        device=device).half()
        out = torch.empty_like(q)
        ws = torch.zeros(kvq.kvq_workspace_bytes(cache, kvq.KVQ_MAX_SPLITS), dtype=torch.uint8,
                         device=device)
        for _ in range(3):
            kvq.kvq_decode_attention(cache, q, out, ws)
        ts = []
        for i in range(reps):
            flush_l2(i)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            kvq.kvq_decode_attention(cache, q, out, ws)
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        # warm: calls enqueued back to back with events between them, so the
        # cache stays in L2 where it fits and no host launch gap is timed
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
        torch.cuda.synchronize()
        ev[0].record()
        for i in range(reps):
            kvq.kvq_decode_attention(cache, q, out, ws)
            ev[i + 1].record()
        torch.cuda.synchronize()
        warm = [ev[i].elapsed_time(ev[i + 1]) for i in range(reps)]
        if kvq.kvq_workspace_error(ws):
            raise RuntimeError("decode kernel reported a timed-out wait")
        us = float(np.mean(ts)) * 1e3
        nb = cache_bytes(cache)
        gbs = nb / (us * 1e-6) / 1e9
        return {"us": us, "GB/s": gbs, "frac": gbs / peak, "bytes": nb,
                "us_warm": float(np.mean(warm)) * 1e3,
                "state": dict(nk=[cache.c.seg[i].nk for i in range(cache.c.n_seg)],
                              nv=[cache.c.seg[i].nv for i in range(cache.c.n_seg)],
                              nkr=cache.c.nkr, nvr=cache.c.nvr)}

    def lengths(cache):
        c = cache.c
        return ([(c.seg[i].nk, c.seg[i].nv) for i in range(c.n_seg)], c.nkr, c.nvr,
                c.k_ring_start, c.v_ring_start)

    def set_lengths(cache, st):
        c = cache.c
        for i, (nk, nv) in enumerate(st[0]):
            c.seg[i].nk, c.seg[i].nv = nk, nv
        c.nkr, c.nvr, c.k_ring_start, c.v_ring_start = st[1:]

    def timed_ingest(cache, fn, reps=5):
        """Mean event time of fn() from the same starting state, L2 flushed."""
        st0 = lengths(cache)
        ts = []
        for i in range(reps):
            set_lengths(cache, st0)
            flush_l2(i)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return float(np.mean(ts)) * 1e3

    res, ing = {}, {}
    for name in ("tiny", "llama3_8b_gqa", "streaming"):
        if only is not None and name != only and not (name == "streaming" and only == "prefill_streaming"):
            continue
        w = synth.WORKLOADS[name]
        B, Hq, H, d, G, R, bits = w["batch"], w["h_q"], w["h_kv"], w["d"], w["G"], w["R"], w["bits"]
        n = w["prompt"] + w["steps"] if name == "streaming" else w["n_packed"] + w["n_resid"]
        cache = kvq.alloc_cache(B, H, Hq, d, G, R, [(bits, n + R)], device=device)
        if name == "streaming":
            # prompt, then decode steps up to the average K residual (R/2)
            K, V = dev_kv(w["seed"], B, H, w["prompt"], d, w["n_out"], w["factor"])

            def prefill():
                if kvq.kvq_quantize_append(cache, K, V) == kvq.KVQ_FLUSH_DUE:
                    kvq.kvq_flush_residual(cache)

            # KIVI prefill of the prompt (bulk quantize-pack, rows a1-a3):
            # fp16 K and V read, packed codes / scales / zeros and ring written
            us = timed_ingest(cache, prefill, reps=reps if only else 5)
            st_prompt = lengths(cache)
            nb = K.numel() * 2 * 2 + cache_bytes(cache)
            ing["prefill_streaming"] = {"us": us, "GB/s": nb / (us * 1e-6) / 1e9,
                                        "frac": nb / (us * 1e-6) / 1e9 / peak, "bytes": nb,
                                        "tokens": int(B * H * w["prompt"])}
            del K, V
            K, V = dev_kv(w["seed"] + 1, B, H, R // 2, d, w["n_out"], w["factor"])
            for t in range(R // 2):
                if kvq.kvq_quantize_append(cache, K[:, :, t:t + 1].contiguous(),
                                           V[:, :, t:t + 1].contiguous()) == kvq.KVQ_FLUSH_DUE:
                    kvq.kvq_flush_residual(cache)
        else:
            # the stated state: the flush a full K ring would trigger is left due
            K, V = dev_kv(w["seed"], B, H, n, d, w["n_out"], w["factor"])
            kvq.kvq_quantize_append(cache, K, V)
        del K, V
        torch.cuda.synchronize()
        if only != "prefill_streaming":
            res[name] = timed(cache, B, Hq, d, w["seed"])
        if name == "streaming" and only in (None, "streaming"):
            res["streaming_steps"] = streaming_steps(cache, w, device, flush_l2, peak,
                                                     lambda: set_lengths(cache, st_prompt))
        del cache
        torch.cuda.empty_cache()
    if only is None or only == "ragged_paged":
        # per-sequence lengths in one paged cache: pages handed out in a
        # shuffled order, prompts of ragged lengths ingested by one call
        w = synth.WORKLOADS["ragged_paged"]
        B, Hq, H, d, G, R, bits, Pg = (w[k] for k in ("batch", "h_q", "h_kv", "d", "G", "R", "bits", "page"))
        lens = synth.ragged_lengths(w)
        need = [-(-int(n) // Pg) + 1 for n in lens]
        max_pages, n_pages = max(need), sum(need)
        order = np.random.default_rng(w["seed"]).permutation(n_pages).astype(np.int32)
        table = np.full((B, max_pages), -1, np.int32)
        k = 0
        for b in range(B):
            table[b, :need[b]] = order[k:k + need[b]]
            k += need[b]
        cache = kvq.alloc_paged_cache(B, H, Hq, d, G, R, bits, Pg, n_pages, max_pages,
                                      block_table=table, device=device)
        K, V = dev_kv(w["seed"], B, H, int(lens.max()), d, w["n_out"], w["factor"])
        seqs = cache.c.seq

        def prefill():
            if kvq.kvq_paged_append(cache, K, V, lens) == kvq.KVQ_FLUSH_DUE:
                kvq.kvq_paged_flush_residual(cache)

        ts = []
        for i in range((reps if only else 5) + 1):  # the first call warms up
            for b in range(B):
                seqs[b].nk = seqs[b].nv = seqs[b].nkr = seqs[b].nvr = 0
                seqs[b].k_ring_start = seqs[b].v_ring_start = 0
            flush_l2(i)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            prefill()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        us = float(np.mean(ts[1:])) * 1e3
        nb = int(lens.sum()) * H * d * 2 * 2 + paged_bytes(cache)
        ing["prefill_ragged_paged"] = {"us": us, "GB/s": nb / (us * 1e-6) / 1e9,
                                       "frac": nb / (us * 1e-6) / 1e9 / peak, "bytes": nb,
                                       "tokens": int(lens.sum()) * H}
        del K, V
        torch.cuda.empty_cache()
        q = torch.randn(B, Hq, d, generator=torch.Generator(device=device).manual_seed(w["seed"] + 7),
                        device=device).half()
        out = torch.empty_like(q)
        ws = torch.zeros(kvq.kvq_paged_workspace_bytes(cache), dtype=torch.uint8, device=device)
        for _ in range(3):
            kvq.kvq_paged_decode_attention(cache, q, out, ws)
        ts = []
        for i in range(reps):
            flush_l2(i)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            kvq.kvq_paged_decode_attention(cache, q, out, ws)
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        if kvq.kvq_workspace_error(ws) or kvq.kvq_workspace_error(cache.t["err"]):
            raise RuntimeError("paged decode reported an error")
        us = float(np.mean(ts)) * 1e3
        nb = paged_bytes(cache)
        res["ragged_paged"] = {"us": us, "GB/s": nb / (us * 1e-6) / 1e9, "frac": nb / (us * 1e-6) / 1e9 / peak,
                               "bytes": nb, "lengths": "%d sequences, %d..%d tokens, %d in all" % (
                                   B, int(lens.min()), int(lens.max()), int(lens.sum()))}
        del cache
        torch.cuda.empty_cache()
    if only is not None and only != "windowquant_llava_ov":
        return res, ing
    # WindowQuant: windows ranked and reordered into INT8/INT4/INT2 segments,
    # 64 fp16 text tokens in the ring
    w = synth.WORKLOADS["windowquant_llava_ov"]
    B, Hq, H, d, G, S = w["batch"], w["h_q"], w["h_kv"], w["d"], w["G"], w["S"]
    vis, txt = synth.window_keys(w["seed"], B, H, w["n_win"], S, w["n_text"], d)
    vd, td = torch.from_numpy(vis).to(device), torch.from_numpy(txt).to(device)
    bits, perm, _ = kvq.kvq_window_assign(vd, td, S, w["frac8"], w["frac4"])
    # row a7 timing: the assignment returns host arrays (synchronous call)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(5):
        kvq.kvq_window_assign(vd, td, S, w["frac8"], w["frac4"])
    ing["windowquant_assign"] = {"us": (time.perf_counter() - t0) / 5 * 1e6,
                                 "note": "host-synchronous call (host arrays out)"}
    # paper-exact assignment (Eq.8 over embeddings of the LLM width, 3584 for
    # the Qwen2-7B of LLaVA-OneVision): device time of its three kernels
    dim = 3584
    g8 = torch.Generator(device=device).manual_seed(w["seed"] + 5)
    emb_v = torch.randn(B, vis.shape[2], dim, generator=g8, device=device).half()
    emb_t = torch.randn(B, txt.shape[2], dim, generator=g8, device=device).half()
    ws8 = torch.empty(kvq.kvq_window_assign_eq8_workspace_bytes(B, dim, emb_v.shape[1], S, emb_t.shape[1]),
                      dtype=torch.uint8, device=device)
    kvq.kvq_window_assign_eq8(emb_v, emb_t, S, 0.1, 2.0, ws=ws8)
    t0 = time.perf_counter()
    for _ in range(5):
        kvq.kvq_window_assign_eq8(emb_v, emb_t, S, 0.1, 2.0, ws=ws8)
    us8 = (time.perf_counter() - t0) / 5 * 1e6
    nb8 = (emb_v.numel() + emb_t.numel()) * 2 * 2  # two passes over the embeddings
    ing["windowquant_assign_eq8"] = {"us": us8, "bytes": nb8, "GB/s": nb8 / (us8 * 1e-6) / 1e9,
                                     "note": "host-synchronous call; embeddings read twice (norms, sums)"}
    del emb_v, emb_t, ws8
    caps = [(b, max(G, int((bits == b).sum()) * S)) for b in (8, 4, 2)]
    cache = kvq.alloc_cache(B, H, Hq, d, G, 128, caps, policy=kvq.KVQ_POLICY_FP16_TAIL, device=device)
    g = torch.Generator(device=device).manual_seed(w["seed"])
    Vv = torch.randn(B, H, vis.shape[2], d, generator=g, device=device).half()
    Vt = torch.randn(B, H, txt.shape[2], d, generator=g, device=device).half()
    plan = kvq.make_plan(S, bits, perm)
    us = timed_ingest(cache, lambda: kvq.kvq_quantize_append(cache, vd, Vv, plan=plan))  # leaves it ingested
    nb = vd.numel() * 2 * 2 + cache_bytes(cache)
    ing["windowquant_ingest"] = {"us": us, "GB/s": nb / (us * 1e-6) / 1e9, "frac": nb / (us * 1e-6) / 1e9 / peak,
                                 "bytes": nb}
    kvq.kvq_quantize_append(cache, td, Vt)
    torch.cuda.synchronize()
    res["windowquant_llava_ov"] = timed(cache, B, Hq, d, w["seed"])
    return res, ing


def max_over_ranks(x, device):
    """The largest x over the ranks of the default process group (x itself
    when there is none or it has one rank)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replicas_value(bytes_per_step, steps, world, total_ms):
    """Whole-job effective GB/s of `world` independent replicas (the pairs
    need no exchange): the bytes all ranks processed over the slowest rank's
    time."""
    return bytes_per_step * steps * world / (total_ms * 1e-3) / 1e9


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    from quantized_kv_cache_kivi_gb300 import kvq, synth

    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    w = synth.WORKLOADS[WORKLOAD]
    B, Hq, H, d = w["batch"], w["h_q"], w["h_kv"], w["d"]
    cache = setup_workload(w, device)
    c = cache.c
    snap = (c.seg[0].nk, c.seg[0].nv, c.nkr, c.nvr, c.k_ring_start, c.v_ring_start)

    def reset():
        c.seg[0].nk, c.seg[0].nv, c.nkr, c.nvr, c.k_ring_start, c.v_ring_start = snap

    n_in = args.steps + args.warmup
    pool = 64  # distinct new tokens / queries cycled through the steps
    kn, vn = synth.kv_block(w["seed"] + 100, B, H, pool, d, w["n_out"], w["factor"])
    kn = torch.from_numpy(np.ascontiguousarray(kn.transpose(2, 0, 1, 3))).to(device)  # [pool][B][H][d]
    vn = torch.from_numpy(np.ascontiguousarray(vn.transpose(2, 0, 1, 3))).to(device)
    qp = torch.from_numpy(np.stack([synth.q_block(w["seed"], B, Hq, d, step=i)
                                    for i in range(pool)])).to(device)
    # one device buffer holds a step's inputs (new K, new V, queries), so a
    # step's host inputs arrive in one copy
    n_k, n_q = B * H * d, B * Hq * d
    dev_in = torch.empty(2 * n_k + n_q, dtype=torch.float16, device=device)
    k_in = dev_in[:n_k].view(B, H, 1, d)
    v_in = dev_in[n_k:2 * n_k].view(B, H, 1, d)
    q_in = dev_in[2 * n_k:].view(B, Hq, d)
    out = torch.empty_like(q_in)
    ws = torch.zeros(kvq.kvq_workspace_bytes(cache, kvq.KVQ_MAX_SPLITS), dtype=torch.uint8,
                     device=device)
    l2 = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    l2r = torch.ones(256 << 20, dtype=torch.uint8, device=device)

    def flush_l2(i):
        l2.fill_(i & 255)
        l2r.sum()

    def stage_inputs(i):
        j = i % pool
        k_in.copy_(kn[j].unsqueeze(2))
        v_in.copy_(vn[j].unsqueeze(2))
        q_in.copy_(qp[j])

    def step_append():
        st = kvq.kvq_quantize_append(cache, k_in, v_in)
        assert st == kvq.KVQ_FLUSH_DUE

    def step_attn():
        kvq.kvq_decode_attention(cache, q_in, out, ws)

    def step_flush():
        kvq.kvq_flush_residual(cache)

    # attention reads the state right after the append (flush deferred)
    reset()
    stage_inputs(0)
    step_append()
    attn_state = (c.seg[0].nk, c.nkr, c.seg[0].nv, c.nvr)
    step_attn()
    step_flush()
    reset()
    torch.cuda.synchronize()
    attn_bytes = algorithmic_bytes(w, *attn_state)

    # Timed loop: the whole step as one kvq_decode_step call (append,
    # attention, due flush; the library chains the three kernels with
    # programmatic dependent launch), an event before and after it on the
    # launching stream.  The L2 flush before each step keeps the GPU busy for
    # ~0.1 ms while the host enqueues the step.
    stream = torch.cuda.current_stream()

    def run_step(e):
        e[0].record(stream)
        kvq.kvq_decode_step(cache, k_in, v_in, q_in, out, ws)
        e[1].record(stream)
        reset()

    # The same step as three calls with an event between them: each event
    # interval is that call's device time (the attention's is the roofline's).
    def run_parts(e):
        e[0].record(stream)
        step_append()
        e[1].record(stream)
        step_attn()
        e[2].record(stream)
        step_flush()
        e[3].record(stream)
        reset()

    for i in range(args.warmup):
        flush_l2(i)
        stage_inputs(i)
        run_step([torch.cuda.Event(enable_timing=True) for _ in range(2)])
        flush_l2(i)
        run_parts([torch.cuda.Event(enable_timing=True) for _ in range(4)])
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.2)
    t_wall0 = time.perf_counter()
    for i in range(args.steps):
        flush_l2(i)
        stage_inputs(args.warmup + i)
        run_step(ev[i])
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    step_ms = np.array([e[0].elapsed_time(e[1]) for e in ev])
    total_ms = max_over_ranks(float(step_ms.sum()), device)
    n_parts = min(args.steps, 500)
    evp = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n_parts)]
    for i in range(n_parts):
        flush_l2(i)
        stage_inputs(args.warmup + i)
        run_parts(evp[i])
    torch.cuda.synchronize()
    app_ms = np.array([e[0].elapsed_time(e[1]) for e in evp])
    attn_ms = np.array([e[1].elapsed_time(e[2]) for e in evp])
    fl_ms = np.array([e[2].elapsed_time(e[3]) for e in evp])
    parts_ms = np.array([e[0].elapsed_time(e[3]) for e in evp])

    # end to end through the C ABI with host buffers (kvq_decode_step_host):
    # pinned host inputs copied in, the step, the output copied back
    host_in = torch.cat([kn.reshape(pool, -1), vn.reshape(pool, -1), qp.reshape(pool, -1)], dim=1)
    host_in = host_in.cpu().pin_memory()  # [pool][new K | new V | q], the layout of dev_in
    oh = torch.empty(B, Hq, d, dtype=torch.float16).pin_memory()
    e2e_s = []
    n_e2e = min(args.steps, 500)
    rows = [host_in[j] for j in range(pool)]
    for i in range(n_e2e):
        j = i % pool
        flush_l2(i)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        kvq.kvq_decode_step_host(cache, rows[j], oh, dev_in, out, ws, stream=stream)
        stream.synchronize()
        e2e_s.append(time.perf_counter() - t0)
        reset()
    err = kvq.kvq_workspace_error(ws)
    if err:
        raise RuntimeError("decode kernel reported a timed-out wait")
    e2e_step = float(np.mean(e2e_s))
    others, ingest = (per_workload_attention(device, flush_l2, measured_peak()[0]) if args.per_workload
                      else ({}, {}))
    return dict(w=w, attn_bytes=attn_bytes, total_ms=total_ms, step_ms=step_ms, attn_ms=attn_ms,
                app_ms=app_ms, fl_ms=fl_ms, parts_ms=parts_ms, clocks=clocks, t_wall=t_wall, e2e_step=e2e_step,
                attn_state=attn_state, others=others, ingest=ingest,
                h2d=dev_in.numel() * 2,
                d2h=oh.numel() * 2)


# ---------------------------------------------------------------------------
# the oracle on the host cores (cpu_baseline and --impl reference)
# ---------------------------------------------------------------------------
class OracleStep:
    """One (batch, kv-head) slice of the workload's step, run by the oracle:
    Algorithm 1 decoding update (flush deferred), fp64 attention over the
    serialized cache, then the K flush; the state is restored afterwards."""

    def __init__(self, w, b, h):
        import oracle
        from quantized_kv_cache_kivi_gb300 import synth
        self.oracle = oracle
        self.w = w
        d, G, R, bits = w["d"], w["G"], w["R"], w["bits"]
        L = w["n_packed"] + w["n_resid"]
        K = synth.keys(w["seed"], b, h, L, d, w["n_out"], w["factor"])
        V = synth.values(w["seed"], b, h, L, d)
        self.head = oracle.KiviHead(d, G, R, bits)
        self.head.prefill(K[:L - 1], V[:L - 1])
        self.tk, self.tv = K[L - 1], V[L - 1]
        gq = w["h_q"] // w["h_kv"]
        self.q = synth.queries(w["seed"], b, w["h_q"], d)[h * gq:(h + 1) * gq]
        self.cap = L + R

    def run(self):
        import copy
        o = self.oracle
        w = self.w
        saved = copy.copy(self.head.__dict__)
        saved = {k: (list(v) if isinstance(v, list) else v) for k, v in saved.items()}
        hd = self.head
        hd.decode_update(self.tk, self.tv, flush_k=False)
        segs, kr, vr = o.head_buffers(hd, [self.cap])
        K, V = o.dequant_head(segs, kr, vr, len(hd.kr), len(hd.vr), hd.krs, hd.vrs, w["d"], w["G"],
                              w["R"])
        out = o.attention_head(K, V, self.q.astype(np.float64), 1.0 / math.sqrt(w["d"]))
        hd.flush_k()
        self.head.__dict__.update(saved)
        return out


def cpu_model():
    """CPU model name: lscpu's (it names Arm parts from their part codes),
    else /proc/cpuinfo's model line."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part", "hardware")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_rate(n_pairs_sample, seconds, warm=1):
    """Time the oracle's per-slice step in this process (one core); returns
    (s per slice-step, steps, slices)."""
    from quantized_kv_cache_kivi_gb300 import synth
    w = synth.WORKLOADS[WORKLOAD]
    steps = [OracleStep(w, i % w["batch"], (7 * i) % w["h_kv"]) for i in range(n_pairs_sample)]
    for s in steps[:warm]:
        s.run()
    t0 = time.perf_counter()
    n = 0
    while True:
        for s in steps:
            s.run()
            n += 1
        if time.perf_counter() - t0 > seconds:
            break
    return (time.perf_counter() - t0) / n, n, len(steps)


def _oracle_worker(job):
    """Pool task: build the oracle slice `i`, then run its step either `runs`
    times or for `seconds`; returns (runs done, seconds spent running)."""
    i, runs, seconds, warm = job
    sys.path.insert(0, ROOT)
    import oracle
    oracle.lib()
    from quantized_kv_cache_kivi_gb300 import synth
    w = synth.WORKLOADS[WORKLOAD]
    st = OracleStep(w, i % w["batch"], (7 * i) % w["h_kv"])
    for _ in range(warm):
        st.run()
    t0 = time.perf_counter()
    n = 0
    while (runs and n < runs) or (not runs and time.perf_counter() - t0 < seconds):
        st.run()
        n += 1
    return n, time.perf_counter() - t0


def oracle_pool(workers, runs=0, seconds=0.0, warm=1):
    """The oracle on `workers` processes at once (spawned: no state of this
    process, CUDA included, is inherited), one slice each.  Returns (slice
    steps done, wall seconds of the running phase)."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    with ctx.Pool(workers) as pool:
        res = pool.map(_oracle_worker, [(i, runs, seconds, warm) for i in range(workers)])
    return sum(n for n, _ in res), max(t for _, t in res)


def run_reference(args):
    """The oracle as the reference arm: each step runs one (batch, kv-head)
    slice of the workload's step on every host core at once (a process per
    core); ms_per_step is the measured wall time of those steps, value the
    bytes of the slices processed over that time."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    oracle.lib()
    from quantized_kv_cache_kivi_gb300 import synth
    w = synth.WORKLOADS[WORKLOAD]
    P = w["batch"] * w["h_kv"]
    cores = host_cores()
    slice_bytes = algorithmic_bytes(w, w["n_packed"], w["n_resid"], w["n_packed"], w["n_resid"]) // P
    t_all = time.perf_counter()
    n, wall = oracle_pool(cores, runs=args.steps, warm=args.warmup)
    setup_s = time.perf_counter() - t_all - wall
    value = n * slice_bytes / wall / 1e9
    ms_step = wall / args.steps * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "llama2_7b: batch 8, 32 heads, d_h 128, 3968 packed + 128 fp16 "
                   "tokens (K and V), 2-bit, G 32, R 128",
                   "sample": "each step = one (batch, kv-head) slice of %d per host core, %d cores at once "
                             "(%d slices per step); the whole %d-slice step would take ~%.0f ms at this rate "
                             "(extrapolated, not run)" % (P, cores, cores, P, ms_step * P / cores),
                   "setup_s": setup_s},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": "%d slice-steps, %d processes" % (n, cores), "cpu": cpu_model()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--profile-workload", default=None,
                    choices=["tiny", "llama3_8b_gqa", "streaming", "prefill_streaming", "windowquant_llava_ov",
                             "ragged_paged"],
                    help="run one workload's calls a few times (for an ncu capture) and exit")
    ap.add_argument("--per-workload", type=int, default=1,
                    help="also time the attention alone on the other workloads (0: skip)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
        return
    if args.profile_workload:
        import torch
        device = torch.device("cuda", 0)
        torch.cuda.set_device(device)
        l2 = torch.empty(256 << 20, dtype=torch.uint8, device=device)
        per_workload_attention(device, lambda i: l2.fill_(i & 255), measured_peak()[0], reps=3,
                               only=args.profile_workload)
        torch.cuda.synchronize()
        print(json.dumps({"profiled": args.profile_workload}))
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    import torch
    import torch.distributed as dist
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    from quantized_kv_cache_kivi_gb300 import kvq
    kvq.lib()
    r = run_ours(args, rank, world, local_rank)
    w = r["w"]
    value = replicas_value(r["attn_bytes"], args.steps, world, r["total_ms"])
    peak, peak_kind = measured_peak()
    attn_mean_ms = float(np.mean(r["attn_ms"]))
    achieved = r["attn_bytes"] / (attn_mean_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": float(np.mean(r["step_ms"])), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {
            "workload": "llama2_7b: batch 8, 32 heads (MHA), d_h 128, 3968 packed + 128 fp16 "
                        "tokens for K and V, 2-bit, G 32, R 128; step = kvq_decode_step: quantize-append + "
                        "decode attention + K flush",
            "l2": "flushed between steps (256 MiB write, then 256 MiB read)",
            "launch": "one kvq_decode_step call per step (its three kernels chained by programmatic dependent "
                      "launch), enqueued during the L2 flush", "parallelism": "replicas" if world > 1 else "single",
            "us_per_step": float(np.mean(r["step_ms"])) * 1e3,
            "us_attention": attn_mean_ms * 1e3,
            "us_append": float(np.mean(r["app_ms"])) * 1e3,
            "us_flush": float(np.mean(r["fl_ms"])) * 1e3,
            "us_per_step_three_calls": float(np.mean(r["parts_ms"])) * 1e3,
            "parts_note": "us_append / us_attention / us_flush: the same step as three calls with an event "
                          "between them (the roofline uses us_attention)",
            "attn_state": dict(zip(("nk", "nkr", "nv", "nvr"), r["attn_state"])),
            "algorithmic_bytes_per_step": r["attn_bytes"],
            "wall_s_timed": r["t_wall"],
        },
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": profiled_traffic(),
                     "peak_kind": peak_kind, "kernel": "kvq decode_warp_kernel"},
        "e2e": {"value": r["attn_bytes"] / r["e2e_step"] / 1e9, "unit": UNIT,
                "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"],
                "us_per_step": r["e2e_step"] * 1e6},
        "per_workload_attention": r["others"],
        "per_workload_ingest": r["ingest"],
        "gpu_launches": 3 * args.steps,
        "clocks": r["clocks"],
    }
    if rank == 0 and world == 1 and args.cpu_seconds > 0:
        import oracle
        oracle.lib()
        P = w["batch"] * w["h_kv"]
        cores = host_cores()
        per, n1, ns = oracle_rate(2, args.cpu_seconds / 3)
        v1 = r["attn_bytes"] / (per * P) / 1e9
        n, wall = oracle_pool(cores, seconds=args.cpu_seconds * 2 / 3)
        v = n * (r["attn_bytes"] // P) / wall / 1e9
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": "%d slice-steps of the step's (batch, kv-head) slices on %d "
                                          "processes at once (%.1f s), bytes of the slices run / wall time"
                                          % (n, cores, wall),
                                "single_core": {"value": v1, "cores": 1,
                                                "sample": "%d slice-steps over %d of %d slices" % (n1, ns, P)},
                                "cpu": cpu_model()}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
