"""Helpers shared by the GPU parity tests: drive the CUDA library and the CPU
oracle from the same seeded inputs and compare what they hold.

The CUDA side is only ever called through the C ABI (ctypes binding); the
oracle side only through ``oracle``.  Neither sees the other's results."""
import numpy as np

import oracle
from quantized_kv_cache_kivi_gb300 import kvq, synth

TOL = 2e-3  # max |gpu - oracle| / max |oracle| on attention outputs


def max_abs_rel(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.max(np.abs(ref))
    return float(np.max(np.abs(got - ref)) / (den if den > 0 else 1.0))


def to_dev(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


# ---------------------------------------------------------------------------
# KIVI caches on both sides
# ---------------------------------------------------------------------------
class KiviPair:
    """A GPU cache and per-head oracle caches fed with the same tokens."""

    def __init__(self, batch, h_kv, h_q, d, G, R, bits, cap, policy=kvq.KVQ_POLICY_KIVI,
                 heads=None, zero_point=0, group_v=0):
        self.batch, self.h_kv, self.h_q, self.d, self.G, self.R, self.bits = \
            batch, h_kv, h_q, d, G, R, bits
        self.Gv = group_v or G
        self.gpu = kvq.alloc_cache(batch, h_kv, h_q, d, G, R, [(bits, cap)], policy=policy,
                                   zero_point=zero_point, group_v=group_v)
        self.cap = self.gpu.c.seg[0].capacity
        # oracle heads (optionally only a sample of (b, h) pairs)
        self.heads = heads if heads is not None else [(b, h) for b in range(batch)
                                                      for h in range(h_kv)]
        self.orc = {bh: oracle.KiviHead(d, G, R, bits, intz=zero_point == kvq.KVQ_ZERO_INT,
                                        Gv=self.Gv)
                    for bh in self.heads}
        self.started = False

    # -- stepping ---------------------------------------------------------
    def prefill(self, K, V):
        """K, V fp16 [B][H][l][d]: GPU bulk append (+ flush when due) vs
        Algorithm 1's Prefill."""
        st = kvq.kvq_quantize_append(self.gpu, to_dev(K), to_dev(V))
        if st == kvq.KVQ_FLUSH_DUE:
            kvq.kvq_flush_residual(self.gpu)
        for (b, h), head in self.orc.items():
            head.prefill(K[b, h], V[b, h])
        self.started = True

    def append(self, K, V, flush=True):
        """Token by token through Algorithm 1's decoding update (oracle) vs one
        bulk GPU append of T tokens.  flush=False leaves a full K ring."""
        T = K.shape[2]
        st = kvq.kvq_quantize_append(self.gpu, to_dev(K), to_dev(V))
        if st == kvq.KVQ_FLUSH_DUE and flush:
            kvq.kvq_flush_residual(self.gpu)
        for (b, h), head in self.orc.items():
            for t in range(T):
                last = t == T - 1
                head.decode_update(K[b, h, t], V[b, h, t], flush_k=flush or not last)
        return st

    def flush(self):
        kvq.kvq_flush_residual(self.gpu)
        for head in self.orc.values():
            n = (len(head.kr) // self.G) * self.G
            if n:
                head.flush_k(n)

    # -- comparisons ------------------------------------------------------
    def lengths_match(self):
        c = self.gpu.c
        for head in self.orc.values():
            got = (c.seg[0].nk, c.nkr, c.seg[0].nv, c.nvr, c.k_ring_start, c.v_ring_start)
            want = (head.nk, len(head.kr), head.nv, len(head.vr), head.krs, head.vrs)
            assert got == want, (got, want)

    def gpu_buffers(self):
        import torch
        torch.cuda.synchronize()
        P, cap, d, G, rb = self.batch * self.h_kv, self.cap, self.d, self.G, self.d * self.bits // 8
        t = self.gpu.t["seg0"]
        return dict(
            k_codes=t["k_codes"].cpu().numpy().reshape(P, cap, rb),
            k_scale=t["k_scale"].cpu().numpy().view(np.uint16).reshape(P, cap // G, d),
            k_zero=t["k_zero"].cpu().numpy().view(np.uint16).reshape(P, cap // G, d),
            v_codes=t["v_codes"].cpu().numpy().reshape(P, cap, rb),
            v_scale=t["v_scale"].cpu().numpy().view(np.uint16).reshape(P, cap, d // self.Gv),
            v_zero=t["v_zero"].cpu().numpy().view(np.uint16).reshape(P, cap, d // self.Gv),
            k_resid=self.gpu.t["k_resid"].cpu().numpy().view(np.uint16).reshape(P, self.R, d),
            v_resid=self.gpu.t["v_resid"].cpu().numpy().view(np.uint16).reshape(P, self.R, d))

    def assert_buffers_bit_exact(self):
        """Codes, scales, zeros (valid rows) and ring contents (valid slots)."""
        self.lengths_match()
        g = self.gpu_buffers()
        c = self.gpu.c
        nk, nv, G, R = c.seg[0].nk, c.seg[0].nv, self.G, self.R
        for (b, h), head in self.orc.items():
            p = b * self.h_kv + h
            segs, kr, vr = oracle.head_buffers(head, [self.cap])
            s = segs[0]
            assert np.array_equal(g["k_codes"][p, :nk], s["k_codes"][:nk]), ("k_codes", b, h)
            assert np.array_equal(g["k_scale"][p, :nk // G], s["k_scale"][:nk // G]), ("k_scale", b, h)
            assert np.array_equal(g["k_zero"][p, :nk // G], s["k_zero"][:nk // G]), ("k_zero", b, h)
            assert np.array_equal(g["v_codes"][p, :nv], s["v_codes"][:nv]), ("v_codes", b, h)
            assert np.array_equal(g["v_scale"][p, :nv], s["v_scale"][:nv]), ("v_scale", b, h)
            assert np.array_equal(g["v_zero"][p, :nv], s["v_zero"][:nv]), ("v_zero", b, h)
            for i in range(c.nkr):
                slot = (c.k_ring_start + i) % R
                assert np.array_equal(g["k_resid"][p, slot], kr[slot]), ("k_resid", b, h, i)
            for i in range(c.nvr):
                slot = (c.v_ring_start + i) % R
                assert np.array_equal(g["v_resid"][p, slot], vr[slot]), ("v_resid", b, h, i)

    def oracle_attention(self, q):
        """fp64 outputs for the oracle's heads: {(b, h_kv): [gq][d]}."""
        gq = self.h_q // self.h_kv
        out = {}
        for (b, h), head in self.orc.items():
            segs, kr, vr = oracle.head_buffers(head, [self.cap])
            K, V = oracle.dequant_head(segs, kr, vr, len(head.kr), len(head.vr), head.krs,
                                       head.vrs, self.d, self.G, self.R, self.Gv)
            qh = q[b, h * gq:(h + 1) * gq].astype(np.float64)
            out[(b, h)] = oracle.attention_head(K, V, qh, self.gpu.c.sm_scale)
        return out

    def gpu_attention(self, q, ws_splits=kvq.KVQ_MAX_SPLITS, ws=None):
        import torch
        qd = to_dev(q)
        out = torch.empty_like(qd)
        if ws is None:
            ws = self.workspace(ws_splits)
        kvq.kvq_decode_attention(self.gpu, qd, out, ws)
        torch.cuda.synchronize()
        assert kvq.kvq_workspace_error(ws) == 0
        return out.cpu().numpy()

    def workspace(self, ws_splits=kvq.KVQ_MAX_SPLITS):
        import torch
        return torch.zeros(kvq.kvq_workspace_bytes(self.gpu, ws_splits), dtype=torch.uint8,
                           device="cuda")

    def attention_error(self, q, **kw):
        gq = self.h_q // self.h_kv
        got = self.gpu_attention(q, **kw)
        ref = self.oracle_attention(q)
        g = np.concatenate([got[b, h * gq:(h + 1) * gq] for (b, h) in ref])
        r = np.concatenate([ref[k] for k in ref])
        return max_abs_rel(g, r)


def kv(seed, B, H, n, d, n_out=3, factor=15.0, step=0):
    return synth.kv_block(seed, B, H, n, d, n_out, factor, step)
