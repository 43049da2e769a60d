"""Paged cache with per-sequence lengths against per-sequence oracle heads.

Every sequence of the batch runs KIVI Algorithm 1 (KIVI page, "附录细节") on
its own; the oracle keeps one KiviHead per (sequence, kv head) and is fed the
same tokens one by one.  The GPU's packed rows live in pool pages reached
through a shuffled block table; the test gathers them back per head on the
host and compares codes, scales, zeros and ring contents bit for bit, then
the attention outputs within 2e-3 (max abs error over max abs value)."""
import numpy as np
import pytest

import oracle
from kvq_testutil import TOL, max_abs_rel, to_dev
from quantized_kv_cache_kivi_gb300 import kvq, synth

pytestmark = pytest.mark.gpu


class PagedPair:
    def __init__(self, batch, h_kv, h_q, d, G, R, bits, P, max_pages, seed, zero_point=0,
                 group_v=0, spare=5):
        rng = np.random.default_rng(seed)
        self.n_pages = batch * max_pages + spare
        table = rng.permutation(self.n_pages)[:batch * max_pages].astype(np.int32)
        self.table = table.reshape(batch, max_pages)
        self.gpu = kvq.alloc_paged_cache(batch, h_kv, h_q, d, G, R, bits, P, self.n_pages,
                                         max_pages, block_table=self.table,
                                         zero_point=zero_point, group_v=group_v)
        self.batch, self.h_kv, self.h_q, self.d, self.G, self.R, self.bits, self.P = \
            batch, h_kv, h_q, d, G, R, bits, P
        self.Gv = group_v or G
        self.cap = max_pages * P
        intz = zero_point == kvq.KVQ_ZERO_INT
        self.orc = {(b, h): oracle.KiviHead(d, G, R, bits, intz=intz, Gv=self.Gv)
                    for b in range(batch) for h in range(h_kv)}

    def append(self, K, V, t_seq):
        """K, V fp16 [B][H][T][d]; sequence b takes its first t_seq[b] rows.
        A due K flush runs at once (Algorithm 1)."""
        st = kvq.kvq_paged_append(self.gpu, to_dev(K), to_dev(V), t_seq)
        if st == kvq.KVQ_FLUSH_DUE:
            kvq.kvq_paged_flush_residual(self.gpu)
        for (b, h), head in self.orc.items():
            for i in range(int(t_seq[b])):
                head.decode_update(K[b, h, i], V[b, h, i])
        return st

    def lengths_match(self):
        for (b, h), head in self.orc.items():
            got = self.gpu.lengths(b)
            want = dict(nk=head.nk, nv=head.nv, nkr=len(head.kr), nvr=len(head.vr), krs=head.krs,
                        vrs=head.vrs)
            assert got == want, (b, got, want)

    def gathered(self):
        """Per-head buffers gathered from the pool through the block table."""
        import torch
        torch.cuda.synchronize()
        t = self.gpu.t
        H, P, d, G, Gv = self.h_kv, self.P, self.d, self.G, self.Gv
        rb = d * self.bits // 8
        npg = self.n_pages
        pool = dict(
            k_codes=t["k_codes"].cpu().numpy().reshape(npg, H, P, rb),
            k_scale=t["k_scale"].cpu().numpy().view(np.uint16).reshape(npg, H, P // G, d),
            k_zero=t["k_zero"].cpu().numpy().view(np.uint16).reshape(npg, H, P // G, d),
            v_codes=t["v_codes"].cpu().numpy().reshape(npg, H, P, rb),
            v_scale=t["v_scale"].cpu().numpy().view(np.uint16).reshape(npg, H, P, d // Gv),
            v_zero=t["v_zero"].cpu().numpy().view(np.uint16).reshape(npg, H, P, d // Gv))
        kr = t["k_resid"].cpu().numpy().view(np.uint16).reshape(self.batch, H, self.R, d)
        vr = t["v_resid"].cpu().numpy().view(np.uint16).reshape(self.batch, H, self.R, d)
        out = {}
        for (b, h) in self.orc:
            pages = self.table[b]
            g = {k: np.concatenate([v[p, h] for p in pages]) for k, v in pool.items()}
            g["k_resid"], g["v_resid"] = kr[b, h], vr[b, h]
            out[(b, h)] = g
        return out

    def assert_bit_exact(self):
        self.lengths_match()
        got = self.gathered()
        G, R = self.G, self.R
        for (b, h), head in self.orc.items():
            segs, kr, vr = oracle.head_buffers(head, [self.cap])
            s, g = segs[0], got[(b, h)]
            nk, nv = head.nk, head.nv
            for name, n in (("k_codes", nk), ("k_scale", nk // G), ("k_zero", nk // G),
                            ("v_codes", nv), ("v_scale", nv), ("v_zero", nv)):
                assert np.array_equal(g[name][:n], s[name][:n]), (name, b, h)
            for i in range(len(head.kr)):
                slot = (head.krs + i) % R
                assert np.array_equal(g["k_resid"][slot], kr[slot]), ("k_resid", b, h, i)
            for i in range(len(head.vr)):
                slot = (head.vrs + i) % R
                assert np.array_equal(g["v_resid"][slot], vr[slot]), ("v_resid", b, h, i)

    def attention_error(self, q, max_splits=kvq.KVQ_MAX_SPLITS):
        import torch
        gq = self.h_q // self.h_kv
        ws = torch.zeros(kvq.kvq_paged_workspace_bytes(self.gpu, max_splits), dtype=torch.uint8,
                         device="cuda")
        qd = to_dev(q)
        out = torch.full_like(qd, float("nan"))
        kvq.kvq_paged_decode_attention(self.gpu, qd, out, ws)
        torch.cuda.synchronize()
        assert kvq.kvq_workspace_error(ws) == 0
        assert kvq.kvq_workspace_error(self.gpu.t["err"]) == 0
        got = out.cpu().numpy().astype(np.float64)
        errs = []
        for (b, h), head in self.orc.items():
            g = got[b, h * gq:(h + 1) * gq]
            if head.nk + len(head.kr) == 0:
                assert np.all(g == 0), "a sequence with no tokens must give zeros"
                continue
            segs, kr, vr = oracle.head_buffers(head, [self.cap])
            K, V = oracle.dequant_head(segs, kr, vr, len(head.kr), len(head.vr), head.krs,
                                       head.vrs, self.d, self.G, self.R, self.Gv)
            ref = oracle.attention_head(K, V, q[b, h * gq:(h + 1) * gq].astype(np.float64),
                                        self.gpu.c.sm_scale)
            errs.append(max_abs_rel(g, ref))
        return max(errs) if errs else 0.0


def _tokens(seed, B, H, T, d, step=0):
    return synth.kv_block(seed, B, H, T, d, 3, 15.0, step)


def _q(seed, B, Hq, d):
    return synth.q_block(seed, B, Hq, d)


def _run_ragged(pp, seed, prompt, steps, idle_every=3):
    """Ragged prefill (t_seq = prompt), then `steps` decode steps where
    sequence 1 sits out every `idle_every`-th step."""
    B, H, d = pp.batch, pp.h_kv, pp.d
    T = max(prompt)
    K, V = _tokens(seed, B, H, T, d)
    pp.append(K, V, np.asarray(prompt, np.int32))
    pp.assert_bit_exact()
    for i in range(steps):
        k1, v1 = _tokens(seed + 1 + i, B, H, 1, d, step=i + 1)
        t = np.ones(B, np.int32)
        if B > 1 and i % idle_every == 0:
            t[1] = 0
        pp.append(k1, v1, t)


@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("gq", [1, 4])
def test_paged_ragged_prefill_then_decode(bits, gq):
    pp = PagedPair(batch=5, h_kv=2, h_q=2 * gq, d=128, G=32, R=64, bits=bits, P=128, max_pages=7,
                   seed=11 + bits + gq)
    _run_ragged(pp, 100 + bits, prompt=[0, 37, 300, 128, 700], steps=70)
    pp.assert_bit_exact()
    err = pp.attention_error(_q(7, 5, 2 * gq, 128))
    assert err < TOL, err


def test_paged_chunked_second_prompt_and_empty_sequence():
    """A second prompt-sized append on top of partly filled rings (K groups
    that mix old ring rows with new rows, V evictions from the old ring), one
    sequence left empty throughout, and one split per CTA forced."""
    pp = PagedPair(batch=4, h_kv=3, h_q=3, d=128, G=32, R=128, bits=2, P=256, max_pages=4, seed=5)
    K, V = _tokens(21, 4, 3, 150, 128)
    pp.append(K, V, np.array([150, 0, 70, 129], np.int32))
    K, V = _tokens(22, 4, 3, 600, 128)
    pp.append(K, V, np.array([600, 0, 300, 127], np.int32))
    pp.assert_bit_exact()
    q = _q(9, 4, 3, 128)
    assert pp.attention_error(q) < TOL
    assert pp.attention_error(q, max_splits=1) < TOL


def test_paged_integer_zero_point_and_v_group():
    pp = PagedPair(batch=3, h_kv=2, h_q=4, d=128, G=64, R=128, bits=4, P=256, max_pages=4,
                   seed=8, zero_point=kvq.KVQ_ZERO_INT, group_v=16)
    _run_ragged(pp, 31, prompt=[257, 64, 513], steps=40)
    pp.assert_bit_exact()
    assert pp.attention_error(_q(3, 3, 4, 128)) < TOL


def test_paged_general_kernel_at_head_dim_128():
    """K groups of 16 tokens keep d_h 128 on the general kernel's paged form
    (the tensor-core forms need groups of 32 or more)."""
    pp = PagedPair(batch=4, h_kv=2, h_q=4, d=128, G=16, R=32, bits=4, P=128, max_pages=5, seed=6)
    _run_ragged(pp, 81, prompt=[400, 0, 90, 255], steps=33)
    pp.assert_bit_exact()
    assert pp.attention_error(_q(5, 4, 4, 128)) < TOL


def test_paged_head_dim_64_and_eight_query_heads():
    pp = PagedPair(batch=3, h_kv=1, h_q=8, d=64, G=16, R=32, bits=2, P=128, max_pages=5, seed=2)
    _run_ragged(pp, 41, prompt=[500, 17, 33], steps=35)
    pp.assert_bit_exact()
    assert pp.attention_error(_q(4, 3, 8, 64)) < TOL


def test_paged_decode_many_steps_matches_after_each_flush():
    """Attention right after steps that flushed some sequence's K ring."""
    pp = PagedPair(batch=3, h_kv=2, h_q=2, d=128, G=32, R=32, bits=2, P=128, max_pages=4, seed=3)
    K, V = _tokens(51, 3, 2, 90, 128)
    pp.append(K, V, np.array([90, 31, 64], np.int32))
    for i in range(40):
        k1, v1 = _tokens(52 + i, 3, 2, 1, 128, step=i + 1)
        st = pp.append(k1, v1, np.ones(3, np.int32))
        if st == kvq.KVQ_FLUSH_DUE or i % 13 == 0:
            assert pp.attention_error(_q(60 + i, 3, 2, 128)) < TOL
    pp.assert_bit_exact()


def test_paged_bad_block_table_entry_sets_the_error_word():
    """An entry outside the pool is not followed by the kernels (they read
    page 0 instead and write nothing); the cache's error word says so."""
    import torch
    pp = PagedPair(batch=2, h_kv=1, h_q=1, d=128, G=32, R=32, bits=2, P=128, max_pages=3, seed=4)
    K, V = _tokens(71, 2, 1, 200, 128)
    pp.append(K, V, np.array([200, 40], np.int32))
    bad = pp.gpu.t["block_table"].clone()
    pp.gpu.t["block_table"][0, 0] = pp.n_pages + 7
    ws = torch.zeros(kvq.kvq_paged_workspace_bytes(pp.gpu), dtype=torch.uint8, device="cuda")
    q = to_dev(_q(1, 2, 1, 128))
    out = torch.empty_like(q)
    kvq.kvq_paged_decode_attention(pp.gpu, q, out, ws)
    torch.cuda.synchronize()
    assert kvq.kvq_workspace_error(pp.gpu.t["err"]) == 2
    assert kvq.kvq_workspace_error(ws) == 0
    pp.gpu.t["block_table"].copy_(bad)
    pp.gpu.t["err"].zero_()
