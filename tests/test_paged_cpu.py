"""CPU checks of the paged cache's C ABI: struct layout against the header,
host-side validation and capacity statuses (returned before anything is
launched), workspace arithmetic, and -- without a GPU in the process -- that
the decode plan of many per-sequence states passes the pre-launch geometry
check and reaches the launch (which then fails with KVQ_ERR_CUDA)."""
import ctypes
import os
import subprocess

import numpy as np
import pytest

from quantized_kv_cache_kivi_gb300 import kvq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BASE = 1 << 40


@pytest.fixture(scope="module")
def L():
    return kvq.lib()


def test_paged_struct_layout_matches_header(tmp_path):
    src = tmp_path / "layout.c"
    src.write_text(r'''
#include <stdio.h>
#include <stddef.h>
#include "kvq.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu %zu %zu\n", sizeof(kvq_seq_state), sizeof(kvq_paged_cache),
         offsetof(kvq_paged_cache, sm_scale), offsetof(kvq_paged_cache, k_codes),
         offsetof(kvq_paged_cache, block_table), offsetof(kvq_paged_cache, err),
         offsetof(kvq_paged_cache, seq));
  return 0;
}
''')
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True,
                                          check=True).stdout.split()]
    C = kvq.kvq_paged_cache
    want = [ctypes.sizeof(kvq.kvq_seq_state), ctypes.sizeof(C), C.sm_scale.offset,
            C.k_codes.offset, C.block_table.offset, C.err.offset, C.seq.offset]
    assert got == want


def fake_paged(batch=3, h_kv=2, gq=1, d=128, G=32, R=64, bits=2, P=128, n_pages=20, max_pages=6,
               group_v=0):
    c = kvq.kvq_paged_cache()
    c.batch, c.h_kv, c.h_q, c.d_h, c.group, c.group_v = batch, h_kv, h_kv * gq, d, G, group_v
    c.resid_cap, c.bits, c.zero_point = R, bits, 0
    c.page_tokens, c.n_pages, c.max_pages, c.sm_scale = P, n_pages, max_pages, 0.1
    addr = BASE
    for f in ("k_codes", "k_scale", "k_zero", "v_codes", "v_scale", "v_zero", "block_table",
              "k_resid", "v_resid", "err"):
        setattr(c, f, addr)
        addr += 1 << 32
    return c


def set_seq(c, b, nk, nkr, nv, nvr, krs=0, vrs=0):
    s = c.seq[b]
    s.nk, s.nkr, s.nv, s.nvr, s.k_ring_start, s.v_ring_start = nk, nkr, nv, nvr, krs, vrs


def test_paged_validation_statuses(L):
    flush = lambda c: L.kvq_paged_flush_residual(ctypes.byref(c), None)  # noqa: E731
    c = fake_paged()
    assert flush(c) == kvq.KVQ_OK  # no ring full: nothing launched
    bad = [("batch", 0, kvq.KVQ_ERR_INVALID_ARG), ("batch", kvq.KVQ_MAX_SEQS + 1, kvq.KVQ_ERR_INVALID_ARG),
           ("d_h", 96, kvq.KVQ_ERR_UNSUPPORTED), ("group", 48, kvq.KVQ_ERR_UNSUPPORTED),
           ("group_v", 256, kvq.KVQ_ERR_UNSUPPORTED), ("bits", 3, kvq.KVQ_ERR_UNSUPPORTED),
           ("resid_cap", 40, kvq.KVQ_ERR_INVALID_ARG), ("page_tokens", 192, kvq.KVQ_ERR_INVALID_ARG),
           ("page_tokens", 64, kvq.KVQ_ERR_INVALID_ARG), ("n_pages", 0, kvq.KVQ_ERR_INVALID_ARG),
           ("max_pages", 0, kvq.KVQ_ERR_INVALID_ARG), ("zero_point", 2, kvq.KVQ_ERR_INVALID_ARG),
           ("h_q", 3, kvq.KVQ_ERR_INVALID_ARG), ("h_q", 18, kvq.KVQ_ERR_UNSUPPORTED),
           ("block_table", BASE + 4, kvq.KVQ_ERR_INVALID_ARG), ("err", 0, kvq.KVQ_ERR_INVALID_ARG)]
    for field, value, want in bad:
        c = fake_paged()
        setattr(c, field, value)
        assert flush(c) == want, field
        assert L.kvq_last_error_string()
    # inconsistent per-sequence lengths
    for args in ((16, 0, 16, 0), (32, 65, 33, 64), (32, 5, 30, 6), (0, 0, 0, 0, 64, 0),
                 (6 * 128 + 32, 0, 6 * 128 + 32, 0)):
        c = fake_paged()
        set_seq(c, 1, *args)
        assert flush(c) == kvq.KVQ_ERR_INVALID_ARG, args
    assert L.kvq_paged_flush_residual(None, None) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_paged_decode_attention(None, None, None, None, 0, None) == kvq.KVQ_ERR_INVALID_ARG
    c = fake_paged()
    assert L.kvq_paged_decode_attention(ctypes.byref(c), ctypes.c_void_p(0x1000),
                                        ctypes.c_void_p(0x2000), None, 0, None) == kvq.KVQ_ERR_WORKSPACE


def test_paged_append_capacity_and_arguments(L):
    c = fake_paged(max_pages=2, P=128, R=64)  # 256 packed tokens per sequence
    set_seq(c, 0, 192, 64, 192, 64)          # a full K ring and 192 packed tokens
    t = np.array([65, 1, 1], np.int32)
    tp = t.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    kn, vn = ctypes.c_void_p(BASE - (1 << 20)), ctypes.c_void_p(BASE - (2 << 20))
    # 64 + 65 pushed K tokens: two blocks of R would pass 256
    assert L.kvq_paged_append(ctypes.byref(c), kn, vn, 65, tp, None) == kvq.KVQ_ERR_CAPACITY
    st = c.seq[0]
    assert (st.nk, st.nkr, st.nv, st.nvr) == (192, 64, 192, 64)  # untouched
    t[0] = 66  # t_seq above T
    assert L.kvq_paged_append(ctypes.byref(c), kn, vn, 65, tp, None) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_paged_append(ctypes.byref(c), kn, vn, -1, None, None) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_paged_append(ctypes.byref(c), kn, vn, 0, None, None) == kvq.KVQ_OK
    assert L.kvq_paged_append(ctypes.byref(c), ctypes.c_void_p(BASE + 8), vn, 1, None, None) == \
        kvq.KVQ_ERR_INVALID_ARG


def test_paged_workspace_bytes(L):
    c = fake_paged(batch=3, h_kv=2, gq=4)
    pairs, d = 6, 128
    fixed = 256 + 256
    assert L.kvq_paged_workspace_bytes(ctypes.byref(c), 1) == fixed + pairs * 4 * (d + 2) * 4
    assert L.kvq_paged_workspace_bytes(ctypes.byref(c), 10 ** 6) == \
        fixed + pairs * kvq.KVQ_MAX_SPLITS * 4 * (d + 2) * 4
    c.batch = 0
    assert L.kvq_paged_workspace_bytes(ctypes.byref(c), 4) == 0


def _states(cap, R, G, rng, n):
    out = []
    while len(out) < n:
        nk = int(rng.integers(0, cap // G + 1)) * G
        nkr = int(rng.integers(0, R + 1))
        nvr = int(rng.integers(0, R + 1))
        nv = nk + nkr - nvr
        if 0 <= nv <= cap:
            out.append((nk, nkr, nv, nvr, int(rng.integers(0, R)), int(rng.integers(0, R))))
    return out


@pytest.mark.parametrize("d,G,gv,R,bits,P,gq", [
    (128, 32, 0, 64, 2, 128, 1), (128, 32, 0, 128, 4, 256, 4), (128, 16, 8, 32, 8, 128, 8),
    (64, 16, 0, 32, 2, 128, 8), (128, 256, 128, 256, 8, 256, 2), (64, 64, 16, 128, 4, 512, 1)])
def test_paged_decode_plan_passes_geometry_check(L, d, G, gv, R, bits, P, gq):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("meaningful only without a GPU (the launch must fail)")
    rng = np.random.default_rng(d + G + R + bits + P + gq)
    max_pages = 5
    c = fake_paged(batch=6, h_kv=2, gq=gq, d=d, G=G, R=R, bits=bits, P=P, n_pages=40,
                   max_pages=max_pages, group_v=gv)
    ws = L.kvq_paged_workspace_bytes(ctypes.byref(c), 64)
    for trial in range(20):
        for b, s in enumerate(_states(max_pages * P, R, G, rng, 6)):
            set_seq(c, b, *s)
        st = L.kvq_paged_decode_attention(ctypes.byref(c), ctypes.c_void_p(BASE - 4096),
                                          ctypes.c_void_p(BASE - 8192),
                                          ctypes.c_void_p(BASE // 2), ws, None)
        msg = L.kvq_last_error_string().decode()
        assert st == kvq.KVQ_ERR_CUDA, (st, msg, trial)


def test_paged_tile_geometry_enumeration(tmp_path):
    """Every consistent per-sequence state of several shapes through the
    header's paged tile geometry (host build of tests/paged_geometry.cu)."""
    import shutil
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = tmp_path / "paged_geometry"
    subprocess.run([nvcc, "-std=c++17", "-O2", "--expt-relaxed-constexpr", "-x", "cu",
                    os.path.join(ROOT, "tests", "paged_geometry.cu"), "-o", str(exe)],
                   check=True, capture_output=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:]
    assert "bad 0" in r.stdout


def test_paged_stream_k_planning_against_brute_force(tmp_path):
    """The paged planner's run-based tile costs and forward range walk against
    per-tile costs and a binary search (host build of tests/paged_ranges.cu)."""
    import shutil
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = tmp_path / "paged_ranges"
    subprocess.run([nvcc, "-std=c++17", "-O2", "--expt-relaxed-constexpr", "-x", "cu",
                    os.path.join(ROOT, "tests", "paged_ranges.cu"), "-o", str(exe)],
                   check=True, capture_output=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:]
    assert "bad 0" in r.stdout


class _Lengths:
    """KIVI Algorithm 1 lengths of one sequence (decoding updates, the K
    block quantized when the ring holds R tokens), without the data."""

    def __init__(self, R):
        self.R = R
        self.nk = self.nv = self.nkr = self.nvr = self.krs = self.vrs = 0

    def push(self, n):
        for _ in range(int(n)):
            self.nkr += 1
            self.nvr += 1
            if self.nkr == self.R:
                self.nk += self.R
                self.nkr = 0
            if self.nvr > self.R:
                self.nv += 1
                self.nvr -= 1
                self.vrs = (self.vrs + 1) % self.R


def test_paged_lengths_bookkeeping_matches_the_oracle():
    import oracle
    head, ln = oracle.KiviHead(128, 32, 64, 2), _Lengths(64)
    z = np.zeros(128, np.float16)
    for i in range(300):
        head.decode_update(z, z)
        ln.push(1)
        assert (head.nk, head.nv, len(head.kr), len(head.vr), head.krs, head.vrs) == \
            (ln.nk, ln.nv, ln.nkr, ln.nvr, ln.krs, ln.vrs), i


@pytest.mark.parametrize("d,G,gv,R,bits,P,gq", [
    (128, 32, 0, 64, 2, 128, 1), (128, 32, 0, 64, 8, 128, 4), (128, 64, 16, 128, 4, 256, 2),
    (128, 16, 0, 32, 4, 128, 2), (64, 16, 0, 32, 2, 128, 8), (128, 32, 0, 128, 2, 256, 1)])
def test_paged_decode_plan_on_algorithm1_histories(L, d, G, gv, R, bits, P, gq):
    """States that KIVI Algorithm 1 reaches from ragged prompts and decode
    steps with idle sequences pass the pre-launch checks and reach the
    launch (without a GPU the launch then fails with KVQ_ERR_CUDA)."""
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("meaningful only without a GPU (the launch must fail)")
    rng = np.random.default_rng(d + G + R + bits + gq)
    B, max_pages = 6, 8
    seqs = [_Lengths(R) for _ in range(B)]
    prompt = rng.integers(0, max_pages * P - 3 * R, B)
    prompt[0] = 0
    for s, n in zip(seqs, prompt):
        s.push(n)
    c = fake_paged(batch=B, h_kv=2, gq=gq, d=d, G=G, R=R, bits=bits, P=P, n_pages=B * max_pages,
                   max_pages=max_pages, group_v=gv)
    for step in range(2 * R + 5):
        for b, s in enumerate(seqs):
            if not (b == 1 and step % 3 == 0):
                s.push(1)
        if step % 7 and step != 2 * R + 4:
            continue
        for b, s in enumerate(seqs):
            set_seq(c, b, s.nk, s.nkr, s.nv, s.nvr, s.krs, s.vrs)
        for splits in (64, 1):
            ws = L.kvq_paged_workspace_bytes(ctypes.byref(c), splits)
            st = L.kvq_paged_decode_attention(ctypes.byref(c), ctypes.c_void_p(BASE - 4096),
                                              ctypes.c_void_p(BASE - 8192), ctypes.c_void_p(BASE // 2),
                                              ws, None)
            assert st == kvq.KVQ_ERR_CUDA, (st, L.kvq_last_error_string().decode(), step, splits)
