"""CPU checks of the decode planner: for many cache shapes and states the
host-side plan (runs, tiles, splits) passes the pre-launch check that every
bulk copy is aligned, inside its buffer and sums to the tile's expected byte
count.  With no GPU in the process, a plan that passes reaches the launch and
comes back as KVQ_ERR_CUDA; a plan that fails the check would come back as
KVQ_ERR_INVALID_ARG / KVQ_ERR_UNSUPPORTED before any CUDA call."""
import ctypes
import itertools

import pytest

from quantized_kv_cache_kivi_gb300 import kvq

torch = pytest.importorskip("torch")
if torch.cuda.is_available():
    pytest.skip("meaningful only without a GPU (the launch must fail)", allow_module_level=True)

BASE = 1 << 40


def fake_cache(B, H, gq, d, G, R, segs, nkr, nvr, krs, vrs, policy=kvq.KVQ_POLICY_KIVI):
    c = kvq.kvq_cache()
    c.batch, c.h_kv, c.h_q, c.d_h, c.group, c.resid_cap = B, H, H * gq, d, G, R
    c.policy, c.sm_scale, c.n_seg = policy, 0.1, len(segs)
    addr = BASE
    P = B * H
    for i, (bits, cap, nk, nv) in enumerate(segs):
        s = c.seg[i]
        s.bits, s.capacity, s.nk, s.nv = bits, cap, nk, nv
        rb = d * bits // 8
        sizes = [P * cap * rb, P * (cap // G) * d * 2, P * (cap // G) * d * 2,
                 P * cap * rb, P * cap * (d // G) * 2, P * cap * (d // G) * 2]
        for f, sz in zip(("k_codes", "k_scale", "k_zero", "v_codes", "v_scale", "v_zero"), sizes):
            setattr(s, f, addr)
            addr += (sz + 4095) // 4096 * 4096 + 4096
    c.k_resid = addr
    addr += P * R * d * 2 + 4096
    c.v_resid = addr
    c.nkr, c.nvr, c.k_ring_start, c.v_ring_start = nkr, nvr, krs, vrs
    return c


def decode_status(c, splits=64):
    L = kvq.lib()
    ws = L.kvq_workspace_bytes(ctypes.byref(c), splits)
    return L.kvq_decode_attention(ctypes.byref(c), ctypes.c_void_p(BASE - 4096),
                                  ctypes.c_void_p(BASE - 8192), ctypes.c_void_p(BASE // 2),
                                  ws, None)


CASES = []
for d, G, bits, gq in itertools.product((64, 128), (16, 32, 64, 128), (2, 4, 8), (1, 2, 4, 7, 8)):
    if G > d:
        continue
    R = max(2 * G, 64)
    for nk_blocks, nkr, dv in ((0, 1, 0), (3, 5, 0), (7, R, 0), (5, 17, 3), (2, 0, -G)):
        nk = nk_blocks * R
        nv = nk + nkr - min(nk + nkr, R) if dv == 0 else max(nk + dv, 0)
        nvr = nk + nkr - nv
        if nvr > R or nvr < 0:
            continue
        CASES.append((d, G, bits, gq, R, nk, nkr, nv, nvr))


@pytest.mark.parametrize("d,G,bits,gq,R,nk,nkr,nv,nvr", CASES)
def test_plan_passes_bounds_check(d, G, bits, gq, R, nk, nkr, nv, nvr):
    cap = ((nk + nv + R) // G + 2) * G
    for krs, vrs in ((0, 0), (R - 1, R // 2 + 1)):
        c = fake_cache(2, 3, gq, d, G, R, [(bits, cap, nk, nv)], nkr, nvr, krs % R, vrs % R)
        st = decode_status(c)
        msg = kvq.lib().kvq_last_error_string().decode()
        assert st == kvq.KVQ_ERR_CUDA, (st, msg)


def test_plan_mixed_segments_and_splits():
    G, d, R = 32, 128, 128
    segs = [(8, 1536, 1536, 1536), (4, 4864, 4864, 4864), (2, 9984, 9984, 9984)]
    for gq, splits in itertools.product((1, 7), (1, 2, 5, 64)):
        c = fake_cache(1, 4, gq, d, G, R, segs, 64, 64, 3, 3, policy=kvq.KVQ_POLICY_FP16_TAIL)
        assert decode_status(c, splits) == kvq.KVQ_ERR_CUDA, kvq.lib().kvq_last_error_string()


def test_plan_detects_a_short_buffer():
    """The check really looks at the extents: a segment whose zero buffer
    overlaps the end of the scale buffer region by design still passes, but
    a segment that claims more valid tokens than its capacity is rejected."""
    c = fake_cache(1, 1, 1, 128, 32, 64, [(2, 256, 256, 200)], 8, 64, 0, 0)
    c.seg[0].nk = 288  # beyond capacity
    assert decode_status(c) == kvq.KVQ_ERR_INVALID_ARG


def test_decode_step_checks_arguments_before_any_launch():
    """kvq_decode_step / kvq_decode_step_host reject an unknown order and
    missing buffers before anything is enqueued, and leave the cache's
    lengths as they were."""
    L = kvq.lib()
    c = fake_cache(2, 3, 1, 128, 32, 64, [(2, 256, 128, 96)], 16, 48, 0, 0)
    before = (c.seg[0].nk, c.seg[0].nv, c.nkr, c.nvr, c.k_ring_start, c.v_ring_start)
    ws = L.kvq_workspace_bytes(ctypes.byref(c), 8)
    p = ctypes.c_void_p
    st = L.kvq_decode_step(ctypes.byref(c), p(BASE - 4096 * 4), p(BASE - 4096 * 3), p(BASE - 4096 * 2),
                           p(BASE - 4096), p(BASE // 2), ws, 7, None)
    assert st == kvq.KVQ_ERR_INVALID_ARG
    st = L.kvq_decode_step_host(ctypes.byref(c), None, None, p(BASE - 4096), p(BASE - 8192), p(BASE // 2), ws,
                                kvq.KVQ_STEP_ATTEND_FIRST, None)
    assert st == kvq.KVQ_ERR_INVALID_ARG
    assert (c.seg[0].nk, c.seg[0].nv, c.nkr, c.nvr, c.k_ring_start, c.v_ring_start) == before


@pytest.mark.parametrize("B,H,L", [(64, 32, 8256), (50, 32, 150), (1, 1, 4160)])
def test_plan_one_head_kernel_fills_the_slots(B, H, L):
    """The one-query-head kernel's plan for many pairs (pairs cut into k and
    k - 1 pieces to fill every warp slot), for a pair count near the slot
    count, and for one long pair: the plan passes the pre-launch copy check
    and reaches the launch."""
    G, d, R = 32, 128, 128
    nkr = L % G if L % G else G  # K: whole groups packed, the rest in the ring
    nk = L - nkr
    nvr = min(L, R)  # V: the newest R tokens in the ring
    nv = L - nvr
    cap = (L // G + 2) * G
    c = fake_cache(B, H, 1, d, G, R, [(2, cap, nk, nv)], nkr, nvr, 5, 7)
    assert decode_status(c) == kvq.KVQ_ERR_CUDA, kvq.lib().kvq_last_error_string()


def test_warp_chunk_geometry_enumeration(tmp_path):
    """Many cache states, ring starts, group sizes and pair counts through
    the one-query-head kernel's chunk, piece and copy geometry (host build
    of tests/warp_geometry.cu)."""
    import os
    import shutil
    import subprocess
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = tmp_path / "warp_geometry"
    subprocess.run([nvcc, "-std=c++17", "-O2", "--expt-relaxed-constexpr", "-x", "cu",
                    os.path.join(root, "tests", "warp_geometry.cu"), "-o", str(exe)],
                   check=True, capture_output=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:]
    assert "bad 0" in r.stdout
