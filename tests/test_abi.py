"""CPU checks of the C ABI: libkvq.so builds, loads, exports every function
include/kvq.h declares, its structs have the header's layout, and host-side
validation rejects bad arguments with a status code (no GPU needed: nothing
is launched for a rejected call)."""
import ctypes
import os
import subprocess

import pytest

from quantized_kv_cache_kivi_gb300 import kvq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    return kvq.lib()


def test_exports_every_header_function(L):
    names = kvq.header_symbols()
    assert len(names) >= 10
    for n in names:
        assert hasattr(L, n), n
    for n in ("kvq_quantize_append", "kvq_flush_residual", "kvq_decode_attention",
              "kvq_window_assign"):
        assert n in names


def test_struct_layout_matches_header(tmp_path):
    src = tmp_path / "layout.c"
    src.write_text(r'''
#include <stdio.h>
#include <stddef.h>
#include "kvq.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu %zu %zu %zu\n", sizeof(kvq_segment), sizeof(kvq_cache),
         offsetof(kvq_cache, seg), offsetof(kvq_cache, k_resid), offsetof(kvq_cache, nkr),
         offsetof(kvq_cache, v_ring_start), sizeof(kvq_window_plan), offsetof(kvq_segment, k_codes));
  return 0;
}
''')
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True,
                                          check=True).stdout.split()]
    want = [ctypes.sizeof(kvq.kvq_segment), ctypes.sizeof(kvq.kvq_cache),
            kvq.kvq_cache.seg.offset, kvq.kvq_cache.k_resid.offset, kvq.kvq_cache.nkr.offset,
            kvq.kvq_cache.v_ring_start.offset, ctypes.sizeof(kvq.kvq_window_plan),
            kvq.kvq_segment.k_codes.offset]
    assert got == want


def _fake_cache():
    c = kvq.kvq_cache()
    c.batch, c.h_kv, c.h_q, c.d_h, c.group, c.resid_cap = 2, 2, 4, 128, 32, 64
    c.policy, c.sm_scale, c.n_seg = kvq.KVQ_POLICY_KIVI, 0.088, 1
    s = c.seg[0]
    s.bits, s.capacity = 2, 256
    for i, f in enumerate(("k_codes", "k_scale", "k_zero", "v_codes", "v_scale", "v_zero")):
        setattr(s, f, 0x100000 * (i + 1))
    c.k_resid, c.v_resid = 0x800000, 0x900000
    return c


def _status(L, c):
    return L.kvq_flush_residual(ctypes.byref(c), None)  # validation runs first


def test_validation_statuses(L):
    c = _fake_cache()
    assert _status(L, c) == kvq.KVQ_OK  # nothing due: no launch, no GPU needed
    bad = [("d_h", 96, kvq.KVQ_ERR_UNSUPPORTED), ("group", 48, kvq.KVQ_ERR_UNSUPPORTED),
           ("h_q", 3, kvq.KVQ_ERR_INVALID_ARG), ("h_q", 2 * 9, kvq.KVQ_ERR_UNSUPPORTED),
           ("resid_cap", 40, kvq.KVQ_ERR_INVALID_ARG), ("nkr", 65, kvq.KVQ_ERR_INVALID_ARG),
           ("k_ring_start", 64, kvq.KVQ_ERR_INVALID_ARG), ("policy", 7, kvq.KVQ_ERR_INVALID_ARG),
           ("n_seg", 0, kvq.KVQ_ERR_INVALID_ARG), ("k_resid", 0x800004, kvq.KVQ_ERR_INVALID_ARG)]
    for field, value, want in bad:
        c = _fake_cache()
        setattr(c, field, value)
        assert _status(L, c) == want, field
        assert L.kvq_last_error_string()
    for field, value, want in [("bits", 3, kvq.KVQ_ERR_UNSUPPORTED),
                               ("capacity", 100, kvq.KVQ_ERR_INVALID_ARG),
                               ("nk", 16, kvq.KVQ_ERR_INVALID_ARG),
                               ("k_zero", 0, kvq.KVQ_ERR_INVALID_ARG)]:
        c = _fake_cache()
        setattr(c.seg[0], field, value)
        assert _status(L, c) == want, field
    c = _fake_cache()
    c.seg[0].nk, c.nkr, c.seg[0].nv, c.nvr = 32, 5, 30, 6  # 37 vs 36 tokens
    assert _status(L, c) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_flush_residual(None, None) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_decode_attention(None, None, None, None, 0, None) == kvq.KVQ_ERR_INVALID_ARG
    c = _fake_cache()
    assert L.kvq_decode_attention(ctypes.byref(c), ctypes.c_void_p(0x1000),
                                  ctypes.c_void_p(0x2000), None, 0, None) == kvq.KVQ_ERR_WORKSPACE


def test_workspace_size_arithmetic(L):
    c = _fake_cache()
    pairs, gq, d = 4, 2, 128
    fixed = 256 + 256  # header + counters rounded to 256 bytes
    assert L.kvq_workspace_bytes(ctypes.byref(c), 1) == fixed
    assert L.kvq_workspace_bytes(ctypes.byref(c), 8) == fixed + pairs * 8 * gq * (d + 2) * 4
    # clamped to KVQ_MAX_SPLITS (read from the header)
    import re
    hdr = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "kvq.h")).read()
    cap = int(re.search(r"#define KVQ_MAX_SPLITS (\d+)", hdr).group(1))
    assert cap == kvq.KVQ_MAX_SPLITS
    assert L.kvq_workspace_bytes(ctypes.byref(c), 1000) == fixed + pairs * cap * gq * (d + 2) * 4


def test_status_strings(L):
    for st in (0, 1, -1, -2, -3, -4, -5):
        assert L.kvq_status_string(st)
