"""kvq_decode_attention_noalloc: decode attention for callers that cannot
allocate device memory (a plugin or custom-operator interface that hands
over only its input and output tensors, or a process whose device memory
belongs to another allocator).  Its workspace is the library's own static
device array, so the call needs no buffer from the caller.

Checked through the C ABI against kvq_decode_attention with a caller
workspace and, on two sampled (batch, kv head) pairs, against the oracle, on
two calls in a row, so the second call runs on the array the first one left
behind."""
import ctypes

import numpy as np
import pytest

from kvq_testutil import TOL, KiviPair, kv, max_abs_rel, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from quantized_kv_cache_kivi_gb300 import kvq, synth  # noqa: E402


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    B, H, gq, d, G, R = 4, 8, 4, 128, 32, 128
    pair = KiviPair(B, H, H * gq, d, G, R, 2, cap=3072, heads=[(0, 0), (3, 7)])
    K, V = kv(71, B, H, 2600, d)
    pair.prefill(K[:, :, :2599], V[:, :, :2599])
    pair.append(K[:, :, 2599:], V[:, :, 2599:], flush=False)  # packed + full fp16 ring
    ws = torch.zeros(kvq.kvq_workspace_bytes(pair.gpu, kvq.KVQ_MAX_SPLITS), dtype=torch.uint8,
                     device="cuda")
    for call in range(2):
        qh = synth.q_block(72, B, H * gq, d, step=call)
        q = to_dev(qh)
        ref = torch.empty_like(q)
        got = torch.full_like(q, float("nan"))
        kvq.kvq_decode_attention(pair.gpu, q, ref, ws)
        kvq.kvq_decode_attention_noalloc(pair.gpu, q, got)
        torch.cuda.synchronize()
        assert kvq.kvq_noalloc_error() == 0, call  # no bounded wait ran out
        assert kvq.kvq_workspace_error(ws) == 0, call
        g = got.cpu().numpy().astype(np.float64)
        r = ref.cpu().numpy().astype(np.float64)
        assert np.isfinite(g).all()
        assert max_abs_rel(g, r) < TOL, call
        orc = pair.oracle_attention(qh)
        for (b, h), o in orc.items():
            assert max_abs_rel(g[b, h * gq:(h + 1) * gq], o) < TOL, (call, b, h)


def test_noalloc_rejects_caches_beyond_the_static_array():
    """batch * h_kv large enough that even one split needs more scratch than
    the array holds: rejected before anything touches the device."""
    c = kvq.kvq_cache()
    c.batch, c.h_kv, c.h_q, c.d_h, c.group, c.resid_cap = 1 << 14, 128, 128, 128, 32, 64
    c.policy, c.sm_scale, c.n_seg = kvq.KVQ_POLICY_KIVI, 0.088, 1
    s = c.seg[0]
    s.bits, s.capacity = 2, 64
    for i, f in enumerate(("k_codes", "k_scale", "k_zero", "v_codes", "v_scale", "v_zero")):
        setattr(s, f, (1 << 40) + (i << 32))
    c.k_resid, c.v_resid = (1 << 41), (1 << 41) + (1 << 36)
    L = kvq.lib()
    st = L.kvq_decode_attention_noalloc(ctypes.byref(c), ctypes.c_void_p(4096),
                                        ctypes.c_void_p(8192), None)
    assert st == kvq.KVQ_ERR_CAPACITY
    assert b"KVQ_NOALLOC_SCRATCH_BYTES" in L.kvq_last_error_string()
