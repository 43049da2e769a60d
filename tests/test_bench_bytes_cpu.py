"""CPU checks of the benchmark's byte accounting: the algorithmic bytes that
every effective-bandwidth and roofline figure divides by, against closed
forms worked out by hand for the workloads' states."""
import bench
from quantized_kv_cache_kivi_gb300 import kvq, synth


def test_llama2_step_bytes_closed_form():
    # per (batch, kv head): 3968 packed tokens x (32 B K codes + 16 B K scale
    # and zero per token at G = 32 + 32 B V codes + 16 B V scale and zero)
    # plus 128 fp16 ring tokens x (256 B K + 256 B V); 256 pairs
    w = synth.WORKLOADS["llama2_7b"]
    want = 256 * (3968 * 96 + 128 * 512)
    assert want == 114294784
    assert bench.algorithmic_bytes(w, 3968, 128, 3968, 128) == want


def test_cache_bytes_windowquant_segments():
    # one request, 4 kv heads, d_h 128, G 32: INT8 / INT4 / INT2 segments of
    # 1536 / 4864 / 9984 tokens and 64 fp16 tokens per kv head
    c = kvq.kvq_cache()
    c.batch, c.h_kv, c.h_q, c.d_h, c.group, c.resid_cap = 1, 4, 28, 128, 32, 128
    c.n_seg = 3
    for i, (bits, n) in enumerate(((8, 1536), (4, 4864), (2, 9984))):
        c.seg[i].bits, c.seg[i].capacity, c.seg[i].nk, c.seg[i].nv = bits, n, n, n
    c.nkr = c.nvr = 64
    per_pair = 1536 * (128 + 16 + 128 + 16) + 4864 * (64 + 16 + 64 + 16) + \
        9984 * (32 + 16 + 32 + 16) + 64 * 512
    assert per_pair * 4 == 8847360
    assert bench.cache_bytes(kvq.Cache(c, {})) == 8847360


def test_cache_bytes_separate_v_group():
    # V groups of 16 channels: 8 scale/zero pairs per token instead of 4
    c = kvq.kvq_cache()
    c.batch, c.h_kv, c.h_q, c.d_h, c.group, c.resid_cap, c.group_v = 2, 3, 3, 128, 64, 128, 16
    c.n_seg = 1
    c.seg[0].bits, c.seg[0].capacity, c.seg[0].nk, c.seg[0].nv = 4, 1024, 512, 400
    c.nkr, c.nvr = 16, 128
    per_pair = 512 * 64 + (512 // 64) * 128 * 4 + 400 * 64 + 400 * 8 * 4 + (16 + 128) * 256
    assert bench.cache_bytes(kvq.Cache(c, {})) == 6 * per_pair


def test_paged_bytes_sums_the_sequences():
    c = kvq.kvq_paged_cache()
    c.batch, c.h_kv, c.h_q, c.d_h, c.group, c.bits, c.resid_cap = 3, 2, 2, 128, 32, 2, 128
    states = [(0, 0, 0, 0), (640, 4, 516, 128), (4096, 100, 4068, 128)]  # (nk, nkr, nv, nvr)
    want = 0
    for b, (nk, nkr, nv, nvr) in enumerate(states):
        s = c.seq[b]
        s.nk, s.nkr, s.nv, s.nvr = nk, nkr, nv, nvr
        want += 2 * (nk * 32 + (nk // 32) * 512 + nv * 32 + nv * 16 + (nkr + nvr) * 256)
    assert bench.paged_bytes(kvq.PagedCache(c, {})) == want
    # per packed token 48 B for K (codes + scale/zero share) and 48 B for V
    assert want == 2 * (640 * 48 + 516 * 48 + 132 * 256) + 2 * (4096 * 48 + 4068 * 48 + 228 * 256)
