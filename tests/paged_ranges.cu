// Host check of the paged cache's stream-K planning (kvq_paged.cu:
// paged_tc_costs, paged_tc_ranges) on random ragged batches: the costs built
// from each sequence's runs equal the costs of its tiles taken one by one
// (kvq_internal.h: paged_tile), and the forward walk finds the same range
// boundaries as a binary search over the whole cost prefix, with no range
// empty.  The library's launch functions are stubbed out: nothing runs on a
// GPU.  Built and run on the CPU by tests/test_paged_cpu.py; exits nonzero
// on a mismatch.
#include <cstdio>
#include <random>
#include "../quantized_kv_cache_kivi_gb300/csrc/kvq_paged.cu"
namespace kvq {
void set_last_error(const char*) {}
int sm_count_cached() { return 152; }
cudaError_t launch_paged_append(const PagedAppendArgs&, cudaStream_t) { return cudaSuccess; }
cudaError_t launch_decode_paged(const PagedArgs&, cudaStream_t) { return cudaSuccess; }
cudaError_t launch_decode_tc_paged(const DecodeArgs&, const PagedArgs&, int, int, cudaStream_t) { return cudaSuccess; }
cudaError_t launch_decode_tc_merge(const DecodeArgs&, int, cudaStream_t) { return cudaSuccess; }
int decode_tc_ctas_per_sm() { return 2; }
}
int main() {
  std::mt19937 rng(1);
  long long bad = 0, runs = 0;
  for (int trial = 0; trial < 3000; ++trial) {
    kvq::PagedArgs a{};
    a.n_seq = 1 + rng() % 40; a.tile_pp = 128; a.tile_mix = 32; a.G = 32; a.R = 128; a.d = 128; a.Gv = 32; a.bits = 2; a.P = 256;
    const int h_kv = 1 + rng() % 8;
    int nt = 0;
    for (int b = 0; b < a.n_seq; ++b) {
      kvq::PagedSeq& q = a.seq[b];
      const int L = rng() % 3 == 0 ? 0 : rng() % 9000;
      q.nk = (L / 128) * 128; q.nkr = L - q.nk; q.nvr = std::min(L, 128); q.nv = L - q.nvr;
      q.n_tiles = kvq::paged_tiles(a, q);
      nt = std::max(nt, q.n_tiles);
    }
    if (nt == 0) continue;
    const auto pre = paged_tc_costs(a, nt);
    for (int b = 0; b < a.n_seq; ++b)
      for (int t = 0; t < nt; ++t) {
        long long c = 0;
        if (t < a.seq[b].n_tiles) {
          const kvq::TileInfo ti = kvq::paged_tile(a, a.seq[b], t);
          c = (ti.kseg == 0 && ti.vseg == 0) ? 4 * ((ti.n + 31) / 32) + 1 : 48;
          if (t == 0) c += 16;
        }
        if (pre[(size_t)b * (nt + 1) + t + 1] - pre[(size_t)b * (nt + 1) + t] != c) { if (bad < 5) printf("cost mismatch\n"); ++bad; }
      }
    const long long n_pairs = (long long)a.n_seq * h_kv, T = n_pairs * nt;
    // brute-force prefix and binary search
    std::vector<long long> cum(n_pairs + 1, 0);
    for (long long p = 0; p < n_pairs; ++p) cum[p + 1] = cum[p] + pre[(p / h_kv) * (nt + 1) + nt];
    auto prefix = [&](long long g) { long long p = g / nt; return p >= n_pairs ? cum[n_pairs] : cum[p] + pre[(p / h_kv) * (nt + 1) + g % nt]; };
    for (int N : {1, 2, 7, 64, 304}) {
      if (N > T) continue;
      std::vector<int> b1(N + 1), b2(N + 1);
      paged_tc_ranges(pre, a.n_seq, h_kv, nt, N, b1.data());
      b2[0] = 0;
      for (int i = 1; i < N; ++i) {
        const long long target = cum[n_pairs] * i / N;
        long long lo = 0, hi = T;
        while (lo < hi) { long long mid = (lo + hi) / 2; if (prefix(mid) >= target) hi = mid; else lo = mid + 1; }
        lo = std::max<long long>(lo, b2[i - 1] + 1); lo = std::min<long long>(lo, T - (N - i)); b2[i] = (int)lo;
      }
      b2[N] = (int)T;
      ++runs;
      if (b1 != b2) { if (bad < 5) printf("mismatch trial %d N %d\n", trial, N); ++bad; }
      for (int i = 0; i < N; ++i) if (b1[i] >= b1[i + 1]) { if (bad < 5) printf("empty range\n"); ++bad; }
    }
  }
  printf("runs %lld bad %lld\n", runs, bad);
  return bad != 0;
}
