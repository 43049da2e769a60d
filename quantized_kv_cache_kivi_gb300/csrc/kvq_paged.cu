// C ABI of the paged cache (include/kvq.h, kvq_paged_*): per-sequence KIVI
// Algorithm 1 bookkeeping on the host, packed tokens in a pool of pages
// reached through the caller's block table, one launch per call for the
// whole batch whatever the sequences' lengths.
#include <algorithm>
#include <climits>
#include <cstdarg>
#include <cstdio>
#include <vector>

#include "kvq_internal.h"

// The per-sequence tables travel as kernel parameters (by value, no upload),
// which CUDA limits to 32,764 bytes per launch.
static_assert(sizeof(kvq::PagedAppendArgs) <= 32000, "paged append arguments exceed the kernel parameter limit");
static_assert(sizeof(kvq::PagedArgs) <= 32000, "paged decode arguments exceed the kernel parameter limit");
static_assert(sizeof(kvq::DecodeArgs) + sizeof(kvq::PagedArgs) <= 32000,
              "paged tensor-core arguments exceed the kernel parameter limit");

namespace {

kvq_status pfail(kvq_status st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
kvq_status pfail(kvq_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  kvq::set_last_error(buf);
  return st;
}

kvq_status pcuda(cudaError_t e, const char* what) {
  return pfail(KVQ_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool al16(const void* p) { return p && ((uintptr_t)p & 15u) == 0; }

bool pow2_in(int x, int lo, int hi) { return x >= lo && x <= hi && (x & (x - 1)) == 0; }

int gv_of(const kvq_paged_cache* c) { return c->group_v ? c->group_v : c->group; }

long long seq_cap(const kvq_paged_cache* c) { return (long long)c->max_pages * c->page_tokens; }

kvq_status validate_paged(const kvq_paged_cache* c) {
  if (!c) return pfail(KVQ_ERR_INVALID_ARG, "cache is NULL");
  if (c->batch < 1 || c->batch > KVQ_MAX_SEQS)
    return pfail(KVQ_ERR_INVALID_ARG, "batch must be 1..%d", KVQ_MAX_SEQS);
  if (c->h_kv < 1 || c->h_q < 1 || c->h_q % c->h_kv != 0)
    return pfail(KVQ_ERR_INVALID_ARG, "h_kv, h_q >= 1 and h_q a multiple of h_kv");
  if (c->h_q / c->h_kv > kvq::kMaxGq)
    return pfail(KVQ_ERR_UNSUPPORTED, "more than %d query heads per kv head", kvq::kMaxGq);
  if (c->d_h != 64 && c->d_h != 128) return pfail(KVQ_ERR_UNSUPPORTED, "d_h must be 64 or 128");
  const int G = c->group, Gv = gv_of(c);
  if (!pow2_in(G, 16, 256)) return pfail(KVQ_ERR_UNSUPPORTED, "group must be 16 .. 256, a power of two");
  if (!pow2_in(Gv, 8, 128) || c->d_h % Gv != 0)
    return pfail(KVQ_ERR_UNSUPPORTED, "the V group must be 8 .. 128, a power of two dividing d_h");
  if (c->resid_cap < G || c->resid_cap % G != 0)
    return pfail(KVQ_ERR_INVALID_ARG, "resid_cap must be a positive multiple of group");
  if (c->bits != 2 && c->bits != 4 && c->bits != 8) return pfail(KVQ_ERR_UNSUPPORTED, "bits must be 2, 4 or 8");
  if (c->zero_point != KVQ_ZERO_MIN && c->zero_point != KVQ_ZERO_INT)
    return pfail(KVQ_ERR_INVALID_ARG, "zero_point must be KVQ_ZERO_MIN or KVQ_ZERO_INT");
  if (c->page_tokens < 128 || c->page_tokens % 128 != 0 || c->page_tokens % G != 0)
    return pfail(KVQ_ERR_INVALID_ARG, "page_tokens must be a multiple of 128 and of group");
  if (c->n_pages < 1 || c->max_pages < 1) return pfail(KVQ_ERR_INVALID_ARG, "n_pages, max_pages must be >= 1");
  if (seq_cap(c) > INT_MAX / 2) return pfail(KVQ_ERR_UNSUPPORTED, "max_pages * page_tokens too large");
  if (!al16(c->k_codes) || !al16(c->k_scale) || !al16(c->k_zero) || !al16(c->v_codes) ||
      !al16(c->v_scale) || !al16(c->v_zero) || !al16(c->block_table) || !al16(c->k_resid) ||
      !al16(c->v_resid) || !al16(c->err))
    return pfail(KVQ_ERR_INVALID_ARG, "every device pointer must be non-NULL and 16-byte aligned");
  for (int b = 0; b < c->batch; ++b) {
    const kvq_seq_state& s = c->seq[b];
    if (s.nk < 0 || s.nv < 0 || s.nkr < 0 || s.nvr < 0 || s.nkr > c->resid_cap || s.nvr > c->resid_cap ||
        s.nk % G != 0 || (long long)s.nk + s.nkr != (long long)s.nv + s.nvr || s.nk > seq_cap(c) ||
        s.nv > seq_cap(c) || s.k_ring_start < 0 || s.k_ring_start >= c->resid_cap || s.v_ring_start < 0 ||
        s.v_ring_start >= c->resid_cap)
      return pfail(KVQ_ERR_INVALID_ARG, "inconsistent lengths of sequence %d", b);
  }
  return KVQ_OK;
}

int sms() { return kvq::sm_count_cached(); }

size_t ws_head(int n_pairs) { return kvq::kWorkspaceHeader + (((size_t)n_pairs * 4 + 255) / 256) * 256; }

// Stage bytes of a tile of `t` tokens (K and V widths kb, vb; 16 = fp16),
// counting one K scale group more than an aligned tile can touch.
int stage_bytes(int t, int kb, int vb, int d, int G, int Gv) {
  auto a16 = [](int x) { return (x + 15) & ~15; };
  int b = a16(t * d * kb / 8) + a16(t * d * vb / 8);
  if (kb != 16) b += 2 * ((t + G - 1) / G + 1) * d * 2;
  if (vb != 16) b += 2 * a16(t * (d / Gv) * 2);
  return b;
}

bool tile_fits(int t, int kb, int vb, int d, int G, int Gv, int gq) {
  if (stage_bytes(t, kb, vb, d, G, Gv) > kvq::kStageBytes) return false;
  return kb == 16 || ((t + G - 1) / G + 1) * gq * d * 4 <= kvq::kQsBytes;
}

// Geometry check of a paged plan: every run's first and last tile of every
// sequence (interior tiles repeat the aligned full-size shape) through the
// kernels' own functions: tokens, stage bytes, no page crossed, 16-byte
// copies inside their page (page 0 stands in) or ring, bytes as expected;
// for the tensor-core kernel also the K groups a tile touches and 32-token
// units inside one K group.
kvq_status check_paged_plan(const kvq_paged_cache* c, const kvq::PagedArgs& a, uint32_t stage_cap, bool tc) {
  const int d = a.d, G = a.G, Gv = a.Gv, rb = d * a.bits / 8;
  const size_t n_pairs = (size_t)c->batch * c->h_kv;
  const size_t page_k = (size_t)c->h_kv * a.P * rb;
  const size_t ring = n_pairs * a.R * d * 2;
  for (int b = 0; b < c->batch; ++b) {
    const kvq::PagedSeq& q = a.seq[b];
    const int L = q.nk + q.nkr;
    const int a0 = std::min(q.nk, q.nv), a1 = std::max(q.nk, q.nv);
    const int n0 = kvq::paged_run_tiles(0, a0, a.tile_pp), n1 = kvq::paged_run_tiles(a0, a1, a.tile_mix),
              n2 = kvq::paged_run_tiles(a1, L, a.tile_mix);
    const int ends[6] = {0, n0 - 1, n0, n0 + n1 - 1, n0 + n1, n0 + n1 + n2 - 1};
    for (int t : ends) {
      if (t < 0 || t >= q.n_tiles) continue;
      const kvq::TileInfo ti = kvq::paged_tile(a, q, t);
      if (ti.n < 1 || ti.bytes > stage_cap || ti.n > (tc ? 256 : 128))
        return pfail(KVQ_ERR_UNSUPPORTED, "paged tile %d of sequence %d does not fit a stage", t, b);
      if ((ti.kseg == 0 && (ti.ku0 / a.P != (ti.ku0 + ti.n - 1) / a.P)) ||
          (ti.vseg == 0 && (ti.vu0 / a.P != (ti.vu0 + ti.n - 1) / a.P)))
        return pfail(KVQ_ERR_UNSUPPORTED, "paged tile %d of sequence %d crosses a page", t, b);
      if (tc && ti.kseg == 0 &&
          (ti.ng > kvq::kTcMaxGroups || (ti.ku0 % 32 != 0 && ti.ku0 / 32 != (ti.ku0 + ti.n - 1) / 32)))
        return pfail(KVQ_ERR_UNSUPPORTED, "paged tile %d of sequence %d: K groups or units", t, b);
      uint32_t sum = 0;
      bool ok = true;
      // the buffer a copy must stay in follows from its slot and its side's
      // source (page 0 stands in for the pool page)
      const void* packed[6] = {a.kc, a.ks, a.kz, a.vc, a.vs, a.vz};
      const size_t gsz = page_k / rb / G * d * 2, vsz = page_k / rb * (d / Gv) * 2;
      const size_t psize[6] = {page_k, gsz, gsz, page_k, vsz, vsz};
      kvq::for_each_paged_copy(a, b, c->h_kv - 1, q, ti, [](int) { return 0; },
                               [&](const void* src, uint32_t off, uint32_t bytes, int slot) {
                                 sum += bytes;
                                 if (slot < 0 || slot > 5 || bytes % 16 || off % 16 || ((uintptr_t)src & 15u)) {
                                   ok = false;
                                   return;
                                 }
                                 const bool ring_side = slot < 3 ? ti.kseg != 0 : ti.vseg != 0;
                                 const uint8_t* b0 = static_cast<const uint8_t*>(
                                     ring_side ? (slot < 3 ? (const void*)a.kr : (const void*)a.vr) : packed[slot]);
                                 const size_t n = ring_side ? ring : psize[slot];
                                 const uint8_t* p = static_cast<const uint8_t*>(src);
                                 if (p < b0 || p + bytes > b0 + n) ok = false;
                               });
      if (!ok || sum != ti.bytes)
        return pfail(KVQ_ERR_UNSUPPORTED, "paged tile %d of sequence %d: copy geometry check failed", t, b);
    }
  }
  return KVQ_OK;
}

// Stream-K ranges of the tensor-core kernel over a paged cache: every pair
// padded to nt tiles.  Cost of a live tile: 4 per 32-token unit plus 1 when
// K and V are both packed; a tile that reads a ring (one 32-token unit of
// fp16 K or V) costs 48, and a pair's first tile adds 16 for the pair's
// merge; a padding tile costs nothing.  Such ring tiles keep one consumer
// warp busy each while they hold a pipeline stage; measured on a ragged
// batch (16 sequences, 644-7650 tokens, 2-bit), ring costs of 12 / 20 / 40
// / 56 / 72 / 96 gave 133 / 117 / 94 / 93 / 94 / 101 us.  (In the uniform
// cache every pair has the same mix of tiles, so the weights do not move
// its ranges much; sequences of different lengths put very different mixes
// into one CTA's range.)  CTA i's range starts at the first tile whose cost
// prefix reaches i/N of the total, kept non-empty.  Returns the most ranges
// that meet one pair.
// Cost prefix of each sequence's tiles, padded to nt: [B][nt + 1], built
// from the sequence's runs with arithmetic alone (tiles of the both-packed
// run first, at 4 per 32-token unit + 1; every later tile reads a ring).
std::vector<long long> paged_tc_costs(const kvq::PagedArgs& a, int nt) {
  std::vector<long long> pre((size_t)a.n_seq * (nt + 1), 0);
  for (int b = 0; b < a.n_seq; ++b) {
    const kvq::PagedSeq& q = a.seq[b];
    const int a0 = std::min(q.nk, q.nv), n0 = kvq::paged_run_tiles(0, a0, a.tile_pp);
    long long* pb = pre.data() + (size_t)b * (nt + 1);
    for (int t = 0; t < nt; ++t) {
      long long c = 0;
      if (t < q.n_tiles) {
        c = t < n0 ? 4 * ((std::min(a.tile_pp, a0 - t * a.tile_pp) + 31) / 32) + 1 : 48;
        if (t == 0) c += 16;
      }
      pb[t + 1] = pb[t] + c;
    }
  }
  return pre;
}

int paged_tc_ranges(const std::vector<long long>& pre, int B, int h_kv, int nt, int N, int* bound) {
  const long long n_pairs = (long long)B * h_kv, T = n_pairs * nt;
  std::vector<long long> cum(n_pairs + 1, 0);
  for (long long pr = 0; pr < n_pairs; ++pr) cum[pr + 1] = cum[pr] + pre[(size_t)(pr / h_kv) * (nt + 1) + nt];
  const long long total = cum[n_pairs];
  bound[0] = 0;
  // first g with prefix(g) >= target, prefix(pr nt + t) = cum[pr] + pre_b[t]:
  // targets rise with i, so the pair that holds a target is found by
  // walking forward (the first pair whose end reaches it), then the tile by
  // a lower bound inside that pair
  long long pr = 0;
  for (int i = 1; i < N; ++i) {
    const long long target = total * i / N;
    while (pr < n_pairs && cum[pr + 1] < target) ++pr;
    long long lo = T;
    if (pr < n_pairs) {
      const long long* pb = pre.data() + (size_t)(pr / h_kv) * (nt + 1);
      lo = pr * nt + (std::lower_bound(pb, pb + nt + 1, target - cum[pr]) - pb);
    }
    lo = std::max<long long>(lo, bound[i - 1] + 1);
    lo = std::min<long long>(lo, T - (N - i));
    bound[i] = (int)lo;
  }
  bound[N] = (int)T;
  int most = 1, run = 1;
  long long run_pair = -1;
  for (int i = 1; i < N; ++i) {
    if (bound[i] % nt == 0) continue;
    const long long p = bound[i] / nt;
    run = p == run_pair ? run + 1 : 2;
    run_pair = p;
    most = std::max(most, run);
  }
  return most;
}

// Tensor-core form for a paged cache (the uniform cache's rules): 1 = one
// query head per kv head, 4 = 2-4 heads, 8 = up to 8 heads (no tile with
// fp16 K beside packed V); 0 = the general kernel.
int paged_tc_form(const kvq_paged_cache* c) {
  const int gq = c->h_q / c->h_kv, d = c->d_h, G = c->group, Gv = gv_of(c);
  if (d != 128 || G < 32) return 0;
  if (gq == 1 && Gv >= d / 4) return 1;
  if (gq >= 2 && gq <= 4 && Gv >= 64) return 4;
  if (gq <= kvq::kMaxGq && Gv >= 16) {
    for (int b = 0; b < c->batch; ++b)
      if (c->seq[b].nv > c->seq[b].nk) return 0;
    return 8;
  }
  return 0;
}

kvq::PagedAppendArgs append_base(const kvq_paged_cache* c, int T, const void* k_new, const void* v_new) {
  kvq::PagedAppendArgs a{};
  a.batch = c->batch;
  a.h_kv = c->h_kv;
  a.d = c->d_h;
  a.G = c->group;
  a.Gv = gv_of(c);
  a.R = c->resid_cap;
  a.T = T;
  a.P = c->page_tokens;
  a.bits = c->bits;
  a.intz = c->zero_point == KVQ_ZERO_INT;
  a.k_new = static_cast<const __half*>(k_new);
  a.v_new = static_cast<const __half*>(v_new);
  a.kr = static_cast<__half*>(c->k_resid);
  a.vr = static_cast<__half*>(c->v_resid);
  a.kc = static_cast<uint8_t*>(c->k_codes);
  a.ks = static_cast<__half*>(c->k_scale);
  a.kz = static_cast<__half*>(c->k_zero);
  a.vc = static_cast<uint8_t*>(c->v_codes);
  a.vs = static_cast<__half*>(c->v_scale);
  a.vz = static_cast<__half*>(c->v_zero);
  a.table = c->block_table;
  a.max_pages = c->max_pages;
  a.n_pages = c->n_pages;
  a.page_err = c->err;
  return a;
}

}  // namespace

extern "C" {

kvq_status kvq_paged_append(kvq_paged_cache* c, const void* k_new, const void* v_new, int32_t T,
                            const int32_t* t_seq, void* stream) {
  kvq_status st = validate_paged(c);
  if (st != KVQ_OK) return st;
  if (T < 0) return pfail(KVQ_ERR_INVALID_ARG, "T must be >= 0");
  if (T == 0) return KVQ_OK;
  if (!al16(k_new) || !al16(v_new)) return pfail(KVQ_ERR_INVALID_ARG, "k_new/v_new must be non-NULL and 16-byte aligned");
  const int R = c->resid_cap, G = c->group;
  kvq::PagedAppendArgs a = append_base(c, T, k_new, v_new);
  bool due = false;
  int most = 0;
  long long k_items = 0, v_items = 0;
  // KIVI Algorithm 1 per sequence, as the uniform cache's append
  for (int b = 0; b < c->batch; ++b) {
    const kvq_seq_state& s = c->seq[b];
    const int t = t_seq ? t_seq[b] : T;
    if (t < 0 || t > T) return pfail(KVQ_ERR_INVALID_ARG, "t_seq[%d] = %d outside 0..T", b, t);
    // (a sequence with no new tokens is left as it is; a full K ring left
    // from before still reports the flush as due)
    const long long pushed = (long long)s.nkr + t;
    long long nb = t > 0 ? pushed / R : 0;
    if (t > 0 && nb >= 1 && pushed % R == 0) --nb;
    if (pushed >= R && pushed % R == 0) due = true;
    const int fb = (int)nb;
    const int evict = (int)std::max(0LL, (long long)s.nvr + t - R);
    if ((long long)s.nk + (long long)fb * R > seq_cap(c) || (long long)s.nv + evict > seq_cap(c))
      return pfail(KVQ_ERR_CAPACITY, "sequence %d would pass max_pages * page_tokens tokens", b);
    kvq::PagedAppendSeq& q = a.seq[b];
    q.t = t;
    q.k_groups = fb * R / G;
    q.k_nk0 = s.nk;
    q.ksrc = {s.nkr, s.k_ring_start};
    q.k_ring_groups = std::min(q.k_groups, (s.nkr + G - 1) / G);
    q.v_evict = evict;
    q.v_nv0 = s.nv;
    q.vsrc = {s.nvr, s.v_ring_start};
    q.v_ring_tokens = std::min(evict, s.nvr);
    q.k_first_ring = std::max(0, fb * R - s.nkr);
    q.k_slot0 = s.k_ring_start + s.nkr;
    q.v_first_ring = std::max(0, evict - s.nvr);
    q.v_slot0 = s.v_ring_start + s.nvr;
    const int in_k = q.k_groups - q.k_ring_groups, in_v = q.v_evict - q.v_ring_tokens;
    q.k_item0 = (int)k_items;
    q.v_item0 = (int)v_items;
    k_items += (long long)in_k * c->h_kv;
    v_items += (long long)in_v * c->h_kv;
    most = std::max(most, in_k + (in_v + 63) / 64);
  }
  if (k_items >= INT_MAX || v_items >= INT_MAX) return pfail(KVQ_ERR_UNSUPPORTED, "append too large for one call");
  a.n_seq = c->batch;
  a.k_items = (int)k_items;
  a.v_items = (int)v_items;
  // the new-token work of a prompt-sized append goes to grid-wide kernels;
  // the block kernel keeps the work that reads the old rings
  a.bulk = c->d_h == 128 && k_items + v_items > 0;
  a.chunks = (!a.bulk && most > 0) ? 1 + std::min(256, most) : 1;
  const cudaError_t e = kvq::launch_paged_append(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return pcuda(e, "paged append launch");
  for (int b = 0; b < c->batch; ++b) {
    kvq_seq_state& s = c->seq[b];
    const kvq::PagedAppendSeq& q = a.seq[b];
    s.nk += q.k_groups * G;
    s.nkr = s.nkr + q.t - q.k_groups * G;
    s.nv += q.v_evict;
    s.v_ring_start = (s.v_ring_start + q.v_evict) % R;
    s.nvr = s.nvr + q.t - q.v_evict;
  }
  return due ? KVQ_FLUSH_DUE : KVQ_OK;
}

kvq_status kvq_paged_flush_residual(kvq_paged_cache* c, void* stream) {
  kvq_status st = validate_paged(c);
  if (st != KVQ_OK) return st;
  const int R = c->resid_cap, G = c->group;
  kvq::PagedAppendArgs a = append_base(c, 0, nullptr, nullptr);
  a.flush = 1;
  int most = 0;
  for (int b = 0; b < c->batch; ++b) {
    const kvq_seq_state& s = c->seq[b];
    const int n = s.nkr == R ? R : 0;  // Algorithm 1: len(X_Kr) == R
    if ((long long)s.nk + n > seq_cap(c))
      return pfail(KVQ_ERR_CAPACITY, "sequence %d would pass max_pages * page_tokens tokens", b);
    kvq::PagedAppendSeq& q = a.seq[b];
    q.k_groups = n / G;
    q.k_nk0 = s.nk;
    q.ksrc = {INT_MAX, s.k_ring_start};
    most = std::max(most, q.k_groups);
  }
  if (most == 0) return KVQ_OK;
  a.chunks = most;
  const cudaError_t e = kvq::launch_paged_append(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return pcuda(e, "paged flush launch");
  for (int b = 0; b < c->batch; ++b) {
    kvq_seq_state& s = c->seq[b];
    const int n = a.seq[b].k_groups * G;
    s.nk += n;
    s.nkr -= n;
    s.k_ring_start = (s.k_ring_start + n) % R;
  }
  return KVQ_OK;
}

size_t kvq_paged_workspace_bytes(const kvq_paged_cache* c, int32_t max_splits) {
  if (!c || c->batch < 1 || c->batch > KVQ_MAX_SEQS || c->h_kv < 1 || c->h_q < c->h_kv) return 0;
  max_splits = std::max(1, std::min<int>(max_splits, KVQ_MAX_SPLITS));
  const int n_pairs = c->batch * c->h_kv, gq = c->h_q / c->h_kv;
  return ws_head(n_pairs) + (size_t)n_pairs * max_splits * gq * (c->d_h + 2) * sizeof(float);
}

kvq_status kvq_paged_decode_attention(const kvq_paged_cache* c, const void* q, void* out, void* ws,
                                      size_t ws_bytes, void* stream) {
  kvq_status st = validate_paged(c);
  if (st != KVQ_OK) return st;
  if (!al16(q) || !al16(out)) return pfail(KVQ_ERR_INVALID_ARG, "q/out must be non-NULL and 16-byte aligned");
  const int n_pairs = c->batch * c->h_kv, gq = c->h_q / c->h_kv, d = c->d_h;
  const size_t per_split = (size_t)n_pairs * gq * (d + 2) * sizeof(float);
  if (!al16(ws) || ws_bytes < ws_head(n_pairs) + per_split)
    return pfail(KVQ_ERR_WORKSPACE, "workspace needs at least %zu bytes", ws_head(n_pairs) + per_split);
  const int ws_splits = (int)std::min<size_t>(KVQ_MAX_SPLITS, (ws_bytes - ws_head(n_pairs)) / per_split);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  kvq::PagedArgs a{};
  a.batch = c->batch;
  a.h_kv = c->h_kv;
  a.gq = gq;
  a.d = d;
  a.G = c->group;
  while ((1 << a.log2G) < a.G) ++a.log2G;
  a.Gv = gv_of(c);
  while ((1 << a.log2Gv) < a.Gv) ++a.log2Gv;
  a.R = c->resid_cap;
  a.P = c->page_tokens;
  a.bits = c->bits;
  a.scale_log2 = c->sm_scale * 1.4426950408889634f;
  a.intz = c->zero_point == KVQ_ZERO_INT;
  a.kc = static_cast<const uint8_t*>(c->k_codes);
  a.ks = static_cast<const __half*>(c->k_scale);
  a.kz = static_cast<const __half*>(c->k_zero);
  a.vc = static_cast<const uint8_t*>(c->v_codes);
  a.vs = static_cast<const __half*>(c->v_scale);
  a.vz = static_cast<const __half*>(c->v_zero);
  a.table = c->block_table;
  a.max_pages = c->max_pages;
  a.n_pages = c->n_pages;
  a.kr = static_cast<const __half*>(c->k_resid);
  a.vr = static_cast<const __half*>(c->v_resid);
  a.q = static_cast<const __half*>(q);
  a.out = static_cast<__half*>(out);
  uint8_t* w = static_cast<uint8_t*>(ws);
  a.err = reinterpret_cast<int*>(w);
  a.counters = reinterpret_cast<int*>(w + kvq::kWorkspaceHeader);
  a.part = reinterpret_cast<float*>(w + ws_head(n_pairs));
  a.page_err = c->err;
  a.n_splits = ws_splits;
  // tiles: the largest power of two that fits a stage (packed K and V), and
  // one for tiles that read a ring; both divide the page.  The tensor-core
  // kernel takes 32-token tiles where a ring is involved (a tile starting
  // inside a 32-token unit must end in it).
  const int G = a.G, Gv = a.Gv, bits = a.bits;
  const int form = paged_tc_form(c);
  const bool tc = form != 0;
  auto fits = [&](int t, int kb, int vb) {
    if (tc)
      return stage_bytes(t, kb, vb, d, G, Gv) <= kvq::kTcStageBytes &&
             (kb == 16 || (t + G - 1) / G + 1 <= kvq::kTcMaxGroups);
    return tile_fits(t, kb, vb, d, G, Gv, gq);
  };
  for (int t = tc ? 256 : 128; t >= (tc ? 32 : 16) && !a.tile_pp; t >>= 1)
    if (a.P % t == 0 && fits(t, bits, bits)) a.tile_pp = t;
  for (int t = tc ? 32 : a.tile_pp; t >= 16 && !a.tile_mix; t >>= 1)
    if (t <= a.tile_pp && fits(t, 16, 16) && fits(t, bits, 16) && fits(t, 16, bits)) a.tile_mix = t;
  if (!a.tile_pp || !a.tile_mix) return pfail(KVQ_ERR_UNSUPPORTED, "no tile fits a pipeline stage");
  long long total = 0;
  int nt_max = 0;
  std::vector<int> nt(c->batch);
  for (int b = 0; b < c->batch; ++b) {
    kvq::PagedSeq& q = a.seq[b];
    const kvq_seq_state& cs = c->seq[b];
    q.nk = cs.nk;
    q.nv = cs.nv;
    q.nkr = cs.nkr;
    q.nvr = cs.nvr;
    q.krs = cs.k_ring_start;
    q.vrs = cs.v_ring_start;
    nt[b] = kvq::paged_tiles(a, q);
    q.n_tiles = nt[b];
    nt_max = std::max(nt_max, nt[b]);
    total += (long long)nt[b] * c->h_kv;
  }
  a.n_seq = c->batch;
  if (total == 0) {
    const cudaError_t e = cudaMemsetAsync(out, 0, (size_t)c->batch * c->h_q * d * 2, s);
    return e == cudaSuccess ? KVQ_OK : pcuda(e, "zero output");
  }
  st = check_paged_plan(c, a, tc ? (uint32_t)kvq::kTcStageBytes : (uint32_t)kvq::kStageBytes, tc);
  if (st != KVQ_OK) return st;
  if (tc) {
    // the tensor-core kernel: persistent CTAs over all pairs' tiles, each
    // pair padded to the longest sequence's tile count (padding tiles cost
    // no stage)
    if ((long long)n_pairs * nt_max >= (1LL << 31)) return pfail(KVQ_ERR_UNSUPPORTED, "more than 2^31 tiles");
    kvq::DecodeArgs u{};
    u.batch = c->batch;
    u.h_kv = c->h_kv;
    u.gq = gq;
    u.d = d;
    u.G = G;
    u.log2G = a.log2G;
    u.Gv = Gv;
    u.log2Gv = a.log2Gv;
    u.R = a.R;
    u.scale_log2 = a.scale_log2;
    u.intz = a.intz;
    u.n_seg = 1;
    u.kr = a.kr;
    u.vr = a.vr;
    u.q = a.q;
    u.out = a.out;
    u.err = a.err;
    u.counters = a.counters;
    u.part = a.part;
    u.n_tiles = nt_max;
    u.n_splits = std::max(1, ws_splits);
    const long long T = (long long)n_pairs * nt_max;
    const int cap = std::max(ws_splits, 1);
    long long N = std::min<long long>(T, (long long)sms() * kvq::decode_tc_ctas_per_sm());
    N = std::min<long long>(N, kvq::kTcMaxCtas);
    N = std::min<long long>(N, std::max<long long>(n_pairs, (long long)n_pairs * (cap - 1)));
    const std::vector<long long> costs = paged_tc_costs(a, nt_max);
    while (true) {
      const int most = paged_tc_ranges(costs, c->batch, c->h_kv, nt_max, (int)N, u.tc_bound);
      u.tc_defer = most > 16;  // past 16 records a pair, a merge launch of its own
      if (most <= cap) {
        u.n_cta = (int)N;
        u.tc_whole = 0;
        break;
      }
      if (N <= n_pairs) {
        u.n_cta = n_pairs;  // one pair per CTA: no records
        u.tc_whole = 1;
        u.tc_defer = 0;
        break;
      }
      N = std::max<long long>(n_pairs, N - std::max<long long>(1, N / 32));
    }
    cudaError_t e = kvq::launch_decode_tc_paged(u, a, bits, form, s);
    if (e == cudaSuccess && u.tc_defer) e = kvq::launch_decode_tc_merge(u, n_pairs, s);
    return e == cudaSuccess ? KVQ_OK : pcuda(e, "paged decode launch");
  }
  // the general kernel: about four CTAs per SM over all tiles, each CTA a
  // contiguous range of one sequence's tiles
  const long long per_cta = std::max<long long>(4, (total + 4LL * sms() - 1) / (4LL * sms()));
  int cols = 0;
  for (int b = 0; b < c->batch; ++b) {
    kvq::PagedSeq& q = a.seq[b];
    const long long want = (nt[b] + per_cta - 1) / per_cta;
    q.n_split = (int)std::max<long long>(1, std::min<long long>({want, ws_splits, std::max(nt[b], 1)}));
    q.split0 = cols;
    cols += q.n_split;
  }
  a.n_cols = cols;
  const cudaError_t e = kvq::launch_decode_paged(a, s);
  return e == cudaSuccess ? KVQ_OK : pcuda(e, "paged decode launch");
}

}  // extern "C"
