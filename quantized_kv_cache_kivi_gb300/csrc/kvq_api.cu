// The C ABI of include/kvq.h: argument validation, planning of the launches
// (token runs, tiles, splits, append bookkeeping), and the launches.  All
// state lives in the caller's kvq_cache struct and device buffers.
#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "kvq_internal.h"

namespace {

thread_local std::string g_last_error;

kvq_status fail(kvq_status st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
kvq_status fail(kvq_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

kvq_status cuda_fail(cudaError_t e, const char* what) {
  return fail(KVQ_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// ---------------------------------------------------------------------------
// cache validation
// ---------------------------------------------------------------------------
// V quantization group in channels (group_v, or group when 0).
int group_v(const kvq_cache* c) { return c->group_v ? c->group_v : c->group; }

kvq_status validate_cache(const kvq_cache* c) {
  if (!c) return fail(KVQ_ERR_INVALID_ARG, "cache is NULL");
  if (c->batch < 1 || c->h_kv < 1 || c->h_q < 1)
    return fail(KVQ_ERR_INVALID_ARG, "batch, h_kv, h_q must be >= 1");
  if (c->h_q % c->h_kv != 0) return fail(KVQ_ERR_INVALID_ARG, "h_q must be a multiple of h_kv");
  if (c->h_q / c->h_kv > kvq::kMaxGq)
    return fail(KVQ_ERR_UNSUPPORTED, "more than %d query heads per kv head", kvq::kMaxGq);
  if (c->d_h != 64 && c->d_h != 128) return fail(KVQ_ERR_UNSUPPORTED, "d_h must be 64 or 128");
  const int G = c->group, Gv = group_v(c);
  if (G != 16 && G != 32 && G != 64 && G != 128 && G != 256)
    return fail(KVQ_ERR_UNSUPPORTED, "group must be 16, 32, 64, 128 or 256");
  if (Gv != 8 && Gv != 16 && Gv != 32 && Gv != 64 && Gv != 128)
    return fail(KVQ_ERR_UNSUPPORTED, "the V group (group_v, or group) must be 8 .. 128, a power of two");
  if (c->d_h % Gv != 0) return fail(KVQ_ERR_INVALID_ARG, "d_h must be a multiple of the V group");
  if (c->resid_cap < G || c->resid_cap % G != 0)
    return fail(KVQ_ERR_INVALID_ARG, "resid_cap must be a positive multiple of group");
  if (c->policy != KVQ_POLICY_KIVI && c->policy != KVQ_POLICY_FP16_TAIL)
    return fail(KVQ_ERR_INVALID_ARG, "unknown policy %d", c->policy);
  if (c->zero_point != KVQ_ZERO_MIN && c->zero_point != KVQ_ZERO_INT)
    return fail(KVQ_ERR_INVALID_ARG, "unknown zero_point %d", c->zero_point);
  if (!std::isfinite(c->sm_scale)) return fail(KVQ_ERR_INVALID_ARG, "sm_scale is not finite");
  if (c->n_seg < 1 || c->n_seg > KVQ_MAX_SEGMENTS)
    return fail(KVQ_ERR_INVALID_ARG, "n_seg must be in 1..%d", KVQ_MAX_SEGMENTS);
  if (!c->k_resid || !c->v_resid || !aligned16(c->k_resid) || !aligned16(c->v_resid))
    return fail(KVQ_ERR_INVALID_ARG, "residual rings must be non-NULL and 16-byte aligned");
  const int R = c->resid_cap;
  if (c->nkr < 0 || c->nkr > R || c->nvr < 0 || c->nvr > R)
    return fail(KVQ_ERR_INVALID_ARG, "nkr/nvr must be in 0..resid_cap");
  if (c->k_ring_start < 0 || c->k_ring_start >= R || c->v_ring_start < 0 || c->v_ring_start >= R)
    return fail(KVQ_ERR_INVALID_ARG, "ring starts must be in 0..resid_cap-1");
  long long lk = c->nkr, lv = c->nvr;
  for (int s = 0; s < c->n_seg; ++s) {
    const kvq_segment& g = c->seg[s];
    if (g.bits != 2 && g.bits != 4 && g.bits != 8)
      return fail(KVQ_ERR_UNSUPPORTED, "segment %d: bits must be 2, 4 or 8", s);
    if (g.capacity < 0 || g.capacity % G != 0)
      return fail(KVQ_ERR_INVALID_ARG, "segment %d: capacity must be a multiple of group", s);
    if (g.nk < 0 || g.nk > g.capacity || g.nv < 0 || g.nv > g.capacity || g.nk % G != 0)
      return fail(KVQ_ERR_INVALID_ARG, "segment %d: bad nk/nv", s);
    if (s + 1 < c->n_seg && g.nk != g.nv)
      return fail(KVQ_ERR_INVALID_ARG, "segment %d: only the last segment may have nk != nv", s);
    const void* p[6] = {g.k_codes, g.k_scale, g.k_zero, g.v_codes, g.v_scale, g.v_zero};
    for (int i = 0; i < 6; ++i)
      if (g.capacity > 0 && (!p[i] || !aligned16(p[i])))
        return fail(KVQ_ERR_INVALID_ARG, "segment %d: buffers must be non-NULL, 16-byte aligned", s);
    lk += g.nk;
    lv += g.nv;
  }
  if (lk != lv) return fail(KVQ_ERR_INVALID_ARG, "K and V describe %lld vs %lld tokens", lk, lv);
  if (lk > INT_MAX / 2) return fail(KVQ_ERR_INVALID_ARG, "too many tokens");
  return KVQ_OK;
}

kvq::SegDev seg_dev(const kvq_segment& g, int zero_point = KVQ_ZERO_MIN) {
  kvq::SegDev d;
  d.intz = zero_point == KVQ_ZERO_INT;
  d.kc = static_cast<const uint8_t*>(g.k_codes);
  d.ks = static_cast<const __half*>(g.k_scale);
  d.kz = static_cast<const __half*>(g.k_zero);
  d.vc = static_cast<const uint8_t*>(g.v_codes);
  d.vs = static_cast<const __half*>(g.v_scale);
  d.vz = static_cast<const __half*>(g.v_zero);
  d.bits = g.bits;
  d.cap = g.capacity;
  return d;
}

int sm_count() { return kvq::sm_count_cached(); }

// ---------------------------------------------------------------------------
// decode planning: runs of uniform (K source, V source), tiles, splits
// ---------------------------------------------------------------------------
struct Piece {
  int seg;  // -1 ring
  int u0;
  int len;
};

int tile_bytes(int tile, int kbits, int vbits, int d, int G, int Gv) {
  auto a16 = [](int x) { return (x + 15) & ~15; };
  int b = a16(tile * d * kbits / 8) + a16(tile * d * vbits / 8);
  if (kbits != 16) b += 2 * ((tile + G - 1) / G + 1) * d * 2;
  if (vbits != 16) b += 2 * a16(tile * (d / Gv) * 2);
  return b;
}

// Tile of the one-query-head kernel: nw consumer warps x wt tokens each,
// the largest that fits one stage and the scaled-query table.
// Among equal token counts, more warps (a smaller slice) wins.
void choose_tile_mha(int kbits, int vbits, int d, int G, int Gv, int* tile, int* wt) {
  *tile = *wt = 0;
  int best_nw = 0;
  for (int w = 32; w >= 8; w >>= 1) {
    for (int nw = kvq::kMhaConsumerWarps; nw >= 1; --nw) {
      const int t = w * nw;
      if (tile_bytes(t, kbits, vbits, d, G, Gv) > kvq::kMhaStageBytes) continue;
      if (kbits != 16 && (t + G - 1) / G + 1 > kvq::kMhaMaxGroups) continue;
      if (t > *tile || (t == *tile && nw > best_nw)) {
        *tile = t;
        *wt = w;
        best_nw = nw;
      }
      break;
    }
  }
}

// Tile of the tensor-core kernel: the most tokens (a multiple of the 32-token
// unit) that fit one stage and the K operand table.
void choose_tile_tc(int kbits, int vbits, int d, int G, int Gv, int* tile, int* wt) {
  *tile = *wt = 0;
  for (int t = 256; t >= 32; t -= 32) {
    if (tile_bytes(t, kbits, vbits, d, G, Gv) > kvq::kTcStageBytes) continue;
    if (kbits != 16 && (t + G - 1) / G + 1 > kvq::kTcMaxGroups) continue;
    *tile = t;
    *wt = 32;
    return;
  }
}

int choose_tile(int kbits, int vbits, int d, int G, int Gv, int gq) {
  for (int tile = 128; tile >= 32; tile >>= 1) {
    if (tile_bytes(tile, kbits, vbits, d, G, Gv) > kvq::kStageBytes) continue;
    if (kbits != 16 && ((tile + G - 1) / G + 1) * gq * d * 4 > kvq::kQsBytes) continue;
    return tile;
  }
  return 0;
}

enum Kernel { K_GENERAL = 0, K_MHA = 1, K_TC = 2 };

kvq_status plan_decode(const kvq_cache* c, kvq::DecodeArgs& a, std::vector<int>& tile_cost,
                       int kern) {
  std::vector<Piece> kp, vp;
  for (int s = 0; s < c->n_seg; ++s) {
    if (c->seg[s].nk > 0) kp.push_back({s, 0, c->seg[s].nk});
    if (c->seg[s].nv > 0) vp.push_back({s, 0, c->seg[s].nv});
  }
  if (c->nkr > 0) kp.push_back({-1, 0, c->nkr});
  if (c->nvr > 0) vp.push_back({-1, 0, c->nvr});
  const int gq = c->h_q / c->h_kv;
  a.n_runs = 0;
  a.n_tiles = 0;
  tile_cost.clear();
  size_t i = 0, j = 0;
  int oi = 0, oj = 0;  // offsets consumed inside kp[i], vp[j]
  while (i < kp.size() && j < vp.size()) {
    int len = std::min(kp[i].len - oi, vp[j].len - oj);
    // the tensor-core kernel applies one K group (G >= 32) per 32-token unit:
    // a packed-K run that starts off a multiple of 32 gets a short head run
    const int uk = kp[i].u0 + oi;
    if (kern == K_TC && kp[i].seg >= 0 && uk % 32 != 0) len = std::min(len, 32 - uk % 32);
    if (a.n_runs >= kvq::kMaxRuns) return fail(KVQ_ERR_UNSUPPORTED, "too many token runs");
    kvq::Run& r = a.runs[a.n_runs++];
    r.seg_k = kp[i].seg;
    r.seg_v = vp[j].seg;
    r.u0_k = kp[i].u0 + oi;
    r.u0_v = vp[j].u0 + oj;
    r.len = len;
    const int kb = r.seg_k >= 0 ? c->seg[r.seg_k].bits : 16;
    const int vb = r.seg_v >= 0 ? c->seg[r.seg_v].bits : 16;
    r.wt = 0;
    if (kern == K_TC) choose_tile_tc(kb, vb, c->d_h, c->group, group_v(c), &r.tile, &r.wt);
    else if (kern == K_MHA) choose_tile_mha(kb, vb, c->d_h, c->group, group_v(c), &r.tile, &r.wt);
    else r.tile = choose_tile(kb, vb, c->d_h, c->group, group_v(c), gq);
    if (r.tile == 0) return fail(KVQ_ERR_UNSUPPORTED, "no tile size fits shared memory");
    r.groups = (r.tile + c->group - 1) / c->group + 1;
    r.tile0 = a.n_tiles;
    const int nt = (len + r.tile - 1) / r.tile;
    for (int t = 0; t < nt; ++t) {
      const int n = std::min(r.tile, len - t * r.tile);
      // bytes streamed plus the CUDA-core work of the general kernel (every
      // token costs gq dot products over d channels whatever its width), in
      // byte equivalents: with several query heads the work dominates, and
      // splitting by bytes alone would give the 2-bit splits three times the
      // tokens of the 8-bit ones
      const int work = kern == K_GENERAL ? n * gq * c->d_h / 2 : 0;
      tile_cost.push_back(tile_bytes(n, kb, vb, c->d_h, c->group, group_v(c)) + work);
    }
    a.n_tiles += nt;
    oi += len;
    oj += len;
    if (oi == kp[i].len) { ++i; oi = 0; }
    if (oj == vp[j].len) { ++j; oj = 0; }
  }
  return KVQ_OK;
}

// Splits per (batch, kv head): minimise the load model
// ceil(pairs * s / slots) * (1/s + f), slots = SMs x the 2 CTAs an SM holds
// at once (both split-K kernels fit two), f = fixed cost of one CTA relative
// to a whole head's stream; ties go to fewer splits.
int choose_splits(int n_pairs, int n_tiles, int max_splits) {
  const int n_sm = 2 * sm_count();
  const int cap = std::min(std::min(max_splits, n_tiles), KVQ_MAX_SPLITS);
  const double f = 0.02;
  int best = 1;
  double best_t = 1e300;
  for (int s = 1; s <= cap; ++s) {
    const double rounds = std::ceil((double)n_pairs * s / n_sm);
    const double t = rounds * (1.0 / s + f);
    if (t < best_t * (1.0 - 1e-9)) {
      best_t = t;
      best = s;
    }
  }
  return best;
}

// Stream-K ranges of the tensor-core kernel.  Tile t of a pair costs its
// 32-token units plus a quarter unit of per-tile work, the same in every
// pair; CTA i's range starts at the first tile whose cost prefix reaches
// W(i) / W(N) of the total, kept non-empty, where CTA i weighs w1 if it is
// one of the first nf (the first wave, one per SM) and w2 otherwise (equal
// weights by default: first-wave weights of 8:7 gained 1-2% with one query
// head per kv head on some runs and lost 5% on others and with more heads).
// Returns the most ranges that meet one pair (its partial records).
int tc_ranges(const kvq::DecodeArgs& a, int n_pairs, int N, int* bound, int nf = 0, int w1 = 1, int w2 = 1) {
  const int nt = a.n_tiles;
  std::vector<long long> pre(nt + 1, 0);
  for (int r = 0, t = 0; t < nt; ++t) {  // tokens of tile t from the runs alone
    while (r + 1 < a.n_runs && a.runs[r + 1].tile0 <= t) ++r;
    const kvq::Run& run = a.runs[r];
    const int n = std::min(run.tile, run.len - (t - run.tile0) * run.tile);
    pre[t + 1] = pre[t] + 4 * ((n + 31) / 32) + 1;
  }
  const long long per_pair = pre[nt], T = (long long)n_pairs * nt;
  const long long total = per_pair * n_pairs;
  auto weight = [&](long long i) { return i <= nf ? w1 * i : w1 * (long long)nf + w2 * (i - nf); };
  const long long wn = weight(N);
  bound[0] = 0;
  for (int i = 1; i < N; ++i) {
    const long long target = total * weight(i) / wn;
    // first g with prefix(g) >= target, where prefix(g) = (g / nt) per_pair
    // + pre[g % nt]: every pair has the same prefix, so the pair is
    // target / per_pair and the tile the first one whose prefix reaches the
    // rest (tile costs are >= 1, so pre rises strictly)
    const long long p = target / per_pair, rest = target - p * per_pair;
    long long lo = p * nt;
    if (rest > 0) lo += std::lower_bound(pre.begin(), pre.end(), rest) - pre.begin();
    lo = std::max<long long>(lo, bound[i - 1] + 1);
    lo = std::min<long long>(lo, T - (N - i));
    bound[i] = (int)lo;
  }
  bound[N] = (int)T;
  // ranges meeting pair p: 1 + the range starts strictly inside it
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

// Persistent grid of the tensor-core kernel: as many CTAs as fit on the GPU
// at once (never more than tiles), fewer while some pair could be cut into
// more partial records than the workspace holds; one CTA per pair needs no
// records.  Up to kTcMaxPieces records per pair, the last CTA of the pair
// merges them (one warp); beyond, a launch of its own does.
constexpr int kTcMaxPieces = 16;

kvq_status tc_grid(kvq::DecodeArgs& a, int n_pairs, int records) {
  const long long T = (long long)n_pairs * a.n_tiles;
  const int cap = std::max(records, 1);
  long long N = std::min<long long>(T, (long long)sm_count() * kvq::decode_tc_ctas_per_sm());
  N = std::min<long long>(N, kvq::kTcMaxCtas);
  N = std::min<long long>(N, std::max<long long>(n_pairs, (long long)n_pairs * (cap - 1)));
  a.tc_defer = 0;
  while (true) {
    const int most = tc_ranges(a, n_pairs, (int)N, a.tc_bound);
    a.tc_defer = most > kTcMaxPieces;
    if (most <= cap) break;
    if (N <= n_pairs) {
      a.n_cta = n_pairs;  // one pair per CTA
      a.tc_whole = 1;
      a.tc_defer = 0;
      return KVQ_OK;
    }
    N = std::max<long long>(n_pairs, N - std::max<long long>(1, N / 32));
  }
  a.n_cta = (int)N;
  a.tc_whole = 0;
  return KVQ_OK;
}

// Walk every tile of the first and the last (batch, kv head) through the same
// geometry the kernel uses and check each bulk copy before anything launches:
// 16-byte alignment, source inside its buffer's documented extent, the stage
// and the scaled-query table large enough, and the copies adding up to the
// byte count the tile's mbarrier expects (so no wait can be left short).
kvq_status verify_decode_plan(const kvq_cache* c, const kvq::DecodeArgs& a, int n_pairs,
                              int kern) {
  const bool mha = kern != K_GENERAL;
  const uint32_t stage_cap = kern == K_TC    ? (uint32_t)kvq::kTcStageBytes
                             : kern == K_MHA ? (uint32_t)kvq::kMhaStageBytes
                                             : (uint32_t)kvq::kStageBytes;
  const int max_groups = kern == K_TC ? kvq::kTcMaxGroups : kvq::kMhaMaxGroups;
  const size_t P = (size_t)n_pairs, D = (size_t)a.d, G = (size_t)a.G, R = (size_t)a.R;
  // The bulk copies are walked for the first and last tile of every run:
  // a run's tiles in between have the first one's shape (their K groups
  // can differ in count, checked for every tile below) and their copies lie
  // between the two ends' addresses.
  std::vector<char> walk(a.n_tiles, 0);
  for (int i = 0; i < a.n_runs; ++i) {
    const int t0 = a.runs[i].tile0;
    const int t1 = (i + 1 < a.n_runs ? a.runs[i + 1].tile0 : a.n_tiles) - 1;
    if (t0 >= 0 && t0 < a.n_tiles) walk[t0] = 1;
    if (t1 >= 0 && t1 < a.n_tiles) walk[t1] = 1;
  }
  for (int which = 0; which < 2; ++which) {
    const size_t pair = which == 0 ? 0 : P - 1;
    for (int t = 0; t < a.n_tiles; ++t) {
      const kvq::TileInfo ti = kvq::tile_info(a, t);
      if (ti.n < 1 || ti.n > (mha ? 8 * 32 : 128))
        return fail(KVQ_ERR_UNSUPPORTED, "tile %d has %d tokens", t, ti.n);
      if (ti.bytes > stage_cap)
        return fail(KVQ_ERR_UNSUPPORTED, "tile %d needs %u stage bytes", t, ti.bytes);
      if (!mha && ti.kseg >= 0 && (size_t)ti.ng * a.gq * D * 4 > (size_t)kvq::kQsBytes)
        return fail(KVQ_ERR_UNSUPPORTED, "tile %d: scaled-query table too small", t);
      if (kern == K_TC && ti.kseg >= 0 && ti.ku0 % 32 != 0 && ti.ku0 / 32 != (ti.ku0 + ti.n - 1) / 32)
        return fail(KVQ_ERR_UNSUPPORTED, "tile %d: 32-token unit spans two K groups", t);
      if (mha && ti.kseg >= 0 && ti.ng > max_groups)
        return fail(KVQ_ERR_UNSUPPORTED, "tile %d: %d K groups > %d", t, ti.ng, max_groups);
      if (!walk[t]) continue;
      struct Copy {
        const void* src;
        uint32_t dst_off, bytes;
        int buf, seg;
      } cp[8];
      int n = 0;
      kvq::for_each_tile_copy(a, pair, ti, [&](const void* src, uint32_t off, uint32_t bytes,
                                               int buf, int seg) {
        if (n < 8) cp[n] = {src, off, bytes, buf, seg};
        ++n;
      });
      if (n > 8) return fail(KVQ_ERR_UNSUPPORTED, "tile %d: %d copies", t, n);
      uint64_t sum = 0;
      for (int i = 0; i < n; ++i) {
        const Copy& k = cp[i];
        const uint8_t* base;
        size_t size;
        if (k.buf >= 6) {
          base = static_cast<const uint8_t*>(k.buf == 6 ? c->k_resid : c->v_resid);
          size = P * R * D * 2;
        } else {
          const kvq_segment& g = c->seg[k.seg];
          const size_t cap = (size_t)g.capacity, rb = D * g.bits / 8;
          const void* ptrs[6] = {g.k_codes, g.k_scale, g.k_zero, g.v_codes, g.v_scale, g.v_zero};
          const size_t Dv = (size_t)(D / group_v(c));
          const size_t sizes[6] = {P * cap * rb, P * (cap / G) * D * 2, P * (cap / G) * D * 2,
                                   P * cap * rb, P * cap * Dv * 2, P * cap * Dv * 2};
          base = static_cast<const uint8_t*>(ptrs[k.buf]);
          size = sizes[k.buf];
        }
        const uint8_t* src = static_cast<const uint8_t*>(k.src);
        if (k.bytes == 0 || k.bytes % 16 || (uintptr_t)src % 16 || k.dst_off % 16)
          return fail(KVQ_ERR_INVALID_ARG, "tile %d copy %d: misaligned (%u bytes)", t, i, k.bytes);
        if (src < base || src + k.bytes > base + size)
          return fail(KVQ_ERR_INVALID_ARG, "tile %d copy %d: outside its buffer", t, i);
        if ((uint64_t)k.dst_off + k.bytes > ti.bytes)
          return fail(KVQ_ERR_INVALID_ARG, "tile %d copy %d: outside the stage", t, i);
        sum += k.bytes;
      }
      if (sum != ti.bytes)
        return fail(KVQ_ERR_INVALID_ARG, "tile %d: copies %llu != expected %u bytes", t,
                    (unsigned long long)sum, ti.bytes);
    }
  }
  return KVQ_OK;
}

size_t ws_fixed(int n_pairs) {
  return kvq::kWorkspaceHeader + (((size_t)n_pairs * 4 + 255) / 256) * 256;
}

// ---------------------------------------------------------------------------
// the warp kernel (one query head per kv head, one 2-bit segment, d_h 128)
// ---------------------------------------------------------------------------
constexpr bool kUseWarpKernel = true;
#ifndef KVQ_WARP_FILL
#define KVQ_WARP_FILL 1
#endif
constexpr bool kWarpFill = KVQ_WARP_FILL;  // pieces per pair that fill every warp slot


bool warp_kernel_applies(const kvq_cache* c) {
  const int Gv = group_v(c);
  return c->h_q == c->h_kv && c->n_seg == 1 && c->d_h == 128 && c->seg[0].bits == 2 && c->group >= 32 &&
         c->group % 32 == 0 && Gv >= 32 && 128 % Gv == 0 && c->seg[0].nk % 8 == 0 && c->seg[0].capacity % 32 == 0;
}

// Chunk counts and warps per pair of a cache's state: as many warps per
// pair as the GPU holds (kWarpWarps per SM), each piece at least the largest
// chunk's cost; fewer if the workspace cannot hold the pieces' records.
bool plan_warp(const kvq_cache* c, kvq::WarpArgs& a, size_t ws_bytes) {
  const int P = c->batch * c->h_kv;
  a.nk = c->seg[0].nk;
  a.nv = c->seg[0].nv;
  a.L = a.nk + c->nkr;
  a.npp = std::min(a.nk, a.nv);
  a.npx = std::max(a.nk, a.nv);
  a.n_pp = (a.npp + 31) / 32;
  a.n_x1 = a.npx > a.npp ? (a.npx - 1) / 8 - a.npp / 8 + 1 : 0;
  a.n_x2 = a.L > a.npx ? (a.L - 1) / 8 - a.npx / 8 + 1 : 0;
  a.C = a.n_pp + a.n_x1 + a.n_x2;
  a.Cp = (long long)kvq::kWarpWpp * a.n_pp + (long long)kvq::kWarpWx * (a.n_x1 + a.n_x2);
  a.P = P;
  const long long slots = (long long)sm_count() * kvq::kWarpWarps;
  const long long kcost = a.Cp / std::max(kvq::kWarpWpp, kvq::kWarpWx);  // every piece keeps a chunk
  const size_t room = ws_bytes > ws_fixed(P) ? ws_bytes - ws_fixed(P) : 0;
  const long long krec = (long long)(room / ((size_t)P * (128 + 2) * sizeof(float)));
  // Every slot of the GPU filled: P1 pairs get k pieces and the rest k - 1,
  // so that no SM holds a warp more than the others; else k pieces a pair.
  const long long k_hi = (slots + P - 1) / P;
  long long k, P1 = P;
  if (kWarpFill && k_hi >= 2 && k_hi <= kcost && k_hi <= krec) {
    k = k_hi;
    P1 = slots - (long long)P * (k_hi - 1);
  } else {
    k = std::min(std::min(slots / P, kcost), krec);
    if (k < 1) k = 1;  // one warp per pair writes its output directly: no records
  }
  if ((long long)P * k >= (1LL << 31)) return false;
  a.k = (int)k;
  a.P1 = (int)P1;
  return true;
}

// Every bulk copy of the chunks of the first and the last pair, walked
// against its buffer (in bounds, 16-byte aligned, inside the slot).  The
// full packed chunks' copies are a fixed size at addresses affine in the
// chunk index, so the first and the last of them bound the rest.
kvq_status verify_warp_plan(const kvq_cache* c, const kvq::WarpArgs& a) {
  const int P = a.P, G = c->group;
  const size_t rows = (size_t)P * a.cap;
  const uint8_t* base[8] = {a.kc, (const uint8_t*)a.ks, (const uint8_t*)a.kz, a.vc, (const uint8_t*)a.vs,
                            (const uint8_t*)a.vz, (const uint8_t*)a.kr, (const uint8_t*)a.vr};
  const size_t ext[8] = {rows * 32, (size_t)P * (a.cap / G) * 256, (size_t)P * (a.cap / G) * 256, rows * 32,
                         rows * a.ngv * 2, rows * a.ngv * 2, (size_t)P * a.R * 256, (size_t)P * a.R * 256};
  const long long pairs[2] = {0, P - 1};
  const int n_full = a.npp / 32;  // full packed chunks: copies affine in the chunk index
  for (long long pair : pairs) {
    for (int ci = 0; ci < a.C; ++ci) {
      if (ci > 0 && ci < n_full - 1) continue;  // between the first and the last full chunk
      const kvq::WarpChunk ch = kvq::warp_chunk(a, ci);
      if (ch.n < 1 || ch.n > (ch.pp ? 32 : 8) || ch.o0 < 0 || ch.o0 + ch.n > (ch.pp ? 32 : 8))
        return fail(KVQ_ERR_UNSUPPORTED, "warp plan: chunk %d has a bad token range", ci);
      bool ok = true;
      uint32_t total = 0;
      kvq::warp_chunk_copies(a, pair, ch, [&](const void* src, uint32_t dst, uint32_t n, int buf) {
        const uint8_t* p = static_cast<const uint8_t*>(src);
        total += n;
        if (n == 0 || n % 16 || (uintptr_t)p % 16 || dst % 16 || dst + n > (uint32_t)kvq::kWarpSlot ||
            p < base[buf] || p + n > base[buf] + ext[buf])
          ok = false;
      });
      if (!ok || total >= (1u << 20))
        return fail(KVQ_ERR_UNSUPPORTED, "warp plan: a copy of chunk %d leaves its buffer or the slot", ci);
    }
  }
  return KVQ_OK;
}

// ---------------------------------------------------------------------------
// append bookkeeping (KIVI Algorithm 1 over T pushed tokens)
// ---------------------------------------------------------------------------
kvq_status append_kivi(kvq_cache* c, const void* k_new, const void* v_new, int T,
                       cudaStream_t st, bool pdl = false) {
  const int R = c->resid_cap, G = c->group;
  kvq_segment& last = c->seg[c->n_seg - 1];
  kvq::AppendArgs a{};
  a.batch = c->batch;
  a.h_kv = c->h_kv;
  a.d = c->d_h;
  a.G = G;
  a.Gv = group_v(c);
  a.R = R;
  a.T = T;
  a.k_new = static_cast<const __half*>(k_new);
  a.v_new = static_cast<const __half*>(v_new);
  a.kr = static_cast<__half*>(c->k_resid);
  a.vr = static_cast<__half*>(c->v_resid);
  a.dst = seg_dev(last, c->zero_point);
  a.bits = last.bits;
  int fb = 0, evict = 0;
  bool flush_due = false;
  if (c->policy == KVQ_POLICY_KIVI) {
    // K: blocks of R pushed tokens are quantized; a block ending exactly at
    // the last token is left for kvq_flush_residual.
    const long long pushed = (long long)c->nkr + T;
    long long nb = pushed / R;
    if (nb >= 1 && pushed % R == 0) {
      flush_due = true;
      --nb;
    }
    fb = (int)nb;
    // V: everything but the newest R pushed tokens is quantized.
    evict = (int)std::max(0LL, (long long)c->nvr + T - R);
  } else {
    if (c->nkr + T > R || c->nvr + T > R)
      return fail(KVQ_ERR_CAPACITY, "fp16 ring full: %d + %d tokens > resid_cap %d",
                  std::max(c->nkr, c->nvr), T, R);
  }
  if ((long long)last.nk + (long long)fb * R > last.capacity ||
      (long long)last.nv + evict > last.capacity)
    return fail(KVQ_ERR_CAPACITY, "last segment full (capacity %d)", last.capacity);
  a.k_groups = fb * R / G;
  a.k_nk0 = last.nk;
  a.ksrc = {c->nkr, c->k_ring_start};
  a.k_ring_groups = std::min(a.k_groups, (c->nkr + G - 1) / G);
  a.v_evict = evict;
  a.v_nv0 = last.nv;
  a.vsrc = {c->nvr, c->v_ring_start};
  a.v_ring_tokens = std::min(evict, c->nvr);
  a.k_first_ring = std::max(0, fb * R - c->nkr);
  a.k_slot0 = c->k_ring_start + c->nkr;
  a.v_first_ring = std::max(0, evict - c->nvr);
  a.v_slot0 = c->v_ring_start + c->nvr;
  const int in_k = a.k_groups - a.k_ring_groups;
  const int in_v = a.v_evict - a.v_ring_tokens;
  // new-token work of a bulk append (a prompt) goes to grid-wide kernels;
  // chunk 0 of the append kernel keeps the ring work
  a.bulk = c->d_h == 128 && in_k + in_v > 0;  // V group 8..128 (validated)
  a.chunks = (!a.bulk && in_k + in_v > 0) ? 1 + std::min(256, in_k + (in_v + 63) / 64) : 1;
  if (a.chunks == 2 && a.k_ring_groups == 0 && a.v_ring_tokens == 0 && a.k_first_ring >= T &&
      a.v_first_ring >= T)
    a.chunks = 1;
  const cudaError_t e = kvq::launch_append(a, st, pdl);
  if (e != cudaSuccess) return cuda_fail(e, "append launch");
  // new lengths
  last.nk += fb * R;
  c->nkr = c->nkr + T - fb * R;
  last.nv += evict;
  c->v_ring_start = (c->v_ring_start + evict) % R;
  c->nvr = c->nvr + T - evict;
  return flush_due ? KVQ_FLUSH_DUE : KVQ_OK;
}

kvq_status append_plan(kvq_cache* c, const void* k_new, const void* v_new, int T,
                       const kvq_window_plan* p, cudaStream_t st) {
  const int R = c->resid_cap, G = c->group;
  if (c->policy != KVQ_POLICY_FP16_TAIL)
    return fail(KVQ_ERR_INVALID_ARG, "a window plan needs policy KVQ_POLICY_FP16_TAIL");
  if (p->window < G || p->window % G != 0)
    return fail(KVQ_ERR_INVALID_ARG, "window must be a positive multiple of group");
  if (p->n_windows < 0 || p->n_windows > kvq::kMaxWindowJobs)
    return fail(KVQ_ERR_UNSUPPORTED, "n_windows must be in 0..%d", kvq::kMaxWindowJobs);
  if ((long long)p->n_windows * p->window > T)
    return fail(KVQ_ERR_INVALID_ARG, "windows exceed the %d input tokens", T);
  if (p->n_windows > 0 && (!p->bits || !p->perm))
    return fail(KVQ_ERR_INVALID_ARG, "plan bits/perm are NULL");
  std::vector<char> seen(p->n_windows, 0);
  for (int i = 0; i < p->n_windows; ++i) {
    const int w = p->perm[i];
    if (w < 0 || w >= p->n_windows || seen[w]) return fail(KVQ_ERR_INVALID_ARG, "perm is not a permutation");
    seen[w] = 1;
    const int b = p->bits[w];
    if (b != 2 && b != 4 && b != 8 && b != 16) return fail(KVQ_ERR_INVALID_ARG, "window bits must be 2/4/8/16");
  }
  kvq::IngestArgs a{};
  a.batch = c->batch;
  a.h_kv = c->h_kv;
  a.d = c->d_h;
  a.G = G;
  a.Gv = group_v(c);
  a.R = R;
  a.T = T;
  a.S = p->window;
  a.k_new = static_cast<const __half*>(k_new);
  a.v_new = static_cast<const __half*>(v_new);
  a.kr = static_cast<__half*>(c->k_resid);
  a.vr = static_cast<__half*>(c->v_resid);
  for (int s = 0; s < c->n_seg; ++s) a.seg[s] = seg_dev(c->seg[s], c->zero_point);
  a.krs_push = c->k_ring_start + c->nkr;
  a.vrs_push = c->v_ring_start + c->nvr;
  std::vector<int> add(c->n_seg, 0);
  int ring = 0;
  a.n_jobs = p->n_windows;
  for (int i = 0; i < p->n_windows; ++i) {
    const int w = p->perm[i];
    kvq::WindowJob& job = a.jobs[i];
    job.src_token = w * p->window;
    if (p->bits[w] == 16) {
      job.seg = -1;
      job.dst = ring;
      ring += p->window;
      continue;
    }
    int s = 0;
    while (s < c->n_seg && c->seg[s].bits != p->bits[w]) ++s;
    if (s == c->n_seg) return fail(KVQ_ERR_INVALID_ARG, "no segment of width %d", (int)p->bits[w]);
    if (c->seg[s].nk != c->seg[s].nv)
      return fail(KVQ_ERR_INVALID_ARG, "segment %d has nk != nv", s);
    job.seg = s;
    job.dst = c->seg[s].nk + add[s];
    add[s] += p->window;
  }
  a.tail_src = p->n_windows * p->window;
  a.tail_len = T - a.tail_src;
  a.tail_dst = ring;
  ring += a.tail_len;
  for (int s = 0; s < c->n_seg; ++s)
    if ((long long)c->seg[s].nk + add[s] > c->seg[s].capacity)
      return fail(KVQ_ERR_CAPACITY, "segment %d full (capacity %d)", s, c->seg[s].capacity);
  if (c->nkr + ring > R || c->nvr + ring > R)
    return fail(KVQ_ERR_CAPACITY, "fp16 ring full: %d more tokens", ring);
  const cudaError_t e = kvq::launch_ingest(a, st);
  if (e != cudaSuccess) return cuda_fail(e, "ingest launch");
  for (int s = 0; s < c->n_seg; ++s) {
    c->seg[s].nk += add[s];
    c->seg[s].nv += add[s];
  }
  c->nkr += ring;
  c->nvr += ring;
  return KVQ_OK;
}

}  // namespace

namespace kvq {
int sm_count_cached() {
  static std::atomic<int> cache[64];  // 0 = not looked up yet
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (dev >= 0 && dev < 64 && (n = cache[dev].load(std::memory_order_relaxed)) > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}
void set_last_error(const char* msg) { g_last_error = msg; }
kvq_status check_cache(const kvq_cache* c) { return validate_cache(c); }
}  // namespace kvq

extern "C" {

const char* kvq_status_string(kvq_status s) {
  switch (s) {
    case KVQ_OK: return "ok";
    case KVQ_FLUSH_DUE: return "flush due: the K residual holds resid_cap tokens";
    case KVQ_ERR_INVALID_ARG: return "invalid argument";
    case KVQ_ERR_UNSUPPORTED: return "unsupported configuration";
    case KVQ_ERR_CAPACITY: return "capacity exceeded";
    case KVQ_ERR_CUDA: return "CUDA error";
    case KVQ_ERR_WORKSPACE: return "workspace missing or too small";
  }
  return "unknown status";
}

const char* kvq_last_error_string(void) { return g_last_error.c_str(); }

kvq_status kvq_quantize_append(kvq_cache* cache, const void* k_new, const void* v_new, int32_t T,
                               const kvq_window_plan* plan, void* stream) {
  kvq_status st = validate_cache(cache);
  if (st != KVQ_OK) return st;
  if (T < 0) return fail(KVQ_ERR_INVALID_ARG, "T must be >= 0");
  if (T == 0) return KVQ_OK;
  if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new))
    return fail(KVQ_ERR_INVALID_ARG, "k_new/v_new must be non-NULL and 16-byte aligned");
  if (plan) return append_plan(cache, k_new, v_new, T, plan, as_stream(stream));
  return append_kivi(cache, k_new, v_new, T, as_stream(stream));
}

namespace {
kvq_status flush_impl(kvq_cache* cache, cudaStream_t stream, bool pdl, const void* k_new = nullptr);
kvq_status decode_attention_impl(const kvq_cache* cache, const void* q, void* out, void* ws, size_t ws_bytes,
                                 cudaStream_t s, bool pdl, int dep_t0 = 0);
void flush_bookkeeping(kvq_cache* cache, int n);
}  // namespace

kvq_status kvq_flush_residual(kvq_cache* cache, void* stream) {
  kvq_status st = validate_cache(cache);
  if (st != KVQ_OK) return st;
  return flush_impl(cache, as_stream(stream), false);
}

kvq_status kvq_decode_attention(const kvq_cache* cache, const void* q, void* out, void* ws, size_t ws_bytes,
                                void* stream) {
  kvq_status st = validate_cache(cache);
  if (st != KVQ_OK) return st;
  return decode_attention_impl(cache, q, out, ws, ws_bytes, as_stream(stream), false);
}

kvq_status kvq_decode_step(kvq_cache* cache, const void* k_new, const void* v_new, const void* q, void* out,
                           void* ws, size_t ws_bytes, int32_t order, void* stream) {
  kvq_status st = validate_cache(cache);
  if (st != KVQ_OK) return st;
  if (order != KVQ_STEP_ATTEND_FIRST && order != KVQ_STEP_FLUSH_FIRST)
    return fail(KVQ_ERR_INVALID_ARG, "unknown step order %d", (int)order);
  if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new))
    return fail(KVQ_ERR_INVALID_ARG, "k_new/v_new must be non-NULL and 16-byte aligned");
  if (!q || !out || !aligned16(q) || !aligned16(out))
    return fail(KVQ_ERR_INVALID_ARG, "q/out must be non-NULL and 16-byte aligned");
  const int n_pairs = cache->batch * cache->h_kv;
  if (!ws || !aligned16(ws) || ws_bytes < ws_fixed(n_pairs))
    return fail(KVQ_ERR_WORKSPACE, "workspace needs at least %zu bytes", ws_fixed(n_pairs));
  cudaStream_t s = as_stream(stream);
  const kvq_cache before = *cache;
  const kvq_status ap = append_kivi(cache, k_new, v_new, 1, s, true);
  if (ap < 0) return ap;
  // The flush takes the step's new token from k_new rather than from the
  // ring slot the append writes, so it may start before the append ends.
  const bool flush_first = order == KVQ_STEP_FLUSH_FIRST;
  if (flush_first && ap == KVQ_FLUSH_DUE) {
    st = flush_impl(cache, s, true, k_new);
    if (st != KVQ_OK) {
      *cache = before;
      return st;
    }
  }
  // first token position whose K or V the append (or the flush) wrote: the
  // new token, and the rows they quantized (one segment; else every chunk
  // waits)
  int dep_t0 = 0;
  if (cache->n_seg == 1) {
    long long d = (long long)cache->seg[0].nk + cache->nkr - 1;
    if (cache->seg[0].nk != before.seg[0].nk) d = std::min<long long>(d, before.seg[0].nk);
    if (cache->seg[0].nv != before.seg[0].nv) d = std::min<long long>(d, before.seg[0].nv);
    dep_t0 = (int)std::max(0LL, d);
  }
  // The attention starts beside the append (or the flush) only when that
  // grid is small: the append's blocks hold shared memory the attention's
  // warps need, and with many pairs (more than two append blocks per SM)
  // the attention's pieces would start staggered behind them (measured on
  // 2048 pairs: 416 against 381 us per step).
  const bool pdl_attn = (long long)n_pairs <= 2LL * sm_count();
  st = decode_attention_impl(cache, q, out, ws, ws_bytes, s, pdl_attn, pdl_attn ? dep_t0 : 0);
  if (st != KVQ_OK) {
    *cache = before;  // nothing of the step counts: the caller may retry it
    return st;
  }
  if (!flush_first && ap == KVQ_FLUSH_DUE) return flush_impl(cache, s, true, k_new);
  return KVQ_OK;
}

kvq_status kvq_decode_step_host(kvq_cache* cache, const void* host_in, void* host_out, void* dev_in,
                                void* dev_out, void* ws, size_t ws_bytes, int32_t order, void* stream) {
  kvq_status st = validate_cache(cache);
  if (st != KVQ_OK) return st;
  if (!host_in || !host_out || !dev_in || !dev_out)
    return fail(KVQ_ERR_INVALID_ARG, "host_in, host_out, dev_in and dev_out must be non-NULL");
  if (!aligned16(dev_in) || !aligned16(dev_out))
    return fail(KVQ_ERR_INVALID_ARG, "dev_in/dev_out must be 16-byte aligned");
  const size_t kv = (size_t)cache->batch * cache->h_kv * cache->d_h * sizeof(__half);  // new K (= new V)
  const size_t qb = (size_t)cache->batch * cache->h_q * cache->d_h * sizeof(__half);
  cudaStream_t s = as_stream(stream);
  cudaError_t e = cudaMemcpyAsync(dev_in, host_in, 2 * kv + qb, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_fail(e, "input copy");
  uint8_t* d = static_cast<uint8_t*>(dev_in);
  st = kvq_decode_step(cache, d, d + kv, d + 2 * kv, dev_out, ws, ws_bytes, order, stream);
  if (st < 0) return st;
  e = cudaMemcpyAsync(host_out, dev_out, qb, cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return cuda_fail(e, "output copy");
  return st;
}

namespace {
// k_new (a decode step's new tokens, [batch][h_kv][1][d_h]): the newest ring
// token is read from there instead of its ring slot.
kvq_status flush_impl(kvq_cache* cache, cudaStream_t stream, bool pdl, const void* k_new) {
  const int G = cache->group, R = cache->resid_cap;
  const int n = (cache->nkr / G) * G;
  if (n == 0) return KVQ_OK;
  kvq_segment& last = cache->seg[cache->n_seg - 1];
  if ((long long)last.nk + n > last.capacity)
    return fail(KVQ_ERR_CAPACITY, "last segment full (capacity %d)", last.capacity);
  kvq::AppendArgs a{};
  a.batch = cache->batch;
  a.h_kv = cache->h_kv;
  a.d = cache->d_h;
  a.G = G;
  a.Gv = group_v(cache);
  a.R = R;
  a.kr = static_cast<__half*>(cache->k_resid);
  a.dst = seg_dev(last, cache->zero_point);
  a.bits = last.bits;
  a.k_groups = n / G;
  a.k_nk0 = last.nk;
  a.ksrc = {INT_MAX, cache->k_ring_start};
  if (k_new && cache->nkr >= 1 && cache->nkr - 1 < n) {  // the newest token is among those flushed
    a.k_new = static_cast<const __half*>(k_new);
    a.T = 1;
    a.ksrc.n_old = cache->nkr - 1;
  }
  const cudaError_t e = kvq::launch_flush(a, stream, pdl);
  if (e != cudaSuccess) return cuda_fail(e, "flush launch");
  flush_bookkeeping(cache, n);
  return KVQ_OK;
}

// n oldest K ring tokens now packed at the end of the last segment
void flush_bookkeeping(kvq_cache* cache, int n) {
  cache->seg[cache->n_seg - 1].nk += n;
  cache->nkr -= n;
  cache->k_ring_start = (cache->k_ring_start + n) % cache->resid_cap;
}

}  // namespace

size_t kvq_workspace_bytes(const kvq_cache* cache, int32_t max_splits) {
  if (!cache || cache->batch < 1 || cache->h_kv < 1 || cache->h_q < cache->h_kv) return 0;
  if (max_splits < 1) max_splits = 1;
  if (max_splits > KVQ_MAX_SPLITS) max_splits = KVQ_MAX_SPLITS;
  const int n_pairs = cache->batch * cache->h_kv;
  const int gq = cache->h_q / cache->h_kv;
  size_t b = ws_fixed(n_pairs);
  if (max_splits > 1) b += (size_t)n_pairs * max_splits * gq * (cache->d_h + 2) * sizeof(float);
  return b;
}

kvq_status kvq_workspace_init(void* ws, size_t bytes, void* stream) {
  if (!ws || bytes == 0) return fail(KVQ_ERR_INVALID_ARG, "workspace is NULL/empty");
  const cudaError_t e = cudaMemsetAsync(ws, 0, bytes, as_stream(stream));
  return e == cudaSuccess ? KVQ_OK : cuda_fail(e, "workspace memset");
}

kvq_status kvq_workspace_error(const void* ws, int32_t* err_out, void* stream) {
  if (!ws || !err_out) return fail(KVQ_ERR_INVALID_ARG, "NULL argument");
  cudaError_t e = cudaMemcpyAsync(err_out, ws, sizeof(int32_t), cudaMemcpyDeviceToHost, as_stream(stream));
  if (e == cudaSuccess) e = cudaStreamSynchronize(as_stream(stream));
  return e == cudaSuccess ? KVQ_OK : cuda_fail(e, "reading the workspace error word");
}

namespace {
kvq_status decode_attention_impl(const kvq_cache* cache, const void* q, void* out, void* ws, size_t ws_bytes,
                                 cudaStream_t stream, bool pdl, int dep_t0) {
  kvq_status st = KVQ_OK;
  if (!q || !out || !aligned16(q) || !aligned16(out))
    return fail(KVQ_ERR_INVALID_ARG, "q/out must be non-NULL and 16-byte aligned");
  const int n_pairs = cache->batch * cache->h_kv;
  if (!ws || !aligned16(ws) || ws_bytes < ws_fixed(n_pairs))
    return fail(KVQ_ERR_WORKSPACE, "workspace needs at least %zu bytes", ws_fixed(n_pairs));
  cudaStream_t s = stream;
  const int gq = cache->h_q / cache->h_kv;
  if (kUseWarpKernel && warp_kernel_applies(cache) && cache->seg[0].nk + cache->nkr > 0) {
    kvq::WarpArgs w{};
    w.cap = cache->seg[0].capacity;
    w.R = cache->resid_cap;
    w.krs = cache->k_ring_start;
    w.vrs = cache->v_ring_start;
    w.log2G = 0;
    while ((1 << w.log2G) < cache->group) ++w.log2G;
    w.ngv = cache->d_h / group_v(cache);
    w.intz = cache->zero_point == KVQ_ZERO_INT;
    w.scale_log2 = cache->sm_scale * 1.4426950408889634f;
    const kvq_segment& sg = cache->seg[0];
    w.kc = static_cast<const uint8_t*>(sg.k_codes);
    w.ks = static_cast<const __half*>(sg.k_scale);
    w.kz = static_cast<const __half*>(sg.k_zero);
    w.vc = static_cast<const uint8_t*>(sg.v_codes);
    w.vs = static_cast<const __half*>(sg.v_scale);
    w.vz = static_cast<const __half*>(sg.v_zero);
    w.kr = static_cast<const __half*>(cache->k_resid);
    w.vr = static_cast<const __half*>(cache->v_resid);
    w.q = static_cast<const __half*>(q);
    w.out = static_cast<__half*>(out);
    if (plan_warp(cache, w, ws_bytes)) {
      uint8_t* wb = static_cast<uint8_t*>(ws);
      w.err = reinterpret_cast<int*>(wb);
      w.counters = reinterpret_cast<int*>(wb + kvq::kWorkspaceHeader);
      w.part = reinterpret_cast<float*>(wb + ws_fixed(n_pairs));
      st = verify_warp_plan(cache, w);
      if (st != KVQ_OK) return st;
      // the first chunk that ends past dep_t0 (chunks run in token order)
      int dc = 0;
      if (dep_t0 > 0) {
        if (dep_t0 < w.npp) {
          dc = dep_t0 / 32;
        } else {
          dc = w.n_pp;
          while (dc < w.C) {
            const kvq::WarpChunk ch = kvq::warp_chunk(w, dc);
            if (ch.t0 + ch.n > dep_t0) break;
            ++dc;
          }
        }
      }
      w.dep_c = dc;
      const cudaError_t e = kvq::launch_decode_warp(w, s, pdl);
      return e == cudaSuccess ? KVQ_OK : cuda_fail(e, "decode launch");
    }
  }
  kvq::DecodeArgs a{};
  std::vector<int> cost;
  // one query head per kv head, one segment, each lane's channel quarter
  // inside one V group: the specialised kernel
  int kern = K_GENERAL, form = 0;
  const int Gk = cache->group, Gv = group_v(cache);
  if (gq == 1 && cache->n_seg == 1 && Gv >= cache->d_h / 4 && (cache->d_h != 128 || Gk >= 32)) {
    kern = cache->d_h == 128 ? K_TC : K_MHA;
    form = 1;
  } else if (gq >= 2 && gq <= 4 && cache->n_seg == 1 && cache->d_h == 128 && Gk >= 32 && Gv >= 64) {
    // 2-4 query heads per kv head, at most two V groups per token: the
    // tensor-core kernel's four-head form
    kern = K_TC;
    form = 4;
  } else if (gq <= kvq::kMaxGq && cache->d_h == 128 && Gk >= 32 && Gv >= 16) {
    // up to 8 query heads, any segments: the eight-head form, if every tile
    // is K and V packed at one width, packed K with ring V, or ring only
    kern = K_TC;
    form = 8;
  }
  st = plan_decode(cache, a, cost, kern);
  if (st != KVQ_OK) return st;
  if (form == 8) {
    bool ok = true;
    for (int i = 0; i < a.n_runs; ++i) {
      const kvq::Run& r = a.runs[i];
      if (r.seg_k < 0 ? r.seg_v >= 0
                      : r.seg_v >= 0 && cache->seg[r.seg_k].bits != cache->seg[r.seg_v].bits)
        ok = false;
    }
    if (!ok) {
      kern = K_GENERAL;
      form = 0;
      st = plan_decode(cache, a, cost, kern);
      if (st != KVQ_OK) return st;
    }
  }
  if (a.n_tiles == 0) {
    const size_t bytes = (size_t)cache->batch * cache->h_q * cache->d_h * 2;
    const cudaError_t e = cudaMemsetAsync(out, 0, bytes, s);
    return e == cudaSuccess ? KVQ_OK : cuda_fail(e, "zero output");
  }
  const size_t per_split = (size_t)n_pairs * gq * (cache->d_h + 2) * sizeof(float);
  const int ws_splits = (int)std::min<size_t>(KVQ_MAX_SPLITS, (ws_bytes - ws_fixed(n_pairs)) / per_split);
  if (kern == K_TC) {
    if ((long long)n_pairs * a.n_tiles >= (1LL << 31))
      return fail(KVQ_ERR_UNSUPPORTED, "more than 2^31 tiles");
    // stream-K: a.n_splits is the record stride per pair
    a.n_splits = std::max(1, ws_splits);
    st = tc_grid(a, n_pairs, ws_splits);
    if (st != KVQ_OK) return st;
  }
  const int S = kern == K_TC ? 1 : choose_splits(n_pairs, a.n_tiles, std::max(1, ws_splits));
  // split boundaries with equal byte cost: split k ends at the first tile
  // whose cost midpoint passes k/S of the head's bytes
  std::vector<long long> prefix(a.n_tiles + 1, 0);
  for (int t = 0; t < a.n_tiles; ++t) prefix[t + 1] = prefix[t] + cost[t];
  const long long total = prefix[a.n_tiles];
  if (kern != K_TC) a.n_splits = S;
  a.split_tile[0] = 0;
  for (int k = 1; k < S; ++k) {
    const long long target = total * k / S;
    int t = a.split_tile[k - 1] + 1;
    while (t < a.n_tiles && 2 * prefix[t] + cost[t] <= 2 * target) ++t;
    a.split_tile[k] = std::min(t, a.n_tiles - (S - k));
  }
  a.split_tile[S] = a.n_tiles;
  for (int k = 1; k <= S; ++k)
    if (a.split_tile[k] <= a.split_tile[k - 1])
      return fail(KVQ_ERR_UNSUPPORTED, "split planning failed");
  a.batch = cache->batch;
  a.h_kv = cache->h_kv;
  a.gq = gq;
  a.d = cache->d_h;
  a.G = cache->group;
  a.log2G = 0;
  while ((1 << a.log2G) < a.G) ++a.log2G;
  a.Gv = group_v(cache);
  a.log2Gv = 0;
  while ((1 << a.log2Gv) < a.Gv) ++a.log2Gv;
  a.R = cache->resid_cap;
  a.scale_log2 = cache->sm_scale * 1.4426950408889634f;
  a.intz = cache->zero_point == KVQ_ZERO_INT;
  a.n_seg = cache->n_seg;
  for (int i = 0; i < cache->n_seg; ++i) a.seg[i] = seg_dev(cache->seg[i], cache->zero_point);
  a.kr = static_cast<const __half*>(cache->k_resid);
  a.vr = static_cast<const __half*>(cache->v_resid);
  a.krs = cache->k_ring_start;
  a.vrs = cache->v_ring_start;
  a.q = static_cast<const __half*>(q);
  a.out = static_cast<__half*>(out);
  uint8_t* w = static_cast<uint8_t*>(ws);
  a.err = reinterpret_cast<int*>(w);
  a.counters = reinterpret_cast<int*>(w + kvq::kWorkspaceHeader);
  a.part = reinterpret_cast<float*>(w + ws_fixed(n_pairs));
  st = verify_decode_plan(cache, a, n_pairs, kern);
  if (st != KVQ_OK) return st;
  cudaError_t e = kern == K_TC    ? kvq::launch_decode_tc(a, cache->seg[0].bits, form, s)
                  : kern == K_MHA ? kvq::launch_decode_mha(a, n_pairs, cache->seg[0].bits, s)
                                  : kvq::launch_decode(a, n_pairs, s);
  if (e == cudaSuccess && kern == K_TC && a.tc_defer) e = kvq::launch_decode_tc_merge(a, n_pairs, s);
  return e == cudaSuccess ? KVQ_OK : cuda_fail(e, "decode launch");
}

}  // namespace

size_t kvq_window_assign_workspace_bytes(int32_t batch, int32_t h_kv, int32_t d_h, int32_t M,
                                         int32_t S) {
  if (batch < 1 || h_kv < 1 || d_h < 1 || S < 1 || M < S) return 0;
  const size_t nw = (size_t)M / S;
  auto a256 = [](size_t x) { return (x + 255) / 256 * 256; };
  return a256((size_t)batch * h_kv * d_h * 8) + a256((size_t)batch * nw * 16) + a256(nw * 8) +
         a256(nw) + a256(nw * 4);
}

kvq_status kvq_window_assign(const void* keys, const void* text_keys, int32_t batch, int32_t h_kv,
                             int32_t d_h, int32_t M, int32_t S, int32_t N, float frac8,
                             float frac4, int32_t first_window_fp16, void* ws, size_t ws_bytes,
                             int8_t* bits_out, int32_t* perm_out, double* sim_out, void* stream) {
  if (!keys || !text_keys || !bits_out || !perm_out)
    return fail(KVQ_ERR_INVALID_ARG, "NULL argument");
  if (batch < 1 || h_kv < 1 || d_h < 1 || S < 1 || M < S || N < 1)
    return fail(KVQ_ERR_INVALID_ARG, "bad sizes");
  if (!(frac8 >= 0.f && frac4 >= 0.f && frac8 + frac4 <= 1.f))
    return fail(KVQ_ERR_INVALID_ARG, "fractions must be >= 0 and sum to <= 1");
  const size_t need = kvq_window_assign_workspace_bytes(batch, h_kv, d_h, M, S);
  if (!ws || !aligned16(ws) || ws_bytes < need)
    return fail(KVQ_ERR_WORKSPACE, "window workspace needs %zu bytes", need);
  const int nw = M / S;
  const int ranked = nw - (first_window_fp16 ? 1 : 0);
  int n8 = (int)std::floor((double)frac8 * ranked);
  int n4 = (int)std::floor((double)frac4 * ranked);
  n8 = std::min(n8, ranked);
  n4 = std::min(n4, ranked - n8);
  auto a256 = [](size_t x) { return (x + 255) / 256 * 256; };
  uint8_t* w = static_cast<uint8_t*>(ws);
  kvq::WindowArgs a{};
  a.keys = static_cast<const __half*>(keys);
  a.text = static_cast<const __half*>(text_keys);
  a.batch = batch;
  a.h_kv = h_kv;
  a.d = d_h;
  a.M = M;
  a.S = S;
  a.N = N;
  a.n8 = n8;
  a.n4 = n4;
  a.first_fp16 = first_window_fp16 ? 1 : 0;
  size_t off = 0;
  a.tsum = reinterpret_cast<double*>(w + off);
  off += a256((size_t)batch * h_kv * d_h * 8);
  a.wstat = reinterpret_cast<double*>(w + off);
  off += a256((size_t)batch * nw * 16);
  a.sim = reinterpret_cast<double*>(w + off);
  off += a256((size_t)nw * 8);
  a.bits = reinterpret_cast<int8_t*>(w + off);
  off += a256((size_t)nw);
  a.perm = reinterpret_cast<int32_t*>(w + off);
  cudaStream_t s = as_stream(stream);
  cudaError_t e = kvq::launch_window_assign(a, s);
  if (e != cudaSuccess) return cuda_fail(e, "window assign launch");
  e = cudaMemcpyAsync(bits_out, a.bits, nw, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(perm_out, a.perm, (size_t)nw * 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess && sim_out)
    e = cudaMemcpyAsync(sim_out, a.sim, (size_t)nw * 8, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return e == cudaSuccess ? KVQ_OK : cuda_fail(e, "window assign copy-back");
}

static int eq8_chunks(int batch, int M, int S, int N) {
  const int nw = M / S;
  const int maxlen = std::max(S, N);
  int z = std::max(1, (2 * sm_count() + batch * (nw + 1) - 1) / (batch * (nw + 1)));
  z = std::max(z, (maxlen + 4095) / 4096);  // shared inverse norms of a chunk: at most 32 KB
  return std::min(z, maxlen);
}

size_t kvq_window_assign_eq8_workspace_bytes(int32_t batch, int32_t dim, int32_t M, int32_t S, int32_t N) {
  if (batch < 1 || dim < 1 || S < 1 || M < S || N < 1) return 0;
  const size_t nw = (size_t)M / S;
  const size_t z = (size_t)eq8_chunks(batch, M, S, N);
  auto a256 = [](size_t x) { return (x + 255) / 256 * 256; };
  return a256((size_t)batch * (nw + 1) * z * dim * 8) + a256((size_t)batch * nw * 8) + a256(nw) + a256(nw * 4);
}

kvq_status kvq_window_assign_eq8(const void* vision, const void* text, int32_t batch, int32_t dim, int32_t M,
                                 int32_t S, int32_t N, double layer_sim, double alpha, int32_t first_window_fp16,
                                 void* ws, size_t ws_bytes, int8_t* bits_out, int32_t* perm_out, double* sim_out,
                                 void* stream) {
  if (!vision || !text || !bits_out || !perm_out) return fail(KVQ_ERR_INVALID_ARG, "NULL argument");
  if (batch < 1 || dim < 1 || S < 1 || M < S || N < 1) return fail(KVQ_ERR_INVALID_ARG, "bad sizes");
  if (dim % 8 != 0 || !aligned16(vision) || !aligned16(text))
    return fail(KVQ_ERR_INVALID_ARG, "dim must be a multiple of 8 and the inputs 16-byte aligned");
  if (!(alpha != 0.0 && std::isfinite(alpha) && std::isfinite(layer_sim)))
    return fail(KVQ_ERR_INVALID_ARG, "alpha must be finite and nonzero, layer_sim finite");
  const size_t need = kvq_window_assign_eq8_workspace_bytes(batch, dim, M, S, N);
  if (!ws || !aligned16(ws) || ws_bytes < need)
    return fail(KVQ_ERR_WORKSPACE, "window workspace needs %zu bytes", need);
  const int nw = M / S;
  kvq::Eq8Args a{};
  a.vision = static_cast<const __half*>(vision);
  a.text = static_cast<const __half*>(text);
  a.batch = batch;
  a.dim = dim;
  a.M = M;
  a.S = S;
  a.N = N;
  a.chunks = eq8_chunks(batch, M, S, N);
  // Eq.10 and Eq.11
  a.t_low = std::expm1(alpha * layer_sim) / std::expm1(alpha);
  a.t_high = std::expm1(-alpha * layer_sim) / std::expm1(-alpha);
  a.first_fp16 = first_window_fp16 ? 1 : 0;
  auto a256 = [](size_t x) { return (x + 255) / 256 * 256; };
  uint8_t* w = static_cast<uint8_t*>(ws);
  size_t off = 0;
  a.part = reinterpret_cast<double*>(w + off);
  off += a256((size_t)batch * (nw + 1) * a.chunks * dim * 8);
  a.sims = reinterpret_cast<double*>(w + off);
  off += a256((size_t)batch * nw * 8);
  a.bits = reinterpret_cast<int8_t*>(w + off);
  off += a256((size_t)nw);
  a.perm = reinterpret_cast<int32_t*>(w + off);
  cudaStream_t s = as_stream(stream);
  cudaError_t e = kvq::launch_window_assign_eq8(a, s);
  if (e != cudaSuccess) return cuda_fail(e, "window assign launch");
  e = cudaMemcpyAsync(bits_out, a.bits, nw, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(perm_out, a.perm, (size_t)nw * 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess && sim_out)
    e = cudaMemcpyAsync(sim_out, a.sims, (size_t)batch * nw * 8, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return e == cudaSuccess ? KVQ_OK : cuda_fail(e, "window assign copy-back");
}

}  // extern "C"
