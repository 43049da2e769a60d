// Internal launch descriptors shared by the host planner (kvq_api.cu) and the
// kernels.  Everything is passed to kernels by value; nothing here allocates.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <map>
#include <mutex>
#include <utility>

#include "../../include/kvq.h"

namespace kvq {

constexpr int kMaxRuns = 20;        // token runs of uniform (K source, V source)
constexpr int kTcMaxCtas = 512;      // tensor-core kernel: CTAs of the persistent grid, at most
constexpr int kMaxGq = 8;           // query heads per kv head handled by one CTA
constexpr int kDecodeThreads = 256; // threads of a decode CTA
constexpr int kStageBytes = 20480;  // one pipeline stage of staged tile data
constexpr int kStages = 3;          // pipeline depth
constexpr int kQsBytes = 16384;     // per-tile scaled-query table (K groups)
constexpr int kWorkspaceHeader = 256;  // error word + padding at workspace start
// one-query-head (MHA) kernel: 7 consumer warps + 1 producer warp (2 CTAs and
// 16 warps per SM, so each thread may hold 128 registers)
constexpr int kMhaConsumerWarps = 7;
constexpr int kMhaStageBytes = 25600;   // staged tile data per pipeline stage
constexpr int kMhaMaxGroups = 16;       // K scale groups one tile may touch
constexpr int kMhaQtabBytes = kMhaMaxGroups * 4 * 36 * 4;  // scaled-query rows per stage
// tensor-core kernel (d_h = 128, one query head or 2-4 per kv head): a
// bulk-copy warp and 6-7 consumer warps, 4 stages, two CTAs per SM
constexpr int kTcStages = 4;
constexpr int kTcCtasPerSm = 2;
constexpr int kTcStageBytes = 19456;
constexpr int kTcMaxGroups = 8;                      // K groups one tile may touch

// One packed segment as the kernels see it (base pointers of the whole array).
struct SegDev {
  const uint8_t* kc;
  const __half* ks;
  const __half* kz;
  const uint8_t* vc;
  const __half* vs;
  const __half* vz;
  int bits;
  int cap;
  int intz;  // quantize with the integer zero point (WindowQuant Eq.14-16)
};

// A run of consecutive attention positions whose K comes from one source and
// whose V comes from one source.  seg_* = segment index, or -1 for the ring.
// u0_* = first packed row (segment source) or first ring index (ring source).
struct Run {
  int seg_k, seg_v;
  int u0_k, u0_v;
  int len;    // tokens in the run
  int tile;   // tokens per tile
  int tile0;  // index of the run's first tile among the head's tiles
  int groups; // max K scale groups one tile of this run touches (packed K)
  int wt;     // tokens per consumer-warp slice (one-query-head kernel)
};

struct DecodeArgs {
  int batch, h_kv, gq, d, G, R;
  int log2G;         // G is a power of two
  int Gv, log2Gv;    // V channel group and its log2
  float scale_log2;  // sm_scale * log2(e)
  int intz;          // zero slots hold integer zero points (x' = s (code - z))
  int n_seg;
  SegDev seg[KVQ_MAX_SEGMENTS];
  const __half* kr;
  const __half* vr;
  int krs, vrs;
  int n_runs;
  Run runs[kMaxRuns];
  int n_tiles;   // tiles per (batch, kv head)
  int n_splits;  // CTAs per (batch, kv head); tensor-core kernel: records per pair
  int n_cta;     // tensor-core kernel: CTAs of the persistent grid
  int split_tile[KVQ_MAX_SPLITS + 1];
  int tc_whole;                  // tensor-core kernel: 1 = CTA i takes pair i (tc_bound unused)
  int tc_defer;                  // tensor-core kernel: 1 = records merged by launch_decode_tc_merge
  int tc_bound[kTcMaxCtas + 1];  // tensor-core kernel: first tile of each CTA's range, then T
  const __half* q;
  __half* out;
  float* part;   // [pairs][splits][gq][d + 2]  (o..., m, l)
  int* counters; // [pairs]
  int* err;      // device error word
};

// Where the rows of a K group / V token come from during an append:
// push index p < n_old reads ring slot (start + p) % R, otherwise input row
// (p - n_old) of the new tokens.
struct RowSrc {
  int n_old;
  int start;
};

struct AppendArgs {
  int batch, h_kv, d, G, R, T;
  const __half* k_new;  // [B][H][T][d]
  const __half* v_new;
  __half* kr;           // ring [B][H][R][d]
  __half* vr;
  // destination: last segment (KIVI) or the plan's segment
  SegDev dst;
  int bits;
  // K side: groups of G pushed tokens to quantize into packed rows nk0 + p
  int k_groups;         // number of groups (flushed tokens / G)
  int k_nk0;            // packed K rows already valid
  RowSrc ksrc;
  int k_ring_groups;    // groups that read at least one old ring token
  // V side: pushed tokens p < v_evict are quantized into packed row nv0 + p
  int v_evict;
  int v_nv0;
  RowSrc vsrc;
  int v_ring_tokens;    // evicted tokens that come from the old ring
  // ring writes of new tokens: K new token j (j >= k_first_ring) -> slot
  // (k_slot0 + j) % R, likewise V
  int k_first_ring, k_slot0;
  int v_first_ring, v_slot0;
  int chunks;           // CTAs per (batch, kv head); chunk 0 does ring work
  int Gv;               // V channel group
  int bulk;             // 1: the new-token work goes to the bulk kernels (d_h 128)
};

struct WindowJob {   // one window of the WindowQuant ingest plan
  int src_token;     // first input token of the window
  int seg;           // destination segment, -1 = fp16 ring
  int dst;           // first packed row (segment) or ring push index (ring)
};

constexpr int kMaxWindowJobs = 512;

struct IngestArgs {
  int batch, h_kv, d, G, R, T, S;
  const __half* k_new;
  const __half* v_new;
  __half* kr;
  __half* vr;
  SegDev seg[KVQ_MAX_SEGMENTS];
  int krs_push, vrs_push;  // ring slot of push index 0 (start + count)
  int n_jobs;              // windows; tail handled as job n_jobs
  int tail_src, tail_len, tail_dst;
  int ring_only;           // 1: ingest_kernel leaves quantized windows to the bulk kernels
  int Gv;                  // V channel group
  WindowJob jobs[kMaxWindowJobs];
};

// ---------------------------------------------------------------------------
// Tile geometry and the bulk copies that stage one tile in shared memory.
// Used by the decode kernel to issue its copies and by the host to check,
// before any launch, that every copy stays inside its buffer.
// ---------------------------------------------------------------------------
struct TileInfo {
  int n;           // tokens in the tile
  int kseg, vseg;  // source segment, -1 = ring
  int ku0, vu0;    // first packed row / first ring index
  int g0, ng;      // first K scale group, groups touched (packed K)
  int kbits, vbits;
  uint32_t k_off, ks_off, kz_off, v_off, vs_off, vz_off, bytes;
};

__host__ __device__ inline uint32_t align16u(uint32_t x) { return (x + 15u) & ~15u; }

// Stream-K ranges of the tensor-core kernel: CTA i of n_cta takes the tiles
// [tc_bound[i], tc_bound[i + 1]) of all pairs' tiles (pair-major), none
// empty.  The owner of tile g is the last i with tc_bound[i] <= g.
__host__ __device__ inline int tc_owner(const int* bound, int n_cta, long long g) {
  int lo = 0, hi = n_cta - 1;  // (the caller maps whole-pair grids itself)
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (bound[mid] <= g) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

__host__ __device__ inline TileInfo tile_info(const DecodeArgs& a, int t) {
  int r = 0;
  while (r + 1 < a.n_runs && a.runs[r + 1].tile0 <= t) ++r;
  const Run& run = a.runs[r];
  const int D = a.d;
  const int pos0 = (t - run.tile0) * run.tile;
  TileInfo ti;
  ti.n = run.len - pos0 < run.tile ? run.len - pos0 : run.tile;
  ti.kseg = run.seg_k;
  ti.vseg = run.seg_v;
  ti.ku0 = run.u0_k + pos0;
  ti.vu0 = run.u0_v + pos0;
  ti.kbits = ti.kseg >= 0 ? a.seg[ti.kseg].bits : 16;
  ti.vbits = ti.vseg >= 0 ? a.seg[ti.vseg].bits : 16;
  uint32_t off = 0;
  ti.k_off = off;
  off += align16u((uint32_t)ti.n * (uint32_t)(D * ti.kbits / 8));
  if (ti.kseg >= 0) {
    ti.g0 = ti.ku0 / a.G;
    ti.ng = (ti.ku0 + ti.n - 1) / a.G - ti.g0 + 1;
    ti.ks_off = off;
    off += (uint32_t)ti.ng * D * 2;
    ti.kz_off = off;
    off += (uint32_t)ti.ng * D * 2;
  } else {
    ti.g0 = ti.ng = 0;
    ti.ks_off = ti.kz_off = off;
  }
  ti.v_off = off;
  off += align16u((uint32_t)ti.n * (uint32_t)(D * ti.vbits / 8));
  if (ti.vseg >= 0) {
    const uint32_t sb = align16u((uint32_t)ti.n * (uint32_t)(D / a.Gv) * 2u);
    ti.vs_off = off;
    off += sb;
    ti.vz_off = off;
    off += sb;
  } else {
    ti.vs_off = ti.vz_off = off;
  }
  ti.bytes = off;
  return ti;
}

// Visit the (at most 8) bulk copies that stage tile `ti` of (batch, kv head)
// `pair`: f(src, dst_off, bytes, buf, seg) with buf 0..5 = segment k_codes,
// k_scale, k_zero, v_codes, v_scale, v_zero and 6/7 = the K/V ring.
template <class F>
__host__ __device__ inline void for_each_tile_copy(const DecodeArgs& a, size_t pair,
                                                   const TileInfo& ti, F&& f) {
  const int D = a.d;
  if (ti.kseg >= 0) {
    const SegDev& s = a.seg[ti.kseg];
    const int rb = D * s.bits / 8;
    f(s.kc + (pair * s.cap + ti.ku0) * rb, ti.k_off, (uint32_t)(ti.n * rb), 0, ti.kseg);
    const size_t gbase = (pair * (size_t)(s.cap / a.G) + ti.g0) * D;
    f(s.ks + gbase, ti.ks_off, (uint32_t)(ti.ng * D * 2), 1, ti.kseg);
    f(s.kz + gbase, ti.kz_off, (uint32_t)(ti.ng * D * 2), 2, ti.kseg);
  } else {
    const int s0 = (a.krs + ti.ku0) % a.R;
    const int n1 = ti.n < a.R - s0 ? ti.n : a.R - s0;
    const __half* ring = a.kr + pair * (size_t)a.R * D;
    f(ring + (size_t)s0 * D, ti.k_off, (uint32_t)(n1 * D * 2), 6, -1);
    if (n1 < ti.n) f(ring, ti.k_off + (uint32_t)(n1 * D * 2), (uint32_t)((ti.n - n1) * D * 2), 6, -1);
  }
  if (ti.vseg >= 0) {
    const SegDev& s = a.seg[ti.vseg];
    const int rb = D * s.bits / 8;
    f(s.vc + (pair * s.cap + ti.vu0) * rb, ti.v_off, (uint32_t)(ti.n * rb), 3, ti.vseg);
    const size_t sbase = (pair * (size_t)s.cap + ti.vu0) * (D / a.Gv);
    const uint32_t sb = align16u((uint32_t)ti.n * (uint32_t)(D / a.Gv) * 2u);
    f(s.vs + sbase, ti.vs_off, sb, 4, ti.vseg);
    f(s.vz + sbase, ti.vz_off, sb, 5, ti.vseg);
  } else {
    const int s0 = (a.vrs + ti.vu0) % a.R;
    const int n1 = ti.n < a.R - s0 ? ti.n : a.R - s0;
    const __half* ring = a.vr + pair * (size_t)a.R * D;
    f(ring + (size_t)s0 * D, ti.v_off, (uint32_t)(n1 * D * 2), 7, -1);
    if (n1 < ti.n) f(ring, ti.v_off + (uint32_t)(n1 * D * 2), (uint32_t)((ti.n - n1) * D * 2), 7, -1);
  }
}

// ---------------------------------------------------------------------------
// Decode with one query head per kv head over one 2-bit segment (the warp
// kernel, kvq_decode_warp.cu): every pair is cut into k pieces of equal
// cost, one per warp, and every warp runs a bulk-copy pipeline of its own
// over its piece's chunks.  Per pair the token axis is cut into
//   - PP chunks: 32 tokens [32u, 32u + 32) of [0, npp), K and V packed
//     (npp = min(nk, nv)); the last one may be short;
//   - X chunks: the rest, [npp, L), in the 8-token blocks of the token
//     index, split at npx = max(nk, nv): one side packed below npx, both
//     from the rings above.  An X chunk is staged as its whole 8-row block,
//     its tokens at rows [o0, o0 + n).
// ---------------------------------------------------------------------------
#ifndef KVQ_WARP_SLOTS
#define KVQ_WARP_SLOTS 3
#endif
#ifndef KVQ_WARP_WARPS
#define KVQ_WARP_WARPS 16
#endif
constexpr int kWarpSlot = 4096;               // bytes of one pipeline slot
constexpr int kWarpSlots = KVQ_WARP_SLOTS;    // slots per warp
constexpr int kWarpWarps = KVQ_WARP_WARPS;    // warps (one-warp CTAs) per SM
// slot layout, PP chunk: K codes, K group scales / zeros, V codes, V token
// scales / zeros (the zeros 32 bytes off a 256-byte stride, so the scale and
// zero loads of one instruction hit different banks)
constexpr int kPpKc = 0, kPpKs = 1024, kPpKz = 1280, kPpVc = 1536, kPpVs = 2560, kPpVz = 2848;
// X chunk: K side at 0 (ring rows, or codes / group scales / zeros), V side
// at 2048 (ring rows, or codes / token scales / zeros)
constexpr int kXK = 0, kXV = 2048, kXKs = 256, kXKz = 512, kXVs = 256, kXVz = 320;

struct WarpArgs {
  const uint8_t* kc;  // segment 0: K codes [P][cap][32]
  const __half* ks;   // [P][cap/G][128]
  const __half* kz;
  const uint8_t* vc;  // V codes [P][cap][32]
  const __half* vs;   // [P][cap][128/Gv]
  const __half* vz;
  const __half* kr;   // rings [P][R][128]
  const __half* vr;
  const __half* q;    // [P][128] (one query head per pair)
  __half* out;
  float* part;        // records [P][k][130]
  int* counters;      // [P] pieces of a pair finished (merge)
  int* err;
  int cap, R, krs, vrs, log2G, ngv, intz;
  float scale_log2;
  int nk, nv, L, npp, npx;
  int n_pp, n_x1, n_x2, C;  // chunks per pair
  long long Cp;             // cost of a pair (kWarpWpp, kWarpWx)
  int P, k;                 // pairs, pieces per pair (records when k > 1)
  int P1;                   // pairs [0, P1) have k pieces, pairs [P1, P) k - 1
  // first chunk holding a token that the decode step's append (or flush)
  // wrote (its staging waits for the kernel before this grid); 0 outside a
  // decode step
  int dep_c;
};

struct WarpChunk {
  int t0, n, o0;  // first token, tokens, row of t0 in the staged block
  int kq, vq, pp;
};

__host__ __device__ inline WarpChunk warp_chunk(const WarpArgs& a, int c) {
  WarpChunk ch;
  if (c < a.n_pp) {
    ch.pp = 1;
    ch.t0 = 32 * c;
    ch.n = a.npp - ch.t0 < 32 ? a.npp - ch.t0 : 32;
    ch.o0 = 0;
    ch.kq = ch.vq = 1;
    return ch;
  }
  const bool r1 = c < a.n_pp + a.n_x1;
  const int lo = r1 ? a.npp : a.npx, hi = r1 ? a.npx : a.L;
  const int blk = lo / 8 + (c - (r1 ? a.n_pp : a.n_pp + a.n_x1));
  const int s = 8 * blk > lo ? 8 * blk : lo;
  const int e = 8 * blk + 8 < hi ? 8 * blk + 8 : hi;
  ch.pp = 0;
  ch.t0 = s;
  ch.n = e - s;
  ch.o0 = s - 8 * blk;
  ch.kq = s < a.nk;
  ch.vq = s < a.nv;
  return ch;
}

// Weights of a 32-token packed chunk and of an 8-token ring chunk for
// cutting a pair into pieces of equal cost: about their bytes (6 : 8), the
// ring chunk raised to 10 by measured warp times (a ring chunk took ~18 %
// more time per unit of byte cost than a packed one).
#ifndef KVQ_WARP_WPP
#define KVQ_WARP_WPP 6
#endif
#ifndef KVQ_WARP_WX
#define KVQ_WARP_WX 10
#endif
constexpr int kWarpWpp = KVQ_WARP_WPP, kWarpWx = KVQ_WARP_WX;

// First chunk of piece j of a pair cut into `kp` pieces of equal cost (j =
// kp gives C): the first chunk whose cost offset reaches floor(Cp * j / kp).
__host__ __device__ inline int warp_piece_start(const WarpArgs& a, int kp, int j) {
  const long long r = a.Cp * (long long)j / kp;
  const long long pp_cost = (long long)kWarpWpp * a.n_pp;
  const long long c = r <= pp_cost ? (r + kWarpWpp - 1) / kWarpWpp : a.n_pp + (r - pp_cost + kWarpWx - 1) / kWarpWx;
  return (int)(c < a.C ? c : a.C);
}

// The bulk copies that stage chunk c of `pair` in a slot: f(src, dst_off,
// bytes, buf) with buf 0..5 = K codes, K scales, K zeros, V codes, V scales,
// V zeros and 6/7 = the K / V ring.
template <class F>
__host__ __device__ inline void warp_chunk_copies(const WarpArgs& a, long long pair, const WarpChunk& ch, F&& f) {
  const int G = 1 << a.log2G;
  const long long ksb = (pair * (a.cap / G) + (ch.t0 >> a.log2G)) * 128;  // K group, in halves
  if (ch.pp) {
    const long long row = pair * a.cap + ch.t0;
    const uint32_t sb = (uint32_t)((ch.n * a.ngv * 2 + 15) & ~15);
    f(a.kc + row * 32, kPpKc, (uint32_t)ch.n * 32u, 0);
    f(a.ks + ksb, kPpKs, 256u, 1);
    f(a.kz + ksb, kPpKz, 256u, 2);
    f(a.vc + row * 32, kPpVc, (uint32_t)ch.n * 32u, 3);
    f(a.vs + row * a.ngv, kPpVs, sb, 4);
    f(a.vz + row * a.ngv, kPpVz, sb, 5);
    return;
  }
  const long long blk = pair * a.cap + (ch.t0 - ch.o0);  // the chunk's 8-row block
  if (ch.kq) {
    f(a.kc + blk * 32, kXK, 256u, 0);
    f(a.ks + ksb, kXK + kXKs, 256u, 1);
    f(a.kz + ksb, kXK + kXKz, 256u, 2);
  } else {
    const int s0 = (a.krs + (ch.t0 - a.nk)) % a.R;
    const int n1 = ch.n < a.R - s0 ? ch.n : a.R - s0;
    const __half* ring = a.kr + pair * a.R * 128;
    f(ring + (long long)s0 * 128, kXK + ch.o0 * 256, (uint32_t)n1 * 256u, 6);
    if (n1 < ch.n) f(ring, kXK + (ch.o0 + n1) * 256, (uint32_t)(ch.n - n1) * 256u, 6);
  }
  if (ch.vq) {
    f(a.vc + blk * 32, kXV, 256u, 3);
    f(a.vs + blk * a.ngv, kXV + kXVs, (uint32_t)(16 * a.ngv), 4);
    f(a.vz + blk * a.ngv, kXV + kXVz, (uint32_t)(16 * a.ngv), 5);
  } else {
    const int s0 = (a.vrs + (ch.t0 - a.nv)) % a.R;
    const int n1 = ch.n < a.R - s0 ? ch.n : a.R - s0;
    const __half* ring = a.vr + pair * a.R * 128;
    f(ring + (long long)s0 * 128, kXV + ch.o0 * 256, (uint32_t)n1 * 256u, 7);
    if (n1 < ch.n) f(ring, kXV + (ch.o0 + n1) * 256, (uint32_t)(ch.n - n1) * 256u, 7);
  }
}

// ---------------------------------------------------------------------------
// Paged cache with per-sequence lengths.  A sequence's token axis is cut into
// three runs -- both packed [0, min(nk, nv)), one side packed [min, max),
// both ring [max, L) -- and each run into tiles aligned to multiples of the
// tile size in the token index, so a packed tile never crosses a page
// (the tile sizes divide the page).
// ---------------------------------------------------------------------------
struct PagedSeq {
  int nk, nv, nkr, nvr, krs, vrs;
  int n_tiles;  // tiles of the sequence (the same for each kv head)
  int split0;   // first grid column of the sequence
  int n_split;  // CTAs per kv head of the sequence
};

struct PagedArgs {
  int batch, h_kv, gq, d, G, R, log2G, Gv, log2Gv, P, bits;
  float scale_log2;
  int intz;           // zero slots hold integer zero points (x' = s (code - z))
  const uint8_t* kc;  // pool [n_pages][h_kv][P][d*bits/8]
  const __half* ks;   // pool [n_pages][h_kv][P/G][d]
  const __half* kz;
  const uint8_t* vc;
  const __half* vs;   // pool [n_pages][h_kv][P][d/Gv]
  const __half* vz;
  const int* table;   // [batch][max_pages]
  int max_pages, n_pages;
  const __half* kr;   // rings [batch][h_kv][R][d]
  const __half* vr;
  const __half* q;
  __half* out;
  float* part;        // [pairs][n_splits][gq][d + 2]
  int* counters;      // [pairs]
  int* err;           // workspace error word (timed-out waits)
  int* page_err;      // the cache's error word (bad block-table entries)
  int n_splits;       // records per (sequence, kv head) in the workspace
  int tile_pp;        // tile tokens where K and V are both packed
  int tile_mix;       // tile tokens where the ring is involved
  int n_cols;         // grid columns (sum of n_split)
  int n_seq;
  PagedSeq seq[KVQ_MAX_SEQS];
};

__host__ __device__ inline int paged_run_tiles(int lo, int hi, int ts) {
  return hi > lo ? (hi - 1) / ts - lo / ts + 1 : 0;
}

__host__ __device__ inline int paged_tiles(const PagedArgs& a, const PagedSeq& s) {
  const int L = s.nk + s.nkr;
  const int a0 = s.nk < s.nv ? s.nk : s.nv, a1 = s.nk < s.nv ? s.nv : s.nk;
  return paged_run_tiles(0, a0, a.tile_pp) + paged_run_tiles(a0, a1, a.tile_mix) +
         paged_run_tiles(a1, L, a.tile_mix);
}

// Tile t of sequence s: ku0/vu0 = packed row (absolute token index) when the
// side is packed, else ring index; kseg/vseg = 0 packed, -1 ring.
__host__ __device__ inline TileInfo paged_tile(const PagedArgs& a, const PagedSeq& s, int t) {
  const int L = s.nk + s.nkr;
  const int a0 = s.nk < s.nv ? s.nk : s.nv, a1 = s.nk < s.nv ? s.nv : s.nk;
  const int n0 = paged_run_tiles(0, a0, a.tile_pp), n1 = paged_run_tiles(a0, a1, a.tile_mix);
  int lo, hi, ts;
  if (t < n0) {
    lo = 0, hi = a0, ts = a.tile_pp;
  } else if (t < n0 + n1) {
    t -= n0, lo = a0, hi = a1, ts = a.tile_mix;
  } else {
    t -= n0 + n1, lo = a1, hi = L, ts = a.tile_mix;
  }
  int start = (lo / ts + t) * ts, end = start + ts;
  start = start > lo ? start : lo;
  end = end < hi ? end : hi;
  const int D = a.d;
  TileInfo ti;
  ti.n = end - start;
  ti.kseg = start < s.nk ? 0 : -1;
  ti.vseg = start < s.nv ? 0 : -1;
  ti.ku0 = ti.kseg == 0 ? start : start - s.nk;
  ti.vu0 = ti.vseg == 0 ? start : start - s.nv;
  ti.kbits = ti.kseg == 0 ? a.bits : 16;
  ti.vbits = ti.vseg == 0 ? a.bits : 16;
  uint32_t off = 0;
  ti.k_off = off;
  off += align16u((uint32_t)ti.n * (uint32_t)(D * ti.kbits / 8));
  if (ti.kseg == 0) {
    ti.g0 = ti.ku0 / a.G;
    ti.ng = (ti.ku0 + ti.n - 1) / a.G - ti.g0 + 1;
    ti.ks_off = off;
    off += (uint32_t)ti.ng * D * 2;
    ti.kz_off = off;
    off += (uint32_t)ti.ng * D * 2;
  } else {
    ti.g0 = ti.ng = 0;
    ti.ks_off = ti.kz_off = off;
  }
  ti.v_off = off;
  off += align16u((uint32_t)ti.n * (uint32_t)(D * ti.vbits / 8));
  if (ti.vseg == 0) {
    const uint32_t sb = align16u((uint32_t)ti.n * (uint32_t)(D / a.Gv) * 2u);
    ti.vs_off = off;
    off += sb;
    ti.vz_off = off;
    off += sb;
  } else {
    ti.vs_off = ti.vz_off = off;
  }
  ti.bytes = off;
  return ti;
}

// Visit the bulk copies that stage paged tile `ti` of sequence b, kv head h:
// f(src, dst_off, bytes, slot), slot 0-2 the K side (codes, scales, zeros or
// the ring's one or two pieces), 3-5 the V side.  page(row) maps a packed row to its pool page (the
// caller checks the block-table entry).
template <class Page, class F>
__host__ __device__ inline void for_each_paged_copy(const PagedArgs& a, int b, int h, const PagedSeq& s,
                                                    const TileInfo& ti, Page&& page, F&& f) {
  const int D = a.d, P = a.P;
  const size_t pair = (size_t)b * a.h_kv + h;
  const int rb = D * a.bits / 8;
  if (ti.kseg == 0) {
    const size_t ph = (size_t)page(ti.ku0) * a.h_kv + h;
    const int r = ti.ku0 % P;
    f(a.kc + (ph * P + r) * rb, ti.k_off, (uint32_t)(ti.n * rb), 0);
    const size_t gbase = (ph * (size_t)(P / a.G) + r / a.G) * D;
    f(a.ks + gbase, ti.ks_off, (uint32_t)(ti.ng * D * 2), 1);
    f(a.kz + gbase, ti.kz_off, (uint32_t)(ti.ng * D * 2), 2);
  } else {
    const int s0 = (s.krs + ti.ku0) % a.R;
    const int n1 = ti.n < a.R - s0 ? ti.n : a.R - s0;
    const __half* ring = a.kr + pair * (size_t)a.R * D;
    f(ring + (size_t)s0 * D, ti.k_off, (uint32_t)(n1 * D * 2), 0);
    if (n1 < ti.n) f(ring, ti.k_off + (uint32_t)(n1 * D * 2), (uint32_t)((ti.n - n1) * D * 2), 1);
  }
  if (ti.vseg == 0) {
    const size_t ph = (size_t)page(ti.vu0) * a.h_kv + h;
    const int r = ti.vu0 % P;
    f(a.vc + (ph * P + r) * rb, ti.v_off, (uint32_t)(ti.n * rb), 3);
    const size_t sbase = (ph * P + r) * (D / a.Gv);
    const uint32_t sb = align16u((uint32_t)ti.n * (uint32_t)(D / a.Gv) * 2u);
    f(a.vs + sbase, ti.vs_off, sb, 4);
    f(a.vz + sbase, ti.vz_off, sb, 5);
  } else {
    const int s0 = (s.vrs + ti.vu0) % a.R;
    const int n1 = ti.n < a.R - s0 ? ti.n : a.R - s0;
    const __half* ring = a.vr + pair * (size_t)a.R * D;
    f(ring + (size_t)s0 * D, ti.v_off, (uint32_t)(n1 * D * 2), 3);
    if (n1 < ti.n) f(ring, ti.v_off + (uint32_t)(n1 * D * 2), (uint32_t)((ti.n - n1) * D * 2), 4);
  }
}

// Per-sequence append work (KIVI Algorithm 1 for one sequence), the fields
// of AppendArgs that differ between sequences.
struct PagedAppendSeq {
  int t;              // new tokens of the sequence
  int k_groups, k_nk0, k_ring_groups;
  RowSrc ksrc;
  int v_evict, v_nv0, v_ring_tokens;
  RowSrc vsrc;
  int k_first_ring, k_slot0, v_first_ring, v_slot0;
  int k_item0, v_item0;  // bulk kernels: first work item of the sequence
};

struct PagedAppendArgs {
  int batch, h_kv, d, G, Gv, R, T, P, bits, intz;
  const __half* k_new;  // [B][H][T][d]
  const __half* v_new;
  __half* kr;           // rings [B][H][R][d]
  __half* vr;
  uint8_t* kc;          // pool, as PagedArgs
  __half* ks;
  __half* kz;
  uint8_t* vc;
  __half* vs;
  __half* vz;
  const int* table;
  int max_pages, n_pages;
  int* page_err;
  int chunks;           // CTAs per (sequence, kv head); chunk 0 does ring work
  int flush;            // 1: K flush of the rings only (kvq_paged_flush_residual)
  int bulk;             // 1: new-token groups and tokens go to the bulk kernels (d_h 128)
  int k_items, v_items; // bulk kernels: (sequence, kv head, group / token) work items
  int n_seq;
  PagedAppendSeq seq[KVQ_MAX_SEQS];
};

// Make a kernel's dynamic shared-memory limit at least `bytes` on the
// current device.  The attribute is one maximum per (kernel, device) that
// lives in the device's context; it is raised only when a launch needs more
// than the largest value set so far (never lowered: a smaller value would
// fail later launches that need more), so most launches make no driver call.
inline cudaError_t set_smem_once(const void* kernel, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> raised;
  const auto key = std::make_pair(kernel, dev);
  std::lock_guard<std::mutex> lock(mu);
  const auto it = raised.find(key);
  if (it != raised.end() && it->second >= bytes) return cudaSuccess;
  if (it == raised.end()) {
    // Every kernel of the library asks for the largest shared-memory
    // carveout: an SM runs CTAs of two kernels side by side only under one
    // L1/shared split, so a small quantize kernel with a small carveout would
    // keep the decode kernel (which needs most of the SM's shared memory)
    // off the SM until it drains, and a dependent launch could not overlap.
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
  }
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) raised[key] = bytes;
  return e;
}

// Launch a kernel on stream s; with pdl, allowed to start before the previous
// kernel of the stream completes (programmatic stream serialization): such a
// kernel executes griddepcontrol.wait before it touches anything that kernel
// writes.
template <class... KArgs, class... Args>
inline cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                 bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// host helpers of kvq_api.cu used by other entry points
int sm_count_cached();  // SMs of the current device, looked up once per device
void set_last_error(const char* msg);
kvq_status check_cache(const kvq_cache* c);

// kernels' launchers (return cudaGetLastError())
cudaError_t launch_append(const AppendArgs& a, cudaStream_t s, bool pdl = false);
cudaError_t launch_flush(const AppendArgs& a, cudaStream_t s, bool pdl = false);
cudaError_t launch_ingest(const IngestArgs& a, cudaStream_t s);
cudaError_t launch_decode(const DecodeArgs& a, int n_pairs, cudaStream_t s);
size_t decode_smem_bytes(int gq, int d);
cudaError_t launch_decode_mha(const DecodeArgs& a, int n_pairs, int bits, cudaStream_t s);
cudaError_t launch_decode_tc(const DecodeArgs& a, int bits, int form, cudaStream_t s);
cudaError_t launch_decode_tc_merge(const DecodeArgs& a, int n_pairs, cudaStream_t s);
cudaError_t launch_decode_warp(const WarpArgs& a, cudaStream_t s, bool pdl = false);
cudaError_t launch_decode_paged(const PagedArgs& a, cudaStream_t s);
cudaError_t launch_decode_tc_paged(const DecodeArgs& a, const PagedArgs& p, int bits, int form, cudaStream_t s);
cudaError_t launch_paged_append(const PagedAppendArgs& a, cudaStream_t s);
int decode_tc_ctas_per_sm();
size_t decode_mha_smem_bytes();

struct WindowArgs {
  const __half* keys;  // [B][H][M][d]
  const __half* text;  // [B][H][N][d]
  int batch, h_kv, d, M, S, N;
  int n8, n4, first_fp16;
  double* tsum;        // [B][H*d]
  double* wstat;       // [B][n_win][2] (dot with text sum, squared norm)
  double* sim;         // [n_win]
  int8_t* bits;        // [n_win] device
  int32_t* perm;       // [n_win] device
};
cudaError_t launch_window_assign(const WindowArgs& a, cudaStream_t s);

// WindowQuant paper-exact assignment (Eq.8 scores, Eq.10-11 thresholds).
struct Eq8Args {
  const __half* vision;  // [B][M][dim]
  const __half* text;    // [B][N][dim]
  int batch, dim, M, S, N;
  int chunks;            // token chunks per window / text (partial sums)
  double t_low, t_high;
  int first_fp16;
  double* part;          // [B][n_win + 1][chunks][dim]: sums of unit vectors
  double* sims;          // [B][n_win]
  int8_t* bits;          // [n_win]
  int32_t* perm;         // [n_win]
};
cudaError_t launch_window_assign_eq8(const Eq8Args& a, cudaStream_t s);

}  // namespace kvq
