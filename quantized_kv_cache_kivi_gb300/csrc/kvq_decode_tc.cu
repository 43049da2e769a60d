// Decode attention over a quantized KV cache at d_h = 128 with both
// contractions on the tensor cores (mma.sync m16n8k16, fp16 operands, fp32
// accumulation), in three forms: one query head per kv head over one packed
// segment plus the fp16 ring (the KIVI layout); 2-4 query heads per kv head
// over one segment; up to 8 query heads over any mix of segment widths (the
// WindowQuant layout: INT8 / INT4 / INT2 windows and an fp16 tail).
//
// What is computed (KIVI page, Algorithm 1 decoding branch; WindowQuant
// §3.3.1 for several widths):
//   a_t = sm_scale * q . k_t, p = softmax(a), out = sum_t p_t v_t,
// with packed K dequantized per (group, channel) and packed V per (token,
// channel group).  The algebra that makes both contractions tensor-core
// shaped:
//   K:  q . k_t = sum_c (q_c s_gc) code_tc + sum_c q_c z_gc.  A = codes
//       [token][channel]; B = the scaled query split into an fp16 high part
//       and low part, so every lane ends up with whole scores; plus the
//       per-group bias q . z_g.
//   V (1 and 4 heads):  sum_t p_t (code_tc s_tg(c) + z_tg(c)) = sum_t (p_t
//       s_tg) code_tc + sum_t p_t z_tg.  A = codes [channel][token]; B[t][n]
//       = p_t s_tn for the channel groups n < 4 and p_t z_t(n-4) for n >= 4.
//       Row c keeps column g(c); one more MMA with an all-ones A yields the
//       z sums.  (8 heads: see the section of that form.)
// Codes become fp16 operands without any conversion: a code field left at bit
// p (0 <= p <= 8) of a 16-bit half, every other bit zero, is the fp16
// subnormal code * 2^(p - 24) exactly; one 32-bit AND yields two of them.
// The products are exact in the fp32 accumulators, so the factor 2^(24 - p)
// is folded into B for K (2^-p, scores scaled by 2^24 afterwards) and divided
// out of each channel row for V.
//
// Work split: a persistent grid of CTAs walks the concatenated tile list of
// all (batch, kv head) pairs in contiguous ranges of equal cost (stream-K;
// the host computes the range table); a range that covers part of a pair
// leaves a partial (o, m, l) record and the last CTA of that pair to finish
// merges the records, or, when a pair has many of them, a small launch of
// its own does.  CTA = 5-7 consumer warps that take the 32-token units of
// each staged tile in round-robin order, each building the K operand of its
// unit's K group and keeping its own online softmax, and 1 warp that issues
// the bulk copies (TMA engine) of up to 3-4 tiles ahead.
#include <float.h>

#include <type_traits>

#include "kvq_device.cuh"
#include "kvq_internal.h"
#include "kvq_mma.cuh"

namespace kvq {
namespace {

using namespace mma;

// HQ = query-head columns: 1 (one query head per kv head; every column of
// the K operand carries it), 4 (2-4 query heads per kv head; lane tig of a
// quad owns head tig) or 8 (up to 8 query heads, any segments: column n is
// head n, lane tig owns heads 2 tig and 2 tig + 1).
template <int HQ>
struct TcCfg {
  static constexpr int NCW = HQ == 1 ? 7 : (HQ == 8 ? 5 : 6);  // consumer warps
  static constexpr int NTH = (NCW + 1) * 32;           // + the bulk-copy warp
  static constexpr int NSLOT = HQ == 1 ? 3 : 1;        // merge slots
  static constexpr int NS = HQ == 8 ? 3 : kTcStages;   // pipeline stages
  static constexpr int KTAB = 512 * HQ;                // bytes of a warp's K operand
};

// What the producer records about the tile it staged in a stage.
struct TcRec {
  int n;       // tokens
  int kq, vq;  // 1: K / V come from the packed segment, 0: from the ring
  int kr0;     // first packed K row mod G
  uint32_t k_off, v_off, vs_off, vz_off;
  uint32_t ks_off, kz_off;  // K scales / zeros of the staged groups
  int kb, vb;  // widths of the packed K / V segments (16: ring)
  int pad[4];
};
static_assert(sizeof(TcRec) == 64, "record size");

constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }

template <int HQ>
struct TcSmem {
  static constexpr int NCW = TcCfg<HQ>::NCW, NS = TcCfg<HQ>::NS;
  static constexpr int stages = 0;
  static constexpr int q = stages + NS * kTcStageBytes;               // [stage][HQ][D] f16
  static constexpr int ktab = q + NS * HQ * D * 2;                    // [warp] K operand of its unit
  static constexpr int rec = ktab + NCW * TcCfg<HQ>::KTAB;            // [stage] TcRec
  static constexpr int merge = rec + NS * 64;                         // [slot][NCW][HQ][D + 2] f32
  static constexpr int slot_owner =
      align_up(merge + TcCfg<HQ>::NSLOT * NCW * HQ * (D + 2) * 4, 16);  // [slot] piece served
  static constexpr int slot_count = slot_owner + 16;                  // [slot] warps arrived
  static constexpr int zero = slot_count + 16;                        // 64 zero bytes
  static constexpr int args = zero + 64;                             // DecodeArgs copy
  static constexpr int bars = align_up(args + (int)sizeof(DecodeArgs), 16);
  static constexpr int flags = bars + 2 * NS * 8;
  static constexpr int total = flags + 16;
};
static_assert(TcSmem<1>::q % 16 == 0 && TcSmem<1>::ktab % 16 == 0 && TcSmem<1>::rec % 16 == 0, "align");
static_assert(TcSmem<4>::q % 16 == 0 && TcSmem<4>::ktab % 16 == 0 && TcSmem<4>::rec % 16 == 0, "align");
static_assert(kTcCtasPerSm * (TcSmem<1>::total + 1024) <= 228 * 1024, "CTAs per SM");
static_assert(kTcCtasPerSm * (TcSmem<4>::total + 1024) <= 228 * 1024, "CTAs per SM");
static_assert(TcSmem<8>::q % 16 == 0 && TcSmem<8>::ktab % 16 == 0 && TcSmem<8>::rec % 16 == 0, "align");
static_assert(kTcCtasPerSm * (TcSmem<8>::total + 1024) <= 228 * 1024, "CTAs per SM");

// Bounded wait: about 2^31 SM clocks, then the abort flag is raised.  Every
// warp waits inside the barrier unit (suspend-time hint) rather than
// spinning, so a waiting warp leaves its issue slots to the working ones.
template <bool BACKOFF>
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  const uint32_t addr = smem_u32(bar);
  if (try_wait_at(addr, parity)) return true;
  const long long t0 = clock64();
  while (!try_wait_sleep(addr, parity, 20000u)) {
    if (*abort_flag) return false;
    if (clock64() - t0 > (1ll << 31)) {
      *abort_flag = 1;
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}


// Per-warp online-softmax state.  acc holds, for the channel rows of m-tile
// mt, D = sum_t B[t][n] A[c][t] (packed V: carrying 2^(p - 24) until the first
// ring-V sub-tile or the end); accz columns 4.. hold sum_t p_t z_t(n-4).
struct WarpState {
  float m;  // running max (log2 domain), warp-uniform
  float l;  // sum of p over the rows of this lane (tig-replicated)
  float acc[8][4];
  float accz[4];
  bool vring;  // acc already unscaled (ring V reached)
};

__device__ __forceinline__ void reset_state(WarpState& S) {
  S.m = -INFINITY;
  S.l = 0.f;
  S.vring = false;
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) S.acc[i][e] = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) S.accz[e] = 0.f;
}

template <int B>
__device__ __forceinline__ void unscale_acc(WarpState& S) {
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    const int p = Fields<B>::pos(mt % (16 / B));
    const float us = __uint_as_float((uint32_t)(127 + 24 - p) << 23);  // 2^(24 - p)
#pragma unroll
    for (int e = 0; e < 4; ++e) S.acc[mt][e] *= us;
  }
}

// The dynamic shared memory block of the decode kernel.
__device__ __forceinline__ uint8_t* tc_smem() {
  extern __shared__ __align__(128) uint8_t smem_dyn[];
  return smem_dyn;
}

// Scores (log2 domain) of the rows gid and gid + 8 of the 16-token half at
// s0 + 16 h, packed K: the shared B operand bq of the unit's K group, the
// thread's code words of its two rows, 8 MMAs in two chains.
template <int B>
__device__ __forceinline__ void k_scores_packed(const uint8_t* kc, int s0, int r0, int r1, const uint32_t (&bq)[16],
                                                float bias, float& x0, float& x1) {
  constexpr int PH = 16 / B;
  constexpr int RB = D * B / 8;           // packed row bytes
  constexpr int NW = B;                   // words of a row per thread (32 channels)
  constexpr int WPC = NW < 4 ? NW : 4;    // words per load
  constexpr int NCH = NW / WPC;           // loads per row
  float sc[4] = {0.f, 0.f, 0.f, 0.f};
  float sd[4] = {0.f, 0.f, 0.f, 0.f};  // odd k-tiles: two shorter MMA chains
#pragma unroll
  for (int ch = 0; ch < NCH; ++ch) {
    uint32_t w0[WPC], w1[WPC];
    if constexpr (WPC == 2) {
      const uint2 u0 = *reinterpret_cast<const uint2*>(kc + (s0 + r0) * RB);
      const uint2 u1 = *reinterpret_cast<const uint2*>(kc + (s0 + r1) * RB);
      w0[0] = u0.x; w0[1] = u0.y;
      w1[0] = u1.x; w1[1] = u1.y;
    } else {
      const uint4 u0 = *reinterpret_cast<const uint4*>(kc + (s0 + r0) * RB + 16 * ch);
      const uint4 u1 = *reinterpret_cast<const uint4*>(kc + (s0 + r1) * RB + 16 * ch);
      w0[0] = u0.x; w0[1] = u0.y; w0[2] = u0.z; w0[3] = u0.w;
      w1[0] = u1.x; w1[1] = u1.y; w1[2] = u1.z; w1[3] = u1.w;
    }
#pragma unroll
    for (int kk = 0; kk < 8 / NCH; ++kk) {
      const int kt = ch * (8 / NCH) + kk;
      uint32_t av[4];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int h = 2 * kt + e;
        const int w = h / PH - ch * WPC, j = h % PH;
        av[2 * e + 0] = Fields<B>::get(w0[w], w0[w] >> 6, j);
        av[2 * e + 1] = Fields<B>::get(w1[w], w1[w] >> 6, j);
      }
      mma16816((kt & 1) ? sd : sc, av[0], av[1], av[2], av[3], bq[2 * kt], bq[2 * kt + 1]);
    }
  }
  // the table carries sm_scale log2(e) and 2^-p, the codes 2^(p - 24)
  x0 = fmaf((sc[0] + sd[0]) + (sc[1] + sd[1]), 16777216.0f, bias);  // row gid: high + low column
  x1 = fmaf((sc[2] + sd[2]) + (sc[3] + sd[3]), 16777216.0f, bias);  // row gid + 8
}

// Both halves of a 32-token unit at 2 bits, their MMA chains interleaved
// (four accumulators, an MMA's successor on the same accumulator comes four
// MMAs later).
__device__ __forceinline__ void k_scores_packed2_b2(const uint8_t* kc, int s0, int r0, int r1,
                                                    const uint32_t (&bq)[16], float bias, float (&x)[2][2]) {
  constexpr int RB = D * 2 / 8;
  uint32_t w[2][2][2];  // [half][row][word]
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint2 u0 = *reinterpret_cast<const uint2*>(kc + (s0 + 16 * h + r0) * RB);
    const uint2 u1 = *reinterpret_cast<const uint2*>(kc + (s0 + 16 * h + r1) * RB);
    w[h][0][0] = u0.x; w[h][0][1] = u0.y;
    w[h][1][0] = u1.x; w[h][1][1] = u1.y;
  }
  float acc[2][2][4] = {};  // [half][k-tile parity][fragment]
#pragma unroll
  for (int kt = 0; kt < 8; ++kt) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t av[4];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int hh = 2 * kt + e;
        const int wi = hh / 8, j = hh % 8;
        av[2 * e + 0] = Fields<2>::get(w[h][0][wi], w[h][0][wi] >> 6, j);
        av[2 * e + 1] = Fields<2>::get(w[h][1][wi], w[h][1][wi] >> 6, j);
      }
      mma16816(acc[h][kt & 1], av[0], av[1], av[2], av[3], bq[2 * kt], bq[2 * kt + 1]);
    }
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    x[h][0] = fmaf((acc[h][0][0] + acc[h][1][0]) + (acc[h][0][1] + acc[h][1][1]), 16777216.0f, bias);
    x[h][1] = fmaf((acc[h][0][2] + acc[h][1][2]) + (acc[h][0][3] + acc[h][1][3]), 16777216.0f, bias);
  }
}

// Same for fp16 ring K.  Thread tig reads its 32 channels as four 16-byte
// chunks, chunk kc at position (kc + tig) & 3 of the block (spreads the
// banks), and the query words in the same order: each chunk feeds 2 MMAs.
__device__ __forceinline__ void k_scores_ring(const uint8_t* kr, const uint8_t* qt, uint32_t qmask, int s0, int r0,
                                              int r1, int tig, float scale_log2, float& x0, float& x1) {
  float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int kc = 0; kc < 4; ++kc) {
    const int off = ((kc + tig) & 3) * 16;
    const uint4 u0 = *reinterpret_cast<const uint4*>(kr + (s0 + r0) * (D * 2) + off);
    const uint4 u1 = *reinterpret_cast<const uint4*>(kr + (s0 + r1) * (D * 2) + off);
    const uint4 qw = *reinterpret_cast<const uint4*>(qt + off);
    mma16816(sc, u0.x, u1.x, u0.y, u1.y, qw.x & qmask, qw.y & qmask);
    mma16816(sc, u0.z, u1.z, u0.w, u1.w, qw.z & qmask, qw.w & qmask);
  }
  x0 = sc[0] * scale_log2;  // columns 2 tig and 2 tig + 1 carry the same query
  x1 = sc[2] * scale_log2;
}

// The K operand of one K group, built by the consuming warp itself: lane
// (tig, kt) computes q_c s_gc 2^-p sm_scale log2(e) for the 4 channels of
// the operand entries (tig, kt, e = 0/1) and every query head, splits each
// into an fp16 high and low part and stores both; every lane then reads the
// 16 words of its own column (head, hi or lo; tig) row.  Returns the bias
// q_h . z_g (log2 domain) of the lane's head.  Query heads past `gq` (HQ = 4
// with 2 or 3 heads) read as zero.
template <int B, int HQ>
__device__ __forceinline__ float build_k_operand(const DecodeArgs& a, const uint8_t* stage, const __half* qs,
                                                 const TcRec& r, int gl, uint32_t* scratch, int lane,
                                                 uint32_t (&bq)[16]) {
  const int ptig = lane >> 3, pkt = lane & 7;
  const __half* sg = reinterpret_cast<const __half*>(stage + r.ks_off) + gl * D;
  const __half* zg = reinterpret_cast<const __half*>(stage + r.kz_off) + gl * D;
  int cs[4];
  float f[4];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    int clo, chi, p;
    k_half2_channels<B>(ptig, 2 * pkt + e, &clo, &chi, &p);
    cs[2 * e] = clo;
    cs[2 * e + 1] = chi;
    f[2 * e] = f[2 * e + 1] = __uint_as_float((uint32_t)(127 - p) << 23) * a.scale_log2;  // 2^-p sm_scale log2(e)
  }
  float sv[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) sv[e] = __half2float(sg[cs[e]]) * f[e];
  float zsum[HQ];
#pragma unroll
  for (int h = 0; h < HQ; ++h) {
    const bool live = HQ == 1 || h < a.gq;
    const __half* qh = qs + h * D;
    float hi[4], lo[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float v = live ? __half2float(qh[cs[e]]) * sv[e] : 0.f;
      hi[e] = __half2float(__float2half_rn(v));
      lo[e] = v - hi[e];
    }
    // scratch entry (k = kt / 2, column hp = 2 h + part, tig): 4 words, kt even (b0, b1) then kt odd
    *reinterpret_cast<uint2*>(scratch + (((pkt >> 1) * 2 * HQ + 2 * h) * 4 + ptig) * 4 + (pkt & 1) * 2) =
        make_uint2(pack_half2(hi[0], hi[1]), pack_half2(hi[2], hi[3]));
    *reinterpret_cast<uint2*>(scratch + (((pkt >> 1) * 2 * HQ + 2 * h + 1) * 4 + ptig) * 4 + (pkt & 1) * 2) =
        make_uint2(pack_half2(lo[0], lo[1]), pack_half2(lo[2], lo[3]));
    float z = 0.f;
    if (live) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        z = fmaf(__half2float(qh[lane + 32 * i]),
                 zero_add(__half_as_ushort(zg[lane + 32 * i]), __half_as_ushort(sg[lane + 32 * i]), a.intz), z);
    }
    zsum[h] = z;
  }
#pragma unroll
  for (int h = 0; h < HQ; ++h)
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) zsum[h] += __shfl_xor_sync(kFull, zsum[h], off);
  __syncwarp();
  const int gid = lane >> 2, tig = lane & 3;
  // column n = gid: HQ = 1 -> hi (even) / lo (odd); HQ = 4 -> head gid / 2, hi / lo
  const int hp = HQ == 1 ? (gid & 1) : gid;
  const uint4* tb = reinterpret_cast<const uint4*>(scratch) + hp * 4 + tig;
#pragma unroll
  for (int k = 0; k < 4; ++k) *reinterpret_cast<uint4*>(&bq[4 * k]) = tb[k * 8 * HQ];
  __syncwarp();  // scratch reads done before the next unit rewrites it
  float bias = zsum[0];
#pragma unroll
  for (int h = 1; h < HQ; ++h) bias = tig == h ? zsum[h] : bias;
  return bias * a.scale_log2;
}

// One 32-token unit [s0, s0 + 32) of the staged tile: two 16-token halves
// (rows sigma(r) of half h are tokens s0 + 16 h + sigma(r)).  s0 is a
// multiple of 32 and the unit lies inside one K group (G >= 32, packed runs
// start on 32-token boundaries), so both halves share one K operand.
template <int B, int HQ, bool KQ, bool VQ, bool FULL>
__device__ __forceinline__ void sub_unit(const DecodeArgs& a, int st, const TcRec& r, int s0, int lane, WarpState& S) {
  using SM = TcSmem<HQ>;
  constexpr int PH = 16 / B;
  const int gid = lane >> 2, tig = lane & 3;
  const int r0 = sigma(gid), r1 = sigma(gid + 8);
  uint8_t* const sm = tc_smem();
  const uint8_t* const stage = sm + SM::stages + st * kTcStageBytes;
  const int nv = r.n - s0;  // valid tokens from s0 (>= 32 when FULL)
  // ------------------------------------------------------------- scores
  float x[2][2];  // [half][row gid, row gid + 8]
  if constexpr (KQ) {
    const int gl = (r.kr0 + s0) >> a.log2G;
    uint32_t bq[16];
    const float bias = build_k_operand<B, HQ>(
        a, stage, reinterpret_cast<const __half*>(sm + SM::q + st * HQ * D * 2), r, gl,
        reinterpret_cast<uint32_t*>(sm + SM::ktab) + (threadIdx.x >> 5) * (TcCfg<HQ>::KTAB / 4), lane, bq);
    const uint8_t* kc = stage + r.k_off + tig * (B * 4);
    if constexpr (B == 2) {
      k_scores_packed2_b2(kc, s0, r0, r1, bq, bias, x);  // rows past the tile read stale bytes: masked below
    } else {
      k_scores_packed<B>(kc, s0, r0, r1, bq, bias, x[0][0], x[0][1]);
      if (FULL || nv > 16) k_scores_packed<B>(kc, s0 + 16, r0, r1, bq, bias, x[1][0], x[1][1]);
      else x[1][0] = x[1][1] = -INFINITY;
    }
  } else {
    // column n = gid holds the query of head gid / 2 (HQ = 4) or of the one head
    const int qh = HQ == 1 ? 0 : gid >> 1;
    const uint8_t* qt = sm + SM::q + (st * HQ + qh) * D * 2 + tig * 64;
    const uint32_t qmask = (HQ == 1 || qh < a.gq) ? 0xffffffffu : 0u;
    const uint8_t* kr = stage + r.k_off + tig * 64;
    k_scores_ring(kr, qt, qmask, s0, r0, r1, tig, a.scale_log2, x[0][0], x[0][1]);
    if (FULL || nv > 16) k_scores_ring(kr, qt, qmask, s0 + 16, r0, r1, tig, a.scale_log2, x[1][0], x[1][1]);
    else x[1][0] = x[1][1] = -INFINITY;
  }
  if constexpr (!FULL) {
    if (r0 >= nv) x[0][0] = -INFINITY;
    if (r1 >= nv) x[0][1] = -INFINITY;
    if (16 + r0 >= nv) x[1][0] = -INFINITY;
    if (16 + r1 >= nv) x[1][1] = -INFINITY;
  }
  // ------------------------------------------------------ online softmax
  float mloc = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
  if (__any_sync(kFull, mloc > S.m)) {
    mloc = fmaxf(mloc, __shfl_xor_sync(kFull, mloc, 4));
    mloc = fmaxf(mloc, __shfl_xor_sync(kFull, mloc, 8));
    mloc = fmaxf(mloc, __shfl_xor_sync(kFull, mloc, 16));
    const float alpha = ex2(S.m - mloc);  // 0 while S.m is -inf
    S.l *= alpha;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) S.acc[mt][e] *= alpha;
#pragma unroll
    for (int e = 0; e < 4; ++e) S.accz[e] *= alpha;
    S.m = mloc;
  }
  uint32_t pp[2][2];  // B rows k = 2 tig, 2 tig + 1 | 2 tig + 8, 2 tig + 9 of each half
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const float p0 = ex2(x[h][0] - S.m), p1 = ex2(x[h][1] - S.m);
    S.l += p0 + p1;
    pp[h][0] = movm_trans(pack_half2(p0, p0));
    pp[h][1] = movm_trans(pack_half2(p1, p1));
  }
  const int ta = sigma(2 * tig), tb = sigma(2 * tig + 1), tc = sigma(2 * tig + 8), td = sigma(2 * tig + 9);
  // ------------------------------------------------------------------ PV
  if constexpr (VQ) {
    constexpr int RB = D * B / 8;
    constexpr int NW = B / 2;  // words per token for the thread's 16 channels
    // HQ = 1: column n = gid is the scale (n < 4) or the zero (n >= 4) of
    // group n & 3, and one all-ones MMA sums the zero columns.  HQ = 4:
    // column n = gid is head n / 2 and group n & 1 (group 0 when d/G = 1);
    // the scales go to the code MMAs and the zeros to the all-ones MMA.
    const int ngv = D >> a.log2Gv;
    const uint16_t* sp;
    const uint16_t* zp = nullptr;
    const uint16_t* szp = nullptr;  // integer zero points: the scales beside the zero slots read
    int stride;
    if constexpr (HQ == 1) {
      const int g = gid & 3;
      if (g < ngv) {
        sp = reinterpret_cast<const uint16_t*>(stage + (gid < 4 ? r.vs_off : r.vz_off)) + (s0 * ngv + g);
        if (gid >= 4) szp = reinterpret_cast<const uint16_t*>(stage + r.vs_off) + (s0 * ngv + g);
        stride = ngv;
      } else {
        sp = reinterpret_cast<const uint16_t*>(sm + SM::zero);
        stride = 0;
      }
    } else {
      const int g = ngv == 1 ? 0 : (gid & 1);
      sp = reinterpret_cast<const uint16_t*>(stage + r.vs_off) + (s0 * ngv + g);
      zp = reinterpret_cast<const uint16_t*>(stage + r.vz_off) + (s0 * ngv + g);
      szp = sp;
      stride = ngv;
    }
    const bool zint = a.intz && szp != nullptr;
    uint32_t bv[2][2], bz[2][2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int o = 16 * h;
      const uint32_t ka = (FULL || o + ta < nv) ? 0xffffu : 0u, kb = (FULL || o + tb < nv) ? 0xffffu : 0u;
      const uint32_t kc = (FULL || o + tc < nv) ? 0xffffu : 0u, kd = (FULL || o + td < nv) ? 0xffffu : 0u;
      // padding tokens: p = 0, and their stale scale bits must not make NaN
      const uint32_t e[4] = {sp[(o + ta) * stride] & ka, sp[(o + tb) * stride] & kb,
                             sp[(o + tc) * stride] & kc, sp[(o + td) * stride] & kd};
      if (HQ == 1 && zint) {  // columns 4..7: p times the additive zero -s z, one rounding
        bv[h][0] = p_times_zero(pp[h][0], e[0], e[1], szp[(o + ta) * stride] & ka, szp[(o + tb) * stride] & kb);
        bv[h][1] = p_times_zero(pp[h][1], e[2], e[3], szp[(o + tc) * stride] & kc, szp[(o + td) * stride] & kd);
      } else {
        bv[h][0] = hmul2u(pp[h][0], halves(e[0], e[1]));
        bv[h][1] = hmul2u(pp[h][1], halves(e[2], e[3]));
      }
      if constexpr (HQ != 1) {
        const uint32_t f[4] = {zp[(o + ta) * stride] & ka, zp[(o + tb) * stride] & kb,
                               zp[(o + tc) * stride] & kc, zp[(o + td) * stride] & kd};
        if (zint) {
          bz[h][0] = p_times_zero(pp[h][0], f[0], f[1], e[0], e[1]);
          bz[h][1] = p_times_zero(pp[h][1], f[2], f[3], e[2], e[3]);
        } else {
          bz[h][0] = hmul2u(pp[h][0], halves(f[0], f[1]));
          bz[h][1] = hmul2u(pp[h][1], halves(f[2], f[3]));
        }
      } else {
        bz[h][0] = bv[h][0];
        bz[h][1] = bv[h][1];
      }
    }
    const uint8_t* vc = stage + r.v_off + s0 * RB + gid * (NW * 4);
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      uint32_t lo1[2], hi1[2], lo2[2], hi2[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint8_t* vh = vc + 16 * h * RB + 4 * w;
        const uint32_t wa = *reinterpret_cast<const uint32_t*>(vh + ta * RB);
        const uint32_t wb = *reinterpret_cast<const uint32_t*>(vh + tb * RB);
        const uint32_t wc = *reinterpret_cast<const uint32_t*>(vh + tc * RB);
        const uint32_t wd = *reinterpret_cast<const uint32_t*>(vh + td * RB);
        lo1[h] = __byte_perm(wa, wb, 0x5410);
        hi1[h] = __byte_perm(wa, wb, 0x7632);
        lo2[h] = __byte_perm(wc, wd, 0x5410);
        hi2[h] = __byte_perm(wc, wd, 0x7632);
      }
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int j = 0; j < PH; ++j) {
          const int mt = w * PH + j;
          mma16816(S.acc[mt], Fields<B>::get(lo1[h], lo1[h] >> 6, j), Fields<B>::get(hi1[h], hi1[h] >> 6, j),
                   Fields<B>::get(lo2[h], lo2[h] >> 6, j), Fields<B>::get(hi2[h], hi2[h] >> 6, j), bv[h][0], bv[h][1]);
        }
    }
    constexpr uint32_t ONES = 0x3C003C00u;  // (1.0, 1.0)
    mma16816(S.accz, ONES, ONES, ONES, ONES, bz[0][0], bz[0][1]);
    mma16816(S.accz, ONES, ONES, ONES, ONES, bz[1][0], bz[1][1]);
  } else {
    // fp16 ring V: B = p in every column; A rows are the same channels as
    // for packed V, gathered from the thread's 16 channels of each token
    if (!S.vring) {
      unscale_acc<B>(S);
      S.vring = true;
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int o = 16 * h;
      if (!FULL && o >= nv) break;
      // thread gid's 16 channels of tokens ta, tb, tc, td: 32-bit words (channel
      // pairs) read per m-tile to keep few registers live; padding tokens'
      // stale bytes (possibly NaN) are replaced by zeros
      const uint8_t* vr = stage + r.v_off + (s0 + o) * (D * 2) + gid * 32;
      const uint32_t* va = reinterpret_cast<const uint32_t*>(vr + ta * (D * 2));
      const uint32_t* vb = reinterpret_cast<const uint32_t*>(vr + tb * (D * 2));
      const uint32_t* vcc = reinterpret_cast<const uint32_t*>(vr + tc * (D * 2));
      const uint32_t* vd = reinterpret_cast<const uint32_t*>(vr + td * (D * 2));
      const uint32_t ma = (FULL || o + ta < nv) ? 0xffffffffu : 0u, mb = (FULL || o + tb < nv) ? 0xffffffffu : 0u;
      const uint32_t mc = (FULL || o + tc < nv) ? 0xffffffffu : 0u, md = (FULL || o + td < nv) ? 0xffffffffu : 0u;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        int c0, c8, p;
        v_rows<B>(0, mt, &c0, &c8, &p);  // offsets inside the thread's 16 channels
        const uint32_t s0sel = (c0 & 1) ? 0x7632u : 0x5410u;
        const uint32_t s8sel = (c8 & 1) ? 0x7632u : 0x5410u;
        mma16816(S.acc[mt], __byte_perm(va[c0 >> 1] & ma, vb[c0 >> 1] & mb, s0sel),
                 __byte_perm(va[c8 >> 1] & ma, vb[c8 >> 1] & mb, s8sel),
                 __byte_perm(vcc[c0 >> 1] & mc, vd[c0 >> 1] & md, s0sel),
                 __byte_perm(vcc[c8 >> 1] & mc, vd[c8 >> 1] & md, s8sel), pp[h][0], pp[h][1]);
      }
    }
  }
}

// The 32-token units j, j + NCW, ... of one staged tile (only the last unit
// of a tile can be partial).  Returns this warp's first unit of the next
// tile: the units are dealt out round-robin across tiles.
template <int B, int HQ, bool KQ, bool VQ>
__device__ __forceinline__ int run_tile(const DecodeArgs& a, int st, const TcRec& r, int j, int lane, WarpState& S) {
  constexpr int NCW = TcCfg<HQ>::NCW;
  const int n_full = r.n >> 5, n_unit = (r.n + 31) >> 5;
  for (; j < n_full; j += NCW) sub_unit<B, HQ, KQ, VQ, true>(a, st, r, j * 32, lane, S);
  if (j < n_unit) {
    sub_unit<B, HQ, KQ, VQ, false>(a, st, r, j * 32, lane, S);
    j += NCW;
  }
  return j - n_unit;
}

// ---- eight query-head columns (HQ = 8), any mix of segment widths -----------
// Column n of every MMA is query head n (heads past gq carry zeros); lane
// (gid, tig) ends up with heads 2 tig and 2 tig + 1.  K: A = codes as in the
// other forms, B = the scaled query q_h s_c 2^-p sm_scale log2(e) as an fp16
// high part and an fp16 rest, one MMA for each (no column is left for the
// split, and fp16 alone costs about 1e-3 of the output).  V: the codes
// become exact fp16 integers (field | exponent of 2^(10 - p), minus 2^(10 - p))
// and are scaled by their token's fp16 scale (one rounding), so A carries the
// dequantized values minus the zero points and B = p of the 8 heads; one more
// MMA with A = the zero points of the lane's V group adds sum_t p_t z_t.
// The V accumulator rows follow the field order of the V width (v_rows<B>);
// when a piece moves to a segment of another width the rows are permuted.

struct WarpState8 {
  float m[2];       // running max of heads 2 tig, 2 tig + 1 (log2 domain)
  float l[2];       // sum of p over this lane's rows, per head
  float acc[8][4];  // m-tile mt: rows gid / gid + 8 under row map cm x the two heads
  float accz[4];    // sum_t p_t z_t of the lane's V group (rows alike) x the two heads
  int cm;           // row map in use: V width 2, 4 or 8; 0 before the first tile
};

__device__ __forceinline__ void reset_state(WarpState8& S) {
  S.m[0] = S.m[1] = -INFINITY;
  S.l[0] = S.l[1] = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) S.acc[i][e] = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) S.accz[e] = 0.f;
  S.cm = 0;
}

// Move the accumulator rows from the field order of width F to that of T
// (a permutation inside each lane's 16 channels).
template <int F, int T>
__device__ __forceinline__ void remap_rows(float (&acc)[8][4]) {
  float v[16][2];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    int c0, c8, p;
    v_rows<F>(0, mt, &c0, &c8, &p);
    v[c0][0] = acc[mt][0];
    v[c0][1] = acc[mt][1];
    v[c8][0] = acc[mt][2];
    v[c8][1] = acc[mt][3];
  }
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    int c0, c8, p;
    v_rows<T>(0, mt, &c0, &c8, &p);
    acc[mt][0] = v[c0][0];
    acc[mt][1] = v[c0][1];
    acc[mt][2] = v[c8][0];
    acc[mt][3] = v[c8][1];
  }
}

template <int T>
__device__ __forceinline__ void remap_to(WarpState8& S) {
  if (S.cm != T) {
    if (S.cm == 2) remap_rows<2, T>(S.acc);
    else if (S.cm == 4) remap_rows<4, T>(S.acc);
    else if (S.cm == 8) remap_rows<8, T>(S.acc);
    S.cm = T;
  }
}

// Sum over the warp of z[h] for 8 values per lane (reduce-scatter: 11
// shuffles); lane l returns the total of head 4 b4 + 2 b3 + b2 (bits of l).
__device__ __forceinline__ float warp_sum8(const float (&z)[8], int lane) {
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
  float y[4], w[2];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float send = b4 ? z[i] : z[i + 4];
    y[i] = (b4 ? z[i + 4] : z[i]) + __shfl_xor_sync(kFull, send, 16);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float send = b3 ? y[i] : y[i + 2];
    w[i] = (b3 ? y[i + 2] : y[i]) + __shfl_xor_sync(kFull, send, 8);
  }
  float u = (b2 ? w[1] : w[0]) + __shfl_xor_sync(kFull, b2 ? w[0] : w[1], 4);
  u += __shfl_xor_sync(kFull, u, 2);
  u += __shfl_xor_sync(kFull, u, 1);
  return u;
}

// The K operand of one K group for 8 heads (column n = head n, as an fp16
// high part and the fp16 rest), built by the consuming warp: lane (ptig,
// pkt) computes the 4 channels of entries (ptig, pkt, e = 0/1) for every
// head and stores both parts; each lane then reads the 16 words of each
// part of column gid.  Returns the biases q_h . z_g (log2 domain) of heads
// 2 tig and 2 tig + 1.
template <int B>
__device__ __forceinline__ float2 build_k_operand8(const DecodeArgs& a, const uint8_t* stage, const __half* qs,
                                                   const TcRec& r, int gl, uint32_t* scratch, int lane,
                                                   uint32_t (&bq)[16], uint32_t (&bl)[16]) {
  const int ptig = lane >> 3, pkt = lane & 7;
  const __half* sg = reinterpret_cast<const __half*>(stage + r.ks_off) + gl * D;
  const __half* zg = reinterpret_cast<const __half*>(stage + r.kz_off) + gl * D;
  int cs[4];
  float sv[4];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    int clo, chi, p;
    k_half2_channels<B>(ptig, 2 * pkt + e, &clo, &chi, &p);
    cs[2 * e] = clo;
    cs[2 * e + 1] = chi;
    const float f = __uint_as_float((uint32_t)(127 - p) << 23) * a.scale_log2;  // 2^-p sm_scale log2(e)
    sv[2 * e] = __half2float(sg[clo]) * f;
    sv[2 * e + 1] = __half2float(sg[chi]) * f;
  }
  float z[8];
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    const bool live = h < a.gq;
    const __half* qh = qs + h * D;
    float hi[4], lo[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float v = live ? __half2float(qh[cs[e]]) * sv[e] : 0.f;
      hi[e] = __half2float(__float2half_rn(v));
      lo[e] = v - hi[e];
    }
    // scratch entry (k-tile pair pkt / 2, column 2 h + part, tig): kt even (b0, b1), then kt odd
    *reinterpret_cast<uint2*>(scratch + (((pkt >> 1) * 16 + 2 * h) * 4 + ptig) * 4 + (pkt & 1) * 2) =
        make_uint2(pack_half2(hi[0], hi[1]), pack_half2(hi[2], hi[3]));
    *reinterpret_cast<uint2*>(scratch + (((pkt >> 1) * 16 + 2 * h + 1) * 4 + ptig) * 4 + (pkt & 1) * 2) =
        make_uint2(pack_half2(lo[0], lo[1]), pack_half2(lo[2], lo[3]));
    float zs = 0.f;
    if (live) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        zs = fmaf(__half2float(qh[lane + 32 * i]),
                  zero_add(__half_as_ushort(zg[lane + 32 * i]), __half_as_ushort(sg[lane + 32 * i]), a.intz), zs);
    }
    z[h] = zs;
  }
  const float zh = warp_sum8(z, lane);  // head of lane l: 4 b4 + 2 b3 + b2, i.e. lane l / 4
  __syncwarp();
  const int gid = lane >> 2, tig = lane & 3;
  const uint4* tb = reinterpret_cast<const uint4*>(scratch) + 2 * gid * 4 + tig;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    *reinterpret_cast<uint4*>(&bq[4 * k]) = tb[k * 64];
    *reinterpret_cast<uint4*>(&bl[4 * k]) = tb[k * 64 + 4];
  }
  __syncwarp();  // scratch reads done before the next unit rewrites it
  const float b0 = __shfl_sync(kFull, zh, 8 * tig), b1 = __shfl_sync(kFull, zh, 8 * tig + 4);
  return make_float2(b0 * a.scale_log2, b1 * a.scale_log2);
}

// Scores (log2 domain) of rows gid, gid + 8 of the 16-token half at s0,
// heads 2 tig and 2 tig + 1: x = (row gid: h0, h1, row gid + 8: h0, h1).
template <int B>
__device__ __forceinline__ float4 k_scores8_packed(const uint8_t* kc, int s0, int r0, int r1, const uint32_t (&bq)[16],
                                                   const uint32_t (&bl)[16], float2 bias) {
  constexpr int PH = 16 / B;
  constexpr int RB = D * B / 8;
  constexpr int NW = B;
  constexpr int WPC = NW < 4 ? NW : 4;
  constexpr int NCH = NW / WPC;
  float sc[4] = {0.f, 0.f, 0.f, 0.f};  // high parts
  float sl[4] = {0.f, 0.f, 0.f, 0.f};  // low parts
#pragma unroll
  for (int ch = 0; ch < NCH; ++ch) {
    uint32_t w0[WPC], w1[WPC];
    if constexpr (WPC == 2) {
      const uint2 u0 = *reinterpret_cast<const uint2*>(kc + (s0 + r0) * RB);
      const uint2 u1 = *reinterpret_cast<const uint2*>(kc + (s0 + r1) * RB);
      w0[0] = u0.x; w0[1] = u0.y;
      w1[0] = u1.x; w1[1] = u1.y;
    } else {
      const uint4 u0 = *reinterpret_cast<const uint4*>(kc + (s0 + r0) * RB + 16 * ch);
      const uint4 u1 = *reinterpret_cast<const uint4*>(kc + (s0 + r1) * RB + 16 * ch);
      w0[0] = u0.x; w0[1] = u0.y; w0[2] = u0.z; w0[3] = u0.w;
      w1[0] = u1.x; w1[1] = u1.y; w1[2] = u1.z; w1[3] = u1.w;
    }
#pragma unroll
    for (int kk = 0; kk < 8 / NCH; ++kk) {
      const int kt = ch * (8 / NCH) + kk;
      uint32_t av[4];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int h = 2 * kt + e;
        const int w = h / PH - ch * WPC, j = h % PH;
        av[2 * e + 0] = Fields<B>::get(w0[w], w0[w] >> 6, j);
        av[2 * e + 1] = Fields<B>::get(w1[w], w1[w] >> 6, j);
      }
      mma16816(sc, av[0], av[1], av[2], av[3], bq[2 * kt], bq[2 * kt + 1]);
      mma16816(sl, av[0], av[1], av[2], av[3], bl[2 * kt], bl[2 * kt + 1]);
    }
  }
  return make_float4(fmaf(sc[0] + sl[0], 16777216.0f, bias.x), fmaf(sc[1] + sl[1], 16777216.0f, bias.y),
                     fmaf(sc[2] + sl[2], 16777216.0f, bias.x), fmaf(sc[3] + sl[3], 16777216.0f, bias.y));
}

// Same for fp16 ring K; qt = the query of head gid (column gid).
__device__ __forceinline__ float4 k_scores8_ring(const uint8_t* kr, const uint8_t* qt, uint32_t qmask, int s0, int r0,
                                                 int r1, int tig, float scale_log2) {
  float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int kc = 0; kc < 4; ++kc) {
    const int off = ((kc + tig) & 3) * 16;
    const uint4 u0 = *reinterpret_cast<const uint4*>(kr + (s0 + r0) * (D * 2) + off);
    const uint4 u1 = *reinterpret_cast<const uint4*>(kr + (s0 + r1) * (D * 2) + off);
    const uint4 qw = *reinterpret_cast<const uint4*>(qt + off);
    mma16816(sc, u0.x, u1.x, u0.y, u1.y, qw.x & qmask, qw.y & qmask);
    mma16816(sc, u0.z, u1.z, u0.w, u1.w, qw.z & qmask, qw.w & qmask);
  }
  return make_float4(sc[0] * scale_log2, sc[1] * scale_log2, sc[2] * scale_log2, sc[3] * scale_log2);
}

__device__ __forceinline__ uint32_t hsub2u(uint32_t a, uint32_t b) {
  const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// Code field j of both halves as exact fp16 integers.
template <int B>
__device__ __forceinline__ uint32_t code_int2(uint32_t x, int j) {
  const int p = Fields<B>::pos(j);
  const uint32_t magic = (uint32_t)(25 - p) << 10;  // fp16 2^(10 - p): field f at bit p reads 2^(10 - p) + f
  const uint32_t h = Fields<B>::get(x, x >> 6, j) | (magic | (magic << 16));
  return hsub2u(h, magic | (magic << 16));
}

// One 32-token unit [s0, s0 + 32) for 8 head columns.  BK / BV: packed
// width of K / V (2, 4, 8) or 0 for the fp16 ring.  The V rows are laid out
// in the field order of width CM (BV for packed V; the ring takes any).
template <int BK, int BV, int CM, bool FULL>
__device__ __forceinline__ void sub_unit8(const DecodeArgs& a, int st, const TcRec& r, int s0, int lane,
                                          WarpState8& S) {
  using SM = TcSmem<8>;
  const int gid = lane >> 2, tig = lane & 3;
  const int r0 = sigma(gid), r1 = sigma(gid + 8);
  uint8_t* const sm = tc_smem();
  const uint8_t* const stage = sm + SM::stages + st * kTcStageBytes;
  const int nv = r.n - s0;  // valid tokens from s0 (>= 32 when FULL)
  // ------------------------------------------------------------- scores
  float4 x[2];  // [half] (row gid: h0, h1, row gid + 8: h0, h1)
  if constexpr (BK != 0) {
    const int gl = (r.kr0 + s0) >> a.log2G;
    uint32_t bq[16], bl[16];
    const float2 bias = build_k_operand8<BK>(
        a, stage, reinterpret_cast<const __half*>(sm + SM::q + st * 8 * D * 2), r, gl,
        reinterpret_cast<uint32_t*>(sm + SM::ktab) + (threadIdx.x >> 5) * (TcCfg<8>::KTAB / 4), lane, bq, bl);
    const uint8_t* kc = stage + r.k_off + tig * (BK * 4);
    x[0] = k_scores8_packed<BK>(kc, s0, r0, r1, bq, bl, bias);
    if (FULL || nv > 16) x[1] = k_scores8_packed<BK>(kc, s0 + 16, r0, r1, bq, bl, bias);
    else x[1] = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
  } else {
    const uint8_t* qt = sm + SM::q + (st * 8 + gid) * D * 2 + tig * 64;
    const uint32_t qmask = gid < a.gq ? 0xffffffffu : 0u;
    const uint8_t* kr = stage + r.k_off + tig * 64;
    x[0] = k_scores8_ring(kr, qt, qmask, s0, r0, r1, tig, a.scale_log2);
    if (FULL || nv > 16) x[1] = k_scores8_ring(kr, qt, qmask, s0 + 16, r0, r1, tig, a.scale_log2);
    else x[1] = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
  }
  if constexpr (!FULL) {
    if (r0 >= nv) x[0].x = x[0].y = -INFINITY;
    if (r1 >= nv) x[0].z = x[0].w = -INFINITY;
    if (16 + r0 >= nv) x[1].x = x[1].y = -INFINITY;
    if (16 + r1 >= nv) x[1].z = x[1].w = -INFINITY;
  }
  // ------------------------------------------------------ online softmax
  // every head has a valid row in the unit, so the maxima are finite
  float m0 = fmaxf(fmaxf(x[0].x, x[0].z), fmaxf(x[1].x, x[1].z));
  float m1 = fmaxf(fmaxf(x[0].y, x[0].w), fmaxf(x[1].y, x[1].w));
  if (__any_sync(kFull, m0 > S.m[0] || m1 > S.m[1])) {
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      m0 = fmaxf(m0, __shfl_xor_sync(kFull, m0, off));
      m1 = fmaxf(m1, __shfl_xor_sync(kFull, m1, off));
    }
    m0 = fmaxf(m0, S.m[0]);
    m1 = fmaxf(m1, S.m[1]);
    const float al0 = ex2(S.m[0] - m0), al1 = ex2(S.m[1] - m1);  // 0 while S.m is -inf
    S.l[0] *= al0;
    S.l[1] *= al1;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      S.acc[mt][0] *= al0;
      S.acc[mt][1] *= al1;
      S.acc[mt][2] *= al0;
      S.acc[mt][3] *= al1;
    }
    S.accz[0] *= al0;
    S.accz[1] *= al1;
    S.accz[2] *= al0;
    S.accz[3] *= al1;
    S.m[0] = m0;
    S.m[1] = m1;
  }
  uint32_t pp[2][2];  // B of the V MMAs: head gid, token rows 2 tig.. | 2 tig + 8..
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const float p00 = ex2(x[h].x - S.m[0]), p01 = ex2(x[h].y - S.m[1]);
    const float p10 = ex2(x[h].z - S.m[0]), p11 = ex2(x[h].w - S.m[1]);
    S.l[0] += p00 + p10;
    S.l[1] += p01 + p11;
    pp[h][0] = movm_trans(pack_half2(p00, p01));
    pp[h][1] = movm_trans(pack_half2(p10, p11));
  }
  const int ta = sigma(2 * tig), tb = sigma(2 * tig + 1), tc = sigma(2 * tig + 8), td = sigma(2 * tig + 9);
  // ------------------------------------------------------------------ PV
  if constexpr (BV != 0) {
    static_assert(BV == CM, "packed V rows follow their own width");
    constexpr int RB = D * BV / 8;
    constexpr int NW = BV / 2;  // words per token for the thread's 16 channels
    constexpr int PH = 16 / BV;
    const int ngv = D >> a.log2Gv;
    const int g = (16 * gid) >> a.log2Gv;  // the lane's V group
    const uint16_t* sp = reinterpret_cast<const uint16_t*>(stage + r.vs_off) + s0 * ngv + g;
    const uint16_t* zp = reinterpret_cast<const uint16_t*>(stage + r.vz_off) + s0 * ngv + g;
    uint32_t sv[2][2], zv[2][2];  // [half][tokens (ta, tb) | (tc, td)]
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int o = 16 * h;
      // padding tokens: their stale scale / zero bits must not make NaN
      const uint32_t ka = (FULL || o + ta < nv) ? 0xffffu : 0u, kb = (FULL || o + tb < nv) ? 0xffffu : 0u;
      const uint32_t kc = (FULL || o + tc < nv) ? 0xffffu : 0u, kd = (FULL || o + td < nv) ? 0xffffu : 0u;
      sv[h][0] = halves(sp[(o + ta) * ngv] & ka, sp[(o + tb) * ngv] & kb);
      sv[h][1] = halves(sp[(o + tc) * ngv] & kc, sp[(o + td) * ngv] & kd);
      uint32_t f[4] = {zp[(o + ta) * ngv] & ka, zp[(o + tb) * ngv] & kb, zp[(o + tc) * ngv] & kc,
                       zp[(o + td) * ngv] & kd};
      if (a.intz) {  // the additive zero -s z of the integer zero point
        f[0] = zero_add_h(f[0], sp[(o + ta) * ngv] & ka, true);
        f[1] = zero_add_h(f[1], sp[(o + tb) * ngv] & kb, true);
        f[2] = zero_add_h(f[2], sp[(o + tc) * ngv] & kc, true);
        f[3] = zero_add_h(f[3], sp[(o + td) * ngv] & kd, true);
      }
      zv[h][0] = halves(f[0], f[1]);
      zv[h][1] = halves(f[2], f[3]);
    }
    const uint8_t* vc = stage + r.v_off + s0 * RB + gid * (NW * 4);
#pragma unroll
    for (int w = 0; w < NW; ++w) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint8_t* vh = vc + 16 * h * RB + 4 * w;
        const uint32_t wa = *reinterpret_cast<const uint32_t*>(vh + ta * RB);
        const uint32_t wb = *reinterpret_cast<const uint32_t*>(vh + tb * RB);
        const uint32_t wc = *reinterpret_cast<const uint32_t*>(vh + tc * RB);
        const uint32_t wd = *reinterpret_cast<const uint32_t*>(vh + td * RB);
        const uint32_t lo1 = __byte_perm(wa, wb, 0x5410), hi1 = __byte_perm(wa, wb, 0x7632);
        const uint32_t lo2 = __byte_perm(wc, wd, 0x5410), hi2 = __byte_perm(wc, wd, 0x7632);
#pragma unroll
        for (int j = 0; j < PH; ++j) {
          const int mt = w * PH + j;
          mma16816(S.acc[mt], hmul2u(code_int2<BV>(lo1, j), sv[h][0]), hmul2u(code_int2<BV>(hi1, j), sv[h][0]),
                   hmul2u(code_int2<BV>(lo2, j), sv[h][1]), hmul2u(code_int2<BV>(hi2, j), sv[h][1]), pp[h][0],
                   pp[h][1]);
        }
      }
    }
    mma16816(S.accz, zv[0][0], zv[0][0], zv[0][1], zv[0][1], pp[0][0], pp[0][1]);
    mma16816(S.accz, zv[1][0], zv[1][0], zv[1][1], zv[1][1], pp[1][0], pp[1][1]);
  } else {
    // fp16 ring V: A rows are the channels of row map CM, gathered from the
    // thread's 16 channels of each token; padding tokens read as zeros
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int o = 16 * h;
      if (!FULL && o >= nv) break;
      const uint8_t* vr = stage + r.v_off + (s0 + o) * (D * 2) + gid * 32;
      const uint32_t* va = reinterpret_cast<const uint32_t*>(vr + ta * (D * 2));
      const uint32_t* vb = reinterpret_cast<const uint32_t*>(vr + tb * (D * 2));
      const uint32_t* vcc = reinterpret_cast<const uint32_t*>(vr + tc * (D * 2));
      const uint32_t* vd = reinterpret_cast<const uint32_t*>(vr + td * (D * 2));
      const uint32_t ma = (FULL || o + ta < nv) ? 0xffffffffu : 0u, mb = (FULL || o + tb < nv) ? 0xffffffffu : 0u;
      const uint32_t mc = (FULL || o + tc < nv) ? 0xffffffffu : 0u, md = (FULL || o + td < nv) ? 0xffffffffu : 0u;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        int c0, c8, p;
        v_rows<CM>(0, mt, &c0, &c8, &p);
        const uint32_t s0sel = (c0 & 1) ? 0x7632u : 0x5410u;
        const uint32_t s8sel = (c8 & 1) ? 0x7632u : 0x5410u;
        mma16816(S.acc[mt], __byte_perm(va[c0 >> 1] & ma, vb[c0 >> 1] & mb, s0sel),
                 __byte_perm(va[c8 >> 1] & ma, vb[c8 >> 1] & mb, s8sel),
                 __byte_perm(vcc[c0 >> 1] & mc, vd[c0 >> 1] & md, s0sel),
                 __byte_perm(vcc[c8 >> 1] & mc, vd[c8 >> 1] & md, s8sel), pp[h][0], pp[h][1]);
      }
    }
  }
}

template <int BK, int BV, int CM>
__device__ __forceinline__ void run_tile8_t(const DecodeArgs& a, int st, const TcRec& r, int j, int lane,
                                            WarpState8& S) {
  constexpr int NCW = TcCfg<8>::NCW;
  remap_to<CM>(S);
  // one masked body for full and partial units: the form has many width
  // combinations, and a second body each would crowd the instruction cache
  const int n_unit = (r.n + 31) >> 5;
  for (; j < n_unit; j += NCW) sub_unit8<BK, BV, CM, false>(a, st, r, j * 32, lane, S);
}

// Tile dispatch on the widths it carries (the host admits only these forms:
// K and V packed at one width, K packed with ring V, or both from the ring).
__device__ __forceinline__ void run_tile8(const DecodeArgs& a, int st, const TcRec& r, int j, int lane,
                                          WarpState8& S) {
  if (r.vq) {
    if (r.vb == 2) run_tile8_t<2, 2, 2>(a, st, r, j, lane, S);
    else if (r.vb == 4) run_tile8_t<4, 4, 4>(a, st, r, j, lane, S);
    else run_tile8_t<8, 8, 8>(a, st, r, j, lane, S);
  } else {
    if (!r.kq) {
      run_tile8_t<0, 0, 2>(a, st, r, j, lane, S);  // ring tiles take the 2-bit row map
    } else if (r.kb == 2) {
      run_tile8_t<2, 0, 2>(a, st, r, j, lane, S);
    } else if (r.kb == 4) {
      run_tile8_t<4, 0, 4>(a, st, r, j, lane, S);
    } else {
      run_tile8_t<8, 0, 8>(a, st, r, j, lane, S);
    }
  }
}

// Leave a warp's partial (o, m, l) of both its heads in its merge rows
// [head][REC]: channels of the lane's rows under row map cm.
template <int CM>
__device__ __forceinline__ void write_partial8_t(const WarpState8& S, float* rows, const float (&l)[2], int gid,
                                                 int tig) {
  constexpr int REC = D + 2;
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    float* mg = rows + (2 * tig + hh) * REC;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      int c0, c8, p;
      v_rows<CM>(gid, mt, &c0, &c8, &p);
      mg[c0] = S.acc[mt][hh] + S.accz[hh];
      mg[c8] = S.acc[mt][2 + hh] + S.accz[2 + hh];
    }
    if (gid == 0) {
      mg[D] = S.m[hh];
      mg[D + 1] = l[hh];
    }
  }
}

__device__ __forceinline__ void write_partial8(const DecodeArgs&, const WarpState8& S, float* rows, int gid,
                                               int tig) {
  float l[2] = {S.l[0], S.l[1]};
#pragma unroll
  for (int hh = 0; hh < 2; ++hh)
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) l[hh] += __shfl_xor_sync(kFull, l[hh], off);
  if (S.cm == 4) write_partial8_t<4>(S, rows, l, gid, tig);
  else if (S.cm == 8) write_partial8_t<8>(S, rows, l, gid, tig);
  else write_partial8_t<2>(S, rows, l, gid, tig);  // also a warp without tiles: zeros
}

// Overloads so that the state of the 1/4-head forms has the same interface.
__device__ __forceinline__ void write_partial8(const DecodeArgs&, const WarpState&, float*, int, int) {}

// End of a warp's share of one pair inside this CTA's range (the CTA's k-th
// piece).  The warp leaves its partial (o, m, l) in merge slot k % NSLOT and
// goes on; the last of the NCW warps to arrive combines them and writes the
// output (the pair lies in this range only) or the CTA's record; for a split
// pair the last record to arrive merges all records.  No CTA-wide barrier:
// warps that have drifted apart by a few tiles do not wait for each other.
// Slot reuse: warps are at most NS tiles apart (the stage ring), each piece
// has at least one tile, and the merger of piece k is its last warp, so a
// warp reaching piece k + NSLOT waits (bounded) only if fewer than NSLOT
// slots separate it from a merge still running.
template <int B, int HQ, class State>
__device__ void finish_piece(const DecodeArgs& a, uint8_t* smem, int pair, int piece, int warp,
                             int lane, State& S, volatile int* flags) {
  using SM = TcSmem<HQ>;
  constexpr int NCW = TcCfg<HQ>::NCW, NSLOT = TcCfg<HQ>::NSLOT;
  constexpr int REC = D + 2;  // (o[D], m, l)
  const int gid = lane >> 2, tig = lane & 3;
  const int slot = piece % NSLOT;
  volatile int* owner = reinterpret_cast<volatile int*>(smem + SM::slot_owner);
  int* count = reinterpret_cast<int*>(smem + SM::slot_count);
  // wait until the slot serves this piece (its previous piece merged)
  if (owner[slot] != piece) {
    const long long t0 = clock64();
    while (owner[slot] != piece) {
      if (flags[0] || clock64() - t0 > (1ll << 31)) {
        flags[0] = 1;
        break;
      }
      __nanosleep(64);
    }
  }
  __syncwarp();
  float* slot_base = reinterpret_cast<float*>(smem + SM::merge) + slot * NCW * HQ * REC;
  if constexpr (HQ == 8) {
    write_partial8(a, S, slot_base + warp * 8 * REC, gid, tig);
  } else {
    float* mg = slot_base + (warp * HQ + (HQ == 1 ? 0 : tig)) * REC;  // this lane's head
    if (!S.vring) unscale_acc<B>(S);
    float l = S.l;  // a lane's rows cover gid: sum over gid (lanes of one tig)
    l += __shfl_xor_sync(kFull, l, 4);
    l += __shfl_xor_sync(kFull, l, 8);
    l += __shfl_xor_sync(kFull, l, 16);
  #pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      int c0, c8, p;
      v_rows<B>(gid, mt, &c0, &c8, &p);
      const int g = c0 >> a.log2Gv;  // c0 and c8 share their group
      if constexpr (HQ == 1) {
        // z sum of group g: column 4 + g, held by lanes with tig = 2 + g / 2
        const float z0 = __shfl_sync(kFull, S.accz[0], 2 + (g >> 1));
        const float z1 = __shfl_sync(kFull, S.accz[1], 2 + (g >> 1));
        const float zg = (g & 1) ? z1 : z0;
        if (tig == (g >> 1)) {
          mg[c0] = ((g & 1) ? S.acc[mt][1] : S.acc[mt][0]) + zg;
          mg[c8] = ((g & 1) ? S.acc[mt][3] : S.acc[mt][2]) + zg;
        }
      } else {
        // columns 2 tig + g: head tig, group g (d/G <= 2)
        const float zg = (g & 1) ? S.accz[1] : S.accz[0];
        mg[c0] = ((g & 1) ? S.acc[mt][1] : S.acc[mt][0]) + zg;
        mg[c8] = ((g & 1) ? S.acc[mt][3] : S.acc[mt][2]) + zg;
      }
    }
    if (gid == 0 && (HQ != 1 || tig == 0)) {
      mg[D] = S.m;
      mg[D + 1] = l;
    }
  }
  __threadfence_block();
  __syncwarp();
  int last_warp = 0;
  if (lane == 0) last_warp = atomicAdd(&count[slot], 1) == NCW - 1;
  if (!__shfl_sync(kFull, last_warp, 0)) return;
  __threadfence_block();
  // this warp merges the slot, head by head: lane owns channels lane + 32 i
  const int nh = HQ == 1 ? 1 : a.gq;
  float M[HQ], L[HQ], O[HQ][D / 32];
#pragma unroll
  for (int h = 0; h < HQ; ++h) {
    M[h] = -INFINITY;
    L[h] = 0.f;
#pragma unroll
    for (int i = 0; i < D / 32; ++i) O[h][i] = 0.f;
    if (h >= nh) continue;
    for (int w = 0; w < NCW; ++w) M[h] = fmaxf(M[h], slot_base[(w * HQ + h) * REC + D]);
    for (int w = 0; w < NCW; ++w) {
      const float* mw = slot_base + (w * HQ + h) * REC;
      const float sw = (mw[D] == -INFINITY) ? 0.f : exp2f(mw[D] - M[h]);
      L[h] += mw[D + 1] * sw;
#pragma unroll
      for (int i = 0; i < D / 32; ++i) O[h][i] += mw[lane + 32 * i] * sw;
    }
  }
  // the slot is free for piece + NSLOT
  __syncwarp();
  if (lane == 0) {
    count[slot] = 0;
    __threadfence_block();
    owner[slot] = piece + NSLOT;
  }
  const bool ok = flags[0] == 0;
  if (!ok) {
    if (lane == 0) atomicExch(a.err, 1);
    return;
  }
  const long long nt = a.n_tiles;
  const int* bound = reinterpret_cast<const DecodeArgs*>(smem + SM::args)->tc_bound;
  const int first = a.tc_whole ? pair : tc_owner(bound, a.n_cta, (long long)pair * nt);
  const int last = a.tc_whole ? pair : tc_owner(bound, a.n_cta, (long long)pair * nt + nt - 1);
  const int pieces = last - first + 1;
  const size_t out_base = (size_t)pair * nh * D;  // heads of a pair are consecutive query heads
  if (pieces == 1) {
#pragma unroll
    for (int h = 0; h < HQ; ++h)
      if (h < nh)
#pragma unroll
        for (int i = 0; i < D / 32; ++i) a.out[out_base + h * D + lane + 32 * i] = __float2half_rn(L[h] > 0.f ? O[h][i] / L[h] : 0.f);
    return;
  }
  // records [pair][piece][head][REC]
  float* rec = a.part + ((size_t)pair * a.n_splits + (blockIdx.x - first)) * nh * REC;
#pragma unroll
  for (int h = 0; h < HQ; ++h) {
    if (h >= nh) continue;
#pragma unroll
    for (int i = 0; i < D / 32; ++i) rec[h * REC + lane + 32 * i] = O[h][i];
    if (lane == 0) {
      rec[h * REC + D] = M[h];
      rec[h * REC + D + 1] = L[h];
    }
  }
  if (a.tc_defer) return;  // many records: a separate launch merges them
  __threadfence();
  __syncwarp();
  // the last record of the pair to arrive merges them all
  int last_in = 0;
  if (lane == 0) last_in = atomicAdd(&a.counters[pair], 1) == pieces - 1;
  if (!__shfl_sync(kFull, last_in, 0)) return;
  __threadfence();
  // The records are cold in L2: first the max and the weighted sum of each
  // head with the records spread over the lanes, then the outputs as sums
  // of loads that do not wait for one another.
  const float* recs = a.part + (size_t)pair * a.n_splits * nh * REC;
  float MM[HQ], IL[HQ];
#pragma unroll
  for (int h = 0; h < HQ; ++h) {
    MM[h] = -INFINITY;
    IL[h] = 0.f;
    if (h >= nh) continue;
    float m = -INFINITY;
    for (int s = lane; s < pieces; s += 32) m = fmaxf(m, __ldcg(recs + ((size_t)s * nh + h) * REC + D));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, off));
    float l = 0.f;
    for (int s = lane; s < pieces; s += 32) {
      const float* rr = recs + ((size_t)s * nh + h) * REC;
      if (m != -INFINITY) l += __ldcg(rr + D + 1) * exp2f(__ldcg(rr + D) - m);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(kFull, l, off);
    MM[h] = m;
    IL[h] = l > 0.f ? 1.f / l : 0.f;  // l = 0: a sequence with no tokens, output 0
  }
  float OO[HQ][D / 32];
#pragma unroll
  for (int h = 0; h < HQ; ++h)
#pragma unroll
    for (int i = 0; i < D / 32; ++i) OO[h][i] = 0.f;
#pragma unroll 2
  for (int s = 0; s < pieces; ++s) {
#pragma unroll
    for (int h = 0; h < HQ; ++h) {
      if (h >= nh) continue;
      const float* rr = recs + ((size_t)s * nh + h) * REC;
      const float w = MM[h] == -INFINITY ? 0.f : exp2f(__ldcg(rr + D) - MM[h]) * IL[h];
#pragma unroll
      for (int i = 0; i < D / 32; ++i) OO[h][i] += __ldcg(rr + lane + 32 * i) * w;
    }
  }
#pragma unroll
  for (int h = 0; h < HQ; ++h)
    if (h < nh)
#pragma unroll
      for (int i = 0; i < D / 32; ++i) a.out[out_base + h * D + lane + 32 * i] = __float2half_rn(OO[h][i]);
  if (lane == 0) a.counters[pair] = 0;
}

// Launch arguments of a paged cache (per-sequence lengths), or nothing.
struct TcNoPaged {
  int unused;
};

// PG: a paged cache.  Every (sequence, kv head) is padded to a.n_tiles tiles
// (the longest sequence's count) so the stream-K ranges, owners and merges
// keep their uniform tile index; a padding tile (t >= the sequence's own
// count) takes no pipeline stage: the issue warp and the consumers skip it
// by the same rule.
template <int B, int HQ, bool PG>
__global__ void __launch_bounds__(TcCfg<HQ>::NTH, kTcCtasPerSm)
    decode_tc_kernel(const DecodeArgs a, const typename std::conditional<PG, PagedArgs, TcNoPaged>::type p) {
  using SM = TcSmem<HQ>;
  constexpr int NCW = TcCfg<HQ>::NCW, NTH = TcCfg<HQ>::NTH, NSLOT = TcCfg<HQ>::NSLOT, NS = TcCfg<HQ>::NS;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + SM::bars);
  uint64_t* empty = full + NS;
  volatile int* flags = reinterpret_cast<volatile int*>(smem + SM::flags);
  TcRec* recs = reinterpret_cast<TcRec*>(smem + SM::rec);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = a.batch * a.h_kv * a.n_tiles;  // below 2^31 (checked by the host)
  const int g_begin = a.tc_whole ? (int)blockIdx.x * a.n_tiles : a.tc_bound[blockIdx.x];
  const int g_end = a.tc_whole ? ((int)blockIdx.x + 1) * a.n_tiles : a.tc_bound[blockIdx.x + 1];
  const int ntiles = g_end - g_begin;

  if (tid == 0) {
    flags[0] = 0;
    flags[1] = 0;
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NCW);
    }
    mbar_fence_init();
  }
  if (tid < 16) reinterpret_cast<uint32_t*>(smem + SM::zero)[tid] = 0u;
  // a record merge launched after this grid may start launching now (it
  // waits for this grid's completion before reading the records)
  grid_dep_launch();
  if (tid < NSLOT) {
    reinterpret_cast<int*>(smem + SM::slot_owner)[tid] = tid;
    reinterpret_cast<int*>(smem + SM::slot_count)[tid] = 0;
  }
  static_assert(sizeof(DecodeArgs) % 4 == 0, "word copy");
  for (int i = tid; i < (int)(sizeof(DecodeArgs) / 4); i += NTH)
    reinterpret_cast<uint32_t*>(smem + SM::args)[i] = reinterpret_cast<const uint32_t*>(&a)[i];
  const DecodeArgs* args_s = reinterpret_cast<const DecodeArgs*>(smem + SM::args);
  __syncthreads();

  if (warp == NCW) {
    // ------------------------------------------------- bulk-copy issue warp
    // Lane l works out the record and the copies of tile j0 + l for 32 tiles
    // at once (from the shared-memory copy of the launch arguments: indexing
    // kernel parameters dynamically would go through the constant cache);
    // lane j % 32 then issues tile j, so a tile costs its copy instructions
    // only.  Copy slots: 0-2 K (codes, scales, zeros or the ring's one or two
    // pieces), 3-5 V likewise.
    const DecodeArgs& sa = *args_s;
    TcRec rec;
    int pair = 0;
    uint32_t bytes = 0;
    const void* src[6];
    uint32_t dst[6], nb[6];
    int nissued = 0;  // stages used so far (live tiles issued)
    unsigned live = 0u;  // live tiles among the 32 of the current batch
    for (int j = 0, k = 0; j < ntiles; ++j) {
      if ((j & 31) == 0) {
        const int jl = j + lane;
#pragma unroll
        for (int k = 0; k < 6; ++k) {
          src[k] = nullptr;
          dst[k] = nb[k] = 0u;
        }
        bool mine = false;
        auto fill = [&](const TileInfo& ti) {
          rec.n = ti.n;
          rec.kq = ti.kseg >= 0;
          rec.vq = ti.vseg >= 0;
          rec.kr0 = ti.ku0 & (sa.G - 1);
          rec.k_off = ti.k_off;
          rec.ks_off = ti.ks_off;
          rec.kz_off = ti.kz_off;
          rec.v_off = ti.v_off;
          rec.vs_off = ti.vs_off;
          rec.vz_off = ti.vz_off;
          rec.kb = ti.kbits;
          rec.vb = ti.vbits;
          bytes = ti.bytes + (HQ == 1 ? 1 : sa.gq) * D * 2;
        };
        if (jl < ntiles) {
          const int g = g_begin + jl;
          pair = g / sa.n_tiles;
          const int t = g - pair * sa.n_tiles;
          if constexpr (PG) {
            const int b = pair / sa.h_kv, h = pair - b * sa.h_kv;
            const PagedSeq& ps = p.seq[b];
            mine = t < ps.n_tiles;
            if (mine) {
              const TileInfo ti = paged_tile(p, ps, t);
              fill(ti);
              // a block-table entry outside the pool is not followed: page
              // 0 is read in its place and the cache's error word is set
              auto page = [&](int row) {
                const int jp = row / p.P;
                const int pg = jp < p.max_pages ? p.table[(size_t)b * p.max_pages + jp] : -1;
                if (pg < 0 || pg >= p.n_pages) {
                  atomicExch(p.page_err, 2);
                  return 0;
                }
                return pg;
              };
              for_each_paged_copy(p, b, h, ps, ti, page, [&](const void* s_, uint32_t off, uint32_t n_, int slot) {
                src[slot] = s_;
                dst[slot] = off;
                nb[slot] = n_;
              });
            }
          } else {
            mine = true;
            const TileInfo ti = tile_info(sa, t);
            fill(ti);
            bool k2 = false, v2 = false;
            for_each_tile_copy(sa, (size_t)pair, ti, [&](const void* s_, uint32_t off, uint32_t n_, int buf, int) {
              const int slot = buf < 6 ? buf : (buf == 6 ? (k2 ? 1 : 0) : (v2 ? 4 : 3));
              if (buf == 6) k2 = true;
              if (buf == 7) v2 = true;
              src[slot] = s_;
              dst[slot] = off;
              nb[slot] = n_;
            });
          }
        }
        live = __ballot_sync(kFull, mine);
      }
      if (!((live >> (j & 31)) & 1u)) continue;  // padding tile: no stage
      const int st = k % NS;
      if (k >= NS) {
        if (__any_sync(kFull, !wait_or_abort<true>(&empty[st], (uint32_t)(((k / NS) & 1) ^ 1), flags))) break;
        // consumers that gave up release a stage without waiting for it
        if (!mbar_drain_bounded(&full[st], (uint32_t)(((k / NS) & 1) ^ 1)) && lane == 0) atomicExch(sa.err, 1);
      }
      nissued = ++k;
      if (lane == (j & 31)) {
        recs[st] = rec;
        uint8_t* stage = smem + SM::stages + st * kTcStageBytes;
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(&full[st], bytes);
#pragma unroll
        for (int k = 0; k < 6; ++k)
          if (nb[k]) bulk_g2s(stage + dst[k], src[k], nb[k], &full[st]);
        const int nq = HQ == 1 ? 1 : sa.gq;  // query heads of the pair (consecutive)
        bulk_g2s(smem + SM::q + st * HQ * D * 2, sa.q + (size_t)pair * nq * D, nq * D * 2, &full[st]);
      }
      __syncwarp();
    }
    // no copy of this block may still be in flight when it exits
    for (int j = nissued > NS ? nissued - NS : 0; j < nissued; ++j)
      if (!mbar_drain_bounded(&full[j % NS], (uint32_t)((j / NS) & 1)) && lane == 0) atomicExch(sa.err, 1);
    return;
  }

  // -------------------------------------------------------------- consumers
  typename std::conditional<HQ == 8, WarpState8, WarpState>::type S;
  auto reset = [&]() { reset_state(S); };
  reset();
  int cur_pair = g_begin / a.n_tiles;
  int t_in_pair = g_begin - cur_pair * a.n_tiles;
  int piece = 0;  // pieces (pairs) of this CTA's range finished so far
  int jstart = warp;  // this warp's first sub-tile of the next tile (round-robin)
  bool aborted = false;
  auto live_tiles = [&](int pr) {
    if constexpr (PG) return p.seq[pr / a.h_kv].n_tiles;
    else return a.n_tiles;
  };
  int n_live = live_tiles(cur_pair);
  for (int it = 0, k = 0; it < ntiles; ++it) {
    if (t_in_pair == a.n_tiles) {  // first tile of the next pair
      finish_piece<B, HQ>(a, smem, cur_pair, piece++, warp, lane, S, flags);
      reset();
      ++cur_pair;
      t_in_pair = 0;
      n_live = live_tiles(cur_pair);
    }
    if (t_in_pair++ >= n_live) continue;  // padding tile: no stage
    const int st = k % NS;
    const uint32_t ph = (uint32_t)((k / NS) & 1);
    ++k;
    if (!aborted && __any_sync(kFull, !wait_or_abort<false>(&full[st], ph, flags))) aborted = true;
    if (!aborted) {
      const int4 r0 = *reinterpret_cast<const int4*>(&recs[st].n);
      const int4 r1 = *reinterpret_cast<const int4*>(&recs[st].k_off);
      const int4 r2 = *reinterpret_cast<const int4*>(&recs[st].ks_off);
      TcRec r;
      r.n = r0.x;
      r.kq = r0.y;
      r.vq = r0.z;
      r.kr0 = r0.w;
      r.k_off = (uint32_t)r1.x;
      r.v_off = (uint32_t)r1.y;
      r.vs_off = (uint32_t)r1.z;
      r.vz_off = (uint32_t)r1.w;
      r.ks_off = (uint32_t)r2.x;
      r.kz_off = (uint32_t)r2.y;
      r.kb = r2.z;
      r.vb = r2.w;
      if constexpr (HQ == 8) {
        run_tile8(a, st, r, jstart, lane, S);
        jstart = (jstart - ((r.n + 31) >> 5)) % NCW;
        jstart += jstart < 0 ? NCW : 0;
      } else if (r.kq) {
        jstart = r.vq ? run_tile<B, HQ, true, true>(a, st, r, jstart, lane, S) : run_tile<B, HQ, true, false>(a, st, r, jstart, lane, S);
      } else {
        jstart = r.vq ? run_tile<B, HQ, false, true>(a, st, r, jstart, lane, S) : run_tile<B, HQ, false, false>(a, st, r, jstart, lane, S);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
  }
  if (ntiles > 0) finish_piece<B, HQ>(a, smem, cur_pair, piece, warp, lane, S, flags);
}

template <int B, int HQ, bool PG = false, class PA = TcNoPaged>
cudaError_t launch_tc_b(const DecodeArgs& a, cudaStream_t s, const PA& p = PA{}) {
  const int smem = TcSmem<HQ>::total;
  cudaError_t e = set_smem_once((const void*)decode_tc_kernel<B, HQ, PG>, smem);
  if (e != cudaSuccess) return e;
  decode_tc_kernel<B, HQ, PG><<<a.n_cta, TcCfg<HQ>::NTH, smem, s>>>(a, p);
  return cudaGetLastError();
}

template <int HQ, bool PG = false, class PA = TcNoPaged>
cudaError_t launch_tc_hq(const DecodeArgs& a, int bits, cudaStream_t s, const PA& p = PA{}) {
  if (bits == 2) return launch_tc_b<2, HQ, PG>(a, s, p);
  if (bits == 4) return launch_tc_b<4, HQ, PG>(a, s, p);
  return launch_tc_b<8, HQ, PG>(a, s, p);
}

// Merge of a pair's partial records in a launch of its own (many records):
// block (pair, head) of 4 x 128 threads.  The records' weights
// 2^(m_s - M) / L first (threads over records), then channel c = thread % 128
// summed over a quarter of the records by each of the 4 thread groups.
constexpr int kMergeThreads = 1024;
constexpr int kMergeGroups = kMergeThreads / D;  // record groups: thread (k, c) sums records k, k + 8, ...
constexpr int kMergeRegs = 10;                    // records a thread holds per pass

// Merge of one (pair, head)'s records.  Every load of a pass is issued
// before any is used: the (m, l) of the records (one per thread) and each
// thread's o values of up to kMergeRegs records, so a pass costs one round
// trip to L2; the weights then need two block reductions.
__global__ void __launch_bounds__(kMergeThreads) merge_tc_kernel(const DecodeArgs a) {
  constexpr int REC = D + 2;
  __shared__ float w[KVQ_MAX_SPLITS];  // records of a pair: at most KVQ_MAX_SPLITS (the workspace stride)
  __shared__ float red[kMergeThreads / 32];
  __shared__ float part[kMergeGroups][D];
  __shared__ int bound[kTcMaxCtas + 1];
  const int pair = blockIdx.x, h = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nh = a.gq;
  // the range table in shared memory: one parallel read of the parameter
  // array instead of a search whose every step would wait on the constant
  // cache
  for (int i = tid; i <= a.n_cta; i += kMergeThreads) bound[i] = a.tc_bound[i];
  __syncthreads();
  grid_dep_wait();  // launched as a dependent of the decode grid: its records first
  const long long nt = a.n_tiles;
  const int first = tc_owner(bound, a.n_cta, (long long)pair * nt);
  const int last = tc_owner(bound, a.n_cta, (long long)pair * nt + nt - 1);
  const int pieces = last - first + 1;
  if (pieces == 1) return;  // written by the decode launch itself
  const float* recs = a.part + (size_t)pair * a.n_splits * nh * REC + (size_t)h * REC;
  const int c = tid % D, k = tid / D;
  float ov[kMergeRegs];
#pragma unroll
  for (int i = 0; i < kMergeRegs; ++i) {
    const int s = k + i * kMergeGroups;
    ov[i] = s < pieces ? __ldcg(recs + (size_t)s * nh * REC + c) : 0.f;
  }
  float mt = -INFINITY, lt = 0.f;
  if (tid < pieces) {
    mt = __ldcg(recs + (size_t)tid * nh * REC + D);
    lt = __ldcg(recs + (size_t)tid * nh * REC + D + 1);
  }
  // M
  float m = mt;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, off));
  if (lane == 0) red[warp] = m;
  __syncthreads();
  m = red[0];
#pragma unroll
  for (int i = 1; i < kMergeThreads / 32; ++i) m = fmaxf(m, red[i]);
  __syncthreads();
  // weights and L
  const float wt = (tid < pieces && m != -INFINITY) ? exp2f(mt - m) : 0.f;
  if (tid < pieces) w[tid] = wt;
  float l = lt * wt;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(kFull, l, off);
  if (lane == 0) red[warp] = l;
  __syncthreads();
  l = 0.f;
#pragma unroll
  for (int i = 0; i < kMergeThreads / 32; ++i) l += red[i];
  // O
  float o = 0.f;
#pragma unroll
  for (int i = 0; i < kMergeRegs; ++i) {
    const int s = k + i * kMergeGroups;
    if (s < pieces) o = fmaf(ov[i], w[s], o);
  }
  for (int s = k + kMergeRegs * kMergeGroups; s < pieces; s += kMergeGroups)  // past 80 records
    o = fmaf(__ldcg(recs + (size_t)s * nh * REC + c), w[s], o);
  part[k][c] = o;
  __syncthreads();
  if (k == 0) {
#pragma unroll
    for (int i = 1; i < kMergeGroups; ++i) o += part[i][c];
    a.out[((size_t)pair * nh + h) * D + c] = __float2half_rn(l > 0.f ? o / l : 0.f);
  }
}

}  // namespace

cudaError_t launch_decode_tc_merge(const DecodeArgs& a, int n_pairs, cudaStream_t s) {
  return launch_kernel(merge_tc_kernel, dim3(n_pairs, a.gq), dim3(kMergeThreads), 0, s, true, a);
}

int decode_tc_ctas_per_sm() { return kTcCtasPerSm; }

// form 1: one query head per kv head, one segment of `bits`; form 4: 2-4
// query heads, one segment, d_h / G <= 2; form 8: up to 8 query heads over
// any segments (widths per tile).
cudaError_t launch_decode_tc(const DecodeArgs& a, int bits, int form, cudaStream_t s) {
  if (form == 8) return launch_tc_b<0, 8>(a, s);
  return form == 1 ? launch_tc_hq<1>(a, bits, s) : launch_tc_hq<4>(a, bits, s);
}

// The same kernels over a paged cache (per-sequence lengths).
cudaError_t launch_decode_tc_paged(const DecodeArgs& a, const PagedArgs& p, int bits, int form, cudaStream_t s) {
  if (form == 8) return launch_tc_b<0, 8, true>(a, s, p);
  return form == 1 ? launch_tc_hq<1, true>(a, bits, s, p) : launch_tc_hq<4, true>(a, bits, s, p);
}

}  // namespace kvq
