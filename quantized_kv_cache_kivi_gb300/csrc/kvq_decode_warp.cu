// Decode attention with one query head per kv head (MHA) over a 2-bit packed
// segment and the fp16 rings, d_h = 128, every warp a bulk-copy pipeline of
// its own.
//
// What is computed (KIVI page, Algorithm 1 decoding branch):
//   a_t = sm_scale q . k_t, p = softmax(a), out = sum_t p_t v_t,
// packed K dequantized per (group, channel), packed V per (token, channel
// group), the fp16 rings as they are.  The contractions run on the tensor
// cores with exact operands, as in kvq_decode_tc.cu's one-head form: a code
// field left at bit p of a 16-bit half is the fp16 subnormal code 2^(p-24);
//   K:  q . k_t = sum_c (q_c s_gc) code_tc + sum_c q_c z_gc, A = codes
//       [token][channel], B = the scaled query as an fp16 high part (even
//       columns) and low part (odd columns);
//   V:  sum_t p_t (code_tc s_tg + z_tg), A = codes [channel][token],
//       B[t][n] = p_t s_tn (n < 4) and p_t z_t(n-4) (n >= 4).
//
// Work split.  The token axis of every (batch, kv head) pair is cut into
// chunks (32 tokens with K and V packed; 8-token blocks where a ring is
// involved: kvq_internal.h, warp_chunk) and each pair's chunk list into k
// or k - 1 contiguous pieces of equal cost, so that the pieces of all pairs
// fill the GPU's resident warp slots (kWarpWarps per SM).  Each piece is a
// one-warp CTA that stages its
// own chunks, kWarpSlots ahead, into its own slots: the K and V codes by
// bulk copies (TMA engine, mbarrier completion) that one lane issues, the
// small scale / zero arrays by 16-byte cp.async pieces of every lane
// tracked on the same mbarrier.  With one warp per CTA every shared-memory
// and barrier address is warp-uniform.  No warp ever waits for another:
// there is no producer warp, no stage release and no CTA-wide barrier, and
// a warp loads its pair's query once.  Each piece leaves a partial
// (o, m, l) record; the last piece of a pair to finish (atomic counter)
// merges the records.
#include <float.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"
#include "kvq_mma.cuh"

namespace kvq {
namespace {

using namespace mma;

constexpr int kWB = 2;                   // packed width of this kernel
constexpr int kRB = D * kWB / 8;         // packed row bytes (32)
constexpr int kKtab = 512;               // one K operand table (bytes)
constexpr int kRec = D + 2;              // record (o[D], m, l)

// Shared memory of a CTA (one warp): its slots, the K operand table, the
// pair's query and the slots' mbarriers.
struct WarpSmem {
  static constexpr int slots = 0;                              // [slot][kWarpSlot]
  static constexpr int ktab = slots + kWarpSlots * kWarpSlot;  // [kKtab]
  static constexpr int qbuf = ktab + kKtab;                    // [D] f16
  static constexpr int bars = qbuf + D * 2;                          // [slot] mbarrier
  static constexpr int total = bars + kWarpSlots * 8;
};
static_assert(WarpSmem::ktab % 16 == 0 && WarpSmem::qbuf % 16 == 0 && WarpSmem::bars % 8 == 0, "align");
static_assert(kWarpWarps * (WarpSmem::total + 1024) <= 228 * 1024, "CTAs per SM");

struct WState {
  float m;  // running max (log2 domain), warp-uniform
  float l;  // sum of p over this lane's rows
  float acc[8][4];
  float accz[4];
  bool vring;  // acc unscaled (ring V reached)
};

__device__ __forceinline__ void reset_state(WState& S) {
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

__device__ __forceinline__ void unscale_acc2(WState& S) {
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    const int p = Fields<2>::pos(mt % 8);
    const float us = __uint_as_float((uint32_t)(127 + 24 - p) << 23);  // 2^(24 - p)
#pragma unroll
    for (int e = 0; e < 4; ++e) S.acc[mt][e] *= us;
  }
}

// Per-lane constants.  Fragment role: lane (gid, tig).  K-operand build
// role: lane (btig, bkt) = (lane & 3, lane >> 2) computes the entries of
// column pairs (btig, k-tile bkt): channels c_lo(e), c_hi(e) = c_lo(e) + 8
// for e = 0, 1, with c_lo(1) = c_lo(0) + 1.
struct LaneC {
  int gid, tig, r0, r1, ta, tb, tc, td;
  int btig, bkt, c_lo0;
  uint32_t wr_hi, wr_lo;  // byte offsets of this lane's 8-byte table entries (hi, lo parts)
  uint32_t rd;            // byte offset of this lane's first 16-byte table row (k-pair 0)
};

// K operand table: 16-byte units u = kp * 8 + ((hp * 4 + tig) ^ ((kp & 1) * 4))
// for k-tile pair kp, part hp (0 high, 1 low), column-pair tig: the readers
// of one k-pair and the writers of two k-pairs each cover all 32 banks.
__device__ __forceinline__ uint32_t ktab_unit(int kp, int hp, int tig) {
  return (uint32_t)(kp * 8 + ((hp * 4 + tig) ^ ((kp & 1) * 4)));
}

__device__ __forceinline__ LaneC lane_consts(int lane) {
  LaneC L;
  L.gid = lane >> 2;
  L.tig = lane & 3;
  L.r0 = sigma(L.gid);
  L.r1 = sigma(L.gid + 8);
  L.ta = sigma(2 * L.tig);
  L.tb = sigma(2 * L.tig + 1);
  L.tc = sigma(2 * L.tig + 8);
  L.td = sigma(2 * L.tig + 9);
  L.btig = lane & 3;
  L.bkt = lane >> 2;
  int clo, chi, p;
  k_half2_channels<2>(L.btig, 2 * L.bkt, &clo, &chi, &p);
  L.c_lo0 = clo;
  L.wr_hi = ktab_unit(L.bkt >> 1, 0, L.btig) * 16 + (L.bkt & 1) * 8;
  L.wr_lo = ktab_unit(L.bkt >> 1, 1, L.btig) * 16 + (L.bkt & 1) * 8;
  L.rd = 0;
  return L;
}

// The query of a pair in the lane's build role: qk = q_c sm_scale log2(e)
// 2^-p (the K operand before the group scale), qs = q_c sm_scale log2(e)
// (for the bias q . z), for channels (c_lo0, c_lo0 + 8, c_lo0 + 1, c_lo0 + 9).
struct PairQ {
  float qk[4], qs[4];
};

__device__ __forceinline__ PairQ pair_query(const WarpArgs& a, const __half* qsm, const LaneC& L) {
  PairQ Q;
  const int c[4] = {L.c_lo0, L.c_lo0 + 8, L.c_lo0 + 1, L.c_lo0 + 9};
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    int clo, chi, p;
    k_half2_channels<2>(L.btig, 2 * L.bkt + e, &clo, &chi, &p);
    const float f = __uint_as_float((uint32_t)(127 - p) << 23) * a.scale_log2;  // 2^-p sm_scale log2(e)
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const float qv = __half2float(qsm[c[2 * e + k]]);
      Q.qk[2 * e + k] = qv * f;
      Q.qs[2 * e + k] = qv * a.scale_log2;
    }
  }
  return Q;
}

// The K operand of one K group (the group's scales at ks, zeros at kz in the
// slot): each lane computes its four entries, splits them into an fp16 high
// part and the fp16 rest, writes both to the warp's table; every lane then
// reads the 16 words of its own column.  Returns the bias q . z (log2
// domain) of the group.  tab: the warp's table (the __syncwarp that ends
// each chunk separates one chunk's reads from the next one's writes).
template <bool INTZ>
__device__ __forceinline__ float build_kop(const uint8_t* ks, const uint8_t* kz, const PairQ& Q, const LaneC& L,
                                           uint8_t* tab, uint32_t (&bq)[16]) {
  const uint32_t s_lo = *reinterpret_cast<const uint32_t*>(ks + 2 * L.c_lo0);        // s[c_lo0], s[c_lo0 + 1]
  const uint32_t s_hi = *reinterpret_cast<const uint32_t*>(ks + 2 * (L.c_lo0 + 8));  // s[c_hi0], s[c_hi0 + 1]
  const uint32_t z_lo = *reinterpret_cast<const uint32_t*>(kz + 2 * L.c_lo0);
  const uint32_t z_hi = *reinterpret_cast<const uint32_t*>(kz + 2 * (L.c_lo0 + 8));
  const float2 sl = __half22float2(*reinterpret_cast<const __half2*>(&s_lo));
  const float2 sh = __half22float2(*reinterpret_cast<const __half2*>(&s_hi));
  // entries (e = 0: c_lo0, c_hi0; e = 1: c_lo1, c_hi1)
  const float v0 = Q.qk[0] * sl.x, v1 = Q.qk[1] * sh.x, v2 = Q.qk[2] * sl.y, v3 = Q.qk[3] * sh.y;
  const uint32_t h01 = pack_half2(v0, v1), h23 = pack_half2(v2, v3);
  const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&h01));
  const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&h23));
  const uint32_t l01 = pack_half2(v0 - f01.x, v1 - f01.y), l23 = pack_half2(v2 - f23.x, v3 - f23.y);
  *reinterpret_cast<uint2*>(tab + L.wr_hi) = make_uint2(h01, h23);
  *reinterpret_cast<uint2*>(tab + L.wr_lo) = make_uint2(l01, l23);
  float zl0, zl1, zh0, zh1;
  if constexpr (!INTZ) {
    const float2 zl = __half22float2(*reinterpret_cast<const __half2*>(&z_lo));
    const float2 zh = __half22float2(*reinterpret_cast<const __half2*>(&z_hi));
    zl0 = zl.x, zl1 = zl.y, zh0 = zh.x, zh1 = zh.y;
  } else {  // the additive zero -s z of the integer zero point
    zl0 = -sl.x * (float)(short)(z_lo & 0xffffu);
    zl1 = -sl.y * (float)(short)(z_lo >> 16);
    zh0 = -sh.x * (float)(short)(z_hi & 0xffffu);
    zh1 = -sh.y * (float)(short)(z_hi >> 16);
  }
  float bias = Q.qs[0] * zl0;
  bias = fmaf(Q.qs[1], zh0, bias);
  bias = fmaf(Q.qs[2], zl1, bias);
  bias = fmaf(Q.qs[3], zh1, bias);
  __syncwarp();
  const int hp = L.gid & 1;  // column gid: high part (even) or low part (odd)
#pragma unroll
  for (int kp = 0; kp < 4; ++kp)
    *reinterpret_cast<uint4*>(&bq[4 * kp]) = *reinterpret_cast<const uint4*>(tab + ktab_unit(kp, hp, L.tig) * 16);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) bias += __shfl_xor_sync(kFull, bias, off);
  return bias;
}

// Scores (log2 domain) of rows gid, gid + 8 of NH 16-token halves of packed
// K at kc (row stride 32 bytes, the lane's 8 bytes at tig * 8): 8 MMAs per
// half, the two k-tile parities in separate accumulators.
template <int NH>
__device__ __forceinline__ void k_scores_packed(const uint8_t* kc, const LaneC& L, const uint32_t (&bq)[16], float bias,
                                                float (&x)[2][2]) {
  uint32_t w[NH][2][2];  // [half][row][word]
#pragma unroll
  for (int h = 0; h < NH; ++h) {
    const uint2 u0 = *reinterpret_cast<const uint2*>(kc + (16 * h + L.r0) * kRB + L.tig * 8);
    const uint2 u1 = *reinterpret_cast<const uint2*>(kc + (16 * h + L.r1) * kRB + L.tig * 8);
    w[h][0][0] = u0.x;
    w[h][0][1] = u0.y;
    w[h][1][0] = u1.x;
    w[h][1][1] = u1.y;
  }
  float acc[NH][2][4];
#pragma unroll
  for (int h = 0; h < NH; ++h)
#pragma unroll
    for (int k = 0; k < 2; ++k)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[h][k][e] = 0.f;
#pragma unroll
  for (int kt = 0; kt < 8; ++kt) {
#pragma unroll
    for (int h = 0; h < NH; ++h) {
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
  for (int h = 0; h < NH; ++h) {
    x[h][0] = fmaf((acc[h][0][0] + acc[h][1][0]) + (acc[h][0][1] + acc[h][1][1]), 16777216.0f, bias);
    x[h][1] = fmaf((acc[h][0][2] + acc[h][1][2]) + (acc[h][0][3] + acc[h][1][3]), 16777216.0f, bias);
  }
}

// Scores of rows gid, gid + 8 of one 16-row block of fp16 ring K at kr
// (row stride 256 bytes): lane tig's 32 channels as four 16-byte chunks,
// chunk kc at position (kc + tig) & 3 of its 64-byte block, the query words
// (qsm) in the same order.
__device__ __forceinline__ void k_scores_ring(const uint8_t* kr, const uint8_t* qsm, const LaneC& L, float scale_log2,
                                              float& x0, float& x1) {
  float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int kc = 0; kc < 4; ++kc) {
    const int off = L.tig * 64 + ((kc + L.tig) & 3) * 16;
    const uint4 u0 = *reinterpret_cast<const uint4*>(kr + L.r0 * (D * 2) + off);
    const uint4 u1 = *reinterpret_cast<const uint4*>(kr + L.r1 * (D * 2) + off);
    const uint4 qw = *reinterpret_cast<const uint4*>(qsm + off);
    mma16816(sc, u0.x, u1.x, u0.y, u1.y, qw.x, qw.y);
    mma16816(sc, u0.z, u1.z, u0.w, u1.w, qw.z, qw.w);
  }
  x0 = sc[0] * scale_log2;  // columns 2 tig and 2 tig + 1 carry the same query
  x1 = sc[2] * scale_log2;
}

// Online softmax over the scores x[h][row] of NH halves (rows of this lane:
// r0, r1 of each half; -inf where masked).  Returns P in the V MMA's B
// layout: pp[h][0] = p of tokens (ta, tb), pp[h][1] = (tc, td) of half h.
template <int NH>
__device__ __forceinline__ void softmax_step(WState& S, const float (&x)[2][2], uint32_t (&pp)[2][2]) {
  float mloc = fmaxf(x[0][0], x[0][1]);
  if (NH == 2) mloc = fmaxf(mloc, fmaxf(x[1][0], x[1][1]));
  if (__any_sync(kFull, mloc > S.m)) {
    mloc = fmaxf(mloc, __shfl_xor_sync(kFull, mloc, 4));
    mloc = fmaxf(mloc, __shfl_xor_sync(kFull, mloc, 8));
    mloc = fmaxf(mloc, __shfl_xor_sync(kFull, mloc, 16));
    mloc = fmaxf(mloc, S.m);
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
#pragma unroll
  for (int h = 0; h < NH; ++h) {
    const float p0 = ex2(x[h][0] - S.m), p1 = ex2(x[h][1] - S.m);
    S.l += p0 + p1;
    pp[h][0] = movm_trans(pack_half2(p0, p0));
    pp[h][1] = movm_trans(pack_half2(p1, p1));
  }
}

// PV over NH halves of packed V: codes at vc (row stride 32 bytes, token
// row t at vc + t * 32), token scales / zeros at vs / vz ([token][ngv]).
// Rows whose token lies outside [lo, hi) of the staged block are padding:
// p = 0 there and their stale scale / zero bits are masked (no NaN).
template <int NH, bool FULL, int NGV, bool INTZ>
__device__ __forceinline__ void pv_packed(const uint8_t* vc, const uint8_t* vs, const uint8_t* vz, int lo, int hi,
                                          const LaneC& L, const uint32_t (&pp)[2][2], WState& S) {
  const int g = L.gid & 3;
  const bool live = NGV == 4 || g < NGV;  // columns of groups past d / Gv stay zero
  const uint16_t* sp = reinterpret_cast<const uint16_t*>(L.gid < 4 ? vs : vz) + g;
  const uint16_t* szp = reinterpret_cast<const uint16_t*>(vs) + g;
  constexpr int st = NGV;
  uint32_t bv[2][2];
#pragma unroll
  for (int h = 0; h < NH; ++h) {
    const int o = 16 * h;
    const int t[4] = {o + L.ta, o + L.tb, o + L.tc, o + L.td};
    uint32_t e[4], m[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      m[i] = (live && (FULL || (t[i] >= lo && t[i] < hi))) ? 0xffffu : 0u;
      e[i] = live ? (uint32_t)sp[t[i] * st] & m[i] : 0u;
    }
    if (INTZ && L.gid >= 4 && live) {  // columns 4..7: p times the additive zero -s z, one rounding
      bv[h][0] = p_times_zero(pp[h][0], e[0], e[1], szp[t[0] * st] & m[0], szp[t[1] * st] & m[1]);
      bv[h][1] = p_times_zero(pp[h][1], e[2], e[3], szp[t[2] * st] & m[2], szp[t[3] * st] & m[3]);
    } else {
      bv[h][0] = hmul2u(pp[h][0], halves(e[0], e[1]));
      bv[h][1] = hmul2u(pp[h][1], halves(e[2], e[3]));
    }
  }
  const uint8_t* vg = vc + L.gid * 4;  // the lane's 16 channels: one word per token
#pragma unroll
  for (int h = 0; h < NH; ++h) {
    const uint8_t* vh = vg + 16 * h * kRB;
    const uint32_t wa = *reinterpret_cast<const uint32_t*>(vh + L.ta * kRB);
    const uint32_t wb = *reinterpret_cast<const uint32_t*>(vh + L.tb * kRB);
    const uint32_t wc = *reinterpret_cast<const uint32_t*>(vh + L.tc * kRB);
    const uint32_t wd = *reinterpret_cast<const uint32_t*>(vh + L.td * kRB);
    const uint32_t lo1 = __byte_perm(wa, wb, 0x5410), hi1 = __byte_perm(wa, wb, 0x7632);
    const uint32_t lo2 = __byte_perm(wc, wd, 0x5410), hi2 = __byte_perm(wc, wd, 0x7632);
    const uint32_t lo1s = lo1 >> 6, hi1s = hi1 >> 6, lo2s = lo2 >> 6, hi2s = hi2 >> 6;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t m = ((3u << Fields<2>::pos(j)) | (3u << (Fields<2>::pos(j) + 16)));
      const bool ip = j < Fields<2>::INPLACE;
      mma16816(S.acc[j], (ip ? lo1 : lo1s) & m, (ip ? hi1 : hi1s) & m, (ip ? lo2 : lo2s) & m, (ip ? hi2 : hi2s) & m,
               bv[h][0], bv[h][1]);
    }
  }
  constexpr uint32_t ONES = 0x3C003C00u;  // (1.0, 1.0)
#pragma unroll
  for (int h = 0; h < NH; ++h) mma16816(S.accz, ONES, ONES, ONES, ONES, bv[h][0], bv[h][1]);
}

// PV over an 8-row block of fp16 ring V at vr (row stride 256 bytes): A
// rows are the channels of the 2-bit row map, gathered from the lane's 16
// channels of each token; rows outside [lo, hi) read as zeros, and rows 8..15
// of the MMA's 16 (tokens tc, td) lie past the block: zeros, not read.
__device__ __forceinline__ void pv_ring(const uint8_t* vr, int lo, int hi, const LaneC& L, const uint32_t (&pp)[2],
                                        WState& S) {
  if (!S.vring) {
    unscale_acc2(S);
    S.vring = true;
  }
  const uint8_t* vg = vr + L.gid * 32;
  const uint32_t* va = reinterpret_cast<const uint32_t*>(vg + L.ta * (D * 2));
  const uint32_t* vb = reinterpret_cast<const uint32_t*>(vg + L.tb * (D * 2));
  const uint32_t ma = (L.ta >= lo && L.ta < hi) ? kFull : 0u, mb = (L.tb >= lo && L.tb < hi) ? kFull : 0u;
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    int c0, c8, p;
    v_rows<2>(0, mt, &c0, &c8, &p);  // offsets inside the lane's 16 channels
    const uint32_t s0sel = (c0 & 1) ? 0x7632u : 0x5410u;
    const uint32_t s8sel = (c8 & 1) ? 0x7632u : 0x5410u;
    mma16816(S.acc[mt], __byte_perm(va[c0 >> 1] & ma, vb[c0 >> 1] & mb, s0sel),
             __byte_perm(va[c8 >> 1] & ma, vb[c8 >> 1] & mb, s8sel), 0u, 0u, pp[0], pp[1]);
  }
}

// A 32-token chunk with K and V packed (n tokens valid, 32 when FULL).
template <bool FULL, int NGV, bool INTZ>
__device__ __forceinline__ void run_pp(const uint8_t* slot, int n, const PairQ& Q, const LaneC& L, uint8_t* tab,
                                       WState& S) {
  uint32_t bq[16];
  const float bias = build_kop<INTZ>(slot + kPpKs, slot + kPpKz, Q, L, tab, bq);
  float x[2][2];
  k_scores_packed<2>(slot + kPpKc, L, bq, bias, x);  // rows past n read stale codes: masked below
  if (!FULL) {
    if (L.r0 >= n) x[0][0] = -INFINITY;
    if (L.r1 >= n) x[0][1] = -INFINITY;
    if (16 + L.r0 >= n) x[1][0] = -INFINITY;
    if (16 + L.r1 >= n) x[1][1] = -INFINITY;
  }
  uint32_t pp[2][2];
  softmax_step<2>(S, x, pp);
  pv_packed<2, FULL, NGV, INTZ>(slot + kPpVc, slot + kPpVs, slot + kPpVz, 0, n, L, pp, S);
}

// A chunk of at most 8 tokens at rows [o0, o0 + n) of its staged 8-row
// block (rows 8..15 of the MMA half are padding), K and V each packed or
// from the ring.
template <int NGV, bool INTZ>
__device__ __forceinline__ void run_x(const WarpArgs& a, const uint8_t* slot, const WarpChunk& ch, const PairQ& Q,
                                      const LaneC& L, const uint8_t* qsm, uint8_t* tab, WState& S) {
  const int lo = ch.o0, hi = ch.o0 + ch.n;
  float x[2][2];
  if (ch.kq) {
    uint32_t bq[16];
    const float bias = build_kop<INTZ>(slot + kXK + kXKs, slot + kXK + kXKz, Q, L, tab, bq);
    k_scores_packed<1>(slot + kXK, L, bq, bias, x);
  } else {
    k_scores_ring(slot + kXK, qsm, L, a.scale_log2, x[0][0], x[0][1]);
  }
  if (L.r0 < lo || L.r0 >= hi) x[0][0] = -INFINITY;
  x[0][1] = -INFINITY;  // row gid + 8 lies past the 8-row block
  x[1][0] = x[1][1] = -INFINITY;
  uint32_t pp[2][2];
  softmax_step<1>(S, x, pp);
  if (ch.vq) pv_packed<1, false, NGV, INTZ>(slot + kXV, slot + kXV + kXVs, slot + kXV + kXVz, lo, hi, L, pp, S);
  else pv_ring(slot + kXV, lo, hi, L, pp[0], S);
}

// Base addresses of one pair's slices of the cache arrays.
struct PairPtrs {
  const uint8_t *kc, *vc;
  const __half *ks, *kz, *vs, *vz, *kr, *vr;
};

__device__ __forceinline__ PairPtrs pair_ptrs(const WarpArgs& a, long long pair) {
  PairPtrs p;
  const long long rows = pair * a.cap;
  p.kc = a.kc + rows * kRB;
  p.vc = a.vc + rows * kRB;
  p.ks = a.ks + (rows >> a.log2G) * D;
  p.kz = a.kz + (rows >> a.log2G) * D;
  p.vs = a.vs + rows * a.ngv;
  p.vz = a.vz + rows * a.ngv;
  p.kr = a.kr + pair * a.R * D;
  p.vr = a.vr + pair * a.R * D;
  return p;
}

// Stage chunk c of a pair into a slot.  A slot's mbarrier expects 33
// arrivals per phase: one from each lane and one, with the byte count of the
// bulk copies, from lane 0, in any order.  A full 32-token chunk with K and
// V packed: every lane copies its 16-byte pieces of the K group's scales /
// zeros and the tokens' V scales / zeros (cp.async) and arrives when they
// have landed; lane 0 issues the K and V code copies (TMA engine) -- two
// bulk copies per chunk, as the engine issues small copies at a limited
// rate per SM.  Anything else (ring blocks, a short last chunk) walks the
// general copy list (warp_chunk_copies, the list the host checked) with
// bulk copies only.  The CTA is one warp, so every address is warp-uniform.
// No proxy fence precedes the copies into a slot the warp has just read:
// every shared load of the slot has returned its value (the loop's
// __syncwarp follows the last use) before lane 0 issues them.
constexpr uint32_t kSlotArrivals = 33;

template <int NGV>
__device__ __forceinline__ void stage_chunk(const WarpArgs& a, const PairPtrs& pp, long long pair, int c,
                                            uint8_t* slot, uint64_t* bar, int lane) {
  if (c < a.npp / 32) {
    const int t0 = 32 * c;
    const uint32_t sl = smem_u32(slot);
    const int h = lane & 15;
    const bool lo = lane < 16;
    cp16(sl + (lo ? kPpKs : kPpKz) + h * 16, (lo ? pp.ks : pp.kz) + (t0 >> a.log2G) * D + h * 8);
    constexpr int VB = 32 * NGV * 2;  // bytes of the chunk's token scales (zeros)
    if (h * 16 < VB) cp16(sl + (lo ? kPpVs : kPpVz) + h * 16, (lo ? pp.vs : pp.vz) + t0 * NGV + h * 8);
    cp_mbar_arrive_noinc(bar);
    if (lane == 0) {
      mbar_arrive_expect_tx(bar, 2 * 1024);
      bulk_g2s(slot + kPpKc, pp.kc + t0 * kRB, 1024, bar);
      bulk_g2s(slot + kPpVc, pp.vc + t0 * kRB, 1024, bar);
    }
    return;
  }
  mbar_arrive_plain(bar);
  if (lane == 0) {
    const WarpChunk ch = warp_chunk(a, c);
    uint32_t bytes = 0;
    warp_chunk_copies(a, pair, ch, [&](const void*, uint32_t, uint32_t n, int) { bytes += n; });
    mbar_arrive_expect_tx(bar, bytes);
    warp_chunk_copies(a, pair, ch,
                      [&](const void* src, uint32_t dst, uint32_t n, int) { bulk_g2s(slot + dst, src, n, bar); });
  }
}

__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// End of a warp's piece of a pair: its partial (o, m, l) as the piece's
// record, made visible and counted (lane 0 gets the count found, `ticket`),
// or the output itself when the pair has one piece.  Returns the pair's
// number of records (1: output written).
template <int NGV>
__device__ int write_piece(const WarpArgs& a, long long pair, int piece, int kp, int lane, const LaneC& L,
                           WState& S, int& ticket) {
  if (!S.vring) unscale_acc2(S);
  float l = S.l;  // sum over the lanes of one tig (rows gid)
  l += __shfl_xor_sync(kFull, l, 4);
  l += __shfl_xor_sync(kFull, l, 8);
  l += __shfl_xor_sync(kFull, l, 16);
  const int nrec = kp;
  // o of channel c: column g(c) of its row (lanes tig = g / 2) plus the z sum
  // of group g (column 4 + g, lanes tig = 2 + g / 2)
  float o16[16];
  int c16[16];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    int c0, c8, p;
    v_rows<2>(L.gid, mt, &c0, &c8, &p);
    const int g = (c0 * NGV) >> 7;  // c0 and c8 share their group
    const float z0 = __shfl_sync(kFull, S.accz[0], (lane & ~3) | (2 + (g >> 1)));
    const float z1 = __shfl_sync(kFull, S.accz[1], (lane & ~3) | (2 + (g >> 1)));
    const float zg = (g & 1) ? z1 : z0;
    o16[2 * mt] = ((g & 1) ? S.acc[mt][1] : S.acc[mt][0]) + zg;
    o16[2 * mt + 1] = ((g & 1) ? S.acc[mt][3] : S.acc[mt][2]) + zg;
    c16[2 * mt] = (L.tig == (g >> 1)) ? c0 : -1;
    c16[2 * mt + 1] = (L.tig == (g >> 1)) ? c8 : -1;
  }
  if (nrec == 1) {
    const float il = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i)
      if (c16[i] >= 0) a.out[pair * D + c16[i]] = __float2half_rn(o16[i] * il);
    return 1;
  }
  float* rec = a.part + (pair * a.k + piece) * kRec;
#pragma unroll
  for (int i = 0; i < 16; ++i)
    if (c16[i] >= 0) rec[c16[i]] = o16[i];
  if (lane == 0) {
    rec[D] = S.m;
    rec[D + 1] = l;
  }
  fence_acq_rel_gpu();  // the record is visible before it is counted
  __syncwarp();
  if (lane == 0) ticket = atomicAdd(&a.counters[pair], 1);
  return nrec;
}

// The piece that found nrec - 1 (the last of the pair to arrive) merges the
// pair's records and writes the output.  Records are taken 16 at a time with
// every load of a block (o of 16 records, m and l in lanes 0..15) in flight
// together; the running maximum rescales the sums of earlier blocks.
__device__ __noinline__ void merge_if_last(const WarpArgs& a, long long pair, int nrec, int ticket, int lane) {
  if (!__shfl_sync(kFull, ticket == nrec - 1 ? 1 : 0, 0)) return;
  fence_acq_rel_gpu();  // the other records are visible after their counts
  const float* recs = a.part + pair * a.k * kRec;
  constexpr int kBlk = 16;
  float m = -INFINITY, ls = 0.f;
  float oo[D / 32] = {0.f, 0.f, 0.f, 0.f};
  for (int s0 = 0; s0 < nrec; s0 += kBlk) {
    const int nb = nrec - s0 < kBlk ? nrec - s0 : kBlk;
    float ov[kBlk][D / 32];
#pragma unroll
    for (int j = 0; j < kBlk; ++j)
#pragma unroll
      for (int i = 0; i < D / 32; ++i) ov[j][i] = j < nb ? __ldcg(recs + (s0 + j) * kRec + lane + 32 * i) : 0.f;
    float mj = -INFINITY, lj = 0.f;
    if (lane < nb) {
      mj = __ldcg(recs + (s0 + lane) * kRec + D);
      lj = __ldcg(recs + (s0 + lane) * kRec + D + 1);
    }
    float mb = mj;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, off));
    const float mn = fmaxf(m, mb);
    const float sc = m == -INFINITY ? 0.f : exp2f(m - mn);
    const float wj = mj == -INFINITY ? 0.f : exp2f(mj - mn);
    float lw = lj * wj;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lw += __shfl_xor_sync(kFull, lw, off);
    ls = ls * sc + lw;
#pragma unroll
    for (int i = 0; i < D / 32; ++i) oo[i] *= sc;
#pragma unroll
    for (int j = 0; j < kBlk; ++j) {
      const float w = __shfl_sync(kFull, wj, j);
#pragma unroll
      for (int i = 0; i < D / 32; ++i) oo[i] = fmaf(ov[j][i], w, oo[i]);
    }
    m = mn;
  }
  const float il = ls > 0.f ? 1.f / ls : 0.f;
#pragma unroll
  for (int i = 0; i < D / 32; ++i) a.out[pair * D + lane + 32 * i] = __float2half_rn(oo[i] * il);
  if (lane == 0) a.counters[pair] = 0;  // ready for the next call on this workspace
}

// One warp per CTA, kWarpWarps CTAs per SM: CTAs [0, P1 k) take the pieces
// of the pairs cut into k, pair by pair; the rest those of the pairs cut
// into k - 1.
template <int NGV, bool INTZ>
__global__ void __launch_bounds__(32, kWarpWarps) decode_warp_kernel(const WarpArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int lane = threadIdx.x;
  // CTAs [0, P1 k): pairs with k pieces; then pairs with k - 1
  long long pair;
  int piece, kp;
  {
    const long long b = blockIdx.x, n1 = (long long)a.P1 * a.k;
    kp = b < n1 ? a.k : a.k - 1;
    const long long p0 = b < n1 ? 0 : a.P1, b0 = b < n1 ? 0 : n1;
    pair = p0 + (b - b0) / kp;
    piece = (int)((b - b0) % kp);
  }
  uint8_t* slots = smem + WarpSmem::slots;
  uint8_t* tab = smem + WarpSmem::ktab;
  __half* qsm = reinterpret_cast<__half*>(smem + WarpSmem::qbuf);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + WarpSmem::bars);
  const int c0 = warp_piece_start(a, kp, piece), c1 = warp_piece_start(a, kp, piece + 1);
  const int n = c1 - c0;  // chunks of this piece (at least one)
  const PairPtrs pp = pair_ptrs(a, pair);
  if (lane == 0) {
    for (int s = 0; s < kWarpSlots; ++s) mbar_init(&bars[s], kSlotArrivals);
    mbar_fence_init();
  }
  // Inside a decode step this grid starts while the kernel before it (the
  // step's append, or its flush) runs.  Chunks from a.dep_c on hold tokens
  // those write (the evicted V row, the new ring token, the flushed K
  // rows), so staging the first of them waits for that grid, whose
  // completion implies the step's earlier kernels' (each waits for its own
  // predecessor before it completes); the chunks before it are packed rows
  // that no kernel of the step writes, and the kernels of earlier steps had
  // completed before the step's first kernel let the next one start.
  bool waited = false;
  auto stage = [&](int c, int s) {
    if (!waited && c >= a.dep_c) {
      grid_dep_wait();
      waited = true;
    }
    stage_chunk<NGV>(a, pp, pair, c, slots + s * kWarpSlot, &bars[s], lane);
  };
  grid_dep_launch();
  const uint2 qv = __ldg(reinterpret_cast<const uint2*>(a.q + pair * D) + lane);
  __syncwarp();
  for (int s = 0; s < kWarpSlots && s < n; ++s) stage(c0 + s, s);
  reinterpret_cast<uint2*>(qsm)[lane] = qv;
  __syncwarp();
  const LaneC L = lane_consts(lane);
  const PairQ Q = pair_query(a, qsm, L);
  WState S;
  reset_state(S);
  const int n_full = a.npp / 32;  // full 32-token chunks with K and V packed
  int s = 0;
  uint32_t ph = 0;
  for (int k = 0; k < n; ++k) {
    const int c = c0 + k;
    // wait for the chunk's copies (bounded: about 2^31 clocks), inside the
    // barrier unit (suspend-time hint) rather than spinning through issue
    // slots the other warps of the SM need
    const uint32_t bar_addr = smem_u32(&bars[s]);
    if (!try_wait_at(bar_addr, ph)) {
      const long long t0 = clock64();
      bool ok = true;
      while (!try_wait_sleep(bar_addr, ph, 20000u)) {
        if (clock64() - t0 > (1ll << 31)) {
          ok = false;
          break;
        }
      }
      if (!__all_sync(kFull, ok)) {
        if (lane == 0) {
          atomicExch(a.err, 1);
          // the copies still in flight land before the block may exit
          for (int j = k; j < k + kWarpSlots && j < n; ++j)
            (void)mbar_drain_bounded(&bars[j % kWarpSlots], (uint32_t)((j / kWarpSlots) & 1));
        }
        return;
      }
    }
    const uint8_t* slot = slots + s * kWarpSlot;
    if (c < n_full) {
      run_pp<true, NGV, INTZ>(slot, 32, Q, L, tab, S);
    } else {
      const WarpChunk ch = warp_chunk(a, c);
      if (ch.pp) run_pp<false, NGV, INTZ>(slot, ch.n, Q, L, tab, S);
      else run_x<NGV, INTZ>(a, slot, ch, Q, L, reinterpret_cast<const uint8_t*>(qsm), tab, S);
    }
    __syncwarp();  // every lane has read the slot
    if (k + kWarpSlots < n) stage(c + kWarpSlots, s);
    if (++s == kWarpSlots) s = 0, ph ^= 1u;
  }
  int ticket = 0;
  const int nrec = write_piece<NGV>(a, pair, piece, kp, lane, L, S, ticket);
  if (nrec > 1) merge_if_last(a, pair, nrec, ticket, lane);
}

}  // namespace

template <int NGV, bool INTZ>
static cudaError_t launch_warp_t(const WarpArgs& a, cudaStream_t s, bool pdl) {
  const int bytes = WarpSmem::total;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(decode_warp_kernel<NGV, INTZ>), bytes);
  if (e != cudaSuccess) return e;
  const long long grid = (long long)a.P1 * a.k + (long long)(a.P - a.P1) * (a.k - 1);
  return launch_kernel(decode_warp_kernel<NGV, INTZ>, dim3((unsigned)grid), dim3(32), (size_t)bytes, s, pdl, a);
}

cudaError_t launch_decode_warp(const WarpArgs& a, cudaStream_t s, bool pdl) {
  if (a.ngv == 4) return a.intz ? launch_warp_t<4, true>(a, s, pdl) : launch_warp_t<4, false>(a, s, pdl);
  if (a.ngv == 2) return a.intz ? launch_warp_t<2, true>(a, s, pdl) : launch_warp_t<2, false>(a, s, pdl);
  return a.intz ? launch_warp_t<1, true>(a, s, pdl) : launch_warp_t<1, false>(a, s, pdl);
}

}  // namespace kvq
