// Decode attention for one query head per kv head (MHA), d_h = 128, one
// packed segment plus the fp16 ring (the KIVI layout), with the contractions
// on the tensor cores (mma.sync m16n8k16, f16 operands, f32 accumulation).
//
// What is computed (KIVI page, Algorithm 1 decoding branch):
//   a_t = sm_scale * q . k_t, p = softmax(a), out = sum_t p_t v_t,
// with packed K dequantized per (group, channel) and packed V per (token,
// channel group).  The algebra that makes both contractions tensor-core
// shaped:
//   K:  q . k_t = sum_c (q_c s_gc) code_tc + sum_c q_c z_gc.  A = codes
//       [token][channel], B = the scaled query (split into an fp16 high and
//       low part, columns 0 and 1), plus a per-group bias.
//   V:  sum_t p_t (code_tc s_tg(c) + z_tg(c)) = sum_t (p_t s_tg) code_tc +
//       sum_t p_t z_tg.  A = codes [channel][token], B[t][n] = p_t s_tn for
//       each channel group n: row c keeps only column g(c).
// Codes become fp16 operands without any conversion: a code field left at bit
// p (2 <= p <= 8) of a 16-bit half, all other bits zero, is the fp16
// subnormal code * 2^(p - 24) exactly; one 32-bit AND yields two of them.
// The products are exact in the fp32 accumulators, so the factor 2^(24 - p)
// is applied afterwards: folded into B for K (2^-p) with the scores scaled
// by 2^24, divided out of each channel row for V.
//
// CTA = 4 consumer warps + 1 producer warp, one (batch, kv head), a range of
// its tiles; the producer stages tiles with bulk copies (TMA engine), builds
// the K operand table of each tile's groups and signals "ready"; consumers
// each take a slice of 16-token sub-tiles, keep their own online softmax and
// release the stage.
#include <float.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int NCW = kTcConsumerWarps;
constexpr int NTH = (NCW + 1) * 32;
constexpr int D = 128;

// ---- shared memory layout ---------------------------------------------------
struct TcSmem {
  static constexpr int stages = 0;
  static constexpr int ktab = stages + kTcStages * kTcStageBytes;      // [stage][group][hi/lo][tig][kt][2] u32
  static constexpr int kbias = ktab + kTcStages * kTcKtabBytes;        // [stage][group] f32
  static constexpr int qnat = kbias + kTcStages * kTcMaxGroups * 4;    // [D] f16, natural order
  static constexpr int merge = qnat + D * 2;                          // [NCW][D + 2] f32
  static constexpr int bars = merge + NCW * (D + 2) * 4;
  static constexpr int flags = bars + 3 * kTcStages * 8;
  static constexpr int total = flags + 16;
};

// ---- code fields ------------------------------------------------------------
// A 32-bit word holds 32/B codes.  View it as two 16-bit halves; field j of a
// half (0 <= j < 16/B) holds the code of the channel at bit j*B of that half.
// x << 2 moves fields j < HALFJ to bit j*B + 2; x >> 6 moves the others to
// bit j*B - 6; either way the field sits at bit p in [2, 8] of its half.
template <int B>
struct Fields {
  static constexpr int PER_HALF = 16 / B;  // fields per half
  static constexpr int HALFJ = B == 8 ? 1 : (B == 4 ? 2 : 4);
  __host__ __device__ static constexpr int pos(int j) { return j < HALFJ ? j * B + 2 : j * B - 6; }
  // half2 (c_lo 2^(p-24), c_hi 2^(p-24)): field j of both halves, as subnormals
  __device__ static __forceinline__ uint32_t get(uint32_t xl, uint32_t xr, int j) {
    const uint32_t m = ((1u << B) - 1u) << pos(j);
    return (j < HALFJ ? xl : xr) & (m | (m << 16));
  }
};

// K operand layout.  Consumer thread (gid, tig) of a warp owns the 32
// channels [32 tig, 32 tig + 32) of its tokens.  Its h-th half2 (h < 16)
// holds two channels of one token: word w = h / (2 * PER_HALF), field j = h
// % PER_HALF of the low or high half (h / PER_HALF odd = high half ... see
// below); k-tile kt uses h = 2 kt (cols 2 tig, 2 tig + 1) and h = 2 kt + 1
// (cols 2 tig + 8, 2 tig + 9).
template <int B>
__host__ __device__ constexpr void k_half2_channels(int tig, int h, int* c_lo, int* c_hi, int* p) {
  constexpr int PH = 16 / B;             // fields per half = channels per half
  const int w = h / PH;                  // word index among the thread's words
  const int j = h % PH;                  // field inside each half
  const int base = 32 * tig + w * (32 / B);
  *c_lo = base + j;                      // low half: channels base .. base + PH - 1
  *c_hi = base + PH + j;                 // high half: channels base + PH ..
  *p = Fields<B>::pos(j);
}

// V operand layout: thread gid owns channels [16 gid, 16 gid + 16) of the 4
// tokens it reads; m-tile mt = (word w, field j) with w = mt / PER_HALF,
// j = mt % PER_HALF; row gid <- low-half channel, row gid + 8 <- high-half.
template <int B>
__host__ __device__ constexpr void v_rows(int gid, int mt, int* c_row0, int* c_row8, int* p) {
  constexpr int PH = 16 / B;
  const int w = mt / PH, j = mt % PH;
  const int base = 16 * gid + w * (32 / B);
  *c_row0 = base + j;
  *c_row8 = base + PH + j;
  *p = Fields<B>::pos(j);
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldmatrix_x4_t(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ float2 unpack_half2(uint32_t u) {
  return __half22float2(*reinterpret_cast<const __half2*>(&u));
}

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
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

// Per-thread state of one consumer warp (V: D fragments carry 2^(p - 24)).
struct WarpState {
  float m;            // running max (log2 domain), warp-uniform
  float l;            // sum of p over this thread's tokens (tig == 0 threads)
  float zs;           // sum p z for column gid (packed V), this thread's tokens
  float acc[8][4];    // packed V: D fragments of the 8 channel m-tiles
  float accr[8][4];   // ring V: D fragments, natural channel rows
};

template <int B>
__device__ __forceinline__ void rescale(WarpState& S, float alpha) {
  S.l *= alpha;
  S.zs *= alpha;
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      S.acc[i][e] *= alpha;
      S.accr[i][e] *= alpha;
    }
}

// One 16-token sub-tile [s0, s0 + 16) of a tile (tokens >= n are padding).
template <int B>
__device__ __forceinline__ void sub_tile(const DecodeArgs& a, const TileInfo& ti, const uint8_t* stage,
                                         const uint32_t* kt_hi_lo, const float* kbias,
                                         const __half* qnat, int s0, int lane, WarpState& S) {
  constexpr int RB = D * B / 8;        // packed row bytes
  constexpr int PH = 16 / B;
  const int gid = lane >> 2, tig = lane & 3;
  const int n = ti.n;
  // ------------------------------------------------------------- scores
  float sc[4] = {0.f, 0.f, 0.f, 0.f};  // C fragment: rows gid, gid + 8; cols 2 tig, 2 tig + 1
  if (ti.kseg >= 0) {
    // B operand (scaled query) of this token group: threads with gid 0 (high
    // part) and gid 1 (low part) hold it; the other columns are zero
    const int gl = min(((ti.ku0 + s0) >> a.log2G) - ti.g0, ti.ng - 1);
    uint32_t bq[16];
    if (gid < 2) {
      const uint4* src = reinterpret_cast<const uint4*>(kt_hi_lo + ((gl * 2 + gid) * 4 + tig) * 16);
#pragma unroll
      for (int k = 0; k < 4; ++k) *reinterpret_cast<uint4*>(&bq[4 * k]) = src[k];
    } else {
#pragma unroll
      for (int k = 0; k < 16; ++k) bq[k] = 0u;
    }
    // A operand: the thread's words of tokens s0 + gid and s0 + gid + 8
    constexpr int NW = B;  // 32-bit words per thread per token (32 channels)
    const uint32_t* r0 = reinterpret_cast<const uint32_t*>(stage + ti.k_off + (size_t)(s0 + gid) * RB) + tig * NW;
    const uint32_t* r1 = reinterpret_cast<const uint32_t*>(stage + ti.k_off + (size_t)(s0 + gid + 8) * RB) + tig * NW;
    uint32_t w0[NW], w1[NW];
#pragma unroll
    for (int k = 0; k < NW; ++k) {
      w0[k] = r0[k];
      w1[k] = r1[k];
    }
#pragma unroll
    for (int kt = 0; kt < 8; ++kt) {
      uint32_t a[4];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int h = 2 * kt + e;
        const int w = h / PH, j = h % PH;
        a[2 * e + 0] = Fields<B>::get(w0[w] << 2, w0[w] >> 6, j);
        a[2 * e + 1] = Fields<B>::get(w1[w] << 2, w1[w] >> 6, j);
      }
      // fragment order: a0 (row gid, cols 2tig..), a1 (row gid+8), a2 (row gid, cols 2tig+8..), a3
      mma16816(sc, a[0], a[1], a[2], a[3], bq[2 * kt], bq[2 * kt + 1]);
    }
    const float bias = kbias[gl];
    constexpr float k2p24 = 16777216.0f;  // the A operands carry 2^-24
    sc[0] = (sc[0] + sc[1]) * k2p24 + bias;  // token s0 + gid (valid in tig == 0 threads)
    sc[2] = (sc[2] + sc[3]) * k2p24 + bias;  // token s0 + gid + 8
  } else {
    // fp16 ring K in natural channel order: ldmatrix for A, q (natural) for B
#pragma unroll
    for (int kt = 0; kt < 8; ++kt) {
      uint32_t a[4];
      const int row = s0 + (lane & 15);
      const int col = kt * 16 + (lane >> 4) * 8;
      ldmatrix_x4(a, stage + ti.k_off + ((size_t)row * D + col) * 2);
      uint32_t b0 = 0u, b1 = 0u;
      if (gid == 0) {
        b0 = *reinterpret_cast<const uint32_t*>(qnat + kt * 16 + 2 * tig);
        b1 = *reinterpret_cast<const uint32_t*>(qnat + kt * 16 + 2 * tig + 8);
      }
      // ldmatrix x4 order: [rows 0-7, cols 0-7], [rows 8-15, cols 0-7],
      // [rows 0-7, cols 8-15], [rows 8-15, cols 8-15] = a0, a1, a2, a3
      mma16816(sc, a[0], a[1], a[2], a[3], b0, b1);
    }
    sc[2] = sc[2];
  }
  // ------------------------------------------------------ online softmax
  const bool v0 = s0 + gid < n, v1 = s0 + gid + 8 < n;
  float x0 = (tig == 0 && v0) ? sc[0] * a.scale_log2 : -INFINITY;
  float x1 = (tig == 0 && v1) ? sc[2] * a.scale_log2 : -INFINITY;
  float mx = fmaxf(x0, x1);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  const float m_new = fmaxf(S.m, mx);
  if (m_new != S.m && S.m != -INFINITY) rescale<B>(S, exp2f(S.m - m_new));
  S.m = m_new;
  const float p0 = x0 == -INFINITY ? 0.f : exp2f(x0 - m_new);
  const float p1 = x1 == -INFINITY ? 0.f : exp2f(x1 - m_new);
  S.l += p0 + p1;
  // p of tokens 2 tig, 2 tig + 1, 2 tig + 8, 2 tig + 9 of the sub-tile
  const float pa = __shfl_sync(0xffffffffu, p0, 8 * tig);      // token 2 tig
  const float pb = __shfl_sync(0xffffffffu, p0, 8 * tig + 4);  // token 2 tig + 1
  const float pc = __shfl_sync(0xffffffffu, p1, 8 * tig);      // token 2 tig + 8
  const float pd = __shfl_sync(0xffffffffu, p1, 8 * tig + 4);  // token 2 tig + 9
  const int ta = s0 + 2 * tig, tb = ta + 1, tc = ta + 8, td = ta + 9;
  // ------------------------------------------------------------------ PV
  if (ti.vseg >= 0) {
    const int ngv = D >> a.log2G;
    const __half* vs = reinterpret_cast<const __half*>(stage + ti.vs_off);
    const __half* vz = reinterpret_cast<const __half*>(stage + ti.vz_off);
    uint32_t b0 = 0u, b1 = 0u;
    if (gid < ngv) {
      // padding tokens carry p = 0 and must not read scales (may be NaN)
      const float sa = ta < n ? __half2float(vs[ta * ngv + gid]) : 0.f;
      const float sb = tb < n ? __half2float(vs[tb * ngv + gid]) : 0.f;
      const float sc2 = tc < n ? __half2float(vs[tc * ngv + gid]) : 0.f;
      const float sd = td < n ? __half2float(vs[td * ngv + gid]) : 0.f;
      b0 = pack_half2(pa * sa, pb * sb);
      b1 = pack_half2(pc * sc2, pd * sd);
      S.zs += (ta < n ? pa * __half2float(vz[ta * ngv + gid]) : 0.f) +
              (tb < n ? pb * __half2float(vz[tb * ngv + gid]) : 0.f) +
              (tc < n ? pc * __half2float(vz[tc * ngv + gid]) : 0.f) +
              (td < n ? pd * __half2float(vz[td * ngv + gid]) : 0.f);
    }
    // A: the thread's 16 channels of tokens (ta, tb) and (tc, td)
    constexpr int NW = B / 2;  // words per token for 16 channels
    const uint32_t* ra = reinterpret_cast<const uint32_t*>(stage + ti.v_off + (size_t)ta * RB) + gid * NW;
    const uint32_t* rb = reinterpret_cast<const uint32_t*>(stage + ti.v_off + (size_t)tb * RB) + gid * NW;
    const uint32_t* rc = reinterpret_cast<const uint32_t*>(stage + ti.v_off + (size_t)tc * RB) + gid * NW;
    const uint32_t* rd = reinterpret_cast<const uint32_t*>(stage + ti.v_off + (size_t)td * RB) + gid * NW;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const uint32_t wa = ra[w], wb = rb[w], wc = rc[w], wd = rd[w];
      const uint32_t lo1 = __byte_perm(wa, wb, 0x5410), hi1 = __byte_perm(wa, wb, 0x7632);
      const uint32_t lo2 = __byte_perm(wc, wd, 0x5410), hi2 = __byte_perm(wc, wd, 0x7632);
#pragma unroll
      for (int j = 0; j < PH; ++j) {
        const int mt = w * PH + j;
        mma16816(S.acc[mt], Fields<B>::get(lo1 << 2, lo1 >> 6, j), Fields<B>::get(hi1 << 2, hi1 >> 6, j),
                 Fields<B>::get(lo2 << 2, lo2 >> 6, j), Fields<B>::get(hi2 << 2, hi2 >> 6, j), b0, b1);
      }
    }
  } else {
    // fp16 ring V, natural channel rows: A = V^T tiles by ldmatrix.trans;
    // B column 0 = p; padding rows of the last sub-tile are zeroed
    const uint32_t b0 = gid == 0 ? pack_half2(pa, pb) : 0u;
    const uint32_t b1 = gid == 0 ? pack_half2(pc, pd) : 0u;
    const bool full = s0 + 16 <= n;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      uint32_t r[4];
      // matrices: [tok 0-7, ch mt*16+0..7], [tok 0-7, ch +8..15], [tok 8-15, ch 0..7], [tok 8-15, ch 8..15]
      const int tok = s0 + (lane & 7) + ((lane >> 4) << 3);
      const int ch = mt * 16 + ((lane >> 3) & 1) * 8;
      ldmatrix_x4_t(r, stage + ti.v_off + ((size_t)tok * D + ch) * 2);
      if (!full) {
        // element (row = channel, col = token): r0/r1 hold tokens 2tig, 2tig+1; r2/r3 tokens +8
        if (ta >= n) { r[0] &= 0xffff0000u; r[1] &= 0xffff0000u; }
        if (tb >= n) { r[0] &= 0x0000ffffu; r[1] &= 0x0000ffffu; }
        if (tc >= n) { r[2] &= 0xffff0000u; r[3] &= 0xffff0000u; }
        if (td >= n) { r[2] &= 0x0000ffffu; r[3] &= 0x0000ffffu; }
      }
      mma16816(S.accr[mt], r[0], r[1], r[2], r[3], b0, b1);
    }
  }
}

template <int B>
__global__ void __launch_bounds__(NTH, 2) decode_tc_kernel(const DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + TcSmem::bars);
  uint64_t* ready = full + kTcStages;
  uint64_t* empty = ready + kTcStages;
  volatile int* flags = reinterpret_cast<volatile int*>(smem + TcSmem::flags);
  __half* qnat = reinterpret_cast<__half*>(smem + TcSmem::qnat);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int pair = blockIdx.x / a.n_splits;
  const int split = blockIdx.x % a.n_splits;
  const int t_begin = a.split_tile[split], t_end = a.split_tile[split + 1];
  const int ntiles = t_end - t_begin;
  const int b = pair / a.h_kv, hk = pair % a.h_kv;
  const __half* qg = a.q + ((size_t)b * a.h_kv + hk) * D;

  if (tid == 0) {
    flags[0] = 0;
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&ready[s], 1);
      mbar_init(&empty[s], NCW);
    }
    mbar_fence_init();
  }
  for (int c = tid; c < D; c += NTH) qnat[c] = qg[c];
  __syncthreads();

  if (warp == NCW) {
    // ------------------------------------------------------------ producer
    auto issue = [&](int j) {
      const int st = j % kTcStages;
      if (j >= kTcStages &&
          !wait_or_abort(&empty[st], (uint32_t)(((j / kTcStages) & 1) ^ 1), flags))
        return false;
      if (lane == 0) {
        uint8_t* stage = smem + TcSmem::stages + st * kTcStageBytes;
        const TileInfo ti = tile_info(a, t_begin + j);
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(&full[st], ti.bytes);
        for_each_tile_copy(a, (size_t)pair, ti,
                           [&](const void* src, uint32_t off, uint32_t bytes, int, int) {
                             bulk_g2s(stage + off, src, bytes, &full[st]);
                           });
      }
      return true;
    };
    // lane = (tig, kt): the 4 channels of the K operand entry (tig, kt, b0/b1)
    const int ptig = lane >> 3, pkt = lane & 7;
    int ch[4], pw[4];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      int clo, chi, p;
      k_half2_channels<B>(ptig, 2 * pkt + e, &clo, &chi, &p);
      ch[2 * e] = clo;
      ch[2 * e + 1] = chi;
      pw[2 * e] = pw[2 * e + 1] = p;
    }
    float qv[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      qv[e] = __half2float(qnat[ch[e]]) * __uint_as_float((uint32_t)(127 - pw[e]) << 23);
    const float qz0 = __half2float(qnat[lane]), qz1 = __half2float(qnat[lane + 32]);
    const float qz2 = __half2float(qnat[lane + 64]), qz3 = __half2float(qnat[lane + 96]);
    bool ok = true;
    for (int j = 0; j < kTcStages - 1 && j < ntiles && ok; ++j) ok = issue(j);
    for (int it = 0; it < ntiles && ok; ++it) {
      const int st = it % kTcStages;
      const uint32_t ph = (uint32_t)((it / kTcStages) & 1);
      const TileInfo ti = tile_info(a, t_begin + it);
      if (ti.kseg >= 0) {
        if (!wait_or_abort(&full[st], ph, flags)) break;
        const uint8_t* stage = smem + TcSmem::stages + st * kTcStageBytes;
        const __half* ks = reinterpret_cast<const __half*>(stage + ti.ks_off);
        const __half* kz = reinterpret_cast<const __half*>(stage + ti.kz_off);
        uint32_t* kt_tab = reinterpret_cast<uint32_t*>(smem + TcSmem::ktab + st * kTcKtabBytes);
        float* kb = reinterpret_cast<float*>(smem + TcSmem::kbias) + st * kTcMaxGroups;
        for (int gl = 0; gl < ti.ng; ++gl) {
          const __half* sg = ks + gl * D;
          float v[4], hi[4], lo[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            v[e] = qv[e] * __half2float(sg[ch[e]]);
            hi[e] = __half2float(__float2half_rn(v[e]));
            lo[e] = v[e] - hi[e];
          }
          // entry (gl, part, tig, kt) holds b0 (h = 2kt) and b1 (h = 2kt+1)
          uint2* dh = reinterpret_cast<uint2*>(kt_tab + ((gl * 2 + 0) * 4 + ptig) * 16) + pkt;
          uint2* dl = reinterpret_cast<uint2*>(kt_tab + ((gl * 2 + 1) * 4 + ptig) * 16) + pkt;
          *dh = make_uint2(pack_half2(hi[0], hi[1]), pack_half2(hi[2], hi[3]));
          *dl = make_uint2(pack_half2(lo[0], lo[1]), pack_half2(lo[2], lo[3]));
          const __half* zg = kz + gl * D;
          float zsum = qz0 * __half2float(zg[lane]) + qz1 * __half2float(zg[lane + 32]) +
                       qz2 * __half2float(zg[lane + 64]) + qz3 * __half2float(zg[lane + 96]);
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) zsum += __shfl_xor_sync(0xffffffffu, zsum, off);
          if (lane == 0) kb[gl] = zsum;
        }
        __syncwarp();
      }
      if (lane == 0) mbar_arrive(&ready[st]);
      if (it + kTcStages - 1 < ntiles) ok = issue(it + kTcStages - 1);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  WarpState S;
  S.m = -INFINITY;
  S.l = S.zs = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) S.acc[i][e] = S.accr[i][e] = 0.f;

  for (int it = 0; it < ntiles; ++it) {
    const int st = it % kTcStages;
    const uint32_t ph = (uint32_t)((it / kTcStages) & 1);
    if (!wait_or_abort(&ready[st], ph, flags)) break;
    if (!wait_or_abort(&full[st], ph, flags)) break;
    const uint8_t* stage = smem + TcSmem::stages + st * kTcStageBytes;
    const int t = t_begin + it;
    const TileInfo ti = tile_info(a, t);
    int ri = 0;
    while (ri + 1 < a.n_runs && a.runs[ri + 1].tile0 <= t) ++ri;
    const int wt = a.runs[ri].wt;  // tokens of a warp slice (multiple of 16)
    const uint32_t* kt_tab = reinterpret_cast<const uint32_t*>(smem + TcSmem::ktab + st * kTcKtabBytes);
    const float* kb = reinterpret_cast<const float*>(smem + TcSmem::kbias) + st * kTcMaxGroups;
    for (int s0 = warp * wt; s0 < warp * wt + wt && s0 < ti.n; s0 += 16)
      sub_tile<B>(a, ti, stage, kt_tab, kb, qnat, s0, lane, S);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
  }

  // ---- this warp's output row, o[c] for all channels, into shared memory
  const int gid = lane >> 2, tig = lane & 3;
  float* mg = reinterpret_cast<float*>(smem + TcSmem::merge) + warp * (D + 2);
  // column sums over the 4 threads (tig) of each gid
  float zs = S.zs, l = S.l;
  zs += __shfl_xor_sync(0xffffffffu, zs, 1);
  zs += __shfl_xor_sync(0xffffffffu, zs, 2);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
  // zs of column n now sits in the threads with gid == n
  const int ngv = D >> a.log2G;
  // ring V (natural rows): thread (gid, tig == 0) has rows gid, gid + 8 of col 0
  // packed V: rows gid, gid + 8 of m-tile mt are channels v_rows(gid, mt);
  // their column is the channels' group g; the owner thread has tig == g / 2
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    int c0, c8, p;
    v_rows<B>(gid, mt, &c0, &c8, &p);
    const int g = c0 >> a.log2G;  // c0 and c8 share the group (16-channel block)
    const float zsg = __shfl_sync(0xffffffffu, zs, 4 * g);
    const float unscale = __uint_as_float((uint32_t)(127 + 24 - p) << 23);  // 2^(24 - p)
    if (tig == (g >> 1)) {
      const float d0 = (g & 1) ? S.acc[mt][1] : S.acc[mt][0];
      const float d8 = (g & 1) ? S.acc[mt][3] : S.acc[mt][2];
      mg[c0] = d0 * unscale + zsg;
      mg[c8] = d8 * unscale + zsg;
    }
  }
  __syncwarp();
  if (tig == 0) {
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      mg[mt * 16 + gid] += S.accr[mt][0];
      mg[mt * 16 + gid + 8] += S.accr[mt][2];
    }
  }
  (void)ngv;
  if (lane == 0) {
    mg[D] = S.m;
    mg[D + 1] = l;
  }
  asm volatile("bar.sync 1, %0;" ::"r"(NCW * 32) : "memory");
  if (flags[0]) {
    if (tid == 0) atomicExch(a.err, 1);
    return;
  }
  // ---- merge the consumer warps
  const float* m0 = reinterpret_cast<const float*>(smem + TcSmem::merge);
  float M = -INFINITY;
  for (int w = 0; w < NCW; ++w) M = fmaxf(M, m0[w * (D + 2) + D]);
  const size_t out_base = ((size_t)b * a.h_kv + hk) * D;
  float* rec = a.part + ((size_t)pair * a.n_splits + split) * (D + 2);
  for (int c = tid; c < D; c += NCW * 32) {
    float L = 0.f, O = 0.f;
    for (int w = 0; w < NCW; ++w) {
      const float* mw = m0 + w * (D + 2);
      const float sw = (mw[D] == -INFINITY) ? 0.f : exp2f(mw[D] - M);
      L += mw[D + 1] * sw;
      O += mw[c] * sw;
    }
    if (a.n_splits == 1) {
      a.out[out_base + c] = __float2half_rn(O / L);
    } else {
      rec[c] = O;
      if (c == 0) {
        rec[D] = M;
        rec[D + 1] = L;
      }
    }
  }
  if (a.n_splits == 1) return;
  __threadfence();
  asm volatile("bar.sync 1, %0;" ::"r"(NCW * 32) : "memory");
  if (tid == 0) flags[1] = (atomicAdd(&a.counters[pair], 1) == a.n_splits - 1);
  asm volatile("bar.sync 1, %0;" ::"r"(NCW * 32) : "memory");
  if (!flags[1]) return;
  __threadfence();
  const float* recs = a.part + (size_t)pair * a.n_splits * (D + 2);
  for (int c = tid; c < D; c += NCW * 32) {
    float MM = -INFINITY;
    for (int s = 0; s < a.n_splits; ++s) MM = fmaxf(MM, __ldcg(recs + (size_t)s * (D + 2) + D));
    float L = 0.f, O = 0.f;
    for (int s = 0; s < a.n_splits; ++s) {
      const float* rr = recs + (size_t)s * (D + 2);
      const float w = exp2f(__ldcg(rr + D) - MM);
      L += __ldcg(rr + D + 1) * w;
      O += __ldcg(rr + c) * w;
    }
    a.out[out_base + c] = __float2half_rn(O / L);
  }
  if (tid == 0) a.counters[pair] = 0;
}

template <int B>
cudaError_t launch_tc_b(const DecodeArgs& a, int n_pairs, cudaStream_t s) {
  const int smem = TcSmem::total;
  cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel<B>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  decode_tc_kernel<B><<<n_pairs * a.n_splits, NTH, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_tc(const DecodeArgs& a, int n_pairs, int bits, cudaStream_t s) {
  if (bits == 2) return launch_tc_b<2>(a, n_pairs, s);
  if (bits == 4) return launch_tc_b<4>(a, n_pairs, s);
  return launch_tc_b<8>(a, n_pairs, s);
}

}  // namespace kvq
