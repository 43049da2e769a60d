// Decode attention for one query head per kv head (MHA) over a single packed
// segment plus the fp16 ring: the KIVI cache layout (KIVI page, Algorithm 1
// decoding branch: A = Concat(t_Q Q(X_Kg)^T, t_Q X_Kr^T), softmax,
// t_O = A_g Q(X_Vg) + A_r X_Vr).
//
// One CTA = one producer warp + 8 consumer warps, one (batch, kv head) and a
// contiguous range of its tiles.  The producer stages each tile with bulk
// copies (TMA engine) and, for packed K, builds the tile's scaled-query table
// q_c * s_gc (one row per K group) and bias sum_c q_c z_gc; consumers wait on
// the tile's "ready" mbarrier, each takes its own slice of the tile's tokens,
// and release the stage on an "empty" mbarrier.  Consumers never synchronize
// with each other inside the loop: each warp keeps its own online softmax and
// accumulators and the warps are merged once at the end.
//
// Inner loops, per cached element: one LOP3 turns a packed code field into a
// float (the field is OR-ed into the mantissa of 2^23; fields above bit 21 are
// first shifted down once per word), one packed fp32 add removes 2^23 (two
// elements per instruction) and one packed fp32 FMA accumulates (two elements
// per instruction).  The power of two a field sits at is folded into the
// scaled-query table (K) or removed from the output at the end (V).
#include <float.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int NCW = kMhaConsumerWarps;  // consumer warps
constexpr int NTH = (NCW + 1) * 32;     // + producer warp
constexpr float kMagic = 8388608.0f;    // 2^23

struct MhaSmem {
  // offsets (bytes) from the dynamic shared memory base
  static constexpr int stages = 0;
  static constexpr int qtab = stages + kStages * kMhaStageBytes;      // [stage][groups][4][36] f32
  static constexpr int bias = qtab + kStages * kMhaQtabBytes;         // [stage][groups] f32
  static constexpr int qraw = bias + kStages * kMhaMaxGroups * 4;     // [4][36] f32 (raw q)
  static constexpr int merge = qraw + 4 * 36 * 4;                     // [NCW][128 + 4] f32
  static constexpr int bars = merge + NCW * (128 + 4) * 4;            // full/ready/empty
  static constexpr int flags = bars + 3 * kStages * 8;
  static constexpr int total = flags + 16;
};

// bit offset of code j (0-based within its 32-bit word) after the optional
// down-shift of the word's high fields
template <int B>
__host__ __device__ constexpr int field_shift(int j) {
  return j <= (23 - B) / B ? j * B : j * B - ((23 - B) / B + 1) * B;
}

// 2^-field_shift(j) and 2^field_shift(j) as exact floats
template <int B>
__device__ __forceinline__ float field_unscale(int j) {
  return __uint_as_float((uint32_t)(127 - field_shift<B>(j)) << 23);
}
template <int B>
__device__ __forceinline__ float field_scale(int j) {
  return __uint_as_float((uint32_t)(127 + field_shift<B>(j)) << 23);
}

template <int B>
__device__ __forceinline__ void word_fields(uint32_t w, float (&f)[32 / B]) {
  constexpr int N = 32 / B, direct = (23 - B) / B, sh = (direct + 1) * B;
  constexpr uint32_t mask = (1u << B) - 1u;
  const uint32_t hi = w >> sh;
#pragma unroll
  for (int j = 0; j < N; ++j) {
    const uint32_t m = mask << field_shift<B>(j);
    f[j] = __uint_as_float(((j <= direct ? w : hi) & m) | 0x4B000000u);
  }
}

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity,
                                              volatile int* abort_flag) {
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

// Per-warp state of the online softmax and the PV accumulators of one lane.
// acc[k] holds channels (2k, 2k+1) of the lane's quarter, each scaled by
// 2^field_shift of its code field.
template <int D>
struct LaneState {
  float m;       // running max (log2 domain), warp-uniform
  float l;       // this lane's share of the denominator
  float zsum;    // packed V: sum p z of this lane's V group
  float2 acc[D / 8];
};

// One tile's slice of a warp: TPL tokens per lane (slice of 8 * TPL tokens).
template <int D, int B, int TPL>
__device__ __forceinline__ void consume_slice(const DecodeArgs& a, const TileInfo& ti,
                                              const uint8_t* stage, const float* qt,
                                              const float* bs, const float* qraw, int w0,
                                              int lane, LaneState<D>& S) {
  constexpr int CPL = D / 4, WPL = CPL * B / 32, FPW = 32 / B;
  const int r = lane >> 2, cq = lane & 3;
  float part[4] = {0.f, 0.f, 0.f, 0.f};
  // ---- partial scores over this lane's channel quarter
  if (ti.kseg >= 0) {
    // scaled query of the group of the lane's first token; reloaded only if a
    // later token of the slice lies in another group (unaligned runs, G < 32)
    int gl_cur = min(((ti.ku0 + min(w0 + r, ti.n - 1)) >> a.log2G) - ti.g0, ti.ng - 1);
    float2 qk[CPL / 2];
    {
      const float4* row = reinterpret_cast<const float4*>(qt + (gl_cur * 4 + cq) * 36);
#pragma unroll
      for (int k = 0; k < CPL / 4; ++k) {
        const float4 v = row[k];
        qk[2 * k] = make_float2(v.x, v.y);
        qk[2 * k + 1] = make_float2(v.z, v.w);
      }
    }
#pragma unroll 1
    for (int i = 0; i < TPL; ++i) {
      const int tok = w0 + r + 8 * i;
      if (tok < ti.n) {
        const int gl = min(((ti.ku0 + tok) >> a.log2G) - ti.g0, ti.ng - 1);
        if (gl != gl_cur) {
          gl_cur = gl;
          const float4* row = reinterpret_cast<const float4*>(qt + (gl * 4 + cq) * 36);
#pragma unroll
          for (int k = 0; k < CPL / 4; ++k) {
            const float4 v = row[k];
            qk[2 * k] = make_float2(v.x, v.y);
            qk[2 * k + 1] = make_float2(v.z, v.w);
          }
        }
        const uint32_t* cw = reinterpret_cast<const uint32_t*>(
                                 stage + ti.k_off + (size_t)tok * (D * B / 8)) + cq * WPL;
        uint32_t wv[WPL];
        if (WPL >= 4) {
#pragma unroll
          for (int k = 0; k < WPL; k += 4) *reinterpret_cast<uint4*>(&wv[k]) = *reinterpret_cast<const uint4*>(cw + k);
        } else if (WPL == 2) {
          *reinterpret_cast<uint2*>(&wv[0]) = *reinterpret_cast<const uint2*>(cw);
        } else {
          wv[0] = cw[0];
        }
        float2 s2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int wi = 0; wi < WPL; ++wi) {
          float f[FPW];
          word_fields<B>(wv[wi], f);
#pragma unroll
          for (int j = 0; j < FPW; j += 2) {
            const float2 v = fadd2(make_float2(f[j], f[j + 1]), make_float2(-kMagic, -kMagic));
            s2[(j >> 1) & 1] = ffma2(qk[(wi * FPW + j) / 2], v, s2[(j >> 1) & 1]);
          }
        }
        const float pv = (s2[0].x + s2[1].x) + (s2[0].y + s2[1].y) + (cq == 0 ? bs[gl] : 0.f);
        part[0] = i == 0 ? pv : part[0];
        part[1] = i == 1 ? pv : part[1];
        part[2] = i == 2 ? pv : part[2];
        part[3] = i == 3 ? pv : part[3];
      }
    }
  } else {
#pragma unroll 1
    for (int i = 0; i < TPL; ++i) {
      const int tok = w0 + r + 8 * i;
      if (tok < ti.n) {
        const uint4* row =
            reinterpret_cast<const uint4*>(stage + ti.k_off + (size_t)tok * D * 2 + cq * CPL * 2);
        const float4* qv = reinterpret_cast<const float4*>(qraw + cq * 36);
        float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < CPL / 8; ++k) {
          const uint4 raw = row[k];
          const __half2* h2 = reinterpret_cast<const __half2*>(&raw);
          const float4 q0 = qv[2 * k], q1 = qv[2 * k + 1];
          s2 = ffma2(make_float2(q0.x, q0.y), __half22float2(h2[0]), s2);
          s2 = ffma2(make_float2(q0.z, q0.w), __half22float2(h2[1]), s2);
          s2 = ffma2(make_float2(q1.x, q1.y), __half22float2(h2[2]), s2);
          s2 = ffma2(make_float2(q1.z, q1.w), __half22float2(h2[3]), s2);
        }
        const float pv = s2.x + s2.y;
        part[0] = i == 0 ? pv : part[0];
        part[1] = i == 1 ? pv : part[1];
        part[2] = i == 2 ? pv : part[2];
        part[3] = i == 3 ? pv : part[3];
      }
    }
  }
  // ---- sum the 4 quarters; lane (r, cq) ends with token r + 8 * sel
  float sc;
  int sel;
  if (TPL == 4) {
    const bool hi2 = (cq & 2) != 0, hi1 = (cq & 1) != 0;
    float k0 = hi2 ? part[2] : part[0], k1 = hi2 ? part[3] : part[1];
    const float s0 = hi2 ? part[0] : part[2], s1 = hi2 ? part[1] : part[3];
    k0 += __shfl_xor_sync(0xffffffffu, s0, 2);
    k1 += __shfl_xor_sync(0xffffffffu, s1, 2);
    const float keep = hi1 ? k1 : k0, send = hi1 ? k0 : k1;
    sc = keep + __shfl_xor_sync(0xffffffffu, send, 1);
    sel = (hi2 ? 2 : 0) + (hi1 ? 1 : 0);
  } else if (TPL == 2) {
    const bool hi2 = (cq & 2) != 0;
    float keep = hi2 ? part[1] : part[0];
    const float send = hi2 ? part[0] : part[1];
    keep += __shfl_xor_sync(0xffffffffu, send, 2);
    sc = keep + __shfl_xor_sync(0xffffffffu, keep, 1);
    sel = hi2 ? 1 : 0;
  } else {
    float v = part[0];
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    sc = v + __shfl_xor_sync(0xffffffffu, v, 1);
    sel = 0;
  }
  const bool valid = w0 + r + 8 * sel < ti.n;
  sc = valid ? sc * a.scale_log2 : -INFINITY;
  // ---- online softmax over the warp
  float mx = sc;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  const float m_new = fmaxf(S.m, mx);
  const float alpha = (m_new == -INFINITY) ? 1.f : exp2f(S.m - m_new);
  const float p = valid ? exp2f(sc - m_new) : 0.f;
  const bool owner = (TPL == 4) || (TPL == 2 ? (cq & 1) == 0 : cq == 0);
  S.l = S.l * alpha + (owner ? p : 0.f);
  S.m = m_new;
  if (alpha != 1.f) {
    S.zsum *= alpha;
    const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
    for (int k = 0; k < CPL / 2; ++k) S.acc[k] = make_float2(S.acc[k].x * a2.x, S.acc[k].y * a2.y);
  }
  // ---- PV over this lane's tokens r + 8 i
  const int ngv = D >> a.log2Gv;
  const int gv = (cq * CPL) >> a.log2Gv;
#pragma unroll 1
  for (int i = 0; i < TPL; ++i) {
    const int src = TPL == 4 ? (r * 4 + i) : (TPL == 2 ? (r * 4 + 2 * i) : lane);
    const float pt = __shfl_sync(0xffffffffu, p, src);
    const int tok = w0 + r + 8 * i;
    if (tok < ti.n) {
      if (ti.vseg >= 0) {
        const __half* vs = reinterpret_cast<const __half*>(stage + ti.vs_off);
        const __half* vz = reinterpret_cast<const __half*>(stage + ti.vz_off);
        const float ps = pt * __half2float(vs[tok * ngv + gv]);
        S.zsum = fmaf(pt, zero_add(__half_as_ushort(vz[tok * ngv + gv]), __half_as_ushort(vs[tok * ngv + gv]), a.intz),
                      S.zsum);
        const float2 ps2 = make_float2(ps, ps);
        const uint32_t* cw = reinterpret_cast<const uint32_t*>(
                                 stage + ti.v_off + (size_t)tok * (D * B / 8)) + cq * WPL;
        uint32_t wv[WPL];
        if (WPL >= 4) {
#pragma unroll
          for (int k = 0; k < WPL; k += 4) *reinterpret_cast<uint4*>(&wv[k]) = *reinterpret_cast<const uint4*>(cw + k);
        } else if (WPL == 2) {
          *reinterpret_cast<uint2*>(&wv[0]) = *reinterpret_cast<const uint2*>(cw);
        } else {
          wv[0] = cw[0];
        }
#pragma unroll
        for (int wi = 0; wi < WPL; ++wi) {
          float f[FPW];
          word_fields<B>(wv[wi], f);
#pragma unroll
          for (int j = 0; j < FPW; j += 2) {
            const float2 v = fadd2(make_float2(f[j], f[j + 1]), make_float2(-kMagic, -kMagic));
            S.acc[(wi * FPW + j) / 2] = ffma2(ps2, v, S.acc[(wi * FPW + j) / 2]);
          }
        }
      } else {
        // fp16 ring V: scale by 2^field_shift so it joins the packed sums
        const uint4* row =
            reinterpret_cast<const uint4*>(stage + ti.v_off + (size_t)tok * D * 2 + cq * CPL * 2);
#pragma unroll
        for (int k = 0; k < CPL / 8; ++k) {
          const uint4 raw = row[k];
          const __half2* h2 = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int c0 = 8 * k + 2 * e;
            const float2 pf = make_float2(pt * field_scale<B>(c0 % FPW), pt * field_scale<B>((c0 + 1) % FPW));
            S.acc[4 * k + e] = ffma2(pf, __half22float2(h2[e]), S.acc[4 * k + e]);
          }
        }
      }
    }
  }
}

template <int D, int B>
__global__ void __launch_bounds__(NTH, 2) decode_mha_kernel(const DecodeArgs a) {
  constexpr int CPL = D / 4;
  constexpr int FPW = 32 / B;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + MhaSmem::bars);
  uint64_t* ready = full + kStages;
  uint64_t* empty = ready + kStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + MhaSmem::flags);
  float* qraw = reinterpret_cast<float*>(smem + MhaSmem::qraw);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int pair = blockIdx.x / a.n_splits;
  const int split = blockIdx.x % a.n_splits;
  const int t_begin = a.split_tile[split], t_end = a.split_tile[split + 1];
  const int ntiles = t_end - t_begin;
  const int b = pair / a.h_kv, hk = pair % a.h_kv;
  const __half* qg = a.q + ((size_t)b * a.h_kv + hk) * D;

  if (tid == 0) {
    abort_flag[0] = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&ready[s], 1);
      mbar_init(&empty[s], NCW);
    }
    mbar_fence_init();
  }
  for (int c = tid; c < D; c += NTH) qraw[(c / CPL) * 36 + c % CPL] = __half2float(qg[c]);
  __syncthreads();

  if (warp == NCW) {
    // ------------------------------------------------------------ producer
    // Order per step: build the scaled-query table of tile `it` (its copies
    // were issued kStages-1 steps earlier), release it to the consumers, then
    // issue the copies of tile it + kStages - 1 into the stage that tile
    // it - 1 used.  Loads stay kStages - 1 tiles ahead of the consumers.
    int nissued = 0;
    auto issue = [&](int j) {
      const int st = j % kStages;
      if (j >= kStages) {
        if (!wait_or_abort(&empty[st], (uint32_t)(((j / kStages) & 1) ^ 1), abort_flag)) return false;
        // consumers that gave up release a stage without waiting for it
        if (!mbar_drain_bounded(&full[st], (uint32_t)(((j / kStages) & 1) ^ 1)) && lane == 0) atomicExch(a.err, 1);
      }
      nissued = j + 1;
      if (lane == 0) {
        uint8_t* stage = smem + MhaSmem::stages + st * kMhaStageBytes;
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
    // lane l owns channels 4l .. 4l+3 (lanes >= D/4 idle); q_c * 2^-field_shift
    const bool own = lane < D / 4;
    const int c0 = 4 * lane;
    float qf[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int c = own ? c0 + e : 0;
      qf[e] = qraw[(c / CPL) * 36 + c % CPL] * field_unscale<B>(c % FPW);
    }
    float qz[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int c = own ? c0 + e : 0;
      qz[e] = own ? qraw[(c / CPL) * 36 + c % CPL] : 0.f;
    }
    bool ok = true;
    for (int j = 0; j < kStages - 1 && j < ntiles && ok; ++j) ok = issue(j);
    for (int it = 0; it < ntiles && ok; ++it) {
      const int st = it % kStages;
      const uint32_t ph = (uint32_t)((it / kStages) & 1);
      const TileInfo ti = tile_info(a, t_begin + it);
      if (ti.kseg >= 0) {
        if (!wait_or_abort(&full[st], ph, abort_flag)) break;
        const uint8_t* stage = smem + MhaSmem::stages + st * kMhaStageBytes;
        const __half* ks = reinterpret_cast<const __half*>(stage + ti.ks_off);
        const __half* kz = reinterpret_cast<const __half*>(stage + ti.kz_off);
        float* qt = reinterpret_cast<float*>(smem + MhaSmem::qtab + st * kMhaQtabBytes);
        float* bs = reinterpret_cast<float*>(smem + MhaSmem::bias) + st * kMhaMaxGroups;
        float bp[kMhaMaxGroups];
#pragma unroll
        for (int gl = 0; gl < kMhaMaxGroups; ++gl) {
          bp[gl] = 0.f;
          if (gl < ti.ng && own) {
            const uint2 sr = *reinterpret_cast<const uint2*>(ks + gl * D + c0);
            const uint2 zr = *reinterpret_cast<const uint2*>(kz + gl * D + c0);
            const float2 s01 = __half22float2(*reinterpret_cast<const __half2*>(&sr.x));
            const float2 s23 = __half22float2(*reinterpret_cast<const __half2*>(&sr.y));
            float2 z01 = __half22float2(*reinterpret_cast<const __half2*>(&zr.x));
            float2 z23 = __half22float2(*reinterpret_cast<const __half2*>(&zr.y));
            if (a.intz) {  // the additive zero -s z of the integer zero point
              z01 = make_float2(-s01.x * (float)(short)(zr.x & 0xffffu), -s01.y * (float)(short)(zr.x >> 16));
              z23 = make_float2(-s23.x * (float)(short)(zr.y & 0xffffu), -s23.y * (float)(short)(zr.y >> 16));
            }
            *reinterpret_cast<float4*>(qt + (gl * 4 + c0 / CPL) * 36 + c0 % CPL) =
                make_float4(qf[0] * s01.x, qf[1] * s01.y, qf[2] * s23.x, qf[3] * s23.y);
            bp[gl] = qz[0] * z01.x + qz[1] * z01.y + qz[2] * z23.x + qz[3] * z23.y;
          }
        }
        // bias per group: sum bp[gl] over the lanes (all groups at once)
#pragma unroll
        for (int gl = 0; gl < kMhaMaxGroups; ++gl) {
          if (gl < ti.ng) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) bp[gl] += __shfl_xor_sync(0xffffffffu, bp[gl], off);
          }
        }
        if (lane == 0) {
#pragma unroll
          for (int gl = 0; gl < kMhaMaxGroups; ++gl)
            if (gl < ti.ng) bs[gl] = bp[gl];
        }
        __syncwarp();
      }
      if (lane == 0) mbar_arrive(&ready[st]);
      if (it + kStages - 1 < ntiles) ok = issue(it + kStages - 1);
    }
    // no copy of this block may still be in flight when it exits
    for (int j = nissued > kStages ? nissued - kStages : 0; j < nissued; ++j)
      if (!mbar_drain_bounded(&full[j % kStages], (uint32_t)((j / kStages) & 1)) && lane == 0) atomicExch(a.err, 1);
    return;
  }

  // -------------------------------------------------------------- consumers
  LaneState<D> S;
  S.m = -INFINITY;
  S.l = 0.f;
  S.zsum = 0.f;
#pragma unroll
  for (int k = 0; k < CPL / 2; ++k) S.acc[k] = make_float2(0.f, 0.f);

  for (int it = 0; it < ntiles; ++it) {
    const int st = it % kStages;
    const uint32_t ph = (uint32_t)((it / kStages) & 1);
    if (!wait_or_abort(&ready[st], ph, abort_flag)) break;
    if (!wait_or_abort(&full[st], ph, abort_flag)) break;
    const uint8_t* stage = smem + MhaSmem::stages + st * kMhaStageBytes;
    const int t = t_begin + it;
    const TileInfo ti = tile_info(a, t);
    int ri = 0;
    while (ri + 1 < a.n_runs && a.runs[ri + 1].tile0 <= t) ++ri;
    const int wt = a.runs[ri].wt;  // tokens per warp slice: 8, 16 or 32
    const int w0 = warp * wt;
    if (w0 < ti.n) {
      const float* qt = reinterpret_cast<const float*>(smem + MhaSmem::qtab + st * kMhaQtabBytes);
      const float* bs = reinterpret_cast<const float*>(smem + MhaSmem::bias) + st * kMhaMaxGroups;
      if (wt == 32) consume_slice<D, B, 4>(a, ti, stage, qt, bs, qraw, w0, lane, S);
      else if (wt == 16) consume_slice<D, B, 2>(a, ti, stage, qt, bs, qraw, w0, lane, S);
      else consume_slice<D, B, 1>(a, ti, stage, qt, bs, qraw, w0, lane, S);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
  }

  // ---- per-warp result for this lane's quarter, summed over the 8 rows
  const int r = lane >> 2, cq = lane & 3;
  float* mg = reinterpret_cast<float*>(smem + MhaSmem::merge) + warp * (128 + 4);
  float lw = S.l;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) lw += __shfl_xor_sync(0xffffffffu, lw, off);
#pragma unroll
  for (int k = 0; k < CPL / 2; ++k) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int cl = 2 * k + e;
      float v = (e ? S.acc[k].y : S.acc[k].x) * field_unscale<B>(cl % FPW) + S.zsum;
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      v += __shfl_xor_sync(0xffffffffu, v, 16);
      if (r == 0) mg[cq * CPL + cl] = v;
    }
  }
  if (lane == 0) {
    mg[D] = S.m;
    mg[D + 1] = lw;
  }
  asm volatile("bar.sync 1, %0;" ::"r"(NCW * 32) : "memory");
  if (abort_flag[0]) {
    if (tid == 0) atomicExch(a.err, 1);
    return;
  }
  // ---- merge the consumer warps
  const float* m0 = reinterpret_cast<const float*>(smem + MhaSmem::merge);
  float M = -INFINITY;
  for (int w = 0; w < NCW; ++w) M = fmaxf(M, m0[w * (128 + 4) + D]);
  const size_t out_base = ((size_t)b * a.h_kv + hk) * D;
  float* rec = a.part + ((size_t)pair * a.n_splits + split) * (D + 2);
  for (int c = tid; c < D; c += NCW * 32) {
    float L = 0.f, O = 0.f;
    for (int w = 0; w < NCW; ++w) {
      const float* mw = m0 + w * (128 + 4);
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
  if (tid == 0) abort_flag[1] = (atomicAdd(&a.counters[pair], 1) == a.n_splits - 1);
  asm volatile("bar.sync 1, %0;" ::"r"(NCW * 32) : "memory");
  if (!abort_flag[1]) return;
  __threadfence();
  // Merge of the splits' records: the weights 2^(m_s - M) / L of the splits
  // first (one warp, into the merge area the warps no longer read), then each
  // channel as a sum of independent loads.
  const float* recs = a.part + (size_t)pair * a.n_splits * (D + 2);
  float* wts = reinterpret_cast<float*>(smem + MhaSmem::merge);
  static_assert(KVQ_MAX_SPLITS <= NCW * (128 + 4), "split weights fit the merge area");
  if (warp == 0) {
    float MM = -INFINITY;
    for (int sp = lane; sp < a.n_splits; sp += 32) MM = fmaxf(MM, __ldcg(recs + (size_t)sp * (D + 2) + D));
    for (int off = 16; off > 0; off >>= 1) MM = fmaxf(MM, __shfl_xor_sync(0xffffffffu, MM, off));
    float L = 0.f;
    for (int sp = lane; sp < a.n_splits; sp += 32) {
      const float* rr = recs + (size_t)sp * (D + 2);
      const float w = exp2f(__ldcg(rr + D) - MM);
      wts[sp] = w;
      L += __ldcg(rr + D + 1) * w;
    }
    for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
    __syncwarp();
    const float inv = 1.f / L;
    for (int sp = lane; sp < a.n_splits; sp += 32) wts[sp] *= inv;
  }
  asm volatile("bar.sync 1, %0;" ::"r"(NCW * 32) : "memory");
  for (int c = tid; c < D; c += NCW * 32) {
    float O = 0.f;
#pragma unroll 8
    for (int sp = 0; sp < a.n_splits; ++sp) O += __ldcg(recs + (size_t)sp * (D + 2) + c) * wts[sp];
    a.out[out_base + c] = __float2half_rn(O);
  }
  if (tid == 0) a.counters[pair] = 0;
}

template <int D, int B>
cudaError_t launch_mha_db(const DecodeArgs& a, int n_pairs, cudaStream_t s) {
  const int smem = MhaSmem::total;
  cudaError_t e = set_smem_once((const void*)decode_mha_kernel<D, B>, (int)smem);
  if (e != cudaSuccess) return e;
  decode_mha_kernel<D, B><<<n_pairs * a.n_splits, NTH, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

size_t decode_mha_smem_bytes() { return MhaSmem::total; }

cudaError_t launch_decode_mha(const DecodeArgs& a, int n_pairs, int bits, cudaStream_t s) {
  if (a.d == 128) {
    if (bits == 2) return launch_mha_db<128, 2>(a, n_pairs, s);
    if (bits == 4) return launch_mha_db<128, 4>(a, n_pairs, s);
    return launch_mha_db<128, 8>(a, n_pairs, s);
  }
  if (bits == 2) return launch_mha_db<64, 2>(a, n_pairs, s);
  if (bits == 4) return launch_mha_db<64, 4>(a, n_pairs, s);
  return launch_mha_db<64, 8>(a, n_pairs, s);
}

}  // namespace kvq
