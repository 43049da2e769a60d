// Fused split-K decode attention over a quantized KV cache.
//
// Computes, per (batch, kv head) and for each of its gq query heads,
//   a_t = sm_scale * q . k_t,  p = softmax(a),  out = sum_t p_t v_t
// where k_t / v_t are dequantized packed tokens (code * s + z) or fp16 ring
// tokens (KIVI page, Algorithm 1 decoding branch: A = Concat(t_Q Q(X_Kg)^T,
// t_Q X_Kr^T), t_O = A_g Q(X_Vg) + A_r X_Vr; WindowQuant §3.3.1: the same
// over several bit-width segments).  The token axis of a head is cut into
// tiles and the tiles into splits, one CTA per (head, split); a CTA streams
// its tiles through a bulk-copy (TMA engine) shared-memory pipeline and keeps
// an fp32 online softmax; the last CTA of a head merges the splits
// (FlashDecoding, VQ-LLM page reference [10]).
//
// Algebra used to avoid dequantizing K element by element: for a packed K
// group g, q . k_t = sum_c (q_c s_gc) code_tc + sum_c q_c z_gc, so each tile
// first builds the scaled query q_c s_gc and the bias sum_c q_c z_gc per
// group; for packed V, sum_t p_t (code s_t + z_t) = sum_t (p_t s_t) code +
// sum_t p_t z_t per channel group.
#include <float.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int NT = kDecodeThreads;

// Issue the bulk copies of tile t into `stage` (one thread).
__device__ void issue_tile(const DecodeArgs& a, size_t pair, int t, uint8_t* stage,
                           uint64_t* bar) {
  const TileInfo ti = tile_info(a, t);
  mbar_arrive_expect_tx(bar, ti.bytes);
  for_each_tile_copy(a, pair, ti, [&](const void* src, uint32_t off, uint32_t bytes, int, int) {
    bulk_g2s(stage + off, src, bytes, bar);
  });
}

// Code j (0..7) of a chunk of 8 codes held in `w` (bits per code `B`), as fp32.
template <int B>
__device__ __forceinline__ float code_f(uint32_t w, int j) {
  return __uint_as_float(((w >> (j * B)) & ((1u << B) - 1u)) | 0x4B000000u) - 8388608.0f;
}

// Load the 8-channel chunk of packed codes at byte address p (B bits each).
template <int B>
__device__ __forceinline__ void load_chunk(const uint8_t* p, uint32_t& lo, uint32_t& hi) {
  if (B == 2) {
    lo = *reinterpret_cast<const uint16_t*>(p);
    hi = 0;
  } else if (B == 4) {
    lo = *reinterpret_cast<const uint32_t*>(p);
    hi = 0;
  } else {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    lo = v.x;
    hi = v.y;
  }
}

template <int B>
__device__ __forceinline__ float code8(uint32_t lo, uint32_t hi, int j) {
  if (B == 8) return j < 4 ? code_f<8>(lo, j) : code_f<8>(hi, j - 4);
  return code_f<B>(lo, j);
}

// Scores of the tile's tokens for packed K of B bits: thread-per-token with
// TPT threads sharing a token (channels split), partial sums reduced by
// shuffles.  sc[h][tok] receives the log2-domain score.
template <int D, int GQ, int B, class A>
__device__ void scores_packed(const A& a, const TileInfo& ti, const uint8_t* stage,
                              const float* qs, const float* bias, float* sc) {
  constexpr int RB = D * B / 8;
  const int tpt = NT / max(ti.n <= 32 ? 32 : (ti.n <= 64 ? 64 : 128), 1);
  const int tid = threadIdx.x;
  const int tok = tid / tpt, part = tid % tpt;
  const int ch = D / tpt;  // channels of this thread
  float acc[GQ];
#pragma unroll
  for (int h = 0; h < GQ; ++h) acc[h] = 0.f;
  const bool live = tok < ti.n;
  int gl = 0;
  if (live) {
    gl = (ti.ku0 + tok) / a.G - ti.g0;
    const uint8_t* row = stage + ti.k_off + tok * RB;
    for (int c0 = part * ch; c0 < part * ch + ch; c0 += 8) {
      uint32_t lo, hi;
      load_chunk<B>(row + c0 * B / 8, lo, hi);
#pragma unroll
      for (int h = 0; h < GQ; ++h) {
        if (h >= a.gq) break;
        const float4* qv = reinterpret_cast<const float4*>(qs + ((size_t)gl * a.gq + h) * D + c0);
        const float4 q0 = qv[0], q1 = qv[1];
        acc[h] += q0.x * code8<B>(lo, hi, 0) + q0.y * code8<B>(lo, hi, 1) +
                  q0.z * code8<B>(lo, hi, 2) + q0.w * code8<B>(lo, hi, 3) +
                  q1.x * code8<B>(lo, hi, 4) + q1.y * code8<B>(lo, hi, 5) +
                  q1.z * code8<B>(lo, hi, 6) + q1.w * code8<B>(lo, hi, 7);
      }
    }
  }
#pragma unroll
  for (int h = 0; h < GQ; ++h)
    for (int off = 1; off < tpt; off <<= 1) acc[h] += __shfl_xor_sync(0xffffffffu, acc[h], off);
  if (live && part == 0) {
#pragma unroll
    for (int h = 0; h < GQ; ++h)
      if (h < a.gq) sc[h * 128 + tok] = (acc[h] + bias[gl * a.gq + h]) * a.scale_log2;
  }
}

// Scores for fp16 ring K.
template <int D, int GQ, class A>
__device__ void scores_ring(const A& a, const TileInfo& ti, const uint8_t* stage,
                            const float* q_s, float* sc) {
  const int tpt = NT / (ti.n <= 32 ? 32 : (ti.n <= 64 ? 64 : 128));
  const int tid = threadIdx.x;
  const int tok = tid / tpt, part = tid % tpt;
  const int ch = D / tpt;
  float acc[GQ];
#pragma unroll
  for (int h = 0; h < GQ; ++h) acc[h] = 0.f;
  const bool live = tok < ti.n;
  if (live) {
    const __half* row = reinterpret_cast<const __half*>(stage + ti.k_off) + tok * D;
    for (int c0 = part * ch; c0 < part * ch + ch; c0 += 8) {
      const uint4 raw = *reinterpret_cast<const uint4*>(row + c0);
      const __half2* h2 = reinterpret_cast<const __half2*>(&raw);
      const float2 k0 = __half22float2(h2[0]), k1 = __half22float2(h2[1]);
      const float2 k2 = __half22float2(h2[2]), k3 = __half22float2(h2[3]);
#pragma unroll
      for (int h = 0; h < GQ; ++h) {
        if (h >= a.gq) break;
        const float4* qv = reinterpret_cast<const float4*>(q_s + h * D + c0);
        const float4 q0 = qv[0], q1 = qv[1];
        acc[h] += q0.x * k0.x + q0.y * k0.y + q0.z * k1.x + q0.w * k1.y + q1.x * k2.x +
                  q1.y * k2.y + q1.z * k3.x + q1.w * k3.y;
      }
    }
  }
#pragma unroll
  for (int h = 0; h < GQ; ++h)
    for (int off = 1; off < tpt; off <<= 1) acc[h] += __shfl_xor_sync(0xffffffffu, acc[h], off);
  if (live && part == 0) {
#pragma unroll
    for (int h = 0; h < GQ; ++h)
      if (h < a.gq) sc[h * 128 + tok] = acc[h] * a.scale_log2;
  }
}

// PV for packed V of B bits: thread owns an 8-channel chunk and a token slot.
template <int D, int GQ, int B, class A>
__device__ void pv_packed(const A& a, const TileInfo& ti, const uint8_t* stage,
                          const float* sc, float (&acc)[GQ][8], float (&zsum)[GQ]) {
  constexpr int CHUNKS = D / 8, SLOTS = NT / CHUNKS, RB = D * B / 8;
  const int k = threadIdx.x % CHUNKS, slot = threadIdx.x / CHUNKS;
  const int ngrp = D / a.Gv;
  const int g = (8 * k) / a.Gv;
  const __half* vs = reinterpret_cast<const __half*>(stage + ti.vs_off);
  const __half* vz = reinterpret_cast<const __half*>(stage + ti.vz_off);
  for (int tok = slot; tok < ti.n; tok += SLOTS) {
    uint32_t lo, hi;
    load_chunk<B>(stage + ti.v_off + tok * RB + k * B, lo, hi);
    const float s = __half2float(vs[tok * ngrp + g]);
    const float z = zero_add(__half_as_ushort(vz[tok * ngrp + g]), __half_as_ushort(vs[tok * ngrp + g]), a.intz);
    float c[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) c[j] = code8<B>(lo, hi, j);
#pragma unroll
    for (int h = 0; h < GQ; ++h) {
      if (h >= a.gq) break;
      const float p = sc[h * 128 + tok];
      const float ps = p * s;
      zsum[h] += p * z;
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[h][j] += ps * c[j];
    }
  }
}

template <int D, int GQ, class A>
__device__ void pv_ring(const A& a, const TileInfo& ti, const uint8_t* stage,
                        const float* sc, float (&acc)[GQ][8]) {
  constexpr int CHUNKS = D / 8, SLOTS = NT / CHUNKS;
  const int k = threadIdx.x % CHUNKS, slot = threadIdx.x / CHUNKS;
  const __half* rows = reinterpret_cast<const __half*>(stage + ti.v_off);
  for (int tok = slot; tok < ti.n; tok += SLOTS) {
    const uint4 raw = *reinterpret_cast<const uint4*>(rows + tok * D + 8 * k);
    const __half2* h2 = reinterpret_cast<const __half2*>(&raw);
    float v[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = __half22float2(h2[j]);
      v[2 * j] = f.x;
      v[2 * j + 1] = f.y;
    }
#pragma unroll
    for (int h = 0; h < GQ; ++h) {
      if (h >= a.gq) break;
      const float p = sc[h * 128 + tok];
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[h][j] += p * v[j];
    }
  }
}

// What one CTA does: (batch or sequence, kv head), its split and tile range.
struct CtaWork {
  int b, hk, pair, split, nsplit, t_begin, t_end;
};

__device__ inline CtaWork cta_work(const DecodeArgs& a) {
  CtaWork w;
  w.pair = blockIdx.x / a.n_splits;
  w.split = blockIdx.x % a.n_splits;
  w.nsplit = a.n_splits;
  w.t_begin = a.split_tile[w.split];
  w.t_end = a.split_tile[w.split + 1];
  w.b = w.pair / a.h_kv;
  w.hk = w.pair % a.h_kv;
  return w;
}
__device__ inline TileInfo cta_tile(const DecodeArgs& a, const CtaWork&, int t) { return tile_info(a, t); }
__device__ inline void cta_issue(const DecodeArgs& a, const CtaWork& w, int t, uint8_t* stage, uint64_t* bar) {
  issue_tile(a, w.pair, t, stage, bar);
}

// Paged cache: grid column x belongs to the last sequence whose first
// column is <= x; blockIdx.y is the kv head.  The sequence's tiles are dealt
// to its CTAs in equal contiguous ranges.
__device__ inline CtaWork cta_work(const PagedArgs& a) {
  int lo = 0, hi = a.n_seq - 1;
  const int x = blockIdx.x;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (a.seq[mid].split0 <= x) lo = mid;
    else hi = mid - 1;
  }
  const PagedSeq& s = a.seq[lo];
  CtaWork w;
  w.b = lo;
  w.hk = blockIdx.y;
  w.pair = lo * a.h_kv + w.hk;
  w.split = x - s.split0;
  w.nsplit = s.n_split;
  w.t_begin = (int)((long long)s.n_tiles * w.split / s.n_split);
  w.t_end = (int)((long long)s.n_tiles * (w.split + 1) / s.n_split);
  return w;
}
__device__ inline TileInfo cta_tile(const PagedArgs& a, const CtaWork& w, int t) {
  return paged_tile(a, a.seq[w.b], t);
}
// A block-table entry outside the pool is not followed: page 0 is read
// instead (the copy stays inside the pool and its byte count unchanged) and
// the cache's error word records it.
__device__ inline void cta_issue(const PagedArgs& a, const CtaWork& w, int t, uint8_t* stage, uint64_t* bar) {
  const PagedSeq& s = a.seq[w.b];
  const TileInfo ti = paged_tile(a, s, t);
  mbar_arrive_expect_tx(bar, ti.bytes);
  auto page = [&](int row) {
    const int j = row / a.P;
    const int pg = j < a.max_pages ? a.table[(size_t)w.b * a.max_pages + j] : -1;
    if (pg < 0 || pg >= a.n_pages) {
      atomicExch(a.page_err, 2);
      return 0;
    }
    return pg;
  };
  for_each_paged_copy(a, w.b, w.hk, s, ti, page, [&](const void* src, uint32_t off, uint32_t bytes, int) {
    bulk_g2s(stage + off, src, bytes, bar);
  });
}

template <int D, int GQ, class A>
__device__ __forceinline__ void decode_cta(const A& a) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* stages = smem;
  float* qs = reinterpret_cast<float*>(smem + kStages * kStageBytes);
  float* q_s = qs + kQsBytes / 4;                // [gq][D]
  float* sc = q_s + kMaxGq * D;                  // [gq][128]
  float* bias = sc + kMaxGq * 128;               // [groups][gq]
  float* m_s = bias + (kQsBytes / (4 * D));      // [gq]
  float* l_s = m_s + kMaxGq;
  float* al_s = l_s + kMaxGq;
  int* flag_s = reinterpret_cast<int*>(al_s + kMaxGq);
  uint64_t* bars = reinterpret_cast<uint64_t*>(flag_s + 4);

  const int tid = threadIdx.x;
  const CtaWork cw = cta_work(a);
  const int pair = cw.pair, split = cw.split, nsplit = cw.nsplit;
  const int t_begin = cw.t_begin;
  const int ntiles = cw.t_end - cw.t_begin;
  const int b = cw.b, hk = cw.hk;

  for (int i = tid; i < a.gq * D; i += NT) {
    const int h = i / D, c = i % D;
    q_s[i] = __half2float(a.q[((size_t)b * a.h_kv * a.gq + (size_t)hk * a.gq + h) * D + c]);
  }
  if (tid < kMaxGq) {
    m_s[tid] = -INFINITY;
    l_s[tid] = 0.f;
    al_s[tid] = 1.f;
  }
  if (tid == 0) {
    flag_s[0] = 0;
    for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (tid == 0) {
    for (int i = 0; i < kStages && i < ntiles; ++i)
      cta_issue(a, cw, t_begin + i, stages + i * kStageBytes, &bars[i]);
  }

  float acc[GQ][8];
  float zsum[GQ];
#pragma unroll
  for (int h = 0; h < GQ; ++h) {
    zsum[h] = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[h][j] = 0.f;
  }

  for (int it = 0; it < ntiles; ++it) {
    const int t = t_begin + it;
    const int st = it % kStages;
    uint8_t* stage = stages + st * kStageBytes;
    if (!mbar_wait_bounded(&bars[st], (uint32_t)((it / kStages) & 1))) flag_s[0] = 1;
    __syncthreads();
    if (flag_s[0]) {
      if (tid == 0) {
        atomicExch(a.err, 1);
        // drain (bounded) the copies still in flight before leaving
        for (int j = it + 1; j < ntiles && j < it + kStages; ++j)
          (void)mbar_wait_bounded(&bars[j % kStages], (uint32_t)((j / kStages) & 1));
      }
      return;
    }
    const TileInfo ti = cta_tile(a, cw, t);

    // scaled query and bias per K group of the tile
    if (ti.kseg >= 0) {
      const __half* ks = reinterpret_cast<const __half*>(stage + ti.ks_off);
      const __half* kz = reinterpret_cast<const __half*>(stage + ti.kz_off);
      for (int i = tid; i < ti.ng * a.gq * D; i += NT) {
        const int c = i % D, h = (i / D) % a.gq, gl = i / (D * a.gq);
        qs[i] = q_s[h * D + c] * __half2float(ks[gl * D + c]);
      }
      const int warp = tid >> 5, lane = tid & 31;
      for (int task = warp; task < ti.ng * a.gq; task += NT / 32) {
        const int gl = task / a.gq, h = task % a.gq;
        float s = 0.f;
        for (int c = lane; c < D; c += 32)
          s += q_s[h * D + c] * zero_add(__half_as_ushort(kz[gl * D + c]), __half_as_ushort(ks[gl * D + c]), a.intz);
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        if (lane == 0) bias[task] = s;
      }
      __syncthreads();
      if (ti.kbits == 2) scores_packed<D, GQ, 2>(a, ti, stage, qs, bias, sc);
      else if (ti.kbits == 4) scores_packed<D, GQ, 4>(a, ti, stage, qs, bias, sc);
      else scores_packed<D, GQ, 8>(a, ti, stage, qs, bias, sc);
    } else {
      scores_ring<D, GQ>(a, ti, stage, q_s, sc);
    }
    __syncthreads();

    // online softmax (base 2), one warp per query head
    {
      const int warp = tid >> 5, lane = tid & 31;
      if (warp < a.gq) {
        float* s = sc + warp * 128;
        float mx = -INFINITY;
        for (int i = lane; i < ti.n; i += 32) mx = fmaxf(mx, s[i]);
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        const float m_old = m_s[warp];
        const float m_new = fmaxf(m_old, mx);
        float sum = 0.f;
        for (int i = lane; i < ti.n; i += 32) {
          const float p = exp2f(s[i] - m_new);
          s[i] = p;
          sum += p;
        }
        for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
        __syncwarp();
        if (lane == 0) {
          const float alpha = exp2f(m_old - m_new);
          m_s[warp] = m_new;
          l_s[warp] = l_s[warp] * alpha + sum;
          al_s[warp] = alpha;
        }
      }
    }
    __syncthreads();
#pragma unroll
    for (int h = 0; h < GQ; ++h) {
      if (h < a.gq) {
        const float alpha = al_s[h];
        if (alpha != 1.f) {
          zsum[h] *= alpha;
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[h][j] *= alpha;
        }
      }
    }
    if (ti.vseg >= 0) {
      if (ti.vbits == 2) pv_packed<D, GQ, 2>(a, ti, stage, sc, acc, zsum);
      else if (ti.vbits == 4) pv_packed<D, GQ, 4>(a, ti, stage, sc, acc, zsum);
      else pv_packed<D, GQ, 8>(a, ti, stage, sc, acc, zsum);
    } else {
      pv_ring<D, GQ>(a, ti, stage, sc, acc);
    }
    __syncthreads();
    if (tid == 0 && it + kStages < ntiles) {
      fence_proxy_async_smem();
      cta_issue(a, cw, t + kStages, stage, &bars[st]);
    }
  }

  // ---- reduce the PV partial sums over token slots -> o[h][c] in smem ----
  constexpr int CHUNKS = D / 8;
  const int k = tid % CHUNKS;
  float* red = reinterpret_cast<float*>(stages);  // [NT/32][D], pipeline drained
  float* o_s = reinterpret_cast<float*>(stages) + (NT / 32) * D;  // [gq][D]
  const int warp = tid >> 5, lane = tid & 31;
#pragma unroll
  for (int h = 0; h < GQ; ++h) {
    if (h >= a.gq) break;
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      v[j] = acc[h][j] + zsum[h];
      for (int off = CHUNKS; off < 32; off <<= 1) v[j] += __shfl_xor_sync(0xffffffffu, v[j], off);
    }
    if (lane < CHUNKS) {
#pragma unroll
      for (int j = 0; j < 8; ++j) red[warp * D + 8 * k + j] = v[j];
    }
    __syncthreads();
    for (int c = tid; c < D; c += NT) {
      float s = 0.f;
      for (int w = 0; w < NT / 32; ++w) s += red[w * D + c];
      o_s[h * D + c] = s;
    }
    __syncthreads();
  }

  const size_t out_base = ((size_t)b * a.h_kv * a.gq + (size_t)hk * a.gq) * D;
  if (nsplit == 1) {
    // (l = 0 only for a sequence with no tokens: its output is zero)
    for (int i = tid; i < a.gq * D; i += NT) {
      const int h = i / D;
      a.out[out_base + i] = __float2half_rn(l_s[h] > 0.f ? o_s[i] / l_s[h] : 0.f);
    }
    return;
  }
  float* rec = a.part + ((size_t)pair * a.n_splits + split) * a.gq * (D + 2);
  for (int i = tid; i < a.gq * D; i += NT) {
    const int h = i / D, c = i % D;
    rec[h * (D + 2) + c] = o_s[i];
  }
  if (tid < a.gq) {
    rec[tid * (D + 2) + D] = m_s[tid];
    rec[tid * (D + 2) + D + 1] = l_s[tid];
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int ticket = atomicAdd(&a.counters[pair], 1);
    flag_s[1] = (ticket == nsplit - 1);
  }
  __syncthreads();
  if (!flag_s[1]) return;
  __threadfence();
  // Merge of the splits' records.  First the weight of each (split, head),
  // 2^(m_s - M) / L with M the max and L the weighted sum of l over the
  // splits, one warp per head; then every output element is a sum of
  // independent loads (the records are cold in L2, so a chain of dependent
  // loads per element would cost a round trip per split).
  const float* recs = a.part + (size_t)pair * a.n_splits * a.gq * (D + 2);  // n_splits records a pair
  float* wts = o_s + kMaxGq * D;  // [n_splits][gq]
  static_assert((NT / 32 + 2 * kMaxGq) * 128 + KVQ_MAX_SPLITS * kMaxGq <= kStages * kStageBytes / 4,
                "merge scratch inside the drained stages");
  for (int h = warp; h < a.gq; h += NT / 32) {
    float M = -INFINITY;
    for (int sp = lane; sp < nsplit; sp += 32)
      M = fmaxf(M, __ldcg(recs + ((size_t)sp * a.gq + h) * (D + 2) + D));
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float L = 0.f;
    for (int sp = lane; sp < nsplit; sp += 32) {
      const float* r = recs + ((size_t)sp * a.gq + h) * (D + 2);
      const float w = exp2f(__ldcg(r + D) - M);
      wts[sp * a.gq + h] = w;
      L += __ldcg(r + D + 1) * w;
    }
    for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
    __syncwarp();
    const float inv = 1.f / L;
    for (int sp = lane; sp < nsplit; sp += 32) wts[sp * a.gq + h] *= inv;
  }
  __syncthreads();
  for (int i = tid; i < a.gq * D; i += NT) {
    const int h = i / D, c = i % D;
    float O = 0.f;
#pragma unroll 8
    for (int sp = 0; sp < nsplit; ++sp)
      O += __ldcg(recs + ((size_t)sp * a.gq + h) * (D + 2) + c) * wts[sp * a.gq + h];
    a.out[out_base + i] = __float2half_rn(O);
  }
  if (tid == 0) a.counters[pair] = 0;
}

template <int D, int GQ>
__global__ void __launch_bounds__(NT, 2) decode_kernel(const DecodeArgs a) {
  decode_cta<D, GQ>(a);
}

template <int D, int GQ>
__global__ void __launch_bounds__(NT, 2) decode_paged_kernel(const PagedArgs a) {
  decode_cta<D, GQ>(a);
}

template <int D>
cudaError_t launch_d(const DecodeArgs& a, int n_pairs, cudaStream_t s) {
  const size_t smem = decode_smem_bytes(a.gq, D);
  const dim3 grid(n_pairs * a.n_splits);
  cudaError_t e;
#define KVQ_LAUNCH(GQV)                                                                   \
  e = set_smem_once((const void*)decode_kernel<D, GQV>, (int)smem);                        \
  if (e != cudaSuccess) return e;                                                         \
  decode_kernel<D, GQV><<<grid, NT, smem, s>>>(a);
  if (a.gq == 1) { KVQ_LAUNCH(1) }
  else if (a.gq == 2) { KVQ_LAUNCH(2) }
  else if (a.gq <= 4) { KVQ_LAUNCH(4) }
  else { KVQ_LAUNCH(8) }
#undef KVQ_LAUNCH
  return cudaGetLastError();
}

}  // namespace

size_t decode_smem_bytes(int /*gq*/, int d) {
  size_t b = (size_t)kStages * kStageBytes + kQsBytes;
  b += (size_t)kMaxGq * d * 4 + (size_t)kMaxGq * 128 * 4 + (size_t)kQsBytes / (4 * d) * 4;
  b += 3 * kMaxGq * 4 + 16 + kStages * 8;
  return b;
}

cudaError_t launch_decode(const DecodeArgs& a, int n_pairs, cudaStream_t s) {
  return a.d == 128 ? launch_d<128>(a, n_pairs, s) : launch_d<64>(a, n_pairs, s);
}

namespace {
template <int D>
cudaError_t launch_paged_d(const PagedArgs& a, cudaStream_t s) {
  const size_t smem = decode_smem_bytes(a.gq, D);
  const dim3 grid(a.n_cols, a.h_kv);
  cudaError_t e;
#define KVQ_LAUNCH(GQV)                                                                          \
  e = set_smem_once((const void*)decode_paged_kernel<D, GQV>, (int)smem);                         \
  if (e != cudaSuccess) return e;                                                                \
  decode_paged_kernel<D, GQV><<<grid, NT, smem, s>>>(a);
  if (a.gq == 1) { KVQ_LAUNCH(1) }
  else if (a.gq == 2) { KVQ_LAUNCH(2) }
  else if (a.gq <= 4) { KVQ_LAUNCH(4) }
  else { KVQ_LAUNCH(8) }
#undef KVQ_LAUNCH
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_decode_paged(const PagedArgs& a, cudaStream_t s) {
  return a.d == 128 ? launch_paged_d<128>(a, s) : launch_paged_d<64>(a, s);
}

}  // namespace kvq
