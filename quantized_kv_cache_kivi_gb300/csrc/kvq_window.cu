// WindowQuant window bit-width assignment (WindowQuant page §3.2.1, Eq.7-8:
// windows of S vision tokens scored by cosine similarity to the text;
// §3.3.1: windows of equal width listed contiguously for the reordered
// ingest).  Rank rule: top floor(frac8*n) windows 8 bits, next
// floor(frac4*n) 4 bits, the rest 2 bits; optional window 0 at 16 bits
// (§3.2.2).  Sums of fp16 keys are accumulated in fp64, where they are exact.
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kThreads = 256;

__device__ double block_sum(double v, double* red) {
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  double s = 0.0;
  if (threadIdx.x == 0)
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) s += red[w];
  return s;  // valid in thread 0
}

// tsum[b][h*d + c] = sum over text tokens of text[b][h][t][c]
__global__ void text_sum_kernel(WindowArgs a) {
  const int b = blockIdx.x;
  const int hd = a.h_kv * a.d;
  for (int i = threadIdx.x; i < hd; i += blockDim.x) {
    const int h = i / a.d, c = i % a.d;
    const __half* p = a.text + (((size_t)b * a.h_kv + h) * a.N) * a.d + c;
    double s = 0.0;
    for (int t = 0; t < a.N; ++t) s += (double)__half2float(p[(size_t)t * a.d]);
    a.tsum[(size_t)b * hd + i] = s;
  }
}

// wstat[b][w] = (Wsum . Tsum, |Wsum|^2) for window w of batch b
__global__ void window_stat_kernel(WindowArgs a) {
  __shared__ double red[kThreads / 32];
  const int b = blockIdx.x, w = blockIdx.y;
  const int hd = a.h_kv * a.d;
  double dot = 0.0, nn = 0.0;
  for (int i = threadIdx.x; i < hd; i += blockDim.x) {
    const int h = i / a.d, c = i % a.d;
    const __half* p = a.keys + (((size_t)b * a.h_kv + h) * a.M + (size_t)w * a.S) * a.d + c;
    double s = 0.0;
    for (int t = 0; t < a.S; ++t) s += (double)__half2float(p[(size_t)t * a.d]);
    dot += s * a.tsum[(size_t)b * hd + i];
    nn += s * s;
  }
  const double d_all = block_sum(dot, red);
  const double n_all = block_sum(nn, red);
  if (threadIdx.x == 0) {
    const int nw = a.M / a.S;
    a.wstat[((size_t)b * nw + w) * 2 + 0] = d_all;
    a.wstat[((size_t)b * nw + w) * 2 + 1] = n_all;
  }
}

// One block: cosine per window (mean over the batch), rank, widths, order.
__global__ void window_rank_kernel(WindowArgs a) {
  __shared__ double red[kThreads / 32];
  extern __shared__ double tt[];  // [batch]
  const int nw = a.M / a.S;
  const int hd = a.h_kv * a.d;
  for (int b = 0; b < a.batch; ++b) {
    double v = 0.0;
    for (int i = threadIdx.x; i < hd; i += blockDim.x) {
      const double t = a.tsum[(size_t)b * hd + i];
      v += t * t;
    }
    const double s = block_sum(v, red);
    if (threadIdx.x == 0) tt[b] = s;
  }
  __syncthreads();
  for (int w = threadIdx.x; w < nw; w += blockDim.x) {
    double sum = 0.0;
    for (int b = 0; b < a.batch; ++b) {
      const double dot = a.wstat[((size_t)b * nw + w) * 2 + 0];
      const double nn = a.wstat[((size_t)b * nw + w) * 2 + 1];
      sum += (nn > 0.0 && tt[b] > 0.0) ? dot / (sqrt(nn) * sqrt(tt[b])) : 0.0;
    }
    a.sim[w] = sum / (double)a.batch;
  }
  __syncthreads();
  for (int w = threadIdx.x; w < nw; w += blockDim.x) {
    int bits;
    if (a.first_fp16 && w == 0) {
      bits = 16;
    } else {
      const double sw = a.sim[w];
      int rank = 0;
      for (int v = (a.first_fp16 ? 1 : 0); v < nw; ++v) {
        const double sv = a.sim[v];
        rank += (sv > sw) || (sv == sw && v < w);
      }
      bits = rank < a.n8 ? 8 : (rank < a.n8 + a.n4 ? 4 : 2);
    }
    a.bits[w] = (int8_t)bits;
  }
  __syncthreads();
  for (int w = threadIdx.x; w < nw; w += blockDim.x) {
    const int bw = a.bits[w];
    int pos = 0;
    for (int v = 0; v < nw; ++v) {
      const int bv = a.bits[v];
      pos += (bv > bw) || (bv == bw && v < w);
    }
    a.perm[pos] = w;
  }
}

// ---- paper-exact assignment (WindowQuant §3.2.1 Eq.8, §3.2.3 Eq.10-11) -----
// Eq.8 averages the cosines of every (text token, window token) pair:
// sim = (1 / S N) (sum_j t_j / |t_j|) . (sum_k w_k / |w_k|), so each window and
// the text reduce to one sum of unit vectors (fp64), split over `chunks`
// token chunks (partial sums in a fixed order, no atomics).

// Block (b, unit u, chunk z): unit u < n_win is window u, u = n_win the text.
// Phase 1: one warp per token, its inverse norm; phase 2: one thread per
// 8-channel slice, the sum of x / |x| over the chunk's tokens.  Products of
// fp16 values are exact in fp32; sums run in fp32 over at most 16 terms and
// then in fp64 (GB300's fp64 rate is a small fraction of its fp32 rate).
__global__ void eq8_unit_sum_kernel(Eq8Args a) {
  extern __shared__ float inv[];  // [tokens of the chunk]
  const int b = blockIdx.x, u = blockIdx.y, z = blockIdx.z;
  const int nw = a.M / a.S;
  const bool text = u == nw;
  const int len = text ? a.N : a.S;
  const int per = (len + a.chunks - 1) / a.chunks;
  const int k0 = z * per, k1 = min(len, k0 + per);
  const __half* base = text ? a.text + (size_t)b * a.N * a.dim
                            : a.vision + ((size_t)b * a.M + (size_t)u * a.S) * a.dim;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarp = blockDim.x >> 5;
  const int n8 = a.dim / 8;  // 8-channel slices (dim % 8 == 0, checked by the host)
  for (int k = k0 + warp; k < k1; k += nwarp) {
    const uint4* x = reinterpret_cast<const uint4*>(base + (size_t)k * a.dim);
    double ss = 0.0;
    for (int c0 = 0; c0 < n8; c0 += 32 * 2) {
      float f = 0.f;  // at most 16 exact squares
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int c = c0 + 32 * r + lane;
        if (c < n8) {
          const uint4 v = __ldg(x + c);
          const __half2* h = reinterpret_cast<const __half2*>(&v);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 t = __half22float2(h[e]);
            f = fmaf(t.x, t.x, f);
            f = fmaf(t.y, t.y, f);
          }
        }
      }
      ss += (double)f;
    }
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if (lane == 0) inv[k - k0] = ss > 0.0 ? (float)(1.0 / sqrt(ss)) : 0.f;  // a zero token adds nothing
  }
  __syncthreads();
  double* out = a.part + (((size_t)b * (nw + 1) + u) * a.chunks + z) * a.dim;
  for (int c = threadIdx.x; c < n8; c += blockDim.x) {
    double acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.0;
    for (int k = k0; k < k1; k += 16) {
      float f[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] = 0.f;
      const int kk1 = min(k1, k + 16);
      for (int q = k; q < kk1; ++q) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(base + (size_t)q * a.dim) + c);
        const __half2* h = reinterpret_cast<const __half2*>(&v);
        const float w = inv[q - k0];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 t = __half22float2(h[e]);
          f[2 * e] = fmaf(t.x, w, f[2 * e]);
          f[2 * e + 1] = fmaf(t.y, w, f[2 * e + 1]);
        }
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] += (double)f[e];
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) out[8 * c + e] = acc[e];
  }
}

// sims[b][w] = (window sum . text sum) / (S N), chunk partials added in order.
__global__ void eq8_sim_kernel(Eq8Args a) {
  __shared__ double red[kThreads / 32];
  const int b = blockIdx.x, w = blockIdx.y;
  const int nw = a.M / a.S;
  const double* pw = a.part + ((size_t)b * (nw + 1) + w) * a.chunks * a.dim;
  const double* pt = a.part + ((size_t)b * (nw + 1) + nw) * a.chunks * a.dim;
  double dot = 0.0;
  for (int c = threadIdx.x; c < a.dim; c += blockDim.x) {
    double sw = 0.0, st = 0.0;
    for (int z = 0; z < a.chunks; ++z) {
      sw += pw[(size_t)z * a.dim + c];
      st += pt[(size_t)z * a.dim + c];
    }
    dot += sw * st;
  }
  const double d = block_sum(dot, red);
  if (threadIdx.x == 0) a.sims[(size_t)b * nw + w] = d / ((double)a.S * (double)a.N);
}

// One block: per window the configuration of every request (above T_high
// FP16, below T_low INT2, else INT4), the batch's most frequent one (ties to
// the wider), window 0 pinned to FP16 on request; then the ingest order.
__global__ void eq8_decide_kernel(Eq8Args a) {
  const int nw = a.M / a.S;
  for (int w = threadIdx.x; w < nw; w += blockDim.x) {
    int c16 = 0, c4 = 0, c2 = 0;
    for (int b = 0; b < a.batch; ++b) {
      const double v = a.sims[(size_t)b * nw + w];
      if (v > a.t_high) ++c16;
      else if (v < a.t_low) ++c2;
      else ++c4;
    }
    int bits = (c16 >= c4 && c16 >= c2) ? 16 : (c4 >= c2 ? 4 : 2);
    if (a.first_fp16 && w == 0) bits = 16;
    a.bits[w] = (int8_t)bits;
  }
  __syncthreads();
  for (int w = threadIdx.x; w < nw; w += blockDim.x) {
    const int bw = a.bits[w];
    int pos = 0;
    for (int v = 0; v < nw; ++v) {
      const int bv = a.bits[v];
      pos += (bv > bw) || (bv == bw && v < w);
    }
    a.perm[pos] = w;
  }
}

}  // namespace

cudaError_t launch_window_assign_eq8(const Eq8Args& a, cudaStream_t s) {
  const int nw = a.M / a.S;
  const int maxlen = a.S > a.N ? a.S : a.N;
  const size_t sm = (size_t)((maxlen + a.chunks - 1) / a.chunks) * sizeof(float);
  eq8_unit_sum_kernel<<<dim3(a.batch, nw + 1, a.chunks), kThreads, sm, s>>>(a);
  eq8_sim_kernel<<<dim3(a.batch, nw), kThreads, 0, s>>>(a);
  eq8_decide_kernel<<<1, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_window_assign(const WindowArgs& a, cudaStream_t s) {
  text_sum_kernel<<<a.batch, kThreads, 0, s>>>(a);
  window_stat_kernel<<<dim3(a.batch, a.M / a.S), kThreads, 0, s>>>(a);
  window_rank_kernel<<<1, kThreads, (size_t)a.batch * sizeof(double), s>>>(a);
  return cudaGetLastError();
}

}  // namespace kvq
