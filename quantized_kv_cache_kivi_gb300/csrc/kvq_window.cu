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

}  // namespace

cudaError_t launch_window_assign(const WindowArgs& a, cudaStream_t s) {
  text_sum_kernel<<<a.batch, kThreads, 0, s>>>(a);
  window_stat_kernel<<<dim3(a.batch, a.M / a.S), kThreads, 0, s>>>(a);
  window_rank_kernel<<<1, kThreads, (size_t)a.batch * sizeof(double), s>>>(a);
  return cudaGetLastError();
}

}  // namespace kvq
