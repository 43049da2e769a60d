// Quantize-pack kernels: KIVI appends (V eviction per token, K block flush per
// channel), the explicit K flush, and the WindowQuant reordered ingest.
//
// KIVI page, "方法细节": K is quantized per channel over groups of G tokens
// (the residual block is quantized once it holds R tokens), V per token over
// groups of G channels (the oldest token of the fp16 queue is quantized when
// the queue exceeds R).  WindowQuant page §3.3.1: windows of equal width are
// written contiguously, in the order of the ingest permutation.
#include <climits>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kQuantThreads = 128;

struct PairPtrs {
  const __half* in_k;  // new tokens of this (batch, kv head)
  const __half* in_v;
  __half* ring_k;
  __half* ring_v;
};

template <int D>
__device__ __forceinline__ const __half* src_row(const __half* ring, const __half* in, int R,
                                                 const RowSrc& s, int p) {
  return p < s.n_old ? ring + (size_t)((s.start + p) % R) * D : in + (size_t)(p - s.n_old) * D;
}

// Quantize one K group (G pushed tokens starting at push index p0, all D
// channels, one group per channel) into packed rows [row0, row0 + G) and
// scale/zero row `grow` of the destination segment.  Whole block.  The G
// source rows are first staged in shared memory with 16-byte loads (all in
// flight at once), then each thread reduces and quantizes one channel.
template <int D>
__device__ void quant_k_group(const SegDev& dst, int bits, int G, int R, size_t pair,
                              const __half* ring, const __half* in, const RowSrc& src, int p0,
                              int row0, int grow, __half* xs, uint8_t* codes_s) {
  const int tid = threadIdx.x;
  constexpr int kVec = D * 2 / 16;  // 16-byte vectors per row
  for (int idx = tid; idx < G * kVec; idx += blockDim.x) {
    const int i = idx / kVec, v = idx % kVec;
    reinterpret_cast<int4*>(xs + (size_t)i * D)[v] =
        reinterpret_cast<const int4*>(src_row<D>(ring, in, R, src, p0 + i))[v];
  }
  __syncthreads();
  for (int c = tid; c < D; c += blockDim.x) {
    float mn = __half2float(xs[c]);
    float mx = mn;
    for (int i = 1; i < G; ++i) {
      const float v = __half2float(xs[(size_t)i * D + c]);
      mn = fminf(mn, v);
      mx = fmaxf(mx, v);
    }
    const QParams qp = qparams(mn, mx, bits);
    const float rcp = qp.s != 0.0f ? __frcp_rn(qp.s) : 0.0f;
    const size_t gidx = (pair * (size_t)(dst.cap / G) + grow) * D + c;
    const_cast<__half*>(dst.ks)[gidx] = qp.sh;
    const_cast<__half*>(dst.kz)[gidx] = qp.zh;
    for (int i = 0; i < G; ++i)
      codes_s[(size_t)i * D + c] = (uint8_t)qcode_fast(__half2float(xs[(size_t)i * D + c]), qp, rcp, bits);
  }
  __syncthreads();
  const int per_word = 32 / bits;
  const int words = D * bits / 32;
  const int rb = D * bits / 8;
  uint8_t* base = const_cast<uint8_t*>(dst.kc) + (pair * (size_t)dst.cap + row0) * rb;
  for (int idx = tid; idx < G * words; idx += blockDim.x) {
    const int i = idx / words, w = idx % words;
    uint32_t word = 0;
    for (int j = 0; j < per_word; ++j) word |= (uint32_t)codes_s[(size_t)i * D + w * per_word + j] << (j * bits);
    reinterpret_cast<uint32_t*>(base + (size_t)i * rb)[w] = word;
  }
  __syncthreads();
}

// Quantize one V token (all D channels, one group per G channels) into packed
// row `row` of the destination segment.  One warp; lane l owns channels
// 4l..4l+3 (lanes >= D/4 idle).
template <int D>
__device__ void quant_v_token(const SegDev& dst, int bits, int G, size_t pair, const __half* x,
                              int row) {
  const int lane = threadIdx.x & 31;
  const bool active = lane < D / 4;
  float v[4] = {0.f, 0.f, 0.f, 0.f};
  if (active) {
    const __half2* x2 = reinterpret_cast<const __half2*>(x) + 2 * lane;
    const float2 a = __half22float2(x2[0]);
    const float2 b = __half22float2(x2[1]);
    v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
  }
  float mn = fminf(fminf(v[0], v[1]), fminf(v[2], v[3]));
  float mx = fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3]));
  const int lpg = G / 4;  // lanes per channel group (aligned segments of the warp)
  for (int off = 1; off < lpg; off <<= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  }
  if (!active) return;
  const QParams qp = qparams(mn, mx, bits);
  const float rcp = qp.s != 0.0f ? __frcp_rn(qp.s) : 0.0f;
  uint32_t packed = 0;
  for (int j = 0; j < 4; ++j) packed |= qcode_fast(v[j], qp, rcp, bits) << (j * bits);
  const int rb = D * bits / 8;
  uint8_t* rowp = const_cast<uint8_t*>(dst.vc) + (pair * (size_t)dst.cap + row) * rb;
  if (bits == 2) rowp[lane] = (uint8_t)packed;
  else if (bits == 4) reinterpret_cast<uint16_t*>(rowp)[lane] = (uint16_t)packed;
  else reinterpret_cast<uint32_t*>(rowp)[lane] = packed;
  if ((4 * lane) % G == 0) {
    const size_t sidx = (pair * (size_t)dst.cap + row) * (D / G) + (4 * lane) / G;
    const_cast<__half*>(dst.vs)[sidx] = qp.sh;
    const_cast<__half*>(dst.vz)[sidx] = qp.zh;
  }
}

// Copy `n` token rows: source row i -> ring slot (slot0 + i) % R.  Whole block.
template <int D>
__device__ void copy_to_ring(__half* ring, int R, int slot0, const __half* src, int n) {
  constexpr int kVec = D * 2 / 16;  // 16-byte vectors per row
  for (int idx = threadIdx.x; idx < n * kVec; idx += blockDim.x) {
    const int i = idx / kVec, v = idx % kVec;
    const int4* s = reinterpret_cast<const int4*>(src + (size_t)i * D) + v;
    int4* d = reinterpret_cast<int4*>(ring + (size_t)((slot0 + i) % R) * D) + v;
    *d = *s;
  }
}

template <int D>
__global__ void __launch_bounds__(kQuantThreads) append_kernel(const AppendArgs a) {
  extern __shared__ __align__(16) uint8_t qsm[];
  __half* xs = reinterpret_cast<__half*>(qsm);
  uint8_t* codes_s = qsm + (size_t)a.G * D * 2;
  const size_t pair = blockIdx.x;
  const int chunk = blockIdx.y;
  const __half* in_k = a.k_new + pair * (size_t)a.T * D;
  const __half* in_v = a.v_new + pair * (size_t)a.T * D;
  __half* ring_k = a.kr + pair * (size_t)a.R * D;
  __half* ring_v = a.vr + pair * (size_t)a.R * D;
  const int warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;

  if (chunk == 0) {
    // work that reads old ring slots, before any new token lands in the ring
    for (int gi = 0; gi < a.k_ring_groups; ++gi)
      quant_k_group<D>(a.dst, a.bits, a.G, a.R, pair, ring_k, in_k, a.ksrc, gi * a.G,
                       a.k_nk0 + gi * a.G, a.k_nk0 / a.G + gi, xs, codes_s);
    for (int p = warp; p < a.v_ring_tokens; p += nwarps)
      quant_v_token<D>(a.dst, a.bits, a.G, pair, src_row<D>(ring_v, in_v, a.R, a.vsrc, p),
                       a.v_nv0 + p);
    __syncthreads();
    if (a.k_first_ring < a.T)
      copy_to_ring<D>(ring_k, a.R, a.k_slot0 + a.k_first_ring, in_k + (size_t)a.k_first_ring * D,
                      a.T - a.k_first_ring);
    if (a.v_first_ring < a.T)
      copy_to_ring<D>(ring_v, a.R, a.v_slot0 + a.v_first_ring, in_v + (size_t)a.v_first_ring * D,
                      a.T - a.v_first_ring);
  }
  // work that reads only the new tokens, spread over the chunks (chunk 0
  // takes part only when it is the only one)
  const int workers = a.chunks > 1 ? a.chunks - 1 : 1;
  const int me = a.chunks > 1 ? chunk - 1 : 0;
  if (a.chunks > 1 && chunk == 0) return;
  for (int gi = a.k_ring_groups + me; gi < a.k_groups; gi += workers)
    quant_k_group<D>(a.dst, a.bits, a.G, a.R, pair, ring_k, in_k, a.ksrc, gi * a.G,
                     a.k_nk0 + gi * a.G, a.k_nk0 / a.G + gi, xs, codes_s);
  for (int p = a.v_ring_tokens + me * nwarps + warp; p < a.v_evict; p += workers * nwarps)
    quant_v_token<D>(a.dst, a.bits, a.G, pair, src_row<D>(ring_v, in_v, a.R, a.vsrc, p),
                     a.v_nv0 + p);
}

// K flush: group blockIdx.y of the ring's oldest tokens.
template <int D>
__global__ void __launch_bounds__(kQuantThreads) flush_kernel(const AppendArgs a) {
  extern __shared__ __align__(16) uint8_t qsm[];
  __half* xs = reinterpret_cast<__half*>(qsm);
  uint8_t* codes_s = qsm + (size_t)a.G * D * 2;
  const size_t pair = blockIdx.x;
  const int gi = blockIdx.y;
  const __half* ring_k = a.kr + pair * (size_t)a.R * D;
  quant_k_group<D>(a.dst, a.bits, a.G, a.R, pair, ring_k, nullptr, a.ksrc, gi * a.G,
                   a.k_nk0 + gi * a.G, a.k_nk0 / a.G + gi, xs, codes_s);
}

// WindowQuant ingest: block (pair, job); job n_jobs is the fp16 tail.
template <int D>
__global__ void __launch_bounds__(kQuantThreads) ingest_kernel(const IngestArgs a) {
  extern __shared__ __align__(16) uint8_t qsm[];
  __half* xs = reinterpret_cast<__half*>(qsm);
  uint8_t* codes_s = qsm + (size_t)a.G * D * 2;
  const size_t pair = blockIdx.x;
  const int j = blockIdx.y;
  const __half* in_k = a.k_new + pair * (size_t)a.T * D;
  const __half* in_v = a.v_new + pair * (size_t)a.T * D;
  __half* ring_k = a.kr + pair * (size_t)a.R * D;
  __half* ring_v = a.vr + pair * (size_t)a.R * D;
  if (j == a.n_jobs) {
    if (a.tail_len > 0) {
      copy_to_ring<D>(ring_k, a.R, a.krs_push + a.tail_dst, in_k + (size_t)a.tail_src * D, a.tail_len);
      copy_to_ring<D>(ring_v, a.R, a.vrs_push + a.tail_dst, in_v + (size_t)a.tail_src * D, a.tail_len);
    }
    return;
  }
  const WindowJob job = a.jobs[j];
  if (job.seg < 0) {
    copy_to_ring<D>(ring_k, a.R, a.krs_push + job.dst, in_k + (size_t)job.src_token * D, a.S);
    copy_to_ring<D>(ring_v, a.R, a.vrs_push + job.dst, in_v + (size_t)job.src_token * D, a.S);
    return;
  }
  const SegDev& dst = a.seg[job.seg];
  const RowSrc src{0, 0};
  const __half* wk = in_k + (size_t)job.src_token * D;
  for (int gi = 0; gi < a.S / a.G; ++gi)
    quant_k_group<D>(dst, dst.bits, a.G, a.R, pair, nullptr, wk, src, gi * a.G, job.dst + gi * a.G,
                     job.dst / a.G + gi, xs, codes_s);
  const int warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  for (int p = warp; p < a.S; p += nwarps)
    quant_v_token<D>(dst, dst.bits, a.G, pair, in_v + (size_t)(job.src_token + p) * D, job.dst + p);
}

}  // namespace

size_t quant_smem(int G, int d) { return (size_t)G * d * 3; }

template <class K>
cudaError_t set_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

cudaError_t launch_append(const AppendArgs& a, cudaStream_t s) {
  dim3 grid(a.batch * a.h_kv, a.chunks);
  const size_t sm = quant_smem(a.G, a.d);
  cudaError_t e;
  if (a.d == 128) {
    if ((e = set_smem(append_kernel<128>, sm)) != cudaSuccess) return e;
    append_kernel<128><<<grid, kQuantThreads, sm, s>>>(a);
  } else {
    if ((e = set_smem(append_kernel<64>, sm)) != cudaSuccess) return e;
    append_kernel<64><<<grid, kQuantThreads, sm, s>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t launch_flush(const AppendArgs& a, cudaStream_t s) {
  if (a.k_groups <= 0) return cudaSuccess;
  dim3 grid(a.batch * a.h_kv, a.k_groups);
  const size_t sm = quant_smem(a.G, a.d);
  cudaError_t e;
  if (a.d == 128) {
    if ((e = set_smem(flush_kernel<128>, sm)) != cudaSuccess) return e;
    flush_kernel<128><<<grid, kQuantThreads, sm, s>>>(a);
  } else {
    if ((e = set_smem(flush_kernel<64>, sm)) != cudaSuccess) return e;
    flush_kernel<64><<<grid, kQuantThreads, sm, s>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t launch_ingest(const IngestArgs& a, cudaStream_t s) {
  dim3 grid(a.batch * a.h_kv, a.n_jobs + 1);
  const size_t sm = quant_smem(a.G, a.d);
  cudaError_t e;
  if (a.d == 128) {
    if ((e = set_smem(ingest_kernel<128>, sm)) != cudaSuccess) return e;
    ingest_kernel<128><<<grid, kQuantThreads, sm, s>>>(a);
  } else {
    if ((e = set_smem(ingest_kernel<64>, sm)) != cudaSuccess) return e;
    ingest_kernel<64><<<grid, kQuantThreads, sm, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace kvq
