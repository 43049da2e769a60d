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

// Shared memory of the quantize kernels: the staged K group (G rows of D
// halves), the warps' partial channel minima/maxima and the channel
// parameters (s, 1/s, z) of the group.
struct QuantSmem {
  __half* xs;    // [G][D]
  float* red;    // [2][kQuantThreads / 32][D]
  float* par;    // [3][D]
};

__host__ __device__ inline size_t quant_smem_bytes(int G, int d) {
  return (size_t)G * d * 2 + (size_t)(2 * (kQuantThreads / 32) + 3) * d * 4;
}

__device__ __forceinline__ QuantSmem quant_smem_view(uint8_t* base, int G, int D) {
  QuantSmem q;
  q.xs = reinterpret_cast<__half*>(base);
  q.red = reinterpret_cast<float*>(base + (size_t)G * D * 2);
  q.par = q.red + 2 * (kQuantThreads / 32) * D;
  return q;
}

// Quantize one K group (G pushed tokens starting at push index p0, all D
// channels, one group per channel) into packed rows [row0, row0 + G) and
// scale/zero row `grow` of the destination segment.  Whole block of
// kQuantThreads threads.  The G source rows are staged in shared memory with
// 16-byte loads; thread t then owns the 8-channel chunk t % (D/8) of the
// tokens t / (D/8) + k TL (TL = threads / (D/8)): exact half2 min/max over
// its tokens, a warp and a block reduction give each channel's (min, max),
// one thread per channel turns them into (s, z), and every thread writes
// the codes of its chunk of its tokens (8 codes = `bits` bytes, one store).
template <int D, int BITS, int Z>
__device__ void quant_k_group(const SegDev& dst, int G, int R, size_t pair,
                              const __half* ring, const __half* in, const RowSrc& src, int p0,
                              int row0, int grow, const QuantSmem& q) {
  constexpr int CH = D / 8;                 // 8-channel chunks of a row
  constexpr int TL = kQuantThreads / CH;    // token lanes
  constexpr int NWARP = kQuantThreads / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cch = tid % CH, tl = tid / CH;
  // up to 4 loads per thread in flight before their stores
  for (int b0 = 0; b0 < G * CH; b0 += 4 * kQuantThreads) {
    int4 v4[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int idx = b0 + k * kQuantThreads + tid;
      if (idx < G * CH) v4[k] = reinterpret_cast<const int4*>(src_row<D>(ring, in, R, src, p0 + idx / CH))[idx % CH];
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int idx = b0 + k * kQuantThreads + tid;
      if (idx < G * CH) reinterpret_cast<int4*>(q.xs + (size_t)(idx / CH) * D)[idx % CH] = v4[k];
    }
  }
  __syncthreads();
  // per-thread min/max of 8 channels over tokens tl, tl + TL, ...
  __half2 mn[4], mx[4];
  {
    const uint4 u = reinterpret_cast<const uint4*>(q.xs + (size_t)tl * D)[cch];
    const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
    for (int e = 0; e < 4; ++e) mn[e] = mx[e] = h[e];
  }
  for (int i = tl + TL; i < G; i += TL) {
    const uint4 u = reinterpret_cast<const uint4*>(q.xs + (size_t)i * D)[cch];
    const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      mn[e] = __hmin2(mn[e], h[e]);
      mx[e] = __hmax2(mx[e], h[e]);
    }
  }
  // lanes of one warp that share the chunk: lane ^ CH, lane ^ 2 CH, ...
#pragma unroll
  for (int off = CH; off < 32; off <<= 1)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      mn[e] = __hmin2(mn[e], __shfl_xor_sync(0xffffffffu, mn[e], off));
      mx[e] = __hmax2(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], off));
    }
  if (lane < CH) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 a = __half22float2(mn[e]), b = __half22float2(mx[e]);
      q.red[(0 * NWARP + warp) * D + cch * 8 + 2 * e] = a.x;
      q.red[(0 * NWARP + warp) * D + cch * 8 + 2 * e + 1] = a.y;
      q.red[(1 * NWARP + warp) * D + cch * 8 + 2 * e] = b.x;
      q.red[(1 * NWARP + warp) * D + cch * 8 + 2 * e + 1] = b.y;
    }
  }
  __syncthreads();
  if (tid < D) {
    float lo = q.red[tid], hi = q.red[NWARP * D + tid];
    for (int w = 1; w < NWARP; ++w) {
      lo = fminf(lo, q.red[w * D + tid]);
      hi = fmaxf(hi, q.red[(NWARP + w) * D + tid]);
    }
    const QParams qp = qparams_any(lo, hi, BITS, Z);
    const size_t gidx = (pair * (size_t)(dst.cap / G) + grow) * D + tid;
    const_cast<__half*>(dst.ks)[gidx] = qp.sh;
    const_cast<__half*>(dst.kz)[gidx] = qp.zh;
    q.par[tid] = qp.s;
    q.par[D + tid] = qp.s != 0.0f ? __frcp_rn(qp.s) : 0.0f;
    q.par[2 * D + tid] = qp.z;
  }
  __syncthreads();
  float cs[8], cr[8], cz[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    cs[e] = q.par[cch * 8 + e];
    cr[e] = q.par[D + cch * 8 + e];
    cz[e] = q.par[2 * D + cch * 8 + e];
  }
  constexpr int rb = D * BITS / 8;
  uint8_t* base = const_cast<uint8_t*>(dst.kc) + (pair * (size_t)dst.cap + row0) * rb;
  for (int i = tl; i < G; i += TL) {
    const uint4 u = reinterpret_cast<const uint4*>(q.xs + (size_t)i * D)[cch];
    const __half* h = reinterpret_cast<const __half*>(&u);
    uint32_t c[8];
    bool tie = false;  // some code too close to a rounding tie for the product
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      bool t;
      c[e] = Z ? qcode_intz_guess<BITS>(__half2float(h[e]), cz[e], cr[e], t)
                      : qcode_guess<BITS>(__half2float(h[e]), cz[e], cr[e], t);
      tie |= t;
    }
    if (tie) {  // rare: redo the chunk with IEEE quotients
#pragma unroll
      for (int e = 0; e < 8; ++e)
        c[e] = Z ? qcode_intz_exact<BITS>(__half2float(h[e]), cz[e], cs[e])
                        : qcode_exact<BITS>(__half2float(h[e]), cz[e], cs[e]);
    }
    uint32_t lo = 0, hi = 0;  // codes 0-3 and 4-7 (8 codes = BITS bytes)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      lo |= c[e] << (e * BITS);
      hi |= c[e + 4] << (e * BITS);
    }
    uint8_t* out = base + (size_t)i * rb + cch * BITS;
    if constexpr (BITS == 2) *reinterpret_cast<uint16_t*>(out) = (uint16_t)(lo | (hi << 8));
    else if constexpr (BITS == 4) *reinterpret_cast<uint32_t*>(out) = lo | (hi << 16);
    else *reinterpret_cast<uint2*>(out) = make_uint2(lo, hi);
  }
  __syncthreads();
}

template <int D, int Z>
__device__ __forceinline__ void quant_k_group_any(const SegDev& dst, int bits, int G, int R, size_t pair,
                                                  const __half* ring, const __half* in, const RowSrc& src,
                                                  int p0, int row0, int grow, const QuantSmem& q) {
  if (bits == 2) quant_k_group<D, 2, Z>(dst, G, R, pair, ring, in, src, p0, row0, grow, q);
  else if (bits == 4) quant_k_group<D, 4, Z>(dst, G, R, pair, ring, in, src, p0, row0, grow, q);
  else quant_k_group<D, 8, Z>(dst, G, R, pair, ring, in, src, p0, row0, grow, q);
}

// Quantize one V token (all D channels, one group per G channels) into packed
// row `row` of the destination segment.  One warp; lane l owns channels
// 4l..4l+3 (lanes >= D/4 idle).
template <int D, int Z>
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
  const QParams qp = qparams_any(mn, mx, bits, Z);
  const float rcp = qp.s != 0.0f ? __frcp_rn(qp.s) : 0.0f;
  uint32_t packed = 0;
  for (int j = 0; j < 4; ++j) {
    const uint32_t c = bits == 2 ? qcode_any<2>(v[j], qp.z, qp.s, rcp, Z)
                       : bits == 4 ? qcode_any<4>(v[j], qp.z, qp.s, rcp, Z)
                                   : qcode_any<8>(v[j], qp.z, qp.s, rcp, Z);
    packed |= c << (j * bits);
  }
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

template <int D, int Z>
__global__ void __launch_bounds__(kQuantThreads) append_kernel(const AppendArgs a) {
  extern __shared__ __align__(16) uint8_t qsm[];
  const QuantSmem qs = quant_smem_view(qsm, a.G, D);
  const size_t pair = blockIdx.x;
  const int chunk = blockIdx.y;
  const __half* in_k = a.k_new + pair * (size_t)a.T * D;
  const __half* in_v = a.v_new + pair * (size_t)a.T * D;
  __half* ring_k = a.kr + pair * (size_t)a.R * D;
  __half* ring_v = a.vr + pair * (size_t)a.R * D;
  const int warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  // launched after a kernel of the same decode step: its writes first
  grid_dep_wait();
  grid_dep_launch();

  if (chunk == 0) {
    // A few new tokens (a decode step) are read into registers first, so
    // their load latency overlaps the quantization below; they are written
    // to the ring only after every read of old ring slots.
    constexpr int kVec = D * 2 / 16;
    const int nk_new = a.T - a.k_first_ring, nv_new = a.T - a.v_first_ring;
    const bool few = nk_new * kVec <= (int)blockDim.x && nv_new * kVec <= (int)blockDim.x;
    int4 pk = make_int4(0, 0, 0, 0), pv = make_int4(0, 0, 0, 0);
    const int tid = threadIdx.x;
    if (few) {
      if (tid < nk_new * kVec) pk = reinterpret_cast<const int4*>(in_k + (size_t)a.k_first_ring * D)[tid];
      if (tid < nv_new * kVec) pv = reinterpret_cast<const int4*>(in_v + (size_t)a.v_first_ring * D)[tid];
    }
    // work that reads old ring slots, before any new token lands in the ring
    for (int gi = 0; gi < a.k_ring_groups; ++gi)
      quant_k_group_any<D, Z>(a.dst, a.bits, a.G, a.R, pair, ring_k, in_k, a.ksrc, gi * a.G,
                       a.k_nk0 + gi * a.G, a.k_nk0 / a.G + gi, qs);
    for (int p = warp; p < a.v_ring_tokens; p += nwarps)
      quant_v_token<D, Z>(a.dst, a.bits, a.Gv, pair, src_row<D>(ring_v, in_v, a.R, a.vsrc, p),
                       a.v_nv0 + p);
    __syncthreads();
    if (few) {
      if (tid < nk_new * kVec)
        reinterpret_cast<int4*>(ring_k + (size_t)((a.k_slot0 + a.k_first_ring + tid / kVec) % a.R) * D)[tid % kVec] = pk;
      if (tid < nv_new * kVec)
        reinterpret_cast<int4*>(ring_v + (size_t)((a.v_slot0 + a.v_first_ring + tid / kVec) % a.R) * D)[tid % kVec] = pv;
    } else {
      if (a.k_first_ring < a.T)
        copy_to_ring<D>(ring_k, a.R, a.k_slot0 + a.k_first_ring, in_k + (size_t)a.k_first_ring * D,
                        a.T - a.k_first_ring);
      if (a.v_first_ring < a.T)
        copy_to_ring<D>(ring_v, a.R, a.v_slot0 + a.v_first_ring, in_v + (size_t)a.v_first_ring * D,
                        a.T - a.v_first_ring);
    }
  }
  if (a.bulk) return;  // the bulk kernels quantize the new tokens
  // work that reads only the new tokens, spread over the chunks (chunk 0
  // takes part only when it is the only one)
  const int workers = a.chunks > 1 ? a.chunks - 1 : 1;
  const int me = a.chunks > 1 ? chunk - 1 : 0;
  if (a.chunks > 1 && chunk == 0) return;
  for (int gi = a.k_ring_groups + me; gi < a.k_groups; gi += workers)
    quant_k_group_any<D, Z>(a.dst, a.bits, a.G, a.R, pair, ring_k, in_k, a.ksrc, gi * a.G,
                     a.k_nk0 + gi * a.G, a.k_nk0 / a.G + gi, qs);
  for (int p = a.v_ring_tokens + me * nwarps + warp; p < a.v_evict; p += workers * nwarps)
    quant_v_token<D, Z>(a.dst, a.bits, a.Gv, pair, src_row<D>(ring_v, in_v, a.R, a.vsrc, p),
                     a.v_nv0 + p);
}

// K flush: group blockIdx.y of the ring's oldest tokens.
template <int D, int Z>
__global__ void __launch_bounds__(kQuantThreads) flush_kernel(const AppendArgs a) {
  extern __shared__ __align__(16) uint8_t qsm[];
  const QuantSmem qs = quant_smem_view(qsm, a.G, D);
  const size_t pair = blockIdx.x;
  const int gi = blockIdx.y;
  const __half* ring_k = a.kr + pair * (size_t)a.R * D;
  // Inside a decode step this grid may start while the decode attention
  // still runs, and even before the step's append has finished: it reads
  // only ring slots written by earlier steps (tokens p >= ksrc.n_old, the
  // step's new one, come from the step's input k_new, not from the ring slot
  // the append is writing) and writes packed rows that the attention and the
  // append leave alone.  It completes only after the attention does (the
  // wait at the end), so a kernel waiting on it waits on both.
  grid_dep_launch();
  const __half* in_k = a.k_new ? a.k_new + pair * (size_t)a.T * D : nullptr;
  quant_k_group_any<D, Z>(a.dst, a.bits, a.G, a.R, pair, ring_k, in_k, a.ksrc, gi * a.G,
                   a.k_nk0 + gi * a.G, a.k_nk0 / a.G + gi, qs);
  grid_dep_wait();
}

// WindowQuant ingest: block (pair, job); job n_jobs is the fp16 tail.
template <int D, int Z>
__global__ void __launch_bounds__(kQuantThreads) ingest_kernel(const IngestArgs a) {
  extern __shared__ __align__(16) uint8_t qsm[];
  const QuantSmem qs = quant_smem_view(qsm, a.G, D);
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
  if (a.ring_only && job.seg >= 0) return;  // quantized by the bulk ingest kernels
  if (job.seg < 0) {
    copy_to_ring<D>(ring_k, a.R, a.krs_push + job.dst, in_k + (size_t)job.src_token * D, a.S);
    copy_to_ring<D>(ring_v, a.R, a.vrs_push + job.dst, in_v + (size_t)job.src_token * D, a.S);
    return;
  }
  const SegDev& dst = a.seg[job.seg];
  const RowSrc src{0, 0};
  const __half* wk = in_k + (size_t)job.src_token * D;
  for (int gi = 0; gi < a.S / a.G; ++gi)
    quant_k_group_any<D, Z>(dst, dst.bits, a.G, a.R, pair, nullptr, wk, src, gi * a.G, job.dst + gi * a.G,
                     job.dst / a.G + gi, qs);
  const int warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  for (int p = warp; p < a.S; p += nwarps)
    quant_v_token<D, Z>(dst, dst.bits, a.Gv, pair, in_v + (size_t)(job.src_token + p) * D, job.dst + p);
}

// ---------------------------------------------------------------------------
// Paged cache: KIVI Algorithm 1 per sequence.  Block (sequence, kv head,
// chunk).  A pool page seen through a SegDev of capacity P with the kv head
// as its "pair" index puts every row, K group and V scale row where the
// pool layout [page][h_kv][P][...] wants it, so the quantizers above write
// pages unchanged.  A block-table entry outside the pool writes nothing and
// sets the cache's error word.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int paged_page(const PagedAppendArgs& a, int b, int row) {
  const int j = row / a.P;
  const int pg = j < a.max_pages ? a.table[(size_t)b * a.max_pages + j] : -1;
  return (pg < 0 || pg >= a.n_pages) ? -1 : pg;
}

__device__ __forceinline__ SegDev paged_view(const PagedAppendArgs& a, int pg) {
  const size_t rows = (size_t)pg * a.h_kv * a.P;
  const int rb = a.d * a.bits / 8;
  SegDev v;
  v.kc = a.kc + rows * rb;
  v.ks = a.ks + rows / a.G * a.d;
  v.kz = a.kz + rows / a.G * a.d;
  v.vc = a.vc + rows * rb;
  v.vs = a.vs + rows * (a.d / a.Gv);
  v.vz = a.vz + rows * (a.d / a.Gv);
  v.bits = a.bits;
  v.cap = a.P;
  v.intz = a.intz;
  return v;
}

template <int D, int Z>
__device__ void paged_k_group(const PagedAppendArgs& a, int b, int h, const PagedAppendSeq& q,
                              const __half* ring, const __half* in, int gi, const QuantSmem& qs) {
  const int row = q.k_nk0 + gi * a.G;
  const int pg = paged_page(a, b, row);  // the same in every thread
  if (pg < 0) {
    if (threadIdx.x == 0) atomicExch(a.page_err, 2);
    return;
  }
  const int r = row % a.P;
  quant_k_group_any<D, Z>(paged_view(a, pg), a.bits, a.G, a.R, (size_t)h, ring, in, q.ksrc, gi * a.G, r,
                          r / a.G, qs);
}

template <int D, int Z>
__device__ void paged_v_token(const PagedAppendArgs& a, int b, int h, const PagedAppendSeq& q,
                              const __half* ring, const __half* in, int p) {
  const int row = q.v_nv0 + p;
  const int pg = paged_page(a, b, row);
  if (pg < 0) {
    if ((threadIdx.x & 31) == 0) atomicExch(a.page_err, 2);
    return;
  }
  quant_v_token<D, Z>(paged_view(a, pg), a.bits, a.Gv, (size_t)h, src_row<D>(ring, in, a.R, q.vsrc, p),
                      row % a.P);
}

template <int D, int Z>
__global__ void __launch_bounds__(kQuantThreads) paged_append_kernel(const PagedAppendArgs a) {
  extern __shared__ __align__(16) uint8_t qsm[];
  const QuantSmem qs = quant_smem_view(qsm, a.G, D);
  const int b = blockIdx.x, h = blockIdx.y, chunk = blockIdx.z;
  const PagedAppendSeq& q = a.seq[b];
  const size_t pair = (size_t)b * a.h_kv + h;
  const __half* in_k = a.k_new + pair * (size_t)a.T * D;
  const __half* in_v = a.v_new + pair * (size_t)a.T * D;
  __half* ring_k = a.kr + pair * (size_t)a.R * D;
  __half* ring_v = a.vr + pair * (size_t)a.R * D;
  const int warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  if (a.flush) {  // the ring's oldest K groups, one chunk per group
    for (int gi = chunk; gi < q.k_groups; gi += a.chunks)
      paged_k_group<D, Z>(a, b, h, q, ring_k, nullptr, gi, qs);
    return;
  }
  if (chunk == 0) {
    // work that reads old ring slots, then the new tokens into the ring
    for (int gi = 0; gi < q.k_ring_groups; ++gi) paged_k_group<D, Z>(a, b, h, q, ring_k, in_k, gi, qs);
    for (int p = warp; p < q.v_ring_tokens; p += nwarps) paged_v_token<D, Z>(a, b, h, q, ring_v, in_v, p);
    __syncthreads();
    if (q.k_first_ring < q.t)
      copy_to_ring<D>(ring_k, a.R, q.k_slot0 + q.k_first_ring, in_k + (size_t)q.k_first_ring * D,
                      q.t - q.k_first_ring);
    if (q.v_first_ring < q.t)
      copy_to_ring<D>(ring_v, a.R, q.v_slot0 + q.v_first_ring, in_v + (size_t)q.v_first_ring * D,
                      q.t - q.v_first_ring);
    if (a.chunks > 1 || a.bulk) return;
  }
  // work that reads only new tokens, over chunks 1.. (or chunk 0 alone)
  const int workers = a.chunks > 1 ? a.chunks - 1 : 1;
  const int me = a.chunks > 1 ? chunk - 1 : 0;
  for (int gi = q.k_ring_groups + me; gi < q.k_groups; gi += workers)
    paged_k_group<D, Z>(a, b, h, q, ring_k, in_k, gi, qs);
  for (int p = q.v_ring_tokens + me * nwarps + warp; p < q.v_evict; p += workers * nwarps)
    paged_v_token<D, Z>(a, b, h, q, ring_v, in_v, p);
}

}  // namespace

size_t quant_smem(int G, int d) { return quant_smem_bytes(G, d); }

// ---- bulk quantize of new tokens (prefill-sized appends), d_h = 128 --------
// Rows a1 / a2 for the groups and tokens that read only the appended input:
// independent work items, so a grid of warps walks them with no block-wide
// step.  Codes match quant_k_group / quant_v_token bit for bit (same qparams,
// same product-then-quotient rounding, decided per element).

constexpr int kBulkThreads = 256;

template <int BITS, int Z>
__device__ __forceinline__ uint32_t pack4(const float (&x)[4], const float (&s)[4], const float (&r)[4],
                                          const float (&z)[4]) {
  uint32_t p = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) p |= qcode_any<BITS>(x[e], z[e], s[e], r[e], Z) << (e * BITS);
  return p;
}

__device__ __forceinline__ uint32_t halves_u32(__half lo, __half hi) {
  return (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
}

// One K group of G rows (src, row stride D) into packed rows row0.. of dst
// and scale / zero group grow, by one warp; lane l owns channels 4l .. 4l + 3.
// Pass 1 takes the channel minima / maxima over the G rows, pass 2 re-reads
// the rows (now in L1/L2) and writes the codes.
template <int BITS, int Z>
__device__ __forceinline__ void quant_group_warp(const __half* src, const SegDev& dst, int G, size_t pair, int row0,
                                                 int grow, int lane) {
  constexpr int D = 128;
  src += 4 * lane;
  float mn[4], mx[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    mn[e] = INFINITY;
    mx[e] = -INFINITY;
  }
#pragma unroll 8
  for (int j = 0; j < G; ++j) {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(src + (size_t)j * D));
    const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
    const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
    const float f[4] = {f0.x, f0.y, f1.x, f1.y};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      mn[e] = fminf(mn[e], f[e]);
      mx[e] = fmaxf(mx[e], f[e]);
    }
  }
  float s[4], r[4], z[4];
  __half sh[4], zh[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const QParams qp = qparams_any(mn[e], mx[e], BITS, Z);
    s[e] = qp.s;
    r[e] = qp.s != 0.0f ? __frcp_rn(qp.s) : 0.0f;
    z[e] = qp.z;
    sh[e] = qp.sh;
    zh[e] = qp.zh;
  }
  const size_t gidx = (pair * (size_t)(dst.cap / G) + (size_t)grow) * D + 4 * lane;
  *reinterpret_cast<uint2*>(const_cast<__half*>(dst.ks) + gidx) =
      make_uint2(halves_u32(sh[0], sh[1]), halves_u32(sh[2], sh[3]));
  *reinterpret_cast<uint2*>(const_cast<__half*>(dst.kz) + gidx) =
      make_uint2(halves_u32(zh[0], zh[1]), halves_u32(zh[2], zh[3]));
  constexpr int rb = D * BITS / 8;
  uint8_t* out = const_cast<uint8_t*>(dst.kc) + (pair * (size_t)dst.cap + (size_t)row0) * rb;
#pragma unroll 8
  for (int j = 0; j < G; ++j) {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(src + (size_t)j * D));
    const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
    const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
    const float f[4] = {f0.x, f0.y, f1.x, f1.y};
    const uint32_t p = pack4<BITS, Z>(f, s, r, z);
    uint8_t* o = out + (size_t)j * rb + lane * (BITS / 2);
    if constexpr (BITS == 2) *o = (uint8_t)p;
    else if constexpr (BITS == 4) *reinterpret_cast<uint16_t*>(o) = (uint16_t)p;
    else *reinterpret_cast<uint32_t*>(o) = p;
  }
}

// One V token (8 channels f of half-lane hl, values already loaded) into
// packed row `row` of dst; the min / max shuffles run on the whole warp, so
// both halves call this together (live = this half has a token).
template <int BITS, int Z>
__device__ __forceinline__ void quant_token_half(const float (&f)[8], bool live, const SegDev& dst, int G,
                                                 size_t pair, int row_in_pair, int hl) {
  constexpr int D = 128;
  const int lpg = G / 8;  // lanes per channel group
  float mn = f[0], mx = f[0];
#pragma unroll
  for (int e = 1; e < 8; ++e) {
    mn = fminf(mn, f[e]);
    mx = fmaxf(mx, f[e]);
  }
  for (int off = 1; off < lpg; off <<= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  }
  if (!live) return;
  const QParams qp = qparams_any(mn, mx, BITS, Z);
  const float rcp = qp.s != 0.0f ? __frcp_rn(qp.s) : 0.0f;
  uint32_t lo = 0, hi = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    lo |= qcode_any<BITS>(f[e], qp.z, qp.s, rcp, Z) << (e * BITS);
    hi |= qcode_any<BITS>(f[e + 4], qp.z, qp.s, rcp, Z) << (e * BITS);
  }
  const size_t row = pair * (size_t)dst.cap + (size_t)row_in_pair;
  uint8_t* o = const_cast<uint8_t*>(dst.vc) + row * (D * BITS / 8) + hl * BITS;
  if constexpr (BITS == 2) *reinterpret_cast<uint16_t*>(o) = (uint16_t)(lo | (hi << 8));
  else if constexpr (BITS == 4) *reinterpret_cast<uint32_t*>(o) = lo | (hi << 16);
  else *reinterpret_cast<uint2*>(o) = make_uint2(lo, hi);
  if ((hl & (lpg - 1)) == 0) {
    const size_t sidx = row * (D / G) + (size_t)(8 * hl / G);
    const_cast<__half*>(dst.vs)[sidx] = qp.sh;
    const_cast<__half*>(dst.vz)[sidx] = qp.zh;
  }
}

__device__ __forceinline__ void load8(const __half* p, bool live, float (&f)[8]) {
  uint4 u = make_uint4(0u, 0u, 0u, 0u);
  if (live) u = __ldg(reinterpret_cast<const uint4*>(p));
  const __half2* h2 = reinterpret_cast<const __half2*>(&u);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 t = __half22float2(h2[e]);
    f[2 * e] = t.x;
    f[2 * e + 1] = t.y;
  }
}

// K groups of a bulk append that read only new tokens: one warp per group.
template <int BITS, int Z>
__global__ void __launch_bounds__(kBulkThreads) bulk_k_kernel(const AppendArgs a) {
  constexpr int D = 128;
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * (kBulkThreads / 32);
  const int per_pair = a.k_groups - a.k_ring_groups;
  const long long items = (long long)a.batch * a.h_kv * per_pair;
  for (long long it = blockIdx.x * (kBulkThreads / 32) + (threadIdx.x >> 5); it < items; it += warps) {
    const size_t pair = (size_t)(it / per_pair);
    const int gi = a.k_ring_groups + (int)(it % per_pair);
    const int p0 = gi * a.G;  // push index of the group's first token
    const __half* src = a.k_new + (pair * (size_t)a.T + (size_t)(p0 - a.ksrc.n_old)) * D;
    quant_group_warp<BITS, Z>(src, a.dst, a.G, pair, a.k_nk0 + p0, a.k_nk0 / a.G + gi, lane);
  }
}

// V tokens of a bulk append that read only new tokens: one half-warp each.
template <int BITS, int Z>
__global__ void __launch_bounds__(kBulkThreads) bulk_v_kernel(const AppendArgs a) {
  constexpr int D = 128;
  const int hl = threadIdx.x & 15;
  const long long halves_n = (long long)gridDim.x * (kBulkThreads / 16);
  const int per_pair = a.v_evict - a.v_ring_tokens;
  const long long items = (long long)a.batch * a.h_kv * per_pair;
  // both halves of a warp run the same number of rounds (shuffles)
  const long long first = (long long)blockIdx.x * (kBulkThreads / 16) + (threadIdx.x >> 4);
  const long long rounds = (items + halves_n - 1) / halves_n;
  for (long long k = 0; k < rounds; ++k) {
    const long long it = first + k * halves_n;
    const bool live = it < items;
    const size_t pair = live ? (size_t)(it / per_pair) : 0;
    const int p = live ? a.v_ring_tokens + (int)(it % per_pair) : 0;
    float f[8];
    load8(a.v_new + (pair * (size_t)a.T + (size_t)(p - a.vsrc.n_old)) * D + 8 * hl, live, f);
    quant_token_half<BITS, Z>(f, live, a.dst, a.Gv, pair, a.v_nv0 + p, hl);
  }
}

// Paged cache, bulk appends: the K groups and V tokens that read only new
// tokens, as bulk_k_kernel / bulk_v_kernel, over the work items of all
// sequences (sequence b's items start at k_item0 / v_item0; its kv heads
// are consecutive).  Rows go to the sequence's pages; a block-table entry
// outside the pool writes nothing and sets the cache's error word.
__device__ __forceinline__ int paged_item_seq(const PagedAppendArgs& a, int it, bool k) {
  int lo = 0, hi = a.n_seq - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((k ? a.seq[mid].k_item0 : a.seq[mid].v_item0) <= it) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

template <int BITS, int Z>
__global__ void __launch_bounds__(kBulkThreads) paged_bulk_k_kernel(const PagedAppendArgs a) {
  constexpr int D = 128;
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * (kBulkThreads / 32);
  for (int it = blockIdx.x * (kBulkThreads / 32) + (threadIdx.x >> 5); it < a.k_items; it += warps) {
    const int b = paged_item_seq(a, it, true);
    const PagedAppendSeq& q = a.seq[b];
    const int per_head = q.k_groups - q.k_ring_groups;
    const int local = it - q.k_item0;
    const int h = local / per_head;
    const int gi = q.k_ring_groups + local % per_head;
    const int p0 = gi * a.G;
    const int row = q.k_nk0 + p0;
    const int pg = paged_page(a, b, row);
    if (pg < 0) {
      if (lane == 0) atomicExch(a.page_err, 2);
      continue;
    }
    const size_t pair = (size_t)b * a.h_kv + h;
    const __half* src = a.k_new + (pair * (size_t)a.T + (size_t)(p0 - q.ksrc.n_old)) * D;
    const int r = row % a.P;
    quant_group_warp<BITS, Z>(src, paged_view(a, pg), a.G, (size_t)h, r, r / a.G, lane);
  }
}

template <int BITS, int Z>
__global__ void __launch_bounds__(kBulkThreads) paged_bulk_v_kernel(const PagedAppendArgs a) {
  constexpr int D = 128;
  const int hl = threadIdx.x & 15;
  const int halves_n = gridDim.x * (kBulkThreads / 16);
  const int first = blockIdx.x * (kBulkThreads / 16) + (threadIdx.x >> 4);
  const int rounds = (a.v_items + halves_n - 1) / halves_n;
  // both halves of a warp run the same number of rounds (shuffles)
  for (int k = 0; k < rounds; ++k) {
    const int it = first + k * halves_n;
    bool live = it < a.v_items;
    int b = 0, h = 0, p = 0, pg = 0;
    if (live) {
      b = paged_item_seq(a, it, false);
      const PagedAppendSeq& q = a.seq[b];
      const int per_head = q.v_evict - q.v_ring_tokens;
      const int local = it - q.v_item0;
      h = local / per_head;
      p = q.v_ring_tokens + local % per_head;
      pg = paged_page(a, b, q.v_nv0 + p);
      if (pg < 0) {
        if (hl == 0) atomicExch(a.page_err, 2);
        live = false;
      }
    }
    const PagedAppendSeq& q = a.seq[b];
    const size_t pair = (size_t)b * a.h_kv + h;
    float f[8];
    load8(a.v_new + (pair * (size_t)a.T + (size_t)(p - q.vsrc.n_old)) * D + 8 * hl, live, f);
    quant_token_half<BITS, Z>(f, live, paged_view(a, live ? pg : 0), a.Gv, (size_t)h, (q.v_nv0 + p) % a.P, hl);
  }
}

// WindowQuant reordered ingest: the K groups and V tokens of every quantized
// window go to the rows its job names, in the segment of its width (rings
// and the fp16 tail: ingest_kernel).  Work items are (pair, window, group)
// for K and (pair, window, token) for V.
template <int Z>
__global__ void __launch_bounds__(kBulkThreads) ingest_bulk_k_kernel(const IngestArgs a) {
  constexpr int D = 128;
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * (kBulkThreads / 32);
  const int gpw = a.S / a.G;  // K groups per window
  const long long items = (long long)a.batch * a.h_kv * a.n_jobs * gpw;
  for (long long it = blockIdx.x * (kBulkThreads / 32) + (threadIdx.x >> 5); it < items; it += warps) {
    const size_t pair = (size_t)(it / ((long long)a.n_jobs * gpw));
    const int rest = (int)(it % ((long long)a.n_jobs * gpw));
    const WindowJob job = a.jobs[rest / gpw];
    if (job.seg < 0) continue;
    const int g = rest % gpw;
    const SegDev& dst = a.seg[job.seg];
    const __half* src = a.k_new + (pair * (size_t)a.T + (size_t)(job.src_token + g * a.G)) * D;
    const int row0 = job.dst + g * a.G, grow = job.dst / a.G + g;
    if (dst.bits == 2) quant_group_warp<2, Z>(src, dst, a.G, pair, row0, grow, lane);
    else if (dst.bits == 4) quant_group_warp<4, Z>(src, dst, a.G, pair, row0, grow, lane);
    else quant_group_warp<8, Z>(src, dst, a.G, pair, row0, grow, lane);
  }
}

template <int Z>
__global__ void __launch_bounds__(kBulkThreads) ingest_bulk_v_kernel(const IngestArgs a) {
  constexpr int D = 128;
  const int hl = threadIdx.x & 15;
  const long long halves_n = (long long)gridDim.x * (kBulkThreads / 16);
  const long long per_pair = (long long)a.n_jobs * a.S;
  const long long items = (long long)a.batch * a.h_kv * per_pair;
  const long long first = (long long)blockIdx.x * (kBulkThreads / 16) + (threadIdx.x >> 4);
  const long long rounds = (items + halves_n - 1) / halves_n;
  for (long long k = 0; k < rounds; ++k) {
    const long long it = first + k * halves_n;
    bool live = it < items;
    const size_t pair = live ? (size_t)(it / per_pair) : 0;
    const int rest = live ? (int)(it % per_pair) : 0;
    const WindowJob job = a.jobs[rest / a.S];
    const int t = rest % a.S;
    live = live && job.seg >= 0;
    // a warp's two halves may hold windows of different widths: the group
    // reduction is the same for all widths, so one call site per width with
    // the other half idle keeps the shuffles converged
    const int bits = live ? a.seg[job.seg].bits : 0;
    float f[8];
    load8(a.v_new + (pair * (size_t)a.T + (size_t)(job.src_token + t)) * D + 8 * hl, live, f);
    const SegDev& dst = a.seg[live ? job.seg : 0];
    quant_token_half<2, Z>(f, live && bits == 2, dst, a.Gv, pair, job.dst + t, hl);
    quant_token_half<4, Z>(f, live && bits == 4, dst, a.Gv, pair, job.dst + t, hl);
    quant_token_half<8, Z>(f, live && bits == 8, dst, a.Gv, pair, job.dst + t, hl);
  }
}

template <class K>
cudaError_t set_smem(K kernel, size_t bytes) {
  return set_smem_once((const void*)kernel, (int)bytes);
}

template <int BITS, int Z>
cudaError_t launch_bulk_b(const AppendArgs& a, cudaStream_t s) {
  const long long P = (long long)a.batch * a.h_kv;
  const long long nk = P * (a.k_groups - a.k_ring_groups), nv = P * (a.v_evict - a.v_ring_tokens);
  const long long cap = 4096;  // blocks: enough to fill any GPU, then the warps loop
  if (nk > 0) bulk_k_kernel<BITS, Z><<<(int)std::min(cap, (nk + 7) / 8), kBulkThreads, 0, s>>>(a);
  if (nv > 0) bulk_v_kernel<BITS, Z><<<(int)std::min(cap, (nv + 15) / 16), kBulkThreads, 0, s>>>(a);
  return cudaGetLastError();
}

template <int D, int Z>
cudaError_t launch_append_dz(const AppendArgs& a, cudaStream_t s, bool pdl) {
  dim3 grid(a.batch * a.h_kv, a.chunks);
  const size_t sm = quant_smem(a.G, a.d);
  cudaError_t e;
  if ((e = set_smem(append_kernel<D, Z>, sm)) != cudaSuccess) return e;
  if ((e = launch_kernel(append_kernel<D, Z>, grid, dim3(kQuantThreads), sm, s, pdl && !a.bulk, a)) != cudaSuccess)
    return e;
  if (D == 128 && a.bulk) {
    if (a.bits == 2) return launch_bulk_b<2, Z>(a, s);
    if (a.bits == 4) return launch_bulk_b<4, Z>(a, s);
    return launch_bulk_b<8, Z>(a, s);
  }
  return cudaSuccess;
}

cudaError_t launch_append(const AppendArgs& a, cudaStream_t s, bool pdl) {
  if (a.d == 128) return a.dst.intz ? launch_append_dz<128, 1>(a, s, pdl) : launch_append_dz<128, 0>(a, s, pdl);
  return a.dst.intz ? launch_append_dz<64, 1>(a, s, pdl) : launch_append_dz<64, 0>(a, s, pdl);
}

template <int D, int Z>
cudaError_t launch_flush_dz(const AppendArgs& a, cudaStream_t s, bool pdl) {
  dim3 grid(a.batch * a.h_kv, a.k_groups);
  const size_t sm = quant_smem(a.G, a.d);
  cudaError_t e;
  if ((e = set_smem(flush_kernel<D, Z>, sm)) != cudaSuccess) return e;
  return launch_kernel(flush_kernel<D, Z>, grid, dim3(kQuantThreads), sm, s, pdl, a);
}

cudaError_t launch_flush(const AppendArgs& a, cudaStream_t s, bool pdl) {
  if (a.k_groups <= 0) return cudaSuccess;
  if (a.d == 128) return a.dst.intz ? launch_flush_dz<128, 1>(a, s, pdl) : launch_flush_dz<128, 0>(a, s, pdl);
  return a.dst.intz ? launch_flush_dz<64, 1>(a, s, pdl) : launch_flush_dz<64, 0>(a, s, pdl);
}

template <int D, int Z>
cudaError_t launch_ingest_dz(const IngestArgs& a, cudaStream_t s) {
  dim3 grid(a.batch * a.h_kv, a.n_jobs + 1);
  const size_t sm = quant_smem(a.G, a.d);
  cudaError_t e;
  if ((e = set_smem(ingest_kernel<D, Z>, sm)) != cudaSuccess) return e;
  if (D == 128 && a.Gv >= 8 && a.Gv <= 128) {
    // ring windows and the tail by the block kernel, quantized windows by
    // the grid-wide ones
    IngestArgs r = a;
    r.ring_only = 1;
    ingest_kernel<D, Z><<<grid, kQuantThreads, sm, s>>>(r);
    const long long P = (long long)a.batch * a.h_kv;
    const long long nk = P * a.n_jobs * (a.S / a.G), nv = P * a.n_jobs * a.S;
    const long long cap = 4096;
    if (nk > 0) ingest_bulk_k_kernel<Z><<<(int)std::min(cap, (nk + 7) / 8), kBulkThreads, 0, s>>>(a);
    if (nv > 0) ingest_bulk_v_kernel<Z><<<(int)std::min(cap, (nv + 15) / 16), kBulkThreads, 0, s>>>(a);
  } else {
    ingest_kernel<D, Z><<<grid, kQuantThreads, sm, s>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t launch_ingest(const IngestArgs& a, cudaStream_t s) {
  const int z = a.seg[0].intz;  // one zero-point mode per cache
  if (a.d == 128) return z ? launch_ingest_dz<128, 1>(a, s) : launch_ingest_dz<128, 0>(a, s);
  return z ? launch_ingest_dz<64, 1>(a, s) : launch_ingest_dz<64, 0>(a, s);
}

template <int BITS, int Z>
cudaError_t launch_paged_bulk_b(const PagedAppendArgs& a, cudaStream_t s) {
  const int cap = 4096;  // blocks: enough to fill any GPU, then the warps loop
  if (a.k_items > 0) paged_bulk_k_kernel<BITS, Z><<<std::min(cap, (a.k_items + 7) / 8), kBulkThreads, 0, s>>>(a);
  if (a.v_items > 0) paged_bulk_v_kernel<BITS, Z><<<std::min(cap, (a.v_items + 15) / 16), kBulkThreads, 0, s>>>(a);
  return cudaGetLastError();
}

template <int D, int Z>
cudaError_t launch_paged_append_dz(const PagedAppendArgs& a, cudaStream_t s) {
  dim3 grid(a.batch, a.h_kv, a.chunks);
  const size_t sm = quant_smem(a.G, a.d);
  cudaError_t e;
  if ((e = set_smem(paged_append_kernel<D, Z>, sm)) != cudaSuccess) return e;
  paged_append_kernel<D, Z><<<grid, kQuantThreads, sm, s>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (D == 128 && a.bulk) {
    if (a.bits == 2) return launch_paged_bulk_b<2, Z>(a, s);
    if (a.bits == 4) return launch_paged_bulk_b<4, Z>(a, s);
    return launch_paged_bulk_b<8, Z>(a, s);
  }
  return cudaSuccess;
}

cudaError_t launch_paged_append(const PagedAppendArgs& a, cudaStream_t s) {
  if (a.d == 128) return a.intz ? launch_paged_append_dz<128, 1>(a, s) : launch_paged_append_dz<128, 0>(a, s);
  return a.intz ? launch_paged_append_dz<64, 1>(a, s) : launch_paged_append_dz<64, 0>(a, s);
}

}  // namespace kvq
