// Tensor-core building blocks of the decode kernels at d_h = 128: the token
// order inside a 16-token sub-tile, the code fields of packed words as exact
// fp16 operands, the mma.sync fragment helpers and the mbarrier waits.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "kvq_device.cuh"

namespace kvq {
namespace mma {

constexpr int D = 128;
constexpr uint32_t kFull = 0xffffffffu;

// Token of row r of a 16-token sub-tile.  Swapping neighbours in the upper
// half of each 8-row block keeps both the K row loads (rows gid) and the V
// row loads (rows 2 tig, 2 tig + 1, ...) free of shared-memory bank conflicts.
__host__ __device__ constexpr int sigma(int r) { return r ^ ((r >> 2) & 1); }

// ---- code fields ------------------------------------------------------------
// A 32-bit word holds 32/B codes: two 16-bit halves of 16/B fields each.
// Fields inside bits 0..9 of a half are used in place (p = j B); the others
// are taken from the word shifted right by 6 (p = j B - 6).  Either way the
// field sits at bit p <= 8 with p + B <= 10, inside the fp16 mantissa.
template <int B>
struct Fields {
  static constexpr int INPLACE = B == 2 ? 5 : (B == 4 ? 2 : 1);
  __host__ __device__ static constexpr int pos(int j) { return j < INPLACE ? j * B : j * B - 6; }
  // (code_lo 2^(p-24), code_hi 2^(p-24)) as a half2: field j of both halves
  __device__ static __forceinline__ uint32_t get(uint32_t x, uint32_t x_shr6, int j) {
    const uint32_t m = ((1u << B) - 1u) << pos(j);
    return (j < INPLACE ? x : x_shr6) & (m | (m << 16));
  }
};

// K: thread tig owns channels [32 tig, 32 tig + 32) of its rows; its h-th
// half2 (h = 2 kt + e, e = 0 for k columns 2 tig.., 1 for 2 tig + 8..) holds
// field j = h % PER_HALF of word w = h / PER_HALF: channels c_lo (low half)
// and c_hi (high half).
template <int B>
__host__ __device__ constexpr void k_half2_channels(int tig, int h, int* c_lo, int* c_hi, int* p) {
  constexpr int PH = 16 / B;
  const int w = h / PH, j = h % PH;
  const int base = 32 * tig + w * (32 / B);
  *c_lo = base + j;
  *c_hi = base + PH + j;
  *p = Fields<B>::pos(j);
}

// V: thread gid owns channels [16 gid, 16 gid + 16) of its tokens; m-tile mt
// = (word w, field j), w = mt / PER_HALF, j = mt % PER_HALF; row gid <- the
// low-half channel, row gid + 8 <- the high-half channel.
template <int B>
__host__ __device__ constexpr void v_rows(int gid, int mt, int* c_row0, int* c_row8, int* p) {
  constexpr int PH = 16 / B;
  const int w = mt / PH, j = mt % PH;
  const int base = 16 * gid + w * (32 / B);
  *c_row0 = base + j;
  *c_row8 = base + PH + j;
  *p = Fields<B>::pos(j);
}

// Volatile on purpose: the source order of the MMAs is their issue order,
// which is arranged so that two MMAs on one accumulator are several apart.
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 8x8 b16 transpose across the warp: lane (gid, tig) passes row gid, columns
// 2 tig, 2 tig + 1 and receives row gid of the transpose.
__device__ __forceinline__ uint32_t movm_trans(uint32_t x) {
  uint32_t y;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t hmul2u(uint32_t a, uint32_t b) {
  const __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
  return *reinterpret_cast<const uint32_t*>(&r);
}
__device__ __forceinline__ uint32_t halves(uint32_t lo, uint32_t hi) {
  return (lo & 0xffffu) | (hi << 16);
}
// (p_lo z_lo, p_hi z_hi) as fp16 for integer zero points: p2 holds two fp16
// probabilities, z and s the 16 bits of the zero slots and of their scales;
// z' = -s z and the product p z' are formed in fp32 and rounded once.
__device__ __forceinline__ uint32_t p_times_zero(uint32_t p2, uint32_t z_lo, uint32_t z_hi, uint32_t s_lo,
                                                 uint32_t s_hi) {
  const float2 p = __half22float2(*reinterpret_cast<const __half2*>(&p2));
  return pack_half2(p.x * zero_add((uint16_t)z_lo, (uint16_t)s_lo, true),
                    p.y * zero_add((uint16_t)z_hi, (uint16_t)s_hi, true));
}

__device__ __forceinline__ bool try_wait_at(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// The same with a suspend-time hint: the waiting thread may sleep in the
// barrier unit until the phase completes (or about `ns` nanoseconds pass)
// instead of spinning through issue slots the working warps need.
__device__ __forceinline__ bool try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}


}  // namespace mma
}  // namespace kvq
