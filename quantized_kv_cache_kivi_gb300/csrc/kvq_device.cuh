// Device helpers: the quantizer's arithmetic, and the bulk-copy / mbarrier
// primitives of the decode pipeline (sm_100+ PTX).
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace kvq {

// ---------------------------------------------------------------------------
// The quantizer (KIVI "方法细节": Q(X) = round((X - z) / s), X' = Q s + z;
// WindowQuant §3.3.3 Eq.14/16: s = (max - min)/(qmax - qmin), clamp to
// [0, 2^b - 1]).  Expression order fixed so codes, scales and zeros are
// reproducible bit for bit: fp32 subtract, IEEE divide, fp16 round-to-nearest
// of s, z = min (exact), codes from the fp16-rounded s, rint half-to-even.
// ---------------------------------------------------------------------------
struct QParams {
  float s;  // fp16-rounded scale as fp32
  float z;  // zero point (the minimum) as fp32
  __half sh, zh;
};

__device__ __forceinline__ QParams qparams(float mn, float mx, int bits) {
  const float qmax = (float)((1 << bits) - 1);
  QParams p;
  const float s32 = __fdiv_rn(__fsub_rn(mx, mn), qmax);
  p.sh = __float2half_rn(s32);
  p.zh = __float2half_rn(mn);
  p.s = __half2float(p.sh);
  p.z = __half2float(p.zh);
  return p;
}

__device__ __forceinline__ uint32_t qcode(float x, const QParams& p, int bits) {
  if (p.s == 0.0f) return 0u;
  const float qmax = (float)((1 << bits) - 1);
  float r = rintf(__fdiv_rn(__fsub_rn(x, p.z), p.s));
  r = fminf(fmaxf(r, 0.0f), qmax);
  return (uint32_t)r;
}

// Same code as qcode, faster: the quotient (x - z) / s is first formed as
// (x - z) * (1/s).  Both that product and the IEEE quotient lie within a few
// fp32 ulps of the exact ratio (ulp <= 2^-16 for ratios below 256), so they
// round to the same integer unless the product is within 1e-4 of a
// half-integer (|t - rint(t)| > 0.4999); only then is the IEEE division
// done.  `rcp` = 1/s rounded, or 0 when s == 0 (then t = 0 and the code is
// 0, as in qcode).  x >= z always (z is the group minimum), so the rounded
// quotient is >= 0; it is clamped to 2^BITS - 1 from above.
template <int BITS>
__device__ __forceinline__ uint32_t qcode_fast(float x, float z, float s, float rcp) {
  const float d = __fsub_rn(x, z);
  const float t = __fmul_rn(d, rcp);
  float r = rintf(t);
  if (fabsf(t - r) > 0.4999f) r = rintf(__fdiv_rn(d, s));
  return min(__float2uint_rn(r), (1u << BITS) - 1u);
}

// The fast half of qcode_fast without its branch: the code from the product,
// and whether the IEEE quotient has to decide instead (qcode_exact).
template <int BITS>
__device__ __forceinline__ uint32_t qcode_guess(float x, float z, float rcp, bool& near_tie) {
  const float t = __fmul_rn(__fsub_rn(x, z), rcp);
  const float r = rintf(t);
  near_tie = fabsf(t - r) > 0.4999f;
  return min(__float2uint_rn(r), (1u << BITS) - 1u);
}
template <int BITS>
__device__ __forceinline__ uint32_t qcode_exact(float x, float z, float s) {
  if (s == 0.0f) return 0u;  // constant group (or an underflowed scale): code 0
  return min(__float2uint_rn(rintf(__fdiv_rn(__fsub_rn(x, z), s))), (1u << BITS) - 1u);
}

// Integer zero point (WindowQuant §3.3.3, qmin = 0): Eq.16 s = (max - min) /
// qmax, z = -round(min / s); Eq.14 Q = clamp(round(x / s) + z, 0, qmax);
// Eq.15 x' = s (Q - z).  s is stored as fp16 and used rounded; z is stored
// as a 16-bit two's-complement integer in the zero slot (p.zh holds those
// bits, p.z the integer as fp32).  Where Eq.16 is undefined or z would not
// fit 16 bits: a constant group (or one whose s rounds to 0) takes
// s = |min|, so z = -sign(min) and its codes are 0; if |round(min / s)|
// exceeds 32767 (8 bits, or 4 bits with a subnormal s) s is raised to the
// smallest fp16 value for which it does not.
__device__ __forceinline__ QParams qparams_intz(float mn, float mx, int bits) {
  const float qmax = (float)((1 << bits) - 1);
  QParams p;
  const float s32 = __fdiv_rn(__fsub_rn(mx, mn), qmax);
  p.sh = __float2half_rn(s32);
  p.s = __half2float(p.sh);
  if (p.s == 0.0f) {
    p.sh = __float2half_rn(fabsf(mn));  // exact: mn is an fp16 value
    p.s = __half2float(p.sh);
  }
  float zr = 0.0f;
  if (p.s != 0.0f) {
    zr = rintf(__fdiv_rn(mn, p.s));
    if (fabsf(zr) > 32767.0f) {
      const float t = __fdiv_rn(fabsf(mn), 32767.0f);
      unsigned short h = __half_as_ushort(__float2half_rn(t));
      if (__half2float(__ushort_as_half(h)) < t) ++h;  // smallest fp16 >= t
      for (int k = 0; k < 8 && fabsf(rintf(__fdiv_rn(mn, __half2float(__ushort_as_half(h))))) > 32767.0f; ++k) ++h;
      p.sh = __ushort_as_half(h);
      p.s = __half2float(p.sh);
      zr = rintf(__fdiv_rn(mn, p.s));
    }
  }
  const int zi = -(int)zr;
  p.z = (float)zi;
  p.zh = __short_as_half((short)zi);
  return p;
}

// clamp(rint(x / s) + z, 0, qmax): the product x * (1/s) decides unless it
// lies near a rounding tie, then the IEEE quotient does.  t = x * rcp and
// the quotient both lie within |t| 2^-22.4 of the exact ratio (two and one
// fp32 roundings), so they round alike when t is farther than |t| 2^-20
// from a half-integer; |t| is up to ~2^15 here (x / s is not bounded by
// qmax as (x - min) / s is), so the window scales with it.
template <int BITS>
__device__ __forceinline__ uint32_t qcode_intz_guess(float x, float zi, float rcp, bool& near_tie) {
  const float t = __fmul_rn(x, rcp);
  const float r = rintf(t);
  near_tie = fabsf(t - r) > 0.5f - fabsf(t) * 0x1p-20f;
  return (uint32_t)min(max(__float2int_rn(r + zi), 0), (1 << BITS) - 1);
}
template <int BITS>
__device__ __forceinline__ uint32_t qcode_intz_exact(float x, float zi, float s) {
  if (s == 0.0f) return 0u;
  return (uint32_t)min(max(__float2int_rn(rintf(__fdiv_rn(x, s)) + zi), 0), (1 << BITS) - 1);
}
template <int BITS>
__device__ __forceinline__ uint32_t qcode_intz_fast(float x, float zi, float s, float rcp) {
  bool tie;
  const uint32_t c = qcode_intz_guess<BITS>(x, zi, rcp, tie);
  return tie ? qcode_intz_exact<BITS>(x, zi, s) : c;
}

// The additive zero of a dequantized value x' = code s + zero, from the 16
// bits of a zero slot and of the matching scale: the stored fp16 zero
// (KIVI, z = min), or -s z for an integer zero point z (WindowQuant Eq.15,
// x' = s (code - z)), formed in fp32.
__device__ __forceinline__ float zero_add(uint16_t zbits, uint16_t sbits, bool intz) {
  if (!intz) return __half2float(__ushort_as_half(zbits));
  return -__half2float(__ushort_as_half(sbits)) * (float)(short)zbits;
}
// The same rounded to fp16 bits, for fp16 tensor-core operands.
__device__ __forceinline__ uint16_t zero_add_h(uint16_t zbits, uint16_t sbits, bool intz) {
  if (!intz) return zbits;
  return __half_as_ushort(__float2half_rn(-__half2float(__ushort_as_half(sbits)) * (float)(short)zbits));
}

// Either quantizer, by the destination's zero point.
__device__ __forceinline__ QParams qparams_any(float mn, float mx, int bits, int intz) {
  return intz ? qparams_intz(mn, mx, bits) : qparams(mn, mx, bits);
}
template <int BITS>
__device__ __forceinline__ uint32_t qcode_any(float x, float z, float s, float rcp, int intz) {
  return intz ? qcode_intz_fast<BITS>(x, z, s, rcp) : qcode_fast<BITS>(x, z, s, rcp);
}

// ---------------------------------------------------------------------------
// Shared-memory address, mbarrier and 1-D bulk copy (TMA engine, no tensor map)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of an mbarrier for at most ~2^31 SM clocks (about a
// second).  Returns false on timeout; the caller records the error and stops.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > (1ll << 31)) return false;
  }
  return true;
}

// Bounded wait that ignores any abort flag (about 2^28 SM clocks): a warp
// that issued bulk copies waits with it for them to land before their stage
// is reused and before its block exits, aborted or not.
// Returns false if the phase did not complete in time.
__device__ __forceinline__ bool mbar_drain_bounded(uint64_t* bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 >= (1ll << 28)) return false;
    __nanosleep(128);
  }
  return true;
}

// global -> shared bulk copy completing on an mbarrier (16-byte aligned
// addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Programmatic dependent launch: wait until the grids this one depends on have
// completed and their writes are visible (returns at once for a grid launched
// without the attribute), and let the grid launched after this one start.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// 16-byte asynchronous global -> shared copy cached in L2 only (cp.async.cg),
// its group commit and the wait for all but the N most recent groups.
__device__ __forceinline__ void cp16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// An arrival on an mbarrier once this thread's cp.async copies issued so far
// have completed (.noinc: counted in the barrier's expected arrivals).
__device__ __forceinline__ void cp_mbar_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_plain(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------------------
// Packed fp32 pair arithmetic (sm_100+): two lanes of fp32 per instruction.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) { return __fmul2_rn(a, b); }

// Code of `bits` width at bit position `pos` of word w, as an exact fp32
// value times 2^pos: (w & mask) is OR-ed into the mantissa of 2^23, and 2^23
// is subtracted.  Exact while the masked field stays below 2^23 (pos <= 21
// for 2-bit fields).
__device__ __forceinline__ float field_scaled(uint32_t w, uint32_t mask) {
  return __uint_as_float((w & mask) | 0x4B000000u) - 8388608.0f;
}

}  // namespace kvq
