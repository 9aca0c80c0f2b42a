// FP8 helpers of the backward operands: E4M3 / E5M2 conversion and the MX
// block exponent (one E8M0 scale per 32 elements, no clipping of the block
// maximum).
#pragma once
#include <cstdint>

namespace fp4attn {

constexpr int kFmtE4M3 = 0, kFmtE5M2 = 1;

// Four fp32 values -> four FP8 codes (round to nearest even, saturating to
// the largest finite value), x0 in the low byte.
template <int FMT>
__device__ __forceinline__ uint32_t cvt_fp8x4(float x0, float x1, float x2, float x3) {
  uint32_t r;
  if constexpr (FMT == kFmtE4M3) {
    asm("{\n.reg .b16 lo, hi;\n"
        "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n"
        "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n"
        "mov.b32 %0, {lo, hi};\n}\n"
        : "=r"(r)
        : "f"(x0), "f"(x1), "f"(x2), "f"(x3));
  } else {
    asm("{\n.reg .b16 lo, hi;\n"
        "cvt.rn.satfinite.e5m2x2.f32 lo, %2, %1;\n"
        "cvt.rn.satfinite.e5m2x2.f32 hi, %4, %3;\n"
        "mov.b32 %0, {lo, hi};\n}\n"
        : "=r"(r)
        : "f"(x0), "f"(x1), "f"(x2), "f"(x3));
  }
  return r;
}

// Largest finite value of the format = 1.75 * 2^P.
template <int FMT>
constexpr int kFp8MaxExp = (FMT == kFmtE4M3) ? 8 : 15;

// The smallest e >= -127 with amax <= 1.75 * 2^(P + e), from the bits of a
// non-negative fp32 amax (f 2^k, f in [1, 2): e = k - P if f <= 1.75, else
// k - P + 1; amax = 0 or below 2^-126 gives -127).
template <int FMT>
__device__ __forceinline__ int mx_exp_f32(float amax) {
  const uint32_t a = __float_as_uint(amax);
  const int ebits = static_cast<int>(a >> 23);
  if (ebits == 0) return -127;
  const int e = ebits - 127 - ((a & 0x7FFFFFu) <= 0x600000u ? kFp8MaxExp<FMT> : kFp8MaxExp<FMT> - 1);
  return e < -127 ? -127 : e;
}

// The same from the bits of a non-negative bf16 amax (7 mantissa bits).
template <int FMT>
__device__ __forceinline__ int mx_exp_bf16(uint32_t m) {
  const int ebits = static_cast<int>(m >> 7);
  if (ebits == 0) return -127;
  const int e = ebits - 127 - ((m & 0x7Fu) <= 0x60u ? kFp8MaxExp<FMT> : kFp8MaxExp<FMT> - 1);
  return e < -127 ? -127 : e;
}

// (a0 * b0, a1 * b1) and (a0 - b0, a1 - b1), each rounded once (packed fp32).
__device__ __forceinline__ void fmul2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n.reg .b64 a, b, d;\n"
      "mov.b64 a, {%2, %3};\n"
      "mov.b64 b, {%4, %5};\n"
      "mul.rn.f32x2 d, a, b;\n"
      "mov.b64 {%0, %1}, d;\n}\n"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ void fsub2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n.reg .b64 a, b, d;\n"
      "mov.b64 a, {%2, %3};\n"
      "mov.b64 b, {%4, %5};\n"
      "sub.rn.f32x2 d, a, b;\n"
      "mov.b64 {%0, %1}, d;\n}\n"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// Explicit shared-memory accesses (addresses in the shared window).
__device__ __forceinline__ float4 lds_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ void sts_u4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ void sts_u8(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u8 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void sts_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

// 16 consecutive fp32 TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// 2^-e for -127 <= e <= 126, exact.
__device__ __forceinline__ float pow2_neg(int e) { return __uint_as_float(static_cast<uint32_t>(127 - e) << 23); }

}  // namespace fp4attn
