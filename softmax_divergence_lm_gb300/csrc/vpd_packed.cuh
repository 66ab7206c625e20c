// vpd_packed.cuh -- packed 16-bit logits and fp32x2 arithmetic shared by the
// single-read kernel and the streaming kernels: the bf16 / fp16 input formats
// (two values per 32-bit word, exact upcast folded into x - m), the packed
// max, and fp32x2 helpers over the hardware ex2 / lg2.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "vpd_device.cuh"

namespace vpd {

__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}
// ---------------------------------------------------------------------------
// 16-bit input formats: pairs of values packed in one 32-bit word.
// ---------------------------------------------------------------------------
// -inf can be clamped to a finite floor (twice, packed) so that a difference
// x - m stays finite where it multiplies a probability that is 0: (x - m) log2 e
// cannot overflow while the row max is at most 2^126.
struct InBF16 {
  static constexpr uint32_t kNegInf2 = 0xff80ff80u;
  static constexpr uint32_t kNegBig2 = 0xf180f180u;  // -2^100
  __device__ static __forceinline__ uint32_t max_nan(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
  }
  __device__ static __forceinline__ uint32_t max2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
  }
  __device__ static __forceinline__ float2 unpack(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  }
  // (x - m) for both halves, the exact upcast folded into the subtraction
  __device__ static __forceinline__ float2 sub(uint32_t w, float2 nm) {
    float lo, hi;
    asm("{ .reg .b16 a, b; mov.b32 {a, b}, %2; add.rn.f32.bf16 %0, a, %3; add.rn.f32.bf16 %1, b, %4; }"
        : "=f"(lo), "=f"(hi)
        : "r"(w), "f"(nm.x), "f"(nm.y));
    return make_float2(lo, hi);
  }
  using GSame = GBF16;
};
struct InF16 {
  static constexpr uint32_t kNegInf2 = 0xfc00fc00u;
  static constexpr uint32_t kNegBig2 = 0xfbfffbffu;  // -65504, the most negative finite
  __device__ static __forceinline__ uint32_t max_nan(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.NaN.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
  }
  __device__ static __forceinline__ uint32_t max2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
  }
  __device__ static __forceinline__ float2 unpack(uint32_t w) {
    float lo, hi;
    asm("{ .reg .f16 a, b; mov.b32 {a, b}, %2; cvt.f32.f16 %0, a; cvt.f32.f16 %1, b; }"
        : "=f"(lo), "=f"(hi)
        : "r"(w));
    return make_float2(lo, hi);
  }
  __device__ static __forceinline__ float2 sub(uint32_t w, float2 nm) {
    float lo, hi;
    asm("{ .reg .b16 a, b; mov.b32 {a, b}, %2; add.rn.f32.f16 %0, a, %3; add.rn.f32.f16 %1, b, %4; }"
        : "=f"(lo), "=f"(hi)
        : "r"(w), "f"(nm.x), "f"(nm.y));
    return make_float2(lo, hi);
  }
  using GSame = GF16;
};

__device__ __forceinline__ float2 f2(float a) { return make_float2(a, a); }
__device__ __forceinline__ float2 neg(float2 a) { return make_float2(-a.x, -a.y); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 ex2_2(float2 a) { return make_float2(ex2(a.x), ex2(a.y)); }
__device__ __forceinline__ float2 lg2_2(float2 a) { return make_float2(lg2(a.x), lg2(a.y)); }

}  // namespace vpd
