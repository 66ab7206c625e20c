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
  // The single-read kernels' view: 8-element vectors (16 bytes) of 4 words,
  // each word a packed pair.
  static constexpr int kSize = 2;  // bytes per element
  using Word = uint32_t;
  using Vec = uint4;
  __device__ static __forceinline__ Vec ld(const unsigned char* p) { return *reinterpret_cast<const uint4*>(p); }
  __device__ static __forceinline__ void words(const Vec& v, Word (&w)[4]) {
    w[0] = v.x;
    w[1] = v.y;
    w[2] = v.z;
    w[3] = v.w;
  }
  __device__ static __forceinline__ Word neg_inf_w() { return kNegInf2; }
  __device__ static __forceinline__ Word neg_big_w() { return kNegBig2; }
  __device__ static __forceinline__ Vec fill_neg_big() { return make_uint4(kNegBig2, kNegBig2, kNegBig2, kNegBig2); }
  // nonzero where `oth` is -inf and `tgt` is not (a KL support violation)
  __device__ static __forceinline__ uint32_t viol(Word tgt, Word oth) {
    return __vcmpeq2(oth, kNegInf2) & ~__vcmpeq2(tgt, kNegInf2);
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
  // The single-read kernels' view: 8-element vectors (16 bytes) of 4 words,
  // each word a packed pair.
  static constexpr int kSize = 2;  // bytes per element
  using Word = uint32_t;
  using Vec = uint4;
  __device__ static __forceinline__ Vec ld(const unsigned char* p) { return *reinterpret_cast<const uint4*>(p); }
  __device__ static __forceinline__ void words(const Vec& v, Word (&w)[4]) {
    w[0] = v.x;
    w[1] = v.y;
    w[2] = v.z;
    w[3] = v.w;
  }
  __device__ static __forceinline__ Word neg_inf_w() { return kNegInf2; }
  __device__ static __forceinline__ Word neg_big_w() { return kNegBig2; }
  __device__ static __forceinline__ Vec fill_neg_big() { return make_uint4(kNegBig2, kNegBig2, kNegBig2, kNegBig2); }
  // nonzero where `oth` is -inf and `tgt` is not (a KL support violation)
  __device__ static __forceinline__ uint32_t viol(Word tgt, Word oth) {
    return __vcmpeq2(oth, kNegInf2) & ~__vcmpeq2(tgt, kNegInf2);
  }
  using GSame = GF16;
};
// fp32 logits in the single-read kernels: an 8-element vector is 32 bytes (two
// 16-byte loads), a word is a pair of floats; x - m is one rounded fp32
// subtraction, as in the streaming kernels.
struct InF32 {
  static constexpr int kSize = 4;
  using Word = float2;
  struct Vec {
    uint4 a, b;
  };
  __device__ static __forceinline__ Vec ld(const unsigned char* p) {
    return {*reinterpret_cast<const uint4*>(p), *reinterpret_cast<const uint4*>(p + 16)};
  }
  __device__ static __forceinline__ void words(const Vec& v, Word (&w)[4]) {
    w[0] = make_float2(__uint_as_float(v.a.x), __uint_as_float(v.a.y));
    w[1] = make_float2(__uint_as_float(v.a.z), __uint_as_float(v.a.w));
    w[2] = make_float2(__uint_as_float(v.b.x), __uint_as_float(v.b.y));
    w[3] = make_float2(__uint_as_float(v.b.z), __uint_as_float(v.b.w));
  }
  __device__ static __forceinline__ Word neg_inf_w() {
    return make_float2(__int_as_float(0xff800000), __int_as_float(0xff800000));
  }
  // -2^100: keeps (x - m) log2 e finite for a row max up to 2^126
  __device__ static __forceinline__ Word neg_big_w() { return make_float2(-0x1p100f, -0x1p100f); }
  __device__ static __forceinline__ Vec fill_neg_big() {
    const uint32_t b = __float_as_uint(-0x1p100f);
    return {make_uint4(b, b, b, b), make_uint4(b, b, b, b)};
  }
  __device__ static __forceinline__ Word max_nan(Word a, Word b) {
    float x, y;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(x) : "f"(a.x), "f"(b.x));
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(y) : "f"(a.y), "f"(b.y));
    return make_float2(x, y);
  }
  // the larger of each pair (a NaN loses, as in the packed 16-bit max)
  __device__ static __forceinline__ Word max2(Word a, Word b) { return make_float2(fmaxf(a.x, b.x), fmaxf(a.y, b.y)); }
  __device__ static __forceinline__ float2 unpack(Word w) { return w; }
  __device__ static __forceinline__ float2 sub(Word w, float2 nm) { return __fadd2_rn(w, nm); }
  __device__ static __forceinline__ uint32_t viol(Word tgt, Word oth) {
    const float ni = __int_as_float(0xff800000);
    return ((oth.x == ni) & (tgt.x != ni)) | ((oth.y == ni) & (tgt.y != ni));
  }
  using GSame = GF32;
};

__device__ __forceinline__ float2 f2(float a) { return make_float2(a, a); }
__device__ __forceinline__ float2 neg(float2 a) { return make_float2(-a.x, -a.y); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 ex2_2(float2 a) { return make_float2(ex2(a.x), ex2(a.y)); }
__device__ __forceinline__ float2 lg2_2(float2 a) { return make_float2(lg2(a.x), lg2(a.y)); }

}  // namespace vpd
