// vpd_device.cuh -- device-side building blocks shared by the libvpd kernels:
// exact upcasts of fp32/bf16/fp16 logits, 16-byte vector loads, the hardware
// base-2 exponential and logarithm, the (max, sum-exp) merge used for
// statistics, and warp/block reductions.
//
// The statistics merge follows "Add vocabulary-parallel logprobs, entropy and KL
// ops" (DeepSpeed pull request #8791), section "How": a MAX reduction of the
// per-part max and a SUM reduction of the per-part sum-exp rescaled to it, where
// a part with no finite entry contributes (-inf, 0), and the max and the
// log-sum-exp stay separate.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace vpd {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kThreads = 512;  // threads per CTA of the streaming kernels

enum Dtype : int { kF32 = 0, kBF16 = 1, kF16 = 2 };

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }
__device__ __forceinline__ float pos_inf() { return __int_as_float(0x7f800000); }
__device__ __forceinline__ float qnan() { return __int_as_float(0x7fffffff); }

// Hardware approximations (MUFU): 2^x and log2(x), subnormals flushed.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// e^x for an argument that is already a small difference (x <= 0 in use).
__device__ __forceinline__ float expd(float x) { return ex2(x * kLog2e); }

// ---------------------------------------------------------------------------
// Element types. `bits` is the storage word; unpack() upcasts exactly.
// ---------------------------------------------------------------------------
struct F32 {
  static constexpr int kDtype = kF32;
  static constexpr int kSize = 4;
  static constexpr int kVec = 4;  // elements per 16-byte vector
  __device__ static __forceinline__ float load(const void* p, int64_t j) {
    return __ldg(reinterpret_cast<const float*>(p) + j);
  }
  __device__ static __forceinline__ void unpack(const uint4& v, float (&x)[kVec]) {
    x[0] = __uint_as_float(v.x);
    x[1] = __uint_as_float(v.y);
    x[2] = __uint_as_float(v.z);
    x[3] = __uint_as_float(v.w);
  }
};

struct BF16 {
  static constexpr int kDtype = kBF16;
  static constexpr int kSize = 2;
  static constexpr int kVec = 8;
  __device__ static __forceinline__ float load(const void* p, int64_t j) {
    unsigned short b = __ldg(reinterpret_cast<const unsigned short*>(p) + j);
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
  }
  __device__ static __forceinline__ void unpack(const uint4& v, float (&x)[kVec]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
};

struct F16 {
  static constexpr int kDtype = kF16;
  static constexpr int kSize = 2;
  static constexpr int kVec = 8;
  __device__ static __forceinline__ float h2f(unsigned short b) {
    float f;
    asm("{ .reg .f16 h; mov.b16 h, %1; cvt.f32.f16 %0, h; }" : "=f"(f) : "h"(b));
    return f;
  }
  __device__ static __forceinline__ float load(const void* p, int64_t j) {
    return h2f(__ldg(reinterpret_cast<const unsigned short*>(p) + j));
  }
  __device__ static __forceinline__ void unpack(const uint4& v, float (&x)[kVec]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = h2f(static_cast<unsigned short>(w[i] & 0xffffu));
      x[2 * i + 1] = h2f(static_cast<unsigned short>(w[i] >> 16));
    }
  }
};

// Gradient storage: float32 as is, bf16/fp16 rounded to nearest even.
struct GF32 {
  static constexpr int kSize = 4;
  __device__ static __forceinline__ void store(void* p, int64_t j, float v) {
    reinterpret_cast<float*>(p)[j] = v;
  }
};
struct GBF16 {
  static constexpr int kSize = 2;
  __device__ static __forceinline__ unsigned short cvt(float v) {
    unsigned short b;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(b) : "f"(v));
    return b;
  }
  __device__ static __forceinline__ void store(void* p, int64_t j, float v) {
    reinterpret_cast<unsigned short*>(p)[j] = cvt(v);
  }
};
struct GF16 {
  static constexpr int kSize = 2;
  __device__ static __forceinline__ unsigned short cvt(float v) {
    unsigned short b;
    asm("{ .reg .f16 h; cvt.rn.f16.f32 h, %1; mov.b16 %0, h; }" : "=h"(b) : "f"(v));
    return b;
  }
  __device__ static __forceinline__ void store(void* p, int64_t j, float v) {
    reinterpret_cast<unsigned short*>(p)[j] = cvt(v);
  }
};

// Store n = 4 or 8 consecutive gradient values starting at element j. When
// `vec` is true the destination is 16-byte aligned at j.
template <class G, int N>
__device__ __forceinline__ void store_grads(void* p, int64_t j, const float (&v)[N], bool vec) {
  if constexpr (G::kSize == 4) {
    float* d = reinterpret_cast<float*>(p) + j;
    if (vec) {
#pragma unroll
      for (int i = 0; i < N; i += 4)
        *reinterpret_cast<float4*>(d + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
    } else {
#pragma unroll
      for (int i = 0; i < N; ++i) d[i] = v[i];
    }
  } else {
    unsigned short* d = reinterpret_cast<unsigned short*>(p) + j;
    if (vec && N % 8 == 0) {
#pragma unroll
      for (int i = 0; i < N; i += 8) {
        uint4 w;
        w.x = G::cvt(v[i]) | (static_cast<uint32_t>(G::cvt(v[i + 1])) << 16);
        w.y = G::cvt(v[i + 2]) | (static_cast<uint32_t>(G::cvt(v[i + 3])) << 16);
        w.z = G::cvt(v[i + 4]) | (static_cast<uint32_t>(G::cvt(v[i + 5])) << 16);
        w.w = G::cvt(v[i + 6]) | (static_cast<uint32_t>(G::cvt(v[i + 7])) << 16);
        *reinterpret_cast<uint4*>(d + i) = w;
      }
    } else if (vec) {  // N == 4: 8-byte store
      uint2 w;
      w.x = G::cvt(v[0]) | (static_cast<uint32_t>(G::cvt(v[1])) << 16);
      w.y = G::cvt(v[2]) | (static_cast<uint32_t>(G::cvt(v[3])) << 16);
      *reinterpret_cast<uint2*>(d) = w;
    } else {
#pragma unroll
      for (int i = 0; i < N; ++i) d[i] = G::cvt(v[i]);
    }
  }
}

__device__ __forceinline__ uint4 ldg16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// ---------------------------------------------------------------------------
// Row addressing: element offset of row r in a (possibly batched) view.
// ---------------------------------------------------------------------------
struct RowMap {
  int64_t row_stride;
  int64_t rows_per_batch;
  int64_t batch_stride;
  int64_t first = 0;  // row r of this map is row first + r of the caller's view
  __host__ __device__ __forceinline__ int64_t offset(int64_t r) const {
    r += first;
    if (rows_per_batch > 0)
      return (r / rows_per_batch) * batch_stride + (r % rows_per_batch) * row_stride;
    return r * row_stride;
  }
};

// ---------------------------------------------------------------------------
// (max, sum-exp) statistics. z is relative to m; m = -inf means no finite entry
// yet (z is then 0, or NaN if a NaN was seen). A NaN anywhere makes z NaN and
// +inf makes m = +inf; either marks the row as outside the contract.
// ---------------------------------------------------------------------------
struct Stat {
  float m;
  float z;
};

__device__ __forceinline__ Stat stat_init() { return {neg_inf(), 0.f}; }

// Reference point for exponentials: the max, or 0 while nothing finite is seen
// (so that -inf entries give 0 and NaN entries give NaN).
__device__ __forceinline__ float stat_ref(float m) { return m == neg_inf() ? 0.f : m; }

// e^x to full fp32 accuracy, for the few rescalings of partial sums (the
// hardware approximation's error would compound over a merge tree).
__device__ __forceinline__ float exp_acc(float x) { return expf(x); }

// Merge: MAX of the maxima, SUM of the sums rescaled to it.
__device__ __forceinline__ Stat stat_merge(Stat a, Stat b) {
  float m = fmaxf(a.m, b.m);
  float r = stat_ref(m);
  return {m, a.z * exp_acc(a.m - r) + b.z * exp_acc(b.m - r)};
}

// Add a group of N values (one 16-byte vector) to a running statistic.
template <int N>
__device__ __forceinline__ void stat_add(Stat& st, const float (&x)[N]) {
  float mx = x[0];
#pragma unroll
  for (int i = 1; i < N; ++i) mx = fmaxf(mx, x[i]);
  if (mx > st.m) {
    st.z *= exp_acc(st.m - mx);
    st.m = mx;
  }
  const float r = stat_ref(st.m);
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < N; ++i) acc += expd(x[i] - r);
  st.z += acc;
}

__device__ __forceinline__ void stat_add1(Stat& st, float x) {
  float one[1] = {x};
  stat_add<1>(st, one);
}

// True when the merged statistic marks a NaN or +inf input.
__device__ __forceinline__ bool stat_bad(Stat st) { return isnan(st.z) || st.m == pos_inf(); }

// ---------------------------------------------------------------------------
// Reductions.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ int warp_or(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v |= __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ Stat warp_stat(Stat s) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Stat t{__shfl_xor_sync(0xffffffffu, s.m, o), __shfl_xor_sync(0xffffffffu, s.z, o)};
    s = stat_merge(s, t);
  }
  return s;
}

// Block-wide reduction of K floats (sum) through shared memory. Every thread
// gets the totals. `scratch` holds at least K * 32 floats; the call begins and
// ends with a barrier so scratch can be reused right away.
template <int K>
__device__ __forceinline__ void block_sum(float (&v)[K], float* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int k = 0; k < K; ++k) v[k] = warp_sum(v[k]);
  __syncthreads();
  if (lane == 0) {
#pragma unroll
    for (int k = 0; k < K; ++k) scratch[k * 32 + warp] = v[k];
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < K; ++k) {
    float a = lane < nw ? scratch[k * 32 + lane] : 0.f;
    v[k] = warp_sum(a);
  }
  __syncthreads();
}

// Block-wide merge of K statistics; every thread gets the merged values.
// `scratch` holds at least K * 64 floats.
template <int K>
__device__ __forceinline__ void block_stat(Stat (&s)[K], float* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int k = 0; k < K; ++k) s[k] = warp_stat(s[k]);
  __syncthreads();
  if (lane == 0) {
#pragma unroll
    for (int k = 0; k < K; ++k) {
      scratch[k * 64 + warp] = s[k].m;
      scratch[k * 64 + 32 + warp] = s[k].z;
    }
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < K; ++k) {
    Stat a = lane < nw ? Stat{scratch[k * 64 + lane], scratch[k * 64 + 32 + lane]} : stat_init();
    s[k] = warp_stat(a);
  }
  __syncthreads();
}

__device__ __forceinline__ int block_or(int v, int* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_or(v);
  __syncthreads();
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  int a = lane < nw ? scratch[lane] : 0;
  v = warp_or(a);
  __syncthreads();
  return v;
}

}  // namespace vpd
