// vpd_fused.cuh -- device code of the single-read fused JSD forward+backward
// on thread-block clusters (instantiated per input dtype in
// vpd_fused_bf16.cu / vpd_fused_f16.cu; host dispatch in vpd_fused.cu).
//
// Source: DeepSpeed pull request #8958, "[VocabTP] Add vocabulary-parallel
// generalized JSD with Triton kernels": the op (section Changes: paired softmax
// statistics, the two KL-to-mixture expectations reduced together, a backward
// that recomputes P_s, P_t and M from the inputs; beta = 0 / 1 as explicit KL
// branches) and the reason the pages need two input passes (section Scope and
// limitations: the mixture is nonlinear in the normalised probabilities, so the
// statistics must be global before the divergence).
//
// Design. One cluster of C CTAs (C in {1, 2, 4, 8, 16}) owns one token row at a
// time; CTA c holds columns [c W, (c + 1) W) of both inputs, every thread R
// 16-byte vectors of each, in registers. The row pair is read from HBM once:
//   1. TMA bulk copies (cp.async.bulk, mbarrier completion) stage the CTA's
//      slice of the next rows in shared memory (two stages) while the current
//      row is computed from registers;
//   2. statistics: NaN-propagating max of the raw 16-bit pairs (a NaN or +inf
//      row is outside the contract, and so is a finite row max above 2^126
//      here), then per-thread sum-exp relative to the thread max, merged over
//      the CTA and then over the cluster: the MAX / SUM merge of per-shard
//      statistics, with the CTA slices as shards. These are computed straight
//      from the next row's shared-memory stage while the current row's sums
//      are in flight;
//   3. pass C: log2 p, log2 q, p, q and log2 M, M = (1 - beta) p + beta q; the
//      two expectations A = KL(P_t || M) and B = KL(P_s || M) are reduced
//      together over the CTA and the cluster;
//   4. pass D: dS = g (1 - beta) p (ln p - ln M - B), dT = g beta q (ln q - ln M
//      - A), stored straight from registers with 16-byte stores.
// Two register budgets: the "kept" variant (256 threads, up to 255 registers)
// keeps p, q, log2 p - log2 M and log2 q - log2 M in registers after pass C,
// so pass D is a few multiply-adds per element; the "recompute" variant (480
// threads, up to 128 registers) keeps only log2 M and recomputes p and q.
// When the raw -inf would reach a product, it is clamped first to a finite
// floor so that no 0 * inf forms.
// Arithmetic is fp32 (packed fp32x2 where it pairs up) in base-2 logarithms,
// so the hardware ex2 / lg2 apply without rescaling; sums are converted to
// nats once per row.
//
// Every wait on an mbarrier is bounded: when it gives up, the kernel records
// an error in its device error word, leaves its row loop (every CTA of the
// cluster does, since each then waits in vain for the others), waits
// (bounded) for its own copies in flight, and returns.
#pragma once

#include <cuda_runtime.h>

#include "vpd_internal.h"

namespace vpd {
namespace fused {

constexpr int kStages = 2;                  // shared-memory stages per CTA
constexpr float kTiny = 1e-37f;             // keeps M > 0 so log2 M stays finite
constexpr float kMaxLogit = 8.5070592e37f;  // 2^126: a larger finite row max is out of contract
constexpr int kMaxCluster = 16;
constexpr int kKeepT = 256;     // threads per CTA of the kept-value variant (up to 255 registers each)
constexpr int kKeepMaxR = 5;
constexpr int kRecomputeT = 480;  // threads per CTA of the recompute variant (up to 128 registers each)

enum Mode : int { kInterior = 0, kForwardKL = 1, kReverseKL = 2 };

// Set by a kernel of this translation unit whose bounded wait gave up (each
// translation unit that includes this header has its own word).
static __device__ int g_fused_error = 0;

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* mb, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(mb)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* mb, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(mb)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // a wait gives up after two seconds
constexpr uint32_t kSuspendHintNs = 20000;        // try_wait may sleep this long per round

// One try on an mbarrier phase (CTA-scope acquire); may suspend the thread for
// up to the hint while the phase is incomplete.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* mb, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(mb)), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}
// Wait for a phase, giving up after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t* mb, uint32_t parity) {
  if (mbar_try_wait(mb, parity)) return true;
  const uint64_t t0 = global_ns();
  while (global_ns() - t0 < kWaitLimitNs)
    if (mbar_try_wait(mb, parity)) return true;
  return false;
}
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* mb) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(mb))
      : "memory");
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::
          : "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_index() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// Load a float from the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ float ld_cluster(const float* p, uint32_t rank) {
  uint32_t remote;
  float v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(p)), "r"(rank));
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}
__device__ __forceinline__ uint4 ld_shared16(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_addr(p)));
  return v;
}
__device__ __forceinline__ void st_global16(void* p, uint4 v) {
  asm volatile("st.global.L1::no_allocate.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// ---------------------------------------------------------------------------
// 16-bit input formats: pairs of values packed in one 32-bit word.
// ---------------------------------------------------------------------------
// -inf is clamped to a finite floor (twice, packed) so that every log2 p_j
// computed later stays finite: (x - m) log2 e cannot overflow while the row
// max is at most 2^126 (larger rows are out of contract in this kernel).
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

// Gradient formats for 8 values (one 16-byte input vector).
template <class G>
struct Out;
template <>
struct Out<GBF16> {
  static constexpr int kSize = 2;
  __device__ static __forceinline__ uint32_t pack(float2 v) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(v.y), "f"(v.x));
    return d;
  }
  __device__ static __forceinline__ void store8(char* p, const float2 (&v)[4]) {
    st_global16(p, make_uint4(pack(v[0]), pack(v[1]), pack(v[2]), pack(v[3])));
  }
};
template <>
struct Out<GF16> {
  static constexpr int kSize = 2;
  __device__ static __forceinline__ uint32_t pack(float2 v) {
    uint32_t d;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(v.y), "f"(v.x));
    return d;
  }
  __device__ static __forceinline__ void store8(char* p, const float2 (&v)[4]) {
    st_global16(p, make_uint4(pack(v[0]), pack(v[1]), pack(v[2]), pack(v[3])));
  }
};
template <>
struct Out<GF32> {
  static constexpr int kSize = 4;
  __device__ static __forceinline__ void store8(char* p, const float2 (&v)[4]) {
    st_global16(p, make_uint4(__float_as_uint(v[0].x), __float_as_uint(v[0].y), __float_as_uint(v[1].x),
                              __float_as_uint(v[1].y)));
    st_global16(p + 16, make_uint4(__float_as_uint(v[2].x), __float_as_uint(v[2].y), __float_as_uint(v[3].x),
                                   __float_as_uint(v[3].y)));
  }
};

__device__ __forceinline__ float2 f2(float a) { return make_float2(a, a); }
// A copy the compiler cannot see through: values derived from it in one pass
// are not reused in another, so the passes recompute from the 16-bit inputs
// instead of keeping fp32 copies alive in registers.
__device__ __forceinline__ float2 opaque(float2 a) {
  float2 r;
  asm volatile("mov.b32 %0, %2;\n\tmov.b32 %1, %3;" : "=f"(r.x), "=f"(r.y) : "f"(a.x), "f"(a.y));
  return r;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 ex2_2(float2 a) { return make_float2(ex2(a.x), ex2(a.y)); }
__device__ __forceinline__ float2 lg2_2(float2 a) { return make_float2(lg2(a.x), lg2(a.y)); }

// ---------------------------------------------------------------------------
// Cluster reductions by push. Each CTA reduces its partial over its warps
// (shuffles + shared memory), then one lane per peer sends it with st.async
// into that peer's slot for this CTA; the bytes complete on the peer's
// mbarrier. A receiver arms its own mbarrier for C partials, waits on it and
// merges the C slots from its own shared memory. There is no cluster-wide
// barrier and no fence on the gradient stores in flight. Slots and mbarriers
// are double-buffered by row parity: a CTA cannot run two rows ahead of a
// peer, since it needs that peer's partial of every row to proceed.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t map_rank(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
__device__ __forceinline__ void push16(uint32_t remote, float a, float b, float c, float d, uint32_t remote_bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(remote),
      "f"(a), "f"(b), "f"(c), "f"(d), "r"(remote_bar)
      : "memory");
}
// One try with cluster-scope acquire: the partials arrive from other CTAs.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* mb, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(mb)), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* mb, uint32_t parity) {
  if (mbar_try_wait_cluster(mb, parity)) return true;
  const uint64_t t0 = global_ns();
  while (global_ns() - t0 < kWaitLimitNs)
    if (mbar_try_wait_cluster(mb, parity)) return true;
  return false;
}

struct Pair {  // statistics of both inputs and their out-of-contract flags
  float ms, zs, mt, zt, bad_s, bad_t;
};
struct Sums {  // A, B and the support-violation flag of the KL branches
  float a, b, viol;
};

__device__ __forceinline__ float warp_max_all(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum_all(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Merge the statistics held by the 32 lanes of a warp: MAX of the maxima,
// then each lane's sum rescaled once to it (accurate exp) and summed.
__device__ __forceinline__ Pair warp_merge(const Pair& x) {
  const float ms = warp_max_all(x.ms), mt = warp_max_all(x.mt);
  const float zs = warp_sum_all(x.zs * exp_acc(x.ms - stat_ref(ms)));
  const float zt = warp_sum_all(x.zt * exp_acc(x.mt - stat_ref(mt)));
  return {ms, zs, mt, zt, warp_max_all(x.bad_s), warp_max_all(x.bad_t)};
}
__device__ __forceinline__ Sums warp_merge(const Sums& x) {
  return {warp_sum_all(x.a), warp_sum_all(x.b), warp_max_all(x.viol)};
}

__device__ __forceinline__ Pair pair_identity() { return {neg_inf(), 0.f, neg_inf(), 0.f, 0.f, 0.f}; }
__device__ __forceinline__ Sums sums_identity() { return {0.f, 0.f, 0.f}; }
__device__ __forceinline__ void put(float* p, const Pair& v) {
  p[0] = v.ms, p[1] = v.zs, p[2] = v.mt, p[3] = v.zt, p[4] = v.bad_s, p[5] = v.bad_t;
}
__device__ __forceinline__ void put(float* p, const Sums& v) { p[0] = v.a, p[1] = v.b, p[2] = v.viol; }
__device__ __forceinline__ void get(const float* p, Pair& v) { v = {p[0], p[1], p[2], p[3], p[4], p[5]}; }
__device__ __forceinline__ void get(const float* p, Sums& v) { v = {p[0], p[1], p[2]}; }
__device__ __forceinline__ void identity(Pair& v) { v = pair_identity(); }
__device__ __forceinline__ void identity(Sums& v) { v = sums_identity(); }
template <class V> struct SlotWords;
template <> struct SlotWords<Pair> { static constexpr int kW = 8; };
template <> struct SlotWords<Sums> { static constexpr int kW = 4; };
__device__ __forceinline__ void push(uint32_t dst, const Pair& v, uint32_t bar) {
  push16(dst, v.ms, v.zs, v.mt, v.zt, bar);
  push16(dst + 16, v.bad_s, v.bad_t, 0.f, 0.f, bar);
}
__device__ __forceinline__ void push(uint32_t dst, const Sums& v, uint32_t bar) {
  push16(dst, v.a, v.b, v.viol, 0.f, bar);
}

// Reduce v over this CTA of T threads and push the result to slot `crank` of
// every CTA of the cluster.
template <int T, class V>
__device__ __forceinline__ void reduce_and_push(V v, float* warp_slots, float* slots, uint64_t* bar,
                                                uint32_t crank, uint32_t csize) {
  constexpr int kW = SlotWords<V>::kW;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_merge(v);
  if (lane == 0) put(warp_slots + warp * kW, v);
  __syncthreads();
  if (warp == 0) {
    V w;
    if (lane < T / 32) get(warp_slots + lane * kW, w);
    else identity(w);
    w = warp_merge(w);
    if (lane < static_cast<int>(csize))
      push(map_rank(smem_addr(slots + crank * kW), lane), w, map_rank(smem_addr(bar), lane));
  }
}

// Arm this CTA's mbarrier for the C partials of one row; one thread waits
// (bounded) while the others sleep in the CTA barrier, then every thread
// takes the phase with cluster-scope acquire and merges the slots. `ok`
// becomes false for every thread if the wait gave up.
template <class V>
__device__ __forceinline__ V collect(const float* slots, uint64_t* bar, uint32_t parity, uint32_t csize,
                                     bool& ok) {
  constexpr int kW = SlotWords<V>::kW;
  bool mine = true;
  if (threadIdx.x == 0) {
    mbar_expect_tx(bar, csize * kW * 4u);
    mine = mbar_wait_cluster(bar, parity);
  }
  ok = __syncthreads_and(mine) && ok;
  if (ok && threadIdx.x != 0) mbar_try_wait_cluster(bar, parity);
  const int lane = threadIdx.x & 31;
  V c;
  if (lane < static_cast<int>(csize)) get(slots + lane * kW, c);
  else identity(c);
  return warp_merge(c);
}

struct FusedArgs {
  const char* s;
  const char* t;
  RowMap ms, mt;
  int64_t rows;
  int64_t vocab;
  int W;  // slice width per CTA (elements, multiple of 8)
  float beta;
  const float* grad_loss;
  float* loss;
  float* saved;
  Grad ds, dt;
  int64_t withhold_row;  // test hook: CTA 0 of the owning cluster never copies this row (-1: none)
};

// Shared memory: [kStages][2 inputs][W] 16-bit elements, then this tail.
template <int T>
struct Tail {
  uint64_t tma_bar[kStages];
  uint64_t stat_bar[2];
  uint64_t sum_bar[2];
  float stat_warp[T / 32 * SlotWords<Pair>::kW];
  float sum_warp[T / 32 * SlotWords<Sums>::kW];
  __align__(16) float stat_slot[2][kMaxCluster * SlotWords<Pair>::kW];
  __align__(16) float sum_slot[2][kMaxCluster * SlotWords<Sums>::kW];
};

// Statistics partial of one row read straight from its shared-memory stage:
// NaN-propagating maxima of the raw pairs, then the sum of 2^((x - m) log2 e)
// relative to this thread's max (a -inf entry contributes 2^-inf = 0; the
// rounding of m log2 e is common to every term of the row and cancels in the
// normalisation).
template <class In, int T, int R>
__device__ __forceinline__ Pair stage_stats(const unsigned char* sb, int W, int len) {
  const int tid = threadIdx.x;
  uint32_t mxs = In::kNegInf2, mxt = In::kNegInf2;
#pragma unroll
  for (int k = 0; k < R; ++k) {
    const int e0 = (k * T + tid) * 8;
    if (e0 < len) {
      const uint4 u = ld_shared16(sb + e0 * 2);
      const uint4 v = ld_shared16(sb + static_cast<size_t>(W) * 2 + e0 * 2);
      mxs = In::max_nan(In::max_nan(mxs, u.x), In::max_nan(u.y, In::max_nan(u.z, u.w)));
      mxt = In::max_nan(In::max_nan(mxt, v.x), In::max_nan(v.y, In::max_nan(v.z, v.w)));
    }
  }
  const float2 ms2 = In::unpack(mxs), mt2 = In::unpack(mxt);
  const float m_s = fmaxf(ms2.x, ms2.y), m_t = fmaxf(mt2.x, mt2.y);
  const bool bad_s = isnan(ms2.x) || isnan(ms2.y) || m_s > kMaxLogit;
  const bool bad_t = isnan(mt2.x) || isnan(mt2.y) || m_t > kMaxLogit;
  const float2 l2e2 = f2(kLog2e), ns2 = f2(-stat_ref(m_s)), nt2 = f2(-stat_ref(m_t));
  float2 zs2 = f2(0.f), zt2 = f2(0.f);
#pragma unroll
  for (int k = 0; k < R; ++k) {
    const int e0 = (k * T + tid) * 8;
    if (e0 < len) {
      const uint4 u = ld_shared16(sb + e0 * 2);
      const uint4 v = ld_shared16(sb + static_cast<size_t>(W) * 2 + e0 * 2);
      const uint32_t us[4] = {u.x, u.y, u.z, u.w}, vs[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        // x - m is exact; a -inf entry gives 2^-inf = 0
        zs2 = add2(zs2, ex2_2(mul2(In::sub(us[w], ns2), l2e2)));
        zt2 = add2(zt2, ex2_2(mul2(In::sub(vs[w], nt2), l2e2)));
      }
    }
  }
  return {m_s, zs2.x + zs2.y, m_t, zt2.x + zt2.y, bad_s ? 1.f : 0.f, bad_t ? 1.f : 0.f};
}

// Copy one row's stage into registers with -inf clamped to the floor; flags a
// KL support violation (the target finite where the other side is -inf).
template <class In, int T, int R, int MODE>
__device__ __forceinline__ void stage_to_regs(const unsigned char* sb, int W, int len, uint32_t (&xs)[R][4],
                                              uint32_t (&xt)[R][4], uint32_t& viol) {
  const int tid = threadIdx.x;
  viol = 0;
#pragma unroll
  for (int k = 0; k < R; ++k) {
    const int e0 = (k * T + tid) * 8;
    if (e0 < len) {
      const uint4 u = ld_shared16(sb + e0 * 2);
      const uint4 v = ld_shared16(sb + static_cast<size_t>(W) * 2 + e0 * 2);
      const uint32_t us[4] = {u.x, u.y, u.z, u.w}, vs[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        if (MODE != kInterior) {
          const uint32_t tgt = MODE == kForwardKL ? vs[w] : us[w];
          const uint32_t oth = MODE == kForwardKL ? us[w] : vs[w];
          viol |= __vcmpeq2(oth, In::kNegInf2) & ~__vcmpeq2(tgt, In::kNegInf2);
        }
        xs[k][w] = In::max2(us[w], In::kNegBig2);
        xt[k][w] = In::max2(vs[w], In::kNegBig2);
      }
    } else {
#pragma unroll
      for (int w = 0; w < 4; ++w) xs[k][w] = xt[k][w] = In::kNegBig2;
    }
  }
}

// log2 of the probabilities of one packed pair: (x - m) log2 e - K.
template <class In>
__device__ __forceinline__ float2 lam(uint32_t w, float2 nm, float2 l2e2, float2 nK) {
  return fma2(In::sub(w, nm), l2e2, nK);
}

template <class In, class G, int T, int R, int MODE, bool KEEP>
__global__ void __launch_bounds__(T, 1) k_jsd_fused(FusedArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int W = a.W;
  unsigned char* stage_base = smem;
  Tail<T>* tail = reinterpret_cast<Tail<T>*>(smem + static_cast<size_t>(kStages) * 2 * W * 2);
  auto stage_ptr = [&](int st) { return stage_base + static_cast<size_t>(st) * 2 * W * 2; };

  const uint32_t crank = cluster_rank(), csize = cluster_size();
  const int64_t q = cluster_index(), Q = cluster_count();
  const int tid = threadIdx.x;
  const int64_t col0 = static_cast<int64_t>(crank) * W;
  const int64_t rest = a.vocab - col0;
  const int len = rest <= 0 ? 0 : (rest < W ? static_cast<int>(rest) : W);
  const uint32_t bytes = static_cast<uint32_t>(len) * 2u;

  // The failure-path test hook: this CTA withholds the copy of one row, so
  // its bounded wait on that stage expires.
  auto withheld = [&](int64_t r) { return r == a.withhold_row && crank == 0; };
  auto issue = [&](int64_t r, int st) {  // one thread: both inputs' slices of row r into stage st
    if (withheld(r)) return;
    unsigned char* dst = stage_ptr(st);
    mbar_expect_tx(&tail->tma_bar[st], 2 * bytes);
    bulk_load(dst, a.s + (a.ms.offset(r) + col0) * 2, bytes, &tail->tma_bar[st]);
    bulk_load(dst + static_cast<size_t>(W) * 2, a.t + (a.mt.offset(r) + col0) * 2, bytes, &tail->tma_bar[st]);
  };

  if (tid == 0) {
    for (int st = 0; st < kStages; ++st) mbar_init(&tail->tma_bar[st], 1);
    for (int p = 0; p < 2; ++p) {
      mbar_init(&tail->stat_bar[p], 1);
      mbar_init(&tail->sum_bar[p], 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  uint32_t pending = 0;                  // bit st: a copy into stage st is in flight
  uint32_t tma_done[kStages] = {0, 0};   // completed waits per stage
  if (tid == 0 && bytes) {
    for (int st = 0; st < kStages; ++st)
      if (q + st * Q < a.rows) issue(q + st * Q, st);
  }
  if (bytes)
    for (int st = 0; st < kStages; ++st)
      if (q + st * Q < a.rows && !withheld(q + st * Q)) pending |= 1u << st;
  cluster_sync();  // every CTA's mbarriers are initialised before any push

  bool ok = true;
  auto wait_stage = [&](int st) {  // one thread waits; the others sleep in the barrier
    if (!bytes) return;
    bool mine = true;
    if (tid == 0) mine = mbar_wait(&tail->tma_bar[st], tma_done[st] & 1u);
    ok = __syncthreads_and(mine) && ok;
    if (ok && tid != 0) mbar_try_wait(&tail->tma_bar[st], tma_done[st] & 1u);
    ++tma_done[st];
    pending &= ~(1u << st);
  };

  const float beta = a.beta;
  const float2 ws2 = f2(1.f - beta), wt2 = f2(beta), tiny2 = f2(kTiny), l2e2 = f2(kLog2e), neg2 = f2(-1.f);
  uint32_t xs[R][4], xt[R][4];
  uint32_t viol = 0;

  // Row 0 of this cluster: statistics partial straight from its stage, then registers.
  if (q < a.rows) {
    wait_stage(0);
    reduce_and_push<T, Pair>(stage_stats<In, T, R>(stage_ptr(0), W, len), tail->stat_warp,
                                tail->stat_slot[0], &tail->stat_bar[0], crank, csize);
    stage_to_regs<In, T, R, MODE>(stage_ptr(0), W, len, xs, xt, viol);
    __syncthreads();
    const bool more = ok && q + kStages * Q < a.rows;  // no new copy after a failed wait
    if (tid == 0 && bytes && more) issue(q + kStages * Q, 0);
    if (bytes && more && !withheld(q + kStages * Q)) pending |= 1u;
  }

  int64_t i = 0;
  for (int64_t r = q; r < a.rows && ok; r += Q, ++i) {
    const int par = static_cast<int>(i & 1);
    const uint32_t ph = static_cast<uint32_t>((i >> 1) & 1);
    const bool has_next = r + Q < a.rows;
    const int nst = static_cast<int>((i + 1) % kStages);  // stage of the next row

    // (1) global statistics of row r
    const Pair g_st = collect<Pair>(tail->stat_slot[par], &tail->stat_bar[par], ph, csize, ok);
    const bool row_ok = g_st.bad_s == 0.f && g_st.bad_t == 0.f && g_st.ms != neg_inf() && g_st.mt != neg_inf();
    const float Ks = row_ok ? log2f(g_st.zs) : qnan();  // log2 Z
    const float Kt = row_ok ? log2f(g_st.zt) : qnan();
    const float2 nms2 = f2(-g_st.ms), nmt2 = f2(-g_st.mt), nKs2 = f2(-Ks), nKt2 = f2(-Kt);

    // (2) pass C of row r from registers, in log2 units. Kept: p, q and the two
    // log-ratios (interior: log2 p - log2 M, log2 q - log2 M; KL branches: the
    // log2 ratio target/other). Recompute: -log2 M only.
    float2 kp[KEEP ? R : 1][4], kq[KEEP ? R : 1][4], ku[KEEP ? R : 1][4], kv[KEEP && MODE == kInterior ? R : 1][4];
    float2 nlm_r[KEEP ? 1 : R][4];
    float2 acc_a = f2(0.f), acc_b = f2(0.f);
    if (row_ok) {
      const float2 nmsC = opaque(nms2), nmtC = opaque(nmt2);
#pragma unroll
      for (int k = 0; k < R; ++k)
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const float2 lp = lam<In>(xs[k][w], nmsC, l2e2, nKs2);
          const float2 lq = lam<In>(xt[k][w], nmtC, l2e2, nKt2);
          const float2 p = ex2_2(lp), qv = ex2_2(lq);
          if (MODE == kInterior) {
            const float2 nlm = mul2(lg2_2(fma2(ws2, p, fma2(wt2, qv, tiny2))), neg2);
            const float2 us = add2(lp, nlm), ut = add2(lq, nlm);
            acc_a = fma2(qv, ut, acc_a);
            acc_b = fma2(p, us, acc_b);
            if constexpr (KEEP) {
              kp[k][w] = p, kq[k][w] = qv, ku[k][w] = us, kv[k][w] = ut;
            } else {
              nlm_r[k][w] = nlm;
            }
          } else {
            // forward KL(q || p): d = log2 q - log2 p weighted by q; reverse: mirror
            const float2 d = MODE == kForwardKL ? add2(lq, mul2(lp, neg2)) : add2(lp, mul2(lq, neg2));
            acc_a = fma2(MODE == kForwardKL ? qv : p, d, acc_a);
            if constexpr (KEEP) kp[k][w] = p, kq[k][w] = qv, ku[k][w] = d;
          }
        }
    }
    reduce_and_push<T, Sums>({kLn2 * (acc_a.x + acc_a.y), kLn2 * (acc_b.x + acc_b.y), viol ? 1.f : 0.f},
                               tail->sum_warp, tail->sum_slot[par], &tail->sum_bar[par], crank, csize);

    // (3) statistics partial of the next row, straight from its stage, while
    // this row's sums travel
    if (has_next) {
      wait_stage(nst);
      reduce_and_push<T, Pair>(stage_stats<In, T, R>(stage_ptr(nst), W, len), tail->stat_warp,
                                  tail->stat_slot[par ^ 1], &tail->stat_bar[par ^ 1], crank, csize);
    }

    // (4) global sums of row r; the per-token value and saved statistics
    const Sums g_ab = collect<Sums>(tail->sum_slot[par], &tail->sum_bar[par], ph, csize, ok);
    float A = g_ab.a, B = g_ab.b, value;
    if (!row_ok) {
      value = qnan();
      A = B = qnan();
    } else if (MODE == kInterior) {
      value = beta * A + (1.f - beta) * B;
    } else {
      value = g_ab.viol != 0.f ? pos_inf() : A;
      A = MODE == kForwardKL ? value : 0.f;
      B = MODE == kForwardKL ? 0.f : value;
    }
    if (crank == 0 && tid == 0) {
      a.loss[r] = value;
      float* sv = a.saved + r * VPD_SAVED_PAIR;
      sv[0] = g_st.bad_s != 0.f ? qnan() : g_st.ms;
      sv[1] = g_st.bad_s != 0.f ? qnan() : (g_st.ms == neg_inf() ? neg_inf() : kLn2 * log2f(g_st.zs));
      sv[2] = g_st.bad_t != 0.f ? qnan() : g_st.mt;
      sv[3] = g_st.bad_t != 0.f ? qnan() : (g_st.mt == neg_inf() ? neg_inf() : kLn2 * log2f(g_st.zt));
      sv[4] = A;
      sv[5] = B;
    }

    // (5) pass D of row r: gradients, e.g. dS = p (g (1-beta) ln2 (log2 p - log2 M) - g (1-beta) B)
    const float gr = a.grad_loss ? __ldg(a.grad_loss + r) : 1.f;
    char* ds_row = a.ds.data ? a.ds.data + (r * a.ds.row_stride + col0) * Out<G>::kSize : nullptr;
    char* dt_row = a.dt.data ? a.dt.data + (r * a.dt.row_stride + col0) * Out<G>::kSize : nullptr;
    if (ds_row || dt_row) {
      const bool live = row_ok && isfinite(value);
      const float cs = MODE == kInterior ? gr * (1.f - beta) : gr;
      const float ct = MODE == kInterior ? gr * beta : gr;
      const float2 cs2 = f2(cs * kLn2), ct2 = f2(ct * kLn2);
      const float2 ncs2 = f2(-cs * (MODE == kInterior ? B : value));
      const float2 nct2 = f2(-ct * (MODE == kInterior ? A : value));
      const float2 g2 = f2(gr);
      const float2 nmsD = opaque(nms2), nmtD = opaque(nmt2);
#pragma unroll
      for (int k = 0; k < R; ++k) {
        const int e0 = (k * T + tid) * 8;
        if (e0 >= len) continue;
        float2 gs[4], gt[4];
        if (!live) {
#pragma unroll
          for (int w = 0; w < 4; ++w) gs[w] = gt[w] = f2(0.f);
        } else {
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            float2 p, qv, us, ut;
            if constexpr (KEEP) {
              p = kp[k][w], qv = kq[k][w], us = ku[k][w];
              ut = MODE == kInterior ? kv[k][w] : us;
            } else {
              const float2 lp = lam<In>(xs[k][w], nmsD, l2e2, nKs2);
              const float2 lq = lam<In>(xt[k][w], nmtD, l2e2, nKt2);
              p = ex2_2(lp), qv = ex2_2(lq);
              if (MODE == kInterior) {
                us = add2(lp, nlm_r[k][w]), ut = add2(lq, nlm_r[k][w]);
              } else {
                us = ut = MODE == kForwardKL ? add2(lq, mul2(lp, neg2)) : add2(lp, mul2(lq, neg2));
              }
            }
            if (MODE == kInterior) {
              gs[w] = mul2(p, fma2(cs2, us, ncs2));
              gt[w] = mul2(qv, fma2(ct2, ut, nct2));
            } else if (MODE == kForwardKL) {  // dS = g (p - q), dT = g q (ln q - ln p - KL)
              gs[w] = mul2(g2, add2(p, mul2(qv, neg2)));
              gt[w] = mul2(qv, fma2(ct2, ut, nct2));
            } else {  // dS = g p (ln p - ln q - KL), dT = g (q - p)
              gs[w] = mul2(p, fma2(cs2, us, ncs2));
              gt[w] = mul2(g2, add2(qv, mul2(p, neg2)));
            }
          }
        }
        if (ds_row) Out<G>::store8(ds_row + static_cast<int64_t>(e0) * Out<G>::kSize, gs);
        if (dt_row) Out<G>::store8(dt_row + static_cast<int64_t>(e0) * Out<G>::kSize, gt);
      }
    }

    // (6) the next row into registers; its stage is then free for the row
    // kStages further on
    if (has_next) {
      stage_to_regs<In, T, R, MODE>(stage_ptr(nst), W, len, xs, xt, viol);
      __syncthreads();
      const bool more = ok && r + (kStages + 1) * Q < a.rows;  // no new copy after a failed wait
      if (tid == 0 && bytes && more) issue(r + (kStages + 1) * Q, nst);
      if (bytes && more && !withheld(r + (kStages + 1) * Q)) pending |= 1u << nst;
    }
  }

  // Only after a wait gave up: copies still in flight must land before exit.
  for (int st = 0; st < kStages; ++st)
    if (pending & (1u << st)) mbar_wait(&tail->tma_bar[st], tma_done[st] & 1u);
  if (!ok && tid == 0) atomicExch(&g_fused_error, 1);
  cluster_sync();  // no CTA leaves while a peer may still push into it
}

// ---------------------------------------------------------------------------
// Host side (per input dtype): one configuration, one launch.
// ---------------------------------------------------------------------------
struct Config {
  int C, T, R, W;
  bool keep;
  size_t smem;
};

// Launches the configured kernel; cudaErrorNotSupported (nothing launched)
// when no cluster of that shape can be resident. `clusters_out` reports the
// number of resident clusters.
template <class In>
cudaError_t launch_typed(const FusedArgs& args, const Config& cfg, int mode, bool f32grad, cudaStream_t stream,
                         int* clusters_out);

template <class In, class G, int T, int R, int MODE, bool KEEP>
cudaError_t launch_one(const FusedArgs& args, const Config& cfg, cudaStream_t stream, int* clusters_out) {
  auto kern = k_jsd_fused<In, G, T, R, MODE, KEEP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(cfg.smem));
  if (e != cudaSuccess) return e;
  if (cfg.C > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return cudaErrorNotSupported;
    }
  }
  cudaLaunchConfig_t lc = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cfg.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  lc.blockDim = dim3(T, 1, 1);
  lc.dynamicSmemBytes = cfg.smem;
  lc.stream = stream;
  lc.attrs = attr;
  lc.numAttrs = 1;
  lc.gridDim = dim3(cfg.C, 1, 1);
  int clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&clusters, kern, &lc);
  if (e != cudaSuccess || clusters < 1) {
    cudaGetLastError();
    return cudaErrorNotSupported;
  }
  *clusters_out = clusters;
  const int64_t want = args.rows < clusters ? args.rows : clusters;
  lc.gridDim = dim3(static_cast<unsigned>(want * cfg.C), 1, 1);
  return cudaLaunchKernelEx(&lc, kern, args);
}

template <class In, class G, int MODE>
cudaError_t launch_r(const FusedArgs& args, const Config& cfg, cudaStream_t stream, int* clusters) {
  if (cfg.keep) {
    switch (cfg.R) {
      case 1: return launch_one<In, G, kKeepT, 1, MODE, true>(args, cfg, stream, clusters);
      case 2: return launch_one<In, G, kKeepT, 2, MODE, true>(args, cfg, stream, clusters);
      case 3: return launch_one<In, G, kKeepT, 3, MODE, true>(args, cfg, stream, clusters);
      case 4: return launch_one<In, G, kKeepT, 4, MODE, true>(args, cfg, stream, clusters);
      case 5: return launch_one<In, G, kKeepT, 5, MODE, true>(args, cfg, stream, clusters);
    }
  } else {
    switch (cfg.R) {
      case 1: return launch_one<In, G, kRecomputeT, 1, MODE, false>(args, cfg, stream, clusters);
      case 2: return launch_one<In, G, kRecomputeT, 2, MODE, false>(args, cfg, stream, clusters);
      case 3: return launch_one<In, G, kRecomputeT, 3, MODE, false>(args, cfg, stream, clusters);
      case 4: return launch_one<In, G, kRecomputeT, 4, MODE, false>(args, cfg, stream, clusters);
      case 5: return launch_one<In, G, kRecomputeT, 5, MODE, false>(args, cfg, stream, clusters);
    }
  }
  return cudaErrorNotSupported;
}

template <class In>
cudaError_t launch_typed(const FusedArgs& args, const Config& cfg, int mode, bool f32grad, cudaStream_t stream,
                         int* clusters) {
  using GIn = typename In::GSame;
  if (mode == kForwardKL)
    return f32grad ? launch_r<In, GF32, kForwardKL>(args, cfg, stream, clusters)
                   : launch_r<In, GIn, kForwardKL>(args, cfg, stream, clusters);
  if (mode == kReverseKL)
    return f32grad ? launch_r<In, GF32, kReverseKL>(args, cfg, stream, clusters)
                   : launch_r<In, GIn, kReverseKL>(args, cfg, stream, clusters);
  return f32grad ? launch_r<In, GF32, kInterior>(args, cfg, stream, clusters)
                 : launch_r<In, GIn, kInterior>(args, cfg, stream, clusters);
}

}  // namespace fused
}  // namespace vpd
