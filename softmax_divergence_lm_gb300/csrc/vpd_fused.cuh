// vpd_fused.cuh -- device code of the single-read fused JSD on thread-block
// clusters: the forward+backward kernel (k_jsd_fused) and, for calls that
// want no gradient, the forward-only kernel (k_jsd_fused_fwd, further below);
// instantiated per input dtype in vpd_fused_bf16.cu / vpd_fused_f16.cu /
// vpd_fused_f32.cu (fp32 vectors: 8 floats in 32 bytes), host dispatch in
// vpd_fused.cu.
//
// Source: DeepSpeed pull request #8958, "[VocabTP] Add vocabulary-parallel
// generalized JSD with Triton kernels": the op (section Changes: paired softmax
// statistics, the two KL-to-mixture expectations reduced together, a backward
// that recomputes P_s, P_t and M from the inputs; beta = 0 / 1 as explicit KL
// branches) and the reason the pages need two input passes (section Scope and
// limitations: the mixture is nonlinear in the normalised probabilities, so the
// statistics must be global before the divergence).
//
// Design. One cluster of C CTAs (C from 1 to 16, chosen on the host to cover
// the most SMs) owns one token row at a time; CTA c holds columns
// [c W, (c + 1) W) of both inputs. The row pair is read from HBM once:
//   1. TMA bulk copies (cp.async.bulk, mbarrier completion) stage the CTA's
//      slice of two rows in shared memory (two stages); a stage is refilled
//      as soon as pass C of its row has read it;
//   2. statistics of the next row, straight from its stage while the current
//      row's sums travel: NaN-propagating max of the raw 16-bit pairs reduced
//      over the warp, then the sum of 2^((x - m) log2 e) relative to the warp
//      max, merged over the CTA and then over the cluster: the MAX / SUM merge
//      of per-shard statistics with warps and CTAs as shards;
//   3. pass C from the stage: log2 p, log2 q, p, q and log2 M with
//      M = (1 - beta) p + beta q; the two expectations A = KL(P_t || M) and
//      B = KL(P_s || M) are reduced together over the CTA and the cluster.
//      p and the two log-ratios go to tensor memory (TMEM), q stays in
//      registers;
//   4. pass D: dS = g (1 - beta) p (ln p - ln M - B), dT = g beta q
//      (ln q - ln M - A) from TMEM and registers, stored with 16-byte stores.
// Tensor memory here is plain per-thread storage: each thread owns one TMEM
// lane and a range of 128 columns (the lane quarter of its warp), so pass D
// needs no exponential and no logarithm. When the raw -inf would reach a
// product, it is clamped first to a finite floor so that no 0 * inf forms.
// Arithmetic is fp32 (packed fp32x2 where it pairs up) in base-2 logarithms,
// so the hardware ex2 / lg2 apply without rescaling; sums are converted to
// nats once per row.
//
// Every wait on an mbarrier is bounded: when it gives up, the kernel records
// an error in its device error word, leaves its row loop (every CTA of the
// cluster does, since each then waits in vain for the others), waits
// (bounded) for its own copies in flight, frees its tensor memory and returns.
#pragma once

#include <cuda_runtime.h>

#include <type_traits>

#include "vpd_internal.h"
#include "vpd_packed.cuh"

namespace vpd {
namespace fused {

using vpd::InBF16;
using vpd::InF16;
using vpd::InF32;

constexpr int kStages = 2;                  // shared-memory stages per CTA (forward + backward)
constexpr int kFwdStages = 3;               // stages of the forward-only kernel
constexpr int kRing = 3;                    // cluster slots and their mbarriers, by row
constexpr float kTiny = 1e-37f;             // keeps M > 0 so log2 M stays finite
constexpr float kMaxLogit = 8.5070592e37f;  // 2^126: a larger finite row max is out of contract
constexpr int kMaxCluster = 16;
constexpr int kMaxR = 5;                    // 8-element vectors of each input per worker thread
constexpr int kTmemCols = 512;              // the whole tensor memory of the SM
constexpr int kMinSmem = 120 * 1024;        // keeps one CTA per SM (each takes all TMEM)
constexpr int kMaxWorkers = 19;             // worker warps per CTA (plus one control warp)
// Worker warps per CTA for R vectors per thread. A warp scheduler (SM
// sub-partition) holds a quarter of the register file, so the budget of a
// thread is 16K / (32 ceil((workers + 1) / 4)): 136 registers at R = 5 (15
// warps), 96 below (20 warps).
__host__ __device__ constexpr int max_workers(int R) { return R >= 5 ? 14 : kMaxWorkers; }
// The forward-only kernel keeps nothing across passes (about 70 registers), so
// it runs up to 23 worker warps at any R: more warps hide more of each row's
// hand-over latency.
constexpr int kMaxWorkersFwd = 23;
// TMEM columns of one worker warp: the warps of a lane quarter share its 512
// columns (a multiple of 8 each).
__host__ __device__ constexpr int tmem_cols_per_warp(int nw) { return (kTmemCols / ((nw + 3) / 4)) & ~7; }

enum Mode : int { kInterior = 0, kForwardKL = 1, kReverseKL = 2 };

// TMEM columns a thread uses per 8-element vector: p, log2 p - log2 M and
// log2 q - log2 M (interior); p and the log2 ratio target / other (KL).
template <int MODE>
struct Cols {
  static constexpr int k = MODE == kInterior ? 24 : 16;
};
static_assert(Cols<kInterior>::k * kMaxR <= tmem_cols_per_warp(max_workers(kMaxR)), "TMEM columns per thread");
static_assert(Cols<kInterior>::k * 4 <= tmem_cols_per_warp(max_workers(4)), "TMEM columns per thread");

// Set by a kernel of this translation unit whose bounded wait gave up (each
// translation unit that includes this header has its own word).
static __device__ int g_fused_error = 0;
// The value g_fused_error held when k_take_error last swapped it for 0.
static __device__ int g_fused_taken = 0;

// Reads and clears the error word in one atomic step, so that a failure
// recorded by a kernel on another stream in between is never lost.
static __global__ void k_take_error() { g_fused_taken = atomicExch(&g_fused_error, 0); }

// Host side: the word's value (0 if no wait gave up), cleared, in stream order.
static inline cudaError_t take_error_local(cudaStream_t stream, int* code) {
  k_take_error<<<1, 1, 0, stream>>>();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbolAsync(code, g_fused_taken, sizeof(int), 0, cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(stream);
}

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

// One try on an mbarrier phase (CTA-scope acquire).
__device__ __forceinline__ bool mbar_try_wait(uint64_t* mb, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(mb)), "r"(parity)
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
// One try with cluster-scope acquire: the partials arrive from other CTAs.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* mb, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(mb)), "r"(parity)
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
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* mb) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(mb))
      : "memory");
}
// Bulk copy shared -> global (TMA store), committed as one group per call
// site; wait_read: the shared source may be overwritten; wait_all: the global
// writes are done.
__device__ __forceinline__ void bulk_store(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_addr(src)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Generic-proxy shared-memory writes become visible to the bulk copies.
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
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
__device__ __forceinline__ uint32_t map_rank(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
// 16 bytes into a peer's shared memory; the bytes complete on its mbarrier.
__device__ __forceinline__ void push16(uint32_t remote, float a, float b, float c, float d, uint32_t remote_bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(remote),
      "f"(a), "f"(b), "f"(c), "f"(d), "r"(remote_bar)
      : "memory");
}
// Named CTA barriers over n threads: arrive (no wait, release) and sync (wait, acquire).
__device__ __forceinline__ void bar_arrive(int id, int n) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void bar_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }
__device__ __forceinline__ void st_global16(void* p, uint4 v) {
  asm volatile("st.global.L1::no_allocate.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// Tensor memory: allocation by one warp (the address lands in shared memory),
// and per-thread 32-bit columns of the thread's own lane (32x32b shape).
__device__ __forceinline__ void tmem_alloc(uint32_t* slot) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(slot)),
               "n"(kTmemCols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t base) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "n"(kTmemCols) : "memory");
}
__device__ __forceinline__ void tmem_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// 8 consecutive columns from 4 packed pairs.
__device__ __forceinline__ void tmem_st8(uint32_t ta, const float2 (&v)[4]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(ta),
               "f"(v[0].x), "f"(v[0].y), "f"(v[1].x), "f"(v[1].y), "f"(v[2].x), "f"(v[2].y), "f"(v[3].x),
               "f"(v[3].y));
}
// 8 consecutive columns, waited for within the same statement so that no
// register is read before the load has landed.
__device__ __forceinline__ void tmem_ld8_wait(uint32_t ta, float2 (&v)[4]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=f"(v[0].x), "=f"(v[0].y), "=f"(v[1].x), "=f"(v[1].y), "=f"(v[2].x), "=f"(v[2].y), "=f"(v[3].x),
        "=f"(v[3].y)
      : "r"(ta));
}
// 16 + 8 columns (three groups of 8), one wait.
__device__ __forceinline__ void tmem_ld24_wait(uint32_t ta, float2 (&a)[4], float2 (&b)[4], float2 (&c)[4]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%24];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%16,%17,%18,%19,%20,%21,%22,%23}, [%25];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=f"(a[0].x), "=f"(a[0].y), "=f"(a[1].x), "=f"(a[1].y), "=f"(a[2].x), "=f"(a[2].y), "=f"(a[3].x),
        "=f"(a[3].y), "=f"(b[0].x), "=f"(b[0].y), "=f"(b[1].x), "=f"(b[1].y), "=f"(b[2].x), "=f"(b[2].y),
        "=f"(b[3].x), "=f"(b[3].y), "=f"(c[0].x), "=f"(c[0].y), "=f"(c[1].x), "=f"(c[1].y), "=f"(c[2].x),
        "=f"(c[2].y), "=f"(c[3].x), "=f"(c[3].y)
      : "r"(ta), "r"(ta + 16));
}
// 16 columns (two groups of 8), one wait.
__device__ __forceinline__ void tmem_ld16_wait(uint32_t ta, float2 (&a)[4], float2 (&b)[4]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=f"(a[0].x), "=f"(a[0].y), "=f"(a[1].x), "=f"(a[1].y), "=f"(a[2].x), "=f"(a[2].y), "=f"(a[3].x),
        "=f"(a[3].y), "=f"(b[0].x), "=f"(b[0].y), "=f"(b[1].x), "=f"(b[1].y), "=f"(b[2].x), "=f"(b[2].y),
        "=f"(b[3].x), "=f"(b[3].y)
      : "r"(ta));
}

// Warp-wide NaN-propagating max (every lane gets it).
__device__ __forceinline__ float warp_max_nan(float v) {
  float r;
  asm volatile("redux.sync.max.NaN.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
// Warp sums of a and of b in one butterfly: the half-warps first swap the
// other value, then each reduces its own; lanes 0-15 return the sum of a,
// lanes 16-31 that of b.
__device__ __forceinline__ float warp_sum_pair(float a, float b) {
  const bool hi = (threadIdx.x & 16) != 0;
  float v = (hi ? b : a) + __shfl_xor_sync(0xffffffffu, hi ? a : b, 16);
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

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
  __device__ static __forceinline__ void store8_shared(unsigned char* p, const float2 (&v)[4]) {
    *reinterpret_cast<uint4*>(p) = make_uint4(pack(v[0]), pack(v[1]), pack(v[2]), pack(v[3]));
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
  __device__ static __forceinline__ void store8_shared(unsigned char* p, const float2 (&v)[4]) {
    *reinterpret_cast<uint4*>(p) = make_uint4(pack(v[0]), pack(v[1]), pack(v[2]), pack(v[3]));
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
  __device__ static __forceinline__ void store8_shared(unsigned char*, const float2 (&)[4]) {}
};

// Stage vectors are read with In::ld (plain shared-memory loads: ordered after
// the mbarrier waits and barriers, free to schedule otherwise).

// ---------------------------------------------------------------------------
// Work split inside a CTA. nw worker warps (chosen on the host so that the
// slice divides evenly: each worker thread holds at most R vectors of each
// input) do the element work; one control warp does every wait on another
// CTA, the merges, the pushes, the TMA issue and the per-row outputs. The two
// roles hand over through shared memory and named barriers (one side arrives,
// the other syncs), so the reductions of a row overlap the statistics pass of
// the next and the workers never meet in a CTA-wide barrier.
//
// Cluster reductions by push: the control warp merges the workers' partials
// and lane c sends the CTA's partial with st.async into CTA c's slot for this
// CTA; the bytes complete on the peer's mbarrier. The control warp of each CTA
// arms its own mbarrier for C partials, waits (bounded) and merges the C
// slots. Slots and mbarriers are double-buffered by row parity: a CTA cannot
// run two rows ahead of a peer, since it needs that peer's partial of every
// row to proceed.
//
// Statistics travel as (m_s, z_s, m_t, z_t): z relative to m, with z = NaN
// marking an input outside the contract (a NaN, +inf or a max above 2^126),
// which the merges propagate. Sums travel as (A, B) in nats; a KL support
// violation makes A = +inf.
// ---------------------------------------------------------------------------
enum NamedBar : int {
  kBarStatPart = 1,
  kBarStatReady = 2,
  kBarSumPart = 3,
  kBarSumReady = 4,
  kBarGradFull = 5,
  kBarStatPartOdd = 6,  // forward-only kernel: statistics partials of odd rows
};

struct Tail {
  uint64_t tma_bar[kFwdStages];
  uint64_t stat_bar[kRing];
  uint64_t sum_bar[kRing];
  uint32_t tmem_base;
  int fail;  // set by a worker whose wait on a stage gave up
  __align__(16) float stat_part[2][kMaxWorkersFwd][4];  // per worker warp: m_s, z_s, m_t, z_t
  __align__(16) float sum_part[2][kMaxWorkersFwd][4];   // per worker warp: A, B (nats)
  __align__(16) float stat_res[2][8];  // -m_s, -m_t, -log2 Z_s, -log2 Z_t, row ok, run ok
  __align__(16) float sum_res[2][4];   // A, B, value (nats)
  __align__(16) float stat_slot[kRing][kMaxCluster][4];
  __align__(16) float sum_slot[kRing][kMaxCluster][4];
};

// Merge (m, z) over the lanes of a warp (unused lanes hold (-inf, 0)).
__device__ __forceinline__ float2 merge_warp(float m, float z) {
  const float mx = warp_max_nan(m);
  return make_float2(mx, warp_sum(z * exp_acc(m - stat_ref(mx))));
}

// Control warp: arm this CTA's mbarrier for the C partials of one row and
// wait (bounded, every lane); false if the wait gave up.
__device__ __forceinline__ bool control_wait(uint64_t* bar, uint32_t parity, uint32_t csize) {
  if ((threadIdx.x & 31) == 0) mbar_expect_tx(bar, csize * 16u);
  __syncwarp();
  const bool mine = mbar_wait_cluster(bar, parity);
  return __all_sync(0xffffffffu, mine);
}

// Control warp: merge the workers' statistics partials and push the CTA's to
// every CTA of the cluster (ring slot `par`, entry `crank`).
__device__ __forceinline__ void control_push_stats(const float (*part)[4], int nw, Tail* tail, int par,
                                                   uint32_t crank, uint32_t csize) {
  const int lane = threadIdx.x & 31;
  float4 v = make_float4(neg_inf(), 0.f, neg_inf(), 0.f);
  if (lane < nw) v = *reinterpret_cast<const float4*>(part[lane]);
  const float2 s = merge_warp(v.x, v.y), t = merge_warp(v.z, v.w);
  if (lane < static_cast<int>(csize))
    push16(map_rank(smem_addr(tail->stat_slot[par][crank]), lane), s.x, s.y, t.x, t.y,
           map_rank(smem_addr(&tail->stat_bar[par]), lane));
}

// Which of its R vectors (k Tw + vt, k = 0..R-1, vt the thread's place in the
// vector order) a worker thread holds: the first `kv`; every lane of its warp
// holds the first `kfull`, some lane the first `kwarp` (both warp-uniform).
struct Span {
  int kv, kfull, kwarp;
};
template <int R>
__device__ __forceinline__ Span span_of(int len, int Tw, int vt) {
  const int nv = len >> 3, w0 = vt & ~31;
  auto kv_of = [&](int t) {
    const int k = (nv - t + Tw - 1) / Tw;
    return k < 0 ? 0 : (k > R ? R : k);
  };
  return {kv_of(vt), kv_of(w0 + 31), kv_of(w0)};
}

// The position of worker warp `warp` in the order in which the workers take
// the slice's vectors (vector k Tw + 32 j + lane goes to lane `lane` of the
// j-th warp). A warp scheduler (SM sub-partition, warp % 4) issues only for
// its own warps, and every per-row phase ends with its busiest scheduler, so
// the last, partial round of R vectors goes first to the schedulers with the
// least work: each next warp comes from the scheduler with the fewest vectors
// so far, ties away from the control warp's.
__host__ __device__ __forceinline__ int vector_order(int warp, int nw, int R) {
  int load[4], next[4];
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    load[s] = (nw - s + 3) / 4 * (R - 1);
    next[s] = s;
  }
  const int ctrl = nw & 3;
  for (int j = 0; j < nw; ++j) {
    int b = -1, lb = 0;
#pragma unroll
    for (int s = 0; s < 4; ++s)
      if (next[s] < nw && (b < 0 || load[s] < lb || (load[s] == lb && b == ctrl))) {
        b = s;
        lb = load[s];
      }
#pragma unroll
    for (int s = 0; s < 4; ++s) {  // constant indices keep the arrays in registers
      if (s != b) continue;
      if (next[s] == warp) return j;
      next[s] += 4;
      ++load[s];
    }
  }
  return warp;
}

// Worker warps: statistics partial of one row read from its shared-memory
// stage (`vt`: this thread's place in the vector order); lane 0 writes the
// warp's (m_s, z_s, m_t, z_t) to `part`. KEEP holds the vectors in registers
// between the max and the exponential sweeps (one shared-memory read instead
// of two) where the kernel has registers to spare.
template <class In, int R, bool KEEP = false>
__device__ __forceinline__ void worker_stats(const unsigned char* sb, int W, const Span& sp, int Tw, int vt,
                                             float* part) {
  using Word = typename In::Word;
  using Vec = typename In::Vec;
  constexpr int kVB = 8 * In::kSize;  // bytes of one 8-element vector
  const int lane = threadIdx.x & 31;
  const unsigned char* ps = sb + vt * kVB;
  const size_t tofs = static_cast<size_t>(W) * In::kSize;
  Word mxs = In::neg_inf_w(), mxt = In::neg_inf_w();
  Vec ku[R], kv[R];
#pragma unroll
  for (int k = 0; k < R; ++k) {
    if (k < sp.kv) {
      const Vec u = In::ld(ps + k * Tw * kVB), v = In::ld(ps + tofs + k * Tw * kVB);
      if (KEEP) {
        ku[k] = u;
        kv[k] = v;
      }
      Word uw[4], vw[4];
      In::words(u, uw);
      In::words(v, vw);
      mxs = In::max_nan(mxs, In::max_nan(In::max_nan(uw[0], uw[1]), In::max_nan(uw[2], uw[3])));
      mxt = In::max_nan(mxt, In::max_nan(In::max_nan(vw[0], vw[1]), In::max_nan(vw[2], vw[3])));
    }
  }
  const float2 a = In::unpack(mxs), b = In::unpack(mxt);
  const float m_s = warp_max_nan(max_nan(a.x, a.y)), m_t = warp_max_nan(max_nan(b.x, b.y));
  const float2 l2e2 = f2(kLog2e), ns2 = f2(-stat_ref(m_s)), nt2 = f2(-stat_ref(m_t));
  float2 zs2 = f2(0.f), zt2 = f2(0.f);
#pragma unroll
  for (int k = 0; k < R; ++k) {
    if (k < sp.kv) {
      const Vec u = KEEP ? ku[k] : In::ld(ps + k * Tw * kVB), v = KEEP ? kv[k] : In::ld(ps + tofs + k * Tw * kVB);
      Word us[4], vs[4];
      In::words(u, us);
      In::words(v, vs);
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        // x - m is exact; a -inf entry gives 2^-inf = 0, a NaN gives NaN
        zs2 = add2(zs2, ex2_2(mul2(In::sub(us[w], ns2), l2e2)));
        zt2 = add2(zt2, ex2_2(mul2(In::sub(vs[w], nt2), l2e2)));
      }
    }
  }
  // z_s on lanes 0-15, z_t on lanes 16-31
  float z = warp_sum_pair(zs2.x + zs2.y, zt2.x + zt2.y);
  const float m = lane < 16 ? m_s : m_t;
  if (!(m <= kMaxLogit)) z = qnan();  // NaN, +inf or a max above 2^126
  if ((lane & 15) == 0) *reinterpret_cast<float2*>(part + (lane >> 3)) = make_float2(m, z);
}

struct FusedArgs {
  const char* s;
  const char* t;
  RowMap ms, mt;
  int64_t rows;
  int64_t vocab;
  int W;      // slice width per CTA (elements, multiple of 8)
  int nw;     // worker warps per CTA
  int gstage; // 16-bit gradients go through a shared-memory buffer and bulk stores
  float beta;
  const float* grad_loss;
  float* loss;
  float* saved;
  Grad ds, dt;
  int64_t withhold_row;  // test hook: CTA 0 of the owning cluster never copies this row (-1: none)
};

// log2 of the probabilities of one packed pair: (x - m) log2 e - K.
template <class In>
__device__ __forceinline__ float2 lam(typename In::Word w, float2 nm, float2 l2e2, float2 nK) {
  return fma2(In::sub(w, nm), l2e2, nK);
}

// NW > 0 fixes the worker count at compile time (the common shapes), so that
// the vector offsets k 32 NW are immediates; NW = 0 takes it from the args.
template <class In, class G, int R, int MODE, int NW = 0>
__global__ void __launch_bounds__(32 * (max_workers(R) + 1), 1) k_jsd_fused(FusedArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int kCols = Cols<MODE>::k;
  const int W = a.W, nw = NW > 0 ? NW : a.nw, Tw = 32 * nw, nthreads = Tw + 32;
  // Shared memory: kStages x [s, t] slices, then (staged gradients) the dS and
  // dT slices of one row, then the tail.
  constexpr int kVB = 8 * In::kSize;  // bytes of one 8-element input vector
  using Word = typename In::Word;
  using Vec = typename In::Vec;
  unsigned char* gbuf = smem + static_cast<size_t>(kStages) * 2 * In::kSize * W;
  const bool staged = a.gstage != 0 && (a.ds.data || a.dt.data);
  Tail* tail = reinterpret_cast<Tail*>(gbuf + (a.gstage ? static_cast<size_t>(4) * W : 0));
  auto stage_ptr = [&](int st) { return smem + static_cast<size_t>(st) * 2 * In::kSize * W; };

  const uint32_t crank = cluster_rank(), csize = cluster_size();
  const int64_t q = cluster_index(), Q = cluster_count();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool control = warp == nw;
  const int64_t col0 = static_cast<int64_t>(crank) * W;
  const int64_t rest = a.vocab - col0;
  const int len = rest <= 0 ? 0 : (rest < W ? static_cast<int>(rest) : W);
  const uint32_t bytes = static_cast<uint32_t>(len) * In::kSize;  // of each input's slice
  const uint32_t gbytes = static_cast<uint32_t>(len) * 2u;        // of each staged 16-bit gradient slice

  // The failure-path test hook: this CTA withholds the copy of one row, so
  // its workers' bounded wait on that stage expires.
  auto withheld = [&](int64_t r) { return r == a.withhold_row && crank == 0; };
  // control warp, bit st: copies were issued into stage st / their count is odd
  uint32_t issued_any = 0, issued_odd = 0;
  auto issue = [&](int64_t r, int st) {  // control warp: both inputs' slices of row r into stage st
    if (!bytes || withheld(r)) return;
    if (lane == 0) {
      unsigned char* dst = stage_ptr(st);
      mbar_expect_tx(&tail->tma_bar[st], 2 * bytes);
      bulk_load(dst, a.s + (a.ms.offset(r) + col0) * In::kSize, bytes, &tail->tma_bar[st]);
      bulk_load(dst + static_cast<size_t>(W) * In::kSize, a.t + (a.mt.offset(r) + col0) * In::kSize, bytes,
                &tail->tma_bar[st]);
    }
    issued_any |= 1u << st;
    issued_odd ^= 1u << st;
  };

  // Control warp: bulk stores of the staged (16-bit) gradients of row r.
  auto store_grads = [&](int64_t r) {
    if (lane == 0 && gbytes) {
      if (a.ds.data) bulk_store(a.ds.data + (r * a.ds.row_stride + col0) * 2, gbuf, gbytes);
      if (a.dt.data)
        bulk_store(a.dt.data + (r * a.dt.row_stride + col0) * 2, gbuf + static_cast<size_t>(W) * 2, gbytes);
      bulk_commit();
    }
  };

  if (control) {
    if (lane == 0) {
      for (int st = 0; st < kStages; ++st) mbar_init(&tail->tma_bar[st], 1);
      for (int p = 0; p < kRing; ++p) {
        mbar_init(&tail->stat_bar[p], 1);
        mbar_init(&tail->sum_bar[p], 1);
      }
      tail->fail = 0;
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    tmem_alloc(&tail->tmem_base);
    for (int st = 0; st < kStages; ++st)
      if (q + st * Q < a.rows) issue(q + st * Q, st);
  }
  tmem_fence_before();
  __syncthreads();
  tmem_fence_after();
  cluster_sync();  // every CTA's mbarriers are initialised before any push

  const float beta = a.beta;
  bool ok = true;
  if (control) {
    // ------------------------------------------------------------------
    // Control warp.
    // ------------------------------------------------------------------
    if (q < a.rows) {
      bar_sync(kBarStatPart, nthreads);
      if (tail->fail) ok = false;
      control_push_stats(tail->stat_part[0], nw, tail, 0, crank, csize);
    }
    int64_t i = 0;
    int64_t owed = -1;  // row whose staged gradients the workers write next (not yet stored)
    for (int64_t r = q; r < a.rows; r += Q, ++i) {
      const int par = static_cast<int>(i & 1);
      const uint32_t ph = static_cast<uint32_t>((i >> 1) & 1);
      const bool has_next = r + Q < a.rows;
      const int cst = static_cast<int>(i % kStages);

      // (C1) global statistics of row r, handed to the workers
      float4 g = make_float4(qnan(), qnan(), qnan(), qnan());
      if (ok) ok = control_wait(&tail->stat_bar[par], ph, csize);
      if (ok) {
        float4 v = make_float4(neg_inf(), 0.f, neg_inf(), 0.f);
        if (lane < static_cast<int>(csize)) v = *reinterpret_cast<const float4*>(tail->stat_slot[par][lane]);
        const float2 s = merge_warp(v.x, v.y), t = merge_warp(v.z, v.w);
        g = make_float4(s.x, s.y, t.x, t.y);
      }
      const bool bad_s = isnan(g.y), bad_t = isnan(g.w);
      const bool row_ok = ok && !bad_s && !bad_t && g.x != neg_inf() && g.z != neg_inf();
      const float Ks = row_ok ? log2f(g.y) : qnan();  // log2 Z
      const float Kt = row_ok ? log2f(g.w) : qnan();
      if (lane == 0) {
        float* res = tail->stat_res[par];
        *reinterpret_cast<float4*>(res) = make_float4(-g.x, -g.z, -Ks, -Kt);
        *reinterpret_cast<float2*>(res + 4) = make_float2(row_ok ? 1.f : 0.f, ok ? 1.f : 0.f);
      }
      bar_arrive(kBarStatReady, nthreads);
      if (!ok) break;

      // The previous row's gradients are staged (the workers finished its
      // pass D before taking this row's statistics): store them.
      if (owed >= 0) {
        bar_sync(kBarGradFull, nthreads);
        store_grads(owed);
        owed = -1;
      }

      // (C2) the workers have read this row's stage: refill it with the row
      // kStages on; reduce and push this row's sums
      bar_sync(kBarSumPart, nthreads);
      if (r + kStages * Q < a.rows) issue(r + kStages * Q, cst);
      {
        float2 v = make_float2(0.f, 0.f);
        if (lane < nw) v = *reinterpret_cast<const float2*>(tail->sum_part[par][lane]);
        const float sa = warp_sum(v.x), sb = warp_sum(v.y);
        if (lane < static_cast<int>(csize))
          push16(map_rank(smem_addr(tail->sum_slot[par][crank]), lane), sa, sb, 0.f, 0.f,
                 map_rank(smem_addr(&tail->sum_bar[par]), lane));
      }

      // (C3) global sums of row r, handed to the workers as soon as they
      // arrive; then the per-token value and saved statistics
      float A = qnan(), B = qnan(), value = qnan();
      const bool got = ok && control_wait(&tail->sum_bar[par], ph, csize);
      if (!got) ok = false;
      if (got && row_ok) {
        float2 v = make_float2(0.f, 0.f);
        if (lane < static_cast<int>(csize)) v = *reinterpret_cast<const float2*>(tail->sum_slot[par][lane]);
        A = warp_sum(v.x);
        B = warp_sum(v.y);
        if (MODE == kInterior) {
          value = beta * A + (1.f - beta) * B;
        } else {
          value = A;  // +inf on a support violation
          A = MODE == kForwardKL ? value : 0.f;
          B = MODE == kForwardKL ? 0.f : value;
        }
      }
      if (lane == 0) *reinterpret_cast<float4*>(tail->sum_res[par]) = make_float4(A, B, value, 0.f);
      // the workers overwrite the staging buffer once they have this row's sums
      if (staged && lane == 0) bulk_wait_read();
      bar_arrive(kBarSumReady, nthreads);
      if (staged) owed = r;
      if (lane == 0 && crank == 0) a.loss[r] = value;
      if (lane == 0 && crank == 0 && a.saved) {
        float* sv = a.saved + r * VPD_SAVED_PAIR;
        sv[0] = bad_s ? qnan() : g.x;
        sv[1] = bad_s ? qnan() : (g.x == neg_inf() ? neg_inf() : (row_ok ? kLn2 * Ks : kLn2 * log2f(g.y)));
        sv[2] = bad_t ? qnan() : g.z;
        sv[3] = bad_t ? qnan() : (g.z == neg_inf() ? neg_inf() : (row_ok ? kLn2 * Kt : kLn2 * log2f(g.w)));
        sv[4] = A;
        sv[5] = B;
      }

      // (C4) statistics of the next row
      if (has_next) {
        bar_sync(kBarStatPart, nthreads);
        if (tail->fail) ok = false;
        control_push_stats(tail->stat_part[par ^ 1], nw, tail, par ^ 1, crank, csize);
      }
    }
    if (owed >= 0) {
      bar_sync(kBarGradFull, nthreads);
      store_grads(owed);
    }
    if (lane == 0) bulk_wait_all();
    // Copies still in flight (only after a wait gave up) must land before exit.
    if (lane == 0)
      for (int st = 0; st < kStages; ++st)
        if ((issued_any >> st) & 1u) mbar_wait(&tail->tma_bar[st], ((issued_odd >> st) & 1u) ^ 1u);
    if (!ok && lane == 0) atomicExch(&g_fused_error, 1);
  } else {
    // ------------------------------------------------------------------
    // Worker warps.
    // ------------------------------------------------------------------
    // This thread's TMEM lane (its warp's lane quarter) and column range.
    const uint32_t tmem = tail->tmem_base + (static_cast<uint32_t>(32 * (warp & 3)) << 16) +
                          static_cast<uint32_t>(tmem_cols_per_warp(nw) * (warp >> 2));
    uint32_t tma_parity = 0;  // bit st: parity of the next wait on stage st
    auto wait_stage = [&](int st) {
      if (!bytes) return;
      if (!mbar_wait(&tail->tma_bar[st], (tma_parity >> st) & 1u)) tail->fail = 1;
      tma_parity ^= 1u << st;
    };
    const float2 ws2 = f2(1.f - beta), wt2 = f2(beta), tiny2 = f2(kTiny), l2e2 = f2(kLog2e);
    const int64_t gstride = static_cast<int64_t>(Tw) * 8 * Out<G>::kSize;  // bytes between vectors k, k + 1
    const int vt = 32 * vector_order(warp, nw, R) + lane;  // this thread's place in the vector order
    const Span sp = span_of<R>(len, Tw, vt);

    if (q < a.rows) {
      wait_stage(0);
      worker_stats<In, R>(stage_ptr(0), W, sp, Tw, vt, tail->stat_part[0][warp]);
      bar_arrive(kBarStatPart, nthreads);
    }
    int64_t i = 0;
    for (int64_t r = q; r < a.rows; r += Q, ++i) {
      const int par = static_cast<int>(i & 1);
      const bool has_next = r + Q < a.rows;
      const int cst = static_cast<int>(i % kStages);
      const int nst = static_cast<int>((i + 1) % kStages);

      // upstream gradient of row r, loaded well before pass D needs it
      const float gr = a.grad_loss ? __ldg(a.grad_loss + r) : 1.f;

      // (W1) global statistics of row r
      bar_sync(kBarStatReady, nthreads);
      const float4 st4 = *reinterpret_cast<const float4*>(tail->stat_res[par]);
      const float2 flags = *reinterpret_cast<const float2*>(tail->stat_res[par] + 4);
      if (flags.y == 0.f) break;
      const bool row_ok = flags.x != 0.f;
      const float2 nms2 = f2(st4.x), nmt2 = f2(st4.y), nKs2 = f2(st4.z), nKt2 = f2(st4.w);

      // (W2) pass C of row r from its stage, in log2 units. TMEM per vector:
      // interior p, log2 p - log2 M, log2 q - log2 M; KL p, log2 ratio. q in
      // registers. Warps past the slice skip a vector together; inside a warp,
      // lanes past it compute on the floor value (p = q = 0) so that the TMEM
      // stores stay warp-uniform.
      float2 kq[R][4];
      float2 acc_a = f2(0.f), acc_b = f2(0.f);
      uint32_t viol = 0;
      if (row_ok) {
        const unsigned char* ps = stage_ptr(cst) + vt * kVB;
        const size_t tofs = static_cast<size_t>(W) * In::kSize;
        // One vector: PARTIAL marks the warp that straddles the slice end,
        // whose lanes past it compute on the floor value.
        auto vec_c = [&](int k, auto partial) {
          constexpr bool PARTIAL = decltype(partial)::value;
          Vec u, v;
          if (!PARTIAL || k < sp.kv) {
            u = In::ld(ps + k * Tw * kVB);
            v = In::ld(ps + tofs + k * Tw * kVB);
          } else {
            u = v = In::fill_neg_big();
          }
          Word us[4], vs[4];
          In::words(u, us);
          In::words(v, vs);
          float2 t0[4], t1[4], t2[4];
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            if (MODE != kInterior) {
              const Word tgt = MODE == kForwardKL ? vs[w] : us[w];
              const Word oth = MODE == kForwardKL ? us[w] : vs[w];
              viol |= In::viol(tgt, oth);
            }
            const float2 lp = lam<In>(In::max2(us[w], In::neg_big_w()), nms2, l2e2, nKs2);
            const float2 lq = lam<In>(In::max2(vs[w], In::neg_big_w()), nmt2, l2e2, nKt2);
            const float2 p = ex2_2(lp), qv = ex2_2(lq);
            kq[k][w] = qv;
            t0[w] = p;
            if (MODE == kInterior) {
              const float2 lm = lg2_2(fma2(ws2, p, fma2(wt2, qv, tiny2)));
              const float2 us_ = add2(lp, neg(lm)), ut_ = add2(lq, neg(lm));
              acc_b = fma2(p, us_, acc_b);
              acc_a = fma2(qv, ut_, acc_a);
              t1[w] = us_;
              t2[w] = ut_;
            } else {
              // forward KL(q || p): d = log2 q - log2 p weighted by q; reverse: mirror
              const float2 d = MODE == kForwardKL ? add2(lq, neg(lp)) : add2(lp, neg(lq));
              acc_a = fma2(MODE == kForwardKL ? qv : p, d, acc_a);
              t1[w] = d;
            }
          }
          tmem_st8(tmem + k * kCols, t0);
          tmem_st8(tmem + k * kCols + 8, t1);
          if (MODE == kInterior) tmem_st8(tmem + k * kCols + 16, t2);
        };
#pragma unroll
        for (int k = 0; k < R; ++k) {
          if (k < sp.kfull) vec_c(k, std::false_type{});
          else if (k < sp.kwarp) vec_c(k, std::true_type{});  // warp-uniform branches
        }
        tmem_wait_st();
      }
      if constexpr (MODE == kInterior) {  // A partial on lanes 0-15, B partial on lanes 16-31
        const float v = kLn2 * warp_sum_pair(acc_a.x + acc_a.y, acc_b.x + acc_b.y);
        if ((lane & 15) == 0) tail->sum_part[par][warp][lane >> 4] = v;
      } else {
        float sa = kLn2 * warp_sum(acc_a.x + acc_a.y);
        if (__any_sync(0xffffffffu, viol != 0)) sa = pos_inf();
        if (lane == 0) *reinterpret_cast<float2*>(tail->sum_part[par][warp]) = make_float2(sa, 0.f);
      }
      bar_arrive(kBarSumPart, nthreads);

      // (W3) statistics partial of the next row, straight from its stage,
      // while this row's sums travel
      if (has_next) {
        wait_stage(nst);
        worker_stats<In, R>(stage_ptr(nst), W, sp, Tw, vt, tail->stat_part[par ^ 1][warp]);
        bar_arrive(kBarStatPart, nthreads);
      }

      // (W4) global sums of row r
      bar_sync(kBarSumReady, nthreads);
      const float4 ab = *reinterpret_cast<const float4*>(tail->sum_res[par]);
      const float A = ab.x, B = ab.y, value = ab.z;

      // (W5) pass D of row r: gradients, e.g. dS = p (g (1-beta) ln2 (log2 p - log2 M) - g (1-beta) B)
      char* ds_row = a.ds.data ? a.ds.data + (r * a.ds.row_stride + col0 + vt * 8) * Out<G>::kSize : nullptr;
      char* dt_row = a.dt.data ? a.dt.data + (r * a.dt.row_stride + col0 + vt * 8) * Out<G>::kSize : nullptr;
      if (ds_row || dt_row) {
        const bool live = row_ok && isfinite(value);
        const float cs = MODE == kInterior ? gr * (1.f - beta) : gr;
        const float ct = MODE == kInterior ? gr * beta : gr;
        const float2 cs2 = f2(cs * kLn2), ct2 = f2(ct * kLn2);
        const float2 ncs2 = f2(-cs * (MODE == kInterior ? B : value));
        const float2 nct2 = f2(-ct * (MODE == kInterior ? A : value));
        const float2 g2 = f2(gr);
        // One vector: TMEM loads stay warp-uniform; only lanes holding the
        // vector store it.
        auto vec_d = [&](int k, auto staged_t) {
          constexpr bool STAGED = decltype(staged_t)::value;
          float2 gs[4], gt[4];
          float2 p[4], u1[4], u2[4];
          if (MODE == kInterior) tmem_ld24_wait(tmem + k * kCols, p, u1, u2);
          else tmem_ld16_wait(tmem + k * kCols, p, u1);
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const float2 qv = kq[k][w];
            if (MODE == kInterior) {
              gs[w] = mul2(p[w], fma2(cs2, u1[w], ncs2));
              gt[w] = mul2(qv, fma2(ct2, u2[w], nct2));
            } else if (MODE == kForwardKL) {  // dS = g (p - q), dT = g q (ln q - ln p - KL)
              gs[w] = mul2(g2, add2(p[w], neg(qv)));
              gt[w] = mul2(qv, fma2(ct2, u1[w], nct2));
            } else {  // dS = g p (ln p - ln q - KL), dT = g (q - p)
              gs[w] = mul2(p[w], fma2(cs2, u1[w], ncs2));
              gt[w] = mul2(g2, add2(qv, neg(p[w])));
            }
          }
          if (k < sp.kv) {
            if constexpr (STAGED) {
              unsigned char* pg = gbuf + (k * Tw + vt) * 16;
              if (ds_row) Out<G>::store8_shared(pg, gs);
              if (dt_row) Out<G>::store8_shared(pg + static_cast<size_t>(W) * 2, gt);
            } else {
              if (ds_row) Out<G>::store8(ds_row + k * gstride, gs);
              if (dt_row) Out<G>::store8(dt_row + k * gstride, gt);
            }
          }
        };
        // Rows with no defined value get zero gradients.
        auto zero_d = [&](int k, auto staged_t) {
          constexpr bool STAGED = decltype(staged_t)::value;
          float2 z[4] = {f2(0.f), f2(0.f), f2(0.f), f2(0.f)};
          if (k < sp.kv) {
            if constexpr (STAGED) {
              unsigned char* pg = gbuf + (k * Tw + vt) * 16;
              if (ds_row) Out<G>::store8_shared(pg, z);
              if (dt_row) Out<G>::store8_shared(pg + static_cast<size_t>(W) * 2, z);
            } else {
              if (ds_row) Out<G>::store8(ds_row + k * gstride, z);
              if (dt_row) Out<G>::store8(dt_row + k * gstride, z);
            }
          }
        };
        auto run_d = [&](auto staged_t) {
          if (live) {
#pragma unroll
            for (int k = 0; k < R; ++k)
              if (k < sp.kwarp) vec_d(k, staged_t);  // warp-uniform
          } else {
#pragma unroll
            for (int k = 0; k < R; ++k) zero_d(k, staged_t);
          }
        };
        if (Out<G>::kSize == 2 && staged) run_d(std::true_type{});
        else run_d(std::false_type{});
        if (staged) {
          fence_proxy_async();
          bar_arrive(kBarGradFull, nthreads);
        }
      }
    }
    tmem_wait_st();
  }

  tmem_fence_before();
  __syncthreads();
  if (control) {
    tmem_fence_after();
    tmem_dealloc(tail->tmem_base);
  }
  cluster_sync();  // no CTA leaves while a peer may still push into it
}

// ---------------------------------------------------------------------------
// Forward only (no gradient wanted): the statistics, pass C and the cluster
// reductions of the kernel above without pass D, so nothing goes to tensor
// memory and q is not kept. With no pass D, the exchanges are hidden another
// way: each worker computes the statistics partial of row i + 1 before pass C
// of row i, so that their cluster exchange travels during pass C; and the
// control warp takes the cluster's sums of a row two rows later, when they are
// in, so that this wait never delays a hand-over. Three shared-memory stages
// keep two rows ahead of pass C in flight (a stage is refilled with row i + 3
// once pass C of row i has read it, and is needed again two rows later).
//
// Row indices below count this cluster's rows (row q + i Q is row i).
// Workers, per row i: the statistics partial of row i + 1 from its stage;
// wait for the statistics of row i; pass C of row i (the partials of A and B).
// Control warp, per row i: (C1) merge the cluster's statistics of row i and
// hand them over; (C3) wait for the cluster's sums of row i - 2 and write its
// loss and saved statistics; (C4) merge and push the statistics of row i + 1;
// (C2) once pass C of row i is in, refill its stage with row i + 3 and push
// this CTA's sums. Cluster slots and their mbarriers form rings of three by
// row: a CTA pushes into the slot of row i + 3 only after its own hand-over of
// row i + 3 or i + 2, which needs partials that every peer sends only after
// reading that slot for row i.
// ---------------------------------------------------------------------------
template <class In, int R, int MODE, int NW = 0>  // NW: as for k_jsd_fused
__global__ void __launch_bounds__(32 * (kMaxWorkersFwd + 1), 1) k_jsd_fused_fwd(FusedArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int W = a.W, nw = NW > 0 ? NW : a.nw, Tw = 32 * nw, nthreads = Tw + 32;
  constexpr int kVB = 8 * In::kSize;  // bytes of one 8-element input vector
  using Word = typename In::Word;
  Tail* tail = reinterpret_cast<Tail*>(smem + static_cast<size_t>(kFwdStages) * 2 * In::kSize * W);
  auto stage_ptr = [&](int st) { return smem + static_cast<size_t>(st) * 2 * In::kSize * W; };

  const uint32_t crank = cluster_rank(), csize = cluster_size();
  const int64_t q = cluster_index(), Q = cluster_count();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool control = warp == nw;
  const int64_t col0 = static_cast<int64_t>(crank) * W;
  const int64_t rest = a.vocab - col0;
  const int len = rest <= 0 ? 0 : (rest < W ? static_cast<int>(rest) : W);
  const uint32_t bytes = static_cast<uint32_t>(len) * In::kSize;
  // statistics partials of row i hand over on a named barrier of its parity:
  // the workers may arrive for row i + 1 before the control warp took row i
  auto stat_part_bar = [](int64_t i) { return (i & 1) ? kBarStatPartOdd : kBarStatPart; };

  auto withheld = [&](int64_t r) { return r == a.withhold_row && crank == 0; };
  // control warp, bit st: copies were issued into stage st / their count is odd
  uint32_t issued_any = 0, issued_odd = 0;
  auto issue = [&](int64_t r, int st) {  // control warp: both inputs' slices of row r into stage st
    if (!bytes || withheld(r)) return;
    if (lane == 0) {
      unsigned char* dst = stage_ptr(st);
      mbar_expect_tx(&tail->tma_bar[st], 2 * bytes);
      bulk_load(dst, a.s + (a.ms.offset(r) + col0) * In::kSize, bytes, &tail->tma_bar[st]);
      bulk_load(dst + static_cast<size_t>(W) * In::kSize, a.t + (a.mt.offset(r) + col0) * In::kSize, bytes,
                &tail->tma_bar[st]);
    }
    issued_any |= 1u << st;
    issued_odd ^= 1u << st;
  };

  if (control) {
    if (lane == 0) {
      for (int st = 0; st < kFwdStages; ++st) mbar_init(&tail->tma_bar[st], 1);
      for (int p = 0; p < kRing; ++p) {
        mbar_init(&tail->stat_bar[p], 1);
        mbar_init(&tail->sum_bar[p], 1);
      }
      tail->fail = 0;
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    for (int st = 0; st < kFwdStages; ++st)
      if (q + st * Q < a.rows) issue(q + st * Q, st);
  }
  __syncthreads();
  cluster_sync();  // every CTA's mbarriers are initialised before any push

  const float beta = a.beta;
  bool ok = true;
  if (control) {
    // ------------------------------------------------------------------
    // Control warp.
    // ------------------------------------------------------------------
    struct RowStats {
      float4 g;  // m_s, Z_s, m_t, Z_t
      float Ks, Kt;
      bool bad_s, bad_t, row_ok;
    };
    // (C4) merge the workers' statistics partials of row i and push them
    auto push_stats = [&](int64_t i) {
      bar_sync(stat_part_bar(i), nthreads);
      if (tail->fail) ok = false;
      control_push_stats(tail->stat_part[i & 1], nw, tail, static_cast<int>(i % kRing), crank, csize);
    };
    // (C1) the cluster's statistics of row i, handed to the workers
    auto publish = [&](int64_t i) {
      const int slot = static_cast<int>(i % kRing), par = static_cast<int>(i & 1);
      RowStats rs;
      rs.g = make_float4(qnan(), qnan(), qnan(), qnan());
      if (ok) ok = control_wait(&tail->stat_bar[slot], static_cast<uint32_t>((i / kRing) & 1), csize);
      if (ok) {
        float4 v = make_float4(neg_inf(), 0.f, neg_inf(), 0.f);
        if (lane < static_cast<int>(csize)) v = *reinterpret_cast<const float4*>(tail->stat_slot[slot][lane]);
        const float2 ms = merge_warp(v.x, v.y), mt = merge_warp(v.z, v.w);
        rs.g = make_float4(ms.x, ms.y, mt.x, mt.y);
      }
      rs.bad_s = isnan(rs.g.y);
      rs.bad_t = isnan(rs.g.w);
      rs.row_ok = ok && !rs.bad_s && !rs.bad_t && rs.g.x != neg_inf() && rs.g.z != neg_inf();
      rs.Ks = rs.row_ok ? log2f(rs.g.y) : qnan();  // log2 Z
      rs.Kt = rs.row_ok ? log2f(rs.g.w) : qnan();
      if (lane == 0) {
        float* res = tail->stat_res[par];
        *reinterpret_cast<float4*>(res) = make_float4(-rs.g.x, -rs.g.z, -rs.Ks, -rs.Kt);
        *reinterpret_cast<float2*>(res + 4) = make_float2(rs.row_ok ? 1.f : 0.f, ok ? 1.f : 0.f);
      }
      bar_arrive(kBarStatReady, nthreads);
      return rs;
    };
    // (C3) the cluster's sums of row j (row r): the per-token value and saved statistics
    auto finish = [&](int64_t j, int64_t r, const RowStats& rs) {
      const int slot = static_cast<int>(j % kRing);
      float A = qnan(), B = qnan(), value = qnan();
      const bool got = ok && control_wait(&tail->sum_bar[slot], static_cast<uint32_t>((j / kRing) & 1), csize);
      if (!got) ok = false;
      if (got && rs.row_ok) {
        float2 v = make_float2(0.f, 0.f);
        if (lane < static_cast<int>(csize)) v = *reinterpret_cast<const float2*>(tail->sum_slot[slot][lane]);
        A = warp_sum(v.x);
        B = warp_sum(v.y);
        if (MODE == kInterior) {
          value = beta * A + (1.f - beta) * B;
        } else {
          value = A;  // +inf on a support violation
          A = MODE == kForwardKL ? value : 0.f;
          B = MODE == kForwardKL ? 0.f : value;
        }
      }
      if (lane == 0 && crank == 0) a.loss[r] = value;
      if (lane == 0 && crank == 0 && a.saved) {
        const float4 g = rs.g;
        float* sv = a.saved + r * VPD_SAVED_PAIR;
        sv[0] = rs.bad_s ? qnan() : g.x;
        sv[1] = rs.bad_s ? qnan() : (g.x == neg_inf() ? neg_inf() : (rs.row_ok ? kLn2 * rs.Ks : kLn2 * log2f(g.y)));
        sv[2] = rs.bad_t ? qnan() : g.z;
        sv[3] = rs.bad_t ? qnan() : (g.z == neg_inf() ? neg_inf() : (rs.row_ok ? kLn2 * rs.Kt : kLn2 * log2f(g.w)));
        sv[4] = A;
        sv[5] = B;
      }
    };
    // Rows whose sums are still to be taken: rows i - 2 (old) and i - 1 (new).
    RowStats old_s{}, new_s{};
    int64_t old_r = -1, new_r = -1;
    if (q < a.rows) push_stats(0);
    int64_t i = 0;
    for (int64_t r = q; r < a.rows; r += Q, ++i) {
      const int par = static_cast<int>(i & 1), slot = static_cast<int>(i % kRing);
      const bool has_next = r + Q < a.rows;

      // (C1) statistics of row i (pushed a row earlier) to the workers, who
      // take the row only if no wait gave up
      const RowStats cur = publish(i);
      const bool live = ok;
      // (C3) sums of row i - 2, in by now (every peer pushed them before the
      // statistics of row i that were just merged)
      if (old_r >= 0) finish(i - 2, old_r, old_s);
      old_r = -1;
      // (C4) statistics of row i + 1, which the workers computed before taking row i
      if (has_next) push_stats(i + 1);
      if (!live) break;

      // (C2) pass C of row i is in: refill its stage with row i + 3, push the sums
      bar_sync(kBarSumPart, nthreads);
      if (r + kFwdStages * Q < a.rows) issue(r + kFwdStages * Q, static_cast<int>(i % kFwdStages));
      {
        float2 v = make_float2(0.f, 0.f);
        if (lane < nw) v = *reinterpret_cast<const float2*>(tail->sum_part[par][lane]);
        const float sa = warp_sum(v.x), sb = warp_sum(v.y);
        if (lane < static_cast<int>(csize))
          push16(map_rank(smem_addr(tail->sum_slot[slot][crank]), lane), sa, sb, 0.f, 0.f,
                 map_rank(smem_addr(&tail->sum_bar[slot]), lane));
      }
      old_s = new_s;
      old_r = new_r;
      new_s = cur;
      new_r = r;
    }
    // the last two rows' sums
    if (old_r >= 0) finish(i - 2, old_r, old_s);
    if (new_r >= 0) finish(i - 1, new_r, new_s);
    // Copies still in flight (only after a wait gave up) must land before exit.
    if (lane == 0)
      for (int st = 0; st < kFwdStages; ++st)
        if ((issued_any >> st) & 1u) mbar_wait(&tail->tma_bar[st], ((issued_odd >> st) & 1u) ^ 1u);
  } else {
    // ------------------------------------------------------------------
    // Worker warps.
    // ------------------------------------------------------------------
    uint32_t tma_parity = 0;  // bit st: parity of the next wait on stage st
    const float2 ws2 = f2(1.f - beta), wt2 = f2(beta), tiny2 = f2(kTiny), l2e2 = f2(kLog2e);
    const int vt = 32 * vector_order(warp, nw, R) + lane;  // this thread's place in the vector order
    const Span sp = span_of<R>(len, Tw, vt);
    // statistics partial of row i from its stage
    auto stats_of = [&](int64_t i) {
      const int st = static_cast<int>(i % kFwdStages);
      if (bytes) {
        if (!mbar_wait(&tail->tma_bar[st], (tma_parity >> st) & 1u)) tail->fail = 1;
        tma_parity ^= 1u << st;
      }
      // the vectors stay in registers between the two sweeps for 16-bit
      // inputs (fp32 vectors are twice the registers)
      worker_stats<In, R, In::kSize == 2>(stage_ptr(st), W, sp, Tw, vt, tail->stat_part[i & 1][warp]);
      bar_arrive(stat_part_bar(i), nthreads);
    };
    if (q < a.rows) stats_of(0);
    int64_t i = 0;
    for (int64_t r = q; r < a.rows; r += Q, ++i) {
      const int par = static_cast<int>(i & 1);

      // (W3) statistics partial of row i + 1: its exchange travels during pass C of row i
      if (r + Q < a.rows) stats_of(i + 1);

      // (W1) global statistics of row i
      bar_sync(kBarStatReady, nthreads);
      const float4 st4 = *reinterpret_cast<const float4*>(tail->stat_res[par]);
      const float2 flags = *reinterpret_cast<const float2*>(tail->stat_res[par] + 4);
      if (flags.y == 0.f) break;
      const float2 nms2 = f2(st4.x), nmt2 = f2(st4.y), nKs2 = f2(st4.z), nKt2 = f2(st4.w);

      // (W2) pass C of row i from its stage, in log2 units
      float2 acc_a = f2(0.f), acc_b = f2(0.f);
      uint32_t viol = 0;
      if (flags.x != 0.f) {
        const unsigned char* ps = stage_ptr(static_cast<int>(i % kFwdStages)) + vt * kVB;
        const size_t tofs = static_cast<size_t>(W) * In::kSize;
#pragma unroll
        for (int k = 0; k < R; ++k) {
          if (k < sp.kv) {
            Word us[4], vs[4];
            In::words(In::ld(ps + k * Tw * kVB), us);
            In::words(In::ld(ps + tofs + k * Tw * kVB), vs);
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              if (MODE != kInterior) {
                const Word tgt = MODE == kForwardKL ? vs[w] : us[w];
                const Word oth = MODE == kForwardKL ? us[w] : vs[w];
                viol |= In::viol(tgt, oth);
              }
              const float2 lp = lam<In>(In::max2(us[w], In::neg_big_w()), nms2, l2e2, nKs2);
              const float2 lq = lam<In>(In::max2(vs[w], In::neg_big_w()), nmt2, l2e2, nKt2);
              const float2 p = ex2_2(lp), qv = ex2_2(lq);
              if (MODE == kInterior) {
                const float2 lm = lg2_2(fma2(ws2, p, fma2(wt2, qv, tiny2)));
                acc_b = fma2(p, add2(lp, neg(lm)), acc_b);
                acc_a = fma2(qv, add2(lq, neg(lm)), acc_a);
              } else {
                // forward KL(q || p): d = log2 q - log2 p weighted by q; reverse: mirror
                const float2 d = MODE == kForwardKL ? add2(lq, neg(lp)) : add2(lp, neg(lq));
                acc_a = fma2(MODE == kForwardKL ? qv : p, d, acc_a);
              }
            }
          }
        }
      }
      if constexpr (MODE == kInterior) {  // A partial on lanes 0-15, B partial on lanes 16-31
        const float v = kLn2 * warp_sum_pair(acc_a.x + acc_a.y, acc_b.x + acc_b.y);
        if ((lane & 15) == 0) tail->sum_part[par][warp][lane >> 4] = v;
      } else {
        float sa = kLn2 * warp_sum(acc_a.x + acc_a.y);
        if (__any_sync(0xffffffffu, viol != 0)) sa = pos_inf();
        if (lane == 0) *reinterpret_cast<float2*>(tail->sum_part[par][warp]) = make_float2(sa, 0.f);
      }
      bar_arrive(kBarSumPart, nthreads);
    }
  }

  __syncthreads();
  if (control && lane == 0 && (!ok || tail->fail)) atomicExch(&g_fused_error, 1);
  cluster_sync();  // no CTA leaves while a peer may still push into it
}

// ---------------------------------------------------------------------------
// Host side (per input dtype): one configuration, one launch.
// ---------------------------------------------------------------------------
struct Config {
  int C, R, W, nw;
  size_t smem;
};

// Shared memory of a slice width: both stages of both inputs, then the tail,
// and at least kMinSmem so that no two CTAs share an SM's tensor memory.
inline size_t smem_bytes(int W, bool gstage = false, int esize = 2) {
  const size_t s =
      static_cast<size_t>(kStages) * 2 * esize * W + (gstage ? static_cast<size_t>(4) * W : 0) + sizeof(Tail);
  return s < kMinSmem ? kMinSmem : s;
}
// The forward-only kernel: three stages, then the tail (one CTA per SM too).
inline size_t smem_bytes_fwd(int W, int esize = 2) {
  const size_t s = static_cast<size_t>(kFwdStages) * 2 * esize * W + sizeof(Tail);
  return s < kMinSmem ? kMinSmem : s;
}

// Launches the configured kernel; cudaErrorNotSupported (nothing launched)
// when no cluster of that shape can be resident. `clusters_out` reports the
// number of resident clusters.
// `fwd`: no gradient wanted, the forward-only kernel.
template <class In>
cudaError_t launch_typed(const FusedArgs& args, const Config& cfg, int mode, bool f32grad, bool fwd,
                         cudaStream_t stream, int* clusters_out);
// Resident clusters of C CTAs with nw worker warps (0 when none fit).
template <class In>
int resident_clusters(int C, int nw, size_t smem);

using Kernel = void (*)(FusedArgs);

// Cluster launch of `kern` (at most `maxw` worker warps) in shape `cfg`.
inline cudaError_t setup_one(Kernel kern, int maxw, const Config& cfg, cudaLaunchConfig_t* lc,
                             cudaLaunchAttribute* attr, int* clusters) {
  if (cfg.nw < 1 || cfg.nw > maxw) return cudaErrorNotSupported;
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
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cfg.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  lc->blockDim = dim3(32 * (cfg.nw + 1), 1, 1);
  lc->dynamicSmemBytes = cfg.smem;
  lc->attrs = attr;
  lc->numAttrs = 1;
  lc->gridDim = dim3(cfg.C, 1, 1);
  *clusters = 0;
  e = cudaOccupancyMaxActiveClusters(clusters, kern, lc);
  if (e != cudaSuccess || *clusters < 1) {
    cudaGetLastError();
    return cudaErrorNotSupported;
  }
  return cudaSuccess;
}

inline cudaError_t launch_kernel(Kernel kern, int maxw, const FusedArgs& args, const Config& cfg,
                                 cudaStream_t stream, int* clusters_out) {
  cudaLaunchConfig_t lc = {};
  cudaLaunchAttribute attr[1];
  int clusters = 0;
  cudaError_t e = setup_one(kern, maxw, cfg, &lc, attr, &clusters);
  if (e != cudaSuccess) return e;
  *clusters_out = clusters;
  const int64_t want = args.rows < clusters ? args.rows : clusters;
  lc.gridDim = dim3(static_cast<unsigned>(want * cfg.C), 1, 1);
  lc.stream = stream;
  return cudaLaunchKernelEx(&lc, kern, args);
}

template <class In, class G, int MODE>
cudaError_t launch_r(const FusedArgs& args, const Config& cfg, cudaStream_t stream, int* clusters) {
  switch (cfg.R) {
    case 1: return launch_kernel(k_jsd_fused<In, G, 1, MODE>, max_workers(1), args, cfg, stream, clusters);
    case 2: return launch_kernel(k_jsd_fused<In, G, 2, MODE>, max_workers(2), args, cfg, stream, clusters);
    case 3: return launch_kernel(k_jsd_fused<In, G, 3, MODE>, max_workers(3), args, cfg, stream, clusters);
    case 4:
      if (cfg.nw == kMaxWorkers && MODE == kInterior)
        return launch_kernel(k_jsd_fused<In, G, 4, MODE, kMaxWorkers>, max_workers(4), args, cfg, stream, clusters);
      return launch_kernel(k_jsd_fused<In, G, 4, MODE>, max_workers(4), args, cfg, stream, clusters);
    case 5: return launch_kernel(k_jsd_fused<In, G, 5, MODE>, max_workers(5), args, cfg, stream, clusters);
  }
  return cudaErrorNotSupported;
}

template <class In, int MODE>
cudaError_t launch_fwd(const FusedArgs& args, const Config& cfg, cudaStream_t stream, int* clusters) {
  switch (cfg.R) {
    case 1: return launch_kernel(k_jsd_fused_fwd<In, 1, MODE>, kMaxWorkersFwd, args, cfg, stream, clusters);
    case 2: return launch_kernel(k_jsd_fused_fwd<In, 2, MODE>, kMaxWorkersFwd, args, cfg, stream, clusters);
    case 3:
      if (cfg.nw == kMaxWorkersFwd)
        return launch_kernel(k_jsd_fused_fwd<In, 3, MODE, kMaxWorkersFwd>, kMaxWorkersFwd, args, cfg, stream,
                             clusters);
      return launch_kernel(k_jsd_fused_fwd<In, 3, MODE>, kMaxWorkersFwd, args, cfg, stream, clusters);
    case 4: return launch_kernel(k_jsd_fused_fwd<In, 4, MODE>, kMaxWorkersFwd, args, cfg, stream, clusters);
    case 5: return launch_kernel(k_jsd_fused_fwd<In, 5, MODE>, kMaxWorkersFwd, args, cfg, stream, clusters);
  }
  return cudaErrorNotSupported;
}

template <class In>
cudaError_t launch_typed(const FusedArgs& args, const Config& cfg, int mode, bool f32grad, bool fwd,
                         cudaStream_t stream, int* clusters) {
  if (fwd) {
    if (mode == kForwardKL) return launch_fwd<In, kForwardKL>(args, cfg, stream, clusters);
    if (mode == kReverseKL) return launch_fwd<In, kReverseKL>(args, cfg, stream, clusters);
    return launch_fwd<In, kInterior>(args, cfg, stream, clusters);
  }
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

template <class In>
int resident_clusters(int C, int nw, size_t smem) {
  Config cfg{C, 1, 8, nw, smem};
  cudaLaunchConfig_t lc = {};
  cudaLaunchAttribute attr[1];
  int clusters = 0;
  if (setup_one(k_jsd_fused<In, GF32, 1, kInterior>, max_workers(1), cfg, &lc, attr, &clusters) != cudaSuccess)
    return 0;
  return clusters;
}

}  // namespace fused
}  // namespace vpd
