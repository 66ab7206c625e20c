// vpd_linear.cu -- the fused-linear generalized JSD: student and teacher
// logits s = h_s W_s^T and t = h_t W_t^T are formed tile by tile on the
// tensor cores (tcgen05.mma, bf16 operands staged by TMA, fp32 accumulators in
// tensor memory) and consumed in the epilogue, so the [N, V] logits are never
// written to memory.
//
// Sources (web pages):
//   [JSD page] DeepSpeed pull request #8958, "[VocabTP] Add vocabulary-parallel
//              generalized JSD with Triton kernels": section Scope and
//              limitations names the fused-linear divergence as not included
//              and explains why JSD needs the statistics before the divergence.
//   [ops page] DeepSpeed pull request #8791, "Add vocabulary-parallel logprobs,
//              entropy and KL ops": section Limitations, the fused-linear
//              variant as future work; section How, the (max, sum-exp) merge.
//
// One persistent kernel, k_linear, in four epilogue modes:
//   kStats  logits tiles of both heads -> online (max, sum-exp) per row over
//           the unit's vocabulary tiles -> partials per (vocabulary chunk,
//           column part, row);
//   kDiv    logits tiles again -> the two KL-to-mixture partial sums with the
//           merged statistics (the second of the two passes JSD needs);
//   kGrad   logits tiles again -> dS and dT of a chunk of rows, each split into
//           a bf16 high part and a bf16 low part (x = hi + lo to 16 bits of
//           mantissa) and stored row-major: each epilogue warp stages 32 x 32
//           blocks in shared memory and one lane writes them out with TMA
//           tensor stores;
//   kGemm   a plain C += A B^T over one or two (A, B) operand pairs (used for
//           dh = dS W and dW = dS^T h from the split gradients, hi and lo as the
//           two pairs; for dW the A operand is the same row-major dS, read
//           MN-major), split along K, accumulated into fp32 C by atomics.
// Small kernels merge the per-chunk partials and transpose the chunk's hidden
// states for dW.
//
// Warp roles of k_linear (one instantiation per mode): warp 0 issues the TMA
// loads into a ring of shared-memory stages; warp 1 issues the MMAs (one
// elected lane) into one of two tensor-memory accumulator buffers; the other
// warps are the epilogue, eight (320 threads) or, in kDiv, sixteen (576), that
// is two or four per TMEM lane quarter: thread i owns TMEM lane (and tile
// row) 32 (warp % 4) + lane and one half (one quarter) of each tile's columns.
// Stages hand over through mbarriers (TMA completion -> MMA; tcgen05.commit ->
// producer), and so do the accumulator buffers (commit -> epilogue; epilogue
// arrivals -> MMA), so the epilogue of one tile overlaps the MMAs of the next
// wherever two tiles fit in tensor memory (kStats and kGemm); in kDiv and
// kGrad the s and t tiles of 256 columns fill it, and each epilogue warp hands
// the accumulator back once its last columns are in registers.
// Every mbarrier wait gives up after two seconds, sets the device error word
// and leaves the loops; the CTA waits for copies and MMAs in flight before it
// frees its tensor memory.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "vpd_internal.h"
#include "vpd_linear.h"

namespace vpd {
namespace linear {

constexpr int BM = 128;                     // tile rows (tensor-memory lanes)
constexpr int BN = 256;                     // widest tile: one 128 x 256 MMA per 16 of k
constexpr int BK = 64;                      // k per stage: one 128-byte swizzle row of bf16
constexpr int kTileBytes = BM * BK * 2;     // 16 KB: the A tile of a stage
constexpr int kRingBytes = 4 * (kTileBytes + BN * BK * 2);  // stage ring: 4 of 48 KB (256 columns) or 6 of 32 KB (128)
constexpr int kMaxStages = 6;
// Tile columns of every pass: 256. The statistics pass takes one head's tile
// at a time, in two buffers, and the GEMMs two buffers. The divergence and
// gradient passes need both heads' logits of a tile at once: s and t of one
// 256-column tile fill the tensor memory, so their epilogue overlaps the next
// tile's MMAs only from each warp's last columns on; 128-column tiles, two of
// which fit, overlap fully but draw a third more operand bytes from L2 per
// flop, which costs more than the overlap saves.
constexpr int kGradTN = 256;  // the gradient pass's tile columns (its W maps' box rows)
template <int TN>
struct TileShape {
  static constexpr int kBBytes = TN * BK * 2;             // the B tile of a stage
  static constexpr int kStageBytes = kTileBytes + kBBytes;
  static constexpr int kStages = kRingBytes / kStageBytes;
  static_assert(kStages <= kMaxStages && kStages * kStageBytes <= kRingBytes, "stage ring");
  // instruction descriptor of kind::f16: fp32 accumulator (bits 4-5 = 1),
  // bf16 A and B (bits 7-9, 10-12 = 1), both K-major, N >> 3 at bits 17-22,
  // M >> 4 at bits 24-28
  static constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((TN >> 3) << 17) | ((BM >> 4) << 24);
};
// Gradient pass output blocks: each epilogue warp stages a 32 x 32 bf16 block
// row-major (rows of 64 bytes, 64-byte swizzle) for one tensor store.
constexpr int kStoreBlockBytes = 32 * 64;
constexpr int kStoreWarpBytes = kStoreBlockBytes;
constexpr int kTmemCols = 512;
constexpr float kTinyL = 1e-37f;
constexpr float kLog2eL = 1.4426950408889634f;
constexpr float kLn2L = 0.6931471805599453f;
constexpr uint64_t kWaitNs = 2000000000ull;

enum Mode : int { kStats = 0, kDiv = 1, kGrad = 2, kGemm = 3 };

// Epilogue warps per mode: kParts per tensor-memory lane quarter, each taking
// 1 / kParts of a tile's columns. The divergence pass, whose epilogue overlaps
// the next tile's MMAs only at its end (its s and t tiles fill the tensor
// memory), runs sixteen (at most 96 registers a thread: five warps per SM
// sub-partition); the others run eight (the gradient pass, in the same
// position, needs more registers than sixteen warps leave).
template <int MODE>
struct EpiShape {
  static constexpr int kWarps = MODE == kDiv ? 16 : 8;
  static constexpr int kParts = kWarps / 4;
  static constexpr int kThreads = 32 * (2 + kWarps);
};
// Dynamic shared memory: the stage ring, the per-warp output blocks of the
// gradient pass, and slack for the 1024-byte alignment.
template <int TN, int MODE>
constexpr int smem_bytes() {
  return TileShape<TN>::kStages * TileShape<TN>::kStageBytes +
         (MODE == kGrad ? EpiShape<MODE>::kWarps * kStoreWarpBytes : 0) + 1024;
}

// Tensor maps of the gradient pass's outputs, per head: the row-major high and
// low parts (boxes of 32 x 32).
struct StoreMaps {
  CUtensorMap m[2][2];
};

static __device__ int g_linear_error = 0;

struct Args {
  int mode;
  int jmode;          // 0 interior, 1 forward KL (beta = 0), 2 reverse KL (beta = 1)
  int64_t rows;       // valid rows of the A operands (M)
  int64_t cols;       // valid columns of the output (V for the JSD modes, the N of C for kGemm)
  int nk0, nk1;       // k-blocks of operand pair 0 and 1 (nk1 = 0: one pair)
  int mtiles, ntiles;
  int tiles_per_unit; // JSD modes: vocabulary tiles per work unit
  int ksplit;         // kGemm: parts of the k range
  int64_t units;
  float beta;
  // JSD modes
  const float* saved;      // [rows, 6] merged statistics and sums (kDiv, kGrad)
  const float* loss;       // [rows] (kGrad, endpoint branches)
  const float* grad_loss;  // [rows] or NULL (kGrad)
  float* part;             // [chunks, rows, 4] (kStats) / [chunks, rows, 2] (kDiv)
  // kGrad outputs, chunk-local, row-major [rows, cols] (NULL: head not wanted)
  __nv_bfloat16 *gs_hi, *gs_lo;
  __nv_bfloat16 *gt_hi, *gt_lo;
  // kGemm output
  float* C;
  int64_t ldc;
  int gemm_store;  // 1: C = the product (one k part, nothing to add to); 0: C += by atomics
  int a_mn;        // kGemm: the A operands are stored [K, M] (M contiguous) and read MN-major
  int b_mn;        // kGemm: the B operand is stored [K, N] (N contiguous) and read MN-major
};

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t saddr(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }
__device__ __forceinline__ uint64_t now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mb_init(uint64_t* b, uint32_t n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(b)), "r"(n) : "memory");
}
__device__ __forceinline__ void mb_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mb_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(saddr(b)) : "memory");
}
__device__ __forceinline__ bool mb_try(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(saddr(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for the phase of `parity`, giving up after kWaitNs or when another role
// has already given up.
__device__ __forceinline__ bool mb_wait(uint64_t* b, uint32_t parity, volatile int* abort) {
  if (mb_try(b, parity)) return true;
  const uint64_t t0 = now_ns();
  while (true) {
    if (mb_try(b, parity)) return true;
    if (*abort || now_ns() - t0 > kWaitNs) return false;
  }
}
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          saddr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(saddr(bar))
      : "memory");
}
// Tensor store of a staged shared-memory box to (x, y) of the map's tensor
// (the part inside the tensor's bounds), tracked by the issuing thread's bulk groups.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(saddr(src))
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_async_shared() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tmem_alloc_all(uint32_t* slot) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(slot)), "n"(kTmemCols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_free_all(uint32_t base) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "n"(kTmemCols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Shared-memory matrix descriptor of a K-major bf16 tile stored as rows of 128
// bytes with the 128-byte swizzle (the layout TMA writes for a {64, rows} box):
// 8-row groups 1024 bytes apart (stride byte offset), leading byte offset
// unused for this layout, fixed version bits 0b001 at 46-48, swizzle mode 2.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr) {
  uint64_t d = static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(16u >> 4) << 16;
  d |= static_cast<uint64_t>(1024u >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}
// The same for an MN-major bf16 tile written by two TMA boxes of {64, 64}
// with the 128-byte swizzle: rows of 128 bytes hold 64 consecutive M (or N)
// elements, one row per k; 8-row k groups 1024 bytes apart (stride byte
// offset), the second 64 elements of M 8192 bytes on (leading byte offset).
__device__ __forceinline__ uint64_t sw128_mn_desc(uint32_t addr) {
  uint64_t d = static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(8192u >> 4) << 16;
  d |= static_cast<uint64_t>(1024u >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}
__device__ __forceinline__ void mma_bf16_rt(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
template <uint32_t kIdesc>
__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(kIdesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(saddr(bar))
               : "memory");
}
// 32 consecutive fp32 columns of this thread's lane, waited for in the same statement.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2f(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float ninf() { return __int_as_float(0xff800000); }
// fp32x2: one packed instruction for two values
__device__ __forceinline__ float2 pk(float a, float b) { return make_float2(a, b); }
__device__ __forceinline__ float2 pk_add(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 pk_sub(float2 a, float2 b) { return __fadd2_rn(a, make_float2(-b.x, -b.y)); }
__device__ __forceinline__ float2 pk_fma(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 pk_ex2(float2 a) { return make_float2(ex2f(a.x), ex2f(a.y)); }
__device__ __forceinline__ float2 pk_lg2(float2 a) { return make_float2(lg2f(a.x), lg2f(a.y)); }

// ---------------------------------------------------------------------------
// The sequence of work every role walks through in the same order.
// ---------------------------------------------------------------------------
struct Unit {
  int mt;        // row tile
  int nt0, nt1;  // column tiles [nt0, nt1)
  int kb0, kb1;  // kGemm: k-blocks [kb0, kb1) of the concatenated pairs
  int chunk;     // JSD modes: vocabulary chunk index
};

__device__ __forceinline__ Unit unit_of(const Args& a, int64_t u) {
  Unit w;
  if (a.mode == kGemm) {
    // the column tiles of one row tile are neighbours in the unit order, so
    // the CTAs that run them at the same time share the A tile through L2
    // (A is read from DRAM once, not once per column tile)
    w.nt0 = static_cast<int>(u % a.ntiles);
    w.nt1 = w.nt0 + 1;
    const int64_t rest = u / a.ntiles;
    w.mt = static_cast<int>(rest % a.mtiles);
    const int ks = static_cast<int>(rest / a.mtiles);
    const int nk = a.nk0 + a.nk1;
    w.kb0 = static_cast<int>(static_cast<int64_t>(nk) * ks / a.ksplit);
    w.kb1 = static_cast<int>(static_cast<int64_t>(nk) * (ks + 1) / a.ksplit);
    w.chunk = 0;
  } else {
    w.mt = static_cast<int>(u % a.mtiles);
    w.chunk = static_cast<int>(u / a.mtiles);
    w.nt0 = w.chunk * a.tiles_per_unit;
    w.nt1 = w.nt0 + a.tiles_per_unit < a.ntiles ? w.nt0 + a.tiles_per_unit : a.ntiles;
    w.kb0 = 0;
    w.kb1 = a.nk0 + a.nk1;
  }
  return w;
}

struct __align__(8) Bars {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint32_t tmem_base;
  int abort;
};

template <int TN, int MODE>
__global__ void __launch_bounds__(EpiShape<MODE>::kThreads, 1)
    k_linear(const __grid_constant__ CUtensorMap a0, const __grid_constant__ CUtensorMap b0,
             const __grid_constant__ CUtensorMap a1, const __grid_constant__ CUtensorMap b1, Args a,
             const __grid_constant__ StoreMaps gm) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ Bars bars;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  using S = TileShape<TN>;
  using E = EpiShape<MODE>;
  constexpr int kStages = S::kStages, kStageBytes = S::kStageBytes;
  uint8_t* oblk = smem + kStages * kStageBytes;  // kGrad output blocks
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort = &bars.abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mb_init(&bars.full[s], 1);
      mb_init(&bars.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mb_init(&bars.acc_full[b], 1);
      mb_init(&bars.acc_empty[b], E::kWarps);
    }
    bars.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  if (warp == 0) tmem_alloc_all(&bars.tmem_base);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;
  constexpr bool gemm = MODE == kGemm;
  constexpr bool split = MODE == kStats;  // the two heads' tiles one after the other
  // two accumulator buffers in turn (else one buffer holds s and t of a tile)
  constexpr bool dbuf = gemm || split || TN < BN;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int64_t u = blockIdx.x; u < a.units && ok; u += gridDim.x) {
        const Unit w = unit_of(a, u);
        for (int nt = w.nt0; nt < w.nt1 && ok; ++nt) {
          for (int kb = w.kb0; kb < w.kb1; ++kb) {
            if (!mb_wait(&bars.empty[stage], phase ^ 1u, abort)) {
              ok = false;
              break;
            }
            const bool second = kb >= a.nk0;
            const int kk = second ? kb - a.nk0 : kb;
            uint8_t* sa = smem + stage * kStageBytes;
            mb_expect_tx(&bars.full[stage], kStageBytes);
            if (gemm && a.a_mn) {  // A stored [K, M]: two boxes of 64 M x 64 k
              tma_load_2d(sa, second ? &a1 : &a0, w.mt * BM, kk * BK, &bars.full[stage]);
              tma_load_2d(sa + kTileBytes / 2, second ? &a1 : &a0, w.mt * BM + 64, kk * BK, &bars.full[stage]);
            } else {
              tma_load_2d(sa, second ? &a1 : &a0, kk * BK, w.mt * BM, &bars.full[stage]);
            }
            if (gemm && a.b_mn) {  // B stored [K, N]: TN / 64 boxes of 64 N x 64 k
#pragma unroll
              for (int i = 0; i < TN / 64; ++i)
                tma_load_2d(sa + kTileBytes + i * (kTileBytes / 2), second ? &b1 : &b0, nt * TN + 64 * i, kk * BK,
                            &bars.full[stage]);
            } else {
              tma_load_2d(sa + kTileBytes, second ? &b1 : &b0, kk * BK, nt * TN, &bars.full[stage]);
            }
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      if (!ok) bars.abort = 1;
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int buf = 0;
      uint32_t acc_phase[2] = {0, 0};
      bool ok = true;
      for (int64_t u = blockIdx.x; u < a.units && ok; u += gridDim.x) {
        const Unit w = unit_of(a, u);
        for (int nt = w.nt0; nt < w.nt1 && ok; ++nt) {
         // the statistics mode treats the two heads' tiles as two tiles in
         // alternating buffers (its epilogue needs them one at a time), so one
         // head's epilogue overlaps the other head's MMAs
         int kbs = w.kb0;
         for (int sub = 0; sub < (split ? 2 : 1) && ok; ++sub) {
          const int kbe = split ? (sub == 0 ? a.nk0 : a.nk0 + a.nk1) : w.kb1;
          if (!mb_wait(&bars.acc_empty[buf], acc_phase[buf] ^ 1u, abort)) {
            ok = false;
            break;
          }
          acc_phase[buf] ^= 1u;
          tc_fence_after();
          // kGemm and kStats: one of two 256-column accumulators; the other
          // JSD modes: S at columns 0 .. TN-1 and T at TN .. 2 TN - 1 of one of
          // two buffers (TN = 128) or of the one buffer (TN = 256)
          const uint32_t acc0 = tmem + 256u * buf;
          for (int kb = kbs; kb < kbe; ++kb) {
            if (!mb_wait(&bars.full[stage], phase, abort)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const bool second = kb >= a.nk0;
            const uint32_t dst = (!gemm && !split && second) ? acc0 + TN : acc0;
            // accumulate unless this is the first k-block into this accumulator
            const bool first = (gemm || split) ? kb == kbs : (second ? kb == a.nk0 : kb == 0);
            const uint32_t sa = saddr(smem + stage * kStageBytes);
            if (gemm && (a.a_mn || a.b_mn)) {
              // an MN-major operand (transpose bit 15 for A, 16 for B): 16 k per
              // MMA = two 8-row groups, 2048 bytes: +128 in the address field
              // (a K-major one: 32 bytes, +2)
              const uint64_t da = a.a_mn ? sw128_mn_desc(sa) : sw128_desc(sa);
              const uint64_t db = a.b_mn ? sw128_mn_desc(sa + kTileBytes) : sw128_desc(sa + kTileBytes);
              const uint32_t sta = a.a_mn ? 128u : 2u, stb = a.b_mn ? 128u : 2u;
              const uint32_t idesc = S::kIdesc | (a.a_mn ? 1u << 15 : 0u) | (a.b_mn ? 1u << 16 : 0u);
#pragma unroll
              for (int k = 0; k < BK / 16; ++k)
                mma_bf16_rt(dst, da + sta * k, db + stb * k, idesc, (first && k == 0) ? 0u : 1u);
            } else {
              const uint64_t db = sw128_desc(sa + kTileBytes);
              const uint64_t da = sw128_desc(sa);
#pragma unroll
              for (int k = 0; k < BK / 16; ++k)  // 16 bf16 = 32 bytes per MMA: +2 in the address field
                mma_bf16<S::kIdesc>(dst, da + 2u * k, db + 2u * k, (first && k == 0) ? 0u : 1u);
            }
            mma_commit(&bars.empty[stage]);
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          mma_commit(&bars.acc_full[buf]);
          if (dbuf) buf ^= 1;
          kbs = kbe;
         }
        }
      }
      if (!ok) bars.abort = 1;
    }
  } else {
    // ---------------- epilogue (warps 2-9) ----------------
    const int q = warp & 3;                     // lane quarter of tensor memory
    const int part = (warp - 2) >> 2;           // which 1 / kParts of each tile's columns
    constexpr int kPartCols = TN / E::kParts;
    const int rloc = 32 * q + lane;             // row within the tile
    const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
    int buf = 0;
    uint32_t acc_phase[2] = {0, 0};
    bool ok = true;
    const float beta = a.beta;
    for (int64_t u = blockIdx.x; u < a.units && ok; u += gridDim.x) {
      const Unit w = unit_of(a, u);
      const int64_t row = static_cast<int64_t>(w.mt) * BM + rloc;
      const bool rv = row < a.rows;
      // per-row state
      float ms = ninf(), zs = 0.f, mt = ninf(), zt = 0.f;  // kStats
      float accA = 0.f, accB = 0.f;                       // kDiv (log2 units)
      float nms = 0.f, nmt = 0.f, nKs = 0.f, nKt = 0.f;   // -m, -L log2 e
      float cs = 0.f, ct = 0.f, ks_ = 0.f, kt_ = 0.f;     // kGrad coefficients
      bool live = false;
      if (!gemm && MODE != kStats && rv) {
        const float* sv = a.saved + row * 6;
        nms = -sv[0];
        nKs = -sv[1] * kLog2eL;
        nmt = -sv[2];
        nKt = -sv[3] * kLog2eL;
        live = isfinite(sv[0]) && isfinite(sv[1]) && isfinite(sv[2]) && isfinite(sv[3]);
        if (MODE == kGrad) {
          const float g = a.grad_loss ? a.grad_loss[row] : 1.f;
          const float A = sv[4], B = sv[5], value = a.loss[row];
          live = live && isfinite(value);
          if (a.jmode == 0) {
            cs = g * (1.f - beta);
            ct = g * beta;
            ks_ = -cs * B;
            kt_ = -ct * A;
          } else {
            cs = ct = g;
            ks_ = -g * value;
            kt_ = -g * value;
          }
        }
      }
      for (int nt = w.nt0; nt < w.nt1 && ok; ++nt) {
       for (int sub = 0; sub < (split ? 2 : 1); ++sub) {
        // every lane waits; the warp goes on only together (the tensor-memory
        // loads below are warp-collective)
        if (!__all_sync(0xffffffffu, mb_wait(&bars.acc_full[buf], acc_phase[buf], abort))) {
          ok = false;
          break;
        }
        acc_phase[buf] ^= 1u;
        tc_fence_after();
        const uint32_t accS = tmem + lane_addr + 256u * buf;  // buf stays 0 with one buffer
        const int64_t col0 = static_cast<int64_t>(nt) * TN;
        bool released = false;  // this warp's accumulator columns handed back already
        for (int c = part * kPartCols; c < (part + 1) * kPartCols; c += 32) {
          float x[32];
          tmem_ld32(accS + c, x);
          if (gemm) {
            if (rv) {
              float* crow = a.C + row * a.ldc;
#pragma unroll
              for (int i = 0; i < 32; i += 4) {
                const int64_t j = col0 + c + i;
                if (j + 3 < a.cols) {
                  const float4 v4 = make_float4(x[i], x[i + 1], x[i + 2], x[i + 3]);
                  if (a.gemm_store) *reinterpret_cast<float4*>(crow + j) = v4;
                  else atomicAdd(reinterpret_cast<float4*>(crow + j), v4);
                } else {
                  for (int e = 0; e < 4; ++e)
                    if (j + e < a.cols) {
                      if (a.gemm_store) crow[j + e] = x[i + e];
                      else atomicAdd(crow + j + e, x[i + e]);
                    }
                }
              }
            }
            continue;
          }
          const int nvalid = static_cast<int>(a.cols - (col0 + c) < 32 ? a.cols - (col0 + c) : 32);
          if (split) {  // kStats: one head's tile, online (max, sum-exp)
            float m = sub == 0 ? ms : mt;
            float z = sub == 0 ? zs : zt;
            float cm = ninf();
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (i < nvalid) cm = fmaxf(cm, x[i]);
            if (cm > m) {
              z = m == ninf() ? 0.f : z * expf(m - cm);
              m = cm;
            }
            float e = 0.f;
            if (nvalid >= 32) {  // two columns per packed instruction
              const float2 nm2 = pk(-m, -m), l2e2 = pk(kLog2eL, kLog2eL);
              float2 e2 = pk(0.f, 0.f);
#pragma unroll
              for (int i = 0; i < 32; i += 2) e2 = pk_add(e2, pk_ex2(__fmul2_rn(pk_add(pk(x[i], x[i + 1]), nm2), l2e2)));
              e = e2.x + e2.y;
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (i < nvalid) e += ex2f((x[i] - m) * kLog2eL);
            }
            z += e;
            if (sub == 0) {
              ms = m;
              zs = z;
            } else {
              mt = m;
              zt = z;
            }
            continue;
          }
          float y[32];
          tmem_ld32(accS + TN + c, y);
          if (!dbuf && c + 32 >= (part + 1) * kPartCols) {
            // one buffer (s and t fill the tensor memory): once the last
            // columns are in registers, the MMAs of the next tile may start
            // while this chunk is computed
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mb_arrive(&bars.acc_empty[buf]);
            released = true;
          }
          if (MODE == kDiv) {
            if (!live) continue;
            // two columns per packed instruction; columns past the vocabulary
            // (logits 0 from the zero-filled head rows) get p = q = 0
            const float2 nms2 = pk(nms, nms), nmt2 = pk(nmt, nmt), nKs2 = pk(nKs, nKs), nKt2 = pk(nKt, nKt);
            const float2 l2e2 = pk(kLog2eL, kLog2eL), ws2 = pk(1.f - beta, 1.f - beta), wt2 = pk(beta, beta);
            const float2 tiny2 = pk(kTinyL, kTinyL);
            float2 accA2 = pk(0.f, 0.f), accB2 = pk(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const float2 lp = pk_fma(pk_add(pk(x[i], x[i + 1]), nms2), l2e2, nKs2);
              const float2 lq = pk_fma(pk_add(pk(y[i], y[i + 1]), nmt2), l2e2, nKt2);
              float2 p = pk_ex2(lp), qv = pk_ex2(lq);
              if (nvalid < 32) {  // warp-uniform: the ragged last tile only
                if (i >= nvalid) p.x = qv.x = 0.f;
                if (i + 1 >= nvalid) p.y = qv.y = 0.f;
              }
              if (a.jmode == 0) {
                const float2 lm = pk_lg2(pk_fma(ws2, p, pk_fma(wt2, qv, tiny2)));
                accA2 = pk_fma(qv, pk_sub(lq, lm), accA2);
                accB2 = pk_fma(p, pk_sub(lp, lm), accB2);
              } else if (a.jmode == 1) {
                accA2 = pk_fma(qv, pk_sub(lq, lp), accA2);
              } else {
                accB2 = pk_fma(p, pk_sub(lp, lq), accB2);
              }
            }
            accA += accA2.x + accA2.y;
            accB += accB2.x + accB2.y;
          } else {  // kGrad
            // dS and dT of this thread's row for 32 columns (0 on rows that
            // carry no value; rows past the chunk are not stored)
            float gsv[32], gtv[32];
            const bool want_t = a.gt_hi != nullptr;  // warp-uniform: dT wanted
            const float2 nms2 = pk(nms, nms), nmt2 = pk(nmt, nmt), nKs2 = pk(nKs, nKs), nKt2 = pk(nKt, nKt);
            const float2 l2e2 = pk(kLog2eL, kLog2eL), ws2 = pk(1.f - beta, 1.f - beta), wt2 = pk(beta, beta);
            const float2 tiny2 = pk(kTinyL, kTinyL), cs2 = pk(cs, cs), ct2 = pk(ct, ct);
            const float2 csl2 = pk(cs * kLn2L, cs * kLn2L), ctl2 = pk(ct * kLn2L, ct * kLn2L);
            const float2 ks2 = pk(ks_, ks_), kt2 = pk(kt_, kt_);
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              float2 gs = pk(0.f, 0.f), gt = pk(0.f, 0.f);
              if (live) {
                const float2 lp = pk_fma(pk_add(pk(x[i], x[i + 1]), nms2), l2e2, nKs2);
                const float2 lq = pk_fma(pk_add(pk(y[i], y[i + 1]), nmt2), l2e2, nKt2);
                const float2 p = pk_ex2(lp), qv = pk_ex2(lq);
                if (a.jmode == 0) {
                  const float2 lm = pk_lg2(pk_fma(ws2, p, pk_fma(wt2, qv, tiny2)));
                  gs = __fmul2_rn(p, pk_fma(csl2, pk_sub(lp, lm), ks2));
                  if (want_t) gt = __fmul2_rn(qv, pk_fma(ctl2, pk_sub(lq, lm), kt2));
                } else if (a.jmode == 1) {  // dS = g (p - q), dT = g q (ln q - ln p - KL)
                  gs = __fmul2_rn(cs2, pk_sub(p, qv));
                  if (want_t) gt = __fmul2_rn(qv, pk_fma(ctl2, pk_sub(lq, lp), kt2));
                } else {  // dS = g p (ln p - ln q - KL), dT = g (q - p)
                  gs = __fmul2_rn(p, pk_fma(csl2, pk_sub(lp, lq), ks2));
                  if (want_t) gt = __fmul2_rn(ct2, pk_sub(qv, p));
                }
                if (nvalid < 32) {  // warp-uniform: the ragged last tile only
                  if (i >= nvalid) gs.x = gt.x = 0.f;
                  if (i + 1 >= nvalid) gs.y = gt.y = 0.f;
                }
              }
              gsv[i] = gs.x;
              gsv[i + 1] = gs.y;
              gtv[i] = gt.x;
              gtv[i + 1] = gt.y;
            }
            const int64_t rbase = static_cast<int64_t>(w.mt) * BM + 32 * q;  // this warp's first row
            // This warp's block: lane = its row (16-byte piece j of the 64-byte
            // row at j ^ ((row >> 1) & 3), the 64-byte swizzle).
            uint8_t* blk = oblk + (warp - 2) * kStoreWarpBytes;
            uint4* rmb = reinterpret_cast<uint4*>(blk + lane * 64);
            const int swz = (lane >> 1) & 3;
            // warp-uniform: nothing to store past the chunk's rows or the vocabulary
            const bool store = rbase < a.rows && nvalid > 0;
#pragma unroll
            for (int head = 0; head < 2; ++head) {
              const float* gv = head == 0 ? gsv : gtv;
              if (!(head == 0 ? a.gs_hi : a.gt_hi) || !store) continue;  // warp-uniform
              uint32_t part[2][16];  // high and low bf16 parts, packed in pairs
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const __nv_bfloat162 h = __floats2bfloat162_rn(gv[2 * i], gv[2 * i + 1]);
                const float2 lf = pk_sub(pk(gv[2 * i], gv[2 * i + 1]), __bfloat1622float2(h));
                const __nv_bfloat162 l = __floats2bfloat162_rn(lf.x, lf.y);
                part[0][i] = *reinterpret_cast<const uint32_t*>(&h);
                part[1][i] = *reinterpret_cast<const uint32_t*>(&l);
              }
#pragma unroll
              for (int hl = 0; hl < 2; ++hl) {
                // the block is free once the previous store has read it
                if (lane == 0) bulk_wait_read_all();
                __syncwarp();
#pragma unroll
                for (int j = 0; j < 4; ++j)
                  rmb[j ^ swz] = make_uint4(part[hl][4 * j], part[hl][4 * j + 1], part[hl][4 * j + 2], part[hl][4 * j + 3]);
                fence_async_shared();
                __syncwarp();
                // [rows, V] at (column col0 + c, row rbase); the map clips the
                // block to the rows and columns that exist
                if (lane == 0) {
                  tma_store_2d(&gm.m[head][hl], blk, static_cast<int>(col0 + c), static_cast<int>(rbase));
                  bulk_commit();
                }
              }
            }
          }
        }
        if (!released) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mb_arrive(&bars.acc_empty[buf]);
        }
        if (dbuf) buf ^= 1;
       }
      }
      if (!ok) break;
      if (rv && MODE == kStats) {
        // one partial per (chunk, column part, row)
        reinterpret_cast<float4*>(a.part)[(E::kParts * static_cast<int64_t>(w.chunk) + part) * a.rows + row] =
            make_float4(ms, zs, mt, zt);
      } else if (rv && MODE == kDiv) {
        reinterpret_cast<float2*>(a.part)[(E::kParts * static_cast<int64_t>(w.chunk) + part) * a.rows + row] =
            make_float2(accA, accB);
      }
    }
    if (!ok) bars.abort = 1;
    // the output blocks' tensor stores finish before the shared memory goes
    if (MODE == kGrad && lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (bars.abort) {
    // a wait gave up: let copies and MMAs already issued land before the
    // shared and tensor memory are released
    const uint64_t t0 = now_ns();
    while (now_ns() - t0 < 10000000ull) {
    }
    if (threadIdx.x == 0) atomicExch(&g_linear_error, 1);
  }
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_free_all(tmem);
  }
}

// Per row: merge the (m, z) partials of both heads over the vocabulary chunks
// in chunk order (MAX of maxima, SUM of sums rescaled to it) and store
// (m_s, ln Z_s, m_t, ln Z_t) in `saved`.
__global__ void k_linear_merge_stats(const float4* part, int chunks, int64_t rows, float* saved) {
  const int64_t r = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  if (r >= rows) return;
  float ms = ninf(), mt = ninf();
  for (int c = 0; c < chunks; ++c) {
    const float4 p = part[c * rows + r];
    ms = fmaxf(ms, p.x);
    mt = fmaxf(mt, p.z);
  }
  float zs = 0.f, zt = 0.f;
  for (int c = 0; c < chunks; ++c) {
    const float4 p = part[c * rows + r];
    if (p.x != ninf()) zs += p.y * expf(p.x - ms);
    if (p.z != ninf()) zt += p.w * expf(p.z - mt);
  }
  float* sv = saved + r * 6;
  const bool bad_s = !isfinite(ms) || !isfinite(zs), bad_t = !isfinite(mt) || !isfinite(zt);
  sv[0] = bad_s ? __int_as_float(0x7fffffff) : ms;
  sv[1] = bad_s ? __int_as_float(0x7fffffff) : logf(zs);
  sv[2] = bad_t ? __int_as_float(0x7fffffff) : mt;
  sv[3] = bad_t ? __int_as_float(0x7fffffff) : logf(zt);
}

// Per row: the sums of the two KL-to-mixture partials (log2 units) over the
// chunks, in nats; the per-token value beta A + (1 - beta) B (or the KL of an
// endpoint branch).
__global__ void k_linear_merge_div(const float2* part, int chunks, int64_t rows, int jmode, float beta, float* saved,
                                   float* loss) {
  const int64_t r = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  if (r >= rows) return;
  float A = 0.f, B = 0.f;
  for (int c = 0; c < chunks; ++c) {
    const float2 p = part[c * rows + r];
    A += p.x;
    B += p.y;
  }
  A *= kLn2L;
  B *= kLn2L;
  float* sv = saved + r * 6;
  const bool ok = isfinite(sv[0]) && isfinite(sv[2]);
  float value;
  if (!ok) {
    A = B = value = __int_as_float(0x7fffffff);
  } else if (jmode == 0) {
    value = beta * A + (1.f - beta) * B;
  } else if (jmode == 1) {
    value = A;
    B = 0.f;
  } else {
    value = B;
    A = 0.f;
  }
  sv[4] = A;
  sv[5] = B;
  loss[r] = value;
}

// out[c, r] = in[r, c] for a bf16 [rows, cols] matrix (32 x 32 tiles through
// shared memory; rows and cols of the output are those of the transposed view).
__global__ void k_transpose_bf16(const __nv_bfloat16* in, int64_t rows, int64_t cols, int64_t ld_in,
                                 __nv_bfloat16* out, int64_t ld_out) {
  __shared__ __nv_bfloat16 tile[32][33];
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * 32, c0 = static_cast<int64_t>(blockIdx.x) * 32;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int64_t r = r0 + i, c = c0 + threadIdx.x;
    if (r < rows && c < cols) tile[i][threadIdx.x] = in[r * ld_in + c];
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int64_t c = c0 + i, r = r0 + threadIdx.x;
    if (r < rows && c < cols) out[c * ld_out + r] = tile[threadIdx.x][i];
  }
}


// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// A K-major bf16 operand [rows, k] with row stride `ld` elements, tiled in
// {64, box_rows} boxes with the 128-byte swizzle (A tiles 128 rows, B tiles
// as many as the tile has columns); rows and k past the ends read 0.
cudaError_t make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t k, int64_t ld, int box_rows = BM) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  if ((reinterpret_cast<uintptr_t>(base) & 15u) || (ld * 2) % 16) return cudaErrorInvalidValue;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld * 2)};
  const cuuint32_t box[2] = {BK, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Map of a bf16 output [outer, inner] (row pitch `pitch` elements) for tensor
// stores of 32 x 32 boxes, with the 64-byte swizzle or none.
cudaError_t make_store_map(CUtensorMap* m, void* base, int64_t inner, int64_t outer, int64_t pitch, bool swizzle64) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  if ((reinterpret_cast<uintptr_t>(base) & 15u) || (pitch * 2) % 16) return cudaErrorInvalidValue;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(pitch * 2)};
  const cuuint32_t box[2] = {32, 32};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// k_linear with TN-column tiles (the B maps' boxes must be TN rows high) in
// mode MODE (args.mode must be MODE).
template <int TN, int MODE>
cudaError_t launch(const CUtensorMap& a0, const CUtensorMap& b0, const CUtensorMap& a1, const CUtensorMap& b1,
                   const Args& args, cudaStream_t stream, const StoreMaps* gm = nullptr) {
  using E = EpiShape<MODE>;
  static_assert(smem_bytes<TN, MODE>() <= 232448, "dynamic shared memory above the 227 KB a CTA may take");
  if (args.units <= 0) return cudaSuccess;
  if (args.mode != MODE) return cudaErrorInvalidValue;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err =
        cudaFuncSetAttribute(k_linear<TN, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes<TN, MODE>());
  });
  if (attr_err != cudaSuccess) return attr_err;
  const int64_t grid = args.units < sm_count() ? args.units : sm_count();
  if (MODE == kGrad && !gm) return cudaErrorInvalidValue;
  static const StoreMaps none{};
  k_linear<TN, MODE><<<static_cast<unsigned>(grid), E::kThreads, smem_bytes<TN, MODE>(), stream>>>(a0, b0, a1, b1, args,
                                                                                                   gm ? *gm : none);
  note_launch();
  return cudaGetLastError();
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Vocabulary tiles per work unit of the JSD modes. CTA b of the G resident
// ones takes units b, b + G, ...; a pass lasts as long as its busiest CTA, so
// the unit size t minimises ceil(units / G) x (t + 1/2) (units = row tiles x
// vocabulary chunks, chunks = ceil(ntiles / t); half a tile stands for the
// per-unit cost), with at least 4 tiles per unit, at most `max_chunks` chunks
// (0: no limit; the chunks' partials must fit the workspace) and, on ties, the
// larger t (fewer partials to merge).
int tiles_per_unit(int64_t mtiles, int64_t ntiles, int64_t max_chunks = 0) {
  const int64_t g = sm_count();
  const int64_t t0 = ntiles < 4 ? ntiles : 4;
  int64_t best_t = ntiles, best = -1;
  for (int64_t t = t0; t <= ntiles; ++t) {
    const int64_t chunks = cdiv(ntiles, t);
    if (max_chunks > 0 && chunks > max_chunks) continue;
    const int64_t span = cdiv(mtiles * chunks, g) * (2 * t + 1);
    if (best < 0 || span <= best) {
      best = span;
      best_t = t;
    }
  }
  return static_cast<int>(best_t);
}

// Parts of the k range of a GEMM with `tiles` output tiles and nk k-blocks:
// the k that minimises ceil(tiles k / G) x (ceil(nk / k) + 8) (8 k-blocks
// stand for the per-unit cost of the epilogue's atomics), at most 16 parts
// and at least 8 k-blocks per part; on ties the smaller k.
int64_t gemm_ksplit(int64_t tiles, int64_t nk) {
  const int64_t g = sm_count();
  int64_t kmax = nk / 8;
  if (kmax > 16) kmax = 16;
  if (kmax < 1) kmax = 1;
  int64_t best_k = 1, best = -1;
  for (int64_t k = 1; k <= kmax; ++k) {
    const int64_t span = cdiv(tiles * k, g) * (cdiv(nk, k) + 8);
    if (best < 0 || span < best) {
      best = span;
      best_k = k;
    }
  }
  return best_k;
}

}  // namespace linear

using namespace linear;

// Partials of the forward, 32 bytes per row and vocabulary chunk: the
// statistics pass writes (m_s, z_s, m_t, z_t) per column part (two parts), the
// divergence pass, into the same bytes, (A, B) per column part (four parts).
static_assert(EpiShape<kStats>::kParts * 16 == 32 && EpiShape<kDiv>::kParts * 8 == 32, "partial sizes");
static size_t fwd_partial_bytes(int64_t rows, int64_t chunks) {
  return static_cast<size_t>(chunks) * static_cast<size_t>(rows) * 32u;
}

size_t linear_fwd_workspace(int64_t rows, int64_t vocab) {
  const int64_t mtiles = cdiv(rows, BM), ntiles = cdiv(vocab, BN);
  return fwd_partial_bytes(rows, cdiv(ntiles, tiles_per_unit(mtiles, ntiles)));
}

size_t linear_fwd_min_workspace(int64_t rows) { return fwd_partial_bytes(rows, 1); }

size_t linear_bwd_workspace(int64_t rows, int64_t vocab, int64_t hs, int64_t ht, bool student, bool teacher,
                            int64_t chunk_rows) {
  const int64_t nc = rows < chunk_rows ? cdiv(rows, BM) * BM : chunk_rows;
  size_t b = 0;
  const size_t g = static_cast<size_t>(nc) * static_cast<size_t>(vocab) * 2u;  // one bf16 [nc, V]
  if (student) b += 2 * g + static_cast<size_t>(hs) * nc * 2u;
  if (teacher) b += 2 * g + static_cast<size_t>(ht) * nc * 2u;
  return b + 1024;
}

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

cudaError_t linear_jsd_forward(const LinearProblem& p, float* loss, float* saved, void* ws, size_t ws_bytes,
                               cudaStream_t stream) {
  if (p.rows <= 0) return cudaSuccess;
  const int64_t mtiles = cdiv(p.rows, BM), ntiles = cdiv(p.vocab, BN);
  if (ws_bytes < linear_fwd_min_workspace(p.rows)) return cudaErrorInvalidValue;
  // the fastest plan whose partials fit the workspace (the plan of
  // linear_fwd_workspace when the workspace is at least that large)
  const int64_t max_chunks = static_cast<int64_t>(ws_bytes / fwd_partial_bytes(p.rows, 1));
  const int tpu = tiles_per_unit(mtiles, ntiles, max_chunks);
  const int64_t chunks = cdiv(ntiles, tpu);
  CUtensorMap hs, wsm, ht, wt;
  cudaError_t e;
  if ((e = make_map(&hs, p.h_s, p.rows, p.hs, p.ld_hs)) != cudaSuccess) return e;
  if ((e = make_map(&wsm, p.w_s, p.vocab, p.hs, p.ld_ws, BN)) != cudaSuccess) return e;
  if ((e = make_map(&ht, p.h_t, p.rows, p.ht, p.ld_ht)) != cudaSuccess) return e;
  if ((e = make_map(&wt, p.w_t, p.vocab, p.ht, p.ld_wt, BN)) != cudaSuccess) return e;
  Args a{};
  a.jmode = p.beta == 0.0 ? 1 : p.beta == 1.0 ? 2 : 0;
  a.rows = p.rows;
  a.cols = p.vocab;
  a.nk0 = static_cast<int>(p.hs / BK);
  a.nk1 = static_cast<int>(p.ht / BK);
  a.mtiles = static_cast<int>(mtiles);
  a.ntiles = static_cast<int>(ntiles);
  a.tiles_per_unit = tpu;
  a.units = mtiles * chunks;
  a.beta = static_cast<float>(p.beta);
  a.part = static_cast<float*>(ws);
  a.saved = saved;
  a.mode = kStats;
  if ((e = launch<BN, kStats>(hs, wsm, ht, wt, a, stream)) != cudaSuccess) return e;
  const unsigned mg = static_cast<unsigned>(cdiv(p.rows, 256));
  k_linear_merge_stats<<<mg, 256, 0, stream>>>(reinterpret_cast<const float4*>(ws),
                                               static_cast<int>(EpiShape<kStats>::kParts * chunks), p.rows, saved);
  note_launch();
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  a.mode = kDiv;
  if ((e = launch<BN, kDiv>(hs, wsm, ht, wt, a, stream)) != cudaSuccess) return e;
  k_linear_merge_div<<<mg, 256, 0, stream>>>(reinterpret_cast<const float2*>(ws),
                                             static_cast<int>(EpiShape<kDiv>::kParts * chunks), p.rows, a.jmode,
                                             a.beta, saved, loss);
  note_launch();
  return cudaGetLastError();
}


cudaError_t transpose_bf16(const void* in, int64_t rows, int64_t cols, int64_t ld_in, void* out, int64_t ld_out,
                           cudaStream_t stream) {
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  dim3 grid(static_cast<unsigned>(cdiv(cols, 32)), static_cast<unsigned>(cdiv(rows, 32)));
  k_transpose_bf16<<<grid, dim3(32, 8), 0, stream>>>(static_cast<const __nv_bfloat16*>(in), rows, cols, ld_in,
                                                       static_cast<__nv_bfloat16*>(out), ld_out);
  note_launch();
  return cudaGetLastError();
}

// C[rows, n] += A0 B0^T + A1 B1^T with K-major bf16 operands (A [rows, k],
// B [n, k]), split along k so that the units spread evenly over the SMs; with
// may_store (C holds nothing yet) and a single k part, C = the product.
cudaError_t gemm_acc(const void* a0p, const void* a1p, int64_t lda, const void* bp, int64_t ldb, int64_t rows,
                     int64_t n, int64_t k, float* C, int64_t ldc, bool may_store, cudaStream_t stream,
                     bool a_mn, bool b_mn) {
  CUtensorMap a0, a1, b0;
  cudaError_t e;
  if (a_mn) {  // A stored [k, rows] with row pitch lda, read in boxes of 64 rows x 64 k
    if ((e = make_map(&a0, a0p, k, rows, lda, 64)) != cudaSuccess) return e;
    if ((e = make_map(&a1, a1p, k, rows, lda, 64)) != cudaSuccess) return e;
  } else {
    if ((e = make_map(&a0, a0p, rows, k, lda)) != cudaSuccess) return e;
    if ((e = make_map(&a1, a1p, rows, k, lda)) != cudaSuccess) return e;
  }
  if (b_mn) {  // B stored [k, n] with row pitch ldb, read in boxes of 64 n x 64 k
    if ((e = make_map(&b0, bp, k, n, ldb, 64)) != cudaSuccess) return e;
  } else {
    if ((e = make_map(&b0, bp, n, k, ldb, BN)) != cudaSuccess) return e;
  }
  Args a{};
  a.mode = kGemm;
  a.rows = rows;
  a.cols = n;
  a.nk0 = a.nk1 = static_cast<int>(cdiv(k, BK));
  a.mtiles = static_cast<int>(cdiv(rows, BM));
  a.ntiles = static_cast<int>(cdiv(n, BN));
  const int64_t tiles = static_cast<int64_t>(a.mtiles) * a.ntiles;
  const int64_t ks = gemm_ksplit(tiles, a.nk0 + a.nk1);
  a.ksplit = static_cast<int>(ks);
  a.units = tiles * ks;
  a.C = C;
  a.ldc = ldc;
  // one k part per tile and nothing in C to add to: plain stores
  a.gemm_store = may_store && ks == 1 ? 1 : 0;
  a.a_mn = a_mn ? 1 : 0;
  a.b_mn = b_mn ? 1 : 0;
  return launch<BN, kGemm>(a0, b0, a1, b0, a, stream);
}

cudaError_t linear_jsd_backward(const LinearProblem& p, const float* grad_loss, const float* loss,
                                const float* saved, float* dh_s, float* dw_s, float* dh_t, float* dw_t, void* ws,
                                size_t ws_bytes, int64_t chunk_rows, cudaStream_t stream) {
  const bool student = dh_s || dw_s, teacher = dh_t || dw_t;
  if (!student && !teacher) return cudaSuccess;
  const int64_t nc = p.rows < chunk_rows ? cdiv(p.rows, BM) * BM : chunk_rows;
  if (ws_bytes < linear_bwd_workspace(p.rows, p.vocab, p.hs, p.ht, student, teacher, chunk_rows))
    return cudaErrorInvalidValue;
  // workspace: per head the [hi, lo] gradients of one chunk, row-major, and the
  // chunk's hidden states transposed [H, nc] (the head weight is read in place)
  uint8_t* w = static_cast<uint8_t*>(ws);
  const size_t g = align256(static_cast<size_t>(nc) * p.vocab * 2u);
  auto take = [&](size_t bytes) {
    uint8_t* r = w;
    w += align256(bytes);
    return r;
  };
  __nv_bfloat16* G[2][2] = {};
  void* hT[2] = {nullptr, nullptr};
  const int64_t H[2] = {p.hs, p.ht};
  const void* hp[2] = {p.h_s, p.h_t};
  const int64_t ldh[2] = {p.ld_hs, p.ld_ht};
  const void* wp[2] = {p.w_s, p.w_t};
  const int64_t ldw[2] = {p.ld_ws, p.ld_wt};
  const bool want[2] = {student, teacher};
  float* dh[2] = {dh_s, dh_t};
  float* dw[2] = {dw_s, dw_t};
  cudaError_t e;
  for (int x = 0; x < 2; ++x) {
    if (!want[x]) continue;
    for (int i = 0; i < 2; ++i) G[x][i] = reinterpret_cast<__nv_bfloat16*>(take(g));
    hT[x] = take(static_cast<size_t>(H[x]) * nc * 2u);
    // dh accumulates by atomics: start from zero
    if (dh[x] && (e = cudaMemsetAsync(dh[x], 0, static_cast<size_t>(p.rows) * H[x] * 4u, stream)) != cudaSuccess)
      return e;
    // dW: unless the first chunk's contraction runs unsplit and stores its
    // product (every element once), later chunks add to it
    const int64_t n0 = p.rows < nc ? p.rows : nc;
    const bool dw_stored = gemm_ksplit(cdiv(p.vocab, BM) * cdiv(H[x], BN), 2 * cdiv(n0, BK)) == 1;
    if (dw[x] && !dw_stored &&
        (e = cudaMemsetAsync(dw[x], 0, static_cast<size_t>(p.vocab) * H[x] * 4u, stream)) != cudaSuccess)
      return e;
  }
  CUtensorMap hsm, wsm, htm, wtm;
  for (int64_t r0 = 0; r0 < p.rows; r0 += nc) {
    const int64_t n = p.rows - r0 < nc ? p.rows - r0 : nc;
    const void* hs0 = static_cast<const char*>(p.h_s) + r0 * p.ld_hs * 2;
    const void* ht0 = static_cast<const char*>(p.h_t) + r0 * p.ld_ht * 2;
    if ((e = make_map(&hsm, hs0, n, p.hs, p.ld_hs)) != cudaSuccess) return e;
    if ((e = make_map(&wsm, p.w_s, p.vocab, p.hs, p.ld_ws, kGradTN)) != cudaSuccess) return e;
    if ((e = make_map(&htm, ht0, n, p.ht, p.ld_ht)) != cudaSuccess) return e;
    if ((e = make_map(&wtm, p.w_t, p.vocab, p.ht, p.ld_wt, kGradTN)) != cudaSuccess) return e;
    Args a{};
    a.mode = kGrad;
    a.jmode = p.beta == 0.0 ? 1 : p.beta == 1.0 ? 2 : 0;
    a.rows = n;
    a.cols = p.vocab;
    a.nk0 = static_cast<int>(p.hs / BK);
    a.nk1 = static_cast<int>(p.ht / BK);
    a.mtiles = static_cast<int>(cdiv(n, BM));
    a.ntiles = static_cast<int>(cdiv(p.vocab, kGradTN));
    a.tiles_per_unit = tiles_per_unit(a.mtiles, a.ntiles);
    a.units = static_cast<int64_t>(a.mtiles) * cdiv(a.ntiles, a.tiles_per_unit);
    a.beta = static_cast<float>(p.beta);
    a.saved = saved + r0 * 6;
    a.loss = loss + r0;
    a.grad_loss = grad_loss ? grad_loss + r0 : nullptr;
    // row-major only: dW reads the same arrays MN-major
    if (student) {
      a.gs_hi = G[0][0];
      a.gs_lo = G[0][1];
    }
    if (teacher) {
      a.gt_hi = G[1][0];
      a.gt_lo = G[1][1];
    }
    // the gradient blocks' tensor stores, row-major [n, V]
    StoreMaps gm{};
    for (int x = 0; x < 2; ++x) {
      if (!want[x]) continue;
      for (int hl = 0; hl < 2; ++hl)
        if ((e = make_store_map(&gm.m[x][hl], G[x][hl], p.vocab, n, p.vocab, true)) != cudaSuccess) return e;
    }
    if ((e = launch<kGradTN, kGrad>(hsm, wsm, htm, wtm, a, stream, &gm)) != cudaSuccess) return e;
    for (int x = 0; x < 2; ++x) {
      if (!want[x]) continue;
      // dh[r0:r0+n] += G_hi W + G_lo W  (K = V; A = G K-major, B = W [V, H] read MN-major)
      if (dh[x] &&
          (e = gemm_acc(G[x][0], G[x][1], p.vocab, wp[x], ldw[x], n, H[x], p.vocab, dh[x] + r0 * H[x], H[x],
                        true, stream, false, true)) != cudaSuccess)
        return e;
      // dW += G_hi^T h + G_lo^T h  (K = the chunk's n rows; A = G [n, V] read
      // MN-major, B = h^T [H, nc] K-major: h read in place as an MN-major B
      // drew more from DRAM; the maps end K at n, the loads fill zeros past it)
      if (dw[x]) {
        const void* h0 = static_cast<const char*>(hp[x]) + r0 * ldh[x] * 2;
        if ((e = transpose_bf16(h0, n, H[x], ldh[x], hT[x], nc, stream)) != cudaSuccess) return e;
        if ((e = gemm_acc(G[x][0], G[x][1], p.vocab, hT[x], nc, p.vocab, H[x], n, dw[x], H[x], r0 == 0, stream,
                          true, false)) != cudaSuccess)
          return e;
      }
    }
  }
  return cudaSuccess;
}

cudaError_t take_linear_error(cudaStream_t stream, int* code);

// ---------------------------------------------------------------------------
// Forward without caller workspace: the per-chunk statistics partials live in
// one file-scope device array (each GPU that loads the library holds its own
// copy until the process exits). Every entry of it that the forward reads is
// first written by the same call, so nothing needs clearing; two calls that
// overlap on the GPU would write the same entries and race.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_linear_scratch[kLinearNoAllocMaxBytes];

cudaError_t linear_scratch(void** out) {
  static std::mutex mu;
  static void* ptr[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptr[dev]) {
    // the array's device address on the current device (its host-side name is
    // only a stand-in and must never reach a kernel)
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_linear_scratch);
    if (e != cudaSuccess) return e;
    ptr[dev] = p;
  }
  *out = ptr[dev];
  return cudaSuccess;
}

}  // namespace vpd

namespace vpd {
static __device__ int g_linear_taken = 0;
static __global__ void k_take_linear_error2() { g_linear_taken = atomicExch(&linear::g_linear_error, 0); }
cudaError_t take_linear_error(cudaStream_t stream, int* code) {
  k_take_linear_error2<<<1, 1, 0, stream>>>();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbolAsync(code, g_linear_taken, sizeof(int), 0, cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(stream);
}
}  // namespace vpd
