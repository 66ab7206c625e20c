// vpd_shard.cu -- per-row kernels of the vocabulary-parallel JSD / KL: each
// process holds one vocabulary shard of the student and teacher logits, and
// the forward exchanges only [N]-sized statistics between them, as the pages'
// vocabulary-parallel ops do ("Add vocabulary-parallel logprobs, entropy and
// KL ops", section How: one MAX all-reduce and two SUM all-reduces of
// per-token statistics; "[VocabTP] Add vocabulary-parallel generalized JSD
// with Triton kernels", section Changes: uneven and empty shards). The
// all-reduces themselves are the caller's (NCCL or any other collective
// library); these kernels prepare and consume their [N, 2] buffers:
//   1. local statistics (the paired-statistics kernel on the shard), then the
//      maxima (m_s, m_t) packed for a MAX all-reduce;
//   2. the shard's sums rescaled to the global maxima, packed for a SUM
//      all-reduce;
//   3. the global log-sum-exps, the shard's two KL-to-mixture partial sums (the
//      divergence kernel on the shard), packed for a SUM all-reduce;
//   4. the per-token value from the summed partials.
// The backward is local: vpd_jsd_bwd on the shard with the saved statistics.
// A row outside the contract on any shard travels as +inf through the MAX and
// as NaN through the SUMs, so every process ends with the same NaN row.

#include <cuda_runtime.h>

#include "vpd_internal.h"

namespace vpd {
namespace {

__device__ __forceinline__ float nan_f() { return __int_as_float(0x7fffffff); }
__device__ __forceinline__ float pinf_f() { return __int_as_float(0x7f800000); }
__device__ __forceinline__ float ninf_f() { return __int_as_float(0xff800000); }

__global__ void k_shard_maxima(const float* saved, int64_t rows, float* x) {
  const int64_t r = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  if (r >= rows) return;
  const float ms = saved[r * 6], mt = saved[r * 6 + 2];
  x[2 * r] = isnan(ms) ? pinf_f() : ms;
  x[2 * r + 1] = isnan(mt) ? pinf_f() : mt;
}

// z' = e^{L_local + m_local - m} with m the global max: the shard's sum
// relative to the global max; an empty or fully -inf shard gives 0.
__global__ void k_shard_rescale(float* saved, int64_t rows, float* x) {
  const int64_t r = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  if (r >= rows) return;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const float ml = saved[r * 6 + 2 * h], L = saved[r * 6 + 2 * h + 1], mg = x[2 * r + h];
    float z;
    if (isnan(mg) || mg == pinf_f()) z = nan_f();
    else if (ml == ninf_f()) z = 0.f;
    else z = expf(L + (ml - mg));
    saved[r * 6 + 2 * h] = mg;
    x[2 * r + h] = z;
  }
}

// ln Z of the summed z; m = -inf (no shard has a finite logit): no distribution.
__global__ void k_shard_lse(float* saved, int64_t rows, const float* x) {
  const int64_t r = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  if (r >= rows) return;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const float mg = saved[r * 6 + 2 * h], Z = x[2 * r + h];
    if (isnan(Z) || isnan(mg) || mg == pinf_f()) {
      saved[r * 6 + 2 * h] = nan_f();
      saved[r * 6 + 2 * h + 1] = nan_f();
    } else if (mg == ninf_f()) {
      saved[r * 6 + 2 * h + 1] = ninf_f();
    } else {
      saved[r * 6 + 2 * h + 1] = logf(Z);
    }
  }
}

__global__ void k_shard_pack_sums(const float* saved, int64_t rows, float* x) {
  const int64_t r = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  if (r >= rows) return;
  x[2 * r] = saved[r * 6 + 4];
  x[2 * r + 1] = saved[r * 6 + 5];
}

// The per-token value from the summed (A, B): beta A + (1 - beta) B inside,
// the KL sum at the endpoint branches (+inf when any shard saw a support
// violation); NaN where the statistics are undefined.
__global__ void k_shard_finish(float* saved, int64_t rows, const float* x, int jmode, float beta, float* loss) {
  const int64_t r = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  if (r >= rows) return;
  float A = x[2 * r], B = x[2 * r + 1], value;
  if (!isfinite(saved[r * 6]) || !isfinite(saved[r * 6 + 2])) A = B = value = nan_f();
  else if (jmode == 0) value = beta * A + (1.f - beta) * B;
  else if (jmode == 1) value = A;
  else value = B;
  saved[r * 6 + 4] = A;
  saved[r * 6 + 5] = B;
  loss[r] = value;
}

unsigned blocks_for(int64_t rows) { return static_cast<unsigned>((rows + 255) / 256); }

cudaError_t done() {
  note_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t shard_stats(const View& s, const View& t, float* saved, float* x, cudaStream_t st) {
  Segs one;
  one.count = 1;
  one.off[0] = 0;
  one.off[1] = s.vocab;
  cudaError_t e = launch_pair_stats(s, t, one, saved, st);
  if (e != cudaSuccess) return e;
  k_shard_maxima<<<blocks_for(s.rows), 256, 0, st>>>(saved, s.rows, x);
  return done();
}

cudaError_t shard_rescale(int64_t rows, float* saved, float* x, cudaStream_t st) {
  k_shard_rescale<<<blocks_for(rows), 256, 0, st>>>(saved, rows, x);
  return done();
}

cudaError_t shard_divergence(const View& s, const View& t, double beta, float* loss, float* saved, float* x,
                             cudaStream_t st) {
  k_shard_lse<<<blocks_for(s.rows), 256, 0, st>>>(saved, s.rows, x);
  cudaError_t e = done();
  if (e != cudaSuccess) return e;
  e = launch_jsd_div(s, t, beta, loss, saved, st);
  if (e != cudaSuccess) return e;
  k_shard_pack_sums<<<blocks_for(s.rows), 256, 0, st>>>(saved, s.rows, x);
  return done();
}

cudaError_t shard_finish(int64_t rows, double beta, float* saved, const float* x, float* loss, cudaStream_t st) {
  const int jmode = beta == 0.0 ? 1 : beta == 1.0 ? 2 : 0;
  k_shard_finish<<<blocks_for(rows), 256, 0, st>>>(saved, rows, x, jmode, static_cast<float>(beta), loss);
  return done();
}

}  // namespace vpd
