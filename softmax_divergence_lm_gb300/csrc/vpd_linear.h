// vpd_linear.h -- host interface of the fused-linear JSD kernels (vpd_linear.cu).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace vpd {

// Student and teacher heads: logits s = h_s w_s^T, t = h_t w_t^T; every matrix
// bf16, row-major, K-major (hidden index contiguous), rows 16-byte aligned.
struct LinearProblem {
  const void* h_s;  // [rows, hs], row stride ld_hs
  const void* w_s;  // [vocab, hs], row stride ld_ws
  const void* h_t;  // [rows, ht]
  const void* w_t;  // [vocab, ht]
  int64_t rows, vocab, hs, ht;
  int64_t ld_hs, ld_ws, ld_ht, ld_wt;
  double beta;
};

// Rows of one backward chunk (a multiple of the 128-row tile): up to this
// many rows, dW is one contraction over all of them.
constexpr int64_t kLinearChunkRows = 8192;

size_t linear_fwd_workspace(int64_t rows, int64_t vocab);
// The least workspace the forward runs with (its vocabulary in one chunk); a
// workspace between this and linear_fwd_workspace gets fewer, longer chunks.
size_t linear_fwd_min_workspace(int64_t rows);
size_t linear_bwd_workspace(int64_t rows, int64_t vocab, int64_t hs, int64_t ht, bool student, bool teacher,
                            int64_t chunk_rows);
cudaError_t linear_jsd_forward(const LinearProblem& p, float* loss, float* saved, void* ws, size_t ws_bytes,
                               cudaStream_t stream);
cudaError_t linear_jsd_backward(const LinearProblem& p, const float* grad_loss, const float* loss,
                                const float* saved, float* dh_s, float* dw_s, float* dh_t, float* dw_t, void* ws,
                                size_t ws_bytes, int64_t chunk_rows, cudaStream_t stream);
// Size of the file-scope device array the workspace-free forward uses.
constexpr size_t kLinearNoAllocMaxBytes = size_t(4) << 20;
// Device address of that array on the current device (looked up once per device).
cudaError_t linear_scratch(void** out);
// Reads and clears the device error word of the fused-linear kernels.
cudaError_t take_linear_error(cudaStream_t stream, int* code);

}  // namespace vpd
