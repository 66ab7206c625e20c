// vpd_internal.h -- host-side descriptions of views, gradients and segment
// tables after validation, and the kernel launchers the C ABI dispatches to.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "vpd.h"
#include "vpd_device.cuh"

namespace vpd {

// A validated logits view.
struct View {
  const char* data;  // element (0, 0)
  int dtype;         // Dtype
  int64_t rows;
  int64_t vocab;
  RowMap map;
};

// A validated gradient output; data == nullptr means "not wanted".
struct Grad {
  char* data;
  int dtype;
  int64_t row_stride;
};

// Segment table as offsets: segment k spans [off[k], off[k + 1]).
struct Segs {
  int count;
  int64_t off[VPD_MAX_SEGMENTS + 1];
};

// Streaming kernels: one CTA per row at a time (grid-stride over rows).
cudaError_t launch_pair_stats(const View& s, const View& t, const Segs& seg, float* saved,
                              cudaStream_t stream);
cudaError_t launch_jsd_div(const View& s, const View& t, double beta, float* loss, float* saved,
                           cudaStream_t stream);
cudaError_t launch_pair_bwd(const View& s, const View& t, double beta, const float* grad_loss,
                            const float* saved, const Grad& ds, const Grad& dt, cudaStream_t stream);
cudaError_t launch_kl_fwd(const View& s, const View& t, int reverse, const Segs& seg, float* loss,
                          float* saved, cudaStream_t stream);
cudaError_t launch_entropy_fwd(const View& x, const Segs& seg, float* out, float* saved,
                               cudaStream_t stream);
cudaError_t launch_entropy_bwd(const View& x, const float* grad, const float* saved, const Grad& dx,
                               cudaStream_t stream);
// Selected log-probabilities and the ops built on them: mode 0 the log-probs
// at index [N, k] into out [N, k]; mode 1 the cross-entropy at one label per
// row (k = 1) into row_out [N]; mode 2 the teacher top-k forward KL with the
// teacher's log-probs teacher_logp [N, k] into row_out [N]. inv_temperature
// scales the logits before the softmax (1: none).
cudaError_t launch_select_fwd(const View& x, const Segs& seg, const int64_t* index, int k, int64_t ignore_index,
                              float inv_temperature, int mode, const float* teacher_logp, float* out,
                              float* row_out, float* saved, int32_t* err_flag, cudaStream_t stream);
cudaError_t launch_select_bwd(const View& x, const int64_t* index, int k, int64_t ignore_index,
                              float inv_temperature, int mode, const float* teacher_logp, const float* grad,
                              const float* saved, const Grad& dx, cudaStream_t stream);

// Vocabulary-parallel JSD / KL, per shard (vpd_shard.cu); x is the [rows, 2]
// buffer the caller all-reduces between the steps.
cudaError_t shard_stats(const View& s, const View& t, float* saved, float* x, cudaStream_t st);
cudaError_t shard_rescale(int64_t rows, float* saved, float* x, cudaStream_t st);
cudaError_t shard_divergence(const View& s, const View& t, double beta, float* loss, float* saved, float* x,
                             cudaStream_t st);
cudaError_t shard_finish(int64_t rows, double beta, float* saved, const float* x, float* loss, cudaStream_t st);

// Single-read fused JSD forward+backward on thread-block clusters. Returns
// cudaErrorNotSupported (without launching) when the row pair does not fit on
// chip in clusters of at most max_cluster CTAs or the layout does not allow it;
// the caller then uses the streaming path. withhold_row >= 0 is the
// failure-path test hook (vpd_test_withhold_copy). dry_run: only decide
// (cudaSuccess when the kernel would run), launch nothing.
cudaError_t launch_jsd_fused(const View& s, const View& t, double beta, const float* grad_loss,
                             float* loss, float* saved, const Grad& ds, const Grad& dt,
                             cudaStream_t stream, int64_t withhold_row, int max_cluster = 16,
                             bool dry_run = false);

// While alive, sizes every streaming-kernel launch made on this thread for
// `sms` SMs (as many CTAs as fit that many SMs; 0: every SM).
class GridCap {
 public:
  explicit GridCap(int sms);
  ~GridCap();
  GridCap(const GridCap&) = delete;
  GridCap& operator=(const GridCap&) = delete;

 private:
  int prev_;
};

// Rows of a single-read JSD call (forward+backward, or forward only when
// neither gradient is wanted) to hand to the SMs its clusters leave idle, and
// how many SMs those are (0, 0 when the split does not pay).
void fused_idle_split(const View& s, const Grad& ds, const Grad& dt, int max_cluster, int64_t* side_rows,
                      int* idle_sms);

// Number of SMs of the current device (cached per device).
int sm_count();

// Counts every kernel launch the library issues (read by vpd_launch_count).
void note_launch();
uint64_t launch_count();

}  // namespace vpd
