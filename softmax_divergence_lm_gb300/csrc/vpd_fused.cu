// vpd_fused.cu -- host dispatch of the single-read fused JSD forward+backward
// (device code and design notes in vpd_fused.cuh): shape checks, the choice of
// cluster size and register budget, and the device error words read by
// vpd_device_status.

#include <cuda_runtime.h>

#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "vpd_fused.cuh"
#include "vpd_internal.h"

namespace vpd {
namespace fused {
// Instantiated in vpd_fused_bf16.cu and vpd_fused_f16.cu.
extern template cudaError_t launch_typed<InBF16>(const FusedArgs&, const Config&, int, bool, cudaStream_t, int*);
extern template cudaError_t launch_typed<InF16>(const FusedArgs&, const Config&, int, bool, cudaStream_t, int*);
cudaError_t take_error_bf16(int* code);
cudaError_t take_error_f16(int* code);
}  // namespace fused

cudaError_t take_device_error(cudaStream_t stream, int* code) {
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return e;
  int a = 0, b = 0;
  e = fused::take_error_bf16(&a);
  if (e != cudaSuccess) return e;
  e = fused::take_error_f16(&b);
  *code = a | b;
  return e;
}

namespace {

using fused::Config;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// VPD_VERBOSE=1 logs each fused launch configuration to stderr.
bool verbose() {
  static const bool v = [] {
    const char* e = getenv("VPD_VERBOSE");
    return e && e[0] && e[0] != '0';
  }();
  return v;
}

// VPD_FUSED_VARIANT=keep|recompute restricts the choice to one register
// budget (both are complete implementations; the default tries "recompute"
// first).
int variant_choice() {
  static const int v = [] {
    const char* e = getenv("VPD_FUSED_VARIANT");
    if (e && !strcmp(e, "keep")) return 1;
    if (e && !strcmp(e, "recompute")) return 2;
    return 0;
  }();
  return v;
}

// The smallest cluster that holds a row with at most rmax vectors of both
// inputs per thread, for T threads per CTA.
bool fit(int64_t vocab, int T, int rmin, int rmax, bool keep, Config* cfg) {
  for (int C : {1, 2, 4, 8, 16}) {
    const int64_t W = ((vocab + C - 1) / C + 7) / 8 * 8;
    int64_t R = (W + T * 8 - 1) / (T * 8);
    if (R < rmin) R = rmin;
    if (R <= rmax) {
      cfg->C = C;
      cfg->T = T;
      cfg->R = static_cast<int>(R);
      cfg->W = static_cast<int>(W);
      cfg->keep = keep;
      const size_t tail = keep ? sizeof(fused::Tail<fused::kKeepT>) : sizeof(fused::Tail<fused::kRecomputeT>);
      cfg->smem = static_cast<size_t>(fused::kStages) * 2 * W * 2 + tail;
      return true;
    }
  }
  return false;
}

}  // namespace

cudaError_t launch_jsd_fused(const View& s, const View& t, double beta, const float* grad_loss,
                             float* loss, float* saved, const Grad& ds, const Grad& dt,
                             cudaStream_t stream, int64_t withhold_row) {
  // 16-bit inputs only; every row of both inputs and of both gradients must
  // start on a 16-byte boundary, and V must fill whole 16-byte vectors.
  if (s.dtype == kF32 || s.vocab <= 0 || s.vocab % 8 != 0) return cudaErrorNotSupported;
  if (!aligned16(s.data) || !aligned16(t.data)) return cudaErrorNotSupported;
  for (const RowMap* m : {&s.map, &t.map})
    if ((m->row_stride * 2) % 16 || (m->rows_per_batch > 0 && (m->batch_stride * 2) % 16))
      return cudaErrorNotSupported;
  const Grad* gs[2] = {&ds, &dt};
  int gdtype = -1;
  for (const Grad* g : gs) {
    if (!g->data) continue;
    const int esz = g->dtype == kF32 ? 4 : 2;
    if (!aligned16(g->data) || (g->row_stride * esz) % 16) return cudaErrorNotSupported;
    if (g->dtype != kF32 && g->dtype != s.dtype) return cudaErrorNotSupported;
    gdtype = g->dtype;
  }
  // Candidate configurations, best first: the recompute budget (480 threads,
  // R <= 5), then the kept-value budget (256 threads, R <= 5), which needs
  // about twice the CTAs per row.
  Config cand[2];
  int n = 0;
  const int choice = variant_choice();
  if (choice != 1 && fit(s.vocab, fused::kRecomputeT, 1, 5, false, &cand[n])) ++n;
  if (choice != 2 && fit(s.vocab, fused::kKeepT, 1, fused::kKeepMaxR, true, &cand[n])) ++n;
  const int mode = beta == 0.0 ? fused::kForwardKL : beta == 1.0 ? fused::kReverseKL : fused::kInterior;
  const bool f32g = gdtype == kF32;
  for (int i = 0; i < n; ++i) {
    const Config& cfg = cand[i];
    fused::FusedArgs args{s.data, t.data, s.map, t.map, s.rows, s.vocab, cfg.W, static_cast<float>(beta),
                          grad_loss, loss, saved, ds, dt, withhold_row};
    int clusters = 0;
    const cudaError_t e = s.dtype == kBF16
                              ? fused::launch_typed<fused::InBF16>(args, cfg, mode, f32g, stream, &clusters)
                              : fused::launch_typed<fused::InF16>(args, cfg, mode, f32g, stream, &clusters);
    if (e == cudaErrorNotSupported) continue;
    if (e == cudaSuccess) {
      note_launch();
      if (verbose())
        fprintf(stderr, "[vpd] fused JSD: V=%lld %s cluster=%d threads=%d R=%d W=%d smem=%zu B, %d clusters\n",
                static_cast<long long>(s.vocab), cfg.keep ? "kept" : "recompute", cfg.C, cfg.T, cfg.R, cfg.W,
                cfg.smem, clusters);
    }
    return e;
  }
  return cudaErrorNotSupported;
}

}  // namespace vpd
