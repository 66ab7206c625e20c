// vpd_fused.cu -- host dispatch of the single-read fused JSD forward+backward
// (device code and design notes in vpd_fused.cuh): shape checks, the choice of
// cluster size, and the device error words read by vpd_device_status.

#include <cuda_runtime.h>

#include <cstdio>
#include <cstdlib>
#include <cstring>

#include <atomic>

#include "vpd_fused.cuh"
#include "vpd_internal.h"

namespace vpd {
namespace fused {
// Instantiated in vpd_fused_bf16.cu, vpd_fused_f16.cu and vpd_fused_f32.cu.
extern template cudaError_t launch_typed<InBF16>(const FusedArgs&, const Config&, int, bool, bool, cudaStream_t, int*);
extern template cudaError_t launch_typed<InF16>(const FusedArgs&, const Config&, int, bool, bool, cudaStream_t, int*);
extern template cudaError_t launch_typed<InF32>(const FusedArgs&, const Config&, int, bool, bool, cudaStream_t, int*);
extern template int resident_clusters<InBF16>(int, int, size_t);
cudaError_t take_error_bf16(cudaStream_t stream, int* code);
cudaError_t take_error_f16(cudaStream_t stream, int* code);
cudaError_t take_error_f32(cudaStream_t stream, int* code);
}  // namespace fused

cudaError_t take_device_error(cudaStream_t stream, int* code) {
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return e;
  int a = 0, b = 0, c = 0;
  e = fused::take_error_bf16(stream, &a);
  if (e != cudaSuccess) return e;
  e = fused::take_error_f16(stream, &b);
  if (e != cudaSuccess) return e;
  e = fused::take_error_f32(stream, &c);
  *code = a | b | c;
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

constexpr int kMaxDevices = 64;

// Resident clusters of C CTAs on the current device (one CTA per SM whatever
// the dtype, mode, width or worker count), cached.
int clusters_for(int C) {
  static std::atomic<int> cache[kMaxDevices][fused::kMaxCluster + 1];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  int v = cache[dev][C].load(std::memory_order_relaxed);
  if (v == 0) {
    v = fused::resident_clusters<fused::InBF16>(C, 16, fused::kMinSmem);
    cache[dev][C].store(v < 1 ? -1 : v, std::memory_order_relaxed);
  }
  return v < 1 ? 0 : v;
}

size_t max_smem_optin() {
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  int v = cache[dev].load(std::memory_order_relaxed);
  if (v == 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess || v < 1) v = -1;
    cache[dev].store(v, std::memory_order_relaxed);
  }
  return v < 1 ? 0 : static_cast<size_t>(v);
}

// Per-row cost of the cluster exchanges, in units of one 16-byte vector pair
// of work on an SM (about 1.5 us of hand-overs against about 4 ns a vector).
constexpr int64_t kRowOverheadVectors = 400;

// Per-row work of a CTA in vectors, as its busiest warp scheduler sets it:
// each per-row phase ends when the sub-partition (warp % 4) with the most
// warp-wide vectors has issued them, so the cost is 4 x 32 x that count.
int64_t sched_vectors(int64_t nvec, int R, int nw) {
  int64_t load[4] = {0, 0, 0, 0};
  for (int w = 0; w < nw; ++w) {
    const int64_t j = fused::vector_order(w, nw, R);
    for (int k = 0; k < R; ++k)
      if (static_cast<int64_t>(k) * 32 * nw + 32 * j < nvec) ++load[w & 3];
  }
  int64_t m = 0;
  for (int s = 0; s < 4; ++s) m = load[s] > m ? load[s] : m;
  return 128 * m;
}

// The launch shape: the cluster size C with the least time per row batch,
// rows per cluster x (slice work + exchange overhead), among those whose
// slice fits (two stages in shared memory; at most kMaxR vectors per worker
// thread within the register and TMEM budgets); then the smallest R that
// covers the slice and as many workers as the budgets allow without idle
// warps (more warps hide more latency). Ties go to the smaller cluster.
// `fwd`: the forward-only kernel (three stages, no tensor memory); `esize`:
// bytes per input element (2, or 4 for fp32 logits).
bool choose(int64_t vocab, int64_t rows, int max_cluster, bool fwd, Config* cfg, int esize) {
  const size_t smem_cap = max_smem_optin();
  int64_t best = 0;
  for (int C = 1; C <= fused::kMaxCluster && C <= max_cluster; ++C) {
    const int64_t W = ((vocab + C - 1) / C + 7) / 8 * 8;
    const int64_t nvec = W / 8;
    const size_t smem = fwd ? fused::smem_bytes_fwd(static_cast<int>(W), esize)
                            : fused::smem_bytes(static_cast<int>(W), false, esize);
    if (smem > smem_cap) continue;
    int bR = 0, bnw = 0;
    for (int R = 1; R <= fused::kMaxR && !bR; ++R) {
      const int64_t cap = fwd ? fused::kMaxWorkersFwd : fused::max_workers(R);
      if (nvec > 32 * cap * R) continue;
      int64_t nw = R == 1 ? (nvec + 31) / 32 : (nvec + 32 * (R - 1) - 1) / (32 * (R - 1));
      if (nw > cap) nw = cap;
      if (nw < 1) nw = 1;
      if (!fwd && R * fused::Cols<fused::kInterior>::k > fused::tmem_cols_per_warp(static_cast<int>(nw))) continue;
      bR = R, bnw = static_cast<int>(nw);
    }
    if (!bR) continue;
    const int clusters = clusters_for(C);
    if (clusters < 1) continue;
    const int64_t used = rows < clusters ? rows : clusters;
    const int64_t cost = (rows + used - 1) / used * (sched_vectors(nvec, bR, bnw) + kRowOverheadVectors);
    if (!best || cost < best) {
      best = cost;
      *cfg = Config{C, bR, static_cast<int>(W), bnw, smem};
    }
  }
  return best > 0;
}

}  // namespace

// Rate of the streaming path on one otherwise idle SM relative to one SM of a
// fused cluster, in rows per second per SM: for forward+backward (three
// streaming passes against one read) of 16-bit rows 0.5 with clusters of up
// to 15 CTAs and 0.57 with 16 (a cluster of 16 spends more of each row on its
// exchanges), of fp32 rows 0.9 (the fused kernel moves twice the bytes per
// element through its stages); for the forward (two passes) 0.9; measured at
// V = 151936 (clusters of 9), V = 262144 (clusters of 16) and V = 128256 fp32
// (clusters of 9). VPD_IDLE_RATE / VPD_IDLE_RATE_FWD override them (0
// disables the split).
static double idle_rate(bool fwd, int cluster, int esize) {
  static const double r[2] = {[] {
                                const char* e = getenv("VPD_IDLE_RATE");
                                return e && e[0] ? atof(e) : -1.0;
                              }(),
                              [] {
                                const char* e = getenv("VPD_IDLE_RATE_FWD");
                                return e && e[0] ? atof(e) : 0.9;
                              }()};
  if (fwd) return r[1];
  if (r[0] >= 0.0) return r[0];
  if (esize == 4) return 0.9;
  return cluster >= 16 ? 0.57 : 0.5;
}

void fused_idle_split(const View& s, const Grad& ds, const Grad& dt, int max_cluster, int64_t* side_rows,
                      int* idle_sms) {
  *side_rows = 0;
  *idle_sms = 0;
  const bool fwd = !ds.data && !dt.data;
  // long rows only: their streaming CTAs are wide enough (at least three warps
  // of 40 or more registers) that none fits beside a fused CTA on its SM
  if (s.vocab < 100000) return;
  if (!fwd) {
    const int gdtype = ds.data ? ds.dtype : dt.dtype;
    if (gdtype != kF32 && gdtype != s.dtype) return;
  }
  Config cfg;
  const int es = s.dtype == kF32 ? 4 : 2;
  if (!choose(s.vocab, s.rows, max_cluster, fwd, &cfg, es)) return;
  const double rate = idle_rate(fwd, cfg.C, es);
  if (rate <= 0.0) return;
  const int clusters = clusters_for(cfg.C);
  const int used = clusters * cfg.C, idle = sm_count() - used;
  // worth it only with every cluster busy for many rows
  if (idle < 4 || s.rows < 8 * static_cast<int64_t>(clusters)) return;
  const double share = idle * rate / (used + idle * rate);
  const int64_t side = static_cast<int64_t>(s.rows * share);
  if (side < idle) return;
  *side_rows = side;
  *idle_sms = idle;
}

cudaError_t launch_jsd_fused(const View& s, const View& t, double beta, const float* grad_loss,
                             float* loss, float* saved, const Grad& ds, const Grad& dt,
                             cudaStream_t stream, int64_t withhold_row, int max_cluster, bool dry_run) {
  // Every row of both inputs and of both gradients must start on a 16-byte
  // boundary, and V must fill whole 8-element vectors.
  const int es = s.dtype == kF32 ? 4 : 2;
  if (s.vocab <= 0 || s.vocab % 8 != 0) return cudaErrorNotSupported;
  if (!aligned16(s.data) || !aligned16(t.data)) return cudaErrorNotSupported;
  for (const RowMap* m : {&s.map, &t.map})
    if ((m->row_stride * es) % 16 || (m->rows_per_batch > 0 && (m->batch_stride * es) % 16))
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
  const bool fwd = gdtype < 0;  // no gradient wanted: the forward-only kernel
  Config cfg;
  if (!choose(s.vocab, s.rows, max_cluster, fwd, &cfg, es)) return cudaErrorNotSupported;
  const int mode = beta == 0.0 ? fused::kForwardKL : beta == 1.0 ? fused::kReverseKL : fused::kInterior;
  const bool f32g = gdtype == kF32;
  // 16-bit gradients go out through a shared-memory buffer and bulk stores
  // when it fits beside the stages.
  if (dry_run) return cudaSuccess;
  const bool gstage = gdtype >= 0 && !f32g && fused::smem_bytes(cfg.W, true, es) <= max_smem_optin();
  if (gstage) cfg.smem = fused::smem_bytes(cfg.W, true, es);
  fused::FusedArgs args{s.data, t.data, s.map, t.map, s.rows, s.vocab, cfg.W, cfg.nw, gstage ? 1 : 0,
                        static_cast<float>(beta),
                        grad_loss, loss, saved, ds, dt, withhold_row};
  int clusters = 0;
  const cudaError_t e = s.dtype == kBF16  ? fused::launch_typed<fused::InBF16>(args, cfg, mode, f32g, fwd, stream, &clusters)
                        : s.dtype == kF16 ? fused::launch_typed<fused::InF16>(args, cfg, mode, f32g, fwd, stream, &clusters)
                                          : fused::launch_typed<fused::InF32>(args, cfg, mode, f32g, fwd, stream, &clusters);
  if (e == cudaSuccess) {
    note_launch();
    if (verbose())
      fprintf(stderr, "[vpd] fused JSD%s: V=%lld cluster=%d workers=%d R=%d W=%d smem=%zu B%s, %d clusters\n",
              fwd ? " forward" : "", static_cast<long long>(s.vocab), cfg.C, cfg.nw, cfg.R, cfg.W, cfg.smem,
              gstage ? " (staged gradients)" : "", clusters);
  }
  return e;
}

}  // namespace vpd
