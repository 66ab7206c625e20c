// vpd_api.cu -- the extern "C" entry points of libvpd (declared in vpd.h):
// argument validation on the host, before anything is launched, then dispatch
// to the kernels on the caller's stream. Nothing here allocates memory.

#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <vector>

#include "vpd.h"
#include "vpd_internal.h"
#include "vpd_linear.h"

namespace vpd {
// Reads and clears the device error word (defined with the fused kernel).
cudaError_t take_device_error(cudaStream_t stream, int* code);
// The teacher-cache pipeline (vpd_teacher_stream.cu).
cudaError_t teacher_stream(const vpd_view& s, const void* t_host, int32_t t_dtype, int64_t t_row_stride, double beta,
                           const float* grad_loss, float* loss, float* saved, const vpd_grad* ds, const vpd_grad* dt,
                           void* staging, int nstage, int64_t chunk_rows, cudaStream_t stream,
                           cudaStream_t copy_stream, vpd_status* st_out);
}  // namespace vpd

namespace {

thread_local char g_last_error[512] = "";
thread_local int64_t g_withhold_row = -1;  // vpd_test_withhold_copy

vpd_status fail(vpd_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return st;
}

vpd_status ok() {
  g_last_error[0] = '\0';
  return VPD_OK;
}

vpd_status cuda_fail(cudaError_t e, const char* what) {
  return fail(VPD_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

int elem_size(int dtype) { return dtype == VPD_F32 ? 4 : 2; }
bool dtype_ok(int dtype) { return dtype == VPD_F32 || dtype == VPD_BF16 || dtype == VPD_F16; }

vpd_status check_view(const vpd_view* v, const char* name, vpd::View* out) {
  if (!v) return fail(VPD_ERR_ARG, "%s: NULL view", name);
  if (!dtype_ok(v->dtype)) return fail(VPD_ERR_DTYPE, "%s: unknown dtype %d", name, v->dtype);
  if (v->rows < 0 || v->vocab < 0)
    return fail(VPD_ERR_SHAPE, "%s: negative rows or vocab", name);
  if (v->row_stride < v->vocab)
    return fail(VPD_ERR_SHAPE, "%s: row_stride %lld < vocab %lld", name, (long long)v->row_stride,
                (long long)v->vocab);
  if (v->rows_per_batch < 0 || (v->rows_per_batch > 0 && v->batch_stride < 0))
    return fail(VPD_ERR_SHAPE, "%s: bad batch layout", name);
  if (v->rows > 0 && v->vocab > 0) {
    if (!v->data) return fail(VPD_ERR_ARG, "%s: NULL data", name);
    if (reinterpret_cast<uintptr_t>(v->data) % elem_size(v->dtype))
      return fail(VPD_ERR_ARG, "%s: data not aligned to its element size", name);
  }
  out->data = static_cast<const char*>(v->data);
  out->dtype = v->dtype;
  out->rows = v->rows;
  out->vocab = v->vocab;
  out->map = {v->row_stride, v->rows_per_batch, v->batch_stride};
  return VPD_OK;
}

vpd_status check_pair(const vpd_view* s, const vpd_view* t, vpd::View* vs, vpd::View* vt) {
  vpd_status st = check_view(s, "student", vs);
  if (st != VPD_OK) return st;
  st = check_view(t, "teacher", vt);
  if (st != VPD_OK) return st;
  if (vs->rows != vt->rows || vs->vocab != vt->vocab)
    return fail(VPD_ERR_SHAPE, "student [%lld, %lld] and teacher [%lld, %lld] differ",
                (long long)vs->rows, (long long)vs->vocab, (long long)vt->rows,
                (long long)vt->vocab);
  if (vs->dtype != vt->dtype) return fail(VPD_ERR_DTYPE, "student and teacher dtypes differ");
  return VPD_OK;
}

vpd_status check_segments(const vpd_segments* seg, int64_t vocab, vpd::Segs* out) {
  if (!seg || seg->count == 0) {
    out->count = 1;
    out->off[0] = 0;
    out->off[1] = vocab;
    return VPD_OK;
  }
  if (seg->count < 0 || seg->count > VPD_MAX_SEGMENTS)
    return fail(VPD_ERR_ARG, "segment count %d outside [0, %d]", seg->count, VPD_MAX_SEGMENTS);
  if (!seg->widths) return fail(VPD_ERR_ARG, "NULL segment widths");
  out->count = seg->count;
  out->off[0] = 0;
  for (int k = 0; k < seg->count; ++k) {
    if (seg->widths[k] < 0) return fail(VPD_ERR_SHAPE, "segment %d has negative width", k);
    out->off[k + 1] = out->off[k] + seg->widths[k];
  }
  if (out->off[seg->count] != vocab)
    return fail(VPD_ERR_SHAPE, "segment widths sum to %lld, vocab is %lld",
                (long long)out->off[seg->count], (long long)vocab);
  return VPD_OK;
}

vpd_status check_grad(const vpd_grad* g, const char* name, int64_t vocab, int64_t rows,
                      vpd::Grad* out) {
  out->data = nullptr;
  out->dtype = VPD_F32;
  out->row_stride = 0;
  if (!g || !g->data) return VPD_OK;
  if (!dtype_ok(g->dtype)) return fail(VPD_ERR_DTYPE, "%s: unknown gradient dtype %d", name, g->dtype);
  if (g->row_stride < vocab)
    return fail(VPD_ERR_SHAPE, "%s: gradient row_stride < vocab", name);
  if (reinterpret_cast<uintptr_t>(g->data) % elem_size(g->dtype))
    return fail(VPD_ERR_ARG, "%s: gradient not aligned to its element size", name);
  if (rows > 0 && vocab > 0) out->data = static_cast<char*>(g->data);
  out->dtype = g->dtype;
  out->row_stride = g->row_stride;
  return VPD_OK;
}

vpd_status check_beta(double beta) {
  if (!(beta >= 0.0 && beta <= 1.0)) return fail(VPD_ERR_ARG, "beta %g outside [0, 1]", beta);
  return VPD_OK;
}

vpd_status check_grads_pair(const vpd_grad* ds, const vpd_grad* dt, const vpd::View& v,
                            vpd::Grad* gs, vpd::Grad* gt) {
  vpd_status st = check_grad(ds, "ds", v.vocab, v.rows, gs);
  if (st != VPD_OK) return st;
  st = check_grad(dt, "dt", v.vocab, v.rows, gt);
  if (st != VPD_OK) return st;
  if (gs->data && gt->data && gs->dtype != gt->dtype)
    return fail(VPD_ERR_DTYPE, "ds and dt must share one dtype");
  return VPD_OK;
}

// A non-blocking side stream and its fork / join events, per device and
// calling thread, created on first use and kept for the life of the thread.
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};

cudaError_t side_stream(SideStream** out) {
  thread_local SideStream ss[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  SideStream& x = ss[dev];
  if (!x.stream) {
    if ((e = cudaEventCreateWithFlags(&x.fork, cudaEventDisableTiming)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&x.join, cudaEventDisableTiming)) != cudaSuccess) return e;
    if ((e = cudaStreamCreateWithFlags(&x.stream, cudaStreamNonBlocking)) != cudaSuccess) return e;
  }
  *out = &x;
  return cudaSuccess;
}

#define VPD_TRY(x)                     \
  do {                                 \
    vpd_status _st = (x);              \
    if (_st != VPD_OK) return _st;     \
  } while (0)

#define VPD_CUDA(x, what)                          \
  do {                                             \
    cudaError_t _e = (x);                          \
    if (_e != cudaSuccess) return cuda_fail(_e, what); \
  } while (0)

}  // namespace

extern "C" {

// Forward-only calls take the single-read forward kernel in clusters of at
// most kForwardMaxCluster CTAs (130 or more SMs on this GPU); a row that needs
// larger clusters (V = 262144: 16 CTAs, 112 SMs) takes the streaming kernels,
// which use every SM (JSD: 10.7 ms two-pass against 12.1 single-read for
// 32768 rows). At V = 151936 the JSD forward takes 1.43 ms single-read against
// 1.69 two-pass for 8191 rows. The KL forward has a one-read streaming kernel
// of its own, faster than the single-read kernel's KL branch on long rows
// (V = 151936: 1.10 against 1.36 ms) and on short ones (V = 16032: 0.141
// against 0.147 ms), so it takes that kernel at every width.
constexpr int kForwardMaxCluster = 10;

vpd_status vpd_jsd_fwd(const vpd_view* s, const vpd_view* t, double beta, const vpd_segments* seg,
                       float* loss, float* saved, void* stream) {
  vpd::View vs, vt;
  vpd::Segs sg;
  VPD_TRY(check_pair(s, t, &vs, &vt));
  VPD_TRY(check_beta(beta));
  VPD_TRY(check_segments(seg, vs.vocab, &sg));
  if (vs.rows == 0) return ok();
  if (!loss || !saved) return fail(VPD_ERR_ARG, "vpd_jsd_fwd: loss and saved are required");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // beta = 0 / 1 are the KL branches: the online single-pass KL kernel reads
  // the inputs once too and writes the same loss and saved layout (the KL ops
  // take it at every width for that reason: it is faster than the cluster
  // kernel's KL branch)
  if (beta == 0.0 || beta == 1.0) {
    VPD_CUDA(vpd::launch_kl_fwd(vs, vt, beta == 1.0 ? 1 : 0, sg, loss, saved, st), "single-pass KL kernel");
    return ok();
  }
  // One read of the inputs by the single-read forward kernel when it fits in
  // clusters that cover most SMs; else the two streaming passes on every SM.
  // Vocabulary segments change only the grouping of the statistics merge
  // (the kernel merges its CTA slices with the same MAX / SUM merge), so a
  // segmented call takes the single-read kernel too.
  {
    const vpd::Grad none{nullptr, 0, 0};
    // as in vpd_jsd_fwdbwd: the last rows go to the SMs the clusters leave
    // idle; with them the forward kernel may take clusters of up to 16 CTAs
    // (V = 262144: 9.16 ms with 7970 rows on the 40 idle SMs, against 9.93 ms
    // for the two streaming passes, 32768 rows)
    int64_t side = 0;
    int idle = 0;
    vpd::fused_idle_split(vs, none, none, 16, &side, &idle);
    if (side > 0) {
      SideStream* ss = nullptr;
      VPD_CUDA(side_stream(&ss), "creating the side stream");
      const int64_t nf = vs.rows - side;
      vpd::View fs = vs, ft = vt, ss_v = vs, st_v = vt;
      fs.rows = ft.rows = nf;
      ss_v.rows = st_v.rows = side;
      // the side views start at row nf of the caller's views (mid-batch too)
      ss_v.map.first += nf;
      st_v.map.first += nf;
      VPD_CUDA(cudaEventRecord(ss->fork, st), "forking the side stream");
      VPD_CUDA(cudaStreamWaitEvent(ss->stream, ss->fork, 0), "forking the side stream");
      cudaError_t e = vpd::launch_jsd_fused(fs, ft, beta, nullptr, loss, saved, none, none, st, -1, 16);
      if (e == cudaSuccess) {
        {
          vpd::GridCap cap(idle);
          float* sv = saved + nf * VPD_SAVED_PAIR;
          VPD_CUDA(vpd::launch_pair_stats(ss_v, st_v, sg, sv, ss->stream), "paired statistics kernel");
          VPD_CUDA(vpd::launch_jsd_div(ss_v, st_v, beta, loss + nf, sv, ss->stream), "divergence kernel");
        }
        VPD_CUDA(cudaEventRecord(ss->join, ss->stream), "joining the side stream");
        VPD_CUDA(cudaStreamWaitEvent(st, ss->join, 0), "joining the side stream");
        return ok();
      }
      VPD_CUDA(cudaEventRecord(ss->join, ss->stream), "joining the side stream");
      VPD_CUDA(cudaStreamWaitEvent(st, ss->join, 0), "joining the side stream");
      if (e != cudaErrorNotSupported) return cuda_fail(e, "fused single-read kernel");
    }
    cudaError_t e = vpd::launch_jsd_fused(vs, vt, beta, nullptr, loss, saved, none, none, st, -1,
                                          kForwardMaxCluster);
    if (e == cudaSuccess) return ok();
    if (e != cudaErrorNotSupported) return cuda_fail(e, "fused single-read kernel");
  }
  VPD_CUDA(vpd::launch_pair_stats(vs, vt, sg, saved, st), "paired statistics kernel");
  VPD_CUDA(vpd::launch_jsd_div(vs, vt, beta, loss, saved, st), "divergence kernel");
  return ok();
}

vpd_status vpd_jsd_bwd(const vpd_view* s, const vpd_view* t, double beta, const vpd_segments* seg,
                       const float* grad_loss, const float* saved, const vpd_grad* ds,
                       const vpd_grad* dt, void* stream) {
  vpd::View vs, vt;
  vpd::Segs sg;
  vpd::Grad gs, gt;
  VPD_TRY(check_pair(s, t, &vs, &vt));
  VPD_TRY(check_beta(beta));
  VPD_TRY(check_segments(seg, vs.vocab, &sg));
  VPD_TRY(check_grads_pair(ds, dt, vs, &gs, &gt));
  if (vs.rows == 0 || (!gs.data && !gt.data)) return ok();
  if (!saved) return fail(VPD_ERR_ARG, "vpd_jsd_bwd: saved is required");
  VPD_CUDA(vpd::launch_pair_bwd(vs, vt, beta, grad_loss, saved, gs, gt,
                                static_cast<cudaStream_t>(stream)),
           "backward kernel");
  return ok();
}

vpd_status vpd_jsd_fwdbwd(const vpd_view* s, const vpd_view* t, double beta,
                          const vpd_segments* seg, const float* grad_loss, float* loss,
                          float* saved, const vpd_grad* ds, const vpd_grad* dt, void* stream) {
  vpd::View vs, vt;
  vpd::Segs sg;
  vpd::Grad gs, gt;
  VPD_TRY(check_pair(s, t, &vs, &vt));
  VPD_TRY(check_beta(beta));
  VPD_TRY(check_segments(seg, vs.vocab, &sg));
  VPD_TRY(check_grads_pair(ds, dt, vs, &gs, &gt));
  if (vs.rows == 0) return ok();
  if (!loss || !saved) return fail(VPD_ERR_ARG, "vpd_jsd_fwdbwd: loss and saved are required");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The single-read kernel merges statistics over its CTA slices with the
  // same MAX / SUM merge the segments define, so a segmented call takes it
  // too (the side rows' streaming kernels merge segment by segment).
  {
    // The clusters of the single-read kernel leave some SMs idle (at V =
    // 151936, 15 clusters of 9 CTAs use 135 of 152 SMs). The last rows of the
    // call go to the streaming kernels on a side stream, capped to as many
    // CTAs as fit those SMs; the fused grid is submitted first, so its
    // clusters take their SMs before the side CTAs arrive (which cannot share
    // an SM with a fused CTA: its registers are taken).
    int64_t side = 0;
    int idle = 0;
    if (g_withhold_row < 0) vpd::fused_idle_split(vs, gs, gt, 16, &side, &idle);
    if (side > 0) {
      SideStream* ss = nullptr;
      VPD_CUDA(side_stream(&ss), "creating the side stream");
      const int64_t nf = vs.rows - side;
      vpd::View fs = vs, ft = vt, ss_v = vs, st_v = vt;
      fs.rows = ft.rows = nf;
      ss_v.rows = st_v.rows = side;
      // the side views start at row nf of the caller's views (mid-batch too)
      ss_v.map.first += nf;
      st_v.map.first += nf;
      vpd::Grad sgs = gs, sgt = gt;
      if (gs.data) sgs.data = gs.data + nf * gs.row_stride * (gs.dtype == VPD_F32 ? 4 : 2);
      if (gt.data) sgt.data = gt.data + nf * gt.row_stride * (gt.dtype == VPD_F32 ? 4 : 2);
      VPD_CUDA(cudaEventRecord(ss->fork, st), "forking the side stream");
      VPD_CUDA(cudaStreamWaitEvent(ss->stream, ss->fork, 0), "forking the side stream");
      cudaError_t e = vpd::launch_jsd_fused(fs, ft, beta, grad_loss, loss, saved, gs, gt, st, -1);
      if (e == cudaSuccess) {
        {
          // measured: the three streaming passes, two CTAs per idle SM each,
          // run about as fast per SM as one kernel doing all three per row
          vpd::GridCap cap(idle);
          float* sv = saved + nf * VPD_SAVED_PAIR;
          const float* sg_l = grad_loss ? grad_loss + nf : nullptr;
          VPD_CUDA(vpd::launch_pair_stats(ss_v, st_v, sg, sv, ss->stream), "paired statistics kernel");
          VPD_CUDA(vpd::launch_jsd_div(ss_v, st_v, beta, loss + nf, sv, ss->stream), "divergence kernel");
          VPD_CUDA(vpd::launch_pair_bwd(ss_v, st_v, beta, sg_l, sv, sgs, sgt, ss->stream), "backward kernel");
        }
        VPD_CUDA(cudaEventRecord(ss->join, ss->stream), "joining the side stream");
        VPD_CUDA(cudaStreamWaitEvent(st, ss->join, 0), "joining the side stream");
        return ok();
      }
      // no fused launch: join the (empty) side stream and take the plain path below
      VPD_CUDA(cudaEventRecord(ss->join, ss->stream), "joining the side stream");
      VPD_CUDA(cudaStreamWaitEvent(st, ss->join, 0), "joining the side stream");
      if (e != cudaErrorNotSupported) return cuda_fail(e, "fused single-read kernel");
    }
    cudaError_t e = vpd::launch_jsd_fused(vs, vt, beta, grad_loss, loss, saved, gs, gt, st, g_withhold_row);
    if (e == cudaSuccess) g_withhold_row = -1;
    if (e == cudaSuccess) return ok();
    if (e != cudaErrorNotSupported) return cuda_fail(e, "fused single-read kernel");
  }
  VPD_CUDA(vpd::launch_pair_stats(vs, vt, sg, saved, st), "paired statistics kernel");
  VPD_CUDA(vpd::launch_jsd_div(vs, vt, beta, loss, saved, st), "divergence kernel");
  VPD_CUDA(vpd::launch_pair_bwd(vs, vt, beta, grad_loss, saved, gs, gt, st), "backward kernel");
  return ok();
}

vpd_status vpd_jsd_plan(const vpd_view* s, const vpd_view* t, const vpd_segments* seg, const vpd_grad* ds,
                        const vpd_grad* dt, int64_t* fused_rows, int64_t* idle_sm_rows, int32_t* launches) {
  vpd::View vs, vt;
  vpd::Segs sg;
  vpd::Grad gs, gt;
  VPD_TRY(check_pair(s, t, &vs, &vt));
  VPD_TRY(check_segments(seg, vs.vocab, &sg));
  VPD_TRY(check_grads_pair(ds, dt, vs, &gs, &gt));
  const bool fwd = !gs.data && !gt.data;
  int max_cluster = fwd ? kForwardMaxCluster : 16;
  int64_t fr = 0, side = 0;
  int32_t n = 0;
  if (vs.rows > 0) {
    int idle = 0;
    vpd::fused_idle_split(vs, gs, gt, 16, &side, &idle);
    if (side > 0) max_cluster = 16;
    vpd::View fs = vs, ft = vt;
    fs.rows = ft.rows = vs.rows - side;
    const cudaError_t e =
        vpd::launch_jsd_fused(fs, ft, 0.5, nullptr, nullptr, nullptr, gs, gt, nullptr, -1, max_cluster, true);
    if (e == cudaSuccess) {
      fr = fs.rows;
      n = 1 + (side > 0 ? (fwd ? 2 : 3) : 0);
    } else {
      side = 0;
      n = fwd ? 2 : 3;
    }
  }
  if (fused_rows) *fused_rows = fr;
  if (idle_sm_rows) *idle_sm_rows = side;
  if (launches) *launches = n;
  return ok();
}

vpd_status vpd_kl_fwd(const vpd_view* s, const vpd_view* t, int32_t reverse,
                      const vpd_segments* seg, float* loss, float* saved, void* stream) {
  vpd::View vs, vt;
  vpd::Segs sg;
  VPD_TRY(check_pair(s, t, &vs, &vt));
  VPD_TRY(check_segments(seg, vs.vocab, &sg));
  if (vs.rows == 0) return ok();
  if (!loss) return fail(VPD_ERR_ARG, "vpd_kl_fwd: loss is required");
  VPD_CUDA(vpd::launch_kl_fwd(vs, vt, reverse ? 1 : 0, sg, loss, saved,
                              static_cast<cudaStream_t>(stream)),
           "single-pass KL kernel");
  return ok();
}

vpd_status vpd_kl_bwd(const vpd_view* s, const vpd_view* t, int32_t reverse,
                      const vpd_segments* seg, const float* grad_loss, const float* saved,
                      const vpd_grad* ds, const vpd_grad* dt, void* stream) {
  vpd::View vs, vt;
  vpd::Segs sg;
  vpd::Grad gs, gt;
  VPD_TRY(check_pair(s, t, &vs, &vt));
  VPD_TRY(check_segments(seg, vs.vocab, &sg));
  VPD_TRY(check_grads_pair(ds, dt, vs, &gs, &gt));
  if (vs.rows == 0 || (!gs.data && !gt.data)) return ok();
  if (!saved) return fail(VPD_ERR_ARG, "vpd_kl_bwd: saved is required");
  VPD_CUDA(vpd::launch_pair_bwd(vs, vt, reverse ? 1.0 : 0.0, grad_loss, saved, gs, gt,
                                static_cast<cudaStream_t>(stream)),
           "backward kernel");
  return ok();
}

vpd_status vpd_entropy_fwd(const vpd_view* x, const vpd_segments* seg, float* out, float* saved,
                           void* stream) {
  vpd::View vx;
  vpd::Segs sg;
  VPD_TRY(check_view(x, "x", &vx));
  VPD_TRY(check_segments(seg, vx.vocab, &sg));
  if (vx.rows == 0) return ok();
  if (!out) return fail(VPD_ERR_ARG, "vpd_entropy_fwd: out is required");
  VPD_CUDA(vpd::launch_entropy_fwd(vx, sg, out, saved, static_cast<cudaStream_t>(stream)),
           "entropy kernel");
  return ok();
}

vpd_status vpd_entropy_bwd(const vpd_view* x, const vpd_segments* seg, const float* grad_out,
                           const float* saved, const vpd_grad* dx, void* stream) {
  vpd::View vx;
  vpd::Segs sg;
  vpd::Grad gx;
  VPD_TRY(check_view(x, "x", &vx));
  VPD_TRY(check_segments(seg, vx.vocab, &sg));
  VPD_TRY(check_grad(dx, "dx", vx.vocab, vx.rows, &gx));
  if (vx.rows == 0 || !gx.data) return ok();
  if (!saved) return fail(VPD_ERR_ARG, "vpd_entropy_bwd: saved is required");
  VPD_CUDA(vpd::launch_entropy_bwd(vx, grad_out, saved, gx, static_cast<cudaStream_t>(stream)),
           "entropy backward kernel");
  return ok();
}

}  // extern "C"

namespace {

// The pages' synchronising index check ([ops page], review thread "Provide a
// path for reusing validated shard metadata"): without a device flag the
// indices are copied to the host on the caller's stream and checked before
// anything is launched or written.
vpd_status check_indices_on_host(const int64_t* index, int64_t count, int64_t ignore_index, int64_t vocab,
                                 cudaStream_t st, const char* who) {
  std::vector<int64_t> h(static_cast<size_t>(count));
  VPD_CUDA(cudaMemcpyAsync(h.data(), index, h.size() * sizeof(int64_t), cudaMemcpyDeviceToHost, st), "reading index");
  VPD_CUDA(cudaStreamSynchronize(st), "reading index");
  for (size_t i = 0; i < h.size(); ++i)
    if (h[i] != ignore_index && (h[i] < 0 || h[i] >= vocab))
      return fail(VPD_ERR_INDEX, "%s: index[%lld] = %lld outside [0, %lld)", who, static_cast<long long>(i),
                  static_cast<long long>(h[i]), static_cast<long long>(vocab));
  return VPD_OK;
}

vpd_status check_temperature(double temperature, float* inv) {
  if (!(temperature > 0.0) || !std::isfinite(temperature))
    return fail(VPD_ERR_ARG, "temperature %g must be positive and finite", temperature);
  *inv = static_cast<float>(1.0 / temperature);
  return VPD_OK;
}

// Shared forward of the selection ops: validation, the flag or the host index
// check, then the kernel.
vpd_status select_fwd(const vpd_view* x, const vpd_segments* seg, const int64_t* index, int32_t k,
                      int64_t ignore_index, double temperature, int mode, const float* teacher_logp, float* out,
                      float* row_out, float* saved, int32_t* err_flag, void* stream, const char* who) {
  vpd::View vx;
  vpd::Segs sg;
  float inv = 1.f;
  VPD_TRY(check_view(x, "x", &vx));
  VPD_TRY(check_segments(seg, vx.vocab, &sg));
  VPD_TRY(check_temperature(temperature, &inv));
  if (k < 1) return fail(VPD_ERR_ARG, "%s: k must be >= 1", who);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (err_flag) VPD_CUDA(cudaMemsetAsync(err_flag, 0, sizeof(int32_t), st), "clearing err_flag");
  if (vx.rows == 0) return ok();
  if (!index || (mode == 0 && !out) || (mode != 0 && !row_out) || (mode == 2 && !teacher_logp))
    return fail(VPD_ERR_ARG, "%s: a required pointer is NULL", who);
  if (!err_flag) VPD_TRY(check_indices_on_host(index, vx.rows * k, ignore_index, vx.vocab, st, who));
  VPD_CUDA(vpd::launch_select_fwd(vx, sg, index, k, ignore_index, inv, mode, teacher_logp, out, row_out, saved,
                                  err_flag, st),
           "selection kernel");
  return ok();
}

vpd_status select_bwd(const vpd_view* x, const vpd_segments* seg, const int64_t* index, int32_t k,
                      int64_t ignore_index, double temperature, int mode, const float* teacher_logp,
                      const float* grad, const float* saved, const vpd_grad* dx, void* stream, const char* who) {
  vpd::View vx;
  vpd::Segs sg;
  vpd::Grad gx;
  float inv = 1.f;
  VPD_TRY(check_view(x, "x", &vx));
  VPD_TRY(check_segments(seg, vx.vocab, &sg));
  VPD_TRY(check_grad(dx, "dx", vx.vocab, vx.rows, &gx));
  VPD_TRY(check_temperature(temperature, &inv));
  if (k < 1) return fail(VPD_ERR_ARG, "%s: k must be >= 1", who);
  if (vx.rows == 0 || !gx.data) return ok();
  if (!index || !saved || (mode == 2 && !teacher_logp))
    return fail(VPD_ERR_ARG, "%s: index, saved (and the teacher log-probs) are required", who);
  VPD_CUDA(vpd::launch_select_bwd(vx, index, k, ignore_index, inv, mode, teacher_logp, grad, saved, gx,
                                  static_cast<cudaStream_t>(stream)),
           "selection backward kernel");
  return ok();
}

}  // namespace

extern "C" {

vpd_status vpd_logprobs_fwd(const vpd_view* x, const vpd_segments* seg, const int64_t* index, int32_t k,
                            int64_t ignore_index, float* out, float* saved, int32_t* err_flag, void* stream) {
  return select_fwd(x, seg, index, k, ignore_index, 1.0, 0, nullptr, out, nullptr, saved, err_flag, stream,
                    "vpd_logprobs_fwd");
}

vpd_status vpd_logprobs_bwd(const vpd_view* x, const vpd_segments* seg, const int64_t* index, int32_t k,
                            int64_t ignore_index, const float* grad_out, const float* saved, const vpd_grad* dx,
                            void* stream) {
  return select_bwd(x, seg, index, k, ignore_index, 1.0, 0, nullptr, grad_out, saved, dx, stream,
                    "vpd_logprobs_bwd");
}

vpd_status vpd_cross_entropy_fwd(const vpd_view* x, const vpd_segments* seg, const int64_t* labels,
                                 int64_t ignore_index, double temperature, float* loss, float* saved,
                                 int32_t* err_flag, void* stream) {
  return select_fwd(x, seg, labels, 1, ignore_index, temperature, 1, nullptr, nullptr, loss, saved, err_flag, stream,
                    "vpd_cross_entropy_fwd");
}

vpd_status vpd_cross_entropy_bwd(const vpd_view* x, const vpd_segments* seg, const int64_t* labels,
                                 int64_t ignore_index, double temperature, const float* grad_loss, const float* saved,
                                 const vpd_grad* dx, void* stream) {
  return select_bwd(x, seg, labels, 1, ignore_index, temperature, 1, nullptr, grad_loss, saved, dx, stream,
                    "vpd_cross_entropy_bwd");
}

vpd_status vpd_topk_kl_fwd(const vpd_view* s, const vpd_segments* seg, const int64_t* index, int32_t k,
                           int64_t ignore_index, const float* teacher_logp, double temperature, float* kl,
                           float* saved, int32_t* err_flag, void* stream) {
  return select_fwd(s, seg, index, k, ignore_index, temperature, 2, teacher_logp, nullptr, kl, saved, err_flag,
                    stream, "vpd_topk_kl_fwd");
}

vpd_status vpd_topk_kl_bwd(const vpd_view* s, const vpd_segments* seg, const int64_t* index, int32_t k,
                           int64_t ignore_index, const float* teacher_logp, double temperature,
                           const float* grad_kl, const float* saved, const vpd_grad* ds, void* stream) {
  return select_bwd(s, seg, index, k, ignore_index, temperature, 2, teacher_logp, grad_kl, saved, ds, stream,
                    "vpd_topk_kl_bwd");
}

}  // extern "C"

namespace {

vpd_status check_heads(const vpd_linear_heads* p, vpd::LinearProblem* out) {
  if (!p) return fail(VPD_ERR_ARG, "NULL heads");
  if (p->rows < 0 || p->vocab < 1) return fail(VPD_ERR_SHAPE, "rows must be >= 0 and vocab >= 1");
  if (p->vocab % 8) return fail(VPD_ERR_SHAPE, "vocab %lld is not a multiple of 8", (long long)p->vocab);
  if (p->hidden_s < 64 || p->hidden_s % 64 || p->hidden_t < 64 || p->hidden_t % 64)
    return fail(VPD_ERR_SHAPE, "hidden sizes must be positive multiples of 64");
  const int64_t ld[4] = {p->ld_hs, p->ld_ws, p->ld_ht, p->ld_wt};
  const int64_t hid[4] = {p->hidden_s, p->hidden_s, p->hidden_t, p->hidden_t};
  const void* ptr[4] = {p->h_s, p->w_s, p->h_t, p->w_t};
  for (int i = 0; i < 4; ++i) {
    if (ld[i] < hid[i] || ld[i] % 8) return fail(VPD_ERR_SHAPE, "row stride %d must be >= hidden and a multiple of 8", i);
    if (p->rows > 0 && (!ptr[i] || (reinterpret_cast<uintptr_t>(ptr[i]) & 15u)))
      return fail(VPD_ERR_ARG, "heads: NULL or not 16-byte aligned operand %d", i);
  }
  *out = vpd::LinearProblem{p->h_s, p->w_s, p->h_t, p->w_t, p->rows, p->vocab, p->hidden_s, p->hidden_t,
                            p->ld_hs, p->ld_ws, p->ld_ht, p->ld_wt, 0.0};
  return VPD_OK;
}

}  // namespace

extern "C" {

vpd_status vpd_jsd_fwdbwd_teacher_stream(const vpd_view* s, const void* t_host, int32_t t_dtype,
                                         int64_t t_row_stride, double beta, const float* grad_loss, float* loss,
                                         float* saved, const vpd_grad* ds, const vpd_grad* dt, void* staging,
                                         size_t staging_bytes, int64_t chunk_rows, void* stream,
                                         void* copy_stream) {
  vpd::View vs;
  VPD_TRY(check_view(s, "student", &vs));
  VPD_TRY(check_beta(beta));
  if (!dtype_ok(t_dtype) || t_dtype != vs.dtype) return fail(VPD_ERR_DTYPE, "teacher dtype must equal the student's");
  if (vs.map.rows_per_batch > 0) return fail(VPD_ERR_SHAPE, "the student view must be plain 2-D [N, V]");
  if (t_row_stride < vs.vocab) return fail(VPD_ERR_SHAPE, "teacher row stride < vocab");
  if (chunk_rows < 1) return fail(VPD_ERR_ARG, "chunk_rows must be >= 1");
  if (vs.rows == 0) return ok();
  if (!t_host || !loss || !saved || !staging)
    return fail(VPD_ERR_ARG, "vpd_jsd_fwdbwd_teacher_stream: t_host, loss, saved and staging are required");
  if (vs.vocab == 0) return vpd_jsd_fwdbwd(s, s, beta, nullptr, grad_loss, loss, saved, ds, dt, stream);
  // the cache must be pinned (page-locked or registered) host memory: a
  // pageable buffer would be copied through a synchronous temporary
  cudaPointerAttributes attr;
  VPD_CUDA(cudaPointerGetAttributes(&attr, t_host), "inspecting the teacher cache");
  if (attr.type != cudaMemoryTypeHost) return fail(VPD_ERR_ARG, "the teacher cache must be pinned host memory");
  const int64_t es = elem_size(t_dtype);
  const size_t chunk_bytes = static_cast<size_t>(chunk_rows) * static_cast<size_t>(vs.vocab * es);
  int64_t nstage = static_cast<int64_t>(staging_bytes / chunk_bytes);
  if (nstage < 2) return fail(VPD_ERR_ARG, "staging must hold at least two chunks (%zu bytes)", 2 * chunk_bytes);
  if (nstage > 4) nstage = 4;
  if ((vs.vocab * es) % 16 || reinterpret_cast<uintptr_t>(staging) % 16)
    return fail(VPD_ERR_ARG, "staging must be 16-byte aligned and the row size a multiple of 16 bytes");
  vpd::Grad gs, gt;
  VPD_TRY(check_grads_pair(ds, dt, vs, &gs, &gt));
  vpd_status inner = VPD_OK;
  cudaError_t e = vpd::teacher_stream(*s, t_host, t_dtype, t_row_stride, beta, grad_loss, loss, saved, ds, dt,
                                      staging, static_cast<int>(nstage), chunk_rows,
                                      static_cast<cudaStream_t>(stream), static_cast<cudaStream_t>(copy_stream),
                                      &inner);
  if (inner != VPD_OK) return inner;
  VPD_CUDA(e, "teacher-cache pipeline");
  return ok();
}

vpd_status vpd_jsd_shard_stats(const vpd_view* s, const vpd_view* t, float* saved, float* xbuf, void* stream) {
  vpd::View vs, vt;
  VPD_TRY(check_pair(s, t, &vs, &vt));
  if (vs.rows == 0) return ok();
  if (!saved || !xbuf) return fail(VPD_ERR_ARG, "vpd_jsd_shard_stats: saved and xbuf are required");
  VPD_CUDA(vpd::shard_stats(vs, vt, saved, xbuf, static_cast<cudaStream_t>(stream)), "shard statistics");
  return ok();
}

vpd_status vpd_jsd_shard_rescale(int64_t rows, float* saved, float* xbuf, void* stream) {
  if (rows < 0) return fail(VPD_ERR_SHAPE, "rows must be >= 0");
  if (rows == 0) return ok();
  if (!saved || !xbuf) return fail(VPD_ERR_ARG, "vpd_jsd_shard_rescale: saved and xbuf are required");
  VPD_CUDA(vpd::shard_rescale(rows, saved, xbuf, static_cast<cudaStream_t>(stream)), "shard rescale");
  return ok();
}

vpd_status vpd_jsd_shard_divergence(const vpd_view* s, const vpd_view* t, double beta, float* loss, float* saved,
                                    float* xbuf, void* stream) {
  vpd::View vs, vt;
  VPD_TRY(check_pair(s, t, &vs, &vt));
  VPD_TRY(check_beta(beta));
  if (vs.rows == 0) return ok();
  if (!loss || !saved || !xbuf) return fail(VPD_ERR_ARG, "vpd_jsd_shard_divergence: loss, saved and xbuf are required");
  VPD_CUDA(vpd::shard_divergence(vs, vt, beta, loss, saved, xbuf, static_cast<cudaStream_t>(stream)),
           "shard divergence");
  return ok();
}

vpd_status vpd_jsd_shard_finish(int64_t rows, double beta, float* saved, const float* xbuf, float* loss,
                                void* stream) {
  VPD_TRY(check_beta(beta));
  if (rows < 0) return fail(VPD_ERR_SHAPE, "rows must be >= 0");
  if (rows == 0) return ok();
  if (!saved || !xbuf || !loss) return fail(VPD_ERR_ARG, "vpd_jsd_shard_finish: saved, xbuf and loss are required");
  VPD_CUDA(vpd::shard_finish(rows, beta, saved, xbuf, loss, static_cast<cudaStream_t>(stream)), "shard finish");
  return ok();
}

vpd_status vpd_jsd_linear_workspace(const vpd_linear_heads* heads, int32_t student_grads, int32_t teacher_grads,
                                    size_t* fwd_bytes, size_t* bwd_bytes) {
  vpd::LinearProblem p;
  VPD_TRY(check_heads(heads, &p));
  if (fwd_bytes) *fwd_bytes = p.rows ? vpd::linear_fwd_workspace(p.rows, p.vocab) : 0;
  if (bwd_bytes)
    *bwd_bytes = p.rows ? vpd::linear_bwd_workspace(p.rows, p.vocab, p.hs, p.ht, student_grads != 0,
                                                    teacher_grads != 0, vpd::kLinearChunkRows)
                        : 0;
  return ok();
}

vpd_status vpd_jsd_linear_fwd(const vpd_linear_heads* heads, double beta, float* loss, float* saved,
                              void* workspace, size_t workspace_bytes, void* stream) {
  vpd::LinearProblem p;
  VPD_TRY(check_heads(heads, &p));
  VPD_TRY(check_beta(beta));
  if (p.rows == 0) return ok();
  if (!loss || !saved || !workspace) return fail(VPD_ERR_ARG, "vpd_jsd_linear_fwd: loss, saved and workspace are required");
  if (reinterpret_cast<uintptr_t>(workspace) & 15u) return fail(VPD_ERR_ARG, "workspace not 16-byte aligned");
  if (workspace_bytes < vpd::linear_fwd_workspace(p.rows, p.vocab))
    return fail(VPD_ERR_ARG, "workspace of %zu bytes, %zu needed", workspace_bytes,
                vpd::linear_fwd_workspace(p.rows, p.vocab));
  p.beta = beta;
  VPD_CUDA(vpd::linear_jsd_forward(p, loss, saved, workspace, workspace_bytes, static_cast<cudaStream_t>(stream)),
           "fused-linear forward");
  return ok();
}

vpd_status vpd_jsd_linear_fwd_noalloc(const vpd_linear_heads* heads, double beta, float* loss, float* saved,
                                      void* stream) {
  vpd::LinearProblem p;
  VPD_TRY(check_heads(heads, &p));
  VPD_TRY(check_beta(beta));
  if (p.rows == 0) return ok();
  if (!loss || !saved) return fail(VPD_ERR_ARG, "vpd_jsd_linear_fwd_noalloc: loss and saved are required");
  const size_t need = vpd::linear_fwd_min_workspace(p.rows);
  if (need > vpd::kLinearNoAllocMaxBytes)
    return fail(VPD_ERR_SHAPE,
                "vpd_jsd_linear_fwd_noalloc: this problem needs %zu bytes of scratch, the built-in array holds %zu; "
                "use vpd_jsd_linear_fwd with a workspace",
                need, vpd::kLinearNoAllocMaxBytes);
  void* scratch = nullptr;
  VPD_CUDA(vpd::linear_scratch(&scratch), "looking up the built-in scratch array");
  p.beta = beta;
  VPD_CUDA(vpd::linear_jsd_forward(p, loss, saved, scratch, vpd::kLinearNoAllocMaxBytes,
                                   static_cast<cudaStream_t>(stream)),
           "fused-linear forward");
  return ok();
}

vpd_status vpd_jsd_linear_bwd(const vpd_linear_heads* heads, double beta, const float* grad_loss, const float* loss,
                              const float* saved, float* dh_s, float* dw_s, float* dh_t, float* dw_t, void* workspace,
                              size_t workspace_bytes, void* stream) {
  vpd::LinearProblem p;
  VPD_TRY(check_heads(heads, &p));
  VPD_TRY(check_beta(beta));
  const bool student = dh_s || dw_s, teacher = dh_t || dw_t;
  if (p.rows == 0 || (!student && !teacher)) return ok();
  if (!loss || !saved || !workspace) return fail(VPD_ERR_ARG, "vpd_jsd_linear_bwd: loss, saved and workspace are required");
  if (reinterpret_cast<uintptr_t>(workspace) & 15u) return fail(VPD_ERR_ARG, "workspace not 16-byte aligned");
  const size_t need = vpd::linear_bwd_workspace(p.rows, p.vocab, p.hs, p.ht, student, teacher, vpd::kLinearChunkRows);
  if (workspace_bytes < need) return fail(VPD_ERR_ARG, "workspace of %zu bytes, %zu needed", workspace_bytes, need);
  p.beta = beta;
  VPD_CUDA(vpd::linear_jsd_backward(p, grad_loss, loss, saved, dh_s, dw_s, dh_t, dw_t, workspace, workspace_bytes,
                                    vpd::kLinearChunkRows, static_cast<cudaStream_t>(stream)),
           "fused-linear backward");
  return ok();
}

const char* vpd_status_string(vpd_status status) {
  switch (status) {
    case VPD_OK: return "VPD_OK";
    case VPD_ERR_ARG: return "VPD_ERR_ARG";
    case VPD_ERR_DTYPE: return "VPD_ERR_DTYPE";
    case VPD_ERR_SHAPE: return "VPD_ERR_SHAPE";
    case VPD_ERR_INDEX: return "VPD_ERR_INDEX";
    case VPD_ERR_CUDA: return "VPD_ERR_CUDA";
    case VPD_ERR_TIMEOUT: return "VPD_ERR_TIMEOUT";
    case VPD_ERR_UNSUPPORTED: return "VPD_ERR_UNSUPPORTED";
  }
  return "unknown vpd_status";
}

const char* vpd_last_error(void) { return g_last_error; }

int32_t vpd_abi_version(void) { return VPD_ABI_VERSION; }

uint64_t vpd_launch_count(void) { return vpd::launch_count(); }

vpd_status vpd_test_withhold_copy(int64_t row) {
  g_withhold_row = row < 0 ? -1 : row;
  return ok();
}

vpd_status vpd_device_status(void* stream) {
  int code = 0;
  VPD_CUDA(vpd::take_device_error(static_cast<cudaStream_t>(stream), &code), "reading device status");
  int lin = 0;
  VPD_CUDA(vpd::take_linear_error(static_cast<cudaStream_t>(stream), &lin), "reading device status");
  code |= lin;
  if (code)
    return fail(VPD_ERR_TIMEOUT, "a bounded device-side wait gave up (code %d)", code);
  return ok();
}

}  // extern "C"
