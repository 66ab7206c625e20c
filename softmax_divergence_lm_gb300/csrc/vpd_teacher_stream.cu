// vpd_teacher_stream.cu -- JSD forward+backward with the teacher logits in a
// pinned host cache: the teacher rows travel to the device chunk by chunk on
// the caller's copy stream into a ring of caller-owned staging buffers, and
// each chunk's fused JSD runs on the compute stream as soon as its rows have
// arrived, while the next chunks copy. This is the teacher-cache path of
// "Add an opt-in vocabulary-parallel KL route to OPSD" (DeepSpeedExamples pull
// request #1019), section "Update: copy teacher-cache chunks from pinned
// memory": copies from a pinned buffer, never through a pageable temporary,
// overlapped with the loss kernels.
//
// One chunk is one cudaMemcpy2DAsync (rows of the host cache with its own row
// pitch into dense staging rows). Ordering uses two events per staging buffer
// (copied, consumed), created once per device and thread and reused.

#include <cuda_runtime.h>

#include <cstdint>

#include "vpd.h"
#include "vpd_internal.h"

namespace vpd {

namespace {

constexpr int kMaxStage = 4;

struct StreamEvents {
  bool ready = false;
  cudaEvent_t start = nullptr;
  cudaEvent_t copied[kMaxStage] = {};
  cudaEvent_t consumed[kMaxStage] = {};
};

// Events of the calling thread on the current device (created on first use).
cudaError_t events_for(StreamEvents** out) {
  thread_local StreamEvents ev[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  StreamEvents& x = ev[dev];
  if (!x.ready) {
    if ((e = cudaEventCreateWithFlags(&x.start, cudaEventDisableTiming)) != cudaSuccess) return e;
    for (int i = 0; i < kMaxStage; ++i) {
      if ((e = cudaEventCreateWithFlags(&x.copied[i], cudaEventDisableTiming)) != cudaSuccess) return e;
      if ((e = cudaEventCreateWithFlags(&x.consumed[i], cudaEventDisableTiming)) != cudaSuccess) return e;
    }
    x.ready = true;
  }
  *out = &x;
  return cudaSuccess;
}

}  // namespace

// Host-side checks are done by the caller (the C entry point); this runs the
// chunk loop. `run_chunk` launches the fused JSD of rows [r0, r0 + rows) with
// the teacher chunk at `stage`.
template <class RunChunk>
cudaError_t teacher_stream_loop(const void* t_host, int64_t t_pitch_bytes, int64_t row_bytes, int64_t rows,
                                char* staging, int nstage, int64_t chunk_rows, cudaStream_t stream,
                                cudaStream_t copy_stream, RunChunk&& run_chunk) {
  StreamEvents* ev = nullptr;
  cudaError_t e = events_for(&ev);
  if (e != cudaSuccess) return e;
  // the staging buffers may still be read by earlier work on the compute stream
  if ((e = cudaEventRecord(ev->start, stream)) != cudaSuccess) return e;
  if ((e = cudaStreamWaitEvent(copy_stream, ev->start, 0)) != cudaSuccess) return e;
  const int64_t chunk_bytes = chunk_rows * row_bytes;
  int64_t c = 0;
  for (int64_t r0 = 0; r0 < rows; r0 += chunk_rows, ++c) {
    const int b = static_cast<int>(c % nstage);
    const int64_t n = rows - r0 < chunk_rows ? rows - r0 : chunk_rows;
    char* stage = staging + b * chunk_bytes;
    if (c >= nstage && (e = cudaStreamWaitEvent(copy_stream, ev->consumed[b], 0)) != cudaSuccess) return e;
    e = cudaMemcpy2DAsync(stage, static_cast<size_t>(row_bytes),
                          static_cast<const char*>(t_host) + r0 * t_pitch_bytes, static_cast<size_t>(t_pitch_bytes),
                          static_cast<size_t>(row_bytes), static_cast<size_t>(n), cudaMemcpyHostToDevice, copy_stream);
    if (e != cudaSuccess) return e;
    if ((e = cudaEventRecord(ev->copied[b], copy_stream)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(stream, ev->copied[b], 0)) != cudaSuccess) return e;
    if ((e = run_chunk(r0, n, stage)) != cudaSuccess) return e;
    if ((e = cudaEventRecord(ev->consumed[b], stream)) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace vpd

extern "C" vpd_status vpd_jsd_fwdbwd(const vpd_view* s, const vpd_view* t, double beta, const vpd_segments* seg,
                                     const float* grad_loss, float* loss, float* saved, const vpd_grad* ds,
                                     const vpd_grad* dt, void* stream);

namespace vpd {
cudaError_t teacher_stream(const vpd_view& s, const void* t_host, int32_t t_dtype, int64_t t_row_stride, double beta,
                           const float* grad_loss, float* loss, float* saved, const vpd_grad* ds, const vpd_grad* dt,
                           void* staging, int nstage, int64_t chunk_rows, cudaStream_t stream,
                           cudaStream_t copy_stream, vpd_status* st_out) {
  const int64_t es = t_dtype == VPD_F32 ? 4 : 2;
  const int64_t row_bytes = s.vocab * es;
  *st_out = VPD_OK;
  auto run_chunk = [&](int64_t r0, int64_t n, char* stage) -> cudaError_t {
    vpd_view sc = s;
    sc.data = static_cast<const char*>(s.data) + r0 * s.row_stride * (s.dtype == VPD_F32 ? 4 : 2);
    sc.rows = n;
    vpd_view tc{stage, t_dtype, n, s.vocab, s.vocab, 0, 0};
    vpd_grad dsc{}, dtc{};
    const vpd_grad* pds = nullptr;
    const vpd_grad* pdt = nullptr;
    if (ds && ds->data) {
      dsc = *ds;
      dsc.data = static_cast<char*>(ds->data) + r0 * ds->row_stride * (ds->dtype == VPD_F32 ? 4 : 2);
      pds = &dsc;
    }
    if (dt && dt->data) {
      dtc = *dt;
      dtc.data = static_cast<char*>(dt->data) + r0 * dt->row_stride * (dt->dtype == VPD_F32 ? 4 : 2);
      pdt = &dtc;
    }
    const vpd_status st = vpd_jsd_fwdbwd(&sc, &tc, beta, nullptr, grad_loss ? grad_loss + r0 : nullptr, loss + r0,
                                         saved + r0 * VPD_SAVED_PAIR, pds, pdt, stream);
    if (st != VPD_OK) {
      *st_out = st;
      return cudaErrorUnknown;
    }
    return cudaSuccess;
  };
  return teacher_stream_loop(t_host, t_row_stride * es, row_bytes, s.rows, static_cast<char*>(staging), nstage,
                             chunk_rows, stream, copy_stream, run_chunk);
}
}  // namespace vpd
