// vpd_fused.cu -- single-read fused JSD forward+backward on thread-block
// clusters (placeholder until the cluster kernel lands: every shape takes the
// streaming path), and the device error word read by vpd_device_status.

#include <cuda_runtime.h>

#include "vpd_internal.h"

namespace vpd {

// Set (never cleared) by a kernel whose bounded wait gave up; read and cleared
// by take_device_error.
__device__ int g_device_error = 0;

cudaError_t take_device_error(cudaStream_t stream, int* code) {
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbol(code, g_device_error, sizeof(int));
  if (e != cudaSuccess) return e;
  if (*code) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
  }
  return e;
}

cudaError_t launch_jsd_fused(const View&, const View&, double, const float*, float*, float*,
                             const Grad&, const Grad&, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace vpd
