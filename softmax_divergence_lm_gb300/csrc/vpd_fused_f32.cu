// vpd_fused_f32.cu -- the fused single-read JSD kernels for fp32 logits
// (device code in vpd_fused.cuh), and this unit's device error word.
#include "vpd_fused.cuh"

namespace vpd {
namespace fused {

template cudaError_t launch_typed<InF32>(const FusedArgs&, const Config&, int, bool, bool, cudaStream_t, int*);

cudaError_t take_error_f32(cudaStream_t stream, int* code) { return take_error_local(stream, code); }

}  // namespace fused
}  // namespace vpd
