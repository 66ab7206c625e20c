// vpd_fused_bf16.cu -- the fused single-read JSD kernels for bf16 logits
// (device code in vpd_fused.cuh), and this unit's device error word.
#include "vpd_fused.cuh"

namespace vpd {
namespace fused {

template cudaError_t launch_typed<InBF16>(const FusedArgs&, const Config&, int, bool, bool, cudaStream_t, int*);
template int resident_clusters<InBF16>(int, int, size_t);

cudaError_t take_error_bf16(cudaStream_t stream, int* code) { return take_error_local(stream, code); }

}  // namespace fused
}  // namespace vpd
