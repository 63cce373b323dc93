// The single-launch decode kernels instantiated for the IQ2-style grid format.
#include "moe_decode_kernels.cuh"

namespace moe {

cudaError_t launch_decode_fused_iq2g(const DecodeArgs& a, cudaStream_t s) { return launch_decode_t<kIQ2G>(a, s); }
cudaError_t launch_decode_stack_iq2g(const DecodeArgs& a, cudaStream_t s) { return launch_stack_t<kIQ2G>(a, s); }

}  // namespace moe
