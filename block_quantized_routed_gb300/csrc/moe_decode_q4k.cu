// The single-launch decode kernels instantiated for the Q4_K-style format.
#include "moe_decode_kernels.cuh"

namespace moe {

cudaError_t launch_decode_fused_q4k(const DecodeArgs& a, cudaStream_t s) { return launch_decode_t<kQ4K>(a, s); }
cudaError_t launch_decode_stack_q4k(const DecodeArgs& a, cudaStream_t s) { return launch_stack_t<kQ4K>(a, s); }

}  // namespace moe
