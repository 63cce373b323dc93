// The single-launch decode kernels instantiated for the Q5_K-style format.
#include "moe_decode_kernels.cuh"

namespace moe {

cudaError_t launch_decode_fused_q5k(const DecodeArgs& a, cudaStream_t s) { return launch_decode_t<kQ5K>(a, s); }
cudaError_t launch_decode_stack_q5k(const DecodeArgs& a, cudaStream_t s) { return launch_stack_t<kQ5K>(a, s); }

}  // namespace moe
