// moe_layer_forward_noalloc: run one MoE layer without a caller-provided
// workspace and without allocating anything.
//
// Who needs this: callers that cannot call cudaMalloc where they run the
// layer.  Examples are an engine whose memory planner hands every byte of the
// device to its own pool up front (so a later cudaMalloc fails or breaks its
// accounting), a plugin loaded into such a host that receives only the
// tensors it must read and write, and a token loop that must not allocate
// because an allocation can synchronise the device in the middle of a step.
// They already own the inputs and outputs; this entry point supplies the
// intermediate storage from a fixed array that is part of the library.
//
// The scratch is a file-scope __device__ array of kNoAllocScratchBytes.  The
// CUDA runtime creates it on every device that loads this library and keeps
// it until the process exits.  Host code cannot use the array's name as a
// device address, so every call looks the address up with
// cudaGetSymbolAddress in the context current on the calling thread: a
// host-side lookup that allocates nothing, and that stays right for callers
// that run the layer in a context of their own or reset the device between
// calls (a cached address would belong to the context it was taken in).
#include <cstdint>

#include "moe_internal.h"

namespace moe {
namespace {

// Largest workspace (moe_layer_workspace_size) this entry point can serve.
constexpr size_t kNoAllocScratchBytes = MOE_NOALLOC_MAX_WORKSPACE;  // 16 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array in the calling thread's current context.
cudaError_t scratch_address(void** out) {
  void* p = nullptr;
  const cudaError_t err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (err != cudaSuccess) return err;
  *out = p;
  return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace
}  // namespace moe

extern "C" int moe_layer_forward_noalloc(const moe_layer_desc* desc, const moe_expert_ptrs* table,
                                         const float* w_router, const float* router_bias, const float* x,
                                         const float* residual, float* out, int32_t T, int32_t* ids_out,
                                         float* gates_out, void* stream) {
  using namespace moe;
  int why;
  if (!desc_valid(desc, &why)) return why;
  if (T < 0 || T > desc->T_max) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!table || !w_router || !x || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(out) || !aligned16(w_router) || (residual && !aligned16(residual)))
    return MOE_ERR_INVALID_ARG;
  if (moe_layer_workspace_size(desc) > kNoAllocScratchBytes) return MOE_ERR_WORKSPACE;
  void* ws = nullptr;
  if (scratch_address(&ws) != cudaSuccess) return MOE_ERR_CUDA;
  // The array keeps the previous call's contents: the status word, tile count
  // and grid-barrier counter must start at zero.
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, 16, s) != cudaSuccess) return MOE_ERR_CUDA;
  return moe_layer_forward(desc, table, w_router, router_bias, x, residual, out, T, ids_out, gates_out, ws,
                           kNoAllocScratchBytes, stream);
}
