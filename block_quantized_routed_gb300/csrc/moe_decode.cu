// Exported host side of the single-launch decode kernels (the kernels and
// their launch templates are in moe_decode_kernels.cuh; each format's
// instantiations live in their own translation unit, moe_decode_<fmt>.cu, so
// that the build compiles them in parallel).
#include "moe_decode_kernels.cuh"

namespace moe {

size_t decode_route_bytes(int T, int k, int S) { return route_bytes(T, k, S); }

RouteFields route_fields(int T, int k, int S) { return route_fields_of(T, k, S); }

size_t decode_smem_bytes(int T, int H, int I, int E, int k, int S) {
  return decode_smem(T, H, I, E, k, S, kDecWarps, nullptr, nullptr);
}

cudaError_t launch_decode_fused(const DecodeArgs& a, cudaStream_t s) {
  switch (a.fmt) {
    case kQ4K: return launch_decode_fused_q4k(a, s);
    case kQ2K: return launch_decode_fused_q2k(a, s);
    case kQ5K: return launch_decode_fused_q5k(a, s);
    case kQ3K: return launch_decode_fused_q3k(a, s);
    case kQ6K: return launch_decode_fused_q6k(a, s);
    case kIQ2G: return launch_decode_fused_iq2g(a, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_stack(const DecodeArgs& a, cudaStream_t s) {
  switch (a.fmt) {
    case kQ4K: return launch_decode_stack_q4k(a, s);
    case kQ2K: return launch_decode_stack_q2k(a, s);
    case kQ5K: return launch_decode_stack_q5k(a, s);
    case kQ3K: return launch_decode_stack_q3k(a, s);
    case kQ6K: return launch_decode_stack_q6k(a, s);
    case kIQ2G: return launch_decode_stack_iq2g(a, s);
    default: return cudaErrorInvalidValue;
  }
}

StackPlan stack_plan(const moe_layer_desc& d, int n_layers) {
  StackPlan p{};
  const size_t T = (size_t)d.T_max, H = (size_t)d.H, I = (size_t)d.I, E = (size_t)d.E;
  const size_t P = T * (size_t)(d.top_k + d.n_shared);
  auto a256 = [](size_t v) { return (v + 255) / 256 * 256; };
  p.n_layers = n_layers;
  p.n_cnt = kStackCnt + (int)P;
  p.cnt = 0;
  p.layer0 = a256(p.cnt + (size_t)n_layers * p.n_cnt * 8);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = a256(off + bytes);
    return at;
  };
  p.logits = take(T * E * 4);
  p.xq = take(T * H);
  p.xd = take(T * (H / 256) * 4);
  p.xbs = take(T * (H / 16) * 2);
  p.route = take(route_bytes((int)T, d.top_k, d.n_shared));
  p.tptr = take(P * sizeof(moe_expert_ptrs));
  p.h = take(P * I * 4);
  p.y = take(P * H * 4);
  p.layer_bytes = off;
  p.total = p.layer0 + (size_t)n_layers * p.layer_bytes;
  return p;
}

}  // namespace moe
