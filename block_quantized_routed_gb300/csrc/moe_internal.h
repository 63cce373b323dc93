// Host-side internals shared by the translation units of the MoE library.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "moe_q8k.h"

namespace moe {

// Largest (token, slot) pair count handled by the single-CTA top-k+bucket kernel.
constexpr int kSmallPairs = 256;
// Pairs per CTA of the multi-CTA bucketing kernels.
constexpr int kBucketChunk = 1024;

// A unit of expert work: `count` rows of bucket `expert` starting at bucket
// position `start`; flag 1 = the expert's gate pointer is NULL (not present).
struct Tile {
  int expert, start, count, flag;
};

// Full workspace plan of moe_layer_forward (public regions + internal ones).
struct WsPlan {
  moe_ws_layout pub;
  size_t tiles;       // Tile [max_tiles]
  size_t n_tiles;     // int32 (inside the status block: status[1])
  size_t req_cnt;     // int32 [max_tiles * I/256]  arrival counters
  size_t chunk_cnt;   // int32 [n_chunks * (E + S)]
  size_t bar;         // uint64 grid-barrier counter (inside the status block)
  size_t phase_ns;    // uint64 [16]  phase stamps of the single-launch decode kernel
  // second/third buffers of the pipelined decode schedule (0 when absent)
  size_t xq_b[3], xd_b[3], xbs_b[3], logits_b[2], h_b[2], y_b[2];
  size_t route_pub, route_flag;
  bool pipeline;
  // work items of the tensor-core prefill path (0 when the shape never takes it)
  size_t pitems, n_pitems, pxg, psg, pdg;
  int max_pitems;
  int max_tiles;
  int n_chunks;
  size_t total;
};

bool desc_valid(const moe_layer_desc* d, int* why);
WsPlan plan_workspace(const moe_layer_desc& d);

// token-group size of the expert kernels for T tokens of hidden size H
int pick_tile_tokens(int T, int H);

// ---- launchers (return cudaGetLastError of the launch) ---------------------
cudaError_t launch_q8k_quantize(const float* x, int64_t T, int64_t K, int8_t* q, float* d, int16_t* bs,
                                cudaStream_t s);
// status: the workspace status word for the bounded waits of the tensor-core
// router (nullable: a wait that runs out then only ends the kernel)
cudaError_t launch_router(const float* x, const float* w, const float* bias, int T, int H, int E,
                          float* logits, cudaStream_t s, int* status = nullptr);
// the router GEMM on tcgen05 kind::tf32 (three-term split), H a multiple of 32
cudaError_t launch_router_tc(const float* x, const float* w, const float* bias, int T, int H, int E,
                             float* logits, int* status, cudaStream_t s);
cudaError_t launch_topk(const float* logits, int T, int E, int k, int route, int32_t* ids, float* gates,
                        float* gap, cudaStream_t s);
// single CTA: top-k (optional: logits != nullptr), bucketing, tile plan; T*k <= kSmallPairs
cudaError_t launch_route_bucket_small(const float* logits, int T, int E, int k, int route, int S,
                                      int32_t* ids, float* gates, float* gap, int32_t* counts,
                                      int32_t* offsets, int32_t* perm, int32_t* inv,
                                      const moe_expert_ptrs* table, int TT, int nIB, Tile* tiles,
                                      int32_t* n_tiles, int32_t* req_cnt, int* status, cudaStream_t s);
// multi-CTA bucketing for any T*k
cudaError_t launch_bucket_large(const int32_t* ids, int T, int k, int E, int S, int32_t* counts,
                                int32_t* offsets, int32_t* perm, int32_t* inv, int32_t* chunk_cnt,
                                int* status, cudaStream_t s);
// tile plan from counts/offsets (single CTA)
cudaError_t launch_plan(const int32_t* counts, const int32_t* offsets, int EpS,
                        const moe_expert_ptrs* table, int TT, int nIB, Tile* tiles, int32_t* n_tiles,
                        int32_t* req_cnt, cudaStream_t s);

struct FfnArgs {
  int fmt, H, I, T, k, TT;
  const moe_expert_ptrs* table;
  const int8_t* xq;
  const float* xd;
  const int16_t* xbs;
  const int32_t* perm;
  const Tile* tiles;
  const int32_t* n_tiles;
  int max_tiles;
  float* h;
  int8_t* hq;
  float* hd;
  int16_t* hbs;
  int32_t* req_cnt;
  float* y;          // slot-indexed [T*(k+S), H]
  int* status;
};
cudaError_t launch_expert_ffn(const FfnArgs& a, cudaStream_t s);

// profiling hook state (per host thread): records the next event if tracing
void trace_record(cudaStream_t s);
// counts every kernel launch the library issues (moe_kernel_launch_count)
void note_launch();
// remembers a failed CUDA call of this host thread (moe_last_cuda_error); returns e
cudaError_t record_error(cudaError_t e);

// Workspace extension of a decode stack (moe_stack_forward): per-layer
// buffers and dependency counters, placed after a layer workspace.  Offsets
// are relative to the extension's base; a layer's block starts at
// layer0 + l * layer_bytes.
struct StackPlan {
  size_t cnt;          // uint64 [L][kStackCnt + P] counters, zeroed by each launch
  size_t layer0, layer_bytes;
  size_t logits, xq, xd, xbs, route, tptr, h, y;  // inside a layer block (tptr: tile weight pointers)
  int n_layers, n_cnt;                      // n_cnt = kStackCnt + P counters per layer
  size_t total;
};
constexpr int kStackCnt = 4;  // router items, routing, down items, combine items (then one per tile)
StackPlan stack_plan(const moe_layer_desc& d, int n_layers);
// gate/up + down items of one stack layer per SM (decides which stack kernel runs)
double stack_items_per_sm(const moe_layer_desc& d, int T, int sms);  // sms <= 0: the current device's
bool stack_takes_pipelined(const moe_layer_desc& d, int n_layers, int T, int sms);

// Single-launch decode layer (cooperative kernel); see moe_decode.cu.
struct DecodeArgs {
  int fmt, H, I, E, k, S, route, T;
  const moe_expert_ptrs* table;
  const float* w_router;
  const float* bias;
  const float* x;
  const float* residual;
  float* out;
  // workspace buffers; [0] is the one moe_workspace_layout names, the others
  // exist only for the pipelined schedule of a stack (pipeline_ok)
  int8_t* xq[3];
  float* xd[3];
  int16_t* xbs[3];
  float* logits[2];
  float* h[2];
  float* y[2];
  float* gap;
  int32_t* ids;
  float* gates;
  int32_t* counts;
  int32_t* offsets;
  int32_t* perm;
  int32_t* inv;
  int8_t* hq;
  float* hd;
  int16_t* hbs;
  unsigned long long* bar;
  unsigned long long* phase_ns;   // [16] SM-cycle stamps of CTA 0 (nullable)
  int* status;
  int32_t* ids_out;
  float* gates_out;
  int n_layers;                   // layers of this launch (stack); 1 for one layer
  const moe_layer_ptrs* layers;   // device array of n_layers records, or NULL: use the fields above
  int pipeline_ok;                // the workspace holds the extra buffers of the pipelined schedule
  uint8_t* route_pub;             // 4 routing states published by the routing CTA (pipelined schedule)
  unsigned long long* route_flag; // monotonic count of published routing states
  uint8_t* stk;                   // stack extension (decode_stack_kernel), or NULL
  StackPlan sp;
};
cudaError_t launch_decode_stack(const DecodeArgs& a, cudaStream_t s);

size_t decode_smem_bytes(int T, int H, int I, int E, int k, int S);
size_t decode_route_bytes(int T, int k, int S);  // one routing state of the decode kernel
// byte offsets of the fields of one routing state of T tokens (ids, gates
// [T*k]; tok, slot [P]: token and slot index of each bucket position; tiles
// [P]; ok [T*k + S]; n_tiles)
struct RouteFields {
  size_t ids, gates, tok, slot, tiles, ok, n_tiles;
};
RouteFields route_fields(int T, int k, int S);
cudaError_t launch_decode_fused(const DecodeArgs& a, cudaStream_t s);
// the same two launches per weight format (moe_decode_<fmt>.cu)
cudaError_t launch_decode_fused_q4k(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_decode_fused_q2k(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_decode_fused_q5k(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_decode_fused_q3k(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_decode_fused_q6k(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_decode_fused_iq2g(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_decode_stack_q4k(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_decode_stack_q2k(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_decode_stack_q5k(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_decode_stack_q3k(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_decode_stack_q6k(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_decode_stack_iq2g(const DecodeArgs& a, cudaStream_t s);
// largest token count of the single-launch decode path
constexpr int kDecodeMaxT = 16;

// ---- tensor-core prefill path (moe_prefill.cu) ------------------------------
// Experts must average at least this many routed tokens for the tcgen05
// grouped GEMM to beat the dp4a GEMV kernels.
constexpr int kPrefillMinTokensPerExpert = 16;
// Formats the tensor-core path takes: their scale * code products are exact
// fp16 integers (|sc * q| <= 2048) and their half super-block sums stay
// below 2^24 (Q4_K/Q2_K/Q3_K-style).  The Q5_K-style (63 * 31 * 127 * 128
// > 2^24 per half) and Q6_K-style (|127 * 63| > 2048) formats run their
// large batches on the dp4a GEMV kernels.
inline bool prefill_format(int fmt) {
  return fmt == MOE_FMT_Q4K || fmt == MOE_FMT_Q2K || fmt == MOE_FMT_Q3K || fmt == MOE_FMT_IQ2G;
}
inline bool prefill_path(int64_t T, int k, int E, int fmt) {
  return prefill_format(fmt) && T * k > kSmallPairs && T * k >= (int64_t)kPrefillMinTokensPerExpert * E;
}
// TMA coordinates are 32-bit: the code-sum plane has (max(H, I)/256) * 2 * P rows
inline bool prefill_fits(int64_t T, const moe_layer_desc& d) {
  const int64_t P = T * (d.top_k + d.n_shared);
  const int64_t K = d.H > d.I ? d.H : d.I;
  return (K / 256) * 2 * P + 256 < ((int64_t)1 << 31);
}
// one unit of prefill GEMM work: a token tile of one expert x a weight tile
struct PItem {
  int expert;  // expert index (routed, then shared)
  int start;   // first bucket position of the token tile
  int count;   // tokens in the tile (<= 128)
  int wtile;   // gate/up: 64-row group of I (its gate and up rows); down: 128-row group of H
};
int prefill_tile_tokens();
size_t prefill_item_capacity(int64_t P, int E, int S, int H, int I);
struct PrefillArgs {
  int fmt, H, I, E, S, T, k;
  int64_t P;                     // bucket positions = T * (k + S)
  const moe_expert_ptrs* table;
  const int8_t* xq;
  const float* xd;
  const int16_t* xbs;
  const int32_t* counts;
  const int32_t* offsets;
  const int32_t* perm;
  float* h;                      // [P, I] bucket order
  int8_t* hq;
  float* hd;
  int16_t* hbs;
  float* y;                      // slot-indexed [P, H]
  void* xg;                      // fp16 [P, max(H, I)] activation codes in bucket order
  void* sg;                      // fp16 [max(H, I)/256][2][P][8] code sums
  float* dg;                     // fp32 [max(H, I)/256][P] block scales
  PItem* items;
  int32_t* n_items;
  int max_items;
  int* status;
  unsigned long long* stats;     // [16] wait statistics of the GEMMs' CTA 0 (the phase_ns region)
};
cudaError_t launch_prefill_ffn(const PrefillArgs& a, cudaStream_t s);

// Test hook of the tensor-core path: the integer super-block sums S and M of
// a matrix w [N, K] (N a multiple of 128) against q8_K rows, from the same
// GEMM kernel with an epilogue that writes them instead of rescaling.
struct SumsArgs {
  int fmt, N, K, T;
  const void* w;
  const int8_t* q;
  const float* d;
  const int16_t* bs16;
  int32_t* S;  // [T][N][K/256]
  int32_t* M;
  void* ws;
};
struct SumsPlan {
  size_t status, xg, sg, dg, items, n_items, total;
};
SumsPlan sums_plan(int N, int K, int T);
cudaError_t launch_prefill_sums(const SumsArgs& a, cudaStream_t s);

cudaError_t launch_combine(const float* y, const float* gates, int T, int H, int k, int S,
                           const float* residual, float* out, cudaStream_t s);

cudaError_t launch_debug_dots(int fmt, const void* w, int N, int K, const int8_t* q, int T, int32_t* isum,
                              int32_t* bsum, cudaStream_t s);

cudaError_t launch_debug_wait(int* status, const unsigned* flag, long long limit_ns, cudaStream_t s);

int num_sms();

}  // namespace moe
