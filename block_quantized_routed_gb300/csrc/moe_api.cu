// C ABI of the block-quantized MoE layer: argument validation, workspace
// plans and the launch sequences.  Every entry point validates on the host
// before it touches the GPU, so a rejected call launches nothing.
#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr size_t kAlign = 256;
constexpr size_t kDecodeSmemMax = 200 * 1024;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Carve {
  size_t off = 0;
  size_t take(size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes);
    return at;
  }
};

cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

int check(cudaError_t e) { return record_error(e) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

}  // namespace

bool desc_valid(const moe_layer_desc* d, int* why) {
  *why = MOE_ERR_INVALID_ARG;
  if (!d) return false;
  *why = MOE_ERR_UNSUPPORTED;
  if (d->H <= 0 || d->I <= 0 || d->H % 256 || d->I % 256 || d->H > MOE_MAX_DIM || d->I > MOE_MAX_DIM) return false;
  if (d->E < 1 || d->E > MOE_MAX_EXPERTS) return false;
  if (d->top_k < 1 || d->top_k > MOE_MAX_TOPK || d->top_k > d->E) return false;
  if (d->n_shared < 0 || d->n_shared > MOE_MAX_SHARED) return false;
  if (d->route != MOE_ROUTE_SOFTMAX && d->route != MOE_ROUTE_SIGMOID) return false;
  if (d->fmt < MOE_FMT_Q4K || d->fmt > MOE_FMT_IQ2G) return false;
  if (d->T_max < 1 || (int64_t)d->T_max * (d->top_k + d->n_shared) > (int64_t)1 << 28) return false;
  return true;
}

WsPlan plan_workspace(const moe_layer_desc& d) {
  WsPlan p{};
  const size_t T = (size_t)d.T_max, H = (size_t)d.H, I = (size_t)d.I, E = (size_t)d.E;
  const size_t k = (size_t)d.top_k, S = (size_t)d.n_shared, EpS = E + S;
  const size_t P = T * (k + S);
  p.max_tiles = (int)P;
  p.n_chunks = (int)((T * k + kBucketChunk - 1) / kBucketChunk);
  Carve c;
  p.pub.status = c.take(16);
  p.n_tiles = p.pub.status + 4;
  p.bar = p.pub.status + 8;
  p.pub.xq = c.take(T * H);
  p.pub.xd = c.take(T * (H / 256) * 4);
  p.pub.xbs = c.take(T * (H / 16) * 2);
  p.pub.logits = c.take(T * E * 4);
  p.pub.ids = c.take(T * k * 4);
  p.pub.gates = c.take(T * k * 4);
  p.pub.gap = c.take(T * 4);
  p.pub.counts = c.take(EpS * 4);
  p.pub.offsets = c.take((EpS + 1) * 4);
  p.pub.perm = c.take(P * 4);
  p.pub.inv = c.take(P * 4);
  p.pub.h = c.take(P * I * 4);
  p.pub.hq = c.take(P * I);
  p.pub.hd = c.take(P * (I / 256) * 4);
  p.pub.hbs = c.take(P * (I / 16) * 2);
  p.pub.y = c.take(P * H * 4);
  p.tiles = c.take((size_t)p.max_tiles * sizeof(Tile));
  p.req_cnt = c.take((size_t)p.max_tiles * (I / 256) * 4);
  p.chunk_cnt = c.take((size_t)(p.n_chunks > 0 ? p.n_chunks : 1) * EpS * 4);
  p.phase_ns = c.take(16 * 8);
  p.pub.phase_ns = p.phase_ns;
  // the pipelined decode schedule of a stack keeps several layers in flight:
  // 3 copies of q8_K(x), 2 of logits, h and y (only for decode shapes)
  p.xq_b[0] = p.pub.xq; p.xd_b[0] = p.pub.xd; p.xbs_b[0] = p.pub.xbs;
  p.logits_b[0] = p.pub.logits; p.h_b[0] = p.pub.h; p.y_b[0] = p.pub.y;
  p.pipeline = d.T_max <= kDecodeMaxT;
  if (p.pipeline) {
    for (int i = 1; i < 3; ++i) {
      p.xq_b[i] = c.take(T * H);
      p.xd_b[i] = c.take(T * (H / 256) * 4);
      p.xbs_b[i] = c.take(T * (H / 16) * 2);
    }
    p.logits_b[1] = c.take(T * E * 4);
    p.h_b[1] = c.take(P * I * 4);
    p.y_b[1] = c.take(P * H * 4);
    p.route_pub = c.take(4 * decode_route_bytes((int)T, (int)k, (int)S));
    p.route_flag = c.take(8);
  }
  if (prefill_path(d.T_max, d.top_k, d.E, d.fmt) && prefill_fits(d.T_max, d)) {
    p.max_pitems = (int)prefill_item_capacity((int64_t)P, d.E, d.n_shared, d.H, d.I);
    p.pitems = c.take((size_t)p.max_pitems * sizeof(PItem));
    p.n_pitems = c.take(16);
    const size_t Kmax = std::max(H, I);
    p.pxg = c.take(P * Kmax * 2);
    p.psg = c.take((Kmax / 256) * 2 * P * 16);
    p.pdg = c.take((Kmax / 256) * P * 4);
  }
  p.total = c.off;
  p.pub.total = p.total;
  return p;
}

namespace {
thread_local void* const* g_trace_events = nullptr;
thread_local int g_trace_n = 0;
thread_local int g_trace_next = 0;
}  // namespace

namespace {
std::atomic<unsigned long long> g_launches{0};
thread_local int g_last_error = 0;
}  // namespace

cudaError_t record_error(cudaError_t e) {
  if (e != cudaSuccess) g_last_error = (int)e;
  return e;
}
int last_error() { return g_last_error; }

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

// Gate/up and down items of one layer of the dataflow stack per SM (the same
// item sizes as decode_stack_kernel chooses).
constexpr int kFlowMinLayers = 4;  // heavy layers take the dataflow kernel from this many layers on

double stack_items_per_sm(const moe_layer_desc& d, int T, int sms) {
  const int nbH = d.H / 256, nbI = d.I / 256, nRG = d.I / 32, nRGH = d.H / 32;
  const int Tm = T > 16 ? T : 16;
  const int gpi = std::max(1, std::min(16 / nbH, Tm / T));
  const int dpi = nbI <= 2 ? 2 : 1;
  const double P = (double)T * (d.top_k + d.n_shared);
  const double items = P * ((nRG + gpi - 1) / gpi) + P * ((nRGH + 8 * dpi - 1) / (8 * dpi));
  return items / (sms > 0 ? sms : num_sms());
}

// Short stacks of layers with many expert items per CTA (a wide layer on
// its own) run faster on the barrier-pipelined kernel, whose CTAs prefetch
// all of their items of a layer at once; small layers, and heavy layers
// with enough neighbours to overlap (measured: a 48-layer verify stack),
// run as the dataflow of items.
bool stack_takes_pipelined(const moe_layer_desc& d, int n_layers, int T, int sms) {
  return stack_items_per_sm(d, T, sms) > 2.0 && n_layers < kFlowMinLayers;
}

void trace_record(cudaStream_t s) {
  if (!g_trace_events || g_trace_next >= g_trace_n) return;
  cudaEvent_t ev = static_cast<cudaEvent_t>(g_trace_events[g_trace_next]);
  // under stream capture the record must become an event-record node of the
  // graph (the External flag); outside capture that flag is not valid and a
  // plain record is the same operation
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t err = ev ? cudaStreamIsCapturing(s, &cs) : cudaErrorInvalidResourceHandle;
  if (err == cudaSuccess)
    err = cs == cudaStreamCaptureStatusActive ? cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal)
                                              : cudaEventRecord(ev, s);
  if (err != cudaSuccess) {
    // a profiling record must not turn into the next launch's error: consume
    // the error and stop tracing (moe_trace_used counts only what was recorded)
    cudaGetLastError();
    g_trace_events = nullptr;
    return;
  }
  ++g_trace_next;
}

}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_layer_workspace_size(const moe_layer_desc* desc) {
  int why;
  if (!desc_valid(desc, &why)) return 0;
  return plan_workspace(*desc).total;
}

int moe_workspace_layout(const moe_layer_desc* desc, moe_ws_layout* out) {
  int why;
  if (!out) return MOE_ERR_INVALID_ARG;
  if (!desc_valid(desc, &why)) return why;
  *out = plan_workspace(*desc).pub;
  return MOE_OK;
}

int moe_q8k_quantize(const float* x, int64_t T, int64_t K, int8_t* q, float* d, int16_t* bsum16, void* stream) {
  if (T < 0 || K <= 0 || K % 256) return T < 0 || K <= 0 ? MOE_ERR_INVALID_ARG : MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!x || !q || !d) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(q, 16) || !aligned(d, 4) || (bsum16 && !aligned(bsum16, 4)))
    return MOE_ERR_INVALID_ARG;
  return check(launch_q8k_quantize(x, T, K, q, d, bsum16, as_stream(stream)));
}

int moe_route_topk(const float* x, const float* w_router, const float* bias, int32_t T, int32_t H, int32_t E,
                   int32_t k, int32_t route, float* logits, int32_t* ids, float* gates, float* gap, void* stream) {
  if (T < 0 || H <= 0 || E < 1 || k < 1) return MOE_ERR_INVALID_ARG;
  if (H % 4 || E > MOE_MAX_EXPERTS || k > MOE_MAX_TOPK || k > E) return MOE_ERR_UNSUPPORTED;
  if (route != MOE_ROUTE_SOFTMAX && route != MOE_ROUTE_SIGMOID) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!x || !w_router || !logits || !ids || !gates) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(w_router, 16)) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = as_stream(stream);
  cudaError_t e = launch_router(x, w_router, bias, T, H, E, logits, s);
  if (record_error(e) != cudaSuccess) return MOE_ERR_CUDA;
  return check(launch_topk(logits, T, E, k, route, ids, gates, gap, s));
}

size_t moe_bucket_workspace_size(int32_t T, int32_t k, int32_t E, int32_t n_shared) {
  if (T < 0 || k < 1 || E < 1 || n_shared < 0) return 0;
  const size_t n_chunks = ((size_t)T * k + kBucketChunk - 1) / kBucketChunk;
  return 256 + align_up((n_chunks > 0 ? n_chunks : 1) * (size_t)(E + n_shared) * 4);
}

int moe_bucket(const int32_t* ids, int32_t T, int32_t k, int32_t E, int32_t n_shared, int32_t* counts,
               int32_t* offsets, int32_t* perm, int32_t* inv, void* ws, size_t ws_bytes, void* stream) {
  if (T < 0 || k < 1 || E < 1 || n_shared < 0) return MOE_ERR_INVALID_ARG;
  if (E > MOE_MAX_EXPERTS || n_shared > MOE_MAX_SHARED || k > MOE_MAX_TOPK) return MOE_ERR_UNSUPPORTED;
  if (!counts || !offsets || !ws || (T > 0 && (!ids || !perm))) return MOE_ERR_INVALID_ARG;
  if (!aligned(ws, kAlign)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < moe_bucket_workspace_size(T, k, E, n_shared)) return MOE_ERR_WORKSPACE;
  cudaStream_t s = as_stream(stream);
  int* status = static_cast<int*>(ws);
  int32_t* chunk_cnt = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + 256);
  if ((int64_t)T * k <= kSmallPairs)
    return check(launch_route_bucket_small(nullptr, T, E, k, 0, n_shared, const_cast<int32_t*>(ids), nullptr,
                                           nullptr, counts, offsets, perm, inv, nullptr, 1, 0, nullptr, nullptr,
                                           nullptr, status, s));
  return check(launch_bucket_large(ids, T, k, E, n_shared, counts, offsets, perm, inv, chunk_cnt, status, s));
}

size_t moe_expert_ffn_workspace_size(const moe_layer_desc* desc, int32_t T) {
  int why;
  if (!desc_valid(desc, &why) || T < 0 || T > desc->T_max) return 0;
  const size_t P = (size_t)T * (desc->top_k + desc->n_shared), I = (size_t)desc->I;
  Carve c;
  c.take(16);
  c.take(P * sizeof(Tile));
  c.take(P * (I / 256) * 4);
  c.take(P * I * 4);
  c.take(P * I);
  c.take(P * (I / 256) * 4);
  c.take(P * (I / 16) * 2);
  return c.off;
}

int moe_expert_ffn(const moe_layer_desc* desc, const moe_expert_ptrs* table, const int8_t* q, const float* d,
                   const int16_t* bsum16, const int32_t* counts, const int32_t* offsets, const int32_t* perm,
                   int32_t T, float* y_slots, void* ws, size_t ws_bytes, void* stream) {
  int why;
  if (!desc_valid(desc, &why)) return why;
  if (T < 0 || T > desc->T_max) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!table || !q || !d || !bsum16 || !counts || !offsets || !perm || !y_slots || !ws) return MOE_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(bsum16, 16) || !aligned(y_slots, 16) || !aligned(ws, kAlign))
    return MOE_ERR_INVALID_ARG;
  if (ws_bytes < moe_expert_ffn_workspace_size(desc, T)) return MOE_ERR_WORKSPACE;
  const size_t P = (size_t)T * (desc->top_k + desc->n_shared), I = (size_t)desc->I;
  char* base = static_cast<char*>(ws);
  Carve c;
  int* status = reinterpret_cast<int*>(base + c.take(16));
  Tile* tiles = reinterpret_cast<Tile*>(base + c.take(P * sizeof(Tile)));
  int32_t* req_cnt = reinterpret_cast<int32_t*>(base + c.take(P * (I / 256) * 4));
  FfnArgs a{};
  a.h = reinterpret_cast<float*>(base + c.take(P * I * 4));
  a.hq = reinterpret_cast<int8_t*>(base + c.take(P * I));
  a.hd = reinterpret_cast<float*>(base + c.take(P * (I / 256) * 4));
  a.hbs = reinterpret_cast<int16_t*>(base + c.take(P * (I / 16) * 2));
  cudaStream_t s = as_stream(stream);
  const int TT = pick_tile_tokens(T, desc->H);
  const int EpS = desc->E + desc->n_shared;
  int32_t* n_tiles = status + 1;
  if (record_error(launch_plan(counts, offsets, EpS, table, TT, desc->I / 256, tiles, n_tiles, req_cnt, s)) != cudaSuccess)
    return MOE_ERR_CUDA;
  a.fmt = desc->fmt;
  a.H = desc->H;
  a.I = desc->I;
  a.T = T;
  a.k = desc->top_k;
  a.TT = TT;
  a.table = table;
  a.xq = q;
  a.xd = d;
  a.xbs = bsum16;
  a.perm = perm;
  a.tiles = tiles;
  a.n_tiles = n_tiles;
  a.max_tiles = (int)P;
  a.req_cnt = req_cnt;
  a.y = y_slots;
  a.status = status;
  return check(launch_expert_ffn(a, s));
}

int moe_combine(const float* y_slots, const float* gates, int32_t T, int32_t H, int32_t k, int32_t n_shared,
                const float* residual, float* out, void* stream) {
  if (T < 0 || H <= 0 || k < 1 || n_shared < 0) return MOE_ERR_INVALID_ARG;
  if (H % 4) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!y_slots || !gates || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned(y_slots, 16) || !aligned(out, 16) || (residual && !aligned(residual, 16))) return MOE_ERR_INVALID_ARG;
  return check(launch_combine(y_slots, gates, T, H, k, n_shared, residual, out, as_stream(stream)));
}

int moe_layer_forward(const moe_layer_desc* desc, const moe_expert_ptrs* table, const float* w_router,
                      const float* router_bias, const float* x, const float* residual, float* out, int32_t T,
                      int32_t* ids_out, float* gates_out, void* ws, size_t ws_bytes, void* stream) {
  int why;
  if (!desc_valid(desc, &why)) return why;
  if (T < 0 || T > desc->T_max) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!table || !w_router || !x || !out || !ws) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(out, 16) || !aligned(w_router, 16) || !aligned(ws, kAlign) ||
      (residual && !aligned(residual, 16)))
    return MOE_ERR_INVALID_ARG;
  const WsPlan p = plan_workspace(*desc);
  if (ws_bytes < p.total) return MOE_ERR_WORKSPACE;
  char* base = static_cast<char*>(ws);
  auto at = [&](size_t off) { return static_cast<void*>(base + off); };
  int* status = static_cast<int*>(at(p.pub.status));
  int32_t* n_tiles = reinterpret_cast<int32_t*>(at(p.n_tiles));
  int8_t* xq = static_cast<int8_t*>(at(p.pub.xq));
  float* xd = static_cast<float*>(at(p.pub.xd));
  int16_t* xbs = static_cast<int16_t*>(at(p.pub.xbs));
  float* logits = static_cast<float*>(at(p.pub.logits));
  int32_t* ids = static_cast<int32_t*>(at(p.pub.ids));
  float* gates = static_cast<float*>(at(p.pub.gates));
  float* gap = static_cast<float*>(at(p.pub.gap));
  int32_t* counts = static_cast<int32_t*>(at(p.pub.counts));
  int32_t* offsets = static_cast<int32_t*>(at(p.pub.offsets));
  int32_t* perm = static_cast<int32_t*>(at(p.pub.perm));
  int32_t* inv = static_cast<int32_t*>(at(p.pub.inv));
  Tile* tiles = static_cast<Tile*>(at(p.tiles));
  int32_t* req_cnt = static_cast<int32_t*>(at(p.req_cnt));
  int32_t* chunk_cnt = static_cast<int32_t*>(at(p.chunk_cnt));
  const int H = desc->H, E = desc->E, k = desc->top_k, S = desc->n_shared;
  const int TT = pick_tile_tokens(T, H);
  const int nIB = desc->I / 256;
  cudaStream_t s = as_stream(stream);

  if (T <= kDecodeMaxT && (int64_t)T * k <= kSmallPairs) {
    if (decode_smem_bytes(T, H, desc->I, E, k, S) <= kDecodeSmemMax) {
      DecodeArgs d{};
      d.fmt = desc->fmt;
      d.H = H;
      d.I = desc->I;
      d.E = E;
      d.k = k;
      d.S = S;
      d.route = desc->route;
      d.T = T;
      d.table = table;
      d.w_router = w_router;
      d.bias = router_bias;
      d.x = x;
      d.residual = residual;
      d.out = out;
      d.xq[0] = xq;
      d.xd[0] = xd;
      d.xbs[0] = xbs;
      d.logits[0] = logits;
      d.gap = gap;
      d.ids = ids;
      d.gates = gates;
      d.counts = counts;
      d.offsets = offsets;
      d.perm = perm;
      d.inv = inv;
      d.h[0] = static_cast<float*>(at(p.pub.h));
      d.hq = static_cast<int8_t*>(at(p.pub.hq));
      d.hd = static_cast<float*>(at(p.pub.hd));
      d.hbs = static_cast<int16_t*>(at(p.pub.hbs));
      d.y[0] = static_cast<float*>(at(p.pub.y));
      d.bar = static_cast<unsigned long long*>(at(p.bar));
      d.phase_ns = static_cast<unsigned long long*>(at(p.phase_ns));
      d.status = status;
      d.ids_out = ids_out;
      d.gates_out = gates_out;
      d.n_layers = 1;
      d.layers = nullptr;
      trace_record(s);
      const cudaError_t err = record_error(launch_decode_fused(d, s));
      trace_record(s);
      if (err == cudaSuccess) return MOE_OK;
      if (err != cudaErrorCooperativeLaunchTooLarge) return MOE_ERR_CUDA;
      cudaGetLastError();  // not co-resident on this device: use the multi-kernel path
    }
  }
  if (record_error(launch_q8k_quantize(x, T, H, xq, xd, xbs, s)) != cudaSuccess) return MOE_ERR_CUDA;
  if (record_error(launch_router(x, w_router, router_bias, T, H, E, logits, s, status)) != cudaSuccess)
    return MOE_ERR_CUDA;
  const bool use_prefill = prefill_path(T, k, E, desc->fmt) && prefill_fits(desc->T_max, *desc);  // buffers sized by T_max
  if (use_prefill) {
    // prefill chunk: top-k, bucketing, then the tcgen05 grouped GEMMs
    if (record_error(launch_topk(logits, T, E, k, desc->route, ids, gates, gap, s)) != cudaSuccess) return MOE_ERR_CUDA;
    if (record_error(launch_bucket_large(ids, T, k, E, S, counts, offsets, perm, inv, chunk_cnt, status, s)) != cudaSuccess)
      return MOE_ERR_CUDA;
    PrefillArgs a{};
    a.fmt = desc->fmt;
    a.H = H;
    a.I = desc->I;
    a.E = E;
    a.S = S;
    a.T = T;
    a.k = k;
    a.P = (int64_t)T * (k + S);
    a.table = table;
    a.xq = xq;
    a.xd = xd;
    a.xbs = xbs;
    a.counts = counts;
    a.offsets = offsets;
    a.perm = perm;
    a.h = static_cast<float*>(at(p.pub.h));
    a.hq = static_cast<int8_t*>(at(p.pub.hq));
    a.hd = static_cast<float*>(at(p.pub.hd));
    a.hbs = static_cast<int16_t*>(at(p.pub.hbs));
    a.y = static_cast<float*>(at(p.pub.y));
    a.xg = at(p.pxg);
    a.sg = at(p.psg);
    a.dg = static_cast<float*>(at(p.pdg));
    a.items = static_cast<PItem*>(at(p.pitems));
    a.n_items = static_cast<int32_t*>(at(p.n_pitems));
    a.max_items = p.max_pitems;
    a.status = status;
    a.stats = static_cast<unsigned long long*>(at(p.phase_ns));
    if (record_error(launch_prefill_ffn(a, s)) != cudaSuccess) return MOE_ERR_CUDA;
  } else if ((int64_t)T * k <= kSmallPairs) {
    if (record_error(launch_route_bucket_small(logits, T, E, k, desc->route, S, ids, gates, gap, counts, offsets, perm, inv, table,
                                  TT, nIB, tiles, n_tiles, req_cnt, status, s)) != cudaSuccess)
      return MOE_ERR_CUDA;
  } else {
    if (record_error(launch_topk(logits, T, E, k, desc->route, ids, gates, gap, s)) != cudaSuccess) return MOE_ERR_CUDA;
    if (record_error(launch_bucket_large(ids, T, k, E, S, counts, offsets, perm, inv, chunk_cnt, status, s)) != cudaSuccess)
      return MOE_ERR_CUDA;
    if (record_error(launch_plan(counts, offsets, E + S, table, TT, nIB, tiles, n_tiles, req_cnt, s)) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  if (!use_prefill) {
    FfnArgs a{};
    a.fmt = desc->fmt;
    a.H = H;
    a.I = desc->I;
    a.T = T;
    a.k = k;
    a.TT = TT;
    a.table = table;
    a.xq = xq;
    a.xd = xd;
    a.xbs = xbs;
    a.perm = perm;
    a.tiles = tiles;
    a.n_tiles = n_tiles;
    a.max_tiles = p.max_tiles;
    a.h = static_cast<float*>(at(p.pub.h));
    a.hq = static_cast<int8_t*>(at(p.pub.hq));
    a.hd = static_cast<float*>(at(p.pub.hd));
    a.hbs = static_cast<int16_t*>(at(p.pub.hbs));
    a.req_cnt = req_cnt;
    a.y = static_cast<float*>(at(p.pub.y));
    a.status = status;
    if (record_error(launch_expert_ffn(a, s)) != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (record_error(launch_combine(static_cast<float*>(at(p.pub.y)), gates, T, H, k, S, residual, out, s)) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (ids_out && cudaMemcpyAsync(ids_out, ids, sizeof(int32_t) * T * k, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (gates_out &&
      cudaMemcpyAsync(gates_out, gates, sizeof(float) * T * k, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

size_t moe_stack_workspace_size(const moe_layer_desc* desc, int32_t n_layers) {
  int why;
  if (!desc_valid(desc, &why) || n_layers < 1) return 0;
  return (plan_workspace(*desc).total + 255) / 256 * 256 + stack_plan(*desc, n_layers).total;
}

int moe_stack_layer_layout(const moe_layer_desc* desc, int32_t n_layers, int32_t T, int32_t layer,
                           moe_stack_ws_layout* out) {
  int why;
  if (!desc_valid(desc, &why)) return why;
  if (!out || n_layers < 1 || T < 1 || T > desc->T_max || layer < 0 || layer >= n_layers) return MOE_ERR_INVALID_ARG;
  const int k = desc->top_k, S = desc->n_shared;
  if (T > kDecodeMaxT || (int64_t)T * k > kSmallPairs ||
      decode_smem_bytes(T, desc->H, desc->I, desc->E, k, S) > kDecodeSmemMax)
    return MOE_ERR_UNSUPPORTED;
  // the same placement as moe_stack_forward: the layer workspace of desc,
  // then the stack extension planned for the call's T
  moe_layer_desc dT = *desc;
  dT.T_max = T;
  const size_t ext = (plan_workspace(*desc).total + 255) / 256 * 256;
  const StackPlan sp = stack_plan(dT, n_layers);
  const size_t lb = ext + sp.layer0 + (size_t)layer * sp.layer_bytes;
  const RouteFields rf = route_fields(T, k, S);
  out->logits = lb + sp.logits;
  out->xq = lb + sp.xq;
  out->xd = lb + sp.xd;
  out->xbs = lb + sp.xbs;
  out->ids = lb + sp.route + rf.ids;
  out->gates = lb + sp.route + rf.gates;
  out->tok = lb + sp.route + rf.tok;
  out->slot = lb + sp.route + rf.slot;
  out->h = lb + sp.h;
  out->y = lb + sp.y;
  return MOE_OK;
}

int moe_stack_forward(const moe_layer_desc* desc, int32_t n_layers, const moe_layer_ptrs* layers, int32_t T,
                      void* ws, size_t ws_bytes, void* stream) {
  int why;
  if (!desc_valid(desc, &why)) return why;
  if (n_layers < 0 || T < 0 || T > desc->T_max) return MOE_ERR_INVALID_ARG;
  if (n_layers == 0 || T == 0) return MOE_OK;
  if (!layers || !ws || !aligned(ws, kAlign) || !aligned(layers, 8)) return MOE_ERR_INVALID_ARG;
  const int H = desc->H, E = desc->E, k = desc->top_k, S = desc->n_shared;
  if (T > kDecodeMaxT || (int64_t)T * k > kSmallPairs || decode_smem_bytes(T, H, desc->I, E, k, S) > kDecodeSmemMax)
    return MOE_ERR_UNSUPPORTED;
  // the per-layer buffers are sized by the call's T (T_max only bounds it)
  moe_layer_desc dT = *desc;
  dT.T_max = T;
  const WsPlan p = plan_workspace(*desc);
  const size_t ext = (p.total + 255) / 256 * 256;
  const StackPlan sp = stack_plan(dT, n_layers);
  if (ws_bytes < ext + sp.total) return MOE_ERR_WORKSPACE;
  char* base = static_cast<char*>(ws);
  auto at = [&](size_t off) { return static_cast<void*>(base + off); };
  if (stack_takes_pipelined(*desc, n_layers, T, 0)) {
    DecodeArgs d{};
    d.fmt = desc->fmt;
    d.H = H;
    d.I = desc->I;
    d.E = E;
    d.k = k;
    d.S = S;
    d.route = desc->route;
    d.T = T;
    for (int i = 0; i < 3; ++i) {
      d.xq[i] = static_cast<int8_t*>(at(p.xq_b[i]));
      d.xd[i] = static_cast<float*>(at(p.xd_b[i]));
      d.xbs[i] = static_cast<int16_t*>(at(p.xbs_b[i]));
    }
    for (int i = 0; i < 2; ++i) {
      d.logits[i] = static_cast<float*>(at(p.logits_b[i]));
      d.h[i] = static_cast<float*>(at(p.h_b[i]));
      d.y[i] = static_cast<float*>(at(p.y_b[i]));
    }
    d.pipeline_ok = p.pipeline ? 1 : 0;
    d.route_pub = p.pipeline ? static_cast<uint8_t*>(at(p.route_pub)) : nullptr;
    d.route_flag = p.pipeline ? static_cast<unsigned long long*>(at(p.route_flag)) : nullptr;
    d.gap = static_cast<float*>(at(p.pub.gap));
    d.ids = static_cast<int32_t*>(at(p.pub.ids));
    d.gates = static_cast<float*>(at(p.pub.gates));
    d.counts = static_cast<int32_t*>(at(p.pub.counts));
    d.offsets = static_cast<int32_t*>(at(p.pub.offsets));
    d.perm = static_cast<int32_t*>(at(p.pub.perm));
    d.inv = static_cast<int32_t*>(at(p.pub.inv));
    d.hq = static_cast<int8_t*>(at(p.pub.hq));
    d.hd = static_cast<float*>(at(p.pub.hd));
    d.hbs = static_cast<int16_t*>(at(p.pub.hbs));
    d.bar = static_cast<unsigned long long*>(at(p.bar));
    d.phase_ns = static_cast<unsigned long long*>(at(p.phase_ns));
    d.status = static_cast<int*>(at(p.pub.status));
    d.n_layers = n_layers;
    d.layers = layers;
    cudaStream_t s = as_stream(stream);
    trace_record(s);
    const cudaError_t err = record_error(launch_decode_fused(d, s));
    trace_record(s);
    if (err == cudaErrorCooperativeLaunchTooLarge) {
      cudaGetLastError();
      return MOE_ERR_UNSUPPORTED;
    }
    return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  }
  DecodeArgs d{};
  d.fmt = desc->fmt;
  d.H = H;
  d.I = desc->I;
  d.E = E;
  d.k = k;
  d.S = S;
  d.route = desc->route;
  d.T = T;
  d.gap = static_cast<float*>(at(p.pub.gap));
  d.ids = static_cast<int32_t*>(at(p.pub.ids));
  d.gates = static_cast<float*>(at(p.pub.gates));
  d.counts = static_cast<int32_t*>(at(p.pub.counts));
  d.offsets = static_cast<int32_t*>(at(p.pub.offsets));
  d.perm = static_cast<int32_t*>(at(p.pub.perm));
  d.inv = static_cast<int32_t*>(at(p.pub.inv));
  d.bar = static_cast<unsigned long long*>(at(p.bar));
  d.phase_ns = static_cast<unsigned long long*>(at(p.phase_ns));
  d.status = static_cast<int*>(at(p.pub.status));
  d.n_layers = n_layers;
  d.layers = layers;
  d.stk = static_cast<uint8_t*>(at(ext));
  d.sp = sp;
  cudaStream_t s = as_stream(stream);
  trace_record(s);
  const cudaError_t err = record_error(launch_decode_stack(d, s));
  trace_record(s);
  if (err == cudaErrorCooperativeLaunchTooLarge) {
    cudaGetLastError();
    return MOE_ERR_UNSUPPORTED;
  }
  return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int moe_get_status(void* ws, void* stream) {
  if (!ws) return MOE_ERR_INVALID_ARG;
  if (record_error(cudaStreamSynchronize(as_stream(stream))) != cudaSuccess) return MOE_ERR_CUDA;
  int v = 0;
  if (record_error(cudaMemcpy(&v, ws, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess) return MOE_ERR_CUDA;
  // clear the status block (status word, tile count and the grid-barrier
  // counter, which a timed-out barrier leaves out of step)
  if (v != 0 && cudaMemset(ws, 0, 16) != cudaSuccess) return MOE_ERR_CUDA;
  return v;
}

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE_BOUNDS: return "device: index out of range";
    case MOE_ERR_DEVICE_TIMEOUT: return "device: bounded wait ran out";
    default: return "unknown status";
  }
}

int moe_trace_events(void* const* events, int32_t n_events) {
  if (n_events < 0 || (n_events > 0 && !events)) return MOE_ERR_INVALID_ARG;
  g_trace_events = n_events > 0 ? events : nullptr;
  g_trace_n = n_events;
  g_trace_next = 0;
  return MOE_OK;
}

int moe_last_cuda_error(void) { return last_error(); }

unsigned long long moe_kernel_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int moe_layer_path(const moe_layer_desc* desc, int32_t T) {
  int why;
  if (!desc_valid(desc, &why)) return why;
  if (T < 0 || T > desc->T_max) return MOE_ERR_INVALID_ARG;
  const int k = desc->top_k;
  if (T <= kDecodeMaxT && (int64_t)T * k <= kSmallPairs &&
      decode_smem_bytes(T, desc->H, desc->I, desc->E, k, desc->n_shared) <= kDecodeSmemMax)
    return MOE_PATH_DECODE_FUSED;
  return prefill_path(T, k, desc->E, desc->fmt) && prefill_fits(desc->T_max, *desc) ? MOE_PATH_TENSOR_PREFILL
                                                                                      : MOE_PATH_GEMV;
}

int moe_stack_kernel(const moe_layer_desc* desc, int32_t n_layers, int32_t T, int32_t n_sms) {
  int why;
  if (!desc_valid(desc, &why)) return why;
  if (n_layers < 1 || T < 1 || T > desc->T_max) return MOE_ERR_INVALID_ARG;
  const int k = desc->top_k;
  if (T > kDecodeMaxT || (int64_t)T * k > kSmallPairs ||
      decode_smem_bytes(T, desc->H, desc->I, desc->E, k, desc->n_shared) > kDecodeSmemMax)
    return MOE_ERR_UNSUPPORTED;
  return stack_takes_pipelined(*desc, n_layers, T, n_sms) ? MOE_STACK_PIPELINED : MOE_STACK_DATAFLOW;
}

int moe_prefill_tile_tokens(void) { return prefill_tile_tokens(); }

int32_t moe_trace_used(void) { return g_trace_events || g_trace_next > 0 ? g_trace_next : 0; }

int moe_debug_wait_timeout(void* ws, int32_t limit_us, void* stream) {
  if (!ws || !aligned(ws, kAlign) || limit_us < 1 || limit_us > 1000000) return MOE_ERR_INVALID_ARG;
  int* status = static_cast<int*>(ws);
  const unsigned* flag = reinterpret_cast<const unsigned*>(static_cast<char*>(ws) + 4);  // never the magic
  return check(launch_debug_wait(status, flag, (long long)limit_us * 1000, as_stream(stream)));
}

int moe_debug_subblock_dots(int32_t fmt, const void* w, int32_t N, int32_t K, const int8_t* q, int32_t T,
                            int32_t* isum, int32_t* bsum, void* stream) {
  if (fmt < MOE_FMT_Q4K || fmt > MOE_FMT_IQ2G) return MOE_ERR_UNSUPPORTED;
  if (N <= 0 || K <= 0 || N % 256 || K % 256 || T < 1 || T > 16) return MOE_ERR_UNSUPPORTED;
  if (!w || !q || !isum || !bsum) return MOE_ERR_INVALID_ARG;
  if (!aligned(w, 16) || !aligned(q, 16)) return MOE_ERR_INVALID_ARG;
  return check(launch_debug_dots(fmt, w, N, K, q, T, isum, bsum, as_stream(stream)));
}

size_t moe_debug_prefill_sums_workspace_size(int32_t N, int32_t K, int32_t T) {
  if (N <= 0 || K <= 0 || T < 1 || N % 128 || K % 256 || N > MOE_MAX_DIM || K > MOE_MAX_DIM) return 0;
  return sums_plan(N, K, T).total;
}

int moe_debug_prefill_sums(int32_t fmt, const void* w, int32_t N, int32_t K, const int8_t* q, const float* d,
                           const int16_t* bsum16, int32_t T, int32_t* S, int32_t* M, void* ws, size_t ws_bytes,
                           void* stream) {
  if (!prefill_format(fmt)) return MOE_ERR_UNSUPPORTED;
  if (N <= 0 || K <= 0 || T < 1) return MOE_ERR_INVALID_ARG;
  if (N % 128 || K % 256 || N > MOE_MAX_DIM || K > MOE_MAX_DIM || (int64_t)T * (K / 256) * 2 >= ((int64_t)1 << 31))
    return MOE_ERR_UNSUPPORTED;
  if (!w || !q || !d || !bsum16 || !S || !M || !ws) return MOE_ERR_INVALID_ARG;
  if (!aligned(w, 16) || !aligned(q, 16) || !aligned(d, 4) || !aligned(bsum16, 4) || !aligned(ws, kAlign))
    return MOE_ERR_INVALID_ARG;
  if (ws_bytes < sums_plan(N, K, T).total) return MOE_ERR_WORKSPACE;
  SumsArgs a{};
  a.fmt = fmt;
  a.N = N;
  a.K = K;
  a.T = T;
  a.w = w;
  a.q = q;
  a.d = d;
  a.bs16 = bsum16;
  a.S = S;
  a.M = M;
  a.ws = ws;
  return check(launch_prefill_sums(a, as_stream(stream)));
}

}  // extern "C"
