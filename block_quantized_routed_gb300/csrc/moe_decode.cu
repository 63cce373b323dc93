// Single-launch decode: the MoE layer for a few tokens (T <= 16), or a stack
// of such layers, in one cooperative, persistent kernel (one CTA per SM, all
// co-resident).  The work of a layer is cut into five phases:
//
//   router    router logits (warps split expert rows) and q8_K of x
//   routing   every CTA redundantly: top-k of every token, bucketing and the
//             tile plan, in shared memory (no barrier needed after it)
//   gate/up   items (tile, 32-row group), round-robin over CTAs; the 8 warps
//             of a CTA split the super-blocks, partial sums are reduced in a
//             fixed order; h = silu(G) * U goes to global memory
//   down      items (tile, group of row groups) in contiguous blocks per CTA,
//             so the q8_K of a tile's h is made once per CTA; y by slot
//   combine   out = residual + sum_s gate * y (slots in order, then shared)
//
// Two schedules:
//   sequential  router | routing + gate/up | down | combine, with a grid
//               barrier between them (and between layers): layer l+1 may read
//               layer l's output.
//   pipelined   for stacks whose layer inputs do not alias the outputs of the
//               three layers before them (checked on the device): stage s runs
//               routing(s+1) + L2 prefetch of its experts, gate/up(s),
//               down(s-1), router(s+2) and combine(s-2), then one grid
//               barrier.  Every phase of a layer still sees all of its inputs
//               complete; only independent work of neighbouring layers shares
//               a stage, so results equal the sequential schedule's.
// Weights that a later phase will read are prefetched into L2 with bulk
// prefetches (the next gate/up items, the first down items, the next layers'
// router rows and experts).
//
// The barrier is a 64-bit arrival counter; every wait is bounded and sets
// MOE_ERR_DEVICE_TIMEOUT instead of hanging.  Data written inside the kernel
// is read back through L2 (ld.global.cg), never through L1 or the read-only
// path.  CTA 0 stamps its SM cycle counter at phase boundaries of the last
// layer into the workspace.
//
// Sources: Pulsar README, "How the streaming works" (one expert union per
// batch; explicit per-(token, slot) pointers, NULL = not mine; a thread
// prefetches the next layer's experts), "Fidelity notes" (q8_0/q8_K
// activations, integer dp4a dots, the per-slot sum), "What it does today"
// (Q4_K matmuls on q8_K activations); Strata summary (the per-token layer
// loop replayed as captured work, zero allocation on the token path).
#include <algorithm>
#include <cmath>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kDecThreads = 256;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kRSlots = 4;                    // routing states kept (pipelined schedule)
constexpr long long kSpinLimit = 1ll << 24;  // x ~64 ns sleeps: about a second
constexpr int kDownAhead = 4;                // down items of L2 prefetch ahead

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  // bulk prefetch into L2; bytes is a multiple of 16 and p is 16-byte aligned
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Grid-wide barrier on a monotonic 64-bit counter: arrivals are grouped in
// generations of gridDim.x.  Returns false if the wait ran out.
__device__ bool grid_barrier(unsigned long long* bar, int* status) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned long long n = gridDim.x;
    const unsigned long long old = atomicAdd(bar, 1ull);
    const unsigned long long target = (old / n + 1ull) * n;
    int ok = 1;
    long long spins = 0;
    while (ld_acquire_u64(bar) < target) {
      if (++spins > kSpinLimit) {
        set_status(status, MOE_ERR_DEVICE_TIMEOUT);
        ok = 0;
        break;
      }
      __nanosleep(64);
    }
    __threadfence();
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

// Routing state of one layer in shared memory.
struct Route {
  int* ids;       // [T*k]
  float* gates;   // [T*k]
  int* tok;       // [P]  token of each bucket position
  int* slot;      // [P]  slot index of each bucket position
  Tile* tiles;    // [P]
  uint8_t* ok;    // [T*k + S]  expert of the slot / shared expert is present
  int* n_tiles;   // [1]
};

struct Smem {
  int8_t* xq;      // [T][H]
  int16_t* xbs;    // [T][H/16]
  float* xd;       // [T][nbH]
  uint8_t* rbase;  // kRSlots routing states, rstride bytes apart
  uint32_t rstride;
  int* cnt;        // [E+S+1]  counts -> offsets (routing scratch)
  int* scan;       // [E+S+1]  tile-plan scratch
  float* red;      // [8 warps][2][max(T,16)][32] accumulators / partial sums
  int8_t* hq;      // [T][I]
  int16_t* hbs;    // [T][I/16]
  float* hd;       // [T][nbI]
  int* aoff;       // [T]  activation row offsets of the current item
};

__host__ __device__ inline size_t al16(size_t v) { return (v + 15) / 16 * 16; }

// bytes of one routing state: ids, gates [T*k]; tok, slot [P]; tiles [P]; n_tiles
__host__ __device__ inline size_t route_bytes(int T, int k, int S) {
  const size_t P = (size_t)T * (k + S);
  return al16((size_t)T * k * 4) * 2 + al16(P * 4) * 2 + al16(P * sizeof(Tile)) + al16((size_t)T * k + S) + 16;
}

__device__ __forceinline__ Route route_at(uint8_t* base, int T, int k, int S) {
  const size_t P = (size_t)T * (k + S);
  Route r;
  uint8_t* p = base;
  r.ids = reinterpret_cast<int*>(p);      p += al16((size_t)T * k * 4);
  r.gates = reinterpret_cast<float*>(p);  p += al16((size_t)T * k * 4);
  r.tok = reinterpret_cast<int*>(p);      p += al16(P * 4);
  r.slot = reinterpret_cast<int*>(p);     p += al16(P * 4);
  r.tiles = reinterpret_cast<Tile*>(p);   p += al16(P * sizeof(Tile));
  r.ok = p;                               p += al16((size_t)T * k + S);
  r.n_tiles = reinterpret_cast<int*>(p);
  return r;
}

// Shared-memory carve-up (host and device agree on it).
__host__ __device__ inline size_t decode_smem(int T, int H, int I, int E, int k, int S, Smem* sm, uint8_t* base) {
  const int P = T * (k + S);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += al16(bytes);
    return base ? base + at : nullptr;
  };
  uint8_t* p;
  p = take((size_t)T * H);                 if (sm) sm->xq = (int8_t*)p;
  p = take((size_t)T * (H / 16) * 2);      if (sm) sm->xbs = (int16_t*)p;
  p = take((size_t)T * (H / 256) * 4);     if (sm) sm->xd = (float*)p;
  const size_t rstride = route_bytes(T, k, S);
  p = take(rstride * kRSlots);             if (sm) { sm->rbase = p; sm->rstride = (uint32_t)rstride; }
  p = take((size_t)(E + S + 1) * 4);       if (sm) sm->cnt = (int*)p;
  p = take((size_t)(E + S + 1) * 4);       if (sm) sm->scan = (int*)p;
  p = take((size_t)kDecWarps * 2 * (T > 16 ? T : 16) * 32 * 4); if (sm) sm->red = (float*)p;
  p = take((size_t)T * I);                 if (sm) sm->hq = (int8_t*)p;
  p = take((size_t)T * (I / 16) * 2);      if (sm) sm->hbs = (int16_t*)p;
  p = take((size_t)T * (I / 256) * 4);     if (sm) sm->hd = (float*)p;
  p = take((size_t)T * 4);                 if (sm) sm->aoff = (int*)p;
  return off;
}

// The pointers of one layer (from the argument block for a single layer, or
// from the device-resident layer array of a stack).
struct LayerView {
  const moe_expert_ptrs* table;
  const float* w_router;
  const float* bias;
  const float* x;
  const float* residual;
  float* out;
  int32_t* ids_out;
  float* gates_out;
};

__device__ __forceinline__ LayerView layer_view(const DecodeArgs& a, int l) {
  LayerView v;
  if (a.layers) {
    const moe_layer_ptrs lp = a.layers[l];
    v.table = lp.table;
    v.w_router = lp.w_router;
    v.bias = lp.router_bias;
    v.x = lp.x;
    v.residual = lp.residual;
    v.out = lp.out;
    v.ids_out = lp.ids_out;
    v.gates_out = lp.gates_out;
  } else {
    v.table = a.table;
    v.w_router = a.w_router;
    v.bias = a.bias;
    v.x = a.x;
    v.residual = a.residual;
    v.out = a.out;
    v.ids_out = a.ids_out;
    v.gates_out = a.gates_out;
  }
  return v;
}

// Per-launch constants and the shared-memory view, passed to every phase.
template <int FMT>
struct Ctx {
  const DecodeArgs& a;
  Smem sm;
  int T, H, I, E, k, S, P, EpS;
  int nbH, nbI, nRG, nRGH;
  int tid, lane, warp, G;
  int W;                      // CTAs that take items (all, or all but the routing CTA)
  int wpr, rows_cta;          // router split
  int rg_per, n_grp;          // down items: row groups per item, items per tile
  size_t gu_run, dn_rg_bytes;

  __device__ Ctx(const DecodeArgs& args, uint8_t* smem_raw) : a(args) {
    T = a.T; H = a.H; I = a.I; E = a.E; k = a.k; S = a.S;
    P = T * (k + S);
    EpS = E + S;
    decode_smem(T, H, I, E, k, S, &sm, smem_raw);
    nbH = H / 256; nbI = I / 256; nRG = I / 32; nRGH = H / 32;
    tid = threadIdx.x; lane = tid & 31; warp = tid >> 5; G = gridDim.x;
    W = G;
    set_workers(G);
  }
  // item distribution over the first w CTAs
  __device__ void set_workers(int w) {
    W = w;
    const int GW = W * kDecWarps;
    wpr = GW >= 8 * E ? 8 : GW >= 4 * E ? 4 : GW >= 2 * E ? 2 : 1;
    rows_cta = kDecWarps / wpr;
    rg_per = nbI >= kDecWarps ? 1 : kDecWarps / nbI;
    n_grp = (nRGH + rg_per - 1) / rg_per;
    gu_run = (size_t)nbH * Fmt<FMT>::kSlabBytes;
    dn_rg_bytes = (size_t)nbI * Fmt<FMT>::kSlabBytes;
  }
  __device__ Route route(int slot) const { return route_at(sm.rbase + (size_t)slot * sm.rstride, T, k, S); }
  __device__ void stamp(int i, bool on) const {
    if (on && blockIdx.x == 0 && tid == 0 && a.phase_ns) a.phase_ns[i] = (unsigned long long)clock64();
  }
  // Down items of a layer with n_tiles tiles: (tile, group of `per` row
  // groups).  With enough items for every CTA, a warp owns a whole row group
  // (by_warp: 8 row groups per item, no cross-warp reduction); otherwise the
  // warps of a CTA split the super-blocks of rg_per row groups.
  __device__ void down_plan(int n_tiles, int& per, int& ngrp, bool& by_warp) const {
    const int nblk = (nRGH + kDecWarps - 1) / kDecWarps;
    by_warp = (long long)n_tiles * nblk >= W && nbI >= 2;
    per = by_warp ? kDecWarps : rg_per;
    ngrp = by_warp ? nblk : n_grp;
  }
  // down items to keep in flight towards L2 ahead of use (about 192 KB per CTA)
  __device__ int down_ahead(int n_tiles) const {
    int per, ngrp;
    bool bw;
    down_plan(n_tiles, per, ngrp, bw);
    const int n = (int)((size_t)(192 * 1024) / ((size_t)per * dn_rg_bytes));
    return n < 1 ? 1 : n > kDownAhead ? kDownAhead : n;
  }
  // down items [begin, end) of this CTA
  __device__ void down_range(int n_tiles, int& begin, int& end) const {
    int per, ngrp;
    bool bw;
    down_plan(n_tiles, per, ngrp, bw);
    const int n3 = n_tiles * ngrp;
    begin = (int)((long long)n3 * blockIdx.x / W);
    end = (int)((long long)n3 * (blockIdx.x + 1) / W);
  }
};

// ---------------------------------------------------------------- router
// logits[t, e] for this CTA's rows, and (from the last warps of the grid)
// the q8_K of x.
template <int FMT>
__device__ void router_phase(Ctx<FMT>& c, const LayerView& lv, float* logits, int8_t* xq, float* xd,
                             int16_t* xbs) {
  const int T = c.T, H = c.H, E = c.E, lane = c.lane, warp = c.warp, tid = c.tid;
  const int H4 = H >> 2;
  const int rl = warp / c.wpr, ch = warp % c.wpr;
  const int c4 = H4 / c.wpr;  // float4s per chunk
  float* part = c.sm.red;     // [8 warps][T] partial sums
  for (int base = blockIdx.x * c.rows_cta; base < E; base += c.W * c.rows_cta) {
    const int e = base + rl;
    float acc[16];
#pragma unroll
    for (int t = 0; t < 16; ++t) acc[t] = 0.0f;
    if (e < E) {
      const float4* wr = reinterpret_cast<const float4*>(lv.w_router + (size_t)e * H) + ch * c4;
      const float4* xr = reinterpret_cast<const float4*>(lv.x) + ch * c4;
#pragma unroll 2
      for (int h4 = lane; h4 < c4; h4 += 32) {
        const float4 wv = __ldg(wr + h4);
#pragma unroll
        for (int t = 0; t < 16; ++t)
          if (t < T) {
            const float4 xv = __ldcg(xr + (size_t)t * H4 + h4);  // x may be a previous layer's output
            acc[t] = fmaf(wv.x, xv.x, acc[t]);
            acc[t] = fmaf(wv.y, xv.y, acc[t]);
            acc[t] = fmaf(wv.z, xv.z, acc[t]);
            acc[t] = fmaf(wv.w, xv.w, acc[t]);
          }
      }
    }
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      if (t < T) {
        float v = acc[t];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) part[warp * T + t] = v;
      }
    }
    __syncthreads();
    for (int i = tid; i < c.rows_cta * T; i += kDecThreads) {
      const int r = i / T, t = i % T, er = base + r;
      if (er < E) {
        float v = 0.0f;
        for (int q = 0; q < c.wpr; ++q) v += part[(r * c.wpr + q) * T + t];
        logits[(size_t)t * E + er] = v + (lv.bias ? __ldg(lv.bias + er) : 0.0f);
      }
    }
    __syncthreads();
  }
  // q8_K of x: one warp per 256-element block, from the last warps of the grid down
  const int gw = blockIdx.x * kDecWarps + warp, GW = c.W * kDecWarps;
  for (int qb = GW - 1 - gw; qb < T * c.nbH; qb += GW) {
    const float4* src = reinterpret_cast<const float4*>(lv.x + (size_t)qb * 256 + 8 * lane);
    const float4 v0 = __ldcg(src), v1 = __ldcg(src + 1);
    const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    q8k_block_warp(v, lane, xq + (size_t)qb * 256, xd + qb, xbs + (size_t)qb * 16);
  }
}

// L2 prefetch of this CTA's router rows of a layer
template <int FMT>
__device__ void prefetch_router(const Ctx<FMT>& c, const LayerView& lv) {
  if (c.tid != 0) return;
  for (int base = blockIdx.x * c.rows_cta; base < c.E; base += c.W * c.rows_cta)
    prefetch_l2(lv.w_router + (size_t)base * c.H, (uint32_t)((size_t)min(c.rows_cta, c.E - base) * c.H * 4));
}

// L2 prefetch of the shared experts' gate/up items of this CTA (known before routing)
template <int FMT>
__device__ void prefetch_shared_gateup(const Ctx<FMT>& c, const LayerView& lv) {
  if (c.tid != 0) return;
  for (int it = blockIdx.x; it < c.S * c.nRG; it += c.W) {
    const moe_expert_ptrs ep = lv.table[c.E + it / c.nRG];
    if (!ep.gate) continue;
    prefetch_l2(static_cast<const uint8_t*>(ep.gate) + (size_t)(it % c.nRG) * c.gu_run, (uint32_t)c.gu_run);
    prefetch_l2(static_cast<const uint8_t*>(ep.up) + (size_t)(it % c.nRG) * c.gu_run, (uint32_t)c.gu_run);
  }
}

// ---------------------------------------------------------------- routing
// Top-k of every token, bucketing and the tile plan into route slot R (every
// CTA computes the same result).  CTA 0 also writes the routing to global
// memory (ids, gates, gap, counts, offsets, perm, inv and the caller's
// ids_out / gates_out).
template <int FMT>
__device__ void routing_phase(Ctx<FMT>& c, const LayerView& lv, const float* logits, const Route& R, bool stamps,
                              bool writer) {
  const DecodeArgs& a = c.a;
  const int T = c.T, E = c.E, k = c.k, S = c.S, EpS = c.EpS, P = c.P, tid = c.tid;
  Smem& sm = c.sm;
  for (int e = tid; e < EpS; e += kDecThreads) sm.cnt[e] = 0;
  for (int t = c.warp; t < T; t += kDecWarps)
    warp_topk(logits + (size_t)t * E, E, k, a.route, c.lane, R.ids + t * k, R.gates + t * k,
              writer && a.gap ? a.gap + t : nullptr);
  __syncthreads();
  c.stamp(9, stamps);
  // counts per expert (low 16 bits) and one "used" mark (bit 16): a single
  // scan then gives every bucket's offset and every tile's index (tiles in
  // expert order, shared experts last, like the buckets)
  for (int p = tid; p < T * k; p += kDecThreads) atomicAdd(&sm.cnt[R.ids[p]], 1);
  for (int sh = tid; sh < S; sh += kDecThreads) sm.cnt[E + sh] = T;
  // presence of each slot's expert (one read of the pointer table)
  for (int p = tid; p < T * k + S; p += kDecThreads) {
    const int e = p < T * k ? R.ids[p] : E + (p - T * k);
    R.ok[p] = lv.table[e].gate != nullptr ? 1 : 0;
  }
  __syncthreads();
  for (int e = tid; e < EpS; e += kDecThreads) {
    const int cnt = sm.cnt[e];
    if (writer) a.counts[e] = cnt;
    sm.scan[e] = cnt; // keep the counts
    sm.cnt[e] = cnt | (cnt > 0 ? 1 << 16 : 0);
  }
  __syncthreads();
  const int total = block_exclusive_scan(sm.cnt, EpS);
  c.stamp(10, stamps);
  for (int p = tid; p < T * k; p += kDecThreads) {
    const int e = R.ids[p];
    int rank = 0;
    for (int q = 0; q < p; ++q) rank += (R.ids[q] == e);
    const int pos = (sm.cnt[e] & 0xFFFF) + rank;
    R.tok[pos] = p / k;
    R.slot[pos] = p;
    if (rank == 0) {  // the expert's tile
      Tile tl;
      tl.expert = e;
      tl.start = sm.cnt[e] & 0xFFFF;
      tl.count = sm.scan[e];
      tl.flag = R.ok[p] ? 0 : 1;
      R.tiles[sm.cnt[e] >> 16] = tl;
    }
  }
  for (int i = tid; i < S * T; i += kDecThreads) {
    const int sh = i / T, t = i % T, e = E + sh;
    const int pos = (sm.cnt[e] & 0xFFFF) + t;
    R.tok[pos] = t;
    R.slot[pos] = T * k + sh * T + t;
    if (t == 0) {
      Tile tl;
      tl.expert = e;
      tl.start = sm.cnt[e] & 0xFFFF;
      tl.count = T;
      tl.flag = R.ok[T * k + sh] ? 0 : 1;
      R.tiles[sm.cnt[e] >> 16] = tl;
    }
  }
  if (tid == 0) *R.n_tiles = total >> 16;
  __syncthreads();
  c.stamp(11, stamps);
  if (writer) {
    for (int e = tid; e < EpS; e += kDecThreads) a.offsets[e] = sm.cnt[e] & 0xFFFF;
    if (tid == 0) a.offsets[EpS] = total & 0xFFFF;
    for (int j = tid; j < P; j += kDecThreads) {
      a.perm[j] = R.slot[j];
      if (a.inv) a.inv[R.slot[j]] = j;
    }
    for (int p = tid; p < T * k; p += kDecThreads) {
      a.ids[p] = R.ids[p];
      a.gates[p] = R.gates[p];
      if (lv.ids_out) lv.ids_out[p] = R.ids[p];
      if (lv.gates_out) lv.gates_out[p] = R.gates[p];
    }
  }
}

// L2 prefetch of the down weights of this CTA's down items [i0, i1) of a layer
template <int FMT>
__device__ void prefetch_down(const Ctx<FMT>& c, const LayerView& lv, const Route& R, int i0, int i1) {
  int per, ngrp;
  bool bw;
  c.down_plan(*R.n_tiles, per, ngrp, bw);
  while (i0 < i1) {
    const int ti = i0 / ngrp;
    const int last = min(i1, (ti + 1) * ngrp);
    const Tile tl = R.tiles[ti];
    if (!tl.flag) {
      const int rg0 = (i0 % ngrp) * per;
      const int rg1 = min(c.nRGH, ((last - 1) % ngrp + 1) * per);
      prefetch_l2(static_cast<const uint8_t*>(lv.table[tl.expert].down) + (size_t)rg0 * c.dn_rg_bytes,
                  (uint32_t)((size_t)(rg1 - rg0) * c.dn_rg_bytes));
    }
    i0 = last;
  }
}

// L2 prefetch of a gate/up item (both runs)
template <int FMT>
__device__ void prefetch_gateup_item(const Ctx<FMT>& c, const LayerView& lv, const Route& R, int it) {
  if (it >= *R.n_tiles * c.nRG) return;
  const Tile tn = R.tiles[it / c.nRG];
  if (tn.flag) return;
  const moe_expert_ptrs en = lv.table[tn.expert];
  prefetch_l2(static_cast<const uint8_t*>(en.gate) + (size_t)(it % c.nRG) * c.gu_run, (uint32_t)c.gu_run);
  prefetch_l2(static_cast<const uint8_t*>(en.up) + (size_t)(it % c.nRG) * c.gu_run, (uint32_t)c.gu_run);
}

// Everything this CTA will read of a layer's experts (gate/up items and the
// first down items), issued as soon as the layer's routing is known.
template <int FMT>
__device__ void prefetch_layer_experts(const Ctx<FMT>& c, const LayerView& lv, const Route& R) {
  if (c.tid != 0) return;
  const int n2 = *R.n_tiles * c.nRG;
  for (int it = blockIdx.x; it < n2; it += c.W) prefetch_gateup_item(c, lv, R, it);
  int d0, d1;
  c.down_range(*R.n_tiles, d0, d1);
  prefetch_down(c, lv, R, d0, min(d1, d0 + c.down_ahead(*R.n_tiles)));
}

// The whole of every expert a layer uses (gate, up and down matrices), from
// one CTA: the pipelined schedule issues it one stage ahead of the use.
template <int FMT>
__device__ void prefetch_all_experts(const Ctx<FMT>& c, const LayerView& lv, const Route& R) {
  const int nt = *R.n_tiles;
  const size_t gu = (size_t)c.nRG * c.gu_run, dn = (size_t)c.nRGH * c.dn_rg_bytes;
  for (int i = c.tid; i < nt * 3; i += kDecThreads) {
    const Tile tl = R.tiles[i / 3];
    if (tl.flag) continue;
    const moe_expert_ptrs ep = lv.table[tl.expert];
    const int m = i % 3;
    const void* base = m == 0 ? ep.gate : m == 1 ? ep.up : ep.down;
    const size_t bytes = m < 2 ? gu : dn;
    for (size_t off = 0; off < bytes; off += (size_t)1 << 20)   // in pieces of up to 1 MiB
      prefetch_l2(static_cast<const uint8_t*>(base) + off, (uint32_t)min(bytes - off, (size_t)1 << 20));
  }
}

// q8_K rows of x (written in another phase by other CTAs: via L2) into shared memory
template <int FMT>
__device__ void stage_x(Ctx<FMT>& c, const int8_t* xq, const float* xd, const int16_t* xbs) {
  const int T = c.T, H = c.H;
  const int nq = T * H / 16, nb16 = T * H / 128, nd = T * c.nbH;
  for (int i = c.tid; i < nq; i += kDecThreads)
    reinterpret_cast<int4*>(c.sm.xq)[i] = __ldcg(reinterpret_cast<const int4*>(xq) + i);
  for (int i = c.tid; i < nb16; i += kDecThreads)
    reinterpret_cast<int4*>(c.sm.xbs)[i] = __ldcg(reinterpret_cast<const int4*>(xbs) + i);
  for (int i = c.tid; i < nd; i += kDecThreads) c.sm.xd[i] = __ldcg(xd + i);
  __syncthreads();
}

// ---------------------------------------------------------------- gate/up
// pf_next: prefetch this CTA's next gate/up items and first down items while
// the first item's loads are in flight (used when nothing prefetched them).
template <int FMT>
__device__ void gateup_phase(Ctx<FMT>& c, const LayerView& lv, const Route& R, float* h, bool pf_next) {
  using F = Fmt<FMT>;
  const int T = c.T, H = c.H, I = c.I, nbH = c.nbH, nRG = c.nRG, lane = c.lane, warp = c.warp, tid = c.tid;
  Smem& sm = c.sm;
  const int n2 = *R.n_tiles * nRG;
  bool first = true;
  for (int it = blockIdx.x; it < n2; it += c.W) {
    const Tile tl = R.tiles[it / nRG];
    const int rg = it % nRG;
    if (tl.flag) continue;
    const moe_expert_ptrs ep = lv.table[tl.expert];
    const uint8_t* gbase = static_cast<const uint8_t*>(ep.gate) + (size_t)rg * c.gu_run;
    const uint8_t* ubase = static_cast<const uint8_t*>(ep.up) + (size_t)rg * c.gu_run;
    for (int t = tid; t < tl.count; t += kDecThreads) sm.aoff[t] = R.tok[tl.start + t] * H;
    // per-warp accumulators in shared memory: gate [T][32], then up [T][32]
    float* accw = sm.red + (size_t)warp * 2 * T * 32;
    for (int i = lane; i < tl.count * 32; i += 32) accw[i] = accw[T * 32 + i] = 0.0f;
    __syncthreads();
    for (int b = warp; b < nbH; b += kDecWarps) {
      SbRegs<FMT> sg, su;
      load_sb<FMT>(gbase + (size_t)b * F::kSlabBytes, lane, sg);
      load_sb<FMT>(ubase + (size_t)b * F::kSlabBytes, lane, su);
      if (pf_next && tid == 0 && b == warp) {
        if (first) prefetch_gateup_item(c, lv, R, it + c.W);
        prefetch_gateup_item(c, lv, R, it + 2 * c.W);
        if (first) {
          int d0, d1;
          c.down_range(*R.n_tiles, d0, d1);
          prefetch_down(c, lv, R, d0, min(d1, d0 + c.down_ahead(*R.n_tiles)));
        }
      }
      sb_accum<FMT>(sg, sm.xq, sm.xbs, sm.xd, sm.aoff, b, tl.count, accw, lane);
      sb_accum<FMT>(su, sm.xq, sm.xbs, sm.xd, sm.aoff, b, tl.count, accw + T * 32, lane);
    }
    first = false;
    __syncthreads();
    for (int idx = tid; idx < tl.count * 32; idx += kDecThreads) {
      const int t = idx >> 5, r = idx & 31;
      float Gv = 0.0f, Uv = 0.0f;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) {
        Gv += sm.red[((size_t)w * 2 * T + t) * 32 + r];
        Uv += sm.red[((size_t)w * 2 * T + T + t) * 32 + r];
      }
      h[(size_t)(tl.start + t) * I + rg * 32 + r] = Gv / (1.0f + expf(-Gv)) * Uv;
    }
    __syncthreads();
  }
  if (pf_next && first && tid == 0) {
    int d0, d1;
    c.down_range(*R.n_tiles, d0, d1);
    prefetch_down(c, lv, R, d0, min(d1, d0 + c.down_ahead(*R.n_tiles)));
  }
}

// ---------------------------------------------------------------- down
template <int FMT>
__device__ void down_phase(Ctx<FMT>& c, const LayerView& lv, const Route& R, const float* h, float* y,
                           int8_t* hq_keep, float* hd_keep, int16_t* hbs_keep) {
  using F = Fmt<FMT>;
  const int T = c.T, H = c.H, I = c.I, nbI = c.nbI, lane = c.lane, warp = c.warp, tid = c.tid;
  Smem& sm = c.sm;
  int d_begin, d_end;
  c.down_range(*R.n_tiles, d_begin, d_end);
  for (int t = tid; t < T; t += kDecThreads) sm.aoff[t] = t * I;
  __syncthreads();
  int per, ngrp;
  bool by_warp;
  c.down_plan(*R.n_tiles, per, ngrp, by_warp);
  const int ahead = c.down_ahead(*R.n_tiles);
  int staged = -1;  // tile whose q8_K(h) is in shared memory
  for (int it = d_begin; it < d_end; ++it) {
    const int ti = it / ngrp;
    const Tile tl = R.tiles[ti];
    const int grp = it % ngrp;
    const int rg0 = grp * per, nrg = min(per, c.nRGH - rg0);
    if (tid == 0 && it + ahead < d_end) prefetch_down(c, lv, R, it + ahead, it + ahead + 1);
    if (tl.flag) continue;
    if (ti != staged) {
      __syncthreads();  // previous readers of the staged rows are done
      for (int task = warp; task < tl.count * nbI; task += kDecWarps) {
        const int t = task / nbI, blk = task % nbI;
        const float4* src = reinterpret_cast<const float4*>(h + (size_t)(tl.start + t) * I + blk * 256 + 8 * lane);
        const float4 v0 = __ldcg(src), v1 = __ldcg(src + 1);
        const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        q8k_block_warp(v, lane, sm.hq + (size_t)t * I + blk * 256, sm.hd + t * nbI + blk,
                       sm.hbs + (size_t)t * (I / 16) + blk * 16);
      }
      __syncthreads();
      if (grp == 0 && hq_keep) {  // the CTA holding a tile's first item keeps a copy of q8_K(h)
        const size_t r0 = (size_t)tl.start;
        for (int i = tid; i < tl.count * I / 16; i += kDecThreads)
          reinterpret_cast<int4*>(hq_keep + r0 * I)[i] = reinterpret_cast<const int4*>(sm.hq)[i];
        for (int i = tid; i < tl.count * nbI; i += kDecThreads) hd_keep[r0 * nbI + i] = sm.hd[i];
        for (int i = tid; i < tl.count * (I / 16); i += kDecThreads) hbs_keep[r0 * (I / 16) + i] = sm.hbs[i];
      }
      staged = ti;
    }
    const uint8_t* dbase = static_cast<const uint8_t*>(lv.table[tl.expert].down);
    float* accw = sm.red + (size_t)warp * T * 32;
    for (int i = lane; i < tl.count * 32; i += 32) accw[i] = 0.0f;
    __syncwarp();
    if (by_warp) {
      // warp w owns row group rg0 + w: all of its super-blocks, two at a time
      if (warp < nrg) {
        const uint8_t* rbase = dbase + (size_t)(rg0 + warp) * c.dn_rg_bytes;
        for (int b = 0; b < nbI; b += 2) {
          SbRegs<FMT> s0, s1;
          load_sb<FMT>(rbase + (size_t)b * F::kSlabBytes, lane, s0);
          if (b + 1 < nbI) load_sb<FMT>(rbase + (size_t)(b + 1) * F::kSlabBytes, lane, s1);
          sb_accum<FMT>(s0, sm.hq, sm.hbs, sm.hd, sm.aoff, b, tl.count, accw, lane);
          if (b + 1 < nbI) sb_accum<FMT>(s1, sm.hq, sm.hbs, sm.hd, sm.aoff, b + 1, tl.count, accw, lane);
        }
        __syncwarp();
        for (int t = 0; t < tl.count; ++t)
          y[(size_t)R.slot[tl.start + t] * H + (rg0 + warp) * 32 + lane] = accw[t * 32 + lane];
      }
      continue;  // no cross-warp reduction; the next tile's staging synchronizes
    }
    // warp -> (row group, super-blocks)
    const int rgl = nbI >= kDecWarps ? 0 : warp / nbI;
    const int b0 = nbI >= kDecWarps ? warp : warp % nbI;
    const int bstep = nbI >= kDecWarps ? kDecWarps : nbI;
    if (rgl < nrg) {
      const uint8_t* rbase = dbase + (size_t)(rg0 + rgl) * c.dn_rg_bytes;
      for (int b = b0; b < nbI; b += bstep) {
        SbRegs<FMT> sd;
        load_sb<FMT>(rbase + (size_t)b * F::kSlabBytes, lane, sd);
        sb_accum<FMT>(sd, sm.hq, sm.hbs, sm.hd, sm.aoff, b, tl.count, accw, lane);
      }
    }
    __syncthreads();
    // reduce the warps of each row group in a fixed order; y by slot index
    const int wpr = nbI >= kDecWarps ? kDecWarps : nbI;  // warps per row group
    for (int idx = tid; idx < nrg * tl.count * 32; idx += kDecThreads) {
      const int r = idx & 31, t = (idx >> 5) % tl.count, g = (idx >> 5) / tl.count;
      float v = 0.0f;
      for (int w = g * wpr; w < g * wpr + wpr; ++w) v += sm.red[((size_t)w * T + t) * 32 + r];
      y[(size_t)R.slot[tl.start + t] * H + (rg0 + g) * 32 + r] = v;
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------- combine
template <int FMT>
__device__ void combine_phase(Ctx<FMT>& c, const LayerView& lv, const Route& R, const float* y) {
  const int T = c.T, H = c.H, E = c.E, k = c.k, S = c.S;
  const int H4 = H / 4;
  const float4* y4 = reinterpret_cast<const float4*>(y);
  for (int idx = blockIdx.x * kDecThreads + c.tid; idx < T * H4; idx += c.W * kDecThreads) {
    const int t = idx / H4, cc = idx % H4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < k; ++s) {
      if (!R.ok[t * k + s]) continue;  // expert not present ("not mine"): contributes nothing
      const float g = R.gates[t * k + s];
      const float4 v = __ldcg(y4 + (size_t)(t * k + s) * H4 + cc);
      acc.x = fmaf(g, v.x, acc.x);
      acc.y = fmaf(g, v.y, acc.y);
      acc.z = fmaf(g, v.z, acc.z);
      acc.w = fmaf(g, v.w, acc.w);
    }
    for (int sh = 0; sh < S; ++sh) {
      if (!R.ok[T * k + sh]) continue;
      const float4 v = __ldcg(y4 + (size_t)(T * k + sh * T + t) * H4 + cc);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    if (lv.residual) {
      const float4 r = __ldcg(reinterpret_cast<const float4*>(lv.residual) + idx);
      acc.x += r.x;
      acc.y += r.y;
      acc.z += r.z;
      acc.w += r.w;
    }
    reinterpret_cast<float4*>(lv.out)[idx] = acc;
  }
}

// Can the layers run pipelined?  Layer l's x is read two stages before
// layer l's gate/up, while layers l-1, l-2, l-3 may still be writing their
// outputs; so x_l must not overlap out_{l-1}, out_{l-2}, out_{l-3}.
__device__ bool layers_independent(const DecodeArgs& a, int n_layers) {
  const size_t bytes = (size_t)a.T * a.H * sizeof(float);
  for (int l = 1; l < n_layers; ++l) {
    const char* x = reinterpret_cast<const char*>(a.layers[l].x);
    for (int j = l - 3 < 0 ? 0 : l - 3; j < l; ++j) {
      const char* o = reinterpret_cast<const char*>(a.layers[j].out);
      if (x < o + bytes && o < x + bytes) return false;
    }
  }
  return true;
}

template <int FMT>
__global__ void __launch_bounds__(kDecThreads, 1) decode_fused_kernel(const __grid_constant__ DecodeArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  Ctx<FMT> c(a, smem_raw);
  const int L = a.n_layers > 0 ? a.n_layers : 1;
  const bool pipelined = a.layers && L > 1 && a.pipeline_ok && layers_independent(a, L);
  if (blockIdx.x == 0 && c.tid == 0 && a.phase_ns) a.phase_ns[15] = pipelined ? 2 : 1;  // which schedule ran

  if (!pipelined) {
    for (int layer = 0; layer < L; ++layer) {
      const LayerView lv = layer_view(a, layer);
      const Route R = c.route(0);
      const bool st = layer == L - 1;
      c.stamp(0, st);
      router_phase(c, lv, a.logits[0], a.xq[0], a.xd[0], a.xbs[0]);
      if (layer == 0) prefetch_shared_gateup(c, lv);
      c.stamp(1, st);
      if (!grid_barrier(a.bar, a.status)) return;
      c.stamp(2, st);
      stage_x(c, a.xq[0], a.xd[0], a.xbs[0]);
      routing_phase(c, lv, a.logits[0], R, st, blockIdx.x == 0);
      c.stamp(3, st);
      gateup_phase(c, lv, R, a.h[0], true);
      c.stamp(4, st);
      if (!grid_barrier(a.bar, a.status)) return;
      c.stamp(5, st);
      if (layer + 1 < L) {
        // the next layer's router rows and shared-expert items do not depend on this layer
        const LayerView nx = layer_view(a, layer + 1);
        prefetch_router(c, nx);
        prefetch_shared_gateup(c, nx);
      }
      down_phase(c, lv, R, a.h[0], a.y[0], a.hq, a.hd, a.hbs);
      c.stamp(6, st);
      if (!grid_barrier(a.bar, a.status)) return;
      c.stamp(7, st);
      combine_phase(c, lv, R, a.y[0]);
      c.stamp(8, st);
      // the next layer may read this layer's output
      if (layer + 1 < L && !grid_barrier(a.bar, a.status)) return;
    }
    return;
  }

  // pipelined: the last CTA computes routing(s+1) and publishes it to the
  // workspace with a per-layer flag; the other CTAs run gate/up(s),
  // down(s-1), router(s+2) and combine(s-2), then take routing(s+1) into
  // shared memory and prefetch their own items of layer s+1 into L2.
  const int D = c.G - 1;
  const bool router_cta = blockIdx.x == D;
  c.set_workers(c.G - 1);
  const size_t rbytes = c.sm.rstride;
  // nobody writes the flag before the first barrier: every CTA reads the same base
  __shared__ int s_ok;
  const unsigned long long flag_base = ld_acquire_u64(a.route_flag);
  for (int s = -2; s <= L + 1; ++s) {
    const bool st = s == L - 2;  // stamps of a steady-state stage (all five phases run)
    c.stamp(0, st);
    if (router_cta) {
      if (s + 1 >= 0 && s + 1 < L) {
        const LayerView lv = layer_view(a, s + 1);
        routing_phase(c, lv, a.logits[(s + 1) & 1], c.route((s + 1) & 3), false, true);
        const int4* src = reinterpret_cast<const int4*>(c.sm.rbase + (size_t)((s + 1) & 3) * rbytes);
        int4* dst = reinterpret_cast<int4*>(a.route_pub + (size_t)((s + 1) & 3) * rbytes);
        for (size_t i = c.tid; i < rbytes / 16; i += kDecThreads) dst[i] = src[i];
        __syncthreads();
        if (c.tid == 0) {
          __threadfence();
          atomicExch(a.route_flag, flag_base + (unsigned long long)(s + 2));  // layer s+1 published
        }
      }
    } else {
      if (s >= 0 && s < L) stage_x(c, a.xq[s % 3], a.xd[s % 3], a.xbs[s % 3]);  // ends with __syncthreads
      c.stamp(3, st);
      if (s >= 0 && s < L) gateup_phase(c, layer_view(a, s), c.route(s & 3), a.h[s & 1], false);
      c.stamp(4, st);
      if (s - 1 >= 0 && s - 1 < L)
        down_phase(c, layer_view(a, s - 1), c.route((s - 1) & 3), a.h[(s - 1) & 1], a.y[(s - 1) & 1],
                   s - 1 == L - 1 ? a.hq : nullptr, a.hd, a.hbs);
      c.stamp(6, st);
      if (s + 2 >= 0 && s + 2 < L) {
        const LayerView lv = layer_view(a, s + 2);
        router_phase(c, lv, a.logits[(s + 2) & 1], a.xq[(s + 2) % 3], a.xd[(s + 2) % 3], a.xbs[(s + 2) % 3]);
      }
      c.stamp(1, st);
      if (s - 2 >= 0 && s - 2 < L)
        combine_phase(c, layer_view(a, s - 2), c.route((s - 2) & 3), a.y[(s - 2) & 1]);
      if (s + 3 < L) prefetch_router(c, layer_view(a, s + 3));
      c.stamp(8, st);
      if (s + 1 >= 0 && s + 1 < L) {
        // take routing(s+1) as soon as the routing CTA has published it (bounded wait)
        if (c.tid == 0) {
          const unsigned long long want = flag_base + (unsigned long long)(s + 2);
          long long spins = 0;
          int ok = 1;
          while (ld_acquire_u64(a.route_flag) < want) {
            if (++spins > kSpinLimit) {
              set_status(a.status, MOE_ERR_DEVICE_TIMEOUT);
              ok = 0;
              break;
            }
            __nanosleep(32);
          }
          s_ok = ok;
        }
        __syncthreads();
        if (!s_ok) return;  // the status word says why; the routing CTA is not waiting on us
        const int4* src = reinterpret_cast<const int4*>(a.route_pub + (size_t)((s + 1) & 3) * rbytes);
        int4* dst = reinterpret_cast<int4*>(c.sm.rbase + (size_t)((s + 1) & 3) * rbytes);
        for (size_t i = c.tid; i < rbytes / 16; i += kDecThreads) dst[i] = __ldcg(src + i);
        __syncthreads();
        prefetch_layer_experts(c, layer_view(a, s + 1), c.route((s + 1) & 3));
      }
      c.stamp(12, st);
    }
    if (s < L + 1 && !grid_barrier(a.bar, a.status)) return;
  }
}

template <int FMT>
cudaError_t launch_decode_t(const DecodeArgs& a, cudaStream_t s) {
  const size_t smem = decode_smem(a.T, a.H, a.I, a.E, a.k, a.S, nullptr, nullptr);
  auto kern = decode_fused_kernel<FMT>;
  static size_t opted = 0;  // per instantiation; the opt-in only grows
  if (smem > opted) {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    opted = smem;
  }
  int per_sm = 0;
  cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kDecThreads, smem);
  if (err != cudaSuccess) return err;
  if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
  const int grid = num_sms() * std::min(per_sm, 2);
  DecodeArgs args = a;
  void* params[] = {&args};
  note_launch();
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(kern), dim3(grid), dim3(kDecThreads), params,
                                     smem, s);
}

}  // namespace

size_t decode_route_bytes(int T, int k, int S) { return route_bytes(T, k, S); }

size_t decode_smem_bytes(int T, int H, int I, int E, int k, int S) {
  return decode_smem(T, H, I, E, k, S, nullptr, nullptr);
}

cudaError_t launch_decode_fused(const DecodeArgs& a, cudaStream_t s) {
  return a.fmt == kQ4K ? launch_decode_t<kQ4K>(a, s) : launch_decode_t<kQ2K>(a, s);
}

}  // namespace moe
