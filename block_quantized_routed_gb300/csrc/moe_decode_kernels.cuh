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
#pragma once
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

// Grid-wide barrier on one 64-bit word: the arrival count in the low 32
// bits, a generation number in the high 32 bits.  The CTA that arrives last
// sets the count back to zero and advances the generation in one atomic
// store; the others wait (bounded) for the generation to change.  Every
// completed barrier leaves the count at zero, so a launch does not depend
// on the grid size of the launch before it on the same workspace.  Returns
// false if the wait ran out (the count is then left partial; the status
// read that reports the timeout clears the word).
__device__ bool grid_barrier(unsigned long long* bar, int* status) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned long long old = atomicAdd(bar, 1ull);
    const unsigned gen = (unsigned)(old >> 32);
    int ok = 1;
    if ((unsigned)(old & 0xFFFFFFFFull) == gridDim.x - 1u) {
      __threadfence();  // every other CTA's arrival (and its writes) is seen before the release
      atomicExch(bar, (unsigned long long)(gen + 1u) << 32);
    } else {
      long long spins = 0;
      while ((unsigned)(ld_acquire_u64(bar) >> 32) == gen) {
        if (++spins > kSpinLimit) {
          set_status(status, MOE_ERR_DEVICE_TIMEOUT);
          ok = 0;
          break;
        }
        __nanosleep(64);
      }
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
  float* red;      // [warps][2][max(T,16)][32] accumulators / partial sums
  int8_t* hq;      // [T][I]
  int16_t* hbs;    // [T][I/16]
  float* hd;       // [T][nbI]
  int* aoff;       // [T]  activation row offsets of the current item
  int* srow;       // [T]  slot rows of the current down item's tokens
};

__host__ __device__ inline size_t al16(size_t v) { return (v + 15) / 16 * 16; }

// bytes of one routing state: ids, gates [T*k]; tok, slot [P]; tiles [P]; n_tiles
__host__ __device__ inline size_t route_bytes(int T, int k, int S) {
  const size_t P = (size_t)T * (k + S);
  return al16((size_t)T * k * 4) * 2 + al16(P * 4) * 2 + al16(P * sizeof(Tile)) + al16((size_t)T * k + S) + 16;
}

// byte offsets of the fields of one routing state (host and device agree on it)
__host__ __device__ inline RouteFields route_fields_of(int T, int k, int S) {
  const size_t P = (size_t)T * (k + S);
  RouteFields f;
  size_t o = 0;
  f.ids = o;     o += al16((size_t)T * k * 4);
  f.gates = o;   o += al16((size_t)T * k * 4);
  f.tok = o;     o += al16(P * 4);
  f.slot = o;    o += al16(P * 4);
  f.tiles = o;   o += al16(P * sizeof(Tile));
  f.ok = o;      o += al16((size_t)T * k + S);
  f.n_tiles = o;
  return f;
}

__device__ __forceinline__ Route route_at(uint8_t* base, int T, int k, int S) {
  const RouteFields f = route_fields_of(T, k, S);
  Route r;
  r.ids = reinterpret_cast<int*>(base + f.ids);
  r.gates = reinterpret_cast<float*>(base + f.gates);
  r.tok = reinterpret_cast<int*>(base + f.tok);
  r.slot = reinterpret_cast<int*>(base + f.slot);
  r.tiles = reinterpret_cast<Tile*>(base + f.tiles);
  r.ok = base + f.ok;
  r.n_tiles = reinterpret_cast<int*>(base + f.n_tiles);
  return r;
}

// Shared-memory carve-up (host and device agree on it) for a CTA of nw warps.
__host__ __device__ inline size_t decode_smem(int T, int H, int I, int E, int k, int S, int nw, Smem* sm,
                                              uint8_t* base) {
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
  p = take((size_t)nw * 2 * (T > 16 ? T : 16) * 32 * 4); if (sm) sm->red = (float*)p;
  p = take((size_t)T * I);                 if (sm) sm->hq = (int8_t*)p;
  p = take((size_t)T * (I / 16) * 2);      if (sm) sm->hbs = (int16_t*)p;
  p = take((size_t)T * (I / 256) * 4);     if (sm) sm->hd = (float*)p;
  p = take((size_t)T * 4);                 if (sm) sm->aoff = (int*)p;
  p = take((size_t)T * 4);                 if (sm) sm->srow = (int*)p;
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
  int nw, nt;                 // warps and threads of this CTA
  int W;                      // CTAs that take items (all, or all but the routing CTA)
  int wpr, rows_cta;          // router split
  int rg_per, n_grp;          // down items: row groups per item, items per tile
  size_t gu_run, dn_rg_bytes;

  __device__ Ctx(const DecodeArgs& args, uint8_t* smem_raw) : a(args) {
    T = a.T; H = a.H; I = a.I; E = a.E; k = a.k; S = a.S;
    P = T * (k + S);
    EpS = E + S;
    nt = blockDim.x;
    nw = nt >> 5;
    decode_smem(T, H, I, E, k, S, nw, &sm, smem_raw);
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
                              bool writer, bool write_out) {
  const DecodeArgs& a = c.a;
  const int T = c.T, E = c.E, k = c.k, S = c.S, EpS = c.EpS, P = c.P, tid = c.tid;
  Smem& sm = c.sm;
  for (int e = tid; e < EpS; e += c.nt) sm.cnt[e] = 0;
  for (int t = c.warp; t < T; t += c.nw)
    warp_topk(logits + (size_t)t * E, E, k, a.route, c.lane, R.ids + t * k, R.gates + t * k,
              writer && a.gap ? a.gap + t : nullptr);
  __syncthreads();
  c.stamp(9, stamps);
  // counts per expert (low 16 bits) and one "used" mark (bit 16): a single
  // scan then gives every bucket's offset and every tile's index (tiles in
  // expert order, shared experts last, like the buckets)
  for (int p = tid; p < T * k; p += c.nt) atomicAdd(&sm.cnt[R.ids[p]], 1);
  for (int sh = tid; sh < S; sh += c.nt) sm.cnt[E + sh] = T;
  // presence of each slot's expert (one read of the pointer table)
  for (int p = tid; p < T * k + S; p += c.nt) {
    const int e = p < T * k ? R.ids[p] : E + (p - T * k);
    R.ok[p] = lv.table[e].gate != nullptr ? 1 : 0;
  }
  __syncthreads();
  for (int e = tid; e < EpS; e += c.nt) {
    const int cnt = sm.cnt[e];
    if (writer) a.counts[e] = cnt;
    sm.scan[e] = cnt; // keep the counts
    sm.cnt[e] = cnt | (cnt > 0 ? 1 << 16 : 0);
  }
  __syncthreads();
  const int total = block_exclusive_scan(sm.cnt, EpS);
  c.stamp(10, stamps);
  for (int p = tid; p < T * k; p += c.nt) {
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
  for (int i = tid; i < S * T; i += c.nt) {
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
    for (int e = tid; e < EpS; e += c.nt) a.offsets[e] = sm.cnt[e] & 0xFFFF;
    if (tid == 0) a.offsets[EpS] = total & 0xFFFF;
    for (int j = tid; j < P; j += c.nt) {
      a.perm[j] = R.slot[j];
      if (a.inv) a.inv[R.slot[j]] = j;
    }
    for (int p = tid; p < T * k; p += c.nt) {
      a.ids[p] = R.ids[p];
      a.gates[p] = R.gates[p];
    }
  }
  if (write_out)
    for (int p = tid; p < T * k; p += c.nt) {
      if (lv.ids_out) lv.ids_out[p] = R.ids[p];
      if (lv.gates_out) lv.gates_out[p] = R.gates[p];
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
  stage_format_tables<FMT>();
  Ctx<FMT> c(a, smem_raw);
  const int L = a.n_layers > 0 ? a.n_layers : 1;
  const bool pipelined = a.layers && L > 1 && a.pipeline_ok && layers_independent(a, L);
  if (blockIdx.x == 0 && c.tid == 0 && a.phase_ns) {
    a.phase_ns[15] = pipelined ? 2 : 1;  // which schedule ran
    a.phase_ns[14] = gridDim.x;
  }

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
      routing_phase(c, lv, a.logits[0], R, st, blockIdx.x == 0, blockIdx.x == 0);
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
        routing_phase(c, lv, a.logits[(s + 1) & 1], c.route((s + 1) & 3), false, true, true);
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

// ---------------------------------------------------------------- dataflow stack
// moe_stack_forward: the stack as one sequence of small work items, handed
// out round-robin (item i to CTA i % G, each CTA in increasing order), with
// per-layer counters instead of grid barriers.  Item kinds of layer l:
//   R   8 router rows (one warp each), part of q8_K(x_l)       -> logits_l
//   Q   top-k, bucketing, tile plan                            -> route_l
//   GU  (tile, gpi 32-row groups) of gate and up, SwiGLU       -> h_l
//   D   (tile, 8 dpi row groups) of down, on q8_K(h) of the tile -> y_l by slot
//   C   a chunk of out_l = residual + sum gate * y (fixed order)
// An item waits (bounded) for the counters of what it reads: Q for all R of
// its layer, GU for Q, D for the GU items of its tile, C for all D; in a
// chained stack the R items of layer l also wait for all C of layer l-1.
// In a chained stack the CTA that finishes the last R item of a layer runs
// its Q at once, and the one that finishes the last D item runs all of its C
// (the Q and C items of the sequence are then empty): two fewer hand-offs
// on the critical path of a layer.
// Every item increments its counter, also when it has nothing to do (a
// tile slot beyond the layer's tiles), so the targets are fixed counts; the
// counters are zeroed at the start of the launch (one grid barrier).  Waits
// point only at earlier items, and each CTA takes its items in order, so
// every wait ends.
// Item order: a stack whose layers neither read nor write each other's
// buffers runs stage by stage, stage s holding R of layer s, Q of s-2, GU of
// s-4, D of s-6 and C of s-8 (two stages of slack between an item and what
// it waits for), so several layers overlap with no grid barrier; otherwise
// layer by layer.  Each layer owns its buffers, so no
// layer's data is overwritten while another still reads it.
// Counters are incremented with a release pattern (barrier, acq_rel fence,
// relaxed add) and read with ld.acquire.  Where shared memory allows
// (kRing), each warp streams its gate/up and down super-block rows through
// a two-stage cp.async ring and the item's small reads are issued ahead of
// that stream; otherwise the rows are loaded into registers and thread 32
// prefetches the CTA's next item towards L2 while thread 0 waits.
constexpr int kCombineVec = 1024;       // float4 elements per C item
// A CTA of nw warps: nw router rows per R item (one per warp); nw * dpi row
// groups per D item (dpi per warp).

__device__ __forceinline__ unsigned long long* stk_cnt(const DecodeArgs& a, int l, int j) {
  return reinterpret_cast<unsigned long long*>(a.stk + a.sp.cnt) + (size_t)l * a.sp.n_cnt + j;
}
__device__ __forceinline__ uint8_t* stk_layer(const DecodeArgs& a, int l) {
  return a.stk + a.sp.layer0 + (size_t)l * a.sp.layer_bytes;
}

__device__ __forceinline__ Route stk_route(const DecodeArgs& a, int l) {
  return route_at(stk_layer(a, l) + a.sp.route, a.T, a.k, a.S);
}
__device__ __forceinline__ Tile ld_tile(const Tile* p) {
  const int4 v = __ldcg(reinterpret_cast<const int4*>(p));
  Tile t;
  t.expert = v.x;
  t.start = v.y;
  t.count = v.z;
  t.flag = v.w;
  return t;
}

__device__ __forceinline__ moe_expert_ptrs ld_ptrs(const moe_expert_ptrs* p) {
  const unsigned long long* q = reinterpret_cast<const unsigned long long*>(p);
  moe_expert_ptrs e;
  e.gate = reinterpret_cast<const void*>(__ldcg(q));
  e.up = reinterpret_cast<const void*>(__ldcg(q + 1));
  e.down = reinterpret_cast<const void*>(__ldcg(q + 2));
  return e;
}

// Thread 0 waits (bounded) until *p >= target; every thread gets the answer.
// Data behind the counter is then read through L2 (ld.global.cg).
// While thread 0 polls, thread 32 runs `side` (the next item's L2 prefetch).
template <typename Side>
__device__ bool wait_count(const unsigned long long* p, unsigned long long target, int* status, Side side) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 32) side();
  if (threadIdx.x == 0) {
    int ok = 1;
    long long spins = 0;
    while (ld_acquire_u64(p) < target) {
      if (++spins > kSpinLimit) {
        set_status(status, MOE_ERR_DEVICE_TIMEOUT);
        ok = 0;
        break;
      }
      __nanosleep(32);
    }
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}
// All of this CTA's writes of the item are done: count the item.  A release
// pattern (acq_rel fence, then a relaxed add; the barrier orders the other
// threads' writes before the fence), lighter than a sequentially consistent
// fence before the add; waiters read the counter with ld.acquire.
__device__ __forceinline__ void release_add(unsigned long long* p, unsigned long long v) {
  asm volatile("fence.acq_rel.gpu;\n red.relaxed.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ void signal_count(unsigned long long* p) {
  __syncthreads();
  if (threadIdx.x == 0) release_add(p, 1ull);
}

// The same, and tells every thread whether this item was the one that
// brought the counter to `target` (then the items counted before it are all
// visible to this CTA).
__device__ bool signal_last(unsigned long long* p, unsigned long long target) {
  __shared__ int s_last;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long old;
    asm volatile("fence.acq_rel.gpu;\n atom.relaxed.gpu.global.add.u64 %0, [%1], 1;\n fence.acq_rel.gpu;"
                 : "=l"(old)
                 : "l"(p)
                 : "memory");
    s_last = old + 1 == target;
  }
  __syncthreads();
  return s_last != 0;
}

// The item sequence of one launch.
struct StackSeq {
  int L, nR, nGU, nD, nC, per_stage, n_stages;
  int gpi, grp_g;  // gate/up: row groups per item, items per tile
  int dpi, grp_d;  // down: row groups per warp (nw dpi per item), items per tile
  bool overlap;
  enum { kR = 0, kQ = 1, kGU = 2, kD = 3, kC = 4 };
  static constexpr int kLag = 2;  // stages between an item kind and the kind it waits for (overlapped order)
  // item i -> (kind, layer, index within the layer's items of that kind); layer < 0 or >= L: none
  __device__ void item(long long i, int& kind, int& l, int& idx) const {
    const int s = (int)(i / per_stage);
    int j = (int)(i % per_stage);
    if (j < nR) { kind = kR; idx = j; l = s; return; }
    j -= nR;
    if (j < 1) { kind = kQ; idx = 0; l = overlap ? s - kLag : s; return; }
    j -= 1;
    if (j < nGU) { kind = kGU; idx = j; l = overlap ? s - 2 * kLag : s; return; }
    j -= nGU;
    if (j < nD) { kind = kD; idx = j; l = overlap ? s - 3 * kLag : s; return; }
    j -= nD;
    kind = kC; idx = j; l = overlap ? s - 4 * kLag : s;
  }
  __device__ long long count() const { return (long long)n_stages * per_stage; }
};

// Do the layers share no buffer except a layer's residual with its own out?
// (x, residual, out of every layer against out of every other layer.)
__device__ bool stack_disjoint(const DecodeArgs& a, int L) {
  __shared__ int s_clash;
  if (threadIdx.x == 0) s_clash = 0;
  __syncthreads();
  const size_t bytes = (size_t)a.T * a.H * sizeof(float);
  auto hit = [&](const void* p, const void* q) {
    const char* x = static_cast<const char*>(p);
    const char* o = static_cast<const char*>(q);
    return x && o && x < o + bytes && o < x + bytes;
  };
  int clash = 0;
  for (int pq = threadIdx.x; pq < L * L; pq += blockDim.x) {
    const int i = pq / L, j = pq % L;
    if (i == j) continue;
    const moe_layer_ptrs li = a.layers[i], lj = a.layers[j];
    if (hit(li.out, lj.x) || hit(li.out, lj.residual) || hit(li.out, lj.out)) clash = 1;
  }
  if (clash) atomicOr(&s_clash, 1);
  __syncthreads();
  return s_clash == 0;
}

// L2 prefetch of the weights item i will read (when already known)
template <int FMT>
__device__ void stack_prefetch(const Ctx<FMT>& c, const StackSeq& q, long long i, unsigned long long ep1) {
  if (i >= q.count()) return;
  const DecodeArgs& a = c.a;
  int kind, l, idx;
  q.item(i, kind, l, idx);
  if (l < 0 || l >= q.L) return;
  const LayerView lv = layer_view(a, l);
  if (kind == StackSeq::kR) {
    const int e0 = idx * c.nw, n = min(c.nw, c.E - e0);
    if (n > 0) prefetch_l2(lv.w_router + (size_t)e0 * c.H, (uint32_t)((size_t)n * c.H * 4));
    return;
  }
  if (kind != StackSeq::kGU && kind != StackSeq::kD) return;
  if (ld_acquire_u64(stk_cnt(a, l, 1)) < ep1) return;  // routing not published yet
  const Route Rg = stk_route(a, l);
  const int per = kind == StackSeq::kGU ? q.grp_g : q.grp_d;
  const int ti = idx / per;
  const int nt = __ldcg(Rg.n_tiles);
  const Tile tl = ld_tile(Rg.tiles + ti);
  const moe_expert_ptrs ep = ld_ptrs(reinterpret_cast<const moe_expert_ptrs*>(stk_layer(a, l) + a.sp.tptr) + ti);
  if (ti >= nt || tl.flag) return;
  if (kind == StackSeq::kGU) {
    const int rg0 = (idx % per) * q.gpi, nrg = min(q.gpi, c.nRG - rg0);
    const size_t off = (size_t)rg0 * c.gu_run;
    prefetch_l2(static_cast<const uint8_t*>(ep.gate) + off, (uint32_t)(nrg * c.gu_run));
    prefetch_l2(static_cast<const uint8_t*>(ep.up) + off, (uint32_t)(nrg * c.gu_run));
  } else {
    const int rg0 = (idx % per) * c.nw * q.dpi, nrg = min(c.nw * q.dpi, c.nRGH - rg0);
    prefetch_l2(static_cast<const uint8_t*>(ep.down) + (size_t)rg0 * c.dn_rg_bytes,
                (uint32_t)((size_t)nrg * c.dn_rg_bytes));
  }
}

// R: router rows [nw idx, nw idx + nw) of layer l, one warp per row
// (The router items also make the q8_K of x: block qb by warp qb % 8 of item
// (qb / 8) % nR, so it is done when all router items of the layer are.)
template <int FMT>
__device__ void stack_router_item(Ctx<FMT>& c, const LayerView& lv, int l, int idx, int nR) {
  const int T = c.T, H = c.H, E = c.E, lane = c.lane, H4 = H / 4;
  uint8_t* lb = stk_layer(c.a, l);
  for (int qb = idx * c.nw + c.warp; qb < T * c.nbH; qb += nR * c.nw) {
    const float4* src = reinterpret_cast<const float4*>(lv.x + (size_t)qb * 256 + 8 * lane);
    const float4 v0 = __ldcg(src), v1 = __ldcg(src + 1);
    const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    q8k_block_warp(v, lane, reinterpret_cast<int8_t*>(lb + c.a.sp.xq) + (size_t)qb * 256,
                   reinterpret_cast<float*>(lb + c.a.sp.xd) + qb,
                   reinterpret_cast<int16_t*>(lb + c.a.sp.xbs) + (size_t)qb * 16);
  }
  float* logits = reinterpret_cast<float*>(lb + c.a.sp.logits);
  const int e = idx * c.nw + c.warp;
  if (e >= E) return;
  const float4* wr = reinterpret_cast<const float4*>(lv.w_router + (size_t)e * H);
  const float4* xr = reinterpret_cast<const float4*>(lv.x);
  float acc[16];
#pragma unroll
  for (int t = 0; t < 16; ++t) acc[t] = 0.0f;
  // 8 chunks of the row in flight at a time (chunks past the row end read as zero)
  const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int h0 = lane; h0 < H4; h0 += 32 * 8) {
    float4 wv[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) wv[u] = h0 + 32 * u < H4 ? __ldg(wr + h0 + 32 * u) : z4;
#pragma unroll
    for (int t = 0; t < 16; ++t)
      if (t < T) {
        float4 xv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)  // x may be a previous layer's output
          xv[u] = h0 + 32 * u < H4 ? __ldcg(xr + (size_t)t * H4 + h0 + 32 * u) : z4;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          acc[t] = fmaf(wv[u].x, xv[u].x, acc[t]);
          acc[t] = fmaf(wv[u].y, xv[u].y, acc[t]);
          acc[t] = fmaf(wv[u].z, xv[u].z, acc[t]);
          acc[t] = fmaf(wv[u].w, xv[u].w, acc[t]);
        }
      }
  }
  const float be = lv.bias ? __ldg(lv.bias + e) : 0.0f;
#pragma unroll
  for (int t = 0; t < 16; ++t) {
    if (t < T) {
      float v = acc[t];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) logits[(size_t)t * E + e] = v + be;
    }
  }
}

// Routing of a stack layer without the expert-wide count and scan: with at
// most 256 (token, slot) pairs, a pair's bucket position is the number of
// pairs of smaller experts plus the earlier pairs of its own expert, and an
// expert's tile index is the number of distinct smaller experts.  Same
// result as routing_phase (tiles by expert, shared experts last), without
// writing the layer's counts and offsets to global memory.
template <int FMT>
__device__ void routing_small(Ctx<FMT>& c, const LayerView& lv, const float* logits, const Route& R,
                              moe_expert_ptrs* tptr) {
  const DecodeArgs& a = c.a;
  const int T = c.T, E = c.E, k = c.k, S = c.S, tid = c.tid, TK = T * k;
  int* first = reinterpret_cast<int*>(c.sm.red);  // [TK]: pair is its expert's first
  // [TK + S]: each pair's expert pointer record (one read of the table
  // serves the presence test here and the published tile pointers)
  moe_expert_ptrs* rec = reinterpret_cast<moe_expert_ptrs*>(c.sm.red + 256);
  for (int t = c.warp; t < T; t += c.nw)
    warp_topk(logits + (size_t)t * E, E, k, a.route, c.lane, R.ids + t * k, R.gates + t * k, nullptr);
  __syncthreads();
  for (int p = tid; p < TK + S; p += c.nt) {
    const int e = p < TK ? R.ids[p] : E + (p - TK);
    rec[p] = lv.table[e];
    R.ok[p] = rec[p].gate != nullptr ? 1 : 0;  // present ("mine")?
  }
  for (int p = tid; p < TK; p += c.nt) {
    const int e = R.ids[p];
    int f = 1;
    for (int q = 0; q < p; ++q) f &= R.ids[q] != e;
    first[p] = f;
  }
  __syncthreads();
  for (int p = tid; p < TK; p += c.nt) {
    const int e = R.ids[p];
    int before = 0, same_before = 0, cnt = 0, tix = 0;
    for (int q = 0; q < TK; ++q) {
      const int f = R.ids[q];
      before += f < e;
      same_before += (f == e) & (q < p);
      cnt += f == e;
      tix += (f < e) & first[q];
    }
    const int pos = before + same_before;
    R.tok[pos] = p / k;
    R.slot[pos] = p;
    if (first[p]) {
      Tile tl;
      tl.expert = e;
      tl.start = before;
      tl.count = cnt;
      tl.flag = R.ok[p] ? 0 : 1;
      R.tiles[tix] = tl;
      if (tptr) tptr[tix] = rec[p];
    }
  }
  __shared__ int s_distinct;
  if (tid == 0) {
    int n = 0;
    for (int q = 0; q < TK; ++q) n += first[q];
    s_distinct = n;
  }
  __syncthreads();
  const int nr = s_distinct;
  for (int i = tid; i < S * T; i += c.nt) {
    const int sh = i / T, t = i % T, pos = TK + sh * T + t;
    R.tok[pos] = t;
    R.slot[pos] = pos;
    if (t == 0) {
      Tile tl;
      tl.expert = E + sh;
      tl.start = TK + sh * T;
      tl.count = T;
      tl.flag = R.ok[TK + sh] ? 0 : 1;
      R.tiles[nr + sh] = tl;
      if (tptr) tptr[nr + sh] = rec[TK + sh];
    }
  }
  if (tid == 0) *R.n_tiles = nr + S;
  for (int p = tid; p < TK; p += c.nt) {
    if (lv.ids_out) lv.ids_out[p] = R.ids[p];
    if (lv.gates_out) lv.gates_out[p] = R.gates[p];
  }
  __syncthreads();
}

// Q: top-k, bucketing and tile plan of layer l, published to route_l
template <int FMT>
__device__ void stack_routing_item(Ctx<FMT>& c, const LayerView& lv, int l, bool last) {
  const DecodeArgs& a = c.a;
  uint8_t* lb = stk_layer(a, l);
  const Route R = c.route(0);
  // each tile's weight pointers beside the tiles: a consumer reads tile and
  // pointers in one round trip (routing_small writes them as it plans)
  moe_expert_ptrs* tp = reinterpret_cast<moe_expert_ptrs*>(lb + a.sp.tptr);
  // the last layer also fills the workspace's counts/offsets/perm: the general routine
  const bool general = last || c.T * c.k > c.nt;
  if (general)
    routing_phase(c, lv, reinterpret_cast<const float*>(lb + a.sp.logits), R, false, last, true);
  else
    routing_small(c, lv, reinterpret_cast<const float*>(lb + a.sp.logits), R, tp);
  __syncthreads();
  const int4* src = reinterpret_cast<const int4*>(c.sm.rbase);
  int4* dst = reinterpret_cast<int4*>(lb + a.sp.route);
  for (size_t i = c.tid; i < c.sm.rstride / 16; i += c.nt) dst[i] = src[i];
  if (general)
    for (int t = c.tid; t < *R.n_tiles; t += c.nt) tp[t] = lv.table[R.tiles[t].expert];
}


// GU: (tile idx / grp_g, row groups gpi (idx % grp_g) ..) of gate and up;
// h = silu(G) * U.  The 8 warps take the (row group, super-block) pairs in
// turn.  staged_x: the layer whose q8_K(x) is in shared memory (-1: none).
template <int FMT>
__device__ void stack_gateup_item(Ctx<FMT>& c, const LayerView& lv, int l, int idx, int gpi, int grp_g,
                                  int& staged_x) {
  using F = Fmt<FMT>;
  const DecodeArgs& a = c.a;
  const int T = c.T, H = c.H, I = c.I, nbH = c.nbH, lane = c.lane, warp = c.warp, tid = c.tid;
  Smem& sm = c.sm;
  uint8_t* lb = stk_layer(a, l);
  const Route Rg = stk_route(a, l);
  const int ti = idx / grp_g, rg0 = (idx % grp_g) * gpi;
  const int nrg = min(gpi, c.nRG - rg0);
  // tile count, tile and its weight pointers: independent loads, one round trip
  const int nt = __ldcg(Rg.n_tiles);
  const Tile tl = ld_tile(Rg.tiles + ti);
  const moe_expert_ptrs ep = ld_ptrs(reinterpret_cast<const moe_expert_ptrs*>(lb + a.sp.tptr) + ti);
  if (ti >= nt || tl.flag) return;
  const uint8_t* gbase = static_cast<const uint8_t*>(ep.gate) + (size_t)rg0 * c.gu_run;
  const uint8_t* ubase = static_cast<const uint8_t*>(ep.up) + (size_t)rg0 * c.gu_run;
  const int npair = nrg * nbH;  // (row group, super-block) pairs; pair p = rgl * nbH + b
  // this warp's first pair is in flight while x is staged
  SbRegs<FMT> sg, su;
  if (warp < npair) {
    load_sb<FMT>(gbase + (size_t)warp * F::kSlabBytes, lane, sg);
    load_sb<FMT>(ubase + (size_t)warp * F::kSlabBytes, lane, su);
  }
  if (staged_x != l) {
    const int8_t* xq = reinterpret_cast<const int8_t*>(lb + a.sp.xq);
    const int16_t* xbs = reinterpret_cast<const int16_t*>(lb + a.sp.xbs);
    const float* xd = reinterpret_cast<const float*>(lb + a.sp.xd);
    for (int i = tid; i < T * H / 16; i += c.nt)
      reinterpret_cast<int4*>(sm.xq)[i] = __ldcg(reinterpret_cast<const int4*>(xq) + i);
    for (int i = tid; i < T * H / 128; i += c.nt)
      reinterpret_cast<int4*>(sm.xbs)[i] = __ldcg(reinterpret_cast<const int4*>(xbs) + i);
    for (int i = tid; i < T * nbH; i += c.nt) sm.xd[i] = __ldcg(xd + i);
    staged_x = l;
  }
  for (int t = tid; t < tl.count; t += c.nt) sm.aoff[t] = __ldcg(Rg.tok + tl.start + t) * H;
  // per-warp accumulators: [row group][gate, up][T][32]
  float* accw = sm.red + (size_t)warp * gpi * 2 * T * 32;
  for (int i = lane; i < gpi * 2 * T * 32; i += 32) accw[i] = 0.0f;
  __syncthreads();
  for (int p = warp; p < npair; p += c.nw) {
    // slabs of consecutive row groups are consecutive: pair p's slab is p slabs from the base
    if (p != warp) {
      load_sb<FMT>(gbase + (size_t)p * F::kSlabBytes, lane, sg);
      load_sb<FMT>(ubase + (size_t)p * F::kSlabBytes, lane, su);
    }
    const int rgl = p / nbH, b = p % nbH;
    float* acc = accw + (size_t)rgl * 2 * T * 32;
    sb_accum<FMT>(sg, sm.xq, sm.xbs, sm.xd, sm.aoff, b, tl.count, acc, lane);
    sb_accum<FMT>(su, sm.xq, sm.xbs, sm.xd, sm.aoff, b, tl.count, acc + T * 32, lane);
  }
  __syncthreads();
  float* h = reinterpret_cast<float*>(lb + a.sp.h);
  for (int i = tid; i < nrg * tl.count * 32; i += c.nt) {
    const int r = i & 31, t = (i >> 5) % tl.count, rgl = (i >> 5) / tl.count;
    float Gv = 0.0f, Uv = 0.0f;
#pragma unroll
    for (int w = 0; w < c.nw; ++w) {
      const float* acc = sm.red + ((size_t)w * gpi + rgl) * 2 * T * 32;
      Gv += acc[t * 32 + r];
      Uv += acc[(T + t) * 32 + r];
    }
    h[(size_t)(tl.start + t) * I + (rg0 + rgl) * 32 + r] = Gv / (1.0f + expf(-Gv)) * Uv;
  }
}

// D: (tile idx / grp_d, 8 dpi row groups) of down on q8_K(h); warp w owns row
// groups w, w + 8, .. of the item; y by slot
template <int FMT>
__device__ void stack_down_item(Ctx<FMT>& c, const LayerView& lv, int l, int idx, int dpi, int grp_d) {
  using F = Fmt<FMT>;
  const DecodeArgs& a = c.a;
  const int T = c.T, H = c.H, I = c.I, nbI = c.nbI, lane = c.lane, warp = c.warp, tid = c.tid;
  Smem& sm = c.sm;
  uint8_t* lb = stk_layer(a, l);
  const Route Rg = stk_route(a, l);
  const int ti = idx / grp_d, rgi = (idx % grp_d) * c.nw * dpi;
  const int nt = __ldcg(Rg.n_tiles);
  const Tile tl = ld_tile(Rg.tiles + ti);
  const void* dn = reinterpret_cast<const void*>(
      __ldcg(reinterpret_cast<const unsigned long long*>(lb + a.sp.tptr) + 3 * ti + 2));
  if (ti >= nt || tl.flag) return;
  const uint8_t* dbase = static_cast<const uint8_t*>(dn);
  SbRegs<FMT> sd;
  if (rgi + warp < c.nRGH) load_sb<FMT>(dbase + (size_t)(rgi + warp) * c.dn_rg_bytes, lane, sd);  // in flight
  const float* h = reinterpret_cast<const float*>(lb + a.sp.h);
  for (int task = warp; task < tl.count * nbI; task += c.nw) {
    const int t = task / nbI, blk = task % nbI;
    const float4* src = reinterpret_cast<const float4*>(h + (size_t)(tl.start + t) * I + blk * 256 + 8 * lane);
    const float4 v0 = __ldcg(src), v1 = __ldcg(src + 1);
    const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    q8k_block_warp(v, lane, sm.hq + (size_t)t * I + blk * 256, sm.hd + t * nbI + blk,
                   sm.hbs + (size_t)t * (I / 16) + blk * 16);
  }
  for (int t = tid; t < tl.count; t += c.nt) sm.aoff[t] = t * I;
  float* accw = sm.red + (size_t)warp * dpi * T * 32;  // [dpi][T][32]
  for (int i = lane; i < dpi * T * 32; i += 32) accw[i] = 0.0f;
  __syncthreads();
  float* y = reinterpret_cast<float*>(lb + a.sp.y);
  for (int j = 0; j < dpi; ++j) {
    const int rg = rgi + j * c.nw + warp;
    if (rg >= c.nRGH) break;
    const uint8_t* rbase = dbase + (size_t)rg * c.dn_rg_bytes;
    float* acc = accw + (size_t)j * T * 32;
    for (int b = 0; b < nbI; ++b) {
      if (b > 0 || j > 0) load_sb<FMT>(rbase + (size_t)b * F::kSlabBytes, lane, sd);
      sb_accum<FMT>(sd, sm.hq, sm.hbs, sm.hd, sm.aoff, b, tl.count, acc, lane);
    }
    __syncwarp();
    for (int t = 0; t < tl.count; ++t)
      y[(size_t)__ldcg(Rg.slot + tl.start + t) * H + rg * 32 + lane] = acc[t * 32 + lane];
  }
}

__host__ __device__ inline size_t ring_offset(size_t decode_bytes) { return (decode_bytes + 127) / 128 * 128; }

// sb_accum on a staged slab: the same sums in the same order, with the code
// lines read from shared memory per token instead of held in registers
template <int FMT>
__device__ __forceinline__ void sb_accum_staged(const uint8_t* slab, const int8_t* act, const int16_t* bs,
                                                const float* d, const int* act_off, int b, int cnt, float* acc,
                                                int lane) {
  using F = Fmt<FMT>;
  if constexpr (FMT != kQ4K && FMT != kQ2K) {
    SbRegs<FMT> h;
    load_sb_head<FMT>(slab, lane, h);
    const uint8_t* code = slab + F::kCodeOff + 16 * lane;
    sb_accum_words<FMT>([&](int l) { return *reinterpret_cast<const uint4*>(code + 512 * l); }, h, act, bs, d,
                        act_off, b, cnt, acc, lane);
  } else {
  SbRegs<FMT> s;  // scale/min words and d|dmin only
  s.dm = *reinterpret_cast<const uint32_t*>(slab + 4 * lane);
  if constexpr (FMT == kQ4K) {
#pragma unroll
    for (int i = 0; i < 3; ++i) s.sm[i] = *reinterpret_cast<const uint32_t*>(slab + F::kSmOff + 12 * lane + 4 * i);
  } else {
    const uint4 v = *reinterpret_cast<const uint4*>(slab + F::kSmOff + 16 * lane);
    s.sm[0] = v.x; s.sm[1] = v.y; s.sm[2] = v.z; s.sm[3] = v.w;
  }
  int sc[F::kNSub], mn[F::kNSub];
#pragma unroll
  for (int j = 0; j < F::kNSub; ++j) sb_scale_min<FMT>(s, j, sc[j], mn[j]);
  const float dw = half_lo(s.dm), dmin = half_hi(s.dm);
  const uint8_t* code = slab + F::kCodeOff + 16 * lane;
#pragma unroll 1
  for (int t = 0; t < cnt; ++t) {
    const int o = act_off[t];
    const int8_t* a = act + o + 256 * b;
    const int16_t* bsp = bs + o / 16 + 16 * b;
    int S = 0, M = 0;
    if constexpr (FMT == kQ4K) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint32_t lo[4], hi[4];
        mask_q4k(*reinterpret_cast<const uint4*>(code + 512 * j), lo, hi);
        S += sc[j] * isum_q4k(lo, hi, *reinterpret_cast<const int4*>(a + 32 * j),
                              *reinterpret_cast<const int4*>(a + 32 * j + 16));
        M += mn[j] * ((int)bsp[2 * j] + (int)bsp[2 * j + 1]);
      }
    } else {
#pragma unroll
      for (int ln = 0; ln < 4; ++ln) {
        const uint4 line = *reinterpret_cast<const uint4*>(code + 512 * ln);
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int j = 4 * ln + jj;
          uint32_t w[4];
          mask_q2k(line, j, w);
          S += sc[j] * isum_q2k(w, *reinterpret_cast<const int4*>(a + 16 * j));
          M += mn[j] * (int)bsp[j];
        }
      }
    }
    acc[t * 32 + lane] += d[o / 256 + b] * fmaf(dw, (float)S, -dmin * (float)M);
  }
  }
}

// sb_accum_staged of the gate and the up slab of one pair at once: the same
// sums in the same order per matrix, with each token's activation words and
// 16-sums read once for both
template <int FMT>
__device__ __forceinline__ void sb_accum_pair_staged(const uint8_t* sg, const uint8_t* su, const int8_t* act,
                                                     const int16_t* bs, const float* d, const int* act_off, int b,
                                                     int cnt, float* accg, float* accu, int lane) {
  using F = Fmt<FMT>;
  if constexpr (FMT != kQ4K && FMT != kQ2K) {  // one matrix at a time
    sb_accum_staged<FMT>(sg, act, bs, d, act_off, b, cnt, accg, lane);
    sb_accum_staged<FMT>(su, act, bs, d, act_off, b, cnt, accu, lane);
  } else {
  SbRegs<FMT> g, u;  // scale/min words and d|dmin only
  g.dm = *reinterpret_cast<const uint32_t*>(sg + 4 * lane);
  u.dm = *reinterpret_cast<const uint32_t*>(su + 4 * lane);
  if constexpr (FMT == kQ4K) {
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      g.sm[i] = *reinterpret_cast<const uint32_t*>(sg + F::kSmOff + 12 * lane + 4 * i);
      u.sm[i] = *reinterpret_cast<const uint32_t*>(su + F::kSmOff + 12 * lane + 4 * i);
    }
  } else {
    const uint4 vg = *reinterpret_cast<const uint4*>(sg + F::kSmOff + 16 * lane);
    const uint4 vu = *reinterpret_cast<const uint4*>(su + F::kSmOff + 16 * lane);
    g.sm[0] = vg.x; g.sm[1] = vg.y; g.sm[2] = vg.z; g.sm[3] = vg.w;
    u.sm[0] = vu.x; u.sm[1] = vu.y; u.sm[2] = vu.z; u.sm[3] = vu.w;
  }
  int scg[F::kNSub], mng[F::kNSub], scu[F::kNSub], mnu[F::kNSub];
#pragma unroll
  for (int j = 0; j < F::kNSub; ++j) {
    sb_scale_min<FMT>(g, j, scg[j], mng[j]);
    sb_scale_min<FMT>(u, j, scu[j], mnu[j]);
  }
  const float dwg = half_lo(g.dm), dming = half_hi(g.dm), dwu = half_lo(u.dm), dminu = half_hi(u.dm);
  const uint8_t* cg = sg + F::kCodeOff + 16 * lane;
  const uint8_t* cu = su + F::kCodeOff + 16 * lane;
#pragma unroll 1
  for (int t = 0; t < cnt; ++t) {
    const int o = act_off[t];
    const int8_t* a = act + o + 256 * b;
    const int16_t* bsp = bs + o / 16 + 16 * b;
    int Sg = 0, Mg = 0, Su = 0, Mu = 0;
    if constexpr (FMT == kQ4K) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int4 alo = *reinterpret_cast<const int4*>(a + 32 * j);
        const int4 ahi = *reinterpret_cast<const int4*>(a + 32 * j + 16);
        const int bsum = (int)bsp[2 * j] + (int)bsp[2 * j + 1];
        uint32_t lo[4], hi[4];
        mask_q4k(*reinterpret_cast<const uint4*>(cg + 512 * j), lo, hi);
        Sg += scg[j] * isum_q4k(lo, hi, alo, ahi);
        Mg += mng[j] * bsum;
        mask_q4k(*reinterpret_cast<const uint4*>(cu + 512 * j), lo, hi);
        Su += scu[j] * isum_q4k(lo, hi, alo, ahi);
        Mu += mnu[j] * bsum;
      }
    } else {
#pragma unroll
      for (int ln = 0; ln < 4; ++ln) {
        const uint4 lg = *reinterpret_cast<const uint4*>(cg + 512 * ln);
        const uint4 lu = *reinterpret_cast<const uint4*>(cu + 512 * ln);
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int j = 4 * ln + jj;
          const int4 av = *reinterpret_cast<const int4*>(a + 16 * j);
          const int bsum = (int)bsp[j];
          uint32_t w[4];
          mask_q2k(lg, j, w);
          Sg += scg[j] * isum_q2k(w, av);
          Mg += mng[j] * bsum;
          mask_q2k(lu, j, w);
          Su += scu[j] * isum_q2k(w, av);
          Mu += mnu[j] * bsum;
        }
      }
    }
    const float da = d[o / 256 + b];
    accg[t * 32 + lane] += da * fmaf(dwg, (float)Sg, -dming * (float)Mg);
    accu[t * 32 + lane] += da * fmaf(dwu, (float)Su, -dminu * (float)Mu);
  }
  }
}

// ---- staged gate/up and down items -------------------------------------------
// Each warp streams its super-block rows of the item through its own ring of
// two shared-memory stages with cp.async (16 bytes per lane per
// instruction, one commit group per unit of up to two slabs), so a warp's
// next unit is in flight while it computes the current one and no
// registers hold weights.  cp.async streams at the load path's rate (a
// bulk copy per unit would not).
constexpr int kRingStages = 2;

template <int FMT>
__host__ __device__ inline uint32_t ring_unit_bytes() { return 2u * Fmt<FMT>::kSlabBytes; }

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

template <int FMT>
struct WarpRing {
  uint8_t* base;        // kRingStages stages of ring_unit_bytes
  uint32_t issued, taken;
  int lane;
  // n0 bytes at s0, then n1 at s1, into the next stage (sizes multiples of 16)
  __device__ void issue(const uint8_t* s0, uint32_t n0, const uint8_t* s1, uint32_t n1) {
    const uint32_t d = static_cast<uint32_t>(
        __cvta_generic_to_shared(base + (size_t)(issued % kRingStages) * ring_unit_bytes<FMT>()));
    for (uint32_t off = 16u * lane; off < n0; off += 512u) cp_async16(d + off, s0 + off);
    for (uint32_t off = 16u * lane; off < n1; off += 512u) cp_async16(d + n0 + off, s1 + off);
    asm volatile("cp.async.commit_group;" ::: "memory");
    ++issued;
  }
  // the oldest unit not yet taken, once this warp's copies of it landed
  // (at most kRingStages = 2 units are issued and not taken)
  static_assert(kRingStages == 2, "take() waits with wait_group 1 / 0");
  __device__ const uint8_t* take() {
    if (issued - taken > 1) asm volatile("cp.async.wait_group 1;" ::: "memory");
    else asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncwarp();
    return base + (size_t)(taken % kRingStages) * ring_unit_bytes<FMT>();
  }
  __device__ void give() {
    __syncwarp();
    ++taken;
  }
};

// GU with the ring: the same item as stack_gateup_item; unit j of warp w =
// the gate and up slabs of pair w + 8 j
template <int FMT>
__device__ void stack_gateup_ring(Ctx<FMT>& c, const LayerView& lv, int l, int idx, int gpi, int grp_g,
                                  int& staged_x, WarpRing<FMT>& rg) {
  using F = Fmt<FMT>;
  const DecodeArgs& a = c.a;
  const int T = c.T, H = c.H, I = c.I, nbH = c.nbH, lane = c.lane, warp = c.warp, tid = c.tid;
  Smem& sm = c.sm;
  uint8_t* lb = stk_layer(a, l);
  const Route Rg = stk_route(a, l);
  const int ti = idx / grp_g, rg0 = (idx % grp_g) * gpi;
  const int nrg = min(gpi, c.nRG - rg0);
  const int nt = __ldcg(Rg.n_tiles);
  const Tile tl = ld_tile(Rg.tiles + ti);
  const moe_expert_ptrs ep = ld_ptrs(reinterpret_cast<const moe_expert_ptrs*>(lb + a.sp.tptr) + ti);
  if (ti >= nt || tl.flag) return;
  const uint8_t* gbase = static_cast<const uint8_t*>(ep.gate) + (size_t)rg0 * c.gu_run;
  const uint8_t* ubase = static_cast<const uint8_t*>(ep.up) + (size_t)rg0 * c.gu_run;
  const int npair = nrg * nbH;
  const int nu = warp < npair ? (npair - warp + c.nw - 1) / c.nw : 0;
  auto issue = [&](int j) {
    const size_t off = (size_t)(warp + c.nw * j) * F::kSlabBytes;
    rg.issue(gbase + off, F::kSlabBytes, ubase + off, F::kSlabBytes);
  };
  // the small reads first (they would otherwise queue behind the weight
  // stream): q8_K(x) of the layer as one copy group, the tile's tokens
  const bool stage = staged_x != l;
  if (stage) {
    const uint8_t* xq = lb + a.sp.xq;
    const uint8_t* xbs = lb + a.sp.xbs;
    const uint8_t* xd = lb + a.sp.xd;
    const uint32_t dq = static_cast<uint32_t>(__cvta_generic_to_shared(sm.xq));
    const uint32_t db = static_cast<uint32_t>(__cvta_generic_to_shared(sm.xbs));
    const uint32_t dd = static_cast<uint32_t>(__cvta_generic_to_shared(sm.xd));
    for (int i = tid; i < T * H / 16; i += c.nt) cp_async16(dq + 16 * i, xq + 16 * i);
    for (int i = tid; i < T * H / 128; i += c.nt) cp_async16(db + 16 * i, xbs + 16 * i);
    for (int i = tid; i < T * nbH; i += c.nt)
      asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dd + 4 * i), "l"(xd + 4 * i) : "memory");
    asm volatile("cp.async.commit_group;" ::: "memory");
    staged_x = l;
  }
  const int tok = tid < tl.count ? __ldcg(Rg.tok + tl.start + tid) : 0;  // tl.count <= 16
  for (int j = 0; j < nu && j < kRingStages; ++j) issue(j);
  float* accw = sm.red + (size_t)warp * gpi * 2 * T * 32;  // [row group][gate, up][T][32]
  for (int i = lane; i < gpi * 2 * T * 32; i += 32) accw[i] = 0.0f;
  if (stage) {  // the x group is done; the weight groups after it may still be in flight
    const int newer = min(nu, kRingStages);
    if (newer >= 2) asm volatile("cp.async.wait_group 2;" ::: "memory");
    else if (newer == 1) asm volatile("cp.async.wait_group 1;" ::: "memory");
    else asm volatile("cp.async.wait_group 0;" ::: "memory");
  }
  if (tid < tl.count) sm.aoff[tid] = tok * H;
  __syncthreads();
  for (int j = 0; j < nu; ++j) {
    const uint8_t* st = rg.take();
    const int p = warp + c.nw * j;
    const int rgl = p / nbH, b = p % nbH;
    float* acc = accw + (size_t)rgl * 2 * T * 32;
    sb_accum_pair_staged<FMT>(st, st + F::kSlabBytes, sm.xq, sm.xbs, sm.xd, sm.aoff, b, tl.count, acc,
                              acc + T * 32, lane);
    rg.give();
    if (j + kRingStages < nu) issue(j + kRingStages);
  }
  __syncthreads();
  float* h = reinterpret_cast<float*>(lb + a.sp.h);
  for (int i = tid; i < nrg * tl.count * 32; i += c.nt) {
    const int r = i & 31, t = (i >> 5) % tl.count, rgl = (i >> 5) / tl.count;
    float Gv = 0.0f, Uv = 0.0f;
#pragma unroll
    for (int w = 0; w < c.nw; ++w) {
      const float* acc = sm.red + ((size_t)w * gpi + rgl) * 2 * T * 32;
      Gv += acc[t * 32 + r];
      Uv += acc[(T + t) * 32 + r];
    }
    h[(size_t)(tl.start + t) * I + (rg0 + rgl) * 32 + r] = Gv / (1.0f + expf(-Gv)) * Uv;
  }
}

// D with the ring: the same item as stack_down_item; warp w's units are, for
// each of its row groups rgi + 8 j + w, the slab pairs (2v, 2v + 1)
template <int FMT>
__device__ void stack_down_ring(Ctx<FMT>& c, const LayerView& lv, int l, int idx, int dpi, int grp_d,
                                WarpRing<FMT>& rg) {
  using F = Fmt<FMT>;
  const DecodeArgs& a = c.a;
  const int T = c.T, H = c.H, I = c.I, nbI = c.nbI, lane = c.lane, warp = c.warp, tid = c.tid;
  Smem& sm = c.sm;
  uint8_t* lb = stk_layer(a, l);
  const Route Rg = stk_route(a, l);
  const int ti = idx / grp_d, rgi = (idx % grp_d) * c.nw * dpi;
  const int nt = __ldcg(Rg.n_tiles);
  const Tile tl = ld_tile(Rg.tiles + ti);
  const void* dn = reinterpret_cast<const void*>(
      __ldcg(reinterpret_cast<const unsigned long long*>(lb + a.sp.tptr) + 3 * ti + 2));
  if (ti >= nt || tl.flag) return;
  const uint8_t* dbase = static_cast<const uint8_t*>(dn);
  const int upr = (nbI + 1) / 2;
  int nj = 0;
  for (int j = 0; j < dpi; ++j) nj += rgi + j * c.nw + warp < c.nRGH;
  const int nu = nj * upr;
  auto issue = [&](int u) {
    const int j = u / upr, v = u % upr;
    rg.issue(dbase + (size_t)(rgi + j * c.nw + warp) * c.dn_rg_bytes + (size_t)(2 * v) * F::kSlabBytes,
             (uint32_t)min(2, nbI - 2 * v) * F::kSlabBytes, nullptr, 0);
  };
  // the warp's first block of h is read before the weight stream is issued
  // (small reads would otherwise queue behind it)
  const float* h = reinterpret_cast<const float*>(lb + a.sp.h);
  auto h_src = [&](int task) {
    const int t = task / nbI, blk = task % nbI;
    return reinterpret_cast<const float4*>(h + (size_t)(tl.start + t) * I + blk * 256 + 8 * lane);
  };
  float4 v0 = make_float4(0.f, 0.f, 0.f, 0.f), v1 = v0;
  if (warp < tl.count * nbI) {
    v0 = __ldcg(h_src(warp));
    v1 = __ldcg(h_src(warp) + 1);
  }
  const int slot = tid < tl.count ? __ldcg(Rg.slot + tl.start + tid) : 0;  // tl.count <= 16
  for (int u = 0; u < nu && u < kRingStages; ++u) issue(u);
  for (int task = warp; task < tl.count * nbI; task += c.nw) {
    const int t = task / nbI, blk = task % nbI;
    if (task != warp) {
      v0 = __ldcg(h_src(task));
      v1 = __ldcg(h_src(task) + 1);
    }
    const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    q8k_block_warp(v, lane, sm.hq + (size_t)t * I + blk * 256, sm.hd + t * nbI + blk,
                   sm.hbs + (size_t)t * (I / 16) + blk * 16);
  }
  for (int t = tid; t < tl.count; t += c.nt) sm.aoff[t] = t * I;
  int* srow = sm.srow;
  if (tid < tl.count) srow[tid] = slot;
  float* accw = sm.red + (size_t)warp * dpi * T * 32;  // [dpi][T][32]
  for (int i = lane; i < dpi * T * 32; i += 32) accw[i] = 0.0f;
  __syncthreads();
  float* y = reinterpret_cast<float*>(lb + a.sp.y);
  for (int j = 0; j < nj; ++j) {
    const int rgrow = rgi + j * c.nw + warp;
    float* acc = accw + (size_t)j * T * 32;
    for (int v = 0; v < upr; ++v) {
      const int u = j * upr + v;
      const uint8_t* st = rg.take();
      for (int bb = 0; bb < 2 && 2 * v + bb < nbI; ++bb)
        sb_accum_staged<FMT>(st + bb * F::kSlabBytes, sm.hq, sm.hbs, sm.hd, sm.aoff, 2 * v + bb, tl.count, acc,
                             lane);
      rg.give();
      if (u + kRingStages < nu) issue(u + kRingStages);
    }
    __syncwarp();
    for (int t = 0; t < tl.count; ++t) y[(size_t)srow[t] * H + rgrow * 32 + lane] = acc[t * 32 + lane];
  }
}

// C: float4 elements [1024 idx, 1024 idx + 1024) of out_l
template <int FMT>
__device__ void stack_combine_item(Ctx<FMT>& c, const LayerView& lv, int l, int idx) {
  const DecodeArgs& a = c.a;
  const int T = c.T, H4 = c.H / 4, k = c.k, S = c.S;
  uint8_t* lb = stk_layer(a, l);
  const Route Rg = stk_route(a, l);
  float* s_g = c.sm.red;                                     // gates [T*k]
  float* s_ok = c.sm.red + T * k;                            // presence [T*k + S]
  for (int i = c.tid; i < T * k; i += c.nt) s_g[i] = __ldcg(Rg.gates + i);
  for (int i = c.tid; i < T * k + S; i += c.nt) s_ok[i] = (float)__ldcg(Rg.ok + i);
  __syncthreads();
  const float4* y4 = reinterpret_cast<const float4*>(lb + a.sp.y);
  const int end = min(T * H4, (idx + 1) * kCombineVec);
  for (int e = idx * kCombineVec + c.tid; e < end; e += c.nt) {
    const int t = e / H4, cc = e % H4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < k; ++s) {
      if (s_ok[t * k + s] == 0.0f) continue;  // expert not present ("not mine"): contributes nothing
      const float g = s_g[t * k + s];
      const float4 v = __ldcg(y4 + (size_t)(t * k + s) * H4 + cc);
      acc.x = fmaf(g, v.x, acc.x);
      acc.y = fmaf(g, v.y, acc.y);
      acc.z = fmaf(g, v.z, acc.z);
      acc.w = fmaf(g, v.w, acc.w);
    }
    for (int sh = 0; sh < S; ++sh) {
      if (s_ok[T * k + sh] == 0.0f) continue;
      const float4 v = __ldcg(y4 + (size_t)(T * k + sh * T + t) * H4 + cc);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    if (lv.residual) {
      const float4 r = __ldcg(reinterpret_cast<const float4*>(lv.residual) + e);
      acc.x += r.x;
      acc.y += r.y;
      acc.z += r.z;
      acc.w += r.w;
    }
    reinterpret_cast<float4*>(lv.out)[e] = acc;
  }
}

template <int FMT, bool kRing, int NW>
__global__ void __launch_bounds__(32 * NW, NW == 4 ? 2 : 1) decode_stack_kernel(const __grid_constant__ DecodeArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const long long t_launch = clock64();
  stage_format_tables<FMT>();
  Ctx<FMT> c(a, smem_raw);
  // kRing: each warp's two weight stages after the decode buffers
  WarpRing<FMT> ring;
  ring.base = smem_raw + ring_offset(decode_smem(c.T, c.H, c.I, c.E, c.k, c.S, c.nw, nullptr, nullptr)) +
              (size_t)c.warp * kRingStages * ring_unit_bytes<FMT>();
  ring.issued = ring.taken = 0;
  ring.lane = c.lane;
  StackSeq q;
  q.L = a.n_layers;
  q.overlap = stack_disjoint(a, q.L);
  q.nR = (c.E + c.nw - 1) / c.nw;
  // bigger items when a row group is little work (short K): fewer waits and
  // signals per byte; bounded by the per-warp accumulators in shared memory
  const int Tm = c.T > 16 ? c.T : 16;
  q.gpi = max(1, min(2 * c.nw / c.nbH, Tm / c.T));
  q.grp_g = (c.nRG + q.gpi - 1) / q.gpi;
  q.nGU = c.P * q.grp_g;
  q.dpi = (c.nbI <= 2 && 2 * c.T <= 2 * Tm) ? 2 : 1;
  q.grp_d = (c.nRGH + c.nw * q.dpi - 1) / (c.nw * q.dpi);
  q.nD = c.P * q.grp_d;
  q.nC = (c.T * (c.H / 4) + kCombineVec - 1) / kCombineVec;
  q.per_stage = q.nR + 1 + q.nGU + q.nD + q.nC;
  q.n_stages = q.overlap ? q.L + 4 * StackSeq::kLag : q.L;
  // this launch's counters start at zero (one grid barrier), so a launch
  // depends on no state a previous launch left behind
  {
    unsigned long long* cnt = stk_cnt(a, 0, 0);
    const size_t n = (size_t)q.L * a.sp.n_cnt;
    for (size_t j = (size_t)blockIdx.x * c.nt + c.tid; j < n; j += (size_t)gridDim.x * c.nt) cnt[j] = 0;
    if (blockIdx.x == 0 && c.tid < 15 && a.phase_ns) a.phase_ns[c.tid] = 0;
  }
  if (!grid_barrier(a.bar, a.status)) return;
  // per item kind: cycles of work, cycles waiting, items (summed over CTAs at the end)
  long long t_work[5] = {0, 0, 0, 0, 0}, t_wait[5] = {0, 0, 0, 0, 0};
  const long long t_ready = clock64();
  long long t_prev = t_ready, t_gaps = 0, t_head = -1, n_items_done = 0;
  const unsigned long long ep1 = 1;  // counter targets are counts x ep1
  if (blockIdx.x == 0 && c.tid == 0 && a.phase_ns) {
    a.phase_ns[15] = q.overlap ? 3 : 4;  // which order ran
    a.phase_ns[14] = gridDim.x;
  }
  const long long n_items = q.count();
  const int G = gridDim.x;
  int staged_x = -1;
  if (!kRing && c.tid == 32) stack_prefetch(c, q, blockIdx.x, ep1);
  for (long long i = blockIdx.x; i < n_items; i += G) {
    int kind, l, idx;
    q.item(i, kind, l, idx);
    if (l < 0 || l >= q.L) continue;
    // the layer's pointer record, read only by the items that use it (router,
    // routing, combine): gate/up and down items do not wait for it
    auto lv = [&]() { return layer_view(a, l); };
    const LayerView none{};
    bool ok = true;
    // while thread 0 waits, thread 32 prefetches the next item's weights
    // towards L2; with the weight rings that lookup only delays the wait's
    // closing barrier (measured), so they go without
    auto next_pf = [&]() {
      if constexpr (!kRing) stack_prefetch(c, q, i + G, ep1);
    };
    const long long t0 = clock64();
    if (t_head < 0) t_head = t0 - t_ready;
    else t_gaps += t0 - t_prev;
    long long t1 = t0;  // end of the wait
    if (kind == StackSeq::kR) {
      if (!q.overlap && l > 0) ok = wait_count(stk_cnt(a, l - 1, 3), ep1 * q.nC, a.status, next_pf);
      else if (c.tid == 32) next_pf();
      t1 = clock64();
      if (ok) {
        stack_router_item(c, lv(), l, idx, q.nR);
        // layer by layer: the CTA of the last router item routes the layer at once
        if (q.overlap) {
          signal_count(stk_cnt(a, l, 0));
        } else if (signal_last(stk_cnt(a, l, 0), ep1 * q.nR)) {
          stack_routing_item(c, lv(), l, l == q.L - 1);
          signal_count(stk_cnt(a, l, 1));
        }
      }
    } else if (kind == StackSeq::kQ) {
      if (q.overlap) {
        ok = wait_count(stk_cnt(a, l, 0), ep1 * q.nR, a.status, next_pf);
        t1 = clock64();
        if (ok) {
          stack_routing_item(c, lv(), l, l == q.L - 1);
          signal_count(stk_cnt(a, l, 1));
        }
      }
    } else if (kind == StackSeq::kGU) {
      ok = wait_count(stk_cnt(a, l, 1), ep1, a.status, next_pf);
      t1 = clock64();
      if (ok) {
        if constexpr (kRing) stack_gateup_ring(c, none, l, idx, q.gpi, q.grp_g, staged_x, ring);
        else stack_gateup_item(c, none, l, idx, q.gpi, q.grp_g, staged_x);
        signal_count(stk_cnt(a, l, kStackCnt + idx / q.grp_g));
      }
    } else if (kind == StackSeq::kD) {
      ok = wait_count(stk_cnt(a, l, kStackCnt + idx / q.grp_d), ep1 * q.grp_g, a.status, next_pf);
      t1 = clock64();
      if (ok) {
        if constexpr (kRing) stack_down_ring(c, none, l, idx, q.dpi, q.grp_d, ring);
        else stack_down_item(c, none, l, idx, q.dpi, q.grp_d);
        // layer by layer: the CTA of the last down item combines the layer at once
        if (q.overlap) {
          signal_count(stk_cnt(a, l, 2));
        } else if (signal_last(stk_cnt(a, l, 2), ep1 * q.nD)) {
          const LayerView lvc = lv();
          for (int ci = 0; ci < q.nC; ++ci) {
            stack_combine_item(c, lvc, l, ci);
            __syncthreads();  // the next chunk restages the gates
          }
          if (c.tid == 0) release_add(stk_cnt(a, l, 3), (unsigned long long)q.nC);
        }
      }
    } else if (q.overlap) {
      ok = wait_count(stk_cnt(a, l, 2), ep1 * q.nD, a.status, next_pf);
      t1 = clock64();
      if (ok) {
        stack_combine_item(c, lv(), l, idx);
        signal_count(stk_cnt(a, l, 3));
      }
    }
    if (!ok) return;  // the status word says why; CTAs waiting on this one run out too
    t_wait[kind] += t1 - t0;
    t_prev = clock64();
    t_work[kind] += t_prev - t1;
    ++n_items_done;
  }
  // totals over all CTAs (SM cycles): [0..4] work per item kind, [5..9] wait
  // per item kind, [10] prologue (counter reset, order check, barrier),
  // [11] before the first item, [12] between items, [13] items done;
  // [14] is the grid size
  if (c.tid == 0 && a.phase_ns) {
    for (int k = 0; k < 5; ++k) {
      atomicAdd(a.phase_ns + k, (unsigned long long)t_work[k]);
      atomicAdd(a.phase_ns + 5 + k, (unsigned long long)t_wait[k]);
    }
    atomicAdd(a.phase_ns + 10, (unsigned long long)(t_ready - t_launch));
    atomicAdd(a.phase_ns + 11, (unsigned long long)(t_head < 0 ? 0 : t_head));
    atomicAdd(a.phase_ns + 12, (unsigned long long)t_gaps);
    atomicAdd(a.phase_ns + 13, (unsigned long long)n_items_done);
  }
}

// One instantiation of the stack kernel: per_sm_max CTAs per SM at most.
// Returns cudaErrorCooperativeLaunchTooLarge (nothing launched) when fewer
// than per_sm_min CTAs of it fit an SM.
template <int FMT, bool kRing, int NW>
cudaError_t launch_stack_variant(const DecodeArgs& a, size_t smem, int per_sm_min, int per_sm_max, cudaStream_t s) {
  auto kern = decode_stack_kernel<FMT, kRing, NW>;
  static size_t opted = 0;  // per instantiation; the opt-in only grows
  cudaError_t err;
  if (smem > opted) {
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    opted = smem;
  }
  int per_sm = 0;
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 32 * NW, smem);
  if (err != cudaSuccess) return err;
  if (per_sm < per_sm_min) return cudaErrorCooperativeLaunchTooLarge;
  const int grid = num_sms() * std::min(per_sm, per_sm_max);
  DecodeArgs args = a;
  void* params[] = {&args};
  note_launch();
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(kern), dim3(grid), dim3(32 * NW), params, smem,
                                     s);
}

// Two CTAs of 4 warps per SM, each streaming its warps' weight rings, where
// both fit an SM (two items in flight per SM: one CTA's waits, lookups and
// reductions overlap the other's weight stream); otherwise one CTA of 8
// warps, with the rings when they fit beside the decode buffers.
template <int FMT>
cudaError_t launch_stack_t(const DecodeArgs& a, cudaStream_t s) {
  int dev = 0, optin = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err == cudaSuccess) err = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (err != cudaSuccess) return err;
  const size_t spare = 1024 + (FMT == kIQ2G ? kIq2gSmemBytes : 0);  // the kernel's static shared variables
  const size_t unit = (size_t)kRingStages * ring_unit_bytes<FMT>();
  const size_t ring4 = ring_offset(decode_smem(a.T, a.H, a.I, a.E, a.k, a.S, 4, nullptr, nullptr)) + 4 * unit;
  if (ring4 + spare <= (size_t)optin) {
    err = launch_stack_variant<FMT, true, 4>(a, ring4, 2, 2, s);
    if (err != cudaErrorCooperativeLaunchTooLarge) return err;
    cudaGetLastError();
  }
  const size_t base8 = decode_smem(a.T, a.H, a.I, a.E, a.k, a.S, 8, nullptr, nullptr);
  const size_t ring8 = ring_offset(base8) + 8 * unit;
  if (ring8 + spare <= (size_t)optin) return launch_stack_variant<FMT, true, 8>(a, ring8, 1, 2, s);
  return launch_stack_variant<FMT, false, 8>(a, base8, 1, 2, s);
}

template <int FMT>
cudaError_t launch_decode_t(const DecodeArgs& a, cudaStream_t s) {
  const size_t smem = decode_smem(a.T, a.H, a.I, a.E, a.k, a.S, kDecWarps, nullptr, nullptr);
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
}  // namespace moe
