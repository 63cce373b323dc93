// Single-launch decode layer: the whole MoE layer for a few tokens in one
// cooperative, persistent kernel (one CTA per SM, all co-resident).
//
//   phase 0  router logits (one warp per expert row), q8_K of x, L2 prefetch
//            of the shared experts' gate/up weights (their use does not
//            depend on routing)
//   -------- grid barrier --------
//   phase 1  every CTA redundantly: top-k of every token, bucketing and the
//            tile plan, all in shared memory (no second barrier needed); the
//            q8_K rows of x are staged in shared memory
//   phase 2  gate/up items (tile, 32-row group), round-robin over CTAs; the
//            8 warps of a CTA split the super-blocks and their partial sums
//            are reduced in a fixed order; h = silu(G) * U goes to global
//            memory.  The weights of this CTA's next items and of its first
//            down items are prefetched into L2 meanwhile.
//   -------- grid barrier --------
//   phase 3  down items (tile, group of row groups), in contiguous blocks per
//            CTA so that the q8_K of a tile's h is made once per CTA;
//            integer-dot GEMV; y to the slot buffer; L2 prefetch runs ahead.
//   -------- grid barrier --------
//   phase 4  combine: out = residual + sum_s gate * y (slots in order, then
//            the shared experts), rows split over all CTAs.
//
// The barrier is a 64-bit arrival counter; every wait is bounded and sets
// MOE_ERR_DEVICE_TIMEOUT instead of hanging.  Data written inside the kernel
// is read back through L2 (ld.global.cg), never through L1 or the read-only
// path.  CTA 0 stamps its SM cycle counter at each phase boundary into the
// workspace.
//
// Sources: Pulsar README, "How the streaming works" (one expert union per
// batch; explicit per-(token, slot) pointers, NULL = not mine), "Fidelity
// notes" (q8_0/q8_K activations, integer dp4a dots, the per-slot sum), "What
// it does today" (Q4_K matmuls on q8_K activations); Strata summary (per-layer
// work captured once and replayed, zero allocation on the token path).
#include <algorithm>
#include <cmath>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kDecThreads = 256;
constexpr int kDecWarps = kDecThreads / 32;
constexpr long long kSpinLimit = 1ll << 24;  // x ~64 ns sleeps: about a second

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

struct Smem {
  int8_t* xq;      // [T][H]
  int16_t* xbs;    // [T][H/16]
  float* xd;       // [T][nbH]
  int* ids;        // [T*k]
  float* gates;    // [T*k]
  int* cnt;        // [E+S+1]  counts -> offsets
  int* scan;       // [E+S+1]  tile-plan scratch
  int* tok;        // [P]      token of each bucket position
  int* slot;       // [P]      slot index of each bucket position
  Tile* tiles;     // [P]
  float* red;      // [8 warps][2][T][32] accumulators / partial sums
  int8_t* hq;      // [T][I]
  int16_t* hbs;    // [T][I/16]
  float* hd;       // [T][nbI]
  int* aoff;       // [T]  activation row offsets of the current item
  int* n_tiles;    // 1
};

__host__ __device__ inline size_t al16(size_t v) { return (v + 15) / 16 * 16; }

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
  p = take((size_t)T * k * 4);             if (sm) sm->ids = (int*)p;
  p = take((size_t)T * k * 4);             if (sm) sm->gates = (float*)p;
  p = take((size_t)(E + S + 1) * 4);       if (sm) sm->cnt = (int*)p;
  p = take((size_t)(E + S + 1) * 4);       if (sm) sm->scan = (int*)p;
  p = take((size_t)P * 4);                 if (sm) sm->tok = (int*)p;
  p = take((size_t)P * 4);                 if (sm) sm->slot = (int*)p;
  p = take((size_t)P * sizeof(Tile));      if (sm) sm->tiles = (Tile*)p;
  p = take((size_t)kDecWarps * 2 * (T > 16 ? T : 16) * 32 * 4); if (sm) sm->red = (float*)p;
  p = take((size_t)T * I);                 if (sm) sm->hq = (int8_t*)p;
  p = take((size_t)T * (I / 16) * 2);      if (sm) sm->hbs = (int16_t*)p;
  p = take((size_t)T * (I / 256) * 4);     if (sm) sm->hd = (float*)p;
  p = take((size_t)T * 4);                 if (sm) sm->aoff = (int*)p;
  p = take(16);                            if (sm) sm->n_tiles = (int*)p;
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

// expert of the o-th entry of the tile order: shared experts first
__device__ __forceinline__ int tile_order_expert(int o, int E, int S) { return o < S ? E + o : o - S; }

template <int FMT>
__global__ void __launch_bounds__(kDecThreads, 1) decode_fused_kernel(DecodeArgs a) {
  using F = Fmt<FMT>;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  Smem sm;
  const int T = a.T, H = a.H, I = a.I, E = a.E, k = a.k, S = a.S;
  decode_smem(T, H, I, E, k, S, &sm, smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = gridDim.x;
  const int nbH = H / 256, nbI = I / 256, nRG = I / 32, nRGH = H / 32;
  const int P = T * (k + S), EpS = E + S;
  auto stamp = [&](int i) {
    if (blockIdx.x == 0 && tid == 0 && a.phase_ns) a.phase_ns[i] = (unsigned long long)clock64();
  };
  // router work split (fixed for the launch): wpr warps per expert row, each
  // over a contiguous 1/wpr of H, so that each lane issues all of its loads
  // in one round; rows_cta rows per CTA and round
  const int GW = G * kDecWarps;
  const int wpr = GW >= 8 * E ? 8 : GW >= 4 * E ? 4 : GW >= 2 * E ? 2 : 1;
  const int rows_cta = kDecWarps / wpr;
  const int n_layers = a.n_layers > 0 ? a.n_layers : 1;

  for (int layer = 0; layer < n_layers; ++layer) {
  const LayerView lv = layer_view(a, layer);
  stamp(0);

  // ------------------------------------------------------------ phase 0
  {
    const int gw = blockIdx.x * kDecWarps + warp;
    const int H4 = H >> 2;
    const int rl = warp / wpr, ch = warp % wpr;
    const int c4 = H4 / wpr;  // float4s per chunk
    float* part = sm.red;     // [8 warps][T] partial sums
    for (int base = blockIdx.x * rows_cta; base < E; base += G * rows_cta) {
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
      for (int i = tid; i < rows_cta * T; i += kDecThreads) {
        const int r = i / T, t = i % T, er = base + r;
        if (er < E) {
          float v = 0.0f;
          for (int c = 0; c < wpr; ++c) v += part[(r * wpr + c) * T + t];
          a.logits[(size_t)t * E + er] = v + (lv.bias ? __ldg(lv.bias + er) : 0.0f);
        }
      }
      __syncthreads();
    }
    // q8_K of x: one warp per 256-element block, from the last warps down
    for (int qb = GW - 1 - gw; qb < T * nbH; qb += GW) {
      const float4* src = reinterpret_cast<const float4*>(lv.x + (size_t)qb * 256 + 8 * lane);
      const float4 v0 = __ldcg(src), v1 = __ldcg(src + 1);
      const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
      q8k_block_warp(v, lane, a.xq + (size_t)qb * 256, a.xd + qb, a.xbs + (size_t)qb * 16);
    }
    // shared experts' gate/up weights: their phase-2 items come first, one per CTA round-robin
    if (tid == 0) {
      const size_t run = (size_t)nbH * F::kSlabBytes;
      for (int it = blockIdx.x; it < S * nRG; it += G) {
        const moe_expert_ptrs ep = lv.table[E + it / nRG];
        if (!ep.gate) continue;
        const size_t off = (size_t)(it % nRG) * run;
        prefetch_l2(static_cast<const uint8_t*>(ep.gate) + off, (uint32_t)run);
        prefetch_l2(static_cast<const uint8_t*>(ep.up) + off, (uint32_t)run);
      }
    }
  }
  stamp(1);
  if (!grid_barrier(a.bar, a.status)) return;
  stamp(2);

  // ------------------------------------------------------------ phase 1
  {
    // q8_K rows of x into shared memory (written in phase 0 by other CTAs: via L2)
    const int nq = T * H / 16, nb16 = T * (H / 16) * 2 / 16, nd = T * nbH;
    for (int i = tid; i < nq; i += kDecThreads)
      reinterpret_cast<int4*>(sm.xq)[i] = __ldcg(reinterpret_cast<const int4*>(a.xq) + i);
    for (int i = tid; i < nb16; i += kDecThreads)
      reinterpret_cast<int4*>(sm.xbs)[i] = __ldcg(reinterpret_cast<const int4*>(a.xbs) + i);
    for (int i = tid; i < nd; i += kDecThreads) sm.xd[i] = __ldcg(a.xd + i);
    // top-k of every token (each CTA computes the same result)
    for (int t = warp; t < T; t += kDecWarps)
      warp_topk(a.logits + (size_t)t * E, E, k, a.route, lane, sm.ids + t * k, sm.gates + t * k,
                blockIdx.x == 0 && a.gap ? a.gap + t : nullptr);
    for (int e = tid; e < EpS; e += kDecThreads) sm.cnt[e] = 0;
    __syncthreads();
    stamp(9);
    for (int p = tid; p < T * k; p += kDecThreads) atomicAdd(&sm.cnt[sm.ids[p]], 1);
    for (int sh = tid; sh < S; sh += kDecThreads) sm.cnt[E + sh] = T;
    __syncthreads();
    if (blockIdx.x == 0)
      for (int e = tid; e < EpS; e += kDecThreads) a.counts[e] = sm.cnt[e];
    __syncthreads();
    const int total = block_exclusive_scan(sm.cnt, EpS);  // sm.cnt: offsets
    if (tid == 0) sm.cnt[EpS] = total;
    __syncthreads();
    stamp(10);
    for (int p = tid; p < T * k; p += kDecThreads) {
      const int e = sm.ids[p];
      int rank = 0;
      for (int q = 0; q < p; ++q) rank += (sm.ids[q] == e);
      const int pos = sm.cnt[e] + rank;
      sm.tok[pos] = p / k;
      sm.slot[pos] = p;
    }
    for (int i = tid; i < S * T; i += kDecThreads) {
      const int sh = i / T, t = i % T;
      const int pos = sm.cnt[E + sh] + t;
      sm.tok[pos] = t;
      sm.slot[pos] = T * k + sh * T + t;
    }
    __syncthreads();
    if (blockIdx.x == 0) {
      for (int e = tid; e <= EpS; e += kDecThreads) a.offsets[e] = sm.cnt[e];
      for (int j = tid; j < P; j += kDecThreads) {
        a.perm[j] = sm.slot[j];
        if (a.inv) a.inv[sm.slot[j]] = j;
      }
      for (int p = tid; p < T * k; p += kDecThreads) {
        a.ids[p] = sm.ids[p];
        a.gates[p] = sm.gates[p];
        if (lv.ids_out) lv.ids_out[p] = sm.ids[p];
        if (lv.gates_out) lv.gates_out[p] = sm.gates[p];
      }
    }
    stamp(11);
    // tile plan: one tile per expert used (a tile holds up to T <= 16 rows), shared experts first
    int* order = sm.scan;
    for (int o = tid; o < EpS; o += kDecThreads) {
      const int e = tile_order_expert(o, E, S);
      const int c = sm.cnt[e + 1] - sm.cnt[e];
      order[o] = c > 0 ? 1 : 0;
    }
    __syncthreads();
    const int nt = block_exclusive_scan(order, EpS);
    for (int o = tid; o < EpS; o += kDecThreads) {
      const int e = tile_order_expert(o, E, S);
      const int c = sm.cnt[e + 1] - sm.cnt[e];
      if (c > 0) {
        Tile tl;
        tl.expert = e;
        tl.start = sm.cnt[e];
        tl.count = c;
        tl.flag = lv.table[e].gate == nullptr ? 1 : 0;
        sm.tiles[order[o]] = tl;
      }
    }
    if (tid == 0) *sm.n_tiles = nt;
    __syncthreads();
  }
  const int n_tiles = *sm.n_tiles;
  stamp(3);

  // down items: groups of row groups over H, in contiguous blocks per CTA
  const int rg_per = nbI >= kDecWarps ? 1 : kDecWarps / nbI;     // row groups per item
  const int n_grp = (nRGH + rg_per - 1) / rg_per;
  const int n3 = n_tiles * n_grp;
  const int d_begin = (int)((long long)n3 * blockIdx.x / G), d_end = (int)((long long)n3 * (blockIdx.x + 1) / G);
  const size_t dn_rg_bytes = (size_t)nbI * F::kSlabBytes;
  // L2 prefetch of the down weights of items [i0, i1) of this CTA (same tile: one contiguous run)
  auto prefetch_down = [&](int i0, int i1) {
    while (i0 < i1) {
      const int ti = i0 / n_grp;
      const int last = min(i1, (ti + 1) * n_grp);
      const Tile tl = sm.tiles[ti];
      if (!tl.flag) {
        const int rg0 = (i0 % n_grp) * rg_per;
        const int rg1 = min(nRGH, ((last - 1) % n_grp + 1) * rg_per);
        prefetch_l2(static_cast<const uint8_t*>(lv.table[tl.expert].down) + (size_t)rg0 * dn_rg_bytes,
                    (uint32_t)((size_t)(rg1 - rg0) * dn_rg_bytes));
      }
      i0 = last;
    }
  };
  constexpr int kDownAhead = 4;  // items of L2 prefetch ahead in phase 3

  // ------------------------------------------------------------ phase 2
  {
    const int n2 = n_tiles * nRG;
    const size_t run = (size_t)nbH * F::kSlabBytes;
    auto prefetch_gu = [&](int it) {
      if (it >= n2) return;
      const Tile tn = sm.tiles[it / nRG];
      if (tn.flag) return;
      const moe_expert_ptrs en = lv.table[tn.expert];
      prefetch_l2(static_cast<const uint8_t*>(en.gate) + (size_t)(it % nRG) * run, (uint32_t)run);
      prefetch_l2(static_cast<const uint8_t*>(en.up) + (size_t)(it % nRG) * run, (uint32_t)run);
    };
    bool first = true;
    for (int it = blockIdx.x; it < n2; it += G) {
      const Tile tl = sm.tiles[it / nRG];
      const int rg = it % nRG;
      if (tl.flag) continue;
      const moe_expert_ptrs ep = lv.table[tl.expert];
      const uint8_t* gbase = static_cast<const uint8_t*>(ep.gate) + (size_t)rg * run;
      const uint8_t* ubase = static_cast<const uint8_t*>(ep.up) + (size_t)rg * run;
      for (int t = tid; t < tl.count; t += kDecThreads) sm.aoff[t] = sm.tok[tl.start + t] * H;
      __syncthreads();
      // per-warp accumulators in shared memory: red[warp][m][t][lane]
      float* accw = sm.red + (size_t)warp * 2 * T * 32;  // gate [T][32], then up [T][32]
      for (int i = lane; i < tl.count * 32; i += 32) accw[i] = accw[T * 32 + i] = 0.0f;
      __syncwarp();
      for (int b = warp; b < nbH; b += kDecWarps) {
        SbRegs<FMT> sg, su;
        load_sb<FMT>(gbase + (size_t)b * F::kSlabBytes, lane, sg);
        load_sb<FMT>(ubase + (size_t)b * F::kSlabBytes, lane, su);
        if (tid == 0 && b == warp) {
          // keep HBM busy: this CTA's next two gate/up items and, once, its first down items
          if (first) prefetch_gu(it + G);
          prefetch_gu(it + 2 * G);
          if (first) prefetch_down(d_begin, min(d_end, d_begin + kDownAhead));
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
        a.h[(size_t)(tl.start + t) * I + rg * 32 + r] = Gv / (1.0f + expf(-Gv)) * Uv;
      }
      __syncthreads();
    }
    if (first && tid == 0) prefetch_down(d_begin, min(d_end, d_begin + kDownAhead));
  }
  stamp(4);
  if (!grid_barrier(a.bar, a.status)) return;
  stamp(5);

  // ------------------------------------------------------------ phase 3
  {
    if (tid == 0 && layer + 1 < n_layers) {
      // the next layer's router rows of this CTA and its shared-expert gate/up
      // items do not depend on this layer: start them towards L2 now
      const LayerView nx = layer_view(a, layer + 1);
      for (int base = blockIdx.x * rows_cta; base < E; base += G * rows_cta)
        prefetch_l2(nx.w_router + (size_t)base * H, (uint32_t)((size_t)min(rows_cta, E - base) * H * 4));
      const size_t run = (size_t)nbH * F::kSlabBytes;
      for (int it = blockIdx.x; it < S * nRG; it += G) {
        const moe_expert_ptrs ep = nx.table[E + it / nRG];
        if (!ep.gate) continue;
        prefetch_l2(static_cast<const uint8_t*>(ep.gate) + (size_t)(it % nRG) * run, (uint32_t)run);
        prefetch_l2(static_cast<const uint8_t*>(ep.up) + (size_t)(it % nRG) * run, (uint32_t)run);
      }
    }
    for (int t = tid; t < T; t += kDecThreads) sm.aoff[t] = t * I;
    __syncthreads();
    int staged = -1;  // tile whose q8_K(h) is in shared memory
    for (int it = d_begin; it < d_end; ++it) {
      const int ti = it / n_grp;
      const Tile tl = sm.tiles[ti];
      const int grp = it % n_grp;
      const int rg0 = grp * rg_per, nrg = min(rg_per, nRGH - rg0);
      if (tid == 0 && it + kDownAhead < d_end) prefetch_down(it + kDownAhead, it + kDownAhead + 1);
      if (tl.flag) continue;
      if (ti != staged) {
        __syncthreads();  // previous readers of the staged rows are done
        for (int task = warp; task < tl.count * nbI; task += kDecWarps) {
          const int t = task / nbI, blk = task % nbI;
          const float4* src =
              reinterpret_cast<const float4*>(a.h + (size_t)(tl.start + t) * I + blk * 256 + 8 * lane);
          const float4 v0 = __ldcg(src), v1 = __ldcg(src + 1);
          const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
          q8k_block_warp(v, lane, sm.hq + (size_t)t * I + blk * 256, sm.hd + t * nbI + blk,
                         sm.hbs + (size_t)t * (I / 16) + blk * 16);
        }
        __syncthreads();
        if (grp == 0) {  // the CTA holding a tile's first item keeps a copy of q8_K(h) in the workspace
          const size_t r0 = (size_t)tl.start;
          for (int i = tid; i < tl.count * I / 16; i += kDecThreads)
            reinterpret_cast<int4*>(a.hq + r0 * I)[i] = reinterpret_cast<const int4*>(sm.hq)[i];
          for (int i = tid; i < tl.count * nbI; i += kDecThreads) a.hd[r0 * nbI + i] = sm.hd[i];
          for (int i = tid; i < tl.count * (I / 16); i += kDecThreads) a.hbs[r0 * (I / 16) + i] = sm.hbs[i];
        }
        staged = ti;
      }
      const uint8_t* dbase = static_cast<const uint8_t*>(lv.table[tl.expert].down);
      float* accw = sm.red + (size_t)warp * T * 32;
      for (int i = lane; i < tl.count * 32; i += 32) accw[i] = 0.0f;
      __syncwarp();
      // warp -> (row group, super-blocks)
      const int rgl = nbI >= kDecWarps ? 0 : warp / nbI;
      const int b0 = nbI >= kDecWarps ? warp : warp % nbI;
      const int bstep = nbI >= kDecWarps ? kDecWarps : nbI;
      if (rgl < nrg) {
        const uint8_t* rbase = dbase + (size_t)(rg0 + rgl) * dn_rg_bytes;
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
        a.y[(size_t)sm.slot[tl.start + t] * H + (rg0 + g) * 32 + r] = v;
      }
      __syncthreads();
    }
  }
  stamp(6);
  if (!grid_barrier(a.bar, a.status)) return;
  stamp(7);

  // ------------------------------------------------------------ phase 4
  {
    const int H4 = H / 4;
    const float4* y4 = reinterpret_cast<const float4*>(a.y);
    for (int idx = blockIdx.x * kDecThreads + tid; idx < T * H4; idx += G * kDecThreads) {
      const int t = idx / H4, c = idx % H4;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int s = 0; s < k; ++s) {
        const int e = sm.ids[t * k + s];
        if (lv.table[e].gate == nullptr) continue;  // not mine: contributes nothing
        const float g = sm.gates[t * k + s];
        const float4 v = __ldcg(y4 + (size_t)(t * k + s) * H4 + c);
        acc.x = fmaf(g, v.x, acc.x);
        acc.y = fmaf(g, v.y, acc.y);
        acc.z = fmaf(g, v.z, acc.z);
        acc.w = fmaf(g, v.w, acc.w);
      }
      for (int sh = 0; sh < S; ++sh) {
        if (lv.table[E + sh].gate == nullptr) continue;
        const float4 v = __ldcg(y4 + (size_t)(T * k + sh * T + t) * H4 + c);
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
  stamp(8);
  // the next layer may read this layer's output
  if (layer + 1 < n_layers && !grid_barrier(a.bar, a.status)) return;
  }  // layers
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
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(kern), dim3(grid), dim3(kDecThreads), params,
                                     smem, s);
}

}  // namespace

size_t decode_smem_bytes(int T, int H, int I, int E, int k, int S) {
  return decode_smem(T, H, I, E, k, S, nullptr, nullptr);
}

cudaError_t launch_decode_fused(const DecodeArgs& a, cudaStream_t s) {
  return a.fmt == kQ4K ? launch_decode_t<kQ4K>(a, s) : launch_decode_t<kQ2K>(a, s);
}

}  // namespace moe
