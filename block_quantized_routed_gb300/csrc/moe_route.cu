// q8_K quantization, router logits, top-k gates, token -> expert bucketing
// and the expert tile plan.
//
// Sources: Pulsar README, "Fidelity notes" (q8_0/q8_K activations), "What it
// does today" (softmax router), "How the streaming works" (one expert union
// per batch or prefill chunk; explicit per-(token, slot) pointers, NULL =
// not mine); Pulsar digest note, section 1 (sigmoid-gated router + shared
// expert); Strata summary (router and shared expert resident on the GPU).
#include <cfloat>
#include <climits>
#include <cmath>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

// ---------------------------------------------------------------- q8_K
// one warp per 256-element block
__global__ void __launch_bounds__(256) q8k_quantize_kernel(const float* __restrict__ x, int64_t nblocks,
                                                           int8_t* __restrict__ q, float* __restrict__ d,
                                                           int16_t* __restrict__ bs) {
  const int lane = threadIdx.x & 31;
  const int64_t blk = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (blk >= nblocks) return;
  const float4* src = reinterpret_cast<const float4*>(x + blk * 256 + 8 * lane);
  float4 a = __ldg(src), b = __ldg(src + 1);
  float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  q8k_block_warp(v, lane, q + blk * 256, d + blk, bs ? bs + blk * 16 : nullptr);
}

// ---------------------------------------------------------------- router
// One warp per expert row e: logits[t, e] = sum_h w[e, h] * x[t, h] (+ bias[e]).
// Each lane accumulates a strided partial sum (h = 4*lane + 128*i), then a
// butterfly reduction: a fixed order, so results are deterministic.
constexpr int kRouterTok = 8;

__global__ void __launch_bounds__(128) router_kernel(const float* __restrict__ x, const float* __restrict__ w,
                                                     const float* __restrict__ bias, int T, int H, int E,
                                                     float* __restrict__ logits) {
  const int lane = threadIdx.x & 31;
  const int nwarps = gridDim.x * (blockDim.x >> 5);
  const int H4 = H >> 2;
  for (int e = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); e < E; e += nwarps) {
    const float4* wr = reinterpret_cast<const float4*>(w + (int64_t)e * H);
    const float be = bias ? __ldg(bias + e) : 0.0f;
    for (int t0 = 0; t0 < T; t0 += kRouterTok) {
      float acc[kRouterTok];
#pragma unroll
      for (int t = 0; t < kRouterTok; ++t) acc[t] = 0.0f;
      for (int h4 = lane; h4 < H4; h4 += 32) {
        const float4 wv = __ldg(wr + h4);
#pragma unroll
        for (int t = 0; t < kRouterTok; ++t) {
          if (t0 + t < T) {
            const float4 xv = __ldg(reinterpret_cast<const float4*>(x + (int64_t)(t0 + t) * H) + h4);
            acc[t] = fmaf(wv.x, xv.x, acc[t]);
            acc[t] = fmaf(wv.y, xv.y, acc[t]);
            acc[t] = fmaf(wv.z, xv.z, acc[t]);
            acc[t] = fmaf(wv.w, xv.w, acc[t]);
          }
        }
      }
#pragma unroll
      for (int t = 0; t < kRouterTok; ++t) {
        float v = acc[t];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0 && t0 + t < T) logits[(int64_t)(t0 + t) * E + e] = v + be;
      }
    }
  }
}

// Router logits of many tokens: logits[T, E] = x[T, H] * W[E, H]^T + bias, an
// fp32 GEMM (the gate stays in fp32: top-k picks are decided on these values).
// Tile 128 tokens x 128 experts per CTA, K steps of 16 staged in shared
// memory (double-buffered), 256 threads each holding an 8 x 8 register tile
// (rows ty*4 + {0..3} and 64 + ty*4 + {0..3}, columns likewise): every thread
// reads float4 pairs from shared memory per k and issues 64 FMAs.
constexpr int kRgTile = 128, kRgK = 16, kRgPad = 4;
// token count from which the tiled GEMM replaces the per-expert GEMV, and
// from which the tensor-core GEMM (128-token tiles) replaces both
constexpr int kRouterGemmMinT = 64;
constexpr int kRouterTcMinT = 128;

__global__ void __launch_bounds__(256) router_gemm_kernel(const float* __restrict__ x, const float* __restrict__ w,
                                                          const float* __restrict__ bias, int T, int H, int E,
                                                          float* __restrict__ logits) {
  __shared__ __align__(16) float sx[2][kRgK][kRgTile + kRgPad];
  __shared__ __align__(16) float sw[2][kRgK][kRgTile + kRgPad];
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int t0 = blockIdx.y * kRgTile, e0 = blockIdx.x * kRgTile;
  // loader: rows lr and lr + 64 of each tile, k quad lk (4 floats)
  const int lr = tid >> 2, lk = (tid & 3) * 4;
  const float* xr0 = t0 + lr < T ? x + (int64_t)(t0 + lr) * H : nullptr;
  const float* xr1 = t0 + lr + 64 < T ? x + (int64_t)(t0 + lr + 64) * H : nullptr;
  const float* wr0 = e0 + lr < E ? w + (int64_t)(e0 + lr) * H : nullptr;
  const float* wr1 = e0 + lr + 64 < E ? w + (int64_t)(e0 + lr + 64) * H : nullptr;
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  auto fetch = [&](int k0, float4 (&v)[4]) {
    v[0] = xr0 ? __ldg(reinterpret_cast<const float4*>(xr0 + k0 + lk)) : z;
    v[1] = xr1 ? __ldg(reinterpret_cast<const float4*>(xr1 + k0 + lk)) : z;
    v[2] = wr0 ? __ldg(reinterpret_cast<const float4*>(wr0 + k0 + lk)) : z;
    v[3] = wr1 ? __ldg(reinterpret_cast<const float4*>(wr1 + k0 + lk)) : z;
  };
  auto stash = [&](int buf, const float4 (&v)[4]) {
    sx[buf][lk + 0][lr] = v[0].x; sx[buf][lk + 1][lr] = v[0].y; sx[buf][lk + 2][lr] = v[0].z; sx[buf][lk + 3][lr] = v[0].w;
    sx[buf][lk + 0][lr + 64] = v[1].x; sx[buf][lk + 1][lr + 64] = v[1].y;
    sx[buf][lk + 2][lr + 64] = v[1].z; sx[buf][lk + 3][lr + 64] = v[1].w;
    sw[buf][lk + 0][lr] = v[2].x; sw[buf][lk + 1][lr] = v[2].y; sw[buf][lk + 2][lr] = v[2].z; sw[buf][lk + 3][lr] = v[2].w;
    sw[buf][lk + 0][lr + 64] = v[3].x; sw[buf][lk + 1][lr + 64] = v[3].y;
    sw[buf][lk + 2][lr + 64] = v[3].z; sw[buf][lk + 3][lr + 64] = v[3].w;
  };
  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;
  float4 v[4];
  fetch(0, v);
  stash(0, v);
  __syncthreads();
  const int nk = H / kRgK;
  for (int kt = 0; kt < nk; ++kt) {
    const int buf = kt & 1;
    if (kt + 1 < nk) fetch((kt + 1) * kRgK, v);
#pragma unroll
    for (int kk = 0; kk < kRgK; ++kk) {
      const float4 a0 = *reinterpret_cast<const float4*>(&sx[buf][kk][ty * 4]);
      const float4 a1 = *reinterpret_cast<const float4*>(&sx[buf][kk][64 + ty * 4]);
      const float4 b0 = *reinterpret_cast<const float4*>(&sw[buf][kk][tx * 4]);
      const float4 b1 = *reinterpret_cast<const float4*>(&sw[buf][kk][64 + tx * 4]);
      const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    if (kt + 1 < nk) stash(buf ^ 1, v);
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int t = t0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + i - 4);
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = e0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + j - 4);
      if (e < E) logits[(int64_t)t * E + e] = acc[i][j] + (bias ? __ldg(bias + e) : 0.0f);
    }
  }
}

// ---------------------------------------------------------------- top-k
__global__ void __launch_bounds__(128) topk_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                   int route, int32_t* __restrict__ ids,
                                                   float* __restrict__ gates, float* __restrict__ gap) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  warp_topk(logits + (int64_t)t * E, E, k, route, lane, ids + (int64_t)t * k, gates + (int64_t)t * k,
            gap ? gap + t : nullptr);
}

// Tile plan from counts/offsets: each expert with count c gets ceil(c/TT)
// tiles of up to TT rows, experts in ascending order.  Also zeroes the
// requant arrival counters of every tile.  All threads of the block call it;
// `scratch` holds >= EpS ints of shared memory.
__device__ void build_tiles(const int32_t* counts, const int32_t* offsets, int EpS,
                            const moe_expert_ptrs* table, int TT, int nIB, Tile* tiles, int32_t* n_tiles,
                            int32_t* req_cnt, int* scratch) {
  for (int e = threadIdx.x; e < EpS; e += blockDim.x) scratch[e] = (counts[e] + TT - 1) / TT;
  __syncthreads();
  const int total = block_exclusive_scan(scratch, EpS);
  for (int e = threadIdx.x; e < EpS; e += blockDim.x) {
    const int c = counts[e];
    if (c == 0) continue;
    const int flag = (table && table[e].gate == nullptr) ? 1 : 0;
    int ti = scratch[e];
    for (int st = 0; st < c; st += TT, ++ti) {
      Tile tl;
      tl.expert = e;
      tl.start = offsets[e] + st;
      tl.count = min(TT, c - st);
      tl.flag = flag;
      tiles[ti] = tl;
    }
  }
  for (int i = threadIdx.x; i < total * nIB; i += blockDim.x) req_cnt[i] = 0;
  if (threadIdx.x == 0) *n_tiles = total;
}

// ---------------------------------------------------------------- small path
// One CTA of 1024 threads: top-k of T tokens (one warp each), bucketing of
// the T*k <= kSmallPairs pairs, and the tile plan.
__global__ void __launch_bounds__(1024) route_bucket_small_kernel(
    const float* __restrict__ logits, int T, int E, int k, int route, int S, int32_t* ids,
    float* gates, float* gap, int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv,
    const moe_expert_ptrs* table, int TT, int nIB, Tile* tiles, int32_t* n_tiles, int32_t* req_cnt,
    int* status) {
  __shared__ int s_ids[kSmallPairs];
  __shared__ int s_cnt[MOE_MAX_EXPERTS + MOE_MAX_SHARED + 1];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int P = T * k, EpS = E + S;
  if (logits) {
    for (int t = warp; t < T; t += blockDim.x >> 5)
      warp_topk(logits + (int64_t)t * E, E, k, route, lane, ids + t * k, gates + t * k, gap ? gap + t : nullptr);
    __syncthreads();
    __threadfence_block();
  }
  for (int e = tid; e < EpS; e += blockDim.x) s_cnt[e] = 0;
  for (int p = tid; p < P; p += blockDim.x) {
    int e = ids[p];
    if (e < 0 || e >= E) {
      set_status(status, MOE_ERR_DEVICE_BOUNDS);
      e = -1;
    }
    s_ids[p] = e;
  }
  __syncthreads();
  for (int p = tid; p < P; p += blockDim.x)
    if (s_ids[p] >= 0) atomicAdd(&s_cnt[s_ids[p]], 1);
  for (int sh = tid; sh < S; sh += blockDim.x) s_cnt[E + sh] = T;
  __syncthreads();
  for (int e = tid; e < EpS; e += blockDim.x) counts[e] = s_cnt[e];
  __syncthreads();
  const int total = block_exclusive_scan(s_cnt, EpS);   // s_cnt now holds offsets
  for (int e = tid; e < EpS; e += blockDim.x) offsets[e] = s_cnt[e];
  if (tid == 0) offsets[EpS] = total;
  // stable positions: rank of p among earlier pairs of the same expert
  for (int p = tid; p < P; p += blockDim.x) {
    const int e = s_ids[p];
    if (e < 0) continue;
    int rank = 0;
    for (int q = 0; q < p; ++q) rank += (s_ids[q] == e);
    const int pos = s_cnt[e] + rank;
    perm[pos] = p;
    if (inv) inv[p] = pos;
  }
  for (int i = tid; i < S * T; i += blockDim.x) {
    const int sh = i / T, t = i % T;
    const int pos = s_cnt[E + sh] + t;
    const int p = P + sh * T + t;
    perm[pos] = p;
    if (inv) inv[p] = pos;
  }
  __syncthreads();
  __threadfence_block();
  if (tiles) build_tiles(counts, offsets, EpS, table, TT, nIB, tiles, n_tiles, req_cnt, s_cnt);
}

// ---------------------------------------------------------------- large path
__global__ void __launch_bounds__(1024) bucket_count_kernel(const int32_t* __restrict__ ids, int P, int E,
                                                            int EpS, int32_t* __restrict__ chunk_cnt,
                                                            int* status) {
  __shared__ int hist[MOE_MAX_EXPERTS + MOE_MAX_SHARED];
  for (int e = threadIdx.x; e < EpS; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int p = blockIdx.x * kBucketChunk + threadIdx.x;
  if (p < P) {
    const int e = ids[p];
    if (e >= 0 && e < E)
      atomicAdd(&hist[e], 1);
    else
      set_status(status, MOE_ERR_DEVICE_BOUNDS);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < EpS; e += blockDim.x) chunk_cnt[(int64_t)blockIdx.x * EpS + e] = hist[e];
}

// chunk_cnt[c][e] -> exclusive base of chunk c within bucket e; counts; offsets
__global__ void __launch_bounds__(1024) bucket_scan_kernel(int32_t* __restrict__ chunk_cnt, int n_chunks,
                                                           int T, int E, int S, int32_t* counts,
                                                           int32_t* offsets) {
  __shared__ int s_cnt[MOE_MAX_EXPERTS + MOE_MAX_SHARED + 1];
  const int EpS = E + S;
  for (int e = threadIdx.x; e < EpS; e += blockDim.x) {
    int run = 0;
    if (e < E) {
      for (int c = 0; c < n_chunks; ++c) {
        const int v = chunk_cnt[(int64_t)c * EpS + e];
        chunk_cnt[(int64_t)c * EpS + e] = run;
        run += v;
      }
    } else {
      run = T;
    }
    s_cnt[e] = run;
    counts[e] = run;
  }
  __syncthreads();
  const int total = block_exclusive_scan(s_cnt, EpS);
  for (int e = threadIdx.x; e < EpS; e += blockDim.x) offsets[e] = s_cnt[e];
  if (threadIdx.x == 0) offsets[EpS] = total;
}

__global__ void __launch_bounds__(1024) bucket_scatter_kernel(const int32_t* __restrict__ ids, int T, int k,
                                                              int E, int S, const int32_t* __restrict__ chunk_cnt,
                                                              const int32_t* __restrict__ offsets,
                                                              int32_t* __restrict__ perm, int32_t* inv) {
  __shared__ int s_ids[kBucketChunk];
  const int P = T * k, EpS = E + S;
  const int base = blockIdx.x * kBucketChunk;
  const int n = min(kBucketChunk, P - base);
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int e = ids[base + i];
    s_ids[i] = (e >= 0 && e < E) ? e : -1;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int e = s_ids[i];
    if (e < 0) continue;
    int rank = 0;
    for (int q = 0; q < i; ++q) rank += (s_ids[q] == e);
    const int pos = offsets[e] + chunk_cnt[(int64_t)blockIdx.x * EpS + e] + rank;
    perm[pos] = base + i;
    if (inv) inv[base + i] = pos;
  }
  if (blockIdx.x == 0) {
    for (int i = threadIdx.x; i < S * T; i += blockDim.x) {
      const int sh = i / T, t = i % T;
      const int pos = offsets[E + sh] + t;
      perm[pos] = P + sh * T + t;
      if (inv) inv[P + sh * T + t] = pos;
    }
  }
}

__global__ void __launch_bounds__(1024) plan_kernel(const int32_t* counts, const int32_t* offsets, int EpS,
                                                    const moe_expert_ptrs* table, int TT, int nIB, Tile* tiles,
                                                    int32_t* n_tiles, int32_t* req_cnt) {
  __shared__ int scratch[MOE_MAX_EXPERTS + MOE_MAX_SHARED + 1];
  build_tiles(counts, offsets, EpS, table, TT, nIB, tiles, n_tiles, req_cnt, scratch);
}

}  // namespace

// ---------------------------------------------------------------- launchers
cudaError_t launch_q8k_quantize(const float* x, int64_t T, int64_t K, int8_t* q, float* d, int16_t* bs,
                                cudaStream_t s) {
  const int64_t nblocks = T * (K / 256);
  if (nblocks == 0) return cudaSuccess;
  const int per = 8;  // warps (blocks of 256 elements) per CTA
  note_launch();
  q8k_quantize_kernel<<<(unsigned)((nblocks + per - 1) / per), 32 * per, 0, s>>>(x, nblocks, q, d, bs);
  return cudaGetLastError();
}

cudaError_t launch_router(const float* x, const float* w, const float* bias, int T, int H, int E, float* logits,
                          cudaStream_t s, int* status) {
  if (T == 0) return cudaSuccess;
  if (T >= kRouterTcMinT && H % 32 == 0) return launch_router_tc(x, w, bias, T, H, E, logits, status, s);
  if (T >= kRouterGemmMinT) {
    const dim3 grid((E + kRgTile - 1) / kRgTile, (T + kRgTile - 1) / kRgTile);
    note_launch();
    router_gemm_kernel<<<grid, 256, 0, s>>>(x, w, bias, T, H, E, logits);
    return cudaGetLastError();
  }
  const int warps = 2;                       // rows per CTA: spread the rows over many SMs
  int grid = (E + warps - 1) / warps;
  note_launch();
  router_kernel<<<grid, 32 * warps, 0, s>>>(x, w, bias, T, H, E, logits);
  return cudaGetLastError();
}

cudaError_t launch_topk(const float* logits, int T, int E, int k, int route, int32_t* ids, float* gates,
                        float* gap, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  note_launch();
  topk_kernel<<<(T + 3) / 4, 128, 0, s>>>(logits, T, E, k, route, ids, gates, gap);
  return cudaGetLastError();
}

cudaError_t launch_route_bucket_small(const float* logits, int T, int E, int k, int route, int S, int32_t* ids,
                                      float* gates, float* gap, int32_t* counts, int32_t* offsets, int32_t* perm,
                                      int32_t* inv, const moe_expert_ptrs* table, int TT, int nIB, Tile* tiles,
                                      int32_t* n_tiles, int32_t* req_cnt, int* status, cudaStream_t s) {
  note_launch();
  route_bucket_small_kernel<<<1, 1024, 0, s>>>(logits, T, E, k, route, S, ids, gates, gap, counts, offsets, perm,
                                                inv, table, TT, nIB, tiles, n_tiles, req_cnt, status);
  return cudaGetLastError();
}

cudaError_t launch_bucket_large(const int32_t* ids, int T, int k, int E, int S, int32_t* counts, int32_t* offsets,
                                int32_t* perm, int32_t* inv, int32_t* chunk_cnt, int* status, cudaStream_t s) {
  const int P = T * k;
  const int n_chunks = (P + kBucketChunk - 1) / kBucketChunk;
  if (n_chunks > 0) {
    note_launch();
    bucket_count_kernel<<<n_chunks, 1024, 0, s>>>(ids, P, E, E + S, chunk_cnt, status);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  note_launch();
  bucket_scan_kernel<<<1, 1024, 0, s>>>(chunk_cnt, n_chunks, T, E, S, counts, offsets);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  note_launch();
  bucket_scatter_kernel<<<n_chunks > 0 ? n_chunks : 1, 1024, 0, s>>>(ids, T, k, E, S, chunk_cnt, offsets, perm,
                                                                     inv);
  return cudaGetLastError();
}

cudaError_t launch_plan(const int32_t* counts, const int32_t* offsets, int EpS, const moe_expert_ptrs* table,
                        int TT, int nIB, Tile* tiles, int32_t* n_tiles, int32_t* req_cnt, cudaStream_t s) {
  note_launch();
  plan_kernel<<<1, 1024, 0, s>>>(counts, offsets, EpS, table, TT, nIB, tiles, n_tiles, req_cnt);
  return cudaGetLastError();
}

}  // namespace moe
