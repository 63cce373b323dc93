// Expert FFN kernels of the decode path: fused dequant + integer-dot GEMVs
// over block-quantized super-blocks on q8_K activations, SwiGLU, q8_K
// re-quantization of the intermediate, the down projection, and the
// gate-weighted combine.
//
// Work is cut into items of (expert tile, 32-row group).  One lane owns one
// weight row, so each 16-byte load of a warp reads 512 contiguous bytes of
// a slab; each expert's weights are read once for all the tokens of its tile
// (Pulsar README, "What it does today": a warp token tile lets several rows
// of activations share one weight read).  Gate/up: the four warps of a CTA
// split the super-blocks of the row group; their partial sums are reduced in
// a fixed order.  The 256-wide q8_K blocks of h span 8 row groups; the last
// of the 8 CTAs to finish a block quantizes it (arrival counter, no waiting).
//
// Sources: Pulsar README, "Fidelity notes" (q8_0/q8_K activations, integer
// dp4a dots; the per-slot sum), "What it does today" (gate/up/down FFN
// triple), "How the streaming works" (explicit per-expert pointers; NULL =
// not mine).
#include <algorithm>
#include <cmath>
#include <map>
#include <mutex>
#include <utility>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kThreads = 128;  // 4 warps per CTA

// shared memory: q8_K rows [TT][K], 16-sums [TT][K/16], scales [TT][K/256],
// row offsets [TT], per-warp accumulators [4][NM][TT][32]
__host__ __device__ constexpr size_t ffn_smem(int TT, int K, int NM) {
  return (size_t)TT * K + (size_t)TT * (K / 8) + (size_t)TT * (K / 256) * 4 + (size_t)TT * 4 +
         (size_t)4 * NM * TT * 32 * 4;
}

// Copy the q8_K rows of `cnt` tokens into shared memory: codes [TT][K],
// 16-code sums [TT][K/16], block scales [TT][K/256].  row_of(tt) gives the
// source row index.
template <class RowOf>
__device__ __forceinline__ void stage_rows(int cnt, int K, const int8_t* __restrict__ q,
                                           const int16_t* __restrict__ bs, const float* __restrict__ d,
                                           RowOf row_of, int8_t* s_q, int16_t* s_bs, float* s_d) {
  const int nq = K / 16, nbs = K / 128, nd = K / 256;
  for (int tt = 0; tt < cnt; ++tt) {
    const int64_t r = row_of(tt);
    const int4* srcq = reinterpret_cast<const int4*>(q + r * K);
    int4* dstq = reinterpret_cast<int4*>(s_q + (size_t)tt * K);
    for (int i = threadIdx.x; i < nq; i += blockDim.x) dstq[i] = srcq[i];
    const int4* srcb = reinterpret_cast<const int4*>(bs + r * (K / 16));
    int4* dstb = reinterpret_cast<int4*>(s_bs + (size_t)tt * (K / 16));
    for (int i = threadIdx.x; i < nbs; i += blockDim.x) dstb[i] = srcb[i];
    for (int i = threadIdx.x; i < nd; i += blockDim.x) s_d[tt * nd + i] = d[r * nd + i];
  }
}

template <int FMT>
__global__ void __launch_bounds__(kThreads, 2) gateup_kernel(FfnArgs a) {
  using F = Fmt<FMT>;
  extern __shared__ __align__(16) uint8_t smem[];
  stage_format_tables<FMT>();
  __shared__ int s_last;
  const int TT = a.TT;
  const int H = a.H, I = a.I, nbH = H / 256, nRG = I / 32, nIB = I / 256;
  int8_t* s_act = reinterpret_cast<int8_t*>(smem);
  int16_t* s_bs = reinterpret_cast<int16_t*>(smem + (size_t)TT * H);
  float* s_da = reinterpret_cast<float*>(smem + (size_t)TT * H + (size_t)TT * (H / 8));
  int* s_off = reinterpret_cast<int*>(s_da + TT * nbH);
  float* s_red = reinterpret_cast<float*>(s_off + TT);  // [4 warps][2][TT][32]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = *a.n_tiles * nRG;

  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int ti = item / nRG, rg = item % nRG;
    const Tile tl = a.tiles[ti];
    if (tl.flag) continue;  // expert not present: its rows are written as zeros by the down kernel
    const moe_expert_ptrs ep = a.table[tl.expert];
    const int cnt = tl.count;
    __syncthreads();  // shared memory of the previous item is free
    stage_rows(cnt, H, a.xq, a.xbs, a.xd,
               [&](int tt) { return (int64_t)token_of_slot(a.perm[tl.start + tt], a.T, a.k); }, s_act, s_bs,
               s_da);
    __syncthreads();

    for (int t = threadIdx.x; t < cnt; t += blockDim.x) s_off[t] = t * H;
    float* accw = s_red + (size_t)warp * 2 * TT * 32;
    for (int i = lane; i < 2 * TT * 32; i += 32) accw[i] = 0.0f;
    __syncthreads();
    const uint8_t* gbase = static_cast<const uint8_t*>(ep.gate) + (size_t)rg * nbH * F::kSlabBytes;
    const uint8_t* ubase = static_cast<const uint8_t*>(ep.up) + (size_t)rg * nbH * F::kSlabBytes;
#pragma unroll 1
    for (int b = warp; b < nbH; b += 4) {
      SbRegs<FMT> sg, su;
      load_sb<FMT>(gbase + (size_t)b * F::kSlabBytes, lane, sg);
      load_sb<FMT>(ubase + (size_t)b * F::kSlabBytes, lane, su);
      sb_accum<FMT>(sg, s_act, s_bs, s_da, s_off, b, cnt, accw, lane);
      sb_accum<FMT>(su, s_act, s_bs, s_da, s_off, b, cnt, accw + TT * 32, lane);
    }
    __syncthreads();
    // h = silu(G) * U for the 32 rows of this group and the tile's tokens
    for (int idx = threadIdx.x; idx < cnt * 32; idx += blockDim.x) {
      const int t = idx >> 5, r = idx & 31;
      float G = 0.0f, U = 0.0f;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        G += s_red[((w * 2 + 0) * TT + t) * 32 + r];
        U += s_red[((w * 2 + 1) * TT + t) * 32 + r];
      }
      const float hv = G / (1.0f + expf(-G)) * U;
      a.h[(size_t)(tl.start + t) * I + rg * 32 + r] = hv;
    }
    // the last of the 8 row groups of a 256-wide block quantizes it to q8_K
    __threadfence();
    __syncthreads();
    const int ib = rg >> 3;
    if (threadIdx.x == 0) s_last = (atomicAdd(&a.req_cnt[ti * nIB + ib], 1) == 7);
    __syncthreads();
    if (s_last) {
      __threadfence();
      for (int t = warp; t < cnt; t += 4) {
        const size_t row = (size_t)(tl.start + t);
        const float4* src = reinterpret_cast<const float4*>(a.h + row * I + ib * 256 + 8 * lane);
        const float4 v0 = __ldcg(src), v1 = __ldcg(src + 1);
        const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        q8k_block_warp(v, lane, a.hq + row * I + ib * 256, a.hd + row * nIB + ib, a.hbs + row * (I / 16) + ib * 16);
      }
      if (threadIdx.x == 0) a.req_cnt[ti * nIB + ib] = 0;
    }
  }
}

template <int FMT>
__global__ void __launch_bounds__(kThreads, 2) down_kernel(FfnArgs a) {
  using F = Fmt<FMT>;
  extern __shared__ __align__(16) uint8_t smem[];
  stage_format_tables<FMT>();
  const int TT = a.TT;
  const int H = a.H, I = a.I, nbI = I / 256, nQuad = H / 128;
  int8_t* s_act = reinterpret_cast<int8_t*>(smem);
  int16_t* s_bs = reinterpret_cast<int16_t*>(smem + (size_t)TT * I);
  float* s_da = reinterpret_cast<float*>(smem + (size_t)TT * I + (size_t)TT * (I / 8));
  int* s_off = reinterpret_cast<int*>(s_da + TT * nbI);
  float* s_red = reinterpret_cast<float*>(s_off + TT);  // [4 warps][TT][32]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = *a.n_tiles * nQuad;

  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int ti = item / nQuad, quad = item % nQuad;
    const Tile tl = a.tiles[ti];
    const int cnt = tl.count;
    const int rg = quad * 4 + warp;
    const int row = rg * 32 + lane;
    if (tl.flag) {  // expert not present ("not mine"): contributes zero
      for (int t = 0; t < cnt; ++t) a.y[(size_t)a.perm[tl.start + t] * H + row] = 0.0f;
      continue;
    }
    const moe_expert_ptrs ep = a.table[tl.expert];
    __syncthreads();
    stage_rows(cnt, I, a.hq, a.hbs, a.hd, [&](int tt) { return (int64_t)(tl.start + tt); }, s_act, s_bs, s_da);
    __syncthreads();
    for (int t = threadIdx.x; t < cnt; t += blockDim.x) s_off[t] = t * I;
    float* accw = s_red + (size_t)warp * TT * 32;
    for (int i = lane; i < TT * 32; i += 32) accw[i] = 0.0f;
    __syncthreads();
    const uint8_t* dbase = static_cast<const uint8_t*>(ep.down) + (size_t)rg * nbI * F::kSlabBytes;
#pragma unroll 1
    for (int b = 0; b < nbI; ++b) {
      SbRegs<FMT> sd;
      load_sb<FMT>(dbase + (size_t)b * F::kSlabBytes, lane, sd);
      sb_accum<FMT>(sd, s_act, s_bs, s_da, s_off, b, cnt, accw, lane);
    }
    __syncwarp();
    for (int t = 0; t < cnt; ++t) a.y[(size_t)a.perm[tl.start + t] * H + row] = accw[t * 32 + lane];
  }
}

// out[t] = (sum_s gates[t,s] * y[t*k+s] + sum_sh y[T*k + sh*T + t]) + residual[t]
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ y, const float* __restrict__ gates,
                                                      int T, int H, int k, int S, const float* residual,
                                                      float* out) {
  const int H4 = H >> 2;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (int64_t)T * H4) return;
  const int t = (int)(idx / H4), h4 = (int)(idx % H4);
  const float4* y4 = reinterpret_cast<const float4*>(y);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s = 0; s < k; ++s) {
    const float g = gates[(int64_t)t * k + s];
    const float4 v = y4[((int64_t)t * k + s) * H4 + h4];
    acc.x = fmaf(g, v.x, acc.x);
    acc.y = fmaf(g, v.y, acc.y);
    acc.z = fmaf(g, v.z, acc.z);
    acc.w = fmaf(g, v.w, acc.w);
  }
  for (int sh = 0; sh < S; ++sh) {
    const float4 v = y4[((int64_t)T * k + (int64_t)sh * T + t) * H4 + h4];
    acc.x += v.x;
    acc.y += v.y;
    acc.z += v.z;
    acc.w += v.w;
  }
  if (residual) {
    const float4 r = reinterpret_cast<const float4*>(residual)[idx];
    acc.x += r.x;
    acc.y += r.y;
    acc.z += r.z;
    acc.w += r.w;
  }
  reinterpret_cast<float4*>(out)[idx] = acc;
}

// test hook: the sub-block integer sums of the device dot routine
template <int FMT>
__global__ void debug_dots_kernel(const uint8_t* __restrict__ w, int N, int K, const int8_t* __restrict__ q, int T,
                                  int32_t* __restrict__ isum, int32_t* __restrict__ bsum) {
  using F = Fmt<FMT>;
  stage_format_tables<FMT>();
  const int nb = K / 256;
  const int rg = blockIdx.x / nb, b = blockIdx.x % nb;
  const int lane = threadIdx.x;
  const int n = rg * 32 + lane;
  SbRegs<FMT> s;
  load_sb<FMT>(w + ((size_t)rg * nb + b) * F::kSlabBytes, lane, s);
  for (int t = 0; t < T; ++t) {
    const int8_t* act = q + (size_t)t * K + 256 * b;
#pragma unroll
    for (int j = 0; j < F::kNSub; ++j) isum[(((size_t)t * N + n) * nb + b) * F::kNSub + j] = sub_isum<FMT>(s, j, act);
    if (rg == 0 && lane < F::kNSub) {
      int sum = 0;
      for (int i = 0; i < F::kSubLen; ++i) sum += act[lane * F::kSubLen + i];
      bsum[((size_t)t * nb + b) * F::kNSub + lane] = sum;
    }
  }
}

// Opt a kernel in to `smem` bytes of dynamic shared memory and return its
// resident CTAs per SM.  The opt-in only ever grows (a smaller value would
// make later launches with more shared memory fail); both answers are cached
// because the queries cost host time on every launch otherwise.
cudaError_t occupancy(const void* kern, size_t smem, int* per_sm) {
  static std::mutex mu;
  static std::map<const void*, size_t> opted;
  static std::map<std::pair<const void*, size_t>, int> cache;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find({kern, smem});
  if (it != cache.end()) {
    *per_sm = it->second;
    return cudaSuccess;
  }
  size_t& cur = opted[kern];
  if (smem > cur) {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    cur = smem;
  }
  cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, kern, kThreads, smem);
  if (err != cudaSuccess) return err;
  cache[{kern, smem}] = *per_sm;
  return cudaSuccess;
}

template <int FMT>
cudaError_t launch_ffn_t(const FfnArgs& a, cudaStream_t s) {
  const int sms = num_sms();
  {
    const size_t smem = ffn_smem(a.TT, a.H, 2);
    auto kern = gateup_kernel<FMT>;
    int per_sm = 0;
    cudaError_t err = occupancy(reinterpret_cast<const void*>(kern), smem, &per_sm);
    if (err != cudaSuccess) return err;
    const int64_t max_items = (int64_t)a.max_tiles * (a.I / 32);
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(max_items, (int64_t)std::max(per_sm, 1) * sms));
    trace_record(s);
    note_launch();
    kern<<<grid, kThreads, smem, s>>>(a);
    err = cudaGetLastError();
    trace_record(s);
    if (err != cudaSuccess) return err;
  }
  {
    const size_t smem = ffn_smem(a.TT, a.I, 1);
    auto kern = down_kernel<FMT>;
    int per_sm = 0;
    cudaError_t err = occupancy(reinterpret_cast<const void*>(kern), smem, &per_sm);
    if (err != cudaSuccess) return err;
    const int64_t max_items = (int64_t)a.max_tiles * (a.H / 128);
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(max_items, (int64_t)std::max(per_sm, 1) * sms));
    trace_record(s);
    note_launch();
    kern<<<grid, kThreads, smem, s>>>(a);
    err = cudaGetLastError();
    trace_record(s);
    return err;
  }
}

}  // namespace

int pick_tile_tokens(int T, int H) {
  int tt = T < 16 ? (T > 0 ? T : 1) : 16;
  const size_t budget = 80 * 1024;
  while (tt > 1 && ffn_smem(tt, H, 2) > budget) --tt;
  return tt;
}

cudaError_t launch_expert_ffn(const FfnArgs& a, cudaStream_t s) {
  switch (a.fmt) {
    case kQ4K: return launch_ffn_t<kQ4K>(a, s);
    case kQ2K: return launch_ffn_t<kQ2K>(a, s);
    case kQ5K: return launch_ffn_t<kQ5K>(a, s);
    case kQ3K: return launch_ffn_t<kQ3K>(a, s);
    case kQ6K: return launch_ffn_t<kQ6K>(a, s);
    case kIQ2G: return launch_ffn_t<kIQ2G>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_combine(const float* y, const float* gates, int T, int H, int k, int S, const float* residual,
                           float* out, cudaStream_t s) {
  const int64_t n = (int64_t)T * (H / 4);
  if (n == 0) return cudaSuccess;
  note_launch();
  combine_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(y, gates, T, H, k, S, residual, out);
  return cudaGetLastError();
}

// A bounded wait on a flag that nothing sets: runs out after limit_ns of
// wall time (%globaltimer), records MOE_ERR_DEVICE_TIMEOUT and returns, like
// every wait of the library's kernels.
__global__ void debug_wait_kernel(int* status, const unsigned* flag, long long limit_ns) {
  unsigned long long t0, t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  while (*reinterpret_cast<const volatile unsigned*>(flag) != 0x7FEEDBEEu) {
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if ((long long)(t - t0) > limit_ns) {
      set_status(status, MOE_ERR_DEVICE_TIMEOUT);
      return;
    }
    __nanosleep(1000);
  }
}

cudaError_t launch_debug_wait(int* status, const unsigned* flag, long long limit_ns, cudaStream_t s) {
  note_launch();
  debug_wait_kernel<<<1, 1, 0, s>>>(status, flag, limit_ns);
  return cudaGetLastError();
}

cudaError_t launch_debug_dots(int fmt, const void* w, int N, int K, const int8_t* q, int T, int32_t* isum,
                              int32_t* bsum, cudaStream_t s) {
  const int blocks = (N / 32) * (K / 256);
  note_launch();
  const uint8_t* wb = static_cast<const uint8_t*>(w);
  switch (fmt) {
    case kQ4K: debug_dots_kernel<kQ4K><<<blocks, 32, 0, s>>>(wb, N, K, q, T, isum, bsum); break;
    case kQ2K: debug_dots_kernel<kQ2K><<<blocks, 32, 0, s>>>(wb, N, K, q, T, isum, bsum); break;
    case kQ5K: debug_dots_kernel<kQ5K><<<blocks, 32, 0, s>>>(wb, N, K, q, T, isum, bsum); break;
    case kQ3K: debug_dots_kernel<kQ3K><<<blocks, 32, 0, s>>>(wb, N, K, q, T, isum, bsum); break;
    case kQ6K: debug_dots_kernel<kQ6K><<<blocks, 32, 0, s>>>(wb, N, K, q, T, isum, bsum); break;
    default: debug_dots_kernel<kIQ2G><<<blocks, 32, 0, s>>>(wb, N, K, q, T, isum, bsum); break;
  }
  return cudaGetLastError();
}

int num_sms() {
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 1;
  }
  return sms;
}

}  // namespace moe
