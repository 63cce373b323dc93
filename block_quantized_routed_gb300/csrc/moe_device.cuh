// Device-side building blocks of the block-quantized MoE layer (sm_103a).
//
//  * decoding of the Q4_K-style / Q2_K-style super-block fields from the slab
//    layout (one lane = one row of a 32-row group);
//  * the integer sub-block dot product sum_i q_w[i] * q_a[i] on dp4a, and the
//    per-super-block combination  d_a * (d_w * sum_j sc_j*isum_j
//                                        - dmin * sum_j mn_j*bsum_j);
//  * the warp-level q8_K quantizer of a 256-element block.
//
// Sources: Pulsar README, "Fidelity notes" (every matmul on q8_0/q8_K
// activations with integer dp4a dots) and "What it does today" (Q4_K/Q6_K
// matmuls on q8_K activations); the Q4_K-style and Q2_K-style field lists
// (fp16 d and dmin, per-sub-block scale and min, 4-/2-bit codes, weight =
// d*scale*q - dmin*min) are the workload definitions.
#pragma once

#include <climits>
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "moe_q8k.h"

namespace moe {

constexpr int kQ4K = MOE_FMT_Q4K;
constexpr int kQ2K = MOE_FMT_Q2K;

template <int FMT>
struct Fmt;

template <>
struct Fmt<kQ4K> {
  static constexpr int kSbBytes = 144;
  static constexpr int kSlabBytes = 32 * 144;  // 4608
  static constexpr int kNSub = 8;
  static constexpr int kSubLen = 32;
  static constexpr int kLines = 8;             // 16-byte code lines per row
  static constexpr int kSmOff = 128;
  static constexpr int kCodeOff = 512;
};

template <>
struct Fmt<kQ2K> {
  static constexpr int kSbBytes = 84;
  static constexpr int kSlabBytes = 32 * 84;   // 2688
  static constexpr int kNSub = 16;
  static constexpr int kSubLen = 16;
  static constexpr int kLines = 4;
  static constexpr int kSmOff = 128;
  static constexpr int kCodeOff = 640;
};

// ---- streaming loads of weight bytes (read once: keep them out of L1) ------
__device__ __forceinline__ uint4 ld_stream128(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ld_stream32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// ---- one row's super-block, held in registers ------------------------------
template <int FMT>
struct SbRegs {
  uint4 code[Fmt<FMT>::kLines];
  uint32_t dm;                 // d | dmin << 16 (fp16 bits)
  uint32_t sm[FMT == kQ4K ? 3 : 4];
};

// Load super-block b of lane r's row from a slab (slab = matrix + (rg*nb + b) * kSlabBytes).
template <int FMT>
__device__ __forceinline__ void load_sb(const uint8_t* slab, int r, SbRegs<FMT>& s) {
  using F = Fmt<FMT>;
#pragma unroll
  for (int l = 0; l < F::kLines; ++l) s.code[l] = ld_stream128(slab + F::kCodeOff + 512 * l + 16 * r);
  s.dm = ld_stream32(slab + 4 * r);
  if constexpr (FMT == kQ4K) {
#pragma unroll
    for (int i = 0; i < 3; ++i) s.sm[i] = ld_stream32(slab + F::kSmOff + 12 * r + 4 * i);
  } else {
    uint4 v = ld_stream128(slab + F::kSmOff + 16 * r);
    s.sm[0] = v.x; s.sm[1] = v.y; s.sm[2] = v.z; s.sm[3] = v.w;
  }
}

// scale and min of sub-block j
template <int FMT>
__device__ __forceinline__ void sb_scale_min(const SbRegs<FMT>& s, int j, int& sc, int& mn) {
  if constexpr (FMT == kQ4K) {
    // 96-bit little-endian string: scale j = bits 6j.., min j = bits 48+6j..
    uint64_t lo = (uint64_t)s.sm[0] | ((uint64_t)s.sm[1] << 32);
    uint64_t hi = (uint64_t)(s.sm[1] >> 16) | ((uint64_t)s.sm[2] << 16);
    sc = (int)((lo >> (6 * j)) & 63);
    mn = (int)((hi >> (6 * j)) & 63);
  } else {
    uint32_t byte = (s.sm[j >> 2] >> (8 * (j & 3))) & 0xFF;
    sc = (int)(byte & 15);
    mn = (int)(byte >> 4);
  }
}

__device__ __forceinline__ float half_lo(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w & 0xFFFF))); }
__device__ __forceinline__ float half_hi(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w >> 16))); }

// ---- the integer sub-block dot, shared by every kernel and the test hook ----
// Q4_K-style code line j: byte i = code i (low nibble) | code i+16 (high
// nibble); lo[w] / hi[w] hold codes 4w..4w+3 / 16+4w..16+4w+3 as bytes.
__device__ __forceinline__ void mask_q4k(const uint4 c, uint32_t (&lo)[4], uint32_t (&hi)[4]) {
  lo[0] = c.x & 0x0F0F0F0Fu; hi[0] = (c.x >> 4) & 0x0F0F0F0Fu;
  lo[1] = c.y & 0x0F0F0F0Fu; hi[1] = (c.y >> 4) & 0x0F0F0F0Fu;
  lo[2] = c.z & 0x0F0F0F0Fu; hi[2] = (c.z >> 4) & 0x0F0F0F0Fu;
  lo[3] = c.w & 0x0F0F0F0Fu; hi[3] = (c.w >> 4) & 0x0F0F0F0Fu;
}
// sum of the 32 products of a Q4_K-style sub-block with its activation codes
// (alo: codes 0..15, ahi: codes 16..31 of the sub-block)
__device__ __forceinline__ int isum_q4k(const uint32_t (&lo)[4], const uint32_t (&hi)[4], const int4 alo,
                                        const int4 ahi) {
  int i = 0;
  i = __dp4a((int)lo[0], alo.x, i);
  i = __dp4a((int)lo[1], alo.y, i);
  i = __dp4a((int)lo[2], alo.z, i);
  i = __dp4a((int)lo[3], alo.w, i);
  i = __dp4a((int)hi[0], ahi.x, i);
  i = __dp4a((int)hi[1], ahi.y, i);
  i = __dp4a((int)hi[2], ahi.z, i);
  i = __dp4a((int)hi[3], ahi.w, i);
  return i;
}
// Q2_K-style sub-block j: word j%4 of code line j/4; bits 2p..2p+1 of byte m
// hold code 4p+m; w[p] holds codes 4p..4p+3 as bytes.
__device__ __forceinline__ void mask_q2k(const uint4 line, int j, uint32_t (&w)[4]) {
  const uint32_t x = (j & 3) == 0 ? line.x : (j & 3) == 1 ? line.y : (j & 3) == 2 ? line.z : line.w;
  w[0] = x & 0x03030303u;
  w[1] = (x >> 2) & 0x03030303u;
  w[2] = (x >> 4) & 0x03030303u;
  w[3] = (x >> 6) & 0x03030303u;
}
__device__ __forceinline__ int isum_q2k(const uint32_t (&w)[4], const int4 a) {
  int i = 0;
  i = __dp4a((int)w[0], a.x, i);
  i = __dp4a((int)w[1], a.y, i);
  i = __dp4a((int)w[2], a.z, i);
  i = __dp4a((int)w[3], a.w, i);
  return i;
}

// Integer dot of sub-block j with the 256 activation codes of the same block.
template <int FMT>
__device__ __forceinline__ int sub_isum(const SbRegs<FMT>& s, int j, const int8_t* act) {
  if constexpr (FMT == kQ4K) {
    uint32_t lo[4], hi[4];
    mask_q4k(s.code[j], lo, hi);
    return isum_q4k(lo, hi, *reinterpret_cast<const int4*>(act + 32 * j),
                    *reinterpret_cast<const int4*>(act + 32 * j + 16));
  } else {
    uint32_t w[4];
    mask_q2k(s.code[j >> 2], j, w);
    return isum_q2k(w, *reinterpret_cast<const int4*>(act + 16 * j));
  }
}

// Contribution of super-block b of one row (this lane's) to `cnt` tokens:
//   acc[t*32 + lane] += d_a(t) * (d_w * S_t - dmin * M_t),
//   S_t = sum_j sc_j * isum_j(t),  M_t = sum_j mn_j * bsum_j(t).
// The code words are masked and the scales/mins extracted once per
// super-block; the token loop is a runtime loop (small code), and the
// accumulators live in shared memory, one slot per (token, lane), owned by
// the calling warp.  act_off[t]: byte offset of token t's q8_K row in `act`
// (row stride K); its 16-code sums start at bs + act_off[t] / 16 and its block
// scales at d + act_off[t] / 256.
template <int FMT>
__device__ __forceinline__ void sb_accum(const SbRegs<FMT>& s, const int8_t* act, const int16_t* bs, const float* d,
                                         const int* act_off, int b, int cnt, float* acc, int lane) {
  using F = Fmt<FMT>;
  int sc[F::kNSub], mn[F::kNSub];
#pragma unroll
  for (int j = 0; j < F::kNSub; ++j) sb_scale_min<FMT>(s, j, sc[j], mn[j]);
  const float dw = half_lo(s.dm), dmin = half_hi(s.dm);
  if constexpr (FMT == kQ4K) {
    uint32_t lo[8][4], hi[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) mask_q4k(s.code[j], lo[j], hi[j]);
#pragma unroll 1
    for (int t = 0; t < cnt; ++t) {
      const int o = act_off[t];
      const int8_t* a = act + o + 256 * b;
      const int16_t* bsp = bs + o / 16 + 16 * b;
      int S = 0, M = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int4 alo = *reinterpret_cast<const int4*>(a + 32 * j);
        const int4 ahi = *reinterpret_cast<const int4*>(a + 32 * j + 16);
        S += sc[j] * isum_q4k(lo[j], hi[j], alo, ahi);
        M += mn[j] * ((int)bsp[2 * j] + (int)bsp[2 * j + 1]);
      }
      acc[t * 32 + lane] += d[o / 256 + b] * fmaf(dw, (float)S, -dmin * (float)M);
    }
  } else {
    uint32_t w[16][4];
#pragma unroll
    for (int j = 0; j < 16; ++j) mask_q2k(s.code[j >> 2], j, w[j]);
#pragma unroll 1
    for (int t = 0; t < cnt; ++t) {
      const int o = act_off[t];
      const int8_t* a = act + o + 256 * b;
      const int16_t* bsp = bs + o / 16 + 16 * b;
      int S = 0, M = 0;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        S += sc[j] * isum_q2k(w[j], *reinterpret_cast<const int4*>(a + 16 * j));
        M += mn[j] * (int)bsp[j];
      }
      acc[t * 32 + lane] += d[o / 256 + b] * fmaf(dw, (float)S, -dmin * (float)M);
    }
  }
}

// ---- q8_K of one 256-element block by one warp ------------------------------
// lane holds elements 8*lane .. 8*lane+7 in v[8].  Writes 8 codes per lane,
// the block scale (lane 0) and the 16 sums of 16 codes (even lanes).
// d = max|x| / 127 and q = round-half-away(x / d) with IEEE fp32 division
// (this file is compiled without fast-math), q = 0 when d == 0.
__device__ __forceinline__ void q8k_block_warp(const float (&v)[8], int lane, int8_t* q, float* d,
                                               int16_t* bs16) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float db = amax / 127.0f;
  int codes[8];
  int sum = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float r = 0.0f;
    if (db != 0.0f) r = fminf(127.0f, fmaxf(-127.0f, roundf(v[i] / db)));
    codes[i] = (int)r;
    sum += codes[i];
  }
  uint32_t lo = (uint32_t)(codes[0] & 0xFF) | ((uint32_t)(codes[1] & 0xFF) << 8) |
                ((uint32_t)(codes[2] & 0xFF) << 16) | ((uint32_t)(codes[3] & 0xFF) << 24);
  uint32_t hi = (uint32_t)(codes[4] & 0xFF) | ((uint32_t)(codes[5] & 0xFF) << 8) |
                ((uint32_t)(codes[6] & 0xFF) << 16) | ((uint32_t)(codes[7] & 0xFF) << 24);
  *reinterpret_cast<uint2*>(q + 8 * lane) = make_uint2(lo, hi);
  sum += __shfl_xor_sync(0xffffffffu, sum, 1);
  if (bs16 && (lane & 1) == 0) bs16[lane >> 1] = (int16_t)sum;
  if (lane == 0) *d = db;
}

// slot index p -> token (p = t*k + s routed; p = T*k + sh*T + t shared)
__device__ __forceinline__ int token_of_slot(int p, int T, int k) {
  const int routed = T * k;
  return p < routed ? p / k : (p - routed) % T;
}

__device__ __forceinline__ void set_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// ---------------------------------------------------------------- top-k
// Order-preserving map of a float logit to an unsigned key: larger logit,
// larger key.  NaN maps to 1 (below every number); key 0 marks a taken entry.
__device__ __forceinline__ uint32_t logit_key(float v) {
  if (v != v) return 1u;
  if (v == 0.0f) v = 0.0f;  // -0 and +0 are the same logit
  const uint32_t b = __float_as_uint(v);
  const uint32_t k = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return k < 1u ? 1u : k;
}
__device__ __forceinline__ float key_logit(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Top-k of one token by one warp.  Lane l owns experts e = l + 32*i
// (i < NPER, E <= 32*NPER); it sorts its own (key, index) pairs once
// (larger key first, equal keys: lower index first), then k+1 rounds merge
// the lanes' heads with warp reductions: the largest key wins, equal keys go
// to the lower expert index.  Gives the k ids in descending logit order, the
// gates renormalised over the k, and the gap l_(k) - l_(k+1).
template <int NPER>
__device__ __forceinline__ void warp_topk_n(const float* l, int E, int k, int route, int lane, int32_t* ids,
                                            float* gates, float* gap) {
  uint32_t key[NPER];
  int idx[NPER];
#pragma unroll
  for (int i = 0; i < NPER; ++i) {
    const int e = lane + 32 * i;
    key[i] = e < E ? logit_key(__ldcg(l + e)) : 0u;
    idx[i] = e < E ? e : INT_MAX;
  }
  // insertion sort of the lane's entries (small NPER; fully unrolled)
#pragma unroll
  for (int i = 1; i < NPER; ++i) {
#pragma unroll
    for (int j = i; j > 0; --j) {
      const bool sw = key[j] > key[j - 1] || (key[j] == key[j - 1] && idx[j] < idx[j - 1]);
      const uint32_t tk = sw ? key[j - 1] : key[j];
      const int ti = sw ? idx[j - 1] : idx[j];
      key[j - 1] = sw ? key[j] : key[j - 1];
      idx[j - 1] = sw ? idx[j] : idx[j - 1];
      key[j] = tk;
      idx[j] = ti;
    }
  }
  // lane r keeps round r's winner; everything stays in registers
  float my_v = 0.0f;
  int my_e = 0;
  float next_v = -INFINITY;
  const int rounds = k < E ? k + 1 : k;
  for (int r = 0; r < rounds; ++r) {
    const uint32_t mk = __reduce_max_sync(0xffffffffu, key[0]);
    const uint32_t cand = key[0] == mk ? (uint32_t)idx[0] : 0xFFFFFFFFu;
    const int win = (int)__reduce_min_sync(0xffffffffu, cand);
    if (r < k) {
      if (lane == r) {
        my_v = key_logit(mk);
        my_e = win;
      }
      if ((win & 31) == lane) {  // the owner drops its head
#pragma unroll
        for (int i = 0; i + 1 < NPER; ++i) {
          key[i] = key[i + 1];
          idx[i] = idx[i + 1];
        }
        key[NPER - 1] = 0u;
        idx[NPER - 1] = INT_MAX;
      }
    } else {
      next_v = key_logit(mk);
    }
  }
  // gates over the k selected: lane s holds selection s
  const float v0 = __shfl_sync(0xffffffffu, my_v, 0);
  float g = 0.0f;
  if (lane < k) g = route == MOE_ROUTE_SOFTMAX ? expf(my_v - v0) : 1.0f / (1.0f + expf(-my_v));
  float z = g;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  if (lane < k) {
    ids[lane] = my_e;
    gates[lane] = g / z;
  }
  const float vk = __shfl_sync(0xffffffffu, my_v, (k - 1) & 31);
  if (lane == 0 && gap) *gap = k < E ? vk - next_v : INFINITY;
}

__device__ __forceinline__ void warp_topk(const float* l, int E, int k, int route, int lane, int32_t* ids,
                                          float* gates, float* gap) {
  if (E <= 256)
    warp_topk_n<8>(l, E, k, route, lane, ids, gates, gap);
  else if (E <= 512)
    warp_topk_n<16>(l, E, k, route, lane, ids, gates, gap);
  else
    warp_topk_n<32>(l, E, k, route, lane, ids, gates, gap);
}

// ---------------------------------------------------------------- scans
// Exclusive scan in place of n ints in shared memory (any n); returns the
// total.  Every thread of the block calls it (blockDim a multiple of 32).
// Thread i owns the contiguous chunk [i*m, i*m + m), m = ceil(n / blockDim).
__device__ __forceinline__ int block_exclusive_scan(int* a, int n) {
  __shared__ int wsum[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
  const int m = (n + blockDim.x - 1) / blockDim.x;
  const int i0 = tid * m, i1 = min(i0 + m, n);
  int s = 0;
  for (int i = i0; i < i1; ++i) s += a[i];
  int x = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int v = lane < nw ? wsum[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += y;
    }
    wsum[lane] = v;
  }
  __syncthreads();
  int run = x - s + (warp > 0 ? wsum[warp - 1] : 0);
  const int total = wsum[nw - 1];
  for (int i = i0; i < i1; ++i) {
    const int v = a[i];
    a[i] = run;
    run += v;
  }
  __syncthreads();
  return total;
}

}  // namespace moe
