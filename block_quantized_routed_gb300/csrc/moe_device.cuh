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

// Integer dot of sub-block j of a super-block with the activation codes of the
// same 256-column block (act: 16-byte aligned, 256 codes; any state space).
template <int FMT>
__device__ __forceinline__ int sub_isum(const SbRegs<FMT>& s, int j, const int8_t* act) {
  int acc = 0;
  if constexpr (FMT == kQ4K) {
    // code line j: byte i = code i (low nibble) | code i+16 (high nibble)
    const int4 alo = *reinterpret_cast<const int4*>(act + 32 * j);
    const int4 ahi = *reinterpret_cast<const int4*>(act + 32 * j + 16);
    const uint4 c = s.code[j];
    acc = __dp4a((int)(c.x & 0x0F0F0F0Fu), alo.x, acc);
    acc = __dp4a((int)(c.y & 0x0F0F0F0Fu), alo.y, acc);
    acc = __dp4a((int)(c.z & 0x0F0F0F0Fu), alo.z, acc);
    acc = __dp4a((int)(c.w & 0x0F0F0F0Fu), alo.w, acc);
    acc = __dp4a((int)((c.x >> 4) & 0x0F0F0F0Fu), ahi.x, acc);
    acc = __dp4a((int)((c.y >> 4) & 0x0F0F0F0Fu), ahi.y, acc);
    acc = __dp4a((int)((c.z >> 4) & 0x0F0F0F0Fu), ahi.z, acc);
    acc = __dp4a((int)((c.w >> 4) & 0x0F0F0F0Fu), ahi.w, acc);
  } else {
    // sub-block j: word j%4 of code line j/4; bits 2p..2p+1 of byte m = code 4p+m
    const uint4 line = s.code[j >> 2];
    const uint32_t w = (j & 3) == 0 ? line.x : (j & 3) == 1 ? line.y : (j & 3) == 2 ? line.z : line.w;
    const int4 a = *reinterpret_cast<const int4*>(act + 16 * j);
    acc = __dp4a((int)(w & 0x03030303u), a.x, acc);
    acc = __dp4a((int)((w >> 2) & 0x03030303u), a.y, acc);
    acc = __dp4a((int)((w >> 4) & 0x03030303u), a.z, acc);
    acc = __dp4a((int)((w >> 6) & 0x03030303u), a.w, acc);
  }
  return acc;
}

// Sum of the activation codes of sub-block j from the 16-code partial sums
// (bs16: the 16 sums of this 256-column block).
template <int FMT>
__device__ __forceinline__ int sub_bsum(const int16_t* bs16, int j) {
  if constexpr (FMT == kQ4K)
    return (int)bs16[2 * j] + (int)bs16[2 * j + 1];
  else
    return (int)bs16[j];
}

// Contribution of one super-block to one row for one token:
//   d_a * (d_w * S - dmin * M),  S = sum_j sc_j * isum_j,  M = sum_j mn_j * bsum_j
// (S and M are exact int32: |S| <= 8*63*32*15*127 < 2^31.)
template <int FMT>
__device__ __forceinline__ float sb_contrib(const SbRegs<FMT>& s, const int8_t* act, const int16_t* bs16,
                                            float da) {
  int S = 0, M = 0;
#pragma unroll
  for (int j = 0; j < Fmt<FMT>::kNSub; ++j) {
    int sc, mn;
    sb_scale_min<FMT>(s, j, sc, mn);
    S += sc * sub_isum<FMT>(s, j, act);
    M += mn * sub_bsum<FMT>(bs16, j);
  }
  const float dw = half_lo(s.dm), dmin = half_hi(s.dm);
  return da * fmaf(dw, (float)S, -dmin * (float)M);
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

}  // namespace moe
