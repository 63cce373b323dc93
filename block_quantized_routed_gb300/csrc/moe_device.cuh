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
constexpr int kQ5K = MOE_FMT_Q5K;
constexpr int kQ3K = MOE_FMT_Q3K;
constexpr int kQ6K = MOE_FMT_Q6K;
constexpr int kIQ2G = MOE_FMT_IQ2G;

// Field sizes of a format (per row of a 32-row slab): header (d | dmin << 16,
// or d alone), scale/min bytes, code bytes; the slab places the 32 headers,
// then the 32 scale/min records, then the 16-byte code lines.  kOff: the
// code offset o of the symmetric formats (weight = d * sc * (q - o)).
template <int HB, int SMB, int CB, int NSUB, int OFF>
struct FmtBase {
  static constexpr int kHdrBytes = HB;
  static constexpr int kSmBytes = SMB;
  static constexpr int kSbBytes = HB + SMB + CB;
  static constexpr int kSlabBytes = 32 * kSbBytes;
  static constexpr int kNSub = NSUB;
  static constexpr int kSubLen = 256 / NSUB;
  static constexpr int kLines = CB / 16;       // 16-byte code lines per row
  static constexpr int kSmOff = 32 * HB;
  static constexpr int kCodeOff = 32 * (HB + SMB);
  static constexpr int kOff = OFF;
  static constexpr bool kSym = OFF != 0;
  static constexpr int kSmWords = (SMB + 3) / 4;
};

template <int FMT>
struct Fmt;
template <> struct Fmt<kQ4K> : FmtBase<4, 12, 128, 8, 0> {};   // 144 B, slab 4608
template <> struct Fmt<kQ2K> : FmtBase<4, 16, 64, 16, 0> {};   // 84 B, slab 2688
template <> struct Fmt<kQ5K> : FmtBase<4, 12, 160, 8, 0> {};   // 176 B, slab 5632
template <> struct Fmt<kQ3K> : FmtBase<2, 12, 96, 16, 4> {};   // 110 B, slab 3520
template <> struct Fmt<kQ6K> : FmtBase<2, 16, 192, 16, 32> {}; // 210 B, slab 6720
template <> struct Fmt<kIQ2G> : FmtBase<2, 4, 64, 8, 0> {};     // 70 B, slab 2240 (no min: mn = 0)

// The IQ2-style grid, built at compile time from its rule: the 256 vectors
// of {1, 3, 5}^8 with the smallest sums of squares, equal sums in increasing
// base-3 order of the digits (v - 1) / 2 with element 0 the most significant
// digit.  Entry u packs element i into byte i.
struct Iq2gGrid {
  uint64_t v[256];
};
constexpr Iq2gGrid make_iq2g_grid() {
  Iq2gGrid g{};
  int sums[6561] = {};
  uint64_t packed[6561] = {};
  for (int t = 0; t < 6561; ++t) {
    int x = t;
    for (int i = 7; i >= 0; --i) {  // the lowest base-3 digit is element 7
      const int v = 1 + 2 * (x % 3);
      x /= 3;
      sums[t] += v * v;
      packed[t] |= (uint64_t)v << (8 * i);
    }
  }
  int n = 0;
  for (int ss = 8; n < 256; ss += 8)  // every sum of squares is 8 + 8a + 24b
    for (int t = 0; t < 6561 && n < 256; ++t)
      if (sums[t] == ss) g.v[n++] = packed[t];
  return g;
}
__device__ const Iq2gGrid g_iq2g_grid = make_iq2g_grid();
// A per-CTA copy in shared memory: the kernels of the grid format fill it
// at their start (stage_format_tables) and the unpacker reads it there
// (random 8-byte lookups conflict less in shared-memory banks than they
// hit distinct L1 lines).
__shared__ uint64_t s_iq2g_grid[256];
// and the byte masks of the 128 sign bytes: byte i is 0xFF when element i is
// negative, the 8th sign (byte 7) set when bits 0-6 hold an odd count
__shared__ uint64_t s_iq2g_sign[128];
constexpr int kIq2gSmemBytes = (256 + 128) * 8;

// Every thread of the CTA calls this at the kernel's start (it ends with a barrier).
template <int FMT>
__device__ __forceinline__ void stage_format_tables() {
  if constexpr (FMT == kIQ2G) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) s_iq2g_grid[i] = g_iq2g_grid.v[i];
    for (int s7 = threadIdx.x; s7 < 128; s7 += blockDim.x) {
      const uint32_t s8 = (uint32_t)s7 | ((uint32_t)(__popc(s7) & 1) << 7);
      uint64_t m = 0;
      for (int i = 0; i < 8; ++i)
        if ((s8 >> i) & 1) m |= (uint64_t)0xFF << (8 * i);
      s_iq2g_sign[s7] = m;
    }
    __syncthreads();
  }
}

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

__device__ __forceinline__ uint32_t ld_stream16(const void* p) {
  unsigned short v;
  asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

// ---- one row's super-block, held in registers ------------------------------
template <int FMT>
struct SbRegs {
  uint4 code[Fmt<FMT>::kLines];
  uint32_t dm;                 // d | dmin << 16 (fp16 bits); d alone for the symmetric formats
  uint32_t sm[Fmt<FMT>::kSmWords];
};

// The header of lane r's row, the scale/min words and the code lines from a
// slab in global memory (slab = matrix + (rg*nb + b) * kSlabBytes).
template <int FMT>
__device__ __forceinline__ void load_sb(const uint8_t* slab, int r, SbRegs<FMT>& s) {
  using F = Fmt<FMT>;
#pragma unroll
  for (int l = 0; l < F::kLines; ++l) s.code[l] = ld_stream128(slab + F::kCodeOff + 512 * l + 16 * r);
  if constexpr (F::kHdrBytes == 4) s.dm = ld_stream32(slab + 4 * r);
  else s.dm = ld_stream16(slab + 2 * r);
  if constexpr (F::kSmBytes == 4) {
    s.sm[0] = ld_stream32(slab + F::kSmOff + 4 * r);
  } else if constexpr (F::kSmBytes == 12) {
#pragma unroll
    for (int i = 0; i < 3; ++i) s.sm[i] = ld_stream32(slab + F::kSmOff + 12 * r + 4 * i);
  } else {
    uint4 v = ld_stream128(slab + F::kSmOff + 16 * r);
    s.sm[0] = v.x; s.sm[1] = v.y; s.sm[2] = v.z; s.sm[3] = v.w;
  }
}

// The same fields from a slab staged in shared memory (code lines are read
// where they are used).
template <int FMT>
__device__ __forceinline__ void load_sb_head(const uint8_t* slab, int r, SbRegs<FMT>& s) {
  using F = Fmt<FMT>;
  if constexpr (F::kHdrBytes == 4) s.dm = *reinterpret_cast<const uint32_t*>(slab + 4 * r);
  else s.dm = *reinterpret_cast<const uint16_t*>(slab + 2 * r);
  if constexpr (F::kSmBytes == 4) {
    s.sm[0] = *reinterpret_cast<const uint32_t*>(slab + F::kSmOff + 4 * r);
  } else if constexpr (F::kSmBytes == 12) {
#pragma unroll
    for (int i = 0; i < 3; ++i) s.sm[i] = *reinterpret_cast<const uint32_t*>(slab + F::kSmOff + 12 * r + 4 * i);
  } else {
    const uint4 v = *reinterpret_cast<const uint4*>(slab + F::kSmOff + 16 * r);
    s.sm[0] = v.x; s.sm[1] = v.y; s.sm[2] = v.z; s.sm[3] = v.w;
  }
}

// Scale and min-term coefficient of sub-block j in the raw-code form
//   y_b = d_a * (d * sum_j sc_j * isum_j - m_scale * sum_j mn_j * bsum_j)
// (isum_j over the raw codes): mn_j is the min (m_scale = dmin) or, for the
// symmetric formats, o * sc_j (m_scale = d).
template <int FMT>
__device__ __forceinline__ void sb_scale_min(const SbRegs<FMT>& s, int j, int& sc, int& mn) {
  if constexpr (FMT == kQ4K || FMT == kQ5K || FMT == kQ3K) {
    // 96-bit little-endian string: field f = bits 6f..6f+5 (Q4_K/Q5_K: scale
    // j = field j, min j = field 8 + j; Q3_K: u_j = field j, scale u_j - 32)
    uint64_t lo = (uint64_t)s.sm[0] | ((uint64_t)s.sm[1] << 32);
    uint64_t hi = (uint64_t)(s.sm[1] >> 16) | ((uint64_t)s.sm[2] << 16);
    if constexpr (FMT == kQ3K) {
      const uint64_t bits = j < 8 ? lo >> (6 * j) : hi >> (6 * (j - 8));
      sc = (int)(bits & 63) - 32;
      mn = 4 * sc;
    } else {
      sc = (int)((lo >> (6 * j)) & 63);
      mn = (int)((hi >> (6 * j)) & 63);
    }
  } else if constexpr (FMT == kQ2K) {
    uint32_t byte = (s.sm[j >> 2] >> (8 * (j & 3))) & 0xFF;
    sc = (int)(byte & 15);
    mn = (int)(byte >> 4);
  } else if constexpr (FMT == kIQ2G) {  // nibble j of the scale word: scale 2t + 1, no min
    sc = 2 * (int)((s.sm[0] >> (4 * j)) & 15) + 1;
    mn = 0;
  } else {  // Q6_K: int8 scales
    sc = (int)(int8_t)((s.sm[j >> 2] >> (8 * (j & 3))) & 0xFF);
    mn = 32 * sc;
  }
}

__device__ __forceinline__ float half_lo(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w & 0xFFFF))); }
__device__ __forceinline__ float half_hi(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w >> 16))); }

// d and the min-term scale (dmin, or d for the symmetric formats) of a header
template <int FMT>
__device__ __forceinline__ void sb_d_mscale(uint32_t dm, float& d, float& ms) {
  d = half_lo(dm);
  ms = Fmt<FMT>::kSym ? d : half_hi(dm);
}

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

// The raw codes of sub-block j as bytes of 32-bit words, in the order of the
// activation codes they meet (word k = codes 4k..4k+3 of the sub-block; for
// 32-code sub-blocks words 0-3 are codes 0..15 and words 4-7 codes 16..31).
// line(l) gives the row's 16-byte code line l (from registers or shared
// memory).  The bit placement is that of synth/layout.py.
template <int FMT, class Line>
__device__ __forceinline__ void sub_words(Line line, int j, uint32_t (&w)[Fmt<FMT>::kSubLen / 4]) {
  if constexpr (FMT == kQ4K || FMT == kQ5K) {
    uint32_t lo[4], hi[4];
    mask_q4k(line(j), lo, hi);
    if constexpr (FMT == kQ5K) {  // 5th bits: line 8 + j/4, bit 2(j%4) + h of byte i -> code i + 16h
      const uint4 h = line(8 + (j >> 2));
      const uint32_t hw[4] = {h.x, h.y, h.z, h.w};
      const int sh = 2 * (j & 3);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        lo[k] |= ((hw[k] >> sh) & 0x01010101u) << 4;
        hi[k] |= ((hw[k] >> (sh + 1)) & 0x01010101u) << 4;
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      w[k] = lo[k];
      w[4 + k] = hi[k];
    }
  } else if constexpr (FMT == kQ2K || FMT == kQ3K) {
    mask_q2k(line(j >> 2), j, w);
    if constexpr (FMT == kQ3K) {  // 3rd bits: word (j/2)%4 of line 4 + j/8, bit p + 4(j%2) of byte m -> code 4p + m
      const uint4 h = line(4 + (j >> 3));
      const int wi = (j >> 1) & 3;
      const uint32_t hv = wi == 0 ? h.x : wi == 1 ? h.y : wi == 2 ? h.z : h.w;
      const int sh = 4 * (j & 1);
#pragma unroll
      for (int p = 0; p < 4; ++p) w[p] |= ((hv >> (p + sh)) & 0x01010101u) << 2;
    }
  } else if constexpr (FMT == kIQ2G) {
    // sub-block j = groups 4j..4j+3: their grid indices are word j%4 of line
    // j/4, their sign bytes word j%4 of line 2 + j/4.  Each group's 8
    // magnitudes come from the grid; a minus sign negates a byte as
    // (v ^ 0xFF) - 0xFF, with the byte masks of the sign byte from a table
    // (the 8th sign makes the count of minus signs even).
    const uint4 li = line(j >> 2), ls = line(2 + (j >> 2));
    const int ws = j & 3;
    const uint32_t iw = ws == 0 ? li.x : ws == 1 ? li.y : ws == 2 ? li.z : li.w;
    const uint32_t sw = ws == 0 ? ls.x : ws == 1 ? ls.y : ws == 2 ? ls.z : ls.w;
#pragma unroll
    for (int gg = 0; gg < 4; ++gg) {
      const uint64_t v = s_iq2g_grid[(iw >> (8 * gg)) & 0xFF];
      const uint64_t m = s_iq2g_sign[(sw >> (8 * gg)) & 0x7Fu];
      const uint32_t mlo = (uint32_t)m, mhi = (uint32_t)(m >> 32);
      w[2 * gg] = __vsub4((uint32_t)v ^ mlo, mlo);
      w[2 * gg + 1] = __vsub4((uint32_t)(v >> 32) ^ mhi, mhi);
    }
  } else {  // Q6_K: low nibbles in line j/2 (nibble j%2), high 2 bits in line 8 + j/4 (bits 2(j%4)..)
    const uint4 lo = line(j >> 1), hi = line(8 + (j >> 2));
    const uint32_t lw[4] = {lo.x, lo.y, lo.z, lo.w}, hw[4] = {hi.x, hi.y, hi.z, hi.w};
    const int sl = 4 * (j & 1), sh = 2 * (j & 3);
#pragma unroll
    for (int k = 0; k < 4; ++k) w[k] = ((lw[k] >> sl) & 0x0F0F0F0Fu) | (((hw[k] >> sh) & 0x03030303u) << 4);
  }
}

// dp4a of a sub-block's code words with its activation codes (a: the first
// code of the sub-block, 16-byte aligned)
template <int NW>
__device__ __forceinline__ int words_dot(const uint32_t (&w)[NW], const int8_t* a) {
  int i = 0;
#pragma unroll
  for (int k = 0; k < NW; k += 4) {
    const int4 v = *reinterpret_cast<const int4*>(a + 4 * k);
    i = __dp4a((int)w[k], v.x, i);
    i = __dp4a((int)w[k + 1], v.y, i);
    i = __dp4a((int)w[k + 2], v.z, i);
    i = __dp4a((int)w[k + 3], v.w, i);
  }
  return i;
}

// Integer dot of sub-block j (raw codes) with the 256 activation codes of the same block.
template <int FMT>
__device__ __forceinline__ int sub_isum(const SbRegs<FMT>& s, int j, const int8_t* act) {
  using F = Fmt<FMT>;
  uint32_t w[F::kSubLen / 4];
  sub_words<FMT>([&](int l) { return s.code[l]; }, j, w);
  return words_dot(w, act + F::kSubLen * j);
}

// Sum of the 16-code sums of sub-block j (one or two of them)
template <int FMT>
__device__ __forceinline__ int sub_bsum(const int16_t* bsp, int j) {
  if constexpr (Fmt<FMT>::kSubLen == 32) return (int)bsp[2 * j] + (int)bsp[2 * j + 1];
  else return (int)bsp[j];
}

// One super-block's contribution to `cnt` tokens for the Q5_K/Q3_K/Q6_K-style
// formats; the code words of every sub-block come from line(l) once per
// super-block.  Asymmetric: d_a (d sum sc isum - dmin sum mn bsum); symmetric:
// d_a d sum_j sc_j (isum_j - o bsum_j), the offset applied in integers.
template <int FMT, class Line>
__device__ __forceinline__ void sb_accum_words(Line line, const SbRegs<FMT>& s, const int8_t* act, const int16_t* bs,
                                               const float* d, const int* act_off, int b, int cnt, float* acc,
                                               int lane) {
  using F = Fmt<FMT>;
  constexpr int NW = F::kSubLen / 4;
  int sc[F::kNSub], mn[F::kNSub];
#pragma unroll
  for (int j = 0; j < F::kNSub; ++j) sb_scale_min<FMT>(s, j, sc[j], mn[j]);
  float dw, ms;
  sb_d_mscale<FMT>(s.dm, dw, ms);
  uint32_t wd[F::kNSub][NW];
#pragma unroll
  for (int j = 0; j < F::kNSub; ++j) sub_words<FMT>(line, j, wd[j]);
#pragma unroll 1
  for (int t = 0; t < cnt; ++t) {
    const int o = act_off[t];
    const int8_t* a = act + o + 256 * b;
    const int16_t* bsp = bs + o / 16 + 16 * b;
    int S = 0, M = 0;
#pragma unroll
    for (int j = 0; j < F::kNSub; ++j) {
      const int isum = words_dot(wd[j], a + F::kSubLen * j);
      if constexpr (F::kSym) {
        S += sc[j] * (isum - F::kOff * sub_bsum<FMT>(bsp, j));
      } else {
        S += sc[j] * isum;
        M += mn[j] * sub_bsum<FMT>(bsp, j);
      }
    }
    if constexpr (F::kSym) acc[t * 32 + lane] += d[o / 256 + b] * (dw * (float)S);
    else acc[t * 32 + lane] += d[o / 256 + b] * fmaf(dw, (float)S, -ms * (float)M);
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
  if constexpr (FMT != kQ4K && FMT != kQ2K) {
    sb_accum_words<FMT>([&](int l) { return s.code[l]; }, s, act, bs, d, act_off, b, cnt, acc, lane);
  } else {
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
