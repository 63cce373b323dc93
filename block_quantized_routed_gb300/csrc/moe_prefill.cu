// Prefill expert FFNs on the 5th-generation tensor cores (tcgen05).
//
// For a prefill chunk every expert sees on average tens to hundreds of
// tokens, so gate/up and down are real dense contractions.  The weights stay
// block-quantized in HBM; each CTA expands one super-block column of a
// 128-row weight tile into shared memory as fp16 values sc_j * q (integers
// <= 945, exact in fp16) and the tokens' q8_K codes as fp16 (exact), and
// issues tcgen05.mma kind::f16 with fp32 accumulation in TMEM.  Every
// partial sum inside one 256-wide super-block is an integer below 2^24, so
// the accumulator holds the exact integer S = sum_j sc_j * isum_j.  The min
// term M = sum_j mn_j * bsum_j is one more K=16 MMA per super-block (Q4_K:
// bsum = 64*hi + lo split into two exact halves against mn and 64*mn; Q2_K:
// |bsum| <= 2032 is exact as is).  The epilogue warps (TMEM lane = weight
// row) read S and M and accumulate d_a * (d_w * S - dmin * M) in fp32.
//
//   D[weight row m, token n] = sum_b d_a[n,b] * (d_w[m,b] * S[m,n,b] - dmin[m,b] * M[m,n,b])
//
// gate/up: a 128-row tile is 64 gate rows + the same 64 up rows, so one CTA
// holds G and U of the same (row, token) and applies SwiGLU; h goes to
// global memory in bucket order.  down: a tile is 128 rows of H; y goes to
// the slot buffer.  h is re-quantized to q8_K between the two (the q8_K
// quantizer kernel, one row per bucket position).
//
// The pages' design does this with int8 MMA (mma.m16n8k32, "mmq-style
// grouped MoE that unpacks each expert super-block to shared memory once per
// prefill chunk and rescales per quant block in registers": Pulsar README,
// "What it does today"; Strata, 长提示 0.1.13: MMQ int8 tensor-core expert
// GEMM).  tcgen05 has no int8 kind on sm_103a, hence the exact-integer fp16
// operands.
#include <algorithm>
#include <cmath>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kPThreads = 256;
constexpr int kTileM = 128;      // weight rows per tile (MMA M)
constexpr int kTileN = 128;      // tokens per tile (MMA N, rounded to 16)
constexpr long long kWaitCycles = 2000000000ll;  // ~1 s at 2 GHz: a wait that long has failed

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Shared-memory matrix descriptor of a K-major operand without swizzle:
// core matrices of 8 rows x 16 bytes; lbo = byte distance of core matrices
// adjacent along K, sbo = along M/N.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFF) >> 4);
  d |= (uint64_t)((lbo & 0x3FFFF) >> 4) << 16;
  d |= (uint64_t)((sbo & 0x3FFFF) >> 4) << 32;
  d |= (uint64_t)1 << 46;  // fixed 0b001 in bits 46..48
  return d;                // base offset 0, no swizzle
}

// Instruction descriptor: kind::f16, A and B fp16, D fp32, K-major A and B.
__device__ __forceinline__ uint32_t idesc_f16(int M, int N) {
  uint32_t d = 0;
  d |= 1u << 4;                       // D format: f32
  // A format bits 7..9 = 0 (f16), B format bits 10..12 = 0 (f16)
  d |= (uint32_t)(N >> 3) << 17;
  d |= (uint32_t)(M >> 4) << 24;
  return d;
}

__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, bool acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"((int)acc));
}

__device__ __forceinline__ void mma_commit(uint32_t mbar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar) : "memory");
}

__device__ __forceinline__ void mbar_init(uint32_t mbar, int count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(mbar), "r"(count) : "memory");
}

// Bounded wait for phase `parity` of an mbarrier: false once about a second
// of SM clock has passed without the phase completing.
__device__ __forceinline__ bool mbar_wait(uint32_t mbar, uint32_t parity) {
  const long long t0 = clock64();
  while (true) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(mbar), "r"(parity)
        : "memory");
    if (ok) return true;
    if (clock64() - t0 > kWaitCycles) return false;
  }
}

__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 lanes x 16 consecutive fp32 columns of TMEM into 16 registers of each lane
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// byte offset of element (row, k) in a K-major canonical tile with kc core
// matrices along K (16-bit elements): core (row/8, k/8), 8 rows x 16 bytes each
__device__ __forceinline__ uint32_t canon_off(int row, int k, int kc) {
  return (uint32_t)(((row >> 3) * kc + (k >> 3)) * 128 + (row & 7) * 16 + (k & 7) * 2);
}

__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// ---------------------------------------------------------------- work items
// One CTA: per expert with tokens and a present gate pointer, its token tiles x
// weight tiles, expert by expert.
__global__ void __launch_bounds__(1024) prefill_plan_kernel(const int32_t* counts, const int32_t* offsets, int EpS,
                                                            const moe_expert_ptrs* table, int n_wtiles, PItem* items,
                                                            int32_t* n_items, int max_items) {
  __shared__ int s_n[MOE_MAX_EXPERTS + MOE_MAX_SHARED + 1];
  for (int e = threadIdx.x; e < EpS; e += blockDim.x) {
    const int c = counts[e];
    s_n[e] = (c > 0 && table[e].gate != nullptr) ? (c + kTileN - 1) / kTileN * n_wtiles : 0;
  }
  __syncthreads();
  const int total = block_exclusive_scan(s_n, EpS);
  for (int e = threadIdx.x; e < EpS; e += blockDim.x) {
    const int c = counts[e];
    if (c <= 0 || table[e].gate == nullptr) continue;
    int idx = s_n[e];
    for (int t0 = 0; t0 < c; t0 += kTileN)
      for (int w = 0; w < n_wtiles; ++w, ++idx) {
        if (idx >= max_items) continue;
        PItem it;
        it.expert = e;
        it.start = offsets[e] + t0;
        it.count = min(kTileN, c - t0);
        it.wtile = w;
        items[idx] = it;
      }
  }
  if (threadIdx.x == 0) *n_items = min(total, max_items);
}

// Rows of NULL ("not mine") experts contribute nothing: zero their y slots.
__global__ void zero_absent_slots_kernel(const int32_t* counts, const int32_t* offsets, const int32_t* perm, int EpS,
                                         const moe_expert_ptrs* table, int H, float* y) {
  const int e = blockIdx.y;
  if (e >= EpS || table[e].gate != nullptr) return;
  const int c = counts[e], o = offsets[e];
  for (int i = blockIdx.x; i < c; i += gridDim.x) {
    float* row = y + (size_t)perm[o + i] * H;
    for (int j = threadIdx.x; j < H; j += blockDim.x) row[j] = 0.0f;
  }
}

// ---------------------------------------------------------------- the GEMM
// Shared memory: A weights [128][256] fp16 canonical (64 KB), B tokens
// [128][256] fp16 canonical (64 KB), A2 mins [128][16] (4 KB), B2 code sums
// [128][16] (4 KB), per-row d/dmin, per-token d_a and row index, the
// mbarrier and the TMEM address.
constexpr int kSmA = 0;
constexpr int kSmB = kSmA + kTileM * 256 * 2;
constexpr int kSmA2 = kSmB + kTileN * 256 * 2;
constexpr int kSmB2 = kSmA2 + kTileM * 16 * 2;
constexpr int kSmDw = kSmB2 + kTileN * 16 * 2;
constexpr int kSmDmin = kSmDw + kTileM * 4;
constexpr int kSmDa = kSmDmin + kTileM * 4;
constexpr int kSmRow = kSmDa + kTileN * 4;
constexpr int kSmBar = kSmRow + kTileN * 4;
constexpr int kSmTmem = kSmBar + 16;
constexpr int kSmTotal = kSmTmem + 16;

template <int FMT, int MODE>  // MODE 0: gate/up + SwiGLU -> h; MODE 1: down -> y
__global__ void __launch_bounds__(kPThreads, 1) prefill_gemm_kernel(const __grid_constant__ PrefillArgs a) {
  using F = Fmt<FMT>;
  extern __shared__ __align__(1024) uint8_t sm[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int K = MODE == 0 ? a.H : a.I;          // reduction length
  const int nb = K / 256;
  const int N_out = MODE == 0 ? a.I : a.H;      // rows of the weight matrices
  const uint32_t bar = smem_u32(sm + kSmBar);
  float* s_dw = reinterpret_cast<float*>(sm + kSmDw);
  float* s_dmin = reinterpret_cast<float*>(sm + kSmDmin);
  float* s_da = reinterpret_cast<float*>(sm + kSmDa);
  int* s_row = reinterpret_cast<int*>(sm + kSmRow);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sm + kSmTmem);

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 256;" ::"r"(smem_u32(s_tmem)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 0) {
    mbar_init(bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  uint32_t phase = 0;
  bool failed = false;

  const int n_items = *a.n_items;
  for (int item = blockIdx.x; item < n_items && !failed; item += gridDim.x) {
    const PItem it = a.items[item];
    const moe_expert_ptrs ep = a.table[it.expert];
    const int ntok = it.count;
    const int N = (ntok + 15) / 16 * 16;  // MMA N
    // token rows of the tile: gate/up gathers x by the bucket permutation, down reads h in bucket order
    for (int n = tid; n < kTileN; n += kPThreads) {
      int row = -1;
      if (n < ntok) row = MODE == 0 ? token_of_slot(a.perm[it.start + n], a.T, a.k) : it.start + n;
      s_row[n] = row;
    }
    float acc[kTileN];
#pragma unroll
    for (int j = 0; j < kTileN; ++j) acc[j] = 0.0f;
    __syncthreads();

    for (int b = 0; b < nb; ++b) {
      // ---- A: 128 weight rows of super-block b, as fp16 sc*q, and the mins
      {
        const int r = tid >> 1, half = tid & 1;  // row r, K half [128*half, +128)
        const uint8_t* base;
        int wrow;
        if (MODE == 0) {
          const int g = r & 63;
          wrow = it.wtile * 64 + g;
          base = static_cast<const uint8_t*>(r < 64 ? ep.gate : ep.up);
        } else {
          wrow = it.wtile * 128 + r;
          base = static_cast<const uint8_t*>(ep.down);
        }
        const uint8_t* slab = base + ((size_t)(wrow >> 5) * nb + b) * F::kSlabBytes;
        const int lr = wrow & 31;
        SbRegs<FMT> s;
        load_sb<FMT>(slab, lr, s);
        if (half == 0) {
          s_dw[r] = half_lo(s.dm);
          s_dmin[r] = half_hi(s.dm);
        }
        uint8_t* A = sm + kSmA;
        if constexpr (FMT == kQ4K) {
          // sub-blocks 4*half .. 4*half+3 (32 codes each)
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const int j = 4 * half + jj;
            int sc, mn;
            sb_scale_min<FMT>(s, j, sc, mn);
            uint32_t lo[4], hi[4];
            mask_q4k(s.code[j], lo, hi);
            const float fs = (float)sc;
            // codes 0..15 of the sub-block are the low nibbles, 16..31 the high ones
#pragma unroll
            for (int w = 0; w < 4; ++w) {
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                const uint32_t v = hh ? hi[w] : lo[w];
                const int k0 = 32 * j + 16 * hh + 4 * w;  // 4 codes k0..k0+3
                uint2 pk;
                pk.x = pack_h2(fs * (float)(v & 0xFF), fs * (float)((v >> 8) & 0xFF));
                pk.y = pack_h2(fs * (float)((v >> 16) & 0xFF), fs * (float)(v >> 24));
                *reinterpret_cast<uint2*>(A + canon_off(r, k0, 32)) = pk;
              }
            }
          }
          if (half == 0) {
            // A2 row r: [mn_0..7, 64*mn_0..7]
            int mnv[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              int sc;
              sb_scale_min<FMT>(s, j, sc, mnv[j]);
            }
            uint4 c0, c1;
            c0.x = pack_h2((float)mnv[0], (float)mnv[1]);
            c0.y = pack_h2((float)mnv[2], (float)mnv[3]);
            c0.z = pack_h2((float)mnv[4], (float)mnv[5]);
            c0.w = pack_h2((float)mnv[6], (float)mnv[7]);
            c1.x = pack_h2(64.f * mnv[0], 64.f * mnv[1]);
            c1.y = pack_h2(64.f * mnv[2], 64.f * mnv[3]);
            c1.z = pack_h2(64.f * mnv[4], 64.f * mnv[5]);
            c1.w = pack_h2(64.f * mnv[6], 64.f * mnv[7]);
            *reinterpret_cast<uint4*>(sm + kSmA2 + canon_off(r, 0, 2)) = c0;
            *reinterpret_cast<uint4*>(sm + kSmA2 + canon_off(r, 8, 2)) = c1;
          }
        } else {
          // sub-blocks 8*half .. 8*half+7 (16 codes each)
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            const int j = 8 * half + jj;
            int sc, mn;
            sb_scale_min<FMT>(s, j, sc, mn);
            uint32_t w[4];
            mask_q2k(s.code[j >> 2], j, w);
            const float fs = (float)sc;
#pragma unroll
            for (int p = 0; p < 4; ++p) {
              const int k0 = 16 * j + 4 * p;
              uint2 pk;
              pk.x = pack_h2(fs * (float)(w[p] & 0xFF), fs * (float)((w[p] >> 8) & 0xFF));
              pk.y = pack_h2(fs * (float)((w[p] >> 16) & 0xFF), fs * (float)(w[p] >> 24));
              *reinterpret_cast<uint2*>(A + canon_off(r, k0, 32)) = pk;
            }
          }
          // A2 row r: mins of the 16 sub-blocks (|bsum| <= 2032 is exact in fp16)
          uint4 c;
          int m0, m1, sc;
          uint32_t pk[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            sb_scale_min<FMT>(s, 8 * half + 2 * q, sc, m0);
            sb_scale_min<FMT>(s, 8 * half + 2 * q + 1, sc, m1);
            pk[q] = pack_h2((float)m0, (float)m1);
          }
          c.x = pk[0]; c.y = pk[1]; c.z = pk[2]; c.w = pk[3];
          *reinterpret_cast<uint4*>(sm + kSmA2 + canon_off(r, 8 * half, 2)) = c;
        }
      }
      // ---- B: the tile's token rows of block b as fp16 codes, and their code sums
      {
        const int n = tid >> 1, half = tid & 1;
        uint8_t* B = sm + kSmB;
        const int row = s_row[n];
        const int8_t* q = MODE == 0 ? a.xq : a.hq;
        const int16_t* bs = MODE == 0 ? a.xbs : a.hbs;
        const float* dq = MODE == 0 ? a.xd : a.hd;
        if (row >= 0) {
          const int4* src = reinterpret_cast<const int4*>(q + (size_t)row * K + 256 * b + 128 * half);
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const int4 v = __ldcg(src + c);
            const uint32_t w4[4] = {(uint32_t)v.x, (uint32_t)v.y, (uint32_t)v.z, (uint32_t)v.w};
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              uint4 pk;
              const uint32_t wa = w4[2 * hh], wb = w4[2 * hh + 1];
              pk.x = pack_h2((float)(int8_t)(wa & 0xFF), (float)(int8_t)((wa >> 8) & 0xFF));
              pk.y = pack_h2((float)(int8_t)((wa >> 16) & 0xFF), (float)(int8_t)(wa >> 24));
              pk.z = pack_h2((float)(int8_t)(wb & 0xFF), (float)(int8_t)((wb >> 8) & 0xFF));
              pk.w = pack_h2((float)(int8_t)((wb >> 16) & 0xFF), (float)(int8_t)(wb >> 24));
              *reinterpret_cast<uint4*>(B + canon_off(n, 128 * half + 16 * c + 8 * hh, 32)) = pk;
            }
          }
          const int16_t* bsp = bs + (size_t)row * (K / 16) + 16 * b;
          if constexpr (FMT == kQ4K) {
            if (half == 0) {
              // 32-code sums bsum_j = 64*hi + lo, lo in [0, 64)
              float lo[8], hi[8];
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const int v = (int)__ldcg(bsp + 2 * j) + (int)__ldcg(bsp + 2 * j + 1);
                const int h = v >> 6;  // floor division
                lo[j] = (float)(v - 64 * h);
                hi[j] = (float)h;
              }
              uint4 c0, c1;
              c0.x = pack_h2(lo[0], lo[1]); c0.y = pack_h2(lo[2], lo[3]);
              c0.z = pack_h2(lo[4], lo[5]); c0.w = pack_h2(lo[6], lo[7]);
              c1.x = pack_h2(hi[0], hi[1]); c1.y = pack_h2(hi[2], hi[3]);
              c1.z = pack_h2(hi[4], hi[5]); c1.w = pack_h2(hi[6], hi[7]);
              *reinterpret_cast<uint4*>(sm + kSmB2 + canon_off(n, 0, 2)) = c0;
              *reinterpret_cast<uint4*>(sm + kSmB2 + canon_off(n, 8, 2)) = c1;
            }
          } else {
            uint4 c;
            c.x = pack_h2((float)__ldcg(bsp + 8 * half + 0), (float)__ldcg(bsp + 8 * half + 1));
            c.y = pack_h2((float)__ldcg(bsp + 8 * half + 2), (float)__ldcg(bsp + 8 * half + 3));
            c.z = pack_h2((float)__ldcg(bsp + 8 * half + 4), (float)__ldcg(bsp + 8 * half + 5));
            c.w = pack_h2((float)__ldcg(bsp + 8 * half + 6), (float)__ldcg(bsp + 8 * half + 7));
            *reinterpret_cast<uint4*>(sm + kSmB2 + canon_off(n, 8 * half, 2)) = c;
          }
          if (half == 0) s_da[n] = __ldcg(dq + (size_t)row * nb + b);
        } else {
          // padding token: zero codes and sums
          const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int c = 0; c < 16; ++c) *reinterpret_cast<uint4*>(B + canon_off(n, 128 * half + 8 * c, 32)) = z;
          *reinterpret_cast<uint4*>(sm + kSmB2 + canon_off(n, 8 * half, 2)) = z;
          if (half == 0) s_da[n] = 0.0f;
        }
      }
      fence_async_smem();
      tc_fence_before();
      __syncthreads();
      // ---- MMAs: S into TMEM columns [0, N), the min term into [128, 128+N)
      if (tid == 0) {
        tc_fence_after();
        const uint32_t idesc = idesc_f16(kTileM, N);
        const uint32_t a0 = smem_u32(sm + kSmA), b0 = smem_u32(sm + kSmB);
        // K-major, 32 core matrices along K: lbo = 128 B, sbo = 32 * 128 B
#pragma unroll 1
        for (int s = 0; s < 16; ++s)
          mma_f16(tmem, smem_desc(a0 + s * 256, 128, 4096), smem_desc(b0 + s * 256, 128, 4096), idesc, s > 0);
        mma_f16(tmem + 128, smem_desc(smem_u32(sm + kSmA2), 128, 256), smem_desc(smem_u32(sm + kSmB2), 128, 256),
                idesc, false);
        mma_commit(bar);
      }
      const bool done = mbar_wait(bar, phase);
      phase ^= 1;
      if (__syncthreads_or(!done)) {  // uniform: every thread leaves together
        if (tid == 0) set_status(a.status, MOE_ERR_DEVICE_TIMEOUT);
        mbar_wait(bar, phase ^ 1);    // one more bounded wait for the MMAs in flight before TMEM is freed
        failed = true;
        break;
      }
      tc_fence_after();
      // ---- epilogue: lane m of warps 0..3 = weight row m
      if (warp < 4) {
        const int m = 32 * warp + lane;
        const float dw = s_dw[m], dmin = s_dmin[m];
        const uint32_t tbase = tmem + ((uint32_t)(32 * warp) << 16);
#pragma unroll
        for (int c = 0; c < kTileN / 16; ++c) {
          if (16 * c < N) {  // N is a multiple of 16 and warp-uniform
            float Sv[16], Mv[16];
            tmem_ld16(tbase + 16 * c, Sv);
            tmem_ld16(tbase + 128 + 16 * c, Mv);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) acc[16 * c + j] += s_da[16 * c + j] * fmaf(dw, Sv[j], -dmin * Mv[j]);
          }
        }
      }
      tc_fence_before();
      __syncthreads();
    }
    if (failed) break;
    // ---- output
    if (MODE == 0) {
      // warps 2,3 hold U of rows 0..63 (lanes 64..127): pass them to warps 0,1 through shared memory
      float* s_u = reinterpret_cast<float*>(sm + kSmA);  // [64][128]
      if (warp == 2 || warp == 3) {
        const int g = 32 * warp + lane - 64;
#pragma unroll
        for (int j = 0; j < kTileN; ++j) s_u[j * 64 + g] = acc[j];
      }
      __syncthreads();
      if (warp < 2) {
        const int g = 32 * warp + lane;
        const int col = it.wtile * 64 + g;
#pragma unroll
        for (int j = 0; j < kTileN; ++j)
          if (j < ntok) {
            const float Gv = acc[j], Uv = s_u[j * 64 + g];
            a.h[(size_t)(it.start + j) * N_out + col] = Gv / (1.0f + expf(-Gv)) * Uv;
          }
      }
      __syncthreads();
    } else {
      if (warp < 4) {
        const int m = 32 * warp + lane;
        const int col = it.wtile * 128 + m;
#pragma unroll
        for (int j = 0; j < kTileN; ++j)
          if (j < ntok) a.y[(size_t)a.perm[it.start + j] * N_out + col] = acc[j];
      }
      __syncthreads();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 256;" ::"r"(tmem));
}

template <int FMT, int MODE>
cudaError_t launch_gemm_t(const PrefillArgs& a, int max_items, cudaStream_t s) {
  auto kern = prefill_gemm_kernel<FMT, MODE>;
  static bool opted = false;
  if (!opted) {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmTotal);
    if (err != cudaSuccess) return err;
    opted = true;
  }
  const int grid = std::max(1, std::min(max_items, num_sms()));
  note_launch();
  kern<<<grid, kPThreads, kSmTotal, s>>>(a);
  return cudaGetLastError();
}

template <int FMT>
cudaError_t launch_prefill_fmt(const PrefillArgs& a0, cudaStream_t s) {
  PrefillArgs a = a0;
  const int EpS = a.E + a.S;
  // gate/up
  int max_items = (int)std::min<int64_t>((a.P / kTileN + EpS) * (a.I / 64), a.max_items);
  note_launch();
  prefill_plan_kernel<<<1, 1024, 0, s>>>(a.counts, a.offsets, EpS, a.table, a.I / 64, a.items, a.n_items, max_items);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  trace_record(s);
  err = launch_gemm_t<FMT, 0>(a, max_items, s);
  trace_record(s);
  if (err != cudaSuccess) return err;
  // q8_K of h, one row per bucket position
  err = launch_q8k_quantize(a.h, a.P, a.I, a.hq, a.hd, a.hbs, s);
  if (err != cudaSuccess) return err;
  // down
  max_items = (int)std::min<int64_t>((a.P / kTileN + EpS) * (a.H / 128), a.max_items);
  note_launch();
  prefill_plan_kernel<<<1, 1024, 0, s>>>(a.counts, a.offsets, EpS, a.table, a.H / 128, a.items, a.n_items, max_items);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  trace_record(s);
  err = launch_gemm_t<FMT, 1>(a, max_items, s);
  trace_record(s);
  if (err != cudaSuccess) return err;
  note_launch();
  zero_absent_slots_kernel<<<dim3(64, EpS), 256, 0, s>>>(a.counts, a.offsets, a.perm, EpS, a.table, a.H, a.y);
  return cudaGetLastError();
}

}  // namespace

size_t prefill_item_capacity(int64_t P, int E, int S, int H, int I) {
  const int64_t EpS = E + S;
  return (size_t)(P / kTileN + EpS) * (size_t)std::max(I / 64, H / 128);
}

cudaError_t launch_prefill_ffn(const PrefillArgs& a, cudaStream_t s) {
  return a.fmt == kQ4K ? launch_prefill_fmt<kQ4K>(a, s) : launch_prefill_fmt<kQ2K>(a, s);
}

}  // namespace moe
