// Prefill expert FFNs on the 5th-generation tensor cores (tcgen05).
//
// In a prefill chunk each expert receives tens to hundreds of tokens, so its
// gate/up and down products are dense contractions.  The weights stay
// block-quantized in HBM and are expanded on chip; the arithmetic is exact
// integer arithmetic carried by fp16 operands:
//
//   A (weights)     sc_j * q  for each weight of sub-block j   (|.| <= 945: exact in fp16)
//   B (activations) the q8_K codes of the tokens               (|q| <= 127: exact)
//   S[m, n, b] = sum over the 256 columns of super-block b of A * B
//
// tcgen05.mma kind::f16 accumulates in fp32 in tensor memory (TMEM).  Each
// half super-block (128 columns) accumulates into its own TMEM region, S0
// and S1: every partial sum of a half is an integer of magnitude at most
// 63*15*127*128 < 2^24 (Q4_K; Q2_K: 15*3*127*128), so S0 and S1 are the
// exact integer sums of their halves.  (A whole Q4_K super-block can reach
// 63*15*127*256 > 2^24, which one fp32 accumulator could not hold.)  The
// epilogue adds them in fp32, which rounds the exact S = S0 + S1 once, as
// the int -> fp32 conversion of the dp4a kernels does.  The min term
// M[m, n, b] = sum_j mn_j * bsum_j(n) is one extra K=16 MMA per super-block
// on the tokens' code sums into a third region (Q4_K: bsum = 64*hi + lo
// against mn and 64*mn, both halves exact; Q2_K: |bsum16| <= 2032 as is;
// |M| <= 63*127*256).  The epilogue rescales per super-block in fp32
// registers:
//
//   D[m, n] = sum_b d_a[n, b] * (d_w[m, b] * (S0 + S1)[m, n, b] - dmin[m, b] * M[m, n, b])
//
// TMEM's 512 columns are a ring of slots of kTileN columns (five of 96):
// super-block number tb of a CTA writes S0, S1, M to slots 3tb, 3tb+1,
// 3tb+2 (mod the slot count), so all MMAs of a super-block but its min MMA
// run while the epilogue still reads the super-block before.  A token tile
// therefore holds at most kTileN tokens; an expert's tokens are split into
// tiles of balanced size.
// This is the same contraction the GEMV kernels compute with dp4a; the
// pages' prefill design reaches it with int8 MMA (Pulsar README, "What it
// does today"; Strata, 0.1.13 prefill notes: grouped int8 tensor-core expert
// GEMM that unpacks super-blocks to shared memory and rescales per block).
// tcgen05 offers no int8 kind on sm_103a, hence exact-integer fp16.  The
// Q4_K, Q2_K and Q3_K-style formats and the IQ2-style grid format run here;
// for the Q3_K-style format (weight = d * sc * (q - 4), sc = u - 32) A =
// sc * q and the min term carries 4 * sc with scale d; for the grid format
// A = (2t + 1) * sign * C[u][i] (|A| <= 155, from fp16 tables of the grid
// and of the sign masks in shared memory) and the min term is zero.  (Q5_K-style products reach 63 * 31 per
// weight and 3.2e7 per half super-block, Q6_K-style 127 * 63 per weight:
// beyond the exact range, so those formats take the dp4a GEMV kernels.)
//
// Kernel organisation (one persistent CTA per SM, 832 threads, warp roles):
//   warp 24      producer: cp.async.bulk of the raw weight slabs and TMA
//                tiles of the activation codes / code sums into rings
//   warps 16-23  expanders: raw slab -> fp16 sc*q tile (two threads per
//                weight row, one swizzle atom each), mins tile for the min MMA
//   warp 25      MMA issuer (one thread): 8 MMAs per half super-block into
//                that half's TMEM region, the min MMA with the last half;
//                commits are grouped (a commit costs the issuing thread
//                several hundred cycles, so each group carries 8+ MMAs)
//   warps 0-15   epilogue: TMEM -> registers in 8-token column blocks (three
//                loads, one wait per block), per-block rescale, output
// (26 warps at 72 registers: the register file is split between the SM's
// four sub-partitions, so the warp count bounds the registers per thread.)
// Rings: 3 activation stages and 2 expanded-weight stages of 128 K each
// (two 128-byte swizzle atoms), 3 raw stages of one super-block column.
// A work item is (expert, token tile of <= kTileN bucket rows, weight tile
// of 128 rows); the items of a launch are laid out by a plan kernel.
//   gate/up: the 128 rows interleave 64 gate rows and the same 64 up rows
//            (even tile row: gate, odd: up), so a lane pair of the epilogue
//            holds G and U of one (row, token): SwiGLU is a shuffle, and h is
//            written in bucket order.
//   down:    128 rows of H; y goes to the (token, slot) rows of the slot buffer.
//   sums:    (test hook) as down, but the epilogue writes the integer S and
//            M of every super-block instead of the rescaled sum.
// Activations are first gathered into bucket order as fp16 codes (and the
// code sums and block scales into TMA-friendly planes) by a small kernel, so
// a token tile is a plain 2-D box for TMA.
#include <algorithm>
#include <cmath>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <mutex>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kTileM = 128;                          // weight rows per tile (MMA M)
#ifndef MOE_PREFILL_TILE_N
#define MOE_PREFILL_TILE_N 96
#endif
constexpr int kTileN = MOE_PREFILL_TILE_N;           // tokens per tile (MMA N <= kTileN)
static_assert(kTileN % 32 == 0 && kTileN >= 32 && kTileN <= 128, "token tile: whole TMA boxes, N <= 128");
// TMEM: 512 columns as a ring of kSlots slots of kTileN columns; a super-block
// takes three (S0, S1, M), so with five or six slots the MMAs of a super-block
// run while the epilogue still reads the one before.
constexpr int kSlots = 512 / kTileN < 6 ? 512 / kTileN : 6;
constexpr int kStageK = 128;                         // K of one A or B stage: half a super-block
constexpr int kAtomK = 64;                           // K of one 128-byte swizzle atom (fp16)
constexpr int kStagesA = 2;                          // expanded-weight stages
constexpr int kStagesB = 3;                          // activation stages
constexpr int kRaw = 3;                              // raw stages (one super-block column each)
constexpr int kBoxRows = 32;                         // token rows per TMA box
constexpr int kEpiWarps = 16, kExpWarps = 8;        // epilogue: 32 tokens per warp; expanders: two threads per row
constexpr int kWarpProducer = kEpiWarps + kExpWarps; // 24
constexpr int kWarpMma = kWarpProducer + 1;          // 25
constexpr int kPThreads = 32 * (kWarpMma + 1);       // 832
constexpr long long kWaitCycles = 2000000000ll;      // ~1 s at 2 GHz: a wait that long has failed

// shared memory (offsets from a 1024-byte aligned base).  A stage holds two
// swizzle atoms of 128 rows x 64 fp16 (16 KB each), K-major, 128-byte swizzle;
// a B stage two atoms of kTileN token rows.
constexpr int kAtomBytes = 128 * 128;
constexpr int kAtomBytesB = kTileN * 128;
constexpr int kBStage = 2 * kAtomBytesB;             // kTileN token rows x 128 codes
constexpr int kAStage = 2 * kAtomBytes;              // 32 KB: 128 weight rows x 128 (sc * q)
constexpr int kRawBytes = 4 * 4608;                  // four slabs (Q4_K size; Q2_K uses less)
constexpr int kSmB = 0;
constexpr int kSmA = kSmB + kStagesB * kBStage;
constexpr int kSmRaw = kSmA + kStagesA * kAStage;
constexpr int kSmA2 = kSmRaw + kRaw * kRawBytes;     // mins tile [128 rows][16] per raw stage
constexpr int kSmB2 = kSmA2 + kRaw * 4096;           // code-sum tile [128 tokens][16] per raw stage
constexpr int kSmDa = kSmB2 + kRaw * 4096;           // per epilogue warp: the block scales of its 32 tokens
constexpr int kSmBar = kSmDa + kEpiWarps * 32 * 4;
constexpr int kNumBars = kStagesA + 2 * kStagesB + 2 * kRaw + 4;
constexpr int kSmMisc = kSmBar + 8 * 32;
constexpr int kSmUsed = kSmMisc + 16;
constexpr int kSmAlloc = kSmUsed + 1024;             // slack for aligning the base
static_assert(kNumBars <= 32, "barrier area");
static_assert(kSmAlloc <= 232448, "shared memory per CTA");

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Shared-memory matrix descriptor, K-major, no swizzle: core matrices of 8
// rows x 16 bytes; lbo = byte distance of core matrices adjacent along K,
// sbo = along M/N.
__device__ __forceinline__ uint64_t desc_plain(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((addr & 0x3FFFF) >> 4);
  d |= (uint64_t)((lbo & 0x3FFFF) >> 4) << 16;
  d |= (uint64_t)((sbo & 0x3FFFF) >> 4) << 32;
  d |= (uint64_t)1 << 46;  // fixed 0b001
  return d;
}
// K-major, 128-byte swizzle (the layout TMA writes with CU_TENSOR_MAP_SWIZZLE_128B):
// 8-row groups 1024 bytes apart; the start may advance by 32-byte K steps inside the atom.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr) {
  uint64_t d = (uint64_t)((addr & 0x3FFFF) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor: kind::f16, A and B fp16, D fp32, both K-major.
__device__ __forceinline__ uint32_t idesc_f16(int M, int N) {
  uint32_t d = 0;
  d |= 1u << 4;                 // D format f32 (A/B format fields 0 = f16)
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
// The four K=16 MMAs of one 64-wide stage: descriptors advance by 32 bytes
// (2 in the start-address field) per step; `acc` = accumulate the first one.
__device__ __forceinline__ void mma_stage4(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, bool acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %11, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %5, %9, p;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %2, %6, %9, 1;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %7, %9, 1;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %4, %8, %9, 1;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(adesc + 2), "l"(adesc + 4), "l"(adesc + 6), "l"(bdesc), "l"(bdesc + 2), "l"(bdesc + 4),
      "l"(bdesc + 6), "r"(idesc), "r"(0), "r"((int)acc));
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_init(uint32_t bar, int count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// the same test without suspending the thread (test_wait): the fast path of a wait
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

constexpr int kEpilogueSleepNs = 0;  // no back-off between the epilogue's polls (a 64 ns one cost 1.7% of the step)

// Bounded wait for phase `parity`.  Gives up when another role has aborted,
// or after about a second, recording a timeout; false = abort.
// `spent` accumulates the cycles waited (per-role wait statistics).  A phase
// already complete costs one non-blocking test and no clock reads (the MMA
// thread runs several such checks per stage).
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* status,
                                         long long& spent, int sleep_ns = 0) {
  if (mbar_test(bar, parity)) return true;
  const long long t0 = clock64();  // before the first try: try_wait itself may suspend the thread
  while (!mbar_try(bar, parity)) {
    if (sleep_ns) __nanosleep(sleep_ns);  // a waiter off the critical path leaves issue slots to the others
    if (*abort_flag) return false;
    if (clock64() - t0 > kWaitCycles) {
      *abort_flag = 1;
      set_status(status, MOE_ERR_DEVICE_TIMEOUT);
      return false;
    }
  }
  spent += clock64() - t0;
  return true;
}

// The same, taken by lane 0 for its whole (converged) warp: every lane gets
// the same answer, so the warp stays converged for .sync.aligned operations.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* status,
                                          long long& spent, int sleep_ns = 0) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = wait_bar(bar, parity, abort_flag, status, spent, sleep_ns);
  ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  __syncwarp();  // orders the other lanes after lane 0's acquire
  return ok;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// packed fp32 pairs (one rounding per lane, as the scalar operations)
__device__ __forceinline__ unsigned long long f2_pack(float x, float y) {
  return (unsigned long long)__float_as_uint(x) | ((unsigned long long)__float_as_uint(y) << 32);
}
__device__ __forceinline__ unsigned long long f2_mul(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b, unsigned long long c) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

// 32 lanes x 8 consecutive fp32 columns of TMEM into 8 registers of each lane
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// TMEM column of slot i of the ring (kSlots slots of kTileN columns)
__device__ __forceinline__ uint32_t tmem_slot(uint32_t i) { return (uint32_t)kTileN * (i % (uint32_t)kSlots); }

// byte offset of element (row, k) in a K-major canonical tile without
// swizzle, kc core matrices along K (16-bit elements)
__device__ __forceinline__ uint32_t canon_off(int row, int k, int kc) {
  return (uint32_t)(((row >> 3) * kc + (k >> 3)) * 128 + (row & 7) * 16 + (k & 7) * 2);
}

// byte offset of element (row, k), k < 128, in a stage of two 128-byte
// swizzled K-major atoms (k / 64 selects the atom): row r at 128*r, its
// 16-byte chunk c stored at chunk c ^ (r % 8)
__device__ __forceinline__ uint32_t sw128_off(int row, int k) {
  return (uint32_t)((k >> 6) * kAtomBytes + row * 128 + (((((k & 63) >> 3) ^ (row & 7)) & 7) << 4) + (k & 7) * 2);
}

__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Two small unsigned codes (bytes `sel` = 0x4140: bytes 0,1; 0x4342: bytes
// 2,3 of w) times the sub-block scale, as an exact fp16 pair:
// 0x64XX is the fp16 number 1024 + XX, and one fused multiply-add
// (1024 + q) * sc - 1024 * sc rounds only the exact result q * sc.
__device__ __forceinline__ uint32_t scaled_pair(uint32_t w, uint32_t sel, __half2 sc2, __half2 off2) {
  const uint32_t v = __byte_perm(w, 0x64u, sel);
  const __half2 h = __hfma2(*reinterpret_cast<const __half2*>(&v), sc2, off2);
  return *reinterpret_cast<const uint32_t*>(&h);
}
// eight codes (bytes of w0, then w1) -> 16 bytes of fp16 sc*q
__device__ __forceinline__ uint4 scaled8(uint32_t w0, uint32_t w1, __half2 sc2, __half2 off2) {
  uint4 o;
  o.x = scaled_pair(w0, 0x4140u, sc2, off2);
  o.y = scaled_pair(w0, 0x4342u, sc2, off2);
  o.z = scaled_pair(w1, 0x4140u, sc2, off2);
  o.w = scaled_pair(w1, 0x4342u, sc2, off2);
  return o;
}

// IQ2-style grid format in the expanders: each grid entry as 8 fp16
// magnitudes, and for each 7-bit sign byte the mask that flips the fp16
// sign bit of the negative elements (the 8th sign from the parity of the
// seven).  Filled at the kernel's start; only the grid-format kernels use it.
__shared__ uint4 s_iq2g_half[256 + 128];

__device__ __forceinline__ void stage_iq2g_half_tables() {
  for (int i = threadIdx.x; i < 256 + 128; i += blockDim.x) {
    uint32_t h[4];
    if (i < 256) {
      const uint64_t v = g_iq2g_grid.v[i];
#pragma unroll
      for (int p = 0; p < 4; ++p)
        h[p] = pack_h2((float)((v >> (16 * p)) & 0xFF), (float)((v >> (16 * p + 8)) & 0xFF));
    } else {
      const uint32_t s7 = (uint32_t)(i - 256);
      const uint32_t s8 = s7 | ((uint32_t)(__popc(s7) & 1) << 7);
#pragma unroll
      for (int p = 0; p < 4; ++p)
        h[p] = (((s8 >> (2 * p)) & 1) ? 0x8000u : 0u) | (((s8 >> (2 * p + 1)) & 1) ? 0x80000000u : 0u);
    }
    s_iq2g_half[i] = make_uint4(h[0], h[1], h[2], h[3]);
  }
}

// ---------------------------------------------------------------- planning
// One CTA: per expert with tokens and a present gate pointer, its token tiles
// (ceil(c/kTileN) tiles of balanced size) x weight tiles, expert by expert.
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
    const int nt = (c + kTileN - 1) / kTileN;
    const int per = (c + nt - 1) / nt;
    int idx = s_n[e];
    for (int t0 = 0; t0 < c; t0 += per)
      for (int w = 0; w < n_wtiles; ++w, ++idx) {
        if (idx >= max_items) continue;
        PItem it;
        it.expert = e;
        it.start = offsets[e] + t0;
        it.count = min(per, c - t0);
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

// Bucket-order planes of the activations for the GEMM (one warp per row p):
//   xg [P][K]          fp16 codes
//   sg [nb][2][P][8]   fp16 code sums of super-block b, two 8-wide halves:
//                      Q4_K: the 32-code sums split as lo (0..63) and hi
//                      (bsum = 64*hi + lo); Q2_K: the 16-code sums 0-7, 8-15
//   dg [nb][P]         fp32 block scales
// Row p comes from token row perm ? token_of_slot(perm[p]) : p.
template <int FMT>
__global__ void __launch_bounds__(256) prefill_gather_kernel(const int8_t* __restrict__ q,
                                                             const int16_t* __restrict__ bs,
                                                             const float* __restrict__ d,
                                                             const int32_t* __restrict__ perm, int T, int k,
                                                             int64_t P, int K, __half* __restrict__ xg,
                                                             __half* __restrict__ sg, float* __restrict__ dg) {
  const int lane = threadIdx.x & 31;
  const int64_t nw = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int nb = K / 256;
  for (int64_t p = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); p < P; p += nw) {
    const int64_t t = perm ? token_of_slot(perm[p], T, k) : p;
    const int4* src = reinterpret_cast<const int4*>(q + t * K);
    uint4* dst = reinterpret_cast<uint4*>(xg + p * K);
    for (int c = lane; c < K / 16; c += 32) {
      const int4 v = __ldg(src + c);
      const uint32_t w[4] = {(uint32_t)v.x, (uint32_t)v.y, (uint32_t)v.z, (uint32_t)v.w};
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const uint32_t a = w[2 * hh], b = w[2 * hh + 1];
        uint4 o;
        o.x = pack_h2((float)(int8_t)(a & 0xFF), (float)(int8_t)((a >> 8) & 0xFF));
        o.y = pack_h2((float)(int8_t)((a >> 16) & 0xFF), (float)(int8_t)(a >> 24));
        o.z = pack_h2((float)(int8_t)(b & 0xFF), (float)(int8_t)((b >> 8) & 0xFF));
        o.w = pack_h2((float)(int8_t)((b >> 16) & 0xFF), (float)(int8_t)(b >> 24));
        dst[2 * c + hh] = o;
      }
    }
    for (int e = lane; e < 2 * nb; e += 32) {
      const int b = e >> 1, hh = e & 1;
      const int16_t* s = bs + t * (K / 16) + 16 * b;
      float v[8];
      if constexpr (FMT == kQ4K) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int sum = (int)s[2 * j] + (int)s[2 * j + 1];
          const int hi = sum >> 6;  // floor
          v[j] = (float)(hh ? hi : sum - 64 * hi);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = (float)s[8 * hh + j];
      }
      uint4 o;
      o.x = pack_h2(v[0], v[1]);
      o.y = pack_h2(v[2], v[3]);
      o.z = pack_h2(v[4], v[5]);
      o.w = pack_h2(v[6], v[7]);
      *reinterpret_cast<uint4*>(sg + ((int64_t)(2 * b + hh) * P + p) * 8) = o;
    }
    for (int b = lane; b < nb; b += 32) dg[(int64_t)b * P + p] = d[t * nb + b];
  }
}

// ---------------------------------------------------------------- the GEMM
struct GemmArgs {
  CUtensorMap map_x;    // xg [P][K] fp16, box {64, 32}, 128-byte swizzle
  CUtensorMap map_s;    // sg rows of 8 fp16, box {8, 128}
  int fmt, H, I, T, k;
  int64_t P;
  const moe_expert_ptrs* table;
  const int32_t* perm;
  const float* dg;
  const PItem* items;
  const int32_t* n_items;
  float* h;
  float* y;
  int* status;
  unsigned long long* stats;  // [16] wait statistics of CTA 0 (nullable)
  // MODE 2 (test hook): the one matrix [N_out, K], and the integer sums out [T][N_out][K/256]
  const void* dbg_w;
  int32_t* dbg_s;
  int32_t* dbg_m;
  int dbg_n;
};

// MODE 0: gate/up + SwiGLU -> h; MODE 1: down -> y; MODE 2: integer S and M of a matrix (test hook)
template <int FMT, int MODE>
__global__ void __launch_bounds__(kPThreads, 1) prefill_gemm_kernel(const __grid_constant__ GemmArgs a) {
  using F = Fmt<FMT>;
  extern __shared__ uint8_t sm_raw[];
  uint8_t* sm = sm_raw + ((1024 - (smem_u32(sm_raw) & 1023)) & 1023);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int K = MODE == 0 ? a.H : a.I;
  const int nb = K / 256;
  const int N_out = MODE == 0 ? a.I : MODE == 1 ? a.H : a.dbg_n;
  const uint32_t sbase = smem_u32(sm);
  const uint32_t bar0 = sbase + kSmBar;
  // barrier slots: full_a, full_b, empty_b, full_raw, empty_raw, tfull, tempty.
  // A weight slot has no barrier of its own: the MMAs of stage m read weight
  // slot m % kStagesA and activation slot m % kStagesB and commit once, to
  // empty_b, which the expanders wait on too.
  auto full_a = [&](int s) { return bar0 + 8 * s; };
  auto full_b = [&](int s) { return bar0 + 8 * (kStagesA + s); };
  auto empty_b = [&](int s) { return bar0 + 8 * (kStagesA + kStagesB + s); };
  auto full_raw = [&](int s) { return bar0 + 8 * (kStagesA + 2 * kStagesB + s); };
  auto empty_raw = [&](int s) { return bar0 + 8 * (kStagesA + 2 * kStagesB + kRaw + s); };
  auto tfull = [&](int s) { return bar0 + 8 * (kStagesA + 2 * kStagesB + 2 * kRaw + s); };
  auto tempty = [&](int s) { return bar0 + 8 * (kStagesA + 2 * kStagesB + 2 * kRaw + 2 + s); };
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sm + kSmMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kSmMisc + 4);

  if constexpr (FMT == kIQ2G) stage_iq2g_half_tables();  // read after the barrier below
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(s_tmem)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 32) {
    for (int s = 0; s < kStagesA; ++s) mbar_init(full_a(s), kExpWarps);
    for (int s = 0; s < kStagesB; ++s) {
      mbar_init(full_b(s), 1);
      mbar_init(empty_b(s), 1);
    }
    for (int s = 0; s < kRaw; ++s) {
      mbar_init(full_raw(s), 1);
      mbar_init(empty_raw(s), kExpWarps + 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(tfull(s), 1);
      mbar_init(tempty(s), kEpiWarps);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const int n_items = *a.n_items;
  const int slab_bytes = F::kSlabBytes;
  const long long t_start = clock64();
  long long w0 = 0, w1 = 0;  // cycles this thread waited on its role's two kinds of barrier

  if (warp == kWarpProducer) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t ri = 0;
      int bs = 0;
      uint32_t pb = 0;
      bool ok = true;
      // the four row groups of an item's weight tile: gate/up -> gate 2w, 2w+1,
      // up 2w, 2w+1; down -> 4w .. 4w+3 (each nb slabs, contiguous)
      auto rows_of = [&](const PItem& it, const uint8_t* (&src)[4]) {
        moe_expert_ptrs ep;
        if (MODE == 2) ep.gate = ep.up = ep.down = a.dbg_w;
        else ep = a.table[it.expert];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          if (MODE == 0) {
            const uint8_t* m = static_cast<const uint8_t*>(g < 2 ? ep.gate : ep.up);
            src[g] = m + (size_t)(it.wtile * 2 + (g & 1)) * nb * slab_bytes;
          } else {
            src[g] = static_cast<const uint8_t*>(ep.down) + (size_t)(it.wtile * 4 + g) * nb * slab_bytes;
          }
        }
      };
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
        const PItem it = a.items[item];
        const uint8_t* src[4];
        rows_of(it, src);
        const int nbox = (it.count + kBoxRows - 1) / kBoxRows;
        for (int b = 0; b < nb && ok; ++b) {
          const int rs = ri % kRaw;
          if (!(ok = wait_bar(empty_raw(rs), ((ri / kRaw) & 1) ^ 1, abort_flag, a.status, w0))) break;
          mbar_expect_tx(full_raw(rs), 4 * slab_bytes + 4096);
          const uint32_t raw = sbase + kSmRaw + rs * kRawBytes;
#pragma unroll
          for (int g = 0; g < 4; ++g)
            bulk_load(raw + g * slab_bytes, src[g] + (size_t)b * slab_bytes, slab_bytes, full_raw(rs));
          const uint32_t b2 = sbase + kSmB2 + rs * 4096;
          tma_load_2d(b2, &a.map_s, 0, (int)((2 * b) * a.P + it.start), full_raw(rs));
          tma_load_2d(b2 + 2048, &a.map_s, 0, (int)((2 * b + 1) * a.P + it.start), full_raw(rs));
          ++ri;
          for (int c = 0; c < 256 / kStageK && ok; ++c) {
            if (!(ok = wait_bar(empty_b(bs), pb ^ 1, abort_flag, a.status, w1))) break;
            mbar_expect_tx(full_b(bs), 2 * nbox * kBoxRows * 128);
            const uint32_t bdst = sbase + kSmB + bs * kBStage;
            for (int at = 0; at < 2; ++at)
              for (int i = 0; i < nbox; ++i)
                tma_load_2d(bdst + at * kAtomBytesB + i * kBoxRows * 128, &a.map_x, 256 * b + kStageK * c + kAtomK * at,
                            it.start + kBoxRows * i, full_b(bs));
            if (++bs == kStagesB) { bs = 0; pb ^= 1; }
          }
        }
      }
    }
  } else if (warp >= kEpiWarps && warp < kWarpProducer) {
    // ------------------------------------------------------------ expanders
    // tile row r: gate/up interleaved (even r: gate row r/2 of the 64-row
    // group, odd r: the same row of up), down: row r of the 128-row group.
    // Two threads per row: `hx` picks the 64-wide atom of each stage.
    const int x = tid - 32 * kEpiWarps;
    const int r = x & 127, hx = x >> 7;
    const int g = MODE == 0 ? ((r & 1) * 2 + (r >> 6)) : (r >> 5);  // slab of the raw stage
    const int lr = MODE == 0 ? ((r >> 1) & 31) : (r & 31);         // row inside the slab
    uint32_t ri = 0;
    int as = 0;
    uint32_t ka = 0;  // stages written so far
    bool ok = true;
    for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
      for (int b = 0; b < nb && ok; ++b) {
        const int rs = ri % kRaw;
        if (!(ok = warp_wait(full_raw(rs), (ri / kRaw) & 1, abort_flag, a.status, w0))) break;
        const uint8_t* slab = sm + kSmRaw + rs * kRawBytes + g * slab_bytes;
        uint8_t* a2 = sm + kSmA2 + rs * 4096;
        // scales and mins, extracted on demand (no per-thread arrays)
        uint64_t sm_lo, sm_hi;
        if constexpr (FMT == kIQ2G) {
          // nibble j = t_j (scale 2 t_j + 1); no min
          sm_lo = *reinterpret_cast<const uint32_t*>(slab + F::kSmOff + 4 * lr);
          sm_hi = 0;
        } else if constexpr (FMT == kQ4K || FMT == kQ3K) {
          // 96-bit string of 6-bit fields: field f = bits 6f.. (Q4_K: scale j = f j,
          // min j = f 8 + j; Q3_K: u_j = f j, scale u_j - 32); sm_hi = bits 48..
          const uint32_t* smw = reinterpret_cast<const uint32_t*>(slab + F::kSmOff + 12 * lr);
          sm_lo = (uint64_t)smw[0] | ((uint64_t)smw[1] << 32);
          sm_hi = (uint64_t)(smw[1] >> 16) | ((uint64_t)smw[2] << 16);
        } else {
          // byte j = scale_j | min_j << 4
          const uint4 v = *reinterpret_cast<const uint4*>(slab + F::kSmOff + 16 * lr);
          sm_lo = (uint64_t)v.x | ((uint64_t)v.y << 32);
          sm_hi = (uint64_t)v.z | ((uint64_t)v.w << 32);
        }
        auto scale_of = [&](int j) -> int {
          if constexpr (FMT == kIQ2G) return 2 * (int)((sm_lo >> (4 * j)) & 15) + 1;
          else if constexpr (FMT == kQ4K) return (int)((sm_lo >> (6 * j)) & 63);
          else if constexpr (FMT == kQ3K) return (int)(((j < 8 ? sm_lo >> (6 * j) : sm_hi >> (6 * (j - 8)))) & 63) - 32;
          else return (int)(((j < 8 ? sm_lo : sm_hi) >> (8 * (j & 7))) & 15);
        };
        // the min-term coefficient: the min, or o * scale (Q3_K-style, o = 4)
        auto min_of = [&](int j) -> int {
          if constexpr (FMT == kIQ2G) return j < 0;  // no min
          else if constexpr (FMT == kQ4K) return (int)((sm_hi >> (6 * j)) & 63);
          else if constexpr (FMT == kQ3K) return 4 * scale_of(j);
          else return (int)(((j < 8 ? sm_lo : sm_hi) >> (8 * (j & 7) + 4)) & 15);
        };
        {
          // A2 row r, K 8*hx .. 8*hx+7: Q4_K [mn_0..7 | 64 * mn_0..7], Q2_K mn_0..15
          float f[8];
#pragma unroll
          for (int i = 0; i < 8; ++i)
            f[i] = FMT == kQ4K ? (hx ? 64.f : 1.f) * (float)min_of(i) : (float)min_of(8 * hx + i);
          uint4 c0;
          c0.x = pack_h2(f[0], f[1]);
          c0.y = pack_h2(f[2], f[3]);
          c0.z = pack_h2(f[4], f[5]);
          c0.w = pack_h2(f[6], f[7]);
          *reinterpret_cast<uint4*>(a2 + canon_off(r, 8 * hx, 2)) = c0;
        }
#pragma unroll
        for (int c = 0; c < 256 / kStageK; ++c) {
          // slot `as` was last read by the MMAs of stage ka - kStagesA: wait for
          // that stage's commit on its activation slot's barrier (stage m
          // completes phase m / kStagesB of empty_b(m % kStagesB))
          if (ka >= (uint32_t)kStagesA) {
            const uint32_t m = ka - kStagesA;
            if (!(ok = warp_wait(empty_b(m % kStagesB), (m / kStagesB) & 1, abort_flag, a.status, w1))) break;
          }
          ++ka;
          uint8_t* A = sm + kSmA + as * kAStage;
          if constexpr (FMT == kIQ2G) {
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
              const int j = 4 * c + 2 * hx + jj;  // sub-block of 32 weights = groups 4j .. 4j + 3
              const uint4 li = *reinterpret_cast<const uint4*>(slab + F::kCodeOff + 512 * (j >> 2) + 16 * lr);
              const uint4 ls = *reinterpret_cast<const uint4*>(slab + F::kCodeOff + 512 * (2 + (j >> 2)) + 16 * lr);
              const int ws = j & 3;
              const uint32_t iw = ws == 0 ? li.x : ws == 1 ? li.y : ws == 2 ? li.z : li.w;
              const uint32_t sw = ws == 0 ? ls.x : ws == 1 ? ls.y : ws == 2 ? ls.z : ls.w;
              const __half2 sc2 = __float2half2_rn((float)scale_of(j));
              const int k0 = 64 * hx + 32 * jj;
#pragma unroll
              for (int gg = 0; gg < 4; ++gg) {
                // 8 weights: the grid magnitudes with their signs flipped, times the scale (exact: |.| <= 155)
                const uint4 mag = s_iq2g_half[(iw >> (8 * gg)) & 0xFF];
                const uint4 neg = s_iq2g_half[256 + ((sw >> (8 * gg)) & 0x7F)];
                const uint32_t hv[4] = {mag.x ^ neg.x, mag.y ^ neg.y, mag.z ^ neg.z, mag.w ^ neg.w};
                uint4 o;
                uint32_t* op = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                  const __half2 prod = __hmul2(*reinterpret_cast<const __half2*>(&hv[p]), sc2);
                  op[p] = *reinterpret_cast<const uint32_t*>(&prod);
                }
                *reinterpret_cast<uint4*>(A + sw128_off(r, k0 + 8 * gg)) = o;
              }
            }
          } else if constexpr (FMT == kQ4K) {
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
              const int j = 4 * c + 2 * hx + jj;  // sub-block of 32 codes
              const uint4 cw = *reinterpret_cast<const uint4*>(slab + F::kCodeOff + 512 * j + 16 * lr);
              uint32_t lo4[4], hi4[4];
              mask_q4k(cw, lo4, hi4);
              const float scf = (float)scale_of(j);
              const __half2 sc2 = __float2half2_rn(scf);
              const __half2 off2 = __float2half2_rn(-1024.0f * scf);
              const int k0 = 64 * hx + 32 * jj;  // K offset inside the stage
              *reinterpret_cast<uint4*>(A + sw128_off(r, k0)) = scaled8(lo4[0], lo4[1], sc2, off2);
              *reinterpret_cast<uint4*>(A + sw128_off(r, k0 + 8)) = scaled8(lo4[2], lo4[3], sc2, off2);
              *reinterpret_cast<uint4*>(A + sw128_off(r, k0 + 16)) = scaled8(hi4[0], hi4[1], sc2, off2);
              *reinterpret_cast<uint4*>(A + sw128_off(r, k0 + 24)) = scaled8(hi4[2], hi4[3], sc2, off2);
            }
          } else {
            const uint4 line = *reinterpret_cast<const uint4*>(slab + F::kCodeOff + 512 * (2 * c + hx) + 16 * lr);
            uint4 hline = make_uint4(0u, 0u, 0u, 0u);  // Q3_K-style: the 3rd bits of sub-blocks 8c .. 8c + 7
            if constexpr (FMT == kQ3K) hline = *reinterpret_cast<const uint4*>(slab + F::kCodeOff + 512 * (4 + c) + 16 * lr);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int j = 8 * c + 4 * hx + q;  // sub-block of 16 codes
              uint32_t w[4];
              mask_q2k(line, q, w);
              if constexpr (FMT == kQ3K) {
                // word (j/2) % 4 = 2 hx + q/2 of the line; bit p + 4 (j % 2) of byte m -> code 4p + m
                const int wi = 2 * hx + (q >> 1);
                const uint32_t hv = wi == 0 ? hline.x : wi == 1 ? hline.y : wi == 2 ? hline.z : hline.w;
#pragma unroll
                for (int p = 0; p < 4; ++p) w[p] |= ((hv >> (p + 4 * (q & 1))) & 0x01010101u) << 2;
              }
              const float scf = (float)scale_of(j);
              const __half2 sc2 = __float2half2_rn(scf);
              const __half2 off2 = __float2half2_rn(-1024.0f * scf);
              const int k0 = 64 * hx + 16 * q;
              *reinterpret_cast<uint4*>(A + sw128_off(r, k0)) = scaled8(w[0], w[1], sc2, off2);
              *reinterpret_cast<uint4*>(A + sw128_off(r, k0 + 8)) = scaled8(w[2], w[3], sc2, off2);
            }
          }
          fence_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(full_a(as));
          if (++as == kStagesA) as = 0;
        }
        if (!ok) break;
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_raw(rs));
        ++ri;
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    // Per super-block: stage 0 (8 MMAs into S0, one commit group), stage 1
    // (8 MMAs into S1, then the min MMA into M, one commit group).  A commit
    // costs the issuing thread a few hundred cycles, so each stage commits
    // once for its slots (empty_b: the expanders read the weight slot's
    // release from it too), plus once per super-block for the raw stage and
    // the epilogue.
    if (lane == 0) {
      const uint64_t dA0 = desc_sw128(sbase + kSmA), dB0 = desc_sw128(sbase + kSmB);
      const uint64_t dA2 = desc_plain(sbase + kSmA2, 128, 256), dB2 = desc_plain(sbase + kSmB2, 2048, 128);
      uint32_t ri = 0, tb = 0;
      uint32_t rel = 0;  // super-blocks whose TMEM slots the epilogue has released (seen in order)
      int as = 0, bs = 0;
      uint32_t pa = 0, pb = 0;
      bool ok = true;
      static_assert(256 / kStageK == 2, "one TMEM slot per half super-block");
      // TMEM slot j of super-block tb is ring slot 3 tb + j; before writing
      // it, wait until the epilogue has released the super-block that used
      // it last, (3 tb + j - kSlots) / 3.  Releases are taken in order, one
      // phase of tempty[sb & 1] per super-block sb.
      auto free_slot = [&](uint32_t slot) -> bool {
        if (slot < (uint32_t)kSlots) return true;
        const uint32_t last = (slot - kSlots) / 3;
        while (rel <= last) {
          if (!wait_bar(tempty(rel & 1), (rel >> 1) & 1, abort_flag, a.status, w0)) return false;
          ++rel;
        }
        return true;
      };
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
        const PItem it = a.items[item];
        const int N = (it.count + 15) / 16 * 16;
        const uint32_t idesc = idesc_f16(kTileM, N);
        for (int b = 0; b < nb && ok; ++b) {
          const int ab = tb & 1;
          const int rs = ri % kRaw;
          for (int c = 0; c < 2 && ok; ++c) {
            if (!(ok = free_slot(3 * tb + c))) break;
            if (!(ok = wait_bar(full_a(as), pa, abort_flag, a.status, w1))) break;
            if (!(ok = wait_bar(full_b(bs), pb, abort_flag, a.status, w1))) break;
            const bool last = c == 1;
            if (last && !(ok = wait_bar(full_raw(rs), (ri / kRaw) & 1, abort_flag, a.status, w1))) break;
            tc_fence_after();
            const uint32_t dS = tmem + tmem_slot(3 * tb + c);
            const uint64_t da = dA0 + (uint64_t)((as * kAStage) >> 4), db = dB0 + (uint64_t)((bs * kBStage) >> 4);
            mma_stage4(dS, da, db, idesc, false);
            mma_stage4(dS, da + (kAtomBytes >> 4), db + (kAtomBytesB >> 4), idesc, true);
            if (last) {
              if (!(ok = free_slot(3 * tb + 2))) break;
              tc_fence_after();
              mma_f16(tmem + tmem_slot(3 * tb + 2), dA2 + (uint64_t)((rs * 4096) >> 4),
                      dB2 + (uint64_t)((rs * 4096) >> 4), idesc, false);
            }
            mma_commit(empty_b(bs));
            if (last) {
              mma_commit(empty_raw(rs));
              mma_commit(tfull(ab));
            }
            if (++as == kStagesA) { as = 0; pa ^= 1; }
            if (++bs == kStagesB) { bs = 0; pb ^= 1; }
          }
          ++ri;
          ++tb;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 0-15)
    // Warp (qd, cg) owns TMEM lanes 32*qd.. (tile rows) and the 8-token
    // column blocks cg, cg + 4, cg + 8, .. (block kb of the warp is block
    // cg + 4 kb), so short tiles spread evenly over the four column groups.
    // Per super-block and block: three 8-column TMEM loads (S0, S1, M), one
    // wait, then the rescale into the block's accumulators.
    constexpr int kBlocksPerWarp = (kTileN / 8 + 3) / 4;
    const int qd = warp & 3, cg = warp >> 2;
    const int m = 32 * qd + lane;             // tile row
    float* s_da = reinterpret_cast<float*>(sm + kSmDa) + 32 * warp;
    uint32_t tb = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
      const PItem it = a.items[item];
      moe_expert_ptrs ep;
      if (MODE == 2) ep.gate = ep.up = ep.down = a.dbg_w;
      else ep = a.table[it.expert];
      const int ntok = it.count;
      const int nblk = (ntok + 7) / 8;
      const uint8_t* hdr;  // header (d | dmin, or d) of this row's super-block 0
      if (MODE == 0) {
        const int i = it.wtile * 64 + (m >> 1);
        hdr = static_cast<const uint8_t*>((m & 1) ? ep.up : ep.gate) + (size_t)(i >> 5) * nb * slab_bytes +
              F::kHdrBytes * (i & 31);
      } else {
        const int i = it.wtile * 128 + m;
        hdr = static_cast<const uint8_t*>(ep.down) + (size_t)(i >> 5) * nb * slab_bytes + F::kHdrBytes * (i & 31);
      }
      auto ld_hdr = [&](const uint8_t* p) -> uint32_t {
        if constexpr (F::kHdrBytes == 4) return __ldg(reinterpret_cast<const uint32_t*>(p));
        else return (uint32_t)__ldg(reinterpret_cast<const unsigned short*>(p));
      };
      unsigned long long acc[kBlocksPerWarp][4];  // block kb: pairs of tokens (2i, 2i+1)
#pragma unroll
      for (int kb = 0; kb < kBlocksPerWarp; ++kb)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[kb][j] = 0ull;
      // this lane's token (for the block scales and the down slot): i = lane % 8 of block lane / 8
      const int tk = 8 * (cg + 4 * (lane >> 3)) + (lane & 7);
      const bool vt = tk < ntok;
      const int slot = (MODE == 1 && vt) ? __ldg(a.perm + it.start + tk) : 0;  // down: its slot row
      const float* dgp = a.dg + it.start + tk;
      // the scales of block b + 1 are loaded while block b is processed
      uint32_t dm_n = ld_hdr(hdr);
      float da_n = vt ? __ldg(dgp) : 0.0f;
      for (int b = 0; b < nb; ++b) {
        const int ab = tb & 1;
        const uint32_t dm = dm_n;
        const float da = da_n;
        if (b + 1 < nb) {
          dm_n = ld_hdr(hdr + (size_t)(b + 1) * slab_bytes);
          da_n = vt ? __ldg(dgp + (int64_t)(b + 1) * a.P) : 0.0f;
        }
        if (!(ok = warp_wait(tfull(ab), (tb >> 1) & 1, abort_flag, a.status, w0, kEpilogueSleepNs))) break;
        tc_fence_after();
        s_da[lane] = da;
        __syncwarp();
        float dw, dmin;  // d and the min-term scale (dmin, or d for the Q3_K-style format)
        sb_d_mscale<FMT>(dm, dw, dmin);
        const unsigned long long dw2 = f2_pack(dw, dw), ndm2 = f2_pack(-dmin, -dmin);
        const uint32_t tl = tmem + ((uint32_t)(32 * qd) << 16);
        const uint32_t tS0 = tl + tmem_slot(3 * tb), tS1 = tl + tmem_slot(3 * tb + 1), tM = tl + tmem_slot(3 * tb + 2);
#pragma unroll
        for (int kb = 0; kb < kBlocksPerWarp; ++kb) {
          const int cb = cg + 4 * kb;  // column block (warp-uniform test)
          if (cb < nblk) {
            float S0v[8], S1v[8], Mv[8];
            tmem_ld8(tS0 + 8 * cb, S0v);
            tmem_ld8(tS1 + 8 * cb, S1v);
            tmem_ld8(tM + 8 * cb, Mv);
            tmem_wait_ld();
            if constexpr (MODE == 2) {
              // the integer sums of the super-block: S = S0 + S1 exactly (each half below 2^24)
              const int row = it.wtile * kTileM + m;
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const int tok = 8 * cb + i;
                if (tok < ntok) {
                  const int64_t o = ((int64_t)(it.start + tok) * N_out + row) * nb + b;
                  a.dbg_s[o] = (int32_t)S0v[i] + (int32_t)S1v[i];
                  a.dbg_m[o] = (int32_t)Mv[i];
                }
              }
            } else {
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                // S0 + S1: both exact integers, so the fp32 sum rounds the exact S once
                const float2 d2 = *reinterpret_cast<const float2*>(s_da + 8 * kb + 2 * j);
                const unsigned long long S2 = f2_pack(S0v[2 * j] + S1v[2 * j], S0v[2 * j + 1] + S1v[2 * j + 1]);
                const unsigned long long t = f2_fma(dw2, S2, f2_mul(ndm2, f2_pack(Mv[2 * j], Mv[2 * j + 1])));
                acc[kb][j] = f2_fma(f2_pack(d2.x, d2.y), t, acc[kb][j]);
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty(ab));
        ++tb;
      }
      if (!ok) break;
      if constexpr (MODE != 2) {
#pragma unroll
        for (int kb = 0; kb < kBlocksPerWarp; ++kb) {
          const int cb = cg + 4 * kb;
          if (cb >= nblk) continue;  // warp-uniform
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int tok = 8 * cb + 2 * j;  // tokens tok, tok + 1 of the tile
            const float lo = __uint_as_float((uint32_t)acc[kb][j]), hi = __uint_as_float((uint32_t)(acc[kb][j] >> 32));
            if (MODE == 0) {
              // lane pairs hold gate (even lane) and up (odd lane) of one row: SwiGLU in registers
              const float G0 = __shfl_sync(0xffffffffu, lo, lane & ~1), G1 = __shfl_sync(0xffffffffu, hi, lane & ~1);
              float* hcol = a.h + (int64_t)(it.start + tok) * N_out + it.wtile * 64 + (m >> 1);
              if (lane & 1) {
                if (tok < ntok) hcol[0] = __fdividef(G0, 1.0f + __expf(-G0)) * lo;
                if (tok + 1 < ntok) hcol[N_out] = __fdividef(G1, 1.0f + __expf(-G1)) * hi;
              }
            } else {
              // the slot rows of the two tokens sit in lanes 8 kb + 2 j and 8 kb + 2 j + 1
              const int s0 = __shfl_sync(0xffffffffu, slot, 8 * kb + 2 * j), s1 = __shfl_sync(0xffffffffu, slot, 8 * kb + 2 * j + 1);
              const int col = it.wtile * 128 + m;
              if (tok < ntok) a.y[(int64_t)s0 * N_out + col] = lo;
              if (tok + 1 < ntok) a.y[(int64_t)s1 * N_out + col] = hi;
            }
          }
        }
      }
    }
  }
  // wait statistics of CTA 0, one thread per role (SM cycles):
  //   [0] producer: raw slot free   [1] producer: activation slot free
  //   [2] expander: raw data        [3] expander: weight slot free
  //   [4] MMA: accumulator free     [5] MMA: operands ready
  //   [6] epilogue: accumulator     [7] total cycles of the CTA
  if (a.stats && blockIdx.x == 0) {
    unsigned long long* st = a.stats + 8 * MODE;
    if (tid == 32 * kWarpProducer) { st[0] = w0; st[1] = w1; }
    if (tid == 32 * kEpiWarps) { st[2] = w0; st[3] = w1; }
    if (tid == 32 * kWarpMma) { st[4] = w0; st[5] = w1; }
    if (tid == 0) st[6] = w0;
  }
  tc_fence_before();
  __syncthreads();
  if (a.stats && blockIdx.x == 0 && tid == 0) a.stats[8 * MODE + 7] = clock64() - t_start;
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem));
  }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D fp16 tensor map: `inner` elements per row, `rows` rows, box {box_inner, box_rows}
bool make_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
              uint32_t box_rows, bool swizzle) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int FMT, int MODE>
cudaError_t launch_gemm_t(const GemmArgs& g, int max_items, cudaStream_t s) {
  auto kern = prefill_gemm_kernel<FMT, MODE>;
  static bool opted = false;
  if (!opted) {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmAlloc);
    if (err != cudaSuccess) return err;
    opted = true;
  }
  const int grid = std::max(1, std::min(max_items, num_sms()));
  note_launch();
  kern<<<grid, kPThreads, kSmAlloc, s>>>(g);
  return cudaGetLastError();
}

template <int FMT>
cudaError_t launch_gather(const int8_t* q, const int16_t* bs, const float* d, const int32_t* perm, int T, int k,
                          int64_t P, int K, __half* xg, __half* sg, float* dg, cudaStream_t s) {
  const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>((P + 7) / 8, 16 * num_sms()));
  note_launch();
  prefill_gather_kernel<FMT><<<(unsigned)blocks, 256, 0, s>>>(q, bs, d, perm, T, k, P, K, xg, sg, dg);
  return cudaGetLastError();
}

template <int FMT>
cudaError_t launch_prefill_fmt(const PrefillArgs& a, cudaStream_t s) {
  const int EpS = a.E + a.S;
  GemmArgs g{};
  g.fmt = a.fmt;
  g.H = a.H;
  g.I = a.I;
  g.T = a.T;
  g.k = a.k;
  g.P = a.P;
  g.table = a.table;
  g.perm = a.perm;
  g.dg = a.dg;
  g.items = a.items;
  g.n_items = a.n_items;
  g.h = a.h;
  g.y = a.y;
  g.status = a.status;
  g.stats = a.stats;
  // ---- gate/up: x codes gathered into bucket order
  __half* xg = static_cast<__half*>(a.xg);
  __half* sg = static_cast<__half*>(a.sg);
  cudaError_t err = launch_gather<FMT>(a.xq, a.xbs, a.xd, a.perm, a.T, a.k, a.P, a.H, xg, sg, a.dg, s);
  if (err != cudaSuccess) return err;
  if (!make_map(&g.map_x, a.xg, (uint64_t)a.H, (uint64_t)a.P, 64, kBoxRows, true) ||
      !make_map(&g.map_s, a.sg, 8, (uint64_t)(a.H / 256) * 2 * a.P, 8, 128, false))
    return cudaErrorInvalidValue;
  int max_items = (int)std::min<int64_t>((a.P / kTileN + EpS) * (a.I / 64), a.max_items);
  note_launch();
  prefill_plan_kernel<<<1, 1024, 0, s>>>(a.counts, a.offsets, EpS, a.table, a.I / 64, a.items, a.n_items, max_items);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  trace_record(s);
  err = launch_gemm_t<FMT, 0>(g, max_items, s);
  trace_record(s);
  if (err != cudaSuccess) return err;
  // ---- q8_K of h (bucket order), its gathered planes, down
  if ((err = launch_q8k_quantize(a.h, a.P, a.I, a.hq, a.hd, a.hbs, s)) != cudaSuccess) return err;
  if ((err = launch_gather<FMT>(a.hq, a.hbs, a.hd, nullptr, a.T, a.k, a.P, a.I, xg, sg, a.dg, s)) != cudaSuccess)
    return err;
  if (!make_map(&g.map_x, a.xg, (uint64_t)a.I, (uint64_t)a.P, 64, kBoxRows, true) ||
      !make_map(&g.map_s, a.sg, 8, (uint64_t)(a.I / 256) * 2 * a.P, 8, 128, false))
    return cudaErrorInvalidValue;
  max_items = (int)std::min<int64_t>((a.P / kTileN + EpS) * (a.H / 128), a.max_items);
  note_launch();
  prefill_plan_kernel<<<1, 1024, 0, s>>>(a.counts, a.offsets, EpS, a.table, a.H / 128, a.items, a.n_items, max_items);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  trace_record(s);
  err = launch_gemm_t<FMT, 1>(g, max_items, s);
  trace_record(s);
  if (err != cudaSuccess) return err;
  note_launch();
  zero_absent_slots_kernel<<<dim3(64, EpS), 256, 0, s>>>(a.counts, a.offsets, a.perm, EpS, a.table, a.H, a.y);
  return cudaGetLastError();
}

// Items of the sums hook: token tiles of up to kTileN rows x the 128-row weight tiles.
__global__ void sums_items_kernel(int T, int n_wtiles, PItem* items, int32_t* n_items) {
  const int nt = (T + kTileN - 1) / kTileN;
  for (int i = threadIdx.x; i < nt * n_wtiles; i += blockDim.x) {
    PItem it;
    it.expert = 0;
    it.start = (i / n_wtiles) * kTileN;
    it.count = min(kTileN, T - it.start);
    it.wtile = i % n_wtiles;
    items[i] = it;
  }
  if (threadIdx.x == 0) *n_items = nt * n_wtiles;
}

template <int FMT>
cudaError_t launch_sums_t(const SumsArgs& a, cudaStream_t s) {
  const SumsPlan p = sums_plan(a.N, a.K, a.T);
  char* base = static_cast<char*>(a.ws);
  __half* xg = reinterpret_cast<__half*>(base + p.xg);
  __half* sg = reinterpret_cast<__half*>(base + p.sg);
  float* dg = reinterpret_cast<float*>(base + p.dg);
  PItem* items = reinterpret_cast<PItem*>(base + p.items);
  int32_t* n_items = reinterpret_cast<int32_t*>(base + p.n_items);
  cudaError_t err = launch_gather<FMT>(a.q, a.bs16, a.d, nullptr, a.T, 1, a.T, a.K, xg, sg, dg, s);
  if (err != cudaSuccess) return err;
  GemmArgs g{};
  g.fmt = FMT;
  g.H = a.N;
  g.I = a.K;
  g.T = a.T;
  g.k = 1;
  g.P = a.T;
  g.dg = dg;
  g.items = items;
  g.n_items = n_items;
  g.status = reinterpret_cast<int*>(base + p.status);
  g.dbg_w = a.w;
  g.dbg_s = a.S;
  g.dbg_m = a.M;
  g.dbg_n = a.N;
  if (!make_map(&g.map_x, xg, (uint64_t)a.K, (uint64_t)a.T, 64, kBoxRows, true) ||
      !make_map(&g.map_s, sg, 8, (uint64_t)(a.K / 256) * 2 * a.T, 8, 128, false))
    return cudaErrorInvalidValue;
  const int n_wtiles = a.N / kTileM;
  note_launch();
  sums_items_kernel<<<1, 256, 0, s>>>(a.T, n_wtiles, items, n_items);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  return launch_gemm_t<FMT, 2>(g, ((a.T + kTileN - 1) / kTileN) * n_wtiles, s);
}

// ---------------------------------------------------------------- router logits on the tensor cores
// logits[t, e] = sum_h x[t, h] * W[e, h] (+ bias[e]) for a prefill chunk, on
// tcgen05 kind::tf32 with the three-term split of each fp32 operand
// (a = a_hi + a_lo, a_hi = tf32(a) rounded to nearest, a_lo = a - a_hi
// exactly): a*b ~ a_hi*b_hi + a_hi*b_lo + a_lo*b_hi.  Each product keeps
// about 21 significant bits and the sums are fp32 in TMEM, an error of the
// order of fp32's own rounding, far inside the forward-error bound
// (H + 8) u sum |w x| that the top-k decisions are checked against.
// (Pulsar README, "What it does today": a softmax or sigmoid router per MoE
// layer; its logits come from the unquantized activations.)
//
// One CTA per 128-token x 256-expert tile, K in a ring of four stages of
// 16 fp32 (64-byte rows, 64-byte swizzle): warp 0 issues the TMA loads of x
// and W, warps 2-5
// split each stage in place (hi) and into a second plane (lo), warp 1
// issues 3 x 4 MMAs per stage into one 256-column TMEM accumulator, and
// warps 2-5 write the tile (+ bias) at the end.
constexpr int kRtM = 128, kRtN = 256, kRtK = 16, kRtStages = 4;
constexpr int kRtABytes = kRtM * kRtK * 4, kRtBBytes = kRtN * kRtK * 4;  // 16 KB, 32 KB
constexpr int kRtStageBytes = 2 * (kRtABytes + kRtBBytes);              // raw/hi and lo planes
constexpr int kRtThreads = 192;
constexpr int kRtSmBar = kRtStages * kRtStageBytes;
constexpr int kRtNumBars = 3 * kRtStages + 1;  // full, split, empty per stage; done
constexpr int kRtSmAlloc = kRtSmBar + 8 * kRtNumBars + 16 + 1024;
static_assert(kRtSmAlloc <= 232448, "router tile shared memory");

struct RouterTcArgs {
  CUtensorMap map_x;  // x [T][H] fp32, box {16, 128}, 64-byte swizzle
  CUtensorMap map_w;  // W [E][H] fp32, box {16, 256}, 64-byte swizzle
  const float* bias;
  float* logits;
  int T, H, E;
  int* status;
};

// Instruction descriptor: kind::tf32, A and B tf32 (format 2), D fp32, both K-major.
__device__ __forceinline__ uint32_t idesc_tf32(int M, int N) {
  uint32_t d = 0;
  d |= 1u << 4;   // D format f32
  d |= 2u << 7;   // A format tf32
  d |= 2u << 10;  // B format tf32
  d |= (uint32_t)(N >> 3) << 17;
  d |= (uint32_t)(M >> 4) << 24;
  return d;
}
__device__ __forceinline__ void mma_tf32(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, bool acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"((int)acc));
}
// K-major, 64-byte swizzle: 8-row groups 512 bytes apart; the start may
// advance by 32-byte K steps inside the 64-byte row.
__device__ __forceinline__ uint64_t desc_sw64(uint32_t addr) {
  uint64_t d = (uint64_t)((addr & 0x3FFFF) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(512 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)4 << 61;
  return d;
}
__device__ __forceinline__ float tf32_rna(float v) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(v));
  return __uint_as_float(r);
}

__global__ void __launch_bounds__(kRtThreads, 1) router_tc_kernel(const __grid_constant__ RouterTcArgs a) {
  extern __shared__ uint8_t sm_raw[];
  uint8_t* sm = sm_raw + ((1024 - (smem_u32(sm_raw) & 1023)) & 1023);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t sbase = smem_u32(sm);
  const uint32_t bar0 = sbase + kRtSmBar;
  auto full = [&](int s) { return bar0 + 8 * s; };                    // TMA bytes landed
  auto split = [&](int s) { return bar0 + 8 * (kRtStages + s); };     // hi/lo planes written
  auto empty = [&](int s) { return bar0 + 8 * (2 * kRtStages + s); }; // MMAs of the stage done
  const uint32_t done = bar0 + 8 * (3 * kRtStages);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sm + kRtSmBar + 8 * kRtNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kRtSmBar + 8 * kRtNumBars + 4);
  // stage s: A hi at 0, B hi at kRtABytes, A lo, B lo after them
  auto a_hi = [&](int s) { return s * kRtStageBytes; };
  auto b_hi = [&](int s) { return s * kRtStageBytes + kRtABytes; };
  auto a_lo = [&](int s) { return s * kRtStageBytes + kRtABytes + kRtBBytes; };
  auto b_lo = [&](int s) { return s * kRtStageBytes + 2 * kRtABytes + kRtBBytes; };
  const int m0 = blockIdx.y * kRtM, n0 = blockIdx.x * kRtN;
  const int nk = a.H / kRtK;

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 256;" ::"r"(smem_u32(s_tmem)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 32) {
    for (int s = 0; s < kRtStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(split(s), 4);
      mbar_init(empty(s), 1);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  long long w0 = 0, w1 = 0;
  bool ok = true;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      for (int kb = 0; kb < nk && ok; ++kb) {
        const int s = kb % kRtStages;
        const uint32_t ph = (kb / kRtStages) & 1;
        if (!(ok = wait_bar(empty(s), ph ^ 1, abort_flag, a.status, w0))) break;
        mbar_expect_tx(full(s), kRtABytes + kRtBBytes);
        tma_load_2d(sbase + a_hi(s), &a.map_x, kRtK * kb, m0, full(s));
        tma_load_2d(sbase + b_hi(s), &a.map_w, kRtK * kb, n0, full(s));
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_tf32(kRtM, kRtN);
      for (int kb = 0; kb < nk && ok; ++kb) {
        const int s = kb % kRtStages;
        const uint32_t ph = (kb / kRtStages) & 1;
        if (!(ok = wait_bar(split(s), ph, abort_flag, a.status, w1))) break;
        tc_fence_after();
        const uint64_t ah = desc_sw64(sbase + a_hi(s)), bh = desc_sw64(sbase + b_hi(s));
        const uint64_t al = desc_sw64(sbase + a_lo(s)), bl = desc_sw64(sbase + b_lo(s));
#pragma unroll
        for (int k8 = 0; k8 < kRtK / 8; ++k8) {  // K = 8 tf32 = 32 bytes per MMA
          const uint64_t o = (uint64_t)(2 * k8);
          mma_tf32(tmem, al + o, bh + o, idesc, kb > 0 || k8 > 0);
          mma_tf32(tmem, ah + o, bl + o, idesc, true);
          mma_tf32(tmem, ah + o, bh + o, idesc, true);
        }
        mma_commit(empty(s));
      }
      if (ok) mma_commit(done);
    }
  } else {
    // ------------------------------------------------ split (warps 2-5), then the epilogue
    const int ct = tid - 64;  // 0..127
    for (int kb = 0; kb < nk && ok; ++kb) {
      const int s = kb % kRtStages;
      const uint32_t ph = (kb / kRtStages) & 1;
      if (!(ok = warp_wait(full(s), ph, abort_flag, a.status, w0))) break;
      // the swizzle permutes 16-byte chunks only, so each chunk splits in place
      float4* hiA = reinterpret_cast<float4*>(sm + a_hi(s));
      float4* loA = reinterpret_cast<float4*>(sm + a_lo(s));
      for (int i = ct; i < (kRtABytes + kRtBBytes) / 16; i += 128) {
        float4 v = hiA[i];  // A and B hi planes are adjacent, as are the lo planes
        float4 h, l;
        h.x = tf32_rna(v.x); l.x = v.x - h.x;
        h.y = tf32_rna(v.y); l.y = v.y - h.y;
        h.z = tf32_rna(v.z); l.z = v.z - h.z;
        h.w = tf32_rna(v.w); l.w = v.w - h.w;
        hiA[i] = h;
        loA[i] = l;
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(split(s));
    }
    if (ok) ok = warp_wait(done, 0, abort_flag, a.status, w1, 128);
    if (ok) {
      tc_fence_after();
      const int qd = warp & 3;  // TMEM lanes 32 qd .. 32 qd + 31
      const int t = m0 + 32 * qd + lane;
      const uint32_t tl = tmem + ((uint32_t)(32 * qd) << 16);
      for (int c0 = 0; c0 < kRtN; c0 += 8) {
        if (n0 + c0 >= a.E) break;  // warp-uniform
        float v[8];
        tmem_ld8(tl + c0, v);
        tmem_wait_ld();
        if (t < a.T) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int e = n0 + c0 + j;
            if (e < a.E) a.logits[(int64_t)t * a.E + e] = v[j] + (a.bias ? __ldg(a.bias + e) : 0.0f);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 256;" ::"r"(tmem));
  }
}

// 2-D fp32 tensor map: `inner` elements per row, `rows` rows, box {box_inner, box_rows}, 64-byte swizzle
bool make_map_f32(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                  uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner * 4};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

SumsPlan sums_plan(int N, int K, int T) {
  SumsPlan p{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = (off + bytes + 255) / 256 * 256;
    return at;
  };
  const size_t nb = (size_t)K / 256;
  p.status = take(16);
  p.xg = take((size_t)T * K * 2);
  p.sg = take(nb * 2 * (size_t)T * 16);
  p.dg = take(nb * (size_t)T * 4);
  p.items = take((size_t)((T + kTileN - 1) / kTileN) * (N / kTileM) * sizeof(PItem));
  p.n_items = take(16);
  p.total = off;
  return p;
}

cudaError_t launch_prefill_sums(const SumsArgs& a, cudaStream_t s) {
  switch (a.fmt) {
    case kQ4K: return launch_sums_t<kQ4K>(a, s);
    case kQ2K: return launch_sums_t<kQ2K>(a, s);
    case kQ3K: return launch_sums_t<kQ3K>(a, s);
    case kIQ2G: return launch_sums_t<kIQ2G>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

int prefill_tile_tokens() { return kTileN; }

size_t prefill_item_capacity(int64_t P, int E, int S, int H, int I) {
  const int64_t EpS = E + S;
  return (size_t)(P / kTileN + EpS) * (size_t)std::max(I / 64, H / 128);
}

cudaError_t launch_router_tc(const float* x, const float* w, const float* bias, int T, int H, int E,
                             float* logits, int* status, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  if (H % kRtK) return cudaErrorInvalidValue;
  RouterTcArgs a{};
  if (!make_map_f32(&a.map_x, x, (uint64_t)H, (uint64_t)T, kRtK, kRtM) ||
      !make_map_f32(&a.map_w, w, (uint64_t)H, (uint64_t)E, kRtK, kRtN))
    return cudaErrorInvalidValue;
  a.bias = bias;
  a.logits = logits;
  a.T = T;
  a.H = H;
  a.E = E;
  a.status = status;
  static bool opted = false;
  if (!opted) {
    cudaError_t err = cudaFuncSetAttribute(router_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRtSmAlloc);
    if (err != cudaSuccess) return err;
    opted = true;
  }
  const dim3 grid((E + kRtN - 1) / kRtN, (T + kRtM - 1) / kRtM);
  note_launch();
  router_tc_kernel<<<grid, kRtThreads, kRtSmAlloc, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_prefill_ffn(const PrefillArgs& a, cudaStream_t s) {
  switch (a.fmt) {
    case kQ4K: return launch_prefill_fmt<kQ4K>(a, s);
    case kQ2K: return launch_prefill_fmt<kQ2K>(a, s);
    case kQ3K: return launch_prefill_fmt<kQ3K>(a, s);
    case kIQ2G: return launch_prefill_fmt<kIQ2G>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace moe
