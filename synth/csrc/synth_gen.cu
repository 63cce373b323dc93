// Device-side generator of random block-quantized weight matrices.
//
// Produces, byte for byte, what synth.gen_matrix() produces on the host (the
// counter-based SplitMix64 stream and the slab layout are described in
// synth/__init__.py and synth/layout.py).  It exists because the large
// workloads hold tens of GB of weights, which are made where they are used.
// Input generation only: nothing here is part of the MoE layer's arithmetic.
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9ull;
  z ^= z >> 27;
  z *= 0x94D049BB133111EBull;
  z ^= z >> 31;
  return z;
}

__device__ __forceinline__ uint64_t draw(uint64_t key, uint64_t sb, uint64_t i) {
  return mix64(key + (sb * 32ull + i + 1ull) * kGamma);
}

__device__ __forceinline__ uint16_t d_bits(uint64_t r) {
  float u = (float)(uint32_t)(r >> 40) * 0x1p-24f;
  float v = __fadd_rn(1e-4f, __fmul_rn(u, 9e-4f));
  return __half_as_ushort(__float2half_rn(v));
}

__device__ __forceinline__ uint16_t dmin_bits(uint64_t r) {
  float u = (float)(uint32_t)(r >> 40) * 0x1p-24f;
  float v = __fmul_rn(u, 5e-4f);
  return __half_as_ushort(__float2half_rn(v));
}

__device__ __forceinline__ uint4 line_of(uint64_t a, uint64_t b) {
  return make_uint4((uint32_t)a, (uint32_t)(a >> 32), (uint32_t)b, (uint32_t)(b >> 32));
}

// one thread per super-block (row n, column block b)
__global__ void fill_q4k(uint8_t* __restrict__ w, int64_t N, int64_t nb, uint64_t key) {
  int64_t sb = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (sb >= N * nb) return;
  int64_t n = sb / nb, b = sb % nb;
  int64_t rg = n >> 5;
  int r = (int)(n & 31);
  uint8_t* slab = w + (rg * nb + b) * 4608;
  uint64_t c[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) c[i] = draw(key, (uint64_t)sb, i);
#pragma unroll
  for (int j = 0; j < 8; ++j)
    *reinterpret_cast<uint4*>(slab + 512 + 512 * j + 16 * r) = line_of(c[2 * j], c[2 * j + 1]);
  uint64_t s0 = draw(key, sb, 16), s1 = draw(key, sb, 17);
  uint32_t* sm = reinterpret_cast<uint32_t*>(slab + 128 + 12 * r);
  sm[0] = (uint32_t)s0;
  sm[1] = (uint32_t)(s0 >> 32);
  sm[2] = (uint32_t)s1;
  uint32_t dm = (uint32_t)d_bits(draw(key, sb, 18)) | ((uint32_t)dmin_bits(draw(key, sb, 19)) << 16);
  *reinterpret_cast<uint32_t*>(slab + 4 * r) = dm;
}

__global__ void fill_q2k(uint8_t* __restrict__ w, int64_t N, int64_t nb, uint64_t key) {
  int64_t sb = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (sb >= N * nb) return;
  int64_t n = sb / nb, b = sb % nb;
  int64_t rg = n >> 5;
  int r = (int)(n & 31);
  uint8_t* slab = w + (rg * nb + b) * 2688;
  uint64_t c[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) c[i] = draw(key, (uint64_t)sb, i);
#pragma unroll
  for (int l = 0; l < 4; ++l)
    *reinterpret_cast<uint4*>(slab + 640 + 512 * l + 16 * r) = line_of(c[2 * l], c[2 * l + 1]);
  *reinterpret_cast<uint4*>(slab + 128 + 16 * r) = line_of(draw(key, sb, 8), draw(key, sb, 9));
  uint32_t dm = (uint32_t)d_bits(draw(key, sb, 10)) | ((uint32_t)dmin_bits(draw(key, sb, 11)) << 16);
  *reinterpret_cast<uint32_t*>(slab + 4 * r) = dm;
}

// The other formats, one thread per super-block: NCODE code draws fill the
// code lines in order (line L = draws 2L, 2L+1, the planes one after the
// other), two draws the scale/min bytes (SMB of them), then d and, with a
// 4-byte header, dmin.  Field offsets: header HB bytes per row, then SMB.
template <int NCODE, int HB, int SMB>
__global__ void fill_generic(uint8_t* __restrict__ w, int64_t N, int64_t nb, uint64_t key) {
  constexpr int kSlab = 32 * (HB + SMB + 8 * NCODE);
  constexpr int kSmOff = 32 * HB, kCodeOff = 32 * (HB + SMB);
  int64_t sb = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (sb >= N * nb) return;
  int64_t n = sb / nb, b = sb % nb;
  int64_t rg = n >> 5;
  int r = (int)(n & 31);
  uint8_t* slab = w + (rg * nb + b) * kSlab;
#pragma unroll
  for (int l = 0; l < NCODE / 2; ++l)
    *reinterpret_cast<uint4*>(slab + kCodeOff + 512 * l + 16 * r) =
        line_of(draw(key, (uint64_t)sb, 2 * l), draw(key, (uint64_t)sb, 2 * l + 1));
  const uint64_t s0 = draw(key, sb, NCODE), s1 = draw(key, sb, NCODE + 1);
  uint32_t* sm = reinterpret_cast<uint32_t*>(slab + kSmOff + SMB * r);
  sm[0] = (uint32_t)s0;
  if (SMB >= 12) {
    sm[1] = (uint32_t)(s0 >> 32);
    sm[2] = (uint32_t)s1;
  }
  if (SMB == 16) sm[3] = (uint32_t)(s1 >> 32);
  const uint16_t db = d_bits(draw(key, sb, NCODE + 2));
  if (HB == 4)
    *reinterpret_cast<uint32_t*>(slab + 4 * r) = (uint32_t)db | ((uint32_t)dmin_bits(draw(key, sb, NCODE + 3)) << 16);
  else
    *reinterpret_cast<uint16_t*>(slab + 2 * r) = db;
}

}  // namespace

extern "C" {

// Fill one [N, K] matrix at dst (device pointer, 16-byte aligned) with the
// stream of `key`.  fmt 0 = Q4_K-style, 1 = Q2_K-style, 2 = Q5_K-style,
// 3 = Q3_K-style, 4 = Q6_K-style, 5 = IQ2-style grid format.  Returns 0 on success, 1 on a bad argument,
// 2 on a CUDA launch error.
int synth_fill_matrix(void* dst, int fmt, int64_t N, int64_t K, uint64_t key, void* stream) {
  if (!dst || N <= 0 || K <= 0 || N % 256 || K % 256 || fmt < 0 || fmt > 5) return 1;
  if (reinterpret_cast<uintptr_t>(dst) & 15) return 1;
  int64_t nb = K / 256;
  int64_t total = N * nb;
  int threads = 256;
  unsigned blocks = (unsigned)((total + threads - 1) / threads);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(dst);
  switch (fmt) {
    case 0: fill_q4k<<<blocks, threads, 0, s>>>(w, N, nb, key); break;
    case 1: fill_q2k<<<blocks, threads, 0, s>>>(w, N, nb, key); break;
    case 2: fill_generic<20, 4, 12><<<blocks, threads, 0, s>>>(w, N, nb, key); break;
    case 3: fill_generic<12, 2, 12><<<blocks, threads, 0, s>>>(w, N, nb, key); break;
    case 4: fill_generic<24, 2, 16><<<blocks, threads, 0, s>>>(w, N, nb, key); break;
    default: fill_generic<8, 2, 4><<<blocks, threads, 0, s>>>(w, N, nb, key); break;
  }
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

// Fill `count` matrices of equal shape: dst[i] receives the stream keys[i].
// Both arrays are host arrays.
int synth_fill_matrices(int count, void* const* dst, const uint64_t* keys, int fmt, int64_t N,
                        int64_t K, void* stream) {
  for (int i = 0; i < count; ++i) {
    int rc = synth_fill_matrix(dst[i], fmt, N, K, keys[i], stream);
    if (rc) return rc;
  }
  return 0;
}

}  // extern "C"
