// ORACLE — test infrastructure, not product code.
//
// A plain, slow CPU definition of the per-token Mixture-of-Experts layer with
// block-quantized experts: q8_K activation quantization, router top-k
// (softmax or sigmoid, renormalised over the selected k), token -> expert
// bucketing, per-expert gate/up integer sub-block dot products, SwiGLU, the
// down projection, and the gate-weighted combine into the residual.
//
// It shares no code with the CUDA path and is only built and called by the
// tests, by __graft_entry__.smoke() and by bench.py's CPU baseline.
// Floating point is fp64 except where a step is defined in fp32 (the q8_K
// quantizer).  Integer sub-block sums are int64.  Parallelism is over rows
// or tokens only; every row is computed by one thread in a fixed order.
//
// Sources of the method (page title, section):
//  * Pulsar README, "Fidelity notes": every matmul runs on activations
//    quantized to q8_0/q8_K with integer dp4a dot products.
//  * Pulsar README, "What it does today" (ThinkingCap paragraph):
//    warp-cooperative Q4_K/Q6_K matmuls on q8_K activations; the FFN triple
//    gate/up/down.  Same section: softmax routers (qwen3moe).
//  * Pulsar digest note (rrlab.tech), section 1: a 512-way sigmoid-gated
//    router plus a shared expert with Q2_K experts.
//  * Pulsar README, "How the streaming works": per token, or per prefill
//    chunk as a union across the batch, each selected expert is resolved
//    once; kernels receive explicit per-(token, slot) gate/up/down pointers
//    and a NULL slot means "not mine".
//  * Pulsar README, "Fidelity notes": the per-slot sum is the combine.
//  * Strata summary (bafh001.com): router and shared expert, ~10 experts per
//    token.
// The pages name the formats but print no field layout or formula; the
// super-block fields (fp16 d, fp16 dmin, per-sub-block scale and min, codes;
// w = d*scale*q - dmin*min), the q8_K rule (d = max|x|/127 in fp32,
// q = round-half-away(x/d)) and the byte placement (synth/layout.py) are the
// workload definitions this oracle follows.  The Q5_K/Q3_K/Q6_K-style
// formats (Pulsar README, "What it does today": Q4_K/Q6_K matmuls; "Get a
// model": q3_K/q5_K/q6_K tensors) are this project's reading of those names:
// Q5_K-style = Q4_K-style with 5-bit codes; Q3_K-style: 16 sub-blocks, 3-bit
// codes, 6-bit signed scales, w = d*scale*(q - 4); Q6_K-style: 16
// sub-blocks, 6-bit codes, int8 scales, w = d*scale*(q - 32).  In general
// w = d*scale*(q - o) - dmin*min, with o = 0 and a min for the first three
// formats and o = 4 / 32 and no min (no dmin) for Q3_K/Q6_K-style.
// The pages also name i-quant codebook formats (Pulsar README, "What it does
// today": IQ2_XXS builds; Strata engine article, finding 7: IQ3 codebook
// lookups cost decode compute that K-quant shifts do not) without printing a
// grid.  The IQ2-style grid format here is this project's own: per group of
// 8 weights a grid index into 256 vectors of magnitudes {1, 3, 5} and 7 sign
// bits (the 8th sign makes the minus signs even), per 32 weights a 4-bit
// scale t (scale 2t + 1), fp16 d: w = d * (2t + 1) * sign * C[u][i].  In the
// (q, sc) form above q is the signed grid value, o = 0, no min.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

constexpr int kQ4K = 0;
constexpr int kQ2K = 1;
constexpr int kQ5K = 2;
constexpr int kQ3K = 3;
constexpr int kQ6K = 4;
constexpr int kIQ2G = 5;

// Per format: sub-blocks, header bytes per row (d|dmin or d), scale/min
// bytes per row, code bytes per row, code offset o.  A slab holds the 32
// rows' headers, then their scale/min bytes, then the code lines.
int n_sub(int fmt) { return (fmt == kQ4K || fmt == kQ5K || fmt == kIQ2G) ? 8 : 16; }
int sub_len(int fmt) { return 256 / n_sub(fmt); }
int hdr_bytes(int fmt) { return (fmt == kQ3K || fmt == kQ6K || fmt == kIQ2G) ? 2 : 4; }
int sm_bytes(int fmt) { return fmt == kIQ2G ? 4 : (fmt == kQ2K || fmt == kQ6K) ? 16 : 12; }
int code_bytes(int fmt) {
  switch (fmt) {
    case kQ4K: return 128;
    case kQ2K: return 64;
    case kQ5K: return 160;
    case kQ3K: return 96;
    case kIQ2G: return 64;
    default: return 192;
  }
}
int code_offset(int fmt) { return fmt == kQ3K ? 4 : fmt == kQ6K ? 32 : 0; }
int64_t slab_bytes(int fmt) { return 32 * (int64_t)(hdr_bytes(fmt) + sm_bytes(fmt) + code_bytes(fmt)); }

// The IQ2-style grid: the 256 vectors of {1, 3, 5}^8 with the smallest sum
// of squares, equal sums ordered by the base-3 number of the digits
// (v_i - 1) / 2 (element 0 most significant); index = rank.  Built by
// listing all 3^8 vectors in increasing base-3 order and sorting them
// stably by their sum of squares.
struct Grid {
  int v[256][8];
};
const Grid& iq2g_grid() {
  static const Grid g = [] {
    std::vector<std::pair<int, int>> all;  // (sum of squares, base-3 number)
    for (int t = 0; t < 6561; ++t) {
      int x = t, ss = 0;
      for (int i = 0; i < 8; ++i) {
        const int v = 1 + 2 * (x % 3);
        ss += v * v;
        x /= 3;
      }
      all.push_back({ss, t});
    }
    std::stable_sort(all.begin(), all.end(),
                     [](const std::pair<int, int>& a, const std::pair<int, int>& b) { return a.first < b.first; });
    Grid out;
    for (int u = 0; u < 256; ++u) {
      int x = all[u].second;
      for (int i = 7; i >= 0; --i) {  // the last digit is element 7
        out.v[u][i] = 1 + 2 * (x % 3);
        x /= 3;
      }
    }
    return out;
  }();
  return g;
}

// IEEE 754 binary16 -> double, written out from the format definition.
double half_to_double(uint16_t h) {
  int sign = h >> 15;
  int e = (h >> 10) & 31;
  int m = h & 1023;
  double v;
  if (e == 0)
    v = std::ldexp((double)m, -24);  // subnormal: m * 2^-24
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = std::ldexp((double)(m + 1024), e - 25);  // (1 + m/1024) * 2^(e-15)
  return sign ? -v : v;
}

uint32_t read_le32(const uint8_t* p) {
  return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}

// bits [start, start+len) of a little-endian bit string
int read_bits(const uint8_t* p, int start, int len) {
  int v = 0;
  for (int i = 0; i < len; ++i) {
    int bit = start + i;
    v |= ((p[bit / 8] >> (bit % 8)) & 1) << i;
  }
  return v;
}

struct SuperBlock {
  int q[256];   // codes (unsigned; the signed grid values for the IQ2-style format)
  int sc[16];   // per-sub-block scale (signed for Q3_K/Q6_K-style)
  int mn[16];   // per-sub-block min (0 where the format has none)
  int off;      // code offset o: w = d * sc * (q - o) - dmin * mn
  double d, dmin;
};

// Unpack super-block b of row n of a matrix with nb super-blocks per row.
void unpack_sb(const uint8_t* w, int fmt, int64_t nb, int64_t n, int64_t b, SuperBlock* o) {
  int64_t rg = n / 32;
  int r = (int)(n % 32);
  const uint8_t* slab = w + (rg * nb + b) * slab_bytes(fmt);
  const int hb = hdr_bytes(fmt), smb = sm_bytes(fmt);
  const uint8_t* sm = slab + 32 * hb + smb * r;
  // code line l of this row
  auto line = [&](int l) { return slab + 32 * (hb + smb) + 512 * l + 16 * r; };
  if (hb == 4) {
    uint32_t dm = read_le32(slab + 4 * r);
    o->d = half_to_double((uint16_t)(dm & 0xFFFF));
    o->dmin = half_to_double((uint16_t)(dm >> 16));
  } else {
    o->d = half_to_double((uint16_t)(slab[2 * r] | (slab[2 * r + 1] << 8)));
    o->dmin = 0.0;
  }
  o->off = code_offset(fmt);
  for (int j = 0; j < 16; ++j) o->mn[j] = 0;
  if (fmt == kQ4K || fmt == kQ5K) {
    for (int j = 0; j < 8; ++j) {
      o->sc[j] = read_bits(sm, 6 * j, 6);
      o->mn[j] = read_bits(sm, 48 + 6 * j, 6);
    }
    for (int j = 0; j < 8; ++j)
      for (int i = 0; i < 16; ++i) {
        o->q[32 * j + i] = line(j)[i] & 15;
        o->q[32 * j + 16 + i] = line(j)[i] >> 4;
      }
    if (fmt == kQ5K)  // 5th bits: line 8 + j/4, byte i, bit 2*(j%4) + h -> code i + 16h of sub-block j
      for (int j = 0; j < 8; ++j)
        for (int i = 0; i < 16; ++i)
          for (int h = 0; h < 2; ++h)
            o->q[32 * j + 16 * h + i] |= ((line(8 + j / 4)[i] >> (2 * (j % 4) + h)) & 1) << 4;
  } else if (fmt == kQ2K || fmt == kQ3K) {
    if (fmt == kQ2K)
      for (int j = 0; j < 16; ++j) {
        o->sc[j] = sm[j] & 15;
        o->mn[j] = sm[j] >> 4;
      }
    else
      for (int j = 0; j < 16; ++j) o->sc[j] = read_bits(sm, 6 * j, 6) - 32;
    // low 2 bits: sub-block j in line j/4, bytes 4*(j%4)..: bits 2p.. of byte m = code 4p + m
    for (int j = 0; j < 16; ++j) {
      const uint8_t* base = line(j / 4) + 4 * (j % 4);
      for (int c = 0; c < 16; ++c) o->q[16 * j + c] = (base[c % 4] >> (2 * (c / 4))) & 3;
    }
    if (fmt == kQ3K)  // 3rd bits: line 4 + j/8, bytes 4*((j/2)%4)..: bit p + 4*(j%2) of byte m -> code 4p + m
      for (int j = 0; j < 16; ++j) {
        const uint8_t* base = line(4 + j / 8) + 4 * ((j / 2) % 4);
        for (int c = 0; c < 16; ++c) o->q[16 * j + c] |= ((base[c % 4] >> (c / 4 + 4 * (j % 2))) & 1) << 2;
      }
  } else if (fmt == kIQ2G) {
    // scales: nibble j of the 4 scale bytes; codes: index byte g in line g/16,
    // sign byte g in line 2 + g/16 (byte g % 16 of each)
    const Grid& C = iq2g_grid();
    for (int j = 0; j < 8; ++j) o->sc[j] = 2 * ((sm[j / 2] >> (4 * (j % 2))) & 15) + 1;
    for (int g = 0; g < 32; ++g) {
      const int u = line(g / 16)[g % 16];
      const int sb7 = line(2 + g / 16)[g % 16] & 127;
      int neg = 0;
      for (int i = 0; i < 7; ++i) neg ^= (sb7 >> i) & 1;  // the 8th sign: an even count of minus signs
      const int signs = sb7 | (neg << 7);
      for (int i = 0; i < 8; ++i) o->q[8 * g + i] = ((signs >> i) & 1) ? -C.v[u][i] : C.v[u][i];
    }
  } else {  // Q6_K-style
    for (int j = 0; j < 16; ++j) o->sc[j] = (int)(int8_t)sm[j];
    for (int j = 0; j < 16; ++j)
      for (int i = 0; i < 16; ++i) {
        const int lo = (line(j / 2)[i] >> (4 * (j % 2))) & 15;
        const int hi = (line(8 + j / 4)[i] >> (2 * (j % 4))) & 3;
        o->q[16 * j + i] = lo | (hi << 4);
      }
  }
}

// The min-term coefficient of sub-block j and its scale in the raw-code
// decomposition: mn_j with dmin, or o * sc_j with d for the symmetric formats.
int m_coef(const SuperBlock& sb, int j) { return sb.off ? sb.off * sb.sc[j] : sb.mn[j]; }
double m_scale(const SuperBlock& sb) { return sb.off ? sb.d : sb.dmin; }

// Run f(i) for i in [0, n) on up to nthreads threads (contiguous ranges).
template <class F>
void parallel_for(int64_t n, int nthreads, F f) {
  if (nthreads <= 1 || n <= 1) {
    for (int64_t i = 0; i < n; ++i) f(i);
    return;
  }
  int nt = (int)std::min<int64_t>(nthreads, n);
  std::vector<std::thread> th;
  for (int t = 0; t < nt; ++t) {
    int64_t lo = n * t / nt, hi = n * (t + 1) / nt;
    th.emplace_back([=, &f] {
      for (int64_t i = lo; i < hi; ++i) f(i);
    });
  }
  for (auto& x : th) x.join();
}

// q8_K quantization of one 256-element block, in fp32 as the format defines:
// d = max|x| / 127 (one IEEE fp32 division), q = round-half-away(x / d)
// (IEEE fp32 division, then rounding; |q| <= 127), q = 0 when d == 0.
void q8k_block(const float* x, int8_t* q, float* d) {
  float amax = 0.0f;
  for (int i = 0; i < 256; ++i) amax = std::max(amax, std::fabs(x[i]));
  float db = amax / 127.0f;
  *d = db;
  for (int i = 0; i < 256; ++i) {
    float v = 0.0f;
    if (db != 0.0f) {
      v = std::round(x[i] / db);  // std::round: halfway cases away from zero
      v = std::min(127.0f, std::max(-127.0f, v));
    }
    q[i] = (int8_t)v;
  }
}

// y[n] for one activation row (codes qa[K], scales da[K/256]):
//   y[n] = sum_b da[b] * (d_w * sum_j sc_j * isum_j  -  dmin * sum_j mn_j * bsum_j)
// with isum_j = sum over sub-block j of (q_w - o) * q_a and bsum_j = sum of q_a.
double row_dot(const uint8_t* w, int fmt, int64_t nb, int64_t n, const int8_t* qa, const float* da) {
  SuperBlock sb;
  double acc = 0.0;
  int ns = n_sub(fmt), sl = sub_len(fmt);
  for (int64_t b = 0; b < nb; ++b) {
    unpack_sb(w, fmt, nb, n, b, &sb);
    int64_t S = 0, M = 0;
    for (int j = 0; j < ns; ++j) {
      int64_t isum = 0, bsum = 0;
      for (int i = 0; i < sl; ++i) {
        int k = j * sl + i;
        isum += (int64_t)(sb.q[k] - sb.off) * qa[256 * b + k];
        bsum += qa[256 * b + k];
      }
      S += (int64_t)sb.sc[j] * isum;
      M += (int64_t)sb.mn[j] * bsum;
    }
    acc += (double)da[b] * (sb.d * (double)S - sb.dmin * (double)M);
  }
  return acc;
}

double silu(double g) { return g / (1.0 + std::exp(-g)); }

// One expert's FFN for one token: G, U = gate/up matvecs on q8_K(x); h =
// silu(G) * U; h is rounded to fp32 and re-quantized to q8_K (all matmuls run
// on q8_K activations); y = down matvec.  y has H entries.
void expert_ffn_token(const uint8_t* gate, const uint8_t* up, const uint8_t* down, int fmt, int64_t H,
                      int64_t I, const int8_t* xq, const float* xd, double* y, int nthreads,
                      float* h_out, int8_t* hq_out, float* hd_out) {
  std::vector<double> G(I), U(I);
  int64_t nbH = H / 256, nbI = I / 256;
  parallel_for(I, nthreads, [&](int64_t n) {
    G[n] = row_dot(gate, fmt, nbH, n, xq, xd);
    U[n] = row_dot(up, fmt, nbH, n, xq, xd);
  });
  std::vector<float> h32(I);
  for (int64_t n = 0; n < I; ++n) h32[n] = (float)(silu(G[n]) * U[n]);
  std::vector<int8_t> hq(I);
  std::vector<float> hd(nbI);
  for (int64_t b = 0; b < nbI; ++b) q8k_block(&h32[256 * b], &hq[256 * b], &hd[b]);
  if (h_out) std::memcpy(h_out, h32.data(), sizeof(float) * I);
  if (hq_out) std::memcpy(hq_out, hq.data(), I);
  if (hd_out) std::memcpy(hd_out, hd.data(), sizeof(float) * nbI);
  parallel_for(H, nthreads, [&](int64_t n) { y[n] = row_dot(down, fmt, nbI, n, hq.data(), hd.data()); });
}

}  // namespace

extern "C" {

// fp16 bit pattern -> double (exposed for the format pins).
double orc_half_to_double(uint16_t h) { return half_to_double(h); }

// The IQ2-style grid as 256 x 8 ints (exposed for the format pins).
void orc_iq2g_grid(int32_t* out) {
  const Grid& C = iq2g_grid();
  for (int u = 0; u < 256; ++u)
    for (int i = 0; i < 8; ++i) out[8 * u + i] = C.v[u][i];
}

// Unpack the fields of super-block (row n, block b) of a [N, K] matrix.
// q: 256 ints, sc/mn: n_sub ints, dd: {d, dmin}.
void orc_unpack_sb(const uint8_t* w, int fmt, int64_t N, int64_t K, int64_t n, int64_t b, int32_t* q,
                   int32_t* sc, int32_t* mn, double* dd) {
  (void)N;
  SuperBlock sb;
  unpack_sb(w, fmt, K / 256, n, b, &sb);
  for (int i = 0; i < 256; ++i) q[i] = sb.q[i];
  for (int j = 0; j < n_sub(fmt); ++j) {
    sc[j] = sb.sc[j];
    mn[j] = sb.mn[j];
  }
  dd[0] = sb.d;
  dd[1] = sb.dmin;
}

// Dequantized matrix W[N, K] in fp64: w = d * sc_j * (q - o) - dmin * mn_j.
void orc_dequant_matrix(const uint8_t* w, int fmt, int64_t N, int64_t K, double* out) {
  int64_t nb = K / 256;
  int sl = sub_len(fmt);
  SuperBlock sb;
  for (int64_t n = 0; n < N; ++n)
    for (int64_t b = 0; b < nb; ++b) {
      unpack_sb(w, fmt, nb, n, b, &sb);
      for (int k = 0; k < 256; ++k) {
        int j = k / sl;
        out[n * K + 256 * b + k] = sb.d * sb.sc[j] * (sb.q[k] - sb.off) - sb.dmin * sb.mn[j];
      }
    }
}

// q8_K quantization of x[T, K] (K a multiple of 256): codes q[T, K],
// scales d[T, K/256], and sums of every 16 consecutive codes bsum16[T, K/16].
void orc_q8k_quantize(const float* x, int64_t T, int64_t K, int8_t* q, float* d, int16_t* bsum16) {
  int64_t nb = K / 256;
  for (int64_t t = 0; t < T; ++t)
    for (int64_t b = 0; b < nb; ++b) q8k_block(x + t * K + 256 * b, q + t * K + 256 * b, d + t * nb + b);
  if (bsum16)
    for (int64_t t = 0; t < T; ++t)
      for (int64_t g = 0; g < K / 16; ++g) {
        int s = 0;
        for (int i = 0; i < 16; ++i) s += q[t * K + 16 * g + i];
        bsum16[t * (K / 16) + g] = (int16_t)s;
      }
}

// Integer sub-block sums of activation rows qa[T, K] against W[N, K]:
// isum[t][n][b][j] = sum_{i in sub-block j of SB b} q_w * q_a  (int32),
// bsum[t][b][j]    = sum_{i in sub-block j of SB b} q_a.
void orc_subblock_dots(const uint8_t* w, int fmt, int64_t N, int64_t K, const int8_t* qa, int64_t T,
                       int32_t* isum, int32_t* bsum) {
  int64_t nb = K / 256;
  int ns = n_sub(fmt), sl = sub_len(fmt);
  SuperBlock sb;
  for (int64_t t = 0; t < T; ++t)
    for (int64_t b = 0; b < nb; ++b)
      for (int j = 0; j < ns; ++j) {
        int64_t s = 0;
        for (int i = 0; i < sl; ++i) s += qa[t * K + 256 * b + j * sl + i];
        bsum[(t * nb + b) * ns + j] = (int32_t)s;
      }
  for (int64_t n = 0; n < N; ++n)
    for (int64_t b = 0; b < nb; ++b) {
      unpack_sb(w, fmt, nb, n, b, &sb);
      for (int64_t t = 0; t < T; ++t)
        for (int j = 0; j < ns; ++j) {
          int64_t s = 0;
          for (int i = 0; i < sl; ++i) s += (int64_t)sb.q[j * sl + i] * qa[t * K + 256 * b + j * sl + i];
          isum[((t * N + n) * nb + b) * ns + j] = (int32_t)s;
        }
    }
}

// Integer super-block sums of activation rows qa[T, K] against W[N, K] on the
// raw codes, the integer part of row_dot before the scales are applied:
//   S[t][n][b] = sum_j sc_j * isum_j  (isum_j = sum of q_w * q_a, raw codes)
//   M[t][n][b] = sum_j m_j * bsum_j   (int64)
// with m_j = mn_j for the formats with a min, and m_j = o * sc_j for the
// symmetric formats; then y = sum_b da * (d * S - m_scale * M), m_scale =
// dmin or d.  (The same value as row_dot: sum_j sc_j sum_i (q - o) a =
// S - o * sum_j sc_j bsum_j.)
void orc_superblock_sums(const uint8_t* w, int fmt, int64_t N, int64_t K, const int8_t* qa, int64_t T,
                         int64_t* S, int64_t* M) {
  int64_t nb = K / 256;
  int ns = n_sub(fmt), sl = sub_len(fmt);
  SuperBlock sb;
  for (int64_t n = 0; n < N; ++n)
    for (int64_t b = 0; b < nb; ++b) {
      unpack_sb(w, fmt, nb, n, b, &sb);
      for (int64_t t = 0; t < T; ++t) {
        const int8_t* q = qa + t * K + 256 * b;
        int64_t s = 0, m = 0;
        for (int j = 0; j < ns; ++j) {
          int64_t isum = 0, bsum = 0;
          for (int i = 0; i < sl; ++i) {
            isum += (int64_t)sb.q[j * sl + i] * q[j * sl + i];
            bsum += q[j * sl + i];
          }
          s += (int64_t)sb.sc[j] * isum;
          m += (int64_t)m_coef(sb, j) * bsum;
        }
        S[(t * N + n) * nb + b] = s;
        M[(t * N + n) * nb + b] = m;
      }
    }
}

// y[T, N] = block-quantized W[N, K] applied to q8_K rows (qa[T, K], da[T, K/256]).
void orc_qmatvec(const uint8_t* w, int fmt, int64_t N, int64_t K, const int8_t* qa, const float* da,
                 int64_t T, double* y, int nthreads) {
  int64_t nb = K / 256;
  parallel_for(N, nthreads, [&](int64_t n) {
    for (int64_t t = 0; t < T; ++t) y[t * N + n] = row_dot(w, fmt, nb, n, qa + t * K, da + t * nb);
  });
}

// Magnitude of the terms that orc_qmatvec sums into y[t][n], for
// floating-point error bounds of an implementation that sums them in fp32:
//   a[t][n] = sum_b |da[b]| * (|d_w| * |S_b| + |m_scale| * |M_b|),
// S_b and M_b the raw-code sums of orc_superblock_sums (m_scale = dmin, or
// d for the symmetric formats).  |y[t][n]| <= a[t][n], with equality when
// no term cancels another.
void orc_qmatvec_absterms(const uint8_t* w, int fmt, int64_t N, int64_t K, const int8_t* qa, const float* da,
                          int64_t T, double* a, int nthreads) {
  int64_t nb = K / 256;
  int ns = n_sub(fmt), sl = sub_len(fmt);
  parallel_for(N, nthreads, [&](int64_t n) {
    SuperBlock sb;
    for (int64_t t = 0; t < T; ++t) {
      const int8_t* q = qa + t * K;
      double acc = 0.0;
      for (int64_t b = 0; b < nb; ++b) {
        unpack_sb(w, fmt, nb, n, b, &sb);
        int64_t S = 0, M = 0;
        for (int j = 0; j < ns; ++j) {
          int64_t isum = 0, bsum = 0;
          for (int i = 0; i < sl; ++i) {
            isum += (int64_t)sb.q[j * sl + i] * q[256 * b + j * sl + i];
            bsum += q[256 * b + j * sl + i];
          }
          S += (int64_t)sb.sc[j] * isum;
          M += (int64_t)m_coef(sb, j) * bsum;
        }
        acc += std::fabs((double)da[t * nb + b]) *
               (std::fabs(sb.d) * std::fabs((double)S) + std::fabs(m_scale(sb)) * std::fabs((double)M));
      }
      a[t * N + n] = acc;
    }
  });
}

// Router: logits[t][e] = sum_h W_r[e][h] * x[t][h] (+ bias[e]) in fp64 from
// the fp32 inputs.  Top-k by a full stable sort on descending logit (equal
// logits: lower expert index first).  Gates renormalised over the k:
//   route 0 (softmax): g_s = exp(l_s - l_max) / sum_sel exp(l - l_max)
//   route 1 (sigmoid): g_s = sigma(l_s) / sum_sel sigma(l)
// gap[t] = l_(k) - l_(k+1) (+inf when k == E).
// forced_ids (nullable): use these ids instead of the top-k (the gates are
// still computed from the logits of the forced ids).
void orc_route(const float* x, const float* wr, const float* bias, int64_t T, int64_t H, int64_t E,
               int64_t k, int route, const int32_t* forced_ids, double* logits, int32_t* ids,
               double* gates, double* gap) {
  std::vector<int> order(E);
  for (int64_t t = 0; t < T; ++t) {
    double* l = logits + t * E;
    for (int64_t e = 0; e < E; ++e) {
      double s = 0.0;
      for (int64_t h = 0; h < H; ++h) s += (double)wr[e * H + h] * (double)x[t * H + h];
      if (bias) s += (double)bias[e];
      l[e] = s;
    }
    for (int64_t e = 0; e < E; ++e) order[e] = (int)e;
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return l[a] > l[b]; });
    if (gap) gap[t] = (k < E) ? l[order[k - 1]] - l[order[k]] : INFINITY;
    int32_t* id = ids + t * k;
    for (int64_t s = 0; s < k; ++s) id[s] = forced_ids ? forced_ids[t * k + s] : order[s];
    double* g = gates + t * k;
    if (route == 0) {
      double lmax = -INFINITY;
      for (int64_t s = 0; s < k; ++s) lmax = std::max(lmax, l[id[s]]);
      double z = 0.0;
      for (int64_t s = 0; s < k; ++s) z += std::exp(l[id[s]] - lmax);
      for (int64_t s = 0; s < k; ++s) g[s] = std::exp(l[id[s]] - lmax) / z;
    } else {
      double z = 0.0;
      for (int64_t s = 0; s < k; ++s) z += 1.0 / (1.0 + std::exp(-l[id[s]]));
      for (int64_t s = 0; s < k; ++s) g[s] = (1.0 / (1.0 + std::exp(-l[id[s]]))) / z;
    }
  }
}

// Bucketing of the T*k (token, slot) pairs by expert, stable by token, plus
// one bucket per shared expert holding every token.
//   counts[e] (E + S entries), offsets[e] (E + S + 1 entries, exclusive sum),
//   perm[offsets[e] + i] = the slot index p of the i-th pair of bucket e,
//   where p = t*k + s for routed pairs and p = T*k + sh*T + t for shared.
void orc_bucket(const int32_t* ids, int64_t T, int64_t k, int64_t E, int64_t S, int32_t* counts,
                int32_t* offsets, int32_t* perm) {
  for (int64_t e = 0; e < E + S; ++e) counts[e] = 0;
  for (int64_t p = 0; p < T * k; ++p) counts[ids[p]]++;
  for (int64_t sh = 0; sh < S; ++sh) counts[E + sh] = (int32_t)T;
  offsets[0] = 0;
  for (int64_t e = 0; e < E + S; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int64_t pos = 0;
  for (int64_t e = 0; e < E; ++e)
    for (int64_t t = 0; t < T; ++t)
      for (int64_t s = 0; s < k; ++s)
        if (ids[t * k + s] == e) perm[pos++] = (int32_t)(t * k + s);
  for (int64_t sh = 0; sh < S; ++sh)
    for (int64_t t = 0; t < T; ++t) perm[pos++] = (int32_t)(T * k + sh * T + t);
}

// One expert FFN (gate/up/down matrices) on T tokens of q8_K activations.
// y[T, H].  Optionally returns h (fp32 [T, I]) and its q8_K codes/scales.
void orc_expert_ffn(const uint8_t* gate, const uint8_t* up, const uint8_t* down, int fmt, int64_t H,
                    int64_t I, const int8_t* xq, const float* xd, int64_t T, double* y, float* h_out,
                    int8_t* hq_out, float* hd_out, int nthreads) {
  for (int64_t t = 0; t < T; ++t)
    expert_ffn_token(gate, up, down, fmt, H, I, xq + t * H, xd + t * (H / 256), y + t * H, nthreads,
                     h_out ? h_out + t * I : nullptr, hq_out ? hq_out + t * I : nullptr,
                     hd_out ? hd_out + t * (I / 256) : nullptr);
}

// The MoE layer on T tokens:
//   out[t] = residual[t] + sum_{s<k} g[t][s] * FFN_{ids[t][s]}(q8_K(x[t]))
//                        + sum_{sh<S} FFN_{E+sh}(q8_K(x[t]))
// gate/up/down: E + S matrix pointers (host); a NULL gate pointer means the
// expert is not present and contributes nothing.  residual may be NULL.
// forced_ids (nullable) replaces the router's top-k.  out is fp64.
void orc_layer_forward(int fmt, int64_t H, int64_t I, int64_t E, int64_t k, int64_t S, int route,
                       const uint8_t* const* gate, const uint8_t* const* up, const uint8_t* const* down,
                       const float* wr, const float* bias, const float* x, const float* residual,
                       int64_t T, const int32_t* forced_ids, double* out, int32_t* ids, double* gates,
                       double* gap, int nthreads) {
  std::vector<int8_t> xq(T * H);
  std::vector<float> xd(T * (H / 256));
  orc_q8k_quantize(x, T, H, xq.data(), xd.data(), nullptr);
  std::vector<double> logits(T * E);
  orc_route(x, wr, bias, T, H, E, k, route, forced_ids, logits.data(), ids, gates, gap);
  std::vector<double> y(H);
  for (int64_t t = 0; t < T; ++t) {
    double* o = out + t * H;
    for (int64_t h = 0; h < H; ++h) o[h] = residual ? (double)residual[t * H + h] : 0.0;
    const int8_t* q = xq.data() + t * H;
    const float* d = xd.data() + t * (H / 256);
    for (int64_t s = 0; s < k; ++s) {
      int e = ids[t * k + s];
      if (!gate[e]) continue;
      expert_ffn_token(gate[e], up[e], down[e], fmt, H, I, q, d, y.data(), nthreads, nullptr, nullptr,
                       nullptr);
      for (int64_t h = 0; h < H; ++h) o[h] += gates[t * k + s] * y[h];
    }
    for (int64_t sh = 0; sh < S; ++sh) {
      int64_t e = E + sh;
      if (!gate[e]) continue;
      expert_ffn_token(gate[e], up[e], down[e], fmt, H, I, q, d, y.data(), nthreads, nullptr, nullptr,
                       nullptr);
      for (int64_t h = 0; h < H; ++h) o[h] += y[h];
    }
  }
}

}  // extern "C"
