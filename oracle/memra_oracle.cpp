// memra CPU oracle -- TEST INFRASTRUCTURE ONLY.
//
// A plain, slow, obviously-correct C++ statement of what the Q8_0 decode hot path
// computes.  Only the test suite, the smoke check and the benchmark's CPU-baseline
// leg may load this library.  It shares no code, header, table or helper with the
// CUDA library under block_quantized_decode_quantize_gb300/csrc, and neither side
// includes or links the other.
//
// Sources.  The pages about memra (memra wiki, github.com/avifenesh/memra/wiki,
// feature list; and "memra performance", docs/PERFORMANCE.md, historical 27B
// board) name Q8_0 decode through split-plane repacked matvecs with warp-level
// dp4a, Q8_0 weights, speculative K+1 verify and routed MoE experts, but print no
// block layout, formula or worked example.  The arithmetic below therefore follows
// the workload definitions this project is built to (GGUF-style Q8_0: 32 int8
// quants and one fp16 scale per 32-element block along K; activations quantised
// per 32-block the same way with the scale kept in fp32; y[n] = sum_b d_w*d_x*s_b
// with exact int32 block sums s_b, accumulated in fp32).  Readings where the text
// is silent are listed in the project design notes and restated beside each
// function here.
//
// Build: g++ -O2 -fno-fast-math -ffp-contract=off [-fopenmp] -shared -fPIC.
// -ffp-contract=off matters: every fp32 multiply and add below is a separately
// rounded IEEE operation, in the order written.
//
// Parity status: every exported function is pinned by tests that do not call it
// through itself (closed forms, invariants, brute force in int64 / fp64, numpy's
// IEEE conversions, libm).  No function here is "parity unpinned".

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

uint32_t bits_of(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  return u;
}

float float_of(uint32_t u) {
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// IEEE binary16 round-to-nearest-even of a finite or infinite fp32 value, written
// from the definition: find the fp16 quantum at |f|'s binade, take the nearest
// integer multiple of it (ties to even via rint in the default rounding mode), and
// encode.  Everything is exact in double: |f| has a 24-bit significand and the
// quantum is a power of two.
uint16_t f16_rne(float f) {
  const uint32_t u = bits_of(f);
  const uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
  if (std::isnan(f)) return (uint16_t)(sign | 0x7e00u);
  if (std::isinf(f)) return (uint16_t)(sign | 0x7c00u);
  const double a = std::fabs((double)f);
  if (a == 0.0) return sign;
  int e2;                      // a = m * 2^e2 with m in [0.5, 1)
  std::frexp(a, &e2);
  int e = e2 - 1;              // a in [2^e, 2^(e+1))
  if (e < -14) e = -14;        // below the normal range the quantum stays 2^-24
  const double quantum = std::ldexp(1.0, e - 10);
  const double n = std::rint(a / quantum);  // ties to even
  // n is in [1024, 2048] for the normal range, [0, 1024] for subnormals.  The
  // binary16 encoding is contiguous in (exponent, mantissa), so the code is
  // (e + 15 - 1) * 1024 + n for normals and n for subnormals.
  uint32_t code;
  if (e == -14 && n < 1024.0) {
    code = (uint32_t)n;
  } else {
    code = (uint32_t)(e + 14) * 1024u + (uint32_t)n;
  }
  if (code >= 0x7c00u) code = 0x7c00u;  // overflow to infinity
  return (uint16_t)(sign | code);
}

// binary16 -> fp32, exact.
float f16_to_f32(uint16_t h) {
  const int sign = (h >> 15) & 1;
  const int ex = (h >> 10) & 0x1f;
  const int man = h & 0x3ff;
  double v;
  if (ex == 0) {
    v = std::ldexp((double)man, -24);
  } else if (ex == 31) {
    v = man ? NAN : INFINITY;
  } else {
    v = std::ldexp((double)(1024 + man), ex - 25);
  }
  return (float)(sign ? -v : v);
}

// bfloat16 -> fp32 is the upper half of the fp32 word: exact.
float bf16_to_f32(uint16_t b) { return float_of((uint32_t)b << 16); }

// q = clamp(round-half-away(v / d), -127, 127); d == 0 gives q = 0.  The division
// is one IEEE fp32 division; roundf rounds halves away from zero.
int8_t quant_one(float v, float d) {
  if (d == 0.0f) return 0;
  float r = roundf(v / d);
  if (r > 127.0f) r = 127.0f;
  if (r < -127.0f) r = -127.0f;
  return (int8_t)r;
}

float block_amax(const float* v) {
  float amax = 0.0f;
  for (int i = 0; i < 32; ++i) {
    const float a = std::fabs(v[i]);
    if (a > amax) amax = a;
  }
  return amax;
}

int threads_or_one(int threads) { return threads > 0 ? threads : 1; }

}  // namespace

extern "C" {

// ---------------------------------------------------------------------------
// Scalar conversions, exported so the tests can pin them against numpy.
// ---------------------------------------------------------------------------
uint16_t oracle_f32_to_f16(float f) { return f16_rne(f); }
float oracle_f16_to_f32(uint16_t h) { return f16_to_f32(h); }
float oracle_bf16_to_f32(uint16_t b) { return bf16_to_f32(b); }

// ---------------------------------------------------------------------------
// Weight ingest (GGUF-style Q8_0 along K, split into two planes).
// w: fp32 [N][K], K % 32 == 0.  q: int8 [N][K].  d: fp16 bits [N][K/32].
// Per block: amax = max|w|; d16 = fp16_rne(amax / 127); q = clamp(round-half-
// away(w / float(d16)), +-127).  Reading: the quotient uses the STORED fp16 scale
// (as the dequantised weight d16*q is what the dot product sees); the clamp only
// acts when fp16 rounding shrank a subnormal scale.
// ---------------------------------------------------------------------------
void oracle_quantize_q8_0(const float* w, int64_t N, int64_t K, int8_t* q, uint16_t* d) {
  const int64_t nb = K / 32;
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t b = 0; b < nb; ++b) {
      const float* blk = w + n * K + b * 32;
      const float amax = block_amax(blk);
      const uint16_t d16 = f16_rne(amax / 127.0f);
      const float dv = f16_to_f32(d16);
      d[n * nb + b] = d16;
      for (int i = 0; i < 32; ++i) q[n * K + b * 32 + i] = quant_one(blk[i], dv);
    }
  }
}

// ---------------------------------------------------------------------------
// Weight ingest to Q4_0 (the pages' other split-plane decode format; memra wiki,
// feature list, which names NVFP4, Q4_0 and Q8_0 decode through split-plane
// matvecs).  The pages name the format and print nothing of it; the reading here is
// GGUF's Q4_0 block restated: 32 consecutive weights of a row share one fp16 scale d and carry
// unsigned 4-bit codes q in [0, 15] with w ~= d * (q - 8).
//   m  = the block element of largest magnitude (the first one on a tie);
//   d  = fp16_rne(m / -8), so that m itself maps to q - 8 = -8 (d = +0 when the
//        block is all zeros);
//   q  = clamp(round-half-away(w / float(d)) + 8, 0, 15); d == 0 gives q = 8.
// Split planes: q4 [N][K/2] bytes and d [N][K/32] fp16 bits.  Byte j < 16 of a
// block holds element j in its low nibble and element j + 16 in its high nibble.
// ---------------------------------------------------------------------------
void oracle_quantize_q4_0(const float* w, int64_t N, int64_t K, uint8_t* q4, uint16_t* d) {
  const int64_t nb = K / 32;
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t b = 0; b < nb; ++b) {
      const float* blk = w + n * K + b * 32;
      float m = 0.0f;
      float amax = 0.0f;
      for (int i = 0; i < 32; ++i) {
        if (std::fabs(blk[i]) > amax) {
          amax = std::fabs(blk[i]);
          m = blk[i];
        }
      }
      const uint16_t d16 = amax == 0.0f ? (uint16_t)0 : f16_rne(m / -8.0f);  // +0 if all zero
      const float dv = f16_to_f32(d16);
      d[n * nb + b] = d16;
      int code[32];
      for (int i = 0; i < 32; ++i) {
        if (dv == 0.0f) {
          code[i] = 8;
        } else {
          int c = (int)std::roundf(blk[i] / dv) + 8;
          code[i] = c < 0 ? 0 : (c > 15 ? 15 : c);
        }
      }
      uint8_t* out = q4 + n * (K / 2) + b * 16;
      for (int j = 0; j < 16; ++j) out[j] = (uint8_t)(code[j] | (code[j + 16] << 4));
    }
  }
}

// Q4_0 codes as signed int8 values q - 8, row-major [N][K]: the weight operand of
// the block dot.  With them the Q4_0 product is the Q8_0 product below, term for
// term: y[m][n] = sum_b (d_w * d_x) * s_b with s_b = sum_i (q_i - 8) * xq_i.
void oracle_unpack_q4_0(const uint8_t* q4, int64_t N, int64_t K, int8_t* wq) {
  for (int64_t n = 0; n < N; ++n)
    for (int64_t b = 0; b < K / 32; ++b)
      for (int j = 0; j < 16; ++j) {
        const uint8_t byte = q4[n * (K / 2) + b * 16 + j];
        wq[n * K + b * 32 + j] = (int8_t)((int)(byte & 0x0F) - 8);
        wq[n * K + b * 32 + j + 16] = (int8_t)((int)(byte >> 4) - 8);
      }
}

// ---------------------------------------------------------------------------
// Repack from GGUF's interleaved block arrays to the two planes (the pages' "split-
// plane repacked" matvecs: memra wiki, feature list).  The pages print neither
// layout; the reading is GGUF's:
//   Q8_0 block, 34 bytes: the fp16 scale (little-endian), then the 32 int8 quants;
//   Q4_0 block, 18 bytes: the fp16 scale (little-endian), then 16 bytes whose byte j
//        holds element j's code in its low nibble and element j+16's in its high one.
// A row of K weights is K/32 consecutive blocks, rows one after another.  The
// repack is byte for byte: no value is changed.
// ---------------------------------------------------------------------------
void oracle_repack_q8_0(const uint8_t* blocks, int64_t N, int64_t K, int8_t* q, uint16_t* d) {
  const int64_t nb = K / 32;
  for (int64_t n = 0; n < N; ++n)
    for (int64_t b = 0; b < nb; ++b) {
      const uint8_t* blk = blocks + (n * nb + b) * 34;
      d[n * nb + b] = (uint16_t)(blk[0] | (blk[1] << 8));
      for (int i = 0; i < 32; ++i) {
        const int v = blk[2 + i];
        q[n * K + b * 32 + i] = (int8_t)(v < 128 ? v : v - 256);
      }
    }
}

void oracle_repack_q4_0(const uint8_t* blocks, int64_t N, int64_t K, uint8_t* q4, uint16_t* d) {
  const int64_t nb = K / 32;
  for (int64_t n = 0; n < N; ++n)
    for (int64_t b = 0; b < nb; ++b) {
      const uint8_t* blk = blocks + (n * nb + b) * 18;
      d[n * nb + b] = (uint16_t)(blk[0] | (blk[1] << 8));
      for (int j = 0; j < 16; ++j) q4[n * (K / 2) + b * 16 + j] = blk[2 + j];
    }
}

// ---------------------------------------------------------------------------
// NVFP4 weights (the pages' third decode format: memra wiki, feature list; their
// safetensors loader reads NVIDIA ModelOpt NVFP4 checkpoints byte for byte).  The
// pages print none of it; the reading is ModelOpt's NVFP4, restated:
//   a block is 16 consecutive weights of a row; each weight is an FP4 E2M1 code
//   (sign, 2 exponent bits, 1 mantissa bit: magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6),
//   each block has an FP8 E4M3 scale s, and the tensor one fp32 scale g, so that
//   w ~= g * s * e2m1(code).  Byte j of a row's code plane holds element 2j in its
//   low nibble and element 2j+1 in its high nibble.
// Quantisation: g = amax|W| / (6 * 448); per block s = e4m3(amax_block / (6 g));
// code = e2m1(w / (float(s) * g)), a block whose scale is 0 gets code 0.  Every
// conversion rounds to nearest, ties to even, and saturates (448, 6).  Each fp32
// operation is one IEEE operation in the order written.
// ---------------------------------------------------------------------------

// FP8 E4M3 ("fn": bias 7, no infinities, largest finite 448) from fp32, written
// from the definition: the quantum of |f|'s binade (2^(e-3) for normals, 2^-9 for
// subnormals), the nearest multiple of it (ties to even via nearbyint), saturation
// at 448, then the encoding.
uint8_t f32_to_e4m3(float f) {
  const uint8_t sign = std::signbit(f) ? 0x80 : 0x00;
  const double a = std::fabs((double)f);
  if (a == 0.0) return sign;
  int e2 = 0;
  std::frexp(a, &e2);  // a = m * 2^e2 with m in [0.5, 1): binade exponent e2 - 1
  const int be = std::max(e2 - 1, -6);
  const double q = std::ldexp(1.0, be - 3);
  double r = std::nearbyint(a / q) * q;
  if (r > 448.0) r = 448.0;
  if (r == 0.0) return sign;
  int re = 0;
  std::frexp(r, &re);
  const int rbe = re - 1;
  if (rbe < -6) return (uint8_t)(sign | (int)std::ldexp(r, 9));  // subnormal: r = m * 2^-9
  const int m = (int)(std::ldexp(r, -rbe) * 8.0) - 8;             // r = 2^rbe * (1 + m/8)
  return (uint8_t)(sign | ((rbe + 7) << 3) | m);
}

// FP8 E4M3 -> fp32, exact (0x7f / 0xff, the NaN codes, never occur here).
float e4m3_to_f32(uint8_t b) {
  const int e = (b >> 3) & 15;
  const int m = b & 7;
  const double mag = e == 0 ? std::ldexp((double)m, -9) : std::ldexp(1.0 + m / 8.0, e - 7);
  return (float)((b & 0x80) ? -mag : mag);
}

// FP4 E2M1 from fp32: the quantum of |f|'s binade (0.5 below 2, 1 below 4, else 2),
// the nearest multiple (ties to even), saturation at 6, then the code of that value.
uint8_t f32_to_e2m1(float f) {
  static const double kVal[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
  const uint8_t sign = std::signbit(f) ? 8 : 0;
  const double a = std::fabs((double)f);
  const double q = a < 2.0 ? 0.5 : (a < 4.0 ? 1.0 : 2.0);
  double r = std::nearbyint(a / q) * q;
  if (r > 6.0) r = 6.0;
  for (int i = 0; i < 8; ++i)
    if (kVal[i] == r) return (uint8_t)(sign | i);
  return sign;  // not reached for finite input
}

// Twice the E2M1 value of a code, an integer in [-12, 12].
int e2m1_twice(uint8_t code) {
  static const int kTwice[8] = {0, 1, 2, 3, 4, 6, 8, 12};
  return (code & 8) ? -kTwice[code & 7] : kTwice[code & 7];
}

uint8_t oracle_f32_to_e4m3(float f) { return f32_to_e4m3(f); }
float oracle_e4m3_to_f32(uint8_t b) { return e4m3_to_f32(b); }
uint8_t oracle_f32_to_e2m1(float f) { return f32_to_e2m1(f); }

// w: fp32 [N][K], K % 32 == 0.  codes: uint8 [N][K/2]; scales: E4M3 bits [N][K/16];
// *g: the tensor scale.
void oracle_quantize_nvfp4(const float* w, int64_t N, int64_t K, uint8_t* codes,
                           uint8_t* scales, float* g_out) {
  float amax = 0.0f;
  for (int64_t i = 0; i < N * K; ++i) amax = std::max(amax, std::fabs(w[i]));
  const float g = amax / 2688.0f;  // 6 * 448
  *g_out = g;
  for (int64_t n = 0; n < N; ++n)
    for (int64_t blk = 0; blk < K / 16; ++blk) {
      const float* v = w + n * K + blk * 16;
      float bmax = 0.0f;
      for (int i = 0; i < 16; ++i) bmax = std::max(bmax, std::fabs(v[i]));
      const uint8_t sc = g == 0.0f ? 0 : f32_to_e4m3(bmax / (6.0f * g));
      scales[n * (K / 16) + blk] = sc;
      const float denom = e4m3_to_f32(sc) * g;
      for (int i = 0; i < 16; ++i) {
        const uint8_t c = denom == 0.0f ? 0 : f32_to_e2m1(v[i] / denom);
        const int64_t e = blk * 16 + i;  // element index within the row
        uint8_t& byte = codes[n * (K / 2) + e / 2];
        if (e % 2 == 0)
          byte = c;
        else
          byte = (uint8_t)(byte | (c << 4));
      }
    }
}

// Codes -> twice their E2M1 values, int8 [N][K].
void oracle_unpack_nvfp4(const uint8_t* codes, int64_t N, int64_t K, int8_t* twice) {
  for (int64_t n = 0; n < N; ++n)
    for (int64_t e = 0; e < K; ++e) {
      const uint8_t byte = codes[n * (K / 2) + e / 2];
      twice[n * K + e] = (int8_t)e2m1_twice(e % 2 == 0 ? (byte & 0x0F) : (byte >> 4));
    }
}

// NVFP4 x q8_1: y[m][n] = (g / 2) * sum_b t_b, summed sequentially in b, with
//   t_b = (s_lo * d_x) * S_lo + (s_hi * d_x) * S_hi,
// S_lo, S_hi the exact int32 sums of (twice the E2M1 value) * xq over the first and
// second 16 elements of activation block b, s_lo, s_hi their blocks' E4M3 scales.
void oracle_nvfp4_gemm(const uint8_t* codes, const uint8_t* scales, float g, int64_t N,
                       int64_t K, int64_t M, const int8_t* xq, const float* xd, float* y,
                       int threads) {
  const int64_t nb = K / 32;
  (void)threads;
#ifdef _OPENMP
#pragma omp parallel for num_threads(threads_or_one(threads)) schedule(static)
#endif
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t m = 0; m < M; ++m) {
      float acc = 0.0f;
      for (int64_t b = 0; b < nb; ++b) {
        int32_t S[2] = {0, 0};
        for (int i = 0; i < 32; ++i) {
          const int64_t e = b * 32 + i;
          const uint8_t byte = codes[n * (K / 2) + e / 2];
          const int c2 = e2m1_twice(e % 2 == 0 ? (byte & 0x0F) : (byte >> 4));
          S[i / 16] += c2 * (int32_t)xq[m * K + e];
        }
        const float dx = xd[m * nb + b];
        const float lo = (e4m3_to_f32(scales[n * (K / 16) + 2 * b]) * dx) * (float)S[0];
        const float hi = (e4m3_to_f32(scales[n * (K / 16) + 2 * b + 1]) * dx) * (float)S[1];
        const float term = lo + hi;
        acc = acc + term;
      }
      y[m * N + n] = (g * 0.5f) * acc;
    }
  }
}

// fp64 brute force of the same product: sum_k (g s e2m1) * (d_x q_x).
void oracle_nvfp4_dequant_gemm_f64(const uint8_t* codes, const uint8_t* scales, float g,
                                   int64_t N, int64_t K, int64_t M, const int8_t* xq,
                                   const float* xd, double* y) {
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n) {
      double acc = 0.0;
      for (int64_t e = 0; e < K; ++e) {
        const uint8_t byte = codes[n * (K / 2) + e / 2];
        const double v = 0.5 * e2m1_twice(e % 2 == 0 ? (byte & 0x0F) : (byte >> 4));
        const double w = (double)g * (double)e4m3_to_f32(scales[n * (K / 16) + e / 16]) * v;
        acc += w * ((double)xd[m * (K / 32) + e / 32] * (double)xq[m * K + e]);
      }
      y[m * N + n] = acc;
    }
}

// ---------------------------------------------------------------------------
// Activation quantisation ("q8_1" blocks with an fp32 scale).
// x: [M][K] fp32 or bf16 bits.  q: int8 [M][K].  d: fp32 [M][K/32].
// Per block: amax = max|x|; d = amax / 127 in fp32; q = clamp(round-half-away(
// x / d), +-127); amax == 0 gives d = 0 and q = 0.
// ---------------------------------------------------------------------------
void oracle_quantize_q8_1_f32(const float* x, int64_t M, int64_t K, int8_t* q, float* d) {
  const int64_t nb = K / 32;
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t b = 0; b < nb; ++b) {
      const float* blk = x + m * K + b * 32;
      const float amax = block_amax(blk);
      const float dv = amax / 127.0f;
      d[m * nb + b] = dv;
      for (int i = 0; i < 32; ++i) q[m * K + b * 32 + i] = quant_one(blk[i], dv);
    }
  }
}

void oracle_quantize_q8_1_bf16(const uint16_t* x, int64_t M, int64_t K, int8_t* q, float* d) {
  std::vector<float> row((size_t)K);
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t k = 0; k < K; ++k) row[(size_t)k] = bf16_to_f32(x[m * K + k]);
    oracle_quantize_q8_1_f32(row.data(), 1, K, q + m * K, d + m * (K / 32));
  }
}

// ---------------------------------------------------------------------------
// Exact int32 block dot products s[m][n][b] = sum_{i<32} wq[n][32b+i]*xq[m][32b+i].
// |s| <= 32 * 127 * 127 = 516128, so int32 (and fp32) hold it exactly.
// ---------------------------------------------------------------------------
void oracle_block_dots(const int8_t* wq, int64_t N, int64_t K, const int8_t* xq, int64_t M,
                       int32_t* s) {
  const int64_t nb = K / 32;
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n)
      for (int64_t b = 0; b < nb; ++b) {
        int32_t acc = 0;
        for (int i = 0; i < 32; ++i)
          acc += (int32_t)wq[n * K + b * 32 + i] * (int32_t)xq[m * K + b * 32 + i];
        s[(m * N + n) * nb + b] = acc;
      }
}

// ---------------------------------------------------------------------------
// Q8_0 x q8_1 product for M activation rows (M = 1 is the plain decode GEMV; M > 1
// is the speculative-verify skinny GEMM, which is the same computation per row).
// y[m][n] = sum_b (d_w[n][b] * d_x[m][b]) * float(s_b), the scale product rounded
// to fp32 first, then the fp32 product, then the fp32 sum, sequentially in b.
// Rows are independent, so `threads` > 1 only splits rows across OpenMP threads;
// every row's arithmetic is identical for any thread count.
// ---------------------------------------------------------------------------
void oracle_q8_0_gemm(const int8_t* wq, const uint16_t* wd, int64_t N, int64_t K, int64_t M,
                      const int8_t* xq, const float* xd, float* y, int threads) {
  const int64_t nb = K / 32;
  (void)threads;
#ifdef _OPENMP
#pragma omp parallel for num_threads(threads_or_one(threads)) schedule(static)
#endif
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t m = 0; m < M; ++m) {
      float acc = 0.0f;
      for (int64_t b = 0; b < nb; ++b) {
        int32_t s = 0;
        for (int i = 0; i < 32; ++i)
          s += (int32_t)wq[n * K + b * 32 + i] * (int32_t)xq[m * K + b * 32 + i];
        const float scale = f16_to_f32(wd[n * nb + b]) * xd[m * nb + b];
        const float term = scale * (float)s;
        acc = acc + term;
      }
      y[m * N + n] = acc;
    }
  }
}

void oracle_q8_0_gemv(const int8_t* wq, const uint16_t* wd, int64_t N, int64_t K,
                      const int8_t* xq, const float* xd, float* y, int threads) {
  oracle_q8_0_gemm(wq, wd, N, K, 1, xq, xd, y, threads);
}

// ---------------------------------------------------------------------------
// fp64 brute force: dequantise both operands and take the plain dot product.
// y[m][n] = sum_k (d_w * q_w) * (d_x * q_x) in fp64.  Used only to pin the fp32
// oracle within its rounding bound.
// ---------------------------------------------------------------------------
void oracle_dequant_gemm_f64(const int8_t* wq, const uint16_t* wd, int64_t N, int64_t K,
                             int64_t M, const int8_t* xq, const float* xd, double* y) {
  const int64_t nb = K / 32;
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n) {
      double acc = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        const double w = (double)f16_to_f32(wd[n * nb + k / 32]) * (double)wq[n * K + k];
        const double x = (double)xd[m * nb + k / 32] * (double)xq[m * K + k];
        acc += w * x;
      }
      y[m * N + n] = acc;
    }
}

// ---------------------------------------------------------------------------
// exp in fp32 by a named published method (Cody & Waite range reduction, "Software
// Manual for the Elementary Functions", 1980, with a truncated Taylor series):
//   k = rint(x * log2(e));  r = (x - k*C1) - k*C2 with C1 + C2 = ln 2, C1 having
//   few significant bits so k*C1 is exact;  p = 1 + r + r^2/2! + ... + r^7/7!
//   evaluated in Horner form;  exp(x) = p * 2^k.
// Each step is one rounded fp32 operation in the order written.  The argument is
// clamped to [-87, 88] so that 2^k stays a normal fp32 number.  This is the exp
// used by the SwiGLU reading below; it is pinned against libm in the tests.
// ---------------------------------------------------------------------------
float oracle_exp_cw(float x) {
  if (x > 88.0f) x = 88.0f;
  if (x < -87.0f) x = -87.0f;
  const float log2e = 1.44269504088896341f;
  const float c1 = 0.693359375f;          // 355/512: 9 significant bits
  const float c2 = -2.12194440e-4f;       // ln 2 - c1, rounded to fp32
  const float kf = rintf(x * log2e);
  float r = x - kf * c1;
  r = r - kf * c2;
  float p = 1.0f / 5040.0f;               // 1/7!
  p = p * r + 1.0f / 720.0f;
  p = p * r + 1.0f / 120.0f;
  p = p * r + 1.0f / 24.0f;
  p = p * r + 1.0f / 6.0f;
  p = p * r + 0.5f;
  p = p * r + 1.0f;
  p = p * r + 1.0f;
  const int k = (int)kf;
  return p * float_of((uint32_t)(k + 127) << 23);
}

// SwiGLU between the MoE gate/up and down projections.  gu: fp32 [R][2F], gate in
// columns [0, F), up in [F, 2F).  h[r][f] = (g / (1 + exp(-g))) * u, each operation
// one fp32 rounding in that order, exp as oracle_exp_cw.
void oracle_swiglu_f32(const float* gu, int64_t R, int64_t F, float* h) {
  for (int64_t r = 0; r < R; ++r)
    for (int64_t f = 0; f < F; ++f) {
      const float g = gu[r * 2 * F + f];
      const float u = gu[r * 2 * F + F + f];
      const float den = 1.0f + oracle_exp_cw(-g);
      const float sg = g / den;
      h[r * F + f] = sg * u;
    }
}

// SwiGLU followed by activation quantisation of each of the R rows.
void oracle_swiglu_quantize_q8_1(const float* gu, int64_t R, int64_t F, int8_t* hq, float* hd) {
  std::vector<float> h((size_t)(R * F));
  oracle_swiglu_f32(gu, R, F, h.data());
  oracle_quantize_q8_1_f32(h.data(), R, F, hq, hd);
}

// ---------------------------------------------------------------------------
// Routed-expert GEMV (top-k MoE).  Bank: wq [E][N][K], wd [E][N][K/32].
// For k < top_k with e = ids[k] in [0, E): y_k = W_e x_k, where x_k is the shared
// activation (x_per_expert == 0) or row k of a [top_k][K] activation.
//   gate_w == NULL: y is [top_k][N], row k = y_k (zero if e is out of range).
//   gate_w != NULL: y is [N] = sum_k gate_w[k] * y_k[n], k ascending, in fp32;
//                   an out-of-range e contributes nothing.
// Returns the number of out-of-range ids (the kernel's status word is 1 if > 0).
// ---------------------------------------------------------------------------
int oracle_q8_0_moe_gemv(const int8_t* wq_bank, const uint16_t* wd_bank, int64_t E, int64_t N,
                         int64_t K, const int32_t* ids, const float* gate_w, int64_t top_k,
                         const int8_t* xq, const float* xd, int x_per_expert, float* y) {
  const int64_t nb = K / 32;
  int bad = 0;
  std::vector<float> yk((size_t)N);
  if (gate_w)
    for (int64_t n = 0; n < N; ++n) y[n] = 0.0f;
  for (int64_t k = 0; k < top_k; ++k) {
    const int32_t e = ids[k];
    const bool ok = e >= 0 && e < E;
    if (!ok) ++bad;
    if (ok) {
      const int8_t* xqk = x_per_expert ? xq + k * K : xq;
      const float* xdk = x_per_expert ? xd + k * nb : xd;
      oracle_q8_0_gemm(wq_bank + (int64_t)e * N * K, wd_bank + (int64_t)e * N * nb, N, K, 1, xqk,
                       xdk, yk.data(), 1);
    } else {
      for (int64_t n = 0; n < N; ++n) yk[(size_t)n] = 0.0f;
    }
    if (gate_w) {
      if (ok)
        for (int64_t n = 0; n < N; ++n) y[n] = y[n] + gate_w[k] * yk[(size_t)n];
    } else {
      for (int64_t n = 0; n < N; ++n) y[k * N + n] = yk[(size_t)n];
    }
  }
  return bad;
}

// One routed MoE FFN layer for a single token:
//   x (fp32 [K]) -> quantise -> gate/up rows y_gu[k] = W_gu[ids[k]] x  ([top_k][2F])
//   -> SwiGLU + quantise per k -> y = sum_k gate_w[k] * W_dn[ids[k]] h_k   ([N_out])
// with K = hidden size, W_gu [E][2F][K], W_dn [E][K_out=N_out][F].
int oracle_moe_ffn(const float* x, int64_t K, const int8_t* gu_q, const uint16_t* gu_d,
                   const int8_t* dn_q, const uint16_t* dn_d, int64_t E, int64_t F, int64_t N_out,
                   const int32_t* ids, const float* gate_w, int64_t top_k, float* y) {
  std::vector<int8_t> xq((size_t)K);
  std::vector<float> xd((size_t)(K / 32));
  oracle_quantize_q8_1_f32(x, 1, K, xq.data(), xd.data());
  std::vector<float> ygu((size_t)(top_k * 2 * F));
  int bad = oracle_q8_0_moe_gemv(gu_q, gu_d, E, 2 * F, K, ids, nullptr, top_k, xq.data(),
                                 xd.data(), 0, ygu.data());
  std::vector<int8_t> hq((size_t)(top_k * F));
  std::vector<float> hd((size_t)(top_k * F / 32));
  oracle_swiglu_quantize_q8_1(ygu.data(), top_k, F, hq.data(), hd.data());
  bad += oracle_q8_0_moe_gemv(dn_q, dn_d, E, N_out, F, ids, gate_w, top_k, hq.data(), hd.data(),
                              1, y);
  return bad;
}

int oracle_openmp_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

}  // extern "C"
