// wq_oracle.cpp -- plain, slow, obviously-correct CPU oracle for the weight-only
// quantized linear layer.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and
// the benchmark's CPU-baseline leg call it; the CUDA library never does, and the two
// share no code, header, table or helper.
//
// Sources (web pages; cited by title and section):
//   [Linnet]   "Quantization" (Linnet language docs, std.quant) -- format table,
//              "Group-wise 4-bit weights", "MXFP4 experts".
//   [L8.5]     "Quantization: int8, int4 group (packed), fp8, KV quant" (OpenLearn
//              TinyLLM module L8.5) -- "2. Principles", "3. Worked example by hand".
//   [Ch20]     "20. Quantization" (Inference Engineering book) -- "Symmetric
//              quantization, from scratch", "Granularity: who shares a scale",
//              "Packing", "A quantized linear layer".
//   [LLM4.8]   "4.8 Quantization II: INT4/INT8/FP8, GGUF, bitsandbytes & QAT" --
//              "Per-Group INT4", "FP8 Inference" (E2M1 element format).
//
// Precision: the quantizers work in f32 because the pages fix that ([L8.5] 2.
// Principles: "every quotient W / s is formed in float32 before rounding").  The
// dequantizers compute (code - zero) * scale in f32 and cast to bf16 ([Linnet] format
// table: "q * scale in f32, cast to T").  The linear layers accumulate in f64; every
// product of two bf16 values is exact in f64.
//
// Readings where the pages are silent or disagree (each is listed in the design notes):
//   R1 code = rint(fl32(w * fl32(Q / a))): reproduces every printed example, which a
//      literal fl32(w / fl32(a / Q)) does not ([Ch20] worked example gives -4 / 4 for
//      -1 / 1; the literal f32 quotient is -3.4999998).  If Q / a overflows f32 (a
//      below ~1e-38) the literal quotient w / s is used instead.
//   R2 rint = round to nearest, ties to even ([L8.5] 2. Principles, 3. Worked example).
//   R3 an all-zero group gets scale 1 and codes 0 ([Ch20] Granularity).
//   R4 symmetric codes are clamped to [-Q, Q]; unpacking accepts nibble 8 = -8.
//   R5 scales are f32, zeros u8.
//   R6 dequant: the integer (q - zero) is formed exactly, converted to f32, multiplied
//      once by the f32 scale, and the product rounded to bf16 (nearest even).
//   R7 asymmetric quantizer (formula lost on the pages): lo = min(0, min w),
//      hi = max(0, max w), s = fl32((hi - lo) / L), r = fl32(L / (hi - lo)),
//      zero = clamp(rint(fl32(-lo * r)), 0, L), code = clamp(rint(fl32(w * r)) + zero,
//      0, L) with L = 2^bits - 1; hi == lo gives s = 1, zero = 2^(bits-1), codes = zero.
//      Parity of this function is pinned by invariants only (range, 0 -> 0 exactly,
//      the half-step bound), not by a printed example.
//   R8 MXFP4 follows the OCP MX v1.0 conventions the pages cite: E8M0 bias 127, scale
//      byte 255 = NaN, E2M1 bit 3 = sign, low 3 bits index {0,.5,1,1.5,2,3,4,6}.
//   R9 bias (bf16) is added to the f64 sum; the layer output type is bf16.
//   R10 a group holding a non-finite weight, or whose range overflows f32, is refused:
//      the function reports it, and writes scale 1 and the code of 0 for that group.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <algorithm>
#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

uint32_t f32_bits(float f) { uint32_t u; std::memcpy(&u, &f, 4); return u; }
float bits_f32(uint32_t u) { float f; std::memcpy(&f, &u, 4); return f; }

// bf16 = the top 16 bits of an IEEE binary32.  Round to nearest, ties to even, on the
// 16 bits dropped; NaN stays NaN (quiet bit set).
uint16_t bf16_from_f32(float f) {
  uint32_t u = f32_bits(f);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0)
    return (uint16_t)((u >> 16) | 0x0040u);
  uint32_t lower = u & 0xFFFFu;
  uint32_t upper = u >> 16;
  if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1;  // carry may
  return (uint16_t)upper;                 // ripple into the exponent: that is correct
}
double bf16_to_f64(uint16_t b) { return (double)bits_f32((uint32_t)b << 16); }

float round_even(float v) { return std::nearbyint(v); }  // default mode: ties to even

}  // namespace

extern "C" {

// Symmetric round-to-nearest quantizer, one scale per group of G consecutive inputs of
// a row ([Ch20] "Symmetric quantization, from scratch" and "Granularity"; [L8.5] 2.
// Principles).  w f32 [N, K] row-major; codes i8 [N, K]; scale f32 [N, ceil(K/G)].
// The last group of a row may be short; it is treated as if padded with zeros.
// bits in {2..8}.  Returns the number of refused groups (R10).
int64_t orc_quantize_sym(const float* w, int64_t N, int64_t K, int64_t G, int bits,
                         int8_t* codes, float* scale) {
  const int64_t groups = (K + G - 1) / G;
  const float Q = (float)((1 << (bits - 1)) - 1);
  int64_t refused = 0;
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t g = 0; g < groups; ++g) {
      const int64_t k0 = g * G, k1 = std::min(K, k0 + G);
      bool finite = true;
      float a = 0.0f;
      for (int64_t k = k0; k < k1; ++k) {
        float v = w[n * K + k];
        if (!std::isfinite(v)) finite = false;
        a = std::max(a, std::fabs(v));
      }
      float s = 1.0f;
      if (!finite) {
        ++refused;
        for (int64_t k = k0; k < k1; ++k) codes[n * K + k] = 0;
      } else if (a > 0.0f) {
        s = a / Q;                 // stored scale
        const float r = Q / a;     // R1: the f32 inverse the codes are rounded against
        for (int64_t k = k0; k < k1; ++k) {
          float v = w[n * K + k];
          float t = std::isinf(r) ? v / s : v * r;
          float q = std::min(Q, std::max(-Q, round_even(t)));
          codes[n * K + k] = (int8_t)q;
        }
      } else {
        for (int64_t k = k0; k < k1; ++k) codes[n * K + k] = 0;   // R3
      }
      scale[n * groups + g] = s;
    }
  }
  return refused;
}

// Asymmetric (zero-point) round-to-nearest quantizer, reading R7.  codes u8 [N, K] in
// [0, 2^bits - 1]; scale f32 and zero u8 [N, ceil(K/G)].  Returns refused groups.
int64_t orc_quantize_asym(const float* w, int64_t N, int64_t K, int64_t G, int bits,
                          uint8_t* codes, float* scale, uint8_t* zero) {
  const int64_t groups = (K + G - 1) / G;
  const float L = (float)((1 << bits) - 1);
  const uint8_t mid = (uint8_t)(1 << (bits - 1));
  int64_t refused = 0;
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t g = 0; g < groups; ++g) {
      const int64_t k0 = g * G, k1 = std::min(K, k0 + G);
      bool finite = true;
      float lo = 0.0f, hi = 0.0f;
      for (int64_t k = k0; k < k1; ++k) {
        float v = w[n * K + k];
        if (!std::isfinite(v)) finite = false;
        lo = std::min(lo, v);
        hi = std::max(hi, v);
      }
      float range = hi - lo;
      if (finite && std::isinf(range)) finite = false;
      float s = 1.0f;
      uint8_t z = mid;
      if (!finite) {
        ++refused;
        for (int64_t k = k0; k < k1; ++k) codes[n * K + k] = mid;
      } else if (range > 0.0f) {
        s = range / L;
        const float r = L / range;
        const bool lit = std::isinf(r);
        float zf = round_even(lit ? (-lo) / s : (-lo) * r);
        zf = std::min(L, std::max(0.0f, zf));
        z = (uint8_t)zf;
        for (int64_t k = k0; k < k1; ++k) {
          float v = w[n * K + k];
          float t = lit ? v / s : v * r;
          float q = std::min(L, std::max(0.0f, round_even(t) + zf));
          codes[n * K + k] = (uint8_t)q;
        }
      } else {
        for (int64_t k = k0; k < k1; ++k) codes[n * K + k] = mid;
      }
      scale[n * groups + g] = s;
      zero[n * groups + g] = z;
    }
  }
  return refused;
}

// Two 4-bit codes per byte, the even column in the low nibble, each as a 4-bit two's
// complement value (signed) or a plain 0..15 value (unsigned) ([Linnet] "Packed 4-bit
// formats hold two values a byte, the even element in the low nibble"; [L8.5] 2.
// Principles, Packing; [Ch20] Packing).  codes [rows, cols] -> packed [rows, cols/2].
// Returns 0, 1 for an odd width, 2 for a code out of range.
int orc_pack_int4(const int8_t* codes, int64_t rows, int64_t cols, int is_unsigned,
                  uint8_t* packed) {
  if (cols % 2 != 0) return 1;
  for (int64_t i = 0; i < rows * cols; ++i) {
    int v = is_unsigned ? (int)(uint8_t)codes[i] : (int)codes[i];
    if (is_unsigned ? (v < 0 || v > 15) : (v < -8 || v > 7)) return 2;
  }
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t j = 0; j < cols / 2; ++j) {
      int lo = codes[r * cols + 2 * j] & 0xF;
      int hi = codes[r * cols + 2 * j + 1] & 0xF;
      packed[r * (cols / 2) + j] = (uint8_t)(lo | (hi << 4));
    }
  }
  return 0;
}

// Inverse of orc_pack_int4.  Signed: a nibble v >= 8 means v - 16 ([L8.5] Packing).
int orc_unpack_int4(const uint8_t* packed, int64_t rows, int64_t cols, int is_unsigned,
                    int8_t* codes) {
  if (cols % 2 != 0) return 1;
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t k = 0; k < cols; ++k) {
      uint8_t byte = packed[r * (cols / 2) + k / 2];
      int v = (k % 2 == 0) ? (byte & 0xF) : (byte >> 4);
      if (!is_unsigned && v >= 8) v -= 16;
      codes[r * cols + k] = (int8_t)v;
    }
  }
  return 0;
}

// Group-wise asymmetric 4-bit dequantization ([Linnet] dequantize_int4_groups:
// "(q - zero) * scale per group"; "Int4GroupLinear ... weight [Out, In/Group, Group/2;
// u8], scale and zero [Out, In/Group]").  The [N, K/G, G/2] byte array is addressed as
// its row-major [N, K/2] view.  w_out bf16 bits [N, K].  Reading R6.
void orc_dequant_int4_groups(const uint8_t* packed, const float* scale,
                             const uint8_t* zero, int64_t N, int64_t K, int64_t G,
                             uint16_t* w_out) {
  const int64_t groups = K / G;
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t k = 0; k < K; ++k) {
      uint8_t byte = packed[n * (K / 2) + k / 2];
      int q = (k % 2 == 0) ? (byte & 0xF) : (byte >> 4);
      int z = zero[n * groups + k / G];
      float s = scale[n * groups + k / G];
      float v = (float)(q - z) * s;
      w_out[n * K + k] = bf16_from_f32(v);
    }
  }
}

// Symmetric per-row int8 ([Linnet] dequantize_int8: "q * scale in f32, cast to T").
void orc_dequant_int8_rows(const int8_t* q, const float* scale, int64_t N, int64_t K,
                           uint16_t* w_out) {
  for (int64_t n = 0; n < N; ++n)
    for (int64_t k = 0; k < K; ++k)
      w_out[n * K + k] = bf16_from_f32((float)q[n * K + k] * scale[n]);
}

// Symmetric per-row signed int4 ([Linnet] dequantize_int4: "unpack, then dequantize";
// Int4Linear weight [Out, In/2; i8], scale [Out; f32]).
void orc_dequant_int4_rows(const uint8_t* packed, const float* scale, int64_t N,
                           int64_t K, uint16_t* w_out) {
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t k = 0; k < K; ++k) {
      uint8_t byte = packed[n * (K / 2) + k / 2];
      int v = (k % 2 == 0) ? (byte & 0xF) : (byte >> 4);
      if (v >= 8) v -= 16;
      w_out[n * K + k] = bf16_from_f32((float)v * scale[n]);
    }
  }
}

// One E2M1 element as a float: bit 3 sign, bits 2..1 exponent, bit 0 mantissa.  The
// magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4, 6 ([L8.5] 2. Principles, MXFP4).  The value
// is computed from the fields (subnormal when the exponent field is 0) rather than
// read from a table, so the table printed on the page pins it.
float e2m1_value(int nib) {
  int sign = (nib >> 3) & 1, e = (nib >> 1) & 3, m = nib & 1;
  float mag = (e == 0) ? 0.5f * (float)m : std::ldexp(1.0f + 0.5f * (float)m, e - 1);
  return sign ? -mag : mag;
}
// E8M0 scale byte -> 2^(byte - 127); 255 is NaN (reading R8).
float e8m0_value(uint8_t b) {
  if (b == 255) return std::nanf("");
  return std::ldexp(1.0f, (int)b - 127);
}

// MXFP4 dequantization ([Linnet] dequantize_mxfp4: "E2M1 values in blocks of 32, one
// E8M0 scale byte a block"; [L8.5] MXFP4).  blocks u8 [E, N, K/32, 16] (two elements a
// byte, even element low), scales u8 [E, N, K/32] -> w_out bf16 bits [E, N, K].
void orc_dequant_mxfp4(const uint8_t* blocks, const uint8_t* scales, int64_t E,
                       int64_t N, int64_t K, uint16_t* w_out) {
  for (int64_t e = 0; e < E; ++e) {
    for (int64_t n = 0; n < N; ++n) {
      const int64_t row = e * N + n;
      for (int64_t k = 0; k < K; ++k) {
        uint8_t byte = blocks[row * (K / 2) + k / 2];
        int nib = (k % 2 == 0) ? (byte & 0xF) : (byte >> 4);
        float v = e2m1_value(nib) * e8m0_value(scales[row * (K / 32) + k / 32]);
        w_out[row * K + k] = bf16_from_f32(v);
      }
    }
  }
}

static int g_threads = 1;
void orc_set_threads(int n) { g_threads = n < 1 ? 1 : n; }
int orc_max_threads(void) {
#ifdef _OPENMP
  return omp_get_num_procs();
#else
  return 1;
#endif
}

// y = x . W^T + bias over an already dequantized bf16 weight: the layer's definition
// ([Ch20] A quantized linear layer: the forward "dequantizes the whole matrix" and runs
// F.linear; [L8.5] "QuantLinear(x) equals x @ dequantize(q)^T + b").  x bf16 [M, K],
// w bf16 [N, K], bias bf16 [N] or NULL.  y f64 [M, N] (unrounded) and
// absdot f64 [M, N] = sum_k |x_k * w_k| (the scale of the output tolerance).
void orc_linear_bf16(const uint16_t* x, int64_t M, int64_t K, const uint16_t* w,
                     const uint16_t* bias, int64_t N, double* y, double* absdot) {
#ifdef _OPENMP
#pragma omp parallel for num_threads(g_threads) schedule(static)
#endif
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t m = 0; m < M; ++m) {
      double acc = 0.0, mag = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        double p = bf16_to_f64(x[m * K + k]) * bf16_to_f64(w[n * K + k]);
        acc += p;
        mag += std::fabs(p);
      }
      if (bias) acc += bf16_to_f64(bias[n]);
      y[m * N + n] = acc;
      if (absdot) absdot[m * N + n] = mag;
    }
  }
}

// linear_int4_groups(x, packed, scale, zero, bias) ([Linnet] format table): dequantize,
// then linear ([Linnet] Group-wise 4-bit weights: "everywhere else: dequantize, then
// linear").  The weight is dequantized one row at a time to bound memory.
void orc_linear_int4_groups(const uint16_t* x, int64_t M, int64_t K,
                            const uint8_t* packed, const float* scale,
                            const uint8_t* zero, const uint16_t* bias, int64_t N,
                            int64_t G, double* y, double* absdot) {
  const int64_t groups = K / G;
#ifdef _OPENMP
#pragma omp parallel for num_threads(g_threads) schedule(static)
#endif
  for (int64_t n = 0; n < N; ++n) {
    uint16_t* row = new uint16_t[K];
    orc_dequant_int4_groups(packed + n * (K / 2), scale + n * groups, zero + n * groups,
                            1, K, G, row);
    for (int64_t m = 0; m < M; ++m) {
      double acc = 0.0, mag = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        double p = bf16_to_f64(x[m * K + k]) * bf16_to_f64(row[k]);
        acc += p;
        mag += std::fabs(p);
      }
      if (bias) acc += bf16_to_f64(bias[n]);
      y[m * N + n] = acc;
      if (absdot) absdot[m * N + n] = mag;
    }
    delete[] row;
  }
}

// Int8Linear forward: dequantize_int8, then linear ([Linnet] format table).
void orc_linear_int8_rows(const uint16_t* x, int64_t M, int64_t K, const int8_t* q,
                          const float* scale, const uint16_t* bias, int64_t N,
                          double* y, double* absdot) {
#ifdef _OPENMP
#pragma omp parallel for num_threads(g_threads) schedule(static)
#endif
  for (int64_t n = 0; n < N; ++n) {
    uint16_t* row = new uint16_t[K];
    orc_dequant_int8_rows(q + n * K, scale + n, 1, K, row);
    for (int64_t m = 0; m < M; ++m) {
      double acc = 0.0, mag = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        double p = bf16_to_f64(x[m * K + k]) * bf16_to_f64(row[k]);
        acc += p;
        mag += std::fabs(p);
      }
      if (bias) acc += bf16_to_f64(bias[n]);
      y[m * N + n] = acc;
      if (absdot) absdot[m * N + n] = mag;
    }
    delete[] row;
  }
}

// Int4Linear forward: dequantize_int4 (signed nibbles, per-row scale), then linear.
void orc_linear_int4_rows(const uint16_t* x, int64_t M, int64_t K,
                          const uint8_t* packed, const float* scale,
                          const uint16_t* bias, int64_t N, double* y, double* absdot) {
#ifdef _OPENMP
#pragma omp parallel for num_threads(g_threads) schedule(static)
#endif
  for (int64_t n = 0; n < N; ++n) {
    uint16_t* row = new uint16_t[K];
    orc_dequant_int4_rows(packed + n * (K / 2), scale + n, 1, K, row);
    for (int64_t m = 0; m < M; ++m) {
      double acc = 0.0, mag = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        double p = bf16_to_f64(x[m * K + k]) * bf16_to_f64(row[k]);
        acc += p;
        mag += std::fabs(p);
      }
      if (bias) acc += bf16_to_f64(bias[n]);
      y[m * N + n] = acc;
      if (absdot) absdot[m * N + n] = mag;
    }
    delete[] row;
  }
}

// mxfp4_experts_shared(x, blocks, scales, experts) ([Linnet] format table: "a
// mixture's chosen experts multiplied from MXFP4 ... each row's slots sharing one
// input (x: [R, 1, In])").  x bf16 [R, K]; experts i32 [R, S]; blocks/scales as in
// orc_dequant_mxfp4; y f64 [R, S, N].  A slot whose expert index is outside [0, E)
// gets zeros and is counted in the return value.  n0/n1 restrict the output columns
// computed to [n0, n1) (the rest of y is left untouched) so callers can sample.
int64_t orc_mxfp4_experts_shared(const uint16_t* x, int64_t R, int64_t K,
                                 const uint8_t* blocks, const uint8_t* scales,
                                 int64_t E, int64_t N, const int32_t* experts,
                                 int64_t S, int64_t n0, int64_t n1, double* y,
                                 double* absdot) {
  int64_t bad = 0;
  for (int64_t r = 0; r < R; ++r) {
    for (int64_t s = 0; s < S; ++s) {
      int32_t e = experts[r * S + s];
      double* yrs = y + (r * S + s) * N;
      double* ars = absdot ? absdot + (r * S + s) * N : nullptr;
      if (e < 0 || e >= E) {
        ++bad;
        for (int64_t n = n0; n < n1; ++n) { yrs[n] = 0.0; if (ars) ars[n] = 0.0; }
        continue;
      }
#ifdef _OPENMP
#pragma omp parallel for num_threads(g_threads) schedule(static)
#endif
      for (int64_t n = n0; n < n1; ++n) {
        uint16_t* row = new uint16_t[K];
        const int64_t erow = (int64_t)e * N + n;
        orc_dequant_mxfp4(blocks + erow * (K / 2), scales + erow * (K / 32), 1, 1, K,
                          row);
        double acc = 0.0, mag = 0.0;
        for (int64_t k = 0; k < K; ++k) {
          double p = bf16_to_f64(x[r * K + k]) * bf16_to_f64(row[k]);
          acc += p;
          mag += std::fabs(p);
        }
        yrs[n] = acc;
        if (ars) ars[n] = mag;
        delete[] row;
      }
    }
  }
  return bad;
}

// Element conversions exposed for pinning against library routines.
uint16_t orc_bf16_from_f32(float f) { return bf16_from_f32(f); }
float orc_e2m1_value(int nib) { return e2m1_value(nib); }

}  // extern "C"
