// quant.cu -- load-time quantize / pack / unpack and the dequantize exports.
//
// Bit-exact by construction: every floating-point step uses an explicitly rounded IEEE
// f32 operation (__fdiv_rn, __fmul_rn, __fsub_rn, rintf with ties to even), so no FMA
// contraction or approximate division can change a code.
//   Quantizer: "20. Quantization" (Inference Engineering book), "Symmetric quantization,
//   from scratch" and "Granularity: who shares a scale"; "Quantization: int8, int4 group
//   (packed), fp8, KV quant" (OpenLearn L8.5), "2. Principles" (rint ties to even,
//   quotients in float32); "Quantization" (Linnet docs), "Quantizing a checkpoint".
//   Packing: "Packed 4-bit formats hold two values a byte, the even element in the low
//   nibble" (Linnet docs); two's complement nibbles (OpenLearn L8.5, Packing).
//   Dequantizers: the Linnet docs' format table ("q * scale in f32, cast to T").
#include <algorithm>

#include "common.cuh"
#include "launch.h"

namespace wq {

namespace {

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_min(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// One warp per (row, group).  Codes are one byte each: i8 (WQ_SYM) or u8.
__global__ void k_quantize(const float* __restrict__ w, int64_t N, int64_t K, int32_t G,
                           int32_t bits, int32_t mode, uint8_t* __restrict__ codes,
                           float* __restrict__ scale, uint8_t* __restrict__ zero,
                           int32_t* dev_status) {
  const int64_t groups = (K + G - 1) / G;
  const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= N * groups) return;
  const int64_t n = gw / groups, g = gw % groups;
  const int64_t k0 = g * G;
  const int64_t k1 = imin64(K, k0 + G);
  const float* row = w + n * K;

  bool finite = true;
  float amax = 0.0f, lo = 0.0f, hi = 0.0f;
  for (int64_t k = k0 + lane; k < k1; k += 32) {
    const float v = row[k];
    if (!isfinite(v)) finite = false;
    amax = fmaxf(amax, fabsf(v));
    lo = fminf(lo, v);
    hi = fmaxf(hi, v);
  }
  finite = __all_sync(0xffffffffu, finite);
  amax = warp_max(amax);
  lo = warp_min(lo);
  hi = warp_max(hi);

  uint8_t* crow = codes + n * K;
  if (mode == WQ_ASYM) {
    const float L = (float)((1 << bits) - 1);
    const uint8_t mid = (uint8_t)(1 << (bits - 1));
    const float range = __fsub_rn(hi, lo);
    if (finite && isinf(range)) finite = false;
    float s = 1.0f;
    uint8_t z = mid;
    if (!finite) {
      if (lane == 0) set_dev_status(dev_status, WQ_DEV_NONFINITE);
      for (int64_t k = k0 + lane; k < k1; k += 32) crow[k] = mid;
    } else if (range > 0.0f) {
      s = __fdiv_rn(range, L);
      const float r = __fdiv_rn(L, range);
      const bool lit = isinf(r);
      float zf = rintf(lit ? __fdiv_rn(-lo, s) : __fmul_rn(-lo, r));
      zf = fminf(L, fmaxf(0.0f, zf));
      z = (uint8_t)zf;
      for (int64_t k = k0 + lane; k < k1; k += 32) {
        const float t = lit ? __fdiv_rn(row[k], s) : __fmul_rn(row[k], r);
        const float q = fminf(L, fmaxf(0.0f, __fadd_rn(rintf(t), zf)));
        crow[k] = (uint8_t)q;
      }
    } else {
      for (int64_t k = k0 + lane; k < k1; k += 32) crow[k] = mid;
    }
    if (lane == 0) {
      scale[n * groups + g] = s;
      zero[n * groups + g] = z;
    }
    return;
  }

  // symmetric (WQ_SYM, WQ_SYM_U4)
  const float Q = (float)((1 << (bits - 1)) - 1);
  const bool u4 = (mode == WQ_SYM_U4);
  const int off = u4 ? 8 : 0;
  float s = 1.0f;
  if (!finite) {
    if (lane == 0) set_dev_status(dev_status, WQ_DEV_NONFINITE);
    for (int64_t k = k0 + lane; k < k1; k += 32) crow[k] = (uint8_t)off;
  } else if (amax > 0.0f) {
    s = __fdiv_rn(amax, Q);
    const float r = __fdiv_rn(Q, amax);
    const bool lit = isinf(r);
    for (int64_t k = k0 + lane; k < k1; k += 32) {
      const float t = lit ? __fdiv_rn(row[k], s) : __fmul_rn(row[k], r);
      const float q = fminf(Q, fmaxf(-Q, rintf(t)));
      crow[k] = (uint8_t)((int)q + off);
    }
  } else {
    for (int64_t k = k0 + lane; k < k1; k += 32) crow[k] = (uint8_t)off;
  }
  if (lane == 0) {
    scale[n * groups + g] = s;
    if (u4) zero[n * groups + g] = 8;
  }
}

__global__ void k_pack(const uint8_t* __restrict__ codes, int64_t total_bytes,
                       int32_t is_unsigned, uint8_t* __restrict__ packed, int32_t* dev_status) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= total_bytes) return;
  const uint8_t a = codes[2 * i], b = codes[2 * i + 1];
  bool bad;
  if (is_unsigned) {
    bad = a > 15 || b > 15;
  } else {
    const int sa = (int8_t)a, sb = (int8_t)b;
    bad = sa < -8 || sa > 7 || sb < -8 || sb > 7;
  }
  if (bad) set_dev_status(dev_status, WQ_DEV_BAD_CODE);
  packed[i] = (uint8_t)((a & 0xF) | ((b & 0xF) << 4));
}

__global__ void k_unpack(const uint8_t* __restrict__ packed, int64_t total_bytes,
                         int32_t is_unsigned, uint8_t* __restrict__ codes) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= total_bytes) return;
  const uint8_t v = packed[i];
  int lo = v & 0xF, hi = v >> 4;
  if (!is_unsigned) {
    if (lo >= 8) lo -= 16;
    if (hi >= 8) hi -= 16;
  }
  codes[2 * i] = (uint8_t)lo;
  codes[2 * i + 1] = (uint8_t)hi;
}

// One thread per byte of codes (two outputs).
__global__ void k_dequant_i4g(const uint8_t* __restrict__ packed, const float* __restrict__ scale,
                              const uint8_t* __restrict__ zero, int64_t N, int64_t K, int32_t G,
                              __nv_bfloat16* __restrict__ w) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t half = K / 2;
  if (i >= N * half) return;
  const int64_t n = i / half, k = (i % half) * 2;
  const int64_t gi = n * (K / G) + k / G;  // G even: both codes share the group
  const uint8_t v = packed[i];
  const int z = zero[gi];
  const float s = scale[gi];
  const float a = __fmul_rn((float)((int)(v & 0xF) - z), s);
  const float b = __fmul_rn((float)((int)(v >> 4) - z), s);
  w[n * K + k] = __float2bfloat16_rn(a);
  w[n * K + k + 1] = __float2bfloat16_rn(b);
}

__global__ void k_dequant_i8r(const int8_t* __restrict__ q, const float* __restrict__ scale,
                              int64_t N, int64_t K, __nv_bfloat16* __restrict__ w) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= N * K) return;
  w[i] = __float2bfloat16_rn(__fmul_rn((float)q[i], scale[i / K]));
}

__global__ void k_dequant_i4r(const uint8_t* __restrict__ packed, const float* __restrict__ scale,
                              int64_t N, int64_t K, __nv_bfloat16* __restrict__ w) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t half = K / 2;
  if (i >= N * half) return;
  const int64_t n = i / half, k = (i % half) * 2;
  const uint8_t v = packed[i];
  int lo = v & 0xF, hi = v >> 4;
  if (lo >= 8) lo -= 16;
  if (hi >= 8) hi -= 16;
  const float s = scale[n];
  w[n * K + k] = __float2bfloat16_rn(__fmul_rn((float)lo, s));
  w[n * K + k + 1] = __float2bfloat16_rn(__fmul_rn((float)hi, s));
}

__global__ void k_dequant_mxfp4(const uint8_t* __restrict__ blocks,
                                const uint8_t* __restrict__ scales, int64_t rows, int64_t K,
                                __nv_bfloat16* __restrict__ w) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t half = K / 2;
  if (i >= rows * half) return;
  const int64_t r = i / half, k = (i % half) * 2;
  const float X = e8m0_to_f32(scales[r * (K / 32) + k / 32]);
  const float2 v = e2m1x2_to_f32x2(blocks[i]);
  w[r * K + k] = __float2bfloat16_rn(__fmul_rn(v.x, X));
  w[r * K + k + 1] = __float2bfloat16_rn(__fmul_rn(v.y, X));
}

// MXFP4 slots whose expert index is outside [0, E): output row zeroed, status flagged.
__global__ void k_zero_bad_slots(const int32_t* __restrict__ experts, int64_t slots, int64_t E,
                                 int64_t N, __nv_bfloat16* __restrict__ y, int32_t* dev_status) {
  const int64_t slot = blockIdx.x;
  if (slot >= slots) return;
  const int32_t e = experts[slot];
  if (e >= 0 && e < E) return;
  if (threadIdx.x == 0) set_dev_status(dev_status, WQ_DEV_BAD_EXPERT);
  if (y == nullptr) return;
  for (int64_t n = threadIdx.x; n < N; n += blockDim.x)
    y[slot * N + n] = __float2bfloat16_rn(0.0f);
}

// The combine step of mxfp4_combine_experts: the weighted slot results (f32, already
// multiplied by their combine weights) of a row are added in slot order, then rounded
// once to bf16.  Grid: (column chunks of 1024, rows).
__global__ void __launch_bounds__(256) k_combine_slots(const float* __restrict__ y32,
                                                       const int32_t* __restrict__ experts,
                                                       int64_t S, int64_t E, int64_t N,
                                                       __nv_bfloat16* __restrict__ y) {
  const int64_t r = blockIdx.y;
  const int64_t n = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (n >= N) return;
  float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  for (int64_t s = 0; s < S; ++s) {
    const int32_t e = __ldg(experts + r * S + s);
    if (e < 0 || e >= E) continue;
    const float* src = y32 + (r * S + s) * N + n;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (n + j < N) acc[j] += __ldcg(src + j);
  }
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if (n + j < N) y[r * N + n + j] = __float2bfloat16_rn(acc[j]);
}

// Activation order: xg[m, j] = x[m, order[j]] ("Quantization" (Linnet docs), "Importing
// GPTQ and AWQ": the layer gathers its inputs first).
__global__ void k_gather_cols(const unsigned short* __restrict__ x, const int32_t* __restrict__ order,
                              int64_t M, int64_t K, unsigned short* __restrict__ xg,
                              int32_t* dev_status) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= M * K) return;
  const int64_t m = i / K, j = i - m * K;
  const int32_t o = __ldg(order + j);
  const bool ok = (uint32_t)o < (uint64_t)K;
  xg[i] = ok ? __ldg(x + m * K + o) : (unsigned short)0;
  if (!ok) set_dev_status(dev_status, WQ_DEV_BAD_ORDER);
}

inline unsigned blocks_for(int64_t n, int threads) {
  return (unsigned)((n + threads - 1) / threads);
}

}  // namespace

cudaError_t launch_quantize(const float* w, int64_t N, int64_t K, int32_t G, int32_t bits,
                            int32_t mode, void* codes, float* scale, uint8_t* zero,
                            int32_t* dev_status, cudaStream_t s) {
  const int64_t warps = N * ((K + G - 1) / G);
  k_quantize<<<blocks_for(warps * 32, 256), 256, 0, s>>>(
      w, N, K, G, bits, mode, static_cast<uint8_t*>(codes), scale, zero, dev_status);
  return cudaGetLastError();
}

cudaError_t launch_pack(const void* codes, int64_t rows, int64_t cols, int32_t is_unsigned,
                        uint8_t* packed, int32_t* dev_status, cudaStream_t s) {
  const int64_t n = rows * cols / 2;
  k_pack<<<blocks_for(n, 256), 256, 0, s>>>(static_cast<const uint8_t*>(codes), n, is_unsigned,
                                            packed, dev_status);
  return cudaGetLastError();
}

cudaError_t launch_unpack(const uint8_t* packed, int64_t rows, int64_t cols,
                          int32_t is_unsigned, void* codes, cudaStream_t s) {
  const int64_t n = rows * cols / 2;
  k_unpack<<<blocks_for(n, 256), 256, 0, s>>>(packed, n, is_unsigned,
                                              static_cast<uint8_t*>(codes));
  return cudaGetLastError();
}

cudaError_t launch_dequant_i4g(const uint8_t* packed, const float* scale, const uint8_t* zero,
                               int64_t N, int64_t K, int32_t G, void* w, cudaStream_t s) {
  const int64_t n = N * K / 2;
  k_dequant_i4g<<<blocks_for(n, 256), 256, 0, s>>>(packed, scale, zero, N, K, G,
                                                   static_cast<__nv_bfloat16*>(w));
  return cudaGetLastError();
}

cudaError_t launch_dequant_i8r(const int8_t* q, const float* scale, int64_t N, int64_t K,
                               void* w, cudaStream_t s) {
  k_dequant_i8r<<<blocks_for(N * K, 256), 256, 0, s>>>(q, scale, N, K,
                                                       static_cast<__nv_bfloat16*>(w));
  return cudaGetLastError();
}

cudaError_t launch_dequant_i4r(const int8_t* packed, const float* scale, int64_t N, int64_t K,
                               void* w, cudaStream_t s) {
  k_dequant_i4r<<<blocks_for(N * K / 2, 256), 256, 0, s>>>(
      reinterpret_cast<const uint8_t*>(packed), scale, N, K, static_cast<__nv_bfloat16*>(w));
  return cudaGetLastError();
}

cudaError_t launch_zero_bad_slots(const int32_t* experts, int64_t slots, int64_t E, int64_t N,
                                  __nv_bfloat16* y, int32_t* dev_status, cudaStream_t s) {
  k_zero_bad_slots<<<(unsigned)slots, 256, 0, s>>>(experts, slots, E, N, y, dev_status);
  return cudaGetLastError();
}

cudaError_t launch_gather_cols(const __nv_bfloat16* x, const int32_t* order, int64_t M, int64_t K,
                               __nv_bfloat16* xg, int32_t* dev_status, cudaStream_t s) {
  k_gather_cols<<<blocks_for(M * K, 256), 256, 0, s>>>(reinterpret_cast<const unsigned short*>(x), order,
                                                      M, K, reinterpret_cast<unsigned short*>(xg),
                                                      dev_status);
  return cudaGetLastError();
}

cudaError_t launch_combine_slots(const float* y32, const int32_t* experts, int64_t R, int64_t S,
                                 int64_t E, int64_t N, __nv_bfloat16* y, cudaStream_t s) {
  const dim3 grid((unsigned)((N + 1023) / 1024), (unsigned)R);
  k_combine_slots<<<grid, 256, 0, s>>>(y32, experts, S, E, N, y);
  return cudaGetLastError();
}

cudaError_t launch_dequant_mxfp4(const uint8_t* blocks, const uint8_t* scales, int64_t E,
                                 int64_t N, int64_t K, void* w, cudaStream_t s) {
  k_dequant_mxfp4<<<blocks_for(E * N * K / 2, 256), 256, 0, s>>>(
      blocks, scales, E * N, K, static_cast<__nv_bfloat16*>(w));
  return cudaGetLastError();
}

}  // namespace wq
