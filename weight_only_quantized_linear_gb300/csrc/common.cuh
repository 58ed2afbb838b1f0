// common.cuh -- device helpers shared by the libwq kernels (sm_103a only).
//
// Inline PTX for the Blackwell data movers and barriers (mbarrier, cp.async.bulk.tensor),
// the legacy warp MMA used by the decode GEMV, and the exact nibble -> f32 conversions
// the dequantizers are built from.  Every wait on a barrier is bounded: it gives up
// after a deadline on the global timer, and the caller records WQ_DEV_TIMEOUT.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/wq.h"

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ < 1000)
#error "libwq is written for sm_103a (Blackwell) only"
#endif

namespace wq {

constexpr int kNumSMsFallback = 152;
// Bounded waits give up after this many nanoseconds of the global timer.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__host__ __device__ __forceinline__ int64_t imin64(int64_t a, int64_t b) { return a < b ? a : b; }
__host__ __device__ __forceinline__ int64_t imax64(int64_t a, int64_t b) { return a > b ? a : b; }

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait until the phase with the given parity has completed.  Returns false if
// `limit_ns` of the global timer passed first (the caller must then stop using the
// barrier's buffers).
__device__ __forceinline__ bool mbar_wait_limit(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  return mbar_wait_limit(bar, parity, kWaitLimitNs);
}

// ------------------------------------------------------------------ thread-block clusters
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster arrives (release) and waits (acquire): shared
// memory written before it is visible to the cluster's CTAs after it.  A hardware
// barrier: all threads must reach it (no early exit before it).
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The shared::cluster address of a shared::cta address in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_shared_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// The two halves of a cluster barrier: arrive (release) early, wait (acquire) just before
// the first access that needs the other CTAs to have passed the arrive.  Every thread of
// every CTA executes each once, warp-uniformly.
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Store a float to shared::cluster address `addr` (another CTA's shared memory).
__device__ __forceinline__ void st_shared_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
// Arrive (release at cluster scope) on the mbarrier at shared::cluster address `addr`: the
// thread's earlier stores, remote ones included, are visible to whoever acquires the phase.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(addr)
               : "memory");
}
// Wait (acquire at cluster scope) for the phase with the given parity of a barrier of this
// CTA that other CTAs of the cluster arrive on; bounded like mbar_wait.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait_cluster(bar, parity)) return true;
    if (global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
}
__device__ __forceinline__ float4 ld_shared_cluster_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// ------------------------------------------------------------------ programmatic dependent launch
// Allow the next kernel of the stream (launched with programmatic stream serialization)
// to be scheduled now; it still waits for this grid's completion in grid_dep_wait().
__device__ __forceinline__ void grid_dep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Wait until the grids this one depends on have completed and their memory is visible.
// Nothing written by an earlier kernel may be read, and nothing an earlier kernel reads
// may be written, before this.
__device__ __forceinline__ void grid_dep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ------------------------------------------------------------------ TMA (bulk tensor)
// 2-D tile load global -> shared, completing `bytes` on the mbarrier.  Coordinates are
// in elements of the tensor map (innermost first).  `policy` is an L2 cache policy.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t c0, int32_t c1, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "l"(policy)
      : "memory");
}
// Untiled bulk copy global -> shared (shared address dst), completing `bytes` on the
// mbarrier: both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// L2 policies: streamed weights are read once (evict first); activations are reused.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ------------------------------------------------------------------ loads
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
__device__ __forceinline__ float2 ld_shared_f32x2(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t ld_shared_u16(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ float ld_shared_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t ld_shared_u8(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
// Read-only 16-byte global load that stays in L1 (activations are reused by every
// thread block of the SM).  Not volatile: the data never changes during a kernel, so the
// compiler may hoist and interleave these loads freely.
__device__ __forceinline__ uint4 ld_global_nc_v4(const void* p) {
  uint4 v;
  asm("ld.global.nc.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Bring the line holding p into L1 ahead of its use (no register, no wait).
__device__ __forceinline__ void prefetch_l1(const void* p) {
  asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}

// Streaming 16-byte global load: read once, so it does not displace L1 lines.
__device__ __forceinline__ uint4 ld_global_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// ------------------------------------------------------------------ warp MMA
// D(16x8, f32) += A(16x16, bf16, row-major) * B(16x8, bf16, column-major).  A pure
// function of its operands (not volatile), so that the compiler can overlap it with loads.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// acc += lo(a) * lo(b) and acc2 += hi(a) * hi(b) for bf16x2 registers a, b: the bf16
// products are exact in f32 and each add rounds once (mixed-precision FMA, f32 result).
__device__ __forceinline__ void fma_bf16x2_f32(uint32_t a, uint32_t b, float& acc, float& acc2) {
  asm("{\n .reg .b16 al, ah, bl, bh;\n mov.b32 {al, ah}, %2;\n mov.b32 {bl, bh}, %3;\n"
      " fma.rn.f32.bf16 %0, al, bl, %0;\n fma.rn.f32.bf16 %1, ah, bh, %1;\n}"
      : "+f"(acc), "+f"(acc2)
      : "r"(a), "r"(b));
}

// acc += half HA of a * half HB of b (0: bits 0..15, 1: bits 16..31), bf16 inputs: the
// product is exact in f32 and the add rounds once.
template <int HA, int HB>
__device__ __forceinline__ void fma_mix(float& acc, uint32_t a, uint32_t b) {
  if constexpr (HA == 0 && HB == 0)
    asm("{\n .reg .b16 a0, a1, b0, b1;\n mov.b32 {a0, a1}, %1;\n mov.b32 {b0, b1}, %2;\n"
        " fma.rn.f32.bf16 %0, a0, b0, %0;\n}" : "+f"(acc) : "r"(a), "r"(b));
  else if constexpr (HA == 0 && HB == 1)
    asm("{\n .reg .b16 a0, a1, b0, b1;\n mov.b32 {a0, a1}, %1;\n mov.b32 {b0, b1}, %2;\n"
        " fma.rn.f32.bf16 %0, a0, b1, %0;\n}" : "+f"(acc) : "r"(a), "r"(b));
  else if constexpr (HA == 1 && HB == 0)
    asm("{\n .reg .b16 a0, a1, b0, b1;\n mov.b32 {a0, a1}, %1;\n mov.b32 {b0, b1}, %2;\n"
        " fma.rn.f32.bf16 %0, a1, b0, %0;\n}" : "+f"(acc) : "r"(a), "r"(b));
  else
    asm("{\n .reg .b16 a0, a1, b0, b1;\n mov.b32 {a0, a1}, %1;\n mov.b32 {b0, b1}, %2;\n"
        " fma.rn.f32.bf16 %0, a1, b1, %0;\n}" : "+f"(acc) : "r"(a), "r"(b));
}

// (a & 0x000F000F) | c as one logic op.  c is passed in a register: with two immediate
// constants the compiler splits the expression into two logic ops.
__device__ __forceinline__ uint32_t and_0f_or(uint32_t a, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, 0x000F000F, %2, 0xEA;" : "=r"(d) : "r"(a), "r"(c));
  return d;
}

// Packed bf16 subtraction a - b, rounded to nearest even (exact for the small integers
// the factored decode subtracts).
__device__ __forceinline__ uint32_t sub_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// ------------------------------------------------------------------ conversions
// Pack two f32 into bf16x2 with round-to-nearest-even: `lo` in bits 0..15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Exact 4-bit dequantization to f32, eight codes of a 32-bit word at a time.
//
// Code p of the word (bits 4p..4p+3) is moved into the mantissa of the float 2^23 by a
// single logic op: the float with bits 0x4B000000 | (code << 4p) equals 2^23 + code * 16^p
// exactly for p <= 3.  Codes 4..7 are first shifted down by 16 bits, landing on the same
// multipliers 1, 16, 256, 4096.  Subtracting the exact constant 2^23 + zero * m leaves
// (code - zero) * m exactly, and multiplying by scale / m (an exact power-of-two rescaling
// of the f32 scale) gives the correctly rounded f32 product (code - zero) * scale: the same
// real number, rounded once.  The conversion to bf16 then rounds to nearest even.  So every
// element equals bf16(f32(code - zero) * scale), bit for bit, for about one logic op, half
// a packed add, half a packed multiply and half a paired conversion an element.
//
// Element pairs (0,1) (2,3) (4,5) (6,7) use the multipliers (1, 16) (256, 4096) (1, 16)
// (256, 4096): two constant pairs a row.  (Exactness needs scale / 4096 to stay a normal
// f32, i.e. |scale| >= 2^-114 or scale == 0.)
struct Nib8Consts {
  float2 negc[2];  // -(2^23 + zero * m) for m = (1, 16) and (256, 4096)
  float2 s[2];     // scale / m
};

__device__ __forceinline__ Nib8Consts make_nib8_consts(float scale, float zero) {
  const float T = 8388608.0f;  // 2^23
  // zero * m is exact (at most 255 * 4096), so each constant is exact
  Nib8Consts k;
  k.negc[0] = make_float2(-(T + zero), fmaf(zero, -16.0f, -T));
  k.negc[1] = make_float2(fmaf(zero, -256.0f, -T), fmaf(zero, -4096.0f, -T));
  k.s[0] = make_float2(scale, scale * 0.0625f);
  k.s[1] = make_float2(scale * 0.00390625f, scale * 0.000244140625f);
  return k;
}
// The same from an integer zero point 0..255 (converted through the 2^23 magic number:
// a logic op and an add instead of an int-to-float conversion).
__device__ __forceinline__ Nib8Consts make_nib8_consts_u(float scale, uint32_t zero) {
  const float zf = __uint_as_float(0x4B000000u | zero) - 8388608.0f;
  return make_nib8_consts(scale, zf);
}

// out[i] = bf16x2 of elements (2i, 2i+1) of the word.
__device__ __forceinline__ void dequant_nib8(uint32_t w, const Nib8Consts& k,
                                             uint32_t (&out)[4]) {
  const uint32_t t = w >> 16;
  const uint32_t M = 0x4B000000u;
  const float2 f01 = make_float2(__uint_as_float(M | (w & 0x000Fu)), __uint_as_float(M | (w & 0x00F0u)));
  const float2 f23 = make_float2(__uint_as_float(M | (w & 0x0F00u)), __uint_as_float(M | (w & 0xF000u)));
  const float2 f45 = make_float2(__uint_as_float(M | (t & 0x000Fu)), __uint_as_float(M | (t & 0x00F0u)));
  const float2 f67 = make_float2(__uint_as_float(M | (t & 0x0F00u)), __uint_as_float(M | (t & 0xF000u)));
  const float2 v01 = __fmul2_rn(__fadd2_rn(f01, k.negc[0]), k.s[0]);
  const float2 v23 = __fmul2_rn(__fadd2_rn(f23, k.negc[1]), k.s[1]);
  const float2 v45 = __fmul2_rn(__fadd2_rn(f45, k.negc[0]), k.s[0]);
  const float2 v67 = __fmul2_rn(__fadd2_rn(f67, k.negc[1]), k.s[1]);
  out[0] = pack_bf16x2(v01.x, v01.y);
  out[1] = pack_bf16x2(v23.x, v23.y);
  out[2] = pack_bf16x2(v45.x, v45.y);
  out[3] = pack_bf16x2(v67.x, v67.y);
}

// Exact int8 dequantization, four codes of a word: the byte (q + 128) is placed in the
// mantissa of 2^23 by a byte permute, 2^23 + 128 is subtracted exactly, and the f32
// product q * scale is rounded once, then to bf16.  out[0] = (b0, b1), out[1] = (b2, b3).
__device__ __forceinline__ void dequant_i8x4(uint32_t w, float2 negc, float2 s,
                                             uint32_t (&out)[2]) {
  const uint32_t u = w ^ 0x80808080u;  // two's complement -> offset binary
  const uint32_t M = 0x4B000000u;
  uint32_t b0, b1, b2, b3;
  asm("prmt.b32 %0, %1, %2, 0x7440;" : "=r"(b0) : "r"(u), "r"(M));
  asm("prmt.b32 %0, %1, %2, 0x7441;" : "=r"(b1) : "r"(u), "r"(M));
  asm("prmt.b32 %0, %1, %2, 0x7442;" : "=r"(b2) : "r"(u), "r"(M));
  asm("prmt.b32 %0, %1, %2, 0x7443;" : "=r"(b3) : "r"(u), "r"(M));
  const float2 v01 =
      __fmul2_rn(__fadd2_rn(make_float2(__uint_as_float(b0), __uint_as_float(b1)), negc), s);
  const float2 v23 =
      __fmul2_rn(__fadd2_rn(make_float2(__uint_as_float(b2), __uint_as_float(b3)), negc), s);
  out[0] = pack_bf16x2(v01.x, v01.y);
  out[1] = pack_bf16x2(v23.x, v23.y);
}

// E8M0 scale byte -> 2^(b - 127) as f32 (b = 0 is the subnormal 2^-127; 255 is NaN).
__device__ __forceinline__ float e8m0_to_f32(uint32_t b) {
  if (b == 255u) return __uint_as_float(0x7FC00000u);
  if (b == 0u) return __uint_as_float(0x00400000u);
  return __uint_as_float(b << 23);
}

// Two E2M1 codes (a byte, even element in the low nibble) -> two f32 values, through
// the hardware E2M1x2 -> f16x2 conversion (exact: every E2M1 value is an f16).
__device__ __forceinline__ float2 e2m1x2_to_f32x2(uint32_t byte_in_low_bits) {
  uint32_t h;
  asm("{\n .reg .b8 t;\n cvt.u8.u32 t, %1;\n cvt.rn.f16x2.e2m1x2 %0, t;\n}"
      : "=r"(h)
      : "r"(byte_in_low_bits));
  const __half2 hh = *reinterpret_cast<const __half2*>(&h);
  return __half22float2(hh);
}

// Eight E2M1 codes of a word times the block scale X -> four bf16x2 (exact products).
__device__ __forceinline__ void dequant_e2m1x8(uint32_t w, float2 X, uint32_t (&out)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 v = __fmul2_rn(e2m1x2_to_f32x2(w >> (8 * i)), X);
    out[i] = pack_bf16x2(v.x, v.y);
  }
}

// ------------------------------------------------------------------ factored decode helpers
// The factored decode kernels form (q - zero) exactly in bf16 and multiply the chunk's
// f32 sum by its scale once (the definition's products reassociated, see gemv.cu).
// Four int8 codes of a word as exact bf16x2 pairs (k0, k1) and (k2, k3).
__device__ __forceinline__ void i8x4_to_bf16x2(uint32_t w, uint32_t (&out)[2]) {
  const uint32_t u = w ^ 0x80808080u;                      // bytes q + 128
  const float2 c = make_float2(-8388736.0f, -8388736.0f);  // -(2^23 + 128)
  const float2 f01 =
      __fadd2_rn(make_float2(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7440)),
                             __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7441))), c);
  const float2 f23 =
      __fadd2_rn(make_float2(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7442)),
                             __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7443))), c);
  out[0] = pack_bf16x2(f01.x, f01.y);
  out[1] = pack_bf16x2(f23.x, f23.y);
}

// Eight 4-bit codes of a word (even element in the low nibble) minus a zero point, as
// exact bf16x2 pairs d[j] = (k j, k j + 4).  zc = bf16x2 of 128 + min(z, 127); zc2 = bf16x2
// of max(z - 127, 0), used only when `big`; magic = 0x43004300 (bf16x2 128, 128) held in a
// register.
template <bool kBig>
__device__ __forceinline__ void nib8_minus_zero(uint32_t w, uint32_t zc, uint32_t zc2,
                                                uint32_t magic, uint32_t (&d)[4]) {
  // plain shifts (measured faster on sm_103a than high halves of products, which move
  // them to the FMA pipe)
  d[0] = sub_bf16x2(and_0f_or(w, magic), zc);
  d[1] = sub_bf16x2(and_0f_or(w >> 4, magic), zc);
  d[2] = sub_bf16x2(and_0f_or(w >> 8, magic), zc);
  d[3] = sub_bf16x2(and_0f_or(w >> 12, magic), zc);
  if constexpr (kBig) {
#pragma unroll
    for (int j = 0; j < 4; ++j) d[j] = sub_bf16x2(d[j], zc2);
  }
}

// ------------------------------------------------------------------ exact MXFP4 unpack
// A code (s, e1 e0, m) with its sign in bf16 bit 15 and e1 e0 m in bits 8..6 is the bf16
// E2M1 * 2^-126 (the 0 / 0.5 codes as subnormals); one packed bf16 multiply by 2^(e - 1)
// (e <= 128) gives bf16(E2M1 * 2^(e - 127)) exactly, two multiplies (by 2^126, then by the
// E8M0 value) any scale byte.  Codes j and j + 4 of a word form one bf16x2 pair.
// bf16x2 a * b, rounded to nearest even
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// (b & 0x80008000) | (a & 0x01C001C0): the sign of a code pair from b, exponent and
// mantissa bits from a
__device__ __forceinline__ uint32_t e2m1_pair_bits(uint32_t a, uint32_t b) {
  uint32_t t, d;
  asm("lop3.b32 %0, %1, 0x01C001C0, 0, 0xC0;" : "=r"(t) : "r"(a));
  asm("lop3.b32 %0, %1, 0x80008000, %2, 0xEA;" : "=r"(d) : "r"(b), "r"(t));
  return d;
}
// The eight codes of a word as four bf16x2 pairs (codes j and j + 4) of E2M1 * 2^-126,
// each multiplied by s2 (bf16x2) and, for kTwo, then by s2b.
template <bool kTwo>
__device__ __forceinline__ void e2m1x8_scaled(uint32_t w, uint32_t s2, uint32_t s2b, uint32_t (&d)[4]) {
  d[0] = e2m1_pair_bits(w << 6, w << 12);
  d[1] = e2m1_pair_bits(w << 2, w << 8);
  d[2] = e2m1_pair_bits(w >> 2, w << 4);
  d[3] = e2m1_pair_bits(w >> 6, w);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    d[j] = mul_bf16x2(d[j], s2);
    if constexpr (kTwo) d[j] = mul_bf16x2(d[j], s2b);
  }
}
// bf16x2 of 2^(e - 1) (e <= 128), and of the E8M0 value 2^(e - 127) (NaN for 255)
__device__ __forceinline__ uint32_t pow2_em1_bf16x2(uint32_t e) { return ((e + 126u) << 7) * 0x00010001u; }
__device__ __forceinline__ uint32_t e8m0_bf16x2(uint32_t e) {
  const uint32_t h = (e == 0u) ? 0x0040u : (e == 255u ? 0x7FC0u : (e << 7));
  return h * 0x00010001u;
}

__device__ __forceinline__ void set_dev_status(int32_t* st, int32_t bits) {
  if (st) atomicOr(st, bits);
}

}  // namespace wq
