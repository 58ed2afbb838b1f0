// gemm_mx.cu -- MXFP4 experts with many routed rows (prefill and serving batches): a
// grouped tcgen05 GEMM over the rows routed to each expert.
//
// "Quantization" (Linnet docs), format table: mxfp4_experts_shared, mxfp4_experts,
// mxfp4_linear_experts_shared ("many rows (x: [R, In])"), mxfp4_combine_experts; "MXFP4
// experts": the work grouped by expert.  The element is the same as in the decode kernels:
// W-hat = bf16(E2M1 * 2^(scale - 127)), formed exactly (common.cuh, exact MXFP4 unpack).
//
// Steps (one stream, three launches):
//   1. k_gx_route   (one block) per-expert counts of the routed slots, each expert's
//                   segment of the sorted slot list and the prefix sums of its 256-row
//                   tiles, then each slot's position in its segment; slots with an expert
//                   index outside [0, E) form a last segment (WQ_DEV_BAD_EXPERT);
//   2. k_gx_gather  the input row of each position (the routed row's shared input, or the
//                   slot's own row for mxfp4_experts), copied in segment order with the
//                   eight elements of every 16 bytes reordered (0, 4, 1, 5, 2, 6, 3, 7): the
//                   pairing the unpack produces for the weights, so both MMA operands hold
//                   the same permutation of k;
//   3. k_gemm_mx_tc one block a (256-row tile of one expert's segment, 256 weight rows):
//                   warp 0 loads the activation tile and the expert's packed codes by TMA,
//                   warps 2..9 unpack the codes into the canonical 128-byte-swizzled bf16
//                   tile, one thread of warp 1 issues tcgen05.mma into two 128 x 256 TMEM
//                   accumulators (one for a tile of at most 128 rows); the epilogue writes
//                   each row to its slot of y (bf16), or its f32 result times the slot's
//                   weight to the combine workspace.  Tiles of the last segment write zero
//                   rows to y and multiply nothing.
// Every wait is bounded; a timeout records WQ_DEV_TIMEOUT and the block winds down.
#include <algorithm>
#include <atomic>

#include "common.cuh"
#include "launch.h"
#include "tc.cuh"

namespace wq {
namespace {

constexpr int kGxBM = 256;  // routed rows a tile
constexpr int kGxBN = 256;  // weight rows a tile
constexpr int kGxBK = 64;   // k a stage
constexpr int kGxStages = 3;
constexpr int kGxDqWarps = 8;
constexpr int kGxThreads = (2 + kGxDqWarps) * 32;
constexpr int kGxABytes = kGxBM * kGxBK * 2;
constexpr int kGxBBytes = kGxBN * kGxBK * 2;
constexpr int kGxPBytes = kGxBN * kGxBK / 2;
constexpr int kGxStageBytes = kGxABytes + kGxBBytes + kGxPBytes;
constexpr int kGxMaxExperts = 256;
constexpr int kGxMinSlots = 512;  // routed slots from which the GEMM takes over (default)

// Workspace: header [2][E + 2] i32 (segment starts, tile starts), sorted slots [RS] i32,
// gathered activations [RS, K] bf16; sections 256-byte aligned.
// Tiles that reach past the gathered rows read zeros (the tensor map's bounds).
struct GxLayout {
  size_t sorted, xg, total;
};
GxLayout gx_layout(int64_t RS, int64_t E, int64_t K) {
  auto al = [](size_t v) { return (v + 255) & ~size_t(255); };
  GxLayout L;
  L.sorted = al(2 * 4 * (size_t)(E + 2));
  L.xg = L.sorted + al(4 * (size_t)RS);
  L.total = L.xg + al((size_t)RS * (size_t)K * 2);
  return L;
}

struct GxParams {
  const int32_t* hdr;      // [2][E + 2]: segment starts, tile starts (segment E: bad slots)
  const int32_t* sorted;   // [RS]
  const uint8_t* escale;   // [E, N, K/32]
  int64_t E, N, K;
  __nv_bfloat16* y;        // [RS, N] or NULL
  float* y32;              // [RS, N] (combine) or NULL
  const float* sw;         // [RS] combine weights or NULL
  int32_t* dev_status;
};

struct SharedGx {
  uint64_t full_tma[kGxStages];
  uint64_t full_b[kGxStages];
  uint64_t empty[kGxStages];
  uint64_t acc_full;
  uint32_t tmem_base;
  int abort;
  int expert, m0, mend;
  int halves;  // 128-row halves of the tile holding routed rows (1 or 2)
};

// One block: the routed slots' segments.  Segment e < E holds the slots routed to expert
// e; segment E the slots whose expert index lies outside [0, E) (zero rows, no product).
// The header gets the segment starts and the prefix sums of each segment's 256-row tiles;
// each slot then takes a position in its segment (the order inside a segment is free:
// every output row is computed on its own).
__global__ void __launch_bounds__(1024) k_gx_route(const int32_t* __restrict__ experts, int RS, int E,
                                                   int32_t* __restrict__ hdr, int32_t* __restrict__ sorted,
                                                   int32_t* __restrict__ dev_status) {
  __shared__ int s_cnt[kGxMaxExperts + 1];
  __shared__ int s_fill[kGxMaxExperts + 1];
  for (int e = threadIdx.x; e <= E; e += blockDim.x) s_cnt[e] = 0;
  __syncthreads();
  auto seg_of = [&](int i) {
    const int e = experts[i];
    return (e >= 0 && e < E) ? e : E;
  };
  for (int i = threadIdx.x; i < RS; i += blockDim.x) atomicAdd(&s_cnt[seg_of(i)], 1);
  __syncthreads();
  if (threadIdx.x == 0) {
    int32_t* const seg = hdr;
    int32_t* const tst = hdr + (E + 2);
    int run = 0, truns = 0;
    for (int e = 0; e <= E; ++e) {
      seg[e] = run;
      tst[e] = truns;
      s_fill[e] = run;
      run += s_cnt[e];
      truns += (s_cnt[e] + kGxBM - 1) / kGxBM;
    }
    seg[E + 1] = run;
    tst[E + 1] = truns;
    if (s_cnt[E] > 0) set_dev_status(dev_status, WQ_DEV_BAD_EXPERT);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < RS; i += blockDim.x) sorted[atomicAdd(&s_fill[seg_of(i)], 1)] = i;
}

__global__ void __launch_bounds__(256) k_gx_gather(const __nv_bfloat16* __restrict__ x, int64_t K, int64_t S,
                                                   int x_per_slot, int E, const int32_t* __restrict__ hdr,
                                                   const int32_t* __restrict__ sorted,
                                                   __nv_bfloat16* __restrict__ xg) {
  const int64_t k8n = K / 8;
  const int64_t total = (int64_t)hdr[E] * k8n;  // routed slots (segments 0 .. E - 1) x 16-byte pieces
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t pos = idx / k8n, k8 = idx - pos * k8n;
    const int slot = sorted[pos];
    const int64_t row = x_per_slot ? slot : slot / S;  // the slot's own row, or its routed row's
    const uint4 v = ld_global_nc_v4(x + row * K + k8 * 8);
    const uint4 o = make_uint4(__byte_perm(v.x, v.z, 0x5410), __byte_perm(v.x, v.z, 0x7632),
                               __byte_perm(v.y, v.w, 0x5410), __byte_perm(v.y, v.w, 0x7632));
    *reinterpret_cast<uint4*>(xg + pos * K + k8 * 8) = o;
  }
}

__global__ void __launch_bounds__(kGxThreads, 1)
    k_gemm_mx_tc(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap,
                 const GxParams p) {
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) &
                                             ~uintptr_t(1023));
  SharedGx* sh = reinterpret_cast<SharedGx*>(smem + kGxStages * kGxStageBytes);
  auto stage_a = [&](int s) { return smem + s * kGxStageBytes; };
  auto stage_b = [&](int s) { return smem + s * kGxStageBytes + kGxABytes; };
  auto stage_p = [&](int s) { return smem + s * kGxStageBytes + kGxABytes + kGxBBytes; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int E = (int)p.E;
  const int64_t N = p.N, K = p.K;
  const int32_t* const seg = p.hdr;
  const int32_t* const tst = p.hdr + (E + 2);

  // this block's tile: the segment whose tile range holds blockIdx.x
  if (threadIdx.x == 0) {
    const int t = (int)blockIdx.x;
    int e = -1;
    if (t < tst[E + 1]) {
      int lo = 0, hi = E;  // largest e with tst[e] <= t (and a tile of its own)
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tst[mid] <= t) lo = mid; else hi = mid - 1;
      }
      e = lo;
    }
    sh->expert = e;
    sh->m0 = (e >= 0) ? seg[e] + (t - tst[e]) * kGxBM : 0;
    sh->mend = (e >= 0) ? seg[e + 1] : 0;
    sh->halves = (sh->mend - sh->m0 > kGxBM / 2) ? 2 : 1;
  }
  __syncthreads();
  const int expert = sh->expert;
  if (expert < 0) return;  // past the last tile (the grid is sized for the worst case)
  const int64_t m0 = sh->m0, mend = sh->mend;
  if (expert == E) {
    // slots with an expert index outside [0, E): zero rows of y (the combine form skips
    // them); no product
    if (p.y != nullptr) {
      const int64_t n0z = (int64_t)blockIdx.y * kGxBN;
      const int64_t nz = imin64(N - n0z, kGxBN);
      const int64_t rows = imin64(mend - m0, kGxBM);
      for (int64_t i = threadIdx.x; i < rows * nz; i += blockDim.x) {
        const int64_t r = i / nz;
        p.y[(int64_t)p.sorted[m0 + r] * N + n0z + (i - r * nz)] = __float2bfloat16_rn(0.0f);
      }
    }
    return;
  }
  // a tile with at most 128 routed rows (small segments, a segment's last tile) loads,
  // multiplies and stores only its first half: one accumulator instead of two
  const int halves = sh->halves;
  const int64_t n0 = (int64_t)blockIdx.y * kGxBN;
  const int nk = (int)((K + kGxBK - 1) / kGxBK);  // K % 64 == 32: the last step's second block reads zeros

  if (threadIdx.x == 0) {
    for (int s = 0; s < kGxStages; ++s) {
      mbar_init(&sh->full_tma[s], 1);
      mbar_init(&sh->full_b[s], kGxDqWarps);
      mbar_init(&sh->empty[s], 1);
    }
    mbar_init(&sh->acc_full, 1);
    fence_mbar_init();
    sh->abort = 0;
  }
  if (warp == 1) tmem_alloc(&sh->tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh->tmem_base;

  if (warp == 0) {
    // ================= TMA producer =================
    if (lane == 0) {
      tma_prefetch_desc(&xmap);
      tma_prefetch_desc(&wmap);
      // the gathered rows are reread for every 256 weight rows: kept in L2; an expert's
      // codes serve only the blocks of its segment, which run together: streamed
      const uint64_t pol = l2_policy_evict_last();
      const uint64_t pol_w = l2_policy_evict_first();
      const int32_t wrow = (int32_t)((int64_t)expert * N + n0);
      int issued = 0;
      for (int kb = 0; kb < nk; ++kb) {
        const int s = kb % kGxStages;
        if (kb >= kGxStages && !mbar_wait(&sh->empty[s], ((kb / kGxStages) - 1) & 1)) {
          set_dev_status(p.dev_status, WQ_DEV_TIMEOUT);
          atomicExch(&sh->abort, 1);
          break;
        }
        if (*reinterpret_cast<volatile int*>(&sh->abort)) break;
        mbar_arrive_expect_tx(&sh->full_tma[s], halves * (kGxABytes / 2) + kGxPBytes);
        for (int h = 0; h < halves; ++h)
          tma_load_2d(stage_a(s) + h * (kGxABytes / 2), &xmap, &sh->full_tma[s], kb * kGxBK,
                      (int32_t)(m0 + h * (kGxBM / 2)), pol);
        tma_load_2d(stage_p(s), &wmap, &sh->full_tma[s], kb * (kGxBK / 2), wrow, pol_w);
        issued = kb + 1;
      }
      for (int kb = std::max(0, issued - kGxStages); kb < issued; ++kb)
        (void)mbar_wait(&sh->full_tma[kb % kGxStages], (uint32_t)(kb / kGxStages) & 1u);
    }
  } else if (warp == 1) {
    // ================= MMA issuer =================
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(128, kGxBN);
      for (int kb = 0; kb < nk; ++kb) {
        const int s = kb % kGxStages;
        if (*reinterpret_cast<volatile int*>(&sh->abort)) break;
        if (!mbar_wait(&sh->full_tma[s], (kb / kGxStages) & 1) ||
            !mbar_wait(&sh->full_b[s], (kb / kGxStages) & 1)) {
          set_dev_status(p.dev_status, WQ_DEV_TIMEOUT);
          atomicExch(&sh->abort, 1);
          break;
        }
        tc_fence_after();
        const uint32_t a_base = smem_u32(stage_a(s));
        const uint32_t b_base = smem_u32(stage_b(s));
        for (int acc = 0; acc < halves; ++acc) {
#pragma unroll
          for (int kk = 0; kk < kGxBK / 16; ++kk) {
            const uint64_t ad = umma_desc_sw128(a_base + acc * (128 * 128) + kk * 32);
            const uint64_t bd = umma_desc_sw128(b_base + kk * 32);
            umma_bf16(tmem + acc * kGxBN, ad, bd, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
          }
        }
        umma_commit(&sh->empty[s]);
      }
      umma_commit(&sh->acc_full);
    }
  } else {
    // ================= unpack (8 warps), then epilogue =================
    // thread t owns weight row n0 + t (rows past N unpack the last row; never stored)
    const int t = threadIdx.x - 64;
    const int64_t n = imin64(n0 + t, N - 1);
    const int64_t kb32 = K / 32;
    const uint8_t* const srow = p.escale + ((int64_t)expert * N + n) * kb32;
    const uint32_t prow = (uint32_t)t * 32;  // packed row, 32-byte swizzle
    const uint32_t pswz = (uint32_t)((t >> 2) & 1);
    const uint32_t pa0 = prow + (pswz << 4), pa1 = prow + ((1u ^ pswz) << 4);
    uint32_t boff[8];
#pragma unroll
    for (int w = 0; w < 8; ++w) boff[w] = (uint32_t)t * 128 + (((uint32_t)w ^ (uint32_t)(t & 7)) << 4);
    // the two E8M0 bytes of a stage (blocks 2 kb and 2 kb + 1), one stage ahead; a block
    // past K (K % 64 == 32) has zero codes and takes scale byte 127
    auto load_e = [&](int kb) -> uint32_t {
      const int64_t b = 2 * (int64_t)kb;
      return (uint32_t)__ldg(srow + b) | ((b + 1 < kb32 ? (uint32_t)__ldg(srow + b + 1) : 127u) << 8);
    };
    uint32_t e_next = load_e(0);
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % kGxStages;
      const uint32_t ecur = e_next;
      if (kb + 1 < nk) e_next = load_e(kb + 1);
      // the warp leaves together (the vote below needs every lane): lane 0's view of the
      // abort flag, and the stage's wait passed by all lanes or by none
      if (__shfl_sync(0xffffffffu, *reinterpret_cast<volatile int*>(&sh->abort), 0)) break;
      if (!__all_sync(0xffffffffu, mbar_wait(&sh->full_tma[s], (kb / kGxStages) & 1))) {
        set_dev_status(p.dev_status, WQ_DEV_TIMEOUT);
        atomicExch(&sh->abort, 1);
        break;
      }
      const uint32_t e0 = ecur & 0xFFu, e1 = ecur >> 8;
      const uint32_t pbase = smem_u32(stage_p(s));
      const uint32_t bbase = smem_u32(stage_b(s));
      const uint4 c0 = ld_shared_v4(pbase + pa0);
      const uint4 c1 = ld_shared_v4(pbase + pa1);
      const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
      auto unpack = [&](auto two_tag, uint32_t sa, uint32_t sb, uint32_t ta, uint32_t tb) {
        constexpr bool kTwo = decltype(two_tag)::value;
#pragma unroll
        for (int w = 0; w < 8; ++w) {
          uint32_t o[4];
          e2m1x8_scaled<kTwo>(words[w], w < 4 ? sa : sb, w < 4 ? ta : tb, o);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(bbase + boff[w]), "r"(o[0]),
                       "r"(o[1]), "r"(o[2]), "r"(o[3])
                       : "memory");
        }
      };
      if (__all_sync(0xffffffffu, max(e0, e1) <= 128u)) {
        unpack(std::false_type{}, pow2_em1_bf16x2(e0), pow2_em1_bf16x2(e1), 0u, 0u);
      } else {
        const uint32_t c126 = 0x7E807E80u;  // bf16x2 (2^126, 2^126)
        unpack(std::true_type{}, c126, c126, e8m0_bf16x2(e0), e8m0_bf16x2(e1));
      }
      fence_async_shared();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->full_b[s]);
    }

    // ---- epilogue: TMEM -> registers -> the rows' slots ----
    if (!mbar_wait(&sh->acc_full, 0)) {
      set_dev_status(p.dev_status, WQ_DEV_TIMEOUT);
      atomicExch(&sh->abort, 1);
    }
    tc_fence_after();
    const int q = warp & 3;
    const int acc = (warp - 2) >> 2;
    const int chunks = (acc < halves) ? kGxBN / 32 : 0;  // the second half of a half tile: no rows
    const int64_t m = m0 + acc * 128 + q * 32 + lane;  // position in the sorted slot list
    const int slot = (m < mend) ? p.sorted[m] : -1;
    const float wgt = (slot >= 0 && p.sw) ? __ldg(p.sw + slot) : 1.0f;
#pragma unroll 1
    for (int ch = 0; ch < chunks; ++ch) {
      uint32_t r[32];
      tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + acc * kGxBN + ch * 32, r);
      const int64_t nb = n0 + ch * 32;
      if (slot < 0 || nb >= N) continue;
      if (p.y32 != nullptr) {
        float* dst = p.y32 + (int64_t)slot * N + nb;
        if (N % 4 == 0 && nb + 32 <= N && (reinterpret_cast<uintptr_t>(p.y32) & 15) == 0) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            *reinterpret_cast<float4*>(dst + 4 * i) =
                make_float4(__uint_as_float(r[4 * i]) * wgt, __uint_as_float(r[4 * i + 1]) * wgt,
                            __uint_as_float(r[4 * i + 2]) * wgt, __uint_as_float(r[4 * i + 3]) * wgt);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (nb + i < N) dst[i] = __uint_as_float(r[i]) * wgt;
        }
      } else {
        __nv_bfloat16* dst = p.y + (int64_t)slot * N + nb;
        if (N % 8 == 0 && nb + 32 <= N && (reinterpret_cast<uintptr_t>(p.y) & 15) == 0) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint4 o;
            o.x = pack_bf16x2(__uint_as_float(r[8 * i + 0]), __uint_as_float(r[8 * i + 1]));
            o.y = pack_bf16x2(__uint_as_float(r[8 * i + 2]), __uint_as_float(r[8 * i + 3]));
            o.z = pack_bf16x2(__uint_as_float(r[8 * i + 4]), __uint_as_float(r[8 * i + 5]));
            o.w = pack_bf16x2(__uint_as_float(r[8 * i + 6]), __uint_as_float(r[8 * i + 7]));
            *reinterpret_cast<uint4*>(dst + 8 * i) = o;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (nb + i < N) dst[i] = __float2bfloat16_rn(__uint_as_float(r[i]));
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

namespace {
int64_t gemm_mx_min_slots() {
  const int64_t v = tuning(kKnobMxGemmMinSlots);
  return v >= 1 ? v : kGxMinSlots;
}
}  // namespace

bool gemm_mx_ok(int64_t R, int64_t S, int64_t E, int64_t N, int64_t K, const void* x, const void* blocks,
                const void* scales) {
  const int64_t RS = R * S;
  if (RS < gemm_mx_min_slots() || E > kGxMaxExperts || K % 32 != 0 || K < 32 || N < 1) return false;
  if (RS >= (int64_t(1) << 30) || E * N >= (int64_t(1) << 31)) return false;
  if ((N + kGxBN - 1) / kGxBN > 65535) return false;  // column blocks: the grid's y extent
  return ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(blocks) |
           reinterpret_cast<uintptr_t>(scales)) & 15) == 0;
}

size_t gemm_mx_ws_bytes(int64_t RS, int64_t E, int64_t K) { return gx_layout(RS, E, K).total; }

cudaError_t launch_gemm_mx(const __nv_bfloat16* x, int64_t R, int64_t S, int x_per_slot, const uint8_t* blocks,
                           const uint8_t* scales, int64_t E, int64_t N, int64_t K, const int32_t* experts,
                           __nv_bfloat16* y, float* y32, const float* sw, void* workspace,
                           int32_t* dev_status, cudaStream_t stream) {
  const int64_t RS = R * S;
  const GxLayout L = gx_layout(RS, E, K);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* hdr = reinterpret_cast<int32_t*>(ws);
  int32_t* sorted = reinterpret_cast<int32_t*>(ws + L.sorted);
  __nv_bfloat16* xg = reinterpret_cast<__nv_bfloat16*>(ws + L.xg);
  CUtensorMap xmap, wmap;
  if (!encode_tensor_map_2d(&xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, xg, (uint64_t)K, (uint64_t)RS,
                            (uint64_t)K * 2, kGxBK, kGxBM / 2, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tensor_map_2d(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, const_cast<uint8_t*>(blocks),
                            (uint64_t)K / 2, (uint64_t)(E * N), (uint64_t)K / 2, kGxBK / 2, kGxBN,
                            CU_TENSOR_MAP_SWIZZLE_32B))
    return cudaErrorInvalidValue;
  const size_t smem = 1024 + (size_t)kGxStages * kGxStageBytes + sizeof(SharedGx);
  static_assert(1024 + (size_t)kGxStages * kGxStageBytes + sizeof(SharedGx) <= 227 * 1024,
                "GEMM stages exceed shared memory");
  static std::atomic<uint64_t> attr_set{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_set.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(k_gemm_mx_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set.fetch_or(bit, std::memory_order_release);
  }
  k_gx_route<<<1, 1024, 0, stream>>>(experts, (int)RS, (int)E, hdr, sorted, dev_status);
  const int64_t pieces = RS * (K / 8);
  const unsigned gblocks = (unsigned)std::min<int64_t>((pieces + 255) / 256, 4096);
  k_gx_gather<<<gblocks, 256, 0, stream>>>(x, K, S, x_per_slot, (int)E, hdr, sorted, xg);
  // tiles: at most RS / 256 + one more for every segment with rows
  const int64_t tiles_max = (RS + kGxBM - 1) / kGxBM + std::min<int64_t>(E + 1, RS);
  const dim3 grid((unsigned)tiles_max, (unsigned)((N + kGxBN - 1) / kGxBN));
  GxParams gp{hdr, sorted, scales, E, N, K, y, y32, sw, dev_status};
  note_launch("k_gemm_mx_tc<grouped by expert,tile=256x256> grid=%ux%u (k_gx_route, k_gx_gather first)",
              grid.x, grid.y);
  k_gemm_mx_tc<<<grid, kGxThreads, smem, stream>>>(xmap, wmap, gp);
  return cudaGetLastError();
}

}  // namespace wq
