// gemm_tc.cu -- prefill-regime (many activation rows) group-wise 4-bit linear on the
// fifth-generation tensor cores.
//
// y[m, n] = sum_k x[m, k] * W-hat[n, k], W-hat[n, k] = bf16(f32(q - zero) * scale)
// ("Quantization" (Linnet docs): linear_int4_groups over Int4GroupLinear; "20.
// Quantization" (Inference Engineering book), "Speed needs a kernel": at large batch
// the product becomes compute-bound and dequantization is extra work, so the weights
// are dequantized once per tile in shared memory and every dequantized weight feeds
// 256 activation rows).
//
// One thread block computes a 256 x 256 tile of y (rows of x by rows of W):
//   warp 0      TMA producer: the x tile (256 rows x 64 k, 128-byte swizzle) and the
//               packed weight tile (256 rows x 32 bytes, 32-byte swizzle) of each k step
//               into a 3-stage ring, completion on an mbarrier;
//   warp 1      allocates 512 TMEM columns (two 128 x 256 f32 accumulators) and one of
//               its threads issues tcgen05.mma kind::f16 (bf16 x bf16 -> f32): 2 x 4
//               MMAs of 128 x 256 x 16 a k step, then tcgen05.commit frees the stage;
//   warps 2..9  dequantize: thread t owns weight row t, turns its 32 packed bytes into
//               64 bf16 values exactly (dequant_nib8) and stores them in the canonical
//               K-major 128-byte-swizzled layout the MMA reads; after the last k step
//               they read the accumulators back (tcgen05.ld), add the bias, round to
//               bf16 and store y.
// Shapes with fewer tiles than half the SMs are split along K (blockIdx.z): each block
// stores its tile's f32 partial sums, and a second kernel adds the partials in split
// order (deterministic), adds the bias and rounds to bf16.
// Every wait is bounded; a timeout records WQ_DEV_TIMEOUT and the block winds down
// after the MMAs it issued have completed, freeing its TMEM.
#include <algorithm>
#include <atomic>
#include <cstdlib>

#include "common.cuh"
#include "launch.h"
#include "tc.cuh"

namespace wq {

namespace {

constexpr int kBK = 64;   // k a stage: one 128-byte swizzle row of bf16
constexpr int kDequantWarps = 8;
constexpr int kThreadsTc = (2 + kDequantWarps) * 32;
constexpr size_t kSmemTcMax = 227 * 1024;

// Tile geometry: kTile x kTile outputs (activation rows x weight rows), kTile / 128
// accumulators of 128 rows in TMEM; stages as many as fit in shared memory (at most 6).
template <int kTile>
struct TileCfg {
  static constexpr int kAcc = kTile / 128;
  static constexpr int kABytes = kTile * kBK * 2;  // activation tile (bf16)
  static constexpr int kBBytes = kTile * kBK * 2;  // dequantized weight tile (bf16)
  static constexpr int kPBytes = kTile * kBK / 2;  // packed codes
  static constexpr int kStageBytes = kABytes + kBBytes + kPBytes;
  static constexpr int kStages = kTile == 256 ? 3 : 6;
  static constexpr uint32_t kTmemCols = (uint32_t)(kAcc * kTile);
};

struct SharedTc {
  uint64_t full_tma[6];  // x + packed landed
  uint64_t full_b[6];    // dequantized weights written
  uint64_t empty[6];     // MMAs of the stage done
  uint64_t acc_full;     // all MMAs done
  uint32_t tmem_base;
  int abort;
};

}  // namespace

// kTile = 256: two 128 x 256 accumulators, each dequantized weight feeding 256 activation
// rows (the large layers).  kTile = 128: one 128 x 128 accumulator and four times the
// tiles, for layers with fewer 256 x 256 tiles than SMs (k and v at M = 2048), which
// would otherwise split K and send f32 partials through HBM; the 256 dequantizing
// threads then take half a weight row each.
template <bool kSplit, int kTile>
__global__ void __launch_bounds__(kThreadsTc, 1)
    k_gemm_w4g_tc(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap pmap,
                  const GemmTcParams p) {
  using C = TileCfg<kTile>;
  constexpr int kStagesTc = C::kStages;
  constexpr int kABytes = C::kABytes, kBBytes = C::kBBytes, kPBytes = C::kPBytes;
  constexpr int kStageTcBytes = C::kStageBytes;
  constexpr int kBM = kTile, kBN = kTile;
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) &
                                             ~uintptr_t(1023));
  SharedTc* sh = reinterpret_cast<SharedTc*>(smem + kStagesTc * kStageTcBytes);
  auto stage_a = [&](int s) { return smem + s * kStageTcBytes; };
  auto stage_b = [&](int s) { return smem + s * kStageTcBytes + kABytes; };
  auto stage_p = [&](int s) { return smem + s * kStageTcBytes + kABytes + kBBytes; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t M = p.M, N = p.N, K = p.K;
  const int64_t m0 = (int64_t)blockIdx.x * kBM;
  const int64_t n0 = (int64_t)blockIdx.y * kBN;
  // this block's k steps: range blockIdx.z of gridDim.z equal ranges
  const int nk_all = (int)((K + kBK - 1) / kBK);
  const int kb0 = (int)(((int64_t)blockIdx.z * nk_all) / gridDim.z);
  const int nk = (int)(((int64_t)(blockIdx.z + 1) * nk_all) / gridDim.z) - kb0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesTc; ++s) {
      mbar_init(&sh->full_tma[s], 1);
      mbar_init(&sh->full_b[s], kDequantWarps);
      mbar_init(&sh->empty[s], 1);
    }
    mbar_init(&sh->acc_full, 1);
    fence_mbar_init();
    sh->abort = 0;
  }
  if (warp == 1) tmem_alloc(&sh->tmem_base, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh->tmem_base;

  if (warp == 0) {
    // ================= TMA producer =================
    if (lane == 0) {
      tma_prefetch_desc(&xmap);
      tma_prefetch_desc(&pmap);
      const uint64_t pol = l2_policy_evict_last();  // x and W tiles are re-read by other blocks
      int issued = 0;
      for (int kb = 0; kb < nk; ++kb) {
        const int s = kb % kStagesTc;
        if (kb >= kStagesTc && !mbar_wait(&sh->empty[s], ((kb / kStagesTc) - 1) & 1)) {
          set_dev_status(p.dev_status, WQ_DEV_TIMEOUT);
          atomicExch(&sh->abort, 1);
          break;
        }
        if (*reinterpret_cast<volatile int*>(&sh->abort)) break;
        mbar_arrive_expect_tx(&sh->full_tma[s], kABytes + kPBytes);
        tma_load_2d(stage_a(s), &xmap, &sh->full_tma[s], (kb0 + kb) * kBK, (int32_t)m0, pol);
        tma_load_2d(stage_p(s), &pmap, &sh->full_tma[s], (kb0 + kb) * (kBK / 2), (int32_t)n0, pol);
        issued = kb + 1;
      }
      // no copy may land in shared memory after the block exits: wait (bounded) for the
      // last copy issued into each stage (long complete unless the block is aborting)
      for (int kb = std::max(0, issued - kStagesTc); kb < issued; ++kb)
        (void)mbar_wait(&sh->full_tma[kb % kStagesTc], (uint32_t)(kb / kStagesTc) & 1u);
    }
  } else if (warp == 1) {
    // ================= MMA issuer =================
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(128, kBN);
      for (int kb = 0; kb < nk; ++kb) {
        const int s = kb % kStagesTc;
        if (*reinterpret_cast<volatile int*>(&sh->abort)) break;
        // the x tile (TMA) and the dequantized weights (dequant warps) of this stage
        if (!mbar_wait(&sh->full_tma[s], (kb / kStagesTc) & 1) ||
            !mbar_wait(&sh->full_b[s], (kb / kStagesTc) & 1)) {
          set_dev_status(p.dev_status, WQ_DEV_TIMEOUT);
          atomicExch(&sh->abort, 1);
          break;
        }
        tc_fence_after();
        const uint32_t a_base = smem_u32(stage_a(s));
        const uint32_t b_base = smem_u32(stage_b(s));
#pragma unroll
        for (int acc = 0; acc < C::kAcc; ++acc) {
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            // +32 bytes a 16-element k slice inside the 128-byte swizzled rows
            const uint64_t ad = umma_desc_sw128(a_base + acc * (128 * 128) + kk * 32);
            const uint64_t bd = umma_desc_sw128(b_base + kk * 32);
            umma_bf16(tmem + acc * kBN, ad, bd, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
          }
        }
        umma_commit(&sh->empty[s]);  // the stage may be refilled once these MMAs finish
      }
      umma_commit(&sh->acc_full);
    }
  } else {
    // ================= dequantize (8 warps), then epilogue =================
    // kTile 256: thread t owns weight row t, all 64 codes of a stage; kTile 128: row
    // t % 128, codes 32 (t / 128) .. + 31
    const int tt = threadIdx.x - 64;
    const int t = (kTile == 256) ? tt : (tt & 127);
    const int half = (kTile == 256) ? 0 : (tt >> 7);
    const int64_t n = imin64(n0 + t, N - 1);
    const int gshift = __ffs(p.group) - 1;
    const uint32_t gpr = (uint32_t)(K >> gshift);  // groups a row (K < 2^31)
    const float* const srow = p.scale + n * (int64_t)gpr;
    const uint8_t* const zrow = p.zero + n * (int64_t)gpr;
    const bool two_groups = (p.group < kBK);  // group 32: two groups a k step

    // scales and zero points four groups at a time: one 16-byte and one 4-byte load a
    // thread when the row's groups are aligned (K / G a multiple of 4), the next four
    // groups prefetched a window ahead; the dequant constants change only with the group
    const bool vec_meta = (gpr % 4u == 0) && ((reinterpret_cast<uintptr_t>(p.scale) & 15) == 0) &&
                          ((reinterpret_cast<uintptr_t>(p.zero) & 3) == 0);
    struct Win {
      float4 s;
      uint32_t z;  // zero points of the four groups, one a byte
    };
    auto load_win = [&](uint32_t gb) -> Win {
      Win w{make_float4(1.0f, 1.0f, 1.0f, 1.0f), 0u};
      if (vec_meta) {
        if (gb < gpr) {
          w.s = __ldg(reinterpret_cast<const float4*>(srow + gb));
          w.z = __ldg(reinterpret_cast<const unsigned int*>(zrow + gb));
        }
      } else {
        float sv[4] = {1.0f, 1.0f, 1.0f, 1.0f};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (gb + i < gpr) {
            sv[i] = __ldg(srow + gb + i);
            w.z |= (uint32_t)__ldg(zrow + gb + i) << (8 * i);
          }
        }
        w.s = make_float4(sv[0], sv[1], sv[2], sv[3]);
      }
      return w;
    };
    auto pick = [](const float4& v, uint32_t i) {
      return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
    };
    uint32_t gb = (((uint32_t)kb0 * (uint32_t)kBK) >> gshift) & ~3u;
    Win cur = load_win(gb), nxt = load_win(gb + 4);
    uint32_t gk = 0xFFFFFFFFu;  // group of the constants below
    Nib8Consts k0{}, k1{};

    const uint32_t prow = (uint32_t)t * 32;  // packed row, 32-byte swizzle
    const uint32_t pswz = (uint32_t)((t >> 2) & 1);
    // this thread's 16-byte pieces of its dequantized row: piece w at w ^ (row mod 8)
    // (128-byte swizzle), offsets inside a stage
    uint32_t boff[8];
#pragma unroll
    for (int w = 0; w < 8; ++w) boff[w] = (uint32_t)t * 128 + (((uint32_t)w ^ (uint32_t)(t & 7)) << 4);
    const uint32_t pa0 = prow + (pswz << 4), pa1 = prow + ((1u ^ pswz) << 4);

    // one k step: the packed row from the stage, dequantized, into the MMA's layout
    auto dequant_step = [&](int s, const Nib8Consts& k0, const Nib8Consts& k1) {
      const uint32_t pbase = smem_u32(stage_p(s));
      const uint32_t bbase = smem_u32(stage_b(s));
      if constexpr (kTile == 256) {
        const uint4 c0 = ld_shared_v4(pbase + pa0);
        const uint4 c1 = ld_shared_v4(pbase + pa1);
        const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
        for (int w = 0; w < 8; ++w) {
          uint32_t o[4];
          dequant_nib8(words[w], (w < 4) ? k0 : k1, o);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(bbase + boff[w]), "r"(o[0]),
                       "r"(o[1]), "r"(o[2]), "r"(o[3])
                       : "memory");
        }
      } else {
        // codes 32 half .. 32 half + 31: the packed 16-byte unit `half` of the row
        const uint4 c = ld_shared_v4(pbase + (half ? pa1 : pa0));
        const uint32_t words[4] = {c.x, c.y, c.z, c.w};
        const Nib8Consts& kc = half ? k1 : k0;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          uint32_t o[4];
          dequant_nib8(words[w], kc, o);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(bbase + boff[4 * half + w]),
                       "r"(o[0]), "r"(o[1]), "r"(o[2]), "r"(o[3])
                       : "memory");
        }
      }
    };

    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % kStagesTc;
      // this step's group (a step of 64 codes lies in one group, or two of 32)
      const uint32_t g0 = ((uint32_t)(kb0 + kb) * (uint32_t)kBK) >> gshift;
      if ((g0 & ~3u) != gb) {  // warp-uniform: the next window of four groups
        gb += 4;
        cur = nxt;
        nxt = load_win(gb + 4);
      }
      if (g0 != gk) {
        gk = g0;
        const uint32_t i0 = g0 - gb;
        k0 = make_nib8_consts_u(pick(cur.s, i0), (cur.z >> (8 * i0)) & 0xFFu);
        k1 = two_groups ? make_nib8_consts_u(pick(cur.s, i0 + 1), (cur.z >> (8 * i0 + 8)) & 0xFFu) : k0;
      }
      if (*reinterpret_cast<volatile int*>(&sh->abort)) break;
      if (!mbar_wait(&sh->full_tma[s], (kb / kStagesTc) & 1)) {
        set_dev_status(p.dev_status, WQ_DEV_TIMEOUT);
        atomicExch(&sh->abort, 1);
        break;
      }
      dequant_step(s, k0, k1);
      fence_async_shared();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->full_b[s]);
    }

    // ---- epilogue: TMEM -> registers -> (+ bias) -> bf16 -> y ----
    if (!mbar_wait(&sh->acc_full, 0)) {
      set_dev_status(p.dev_status, WQ_DEV_TIMEOUT);
      atomicExch(&sh->abort, 1);
    }
    tc_fence_after();
    const int q = warp & 3;  // TMEM lane quarter this warp may read
    // kTile 256: accumulator (warp - 2) / 4, all 256 columns; kTile 128: the one
    // accumulator, columns 64 ((warp - 2) / 4) .. + 63
    const int acc = (kTile == 256) ? ((warp - 2) >> 2) : 0;
    const int col0 = (kTile == 256) ? 0 : ((warp - 2) >> 2) * 64;
    constexpr int kChunks = (kTile == 256) ? kBN / 32 : 2;
    const int64_t m = m0 + acc * 128 + q * 32 + lane;
    const bool vec_ok = (N % 8 == 0) && ((reinterpret_cast<uintptr_t>(p.y) & 15) == 0);
    constexpr bool split = kSplit;  // f32 partials to the workspace, no bias
#pragma unroll 1
    for (int ch = 0; ch < kChunks; ++ch) {
      uint32_t r[32];
      tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + acc * kBN + col0 + ch * 32, r);
      const int64_t nb = n0 + col0 + ch * 32;
      if (split && m < M && nb < N) {
        // f32 partial sums of this k range, no bias (the reduction adds it)
        float* dst = p.part + ((int64_t)blockIdx.z * M + m) * N + nb;
        if (N % 4 == 0 && nb + 32 <= N) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            *reinterpret_cast<float4*>(dst + 4 * i) =
                make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                            __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (nb + i < N) dst[i] = __uint_as_float(r[i]);
        }
      } else if (m < M && nb < N) {
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          v[i] = __uint_as_float(r[i]);
          if (p.bias && nb + i < N) v[i] += __bfloat162float(p.bias[nb + i]);
        }
        __nv_bfloat16* dst = p.y + m * N + nb;
        if (vec_ok && nb + 32 <= N) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint4 o;
            o.x = pack_bf16x2(v[8 * i + 0], v[8 * i + 1]);
            o.y = pack_bf16x2(v[8 * i + 2], v[8 * i + 3]);
            o.z = pack_bf16x2(v[8 * i + 4], v[8 * i + 5]);
            o.w = pack_bf16x2(v[8 * i + 6], v[8 * i + 7]);
            *reinterpret_cast<uint4*>(dst + 8 * i) = o;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (nb + i < N) dst[i] = __float2bfloat16_rn(v[i]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// y[m, n] = bf16(sum over splits z, in order, of part[z, m, n] + bias[n]).  The partials are
// zeroed as they are read: the workspace is left zero-filled, as every entry point of
// the library leaves it.  Grid: (column chunks of 4 x 256, rows); all splits' loads of a
// thread are issued before any of its stores.
constexpr int kMaxSplits = 8;

__global__ void __launch_bounds__(256) k_splitk_reduce(float* __restrict__ part, int splits,
                                                       int64_t M, int64_t N,
                                                       const __nv_bfloat16* __restrict__ bias,
                                                       __nv_bfloat16* __restrict__ y) {
  const int64_t m = blockIdx.y;
  const int64_t n = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (n >= N) return;
  const int64_t total = M * N;
  float* const row = part + m * N + n;
  float v[kMaxSplits][4];
  if (N % 4 == 0) {
#pragma unroll
    for (int z = 0; z < kMaxSplits; ++z) {
      if (z < splits) {
        const float4 u = __ldcg(reinterpret_cast<const float4*>(row + (int64_t)z * total));
        v[z][0] = u.x;
        v[z][1] = u.y;
        v[z][2] = u.z;
        v[z][3] = u.w;
      }
    }
#pragma unroll
    for (int z = 0; z < kMaxSplits; ++z)
      if (z < splits)
        __stcg(reinterpret_cast<float4*>(row + (int64_t)z * total), make_float4(0.f, 0.f, 0.f, 0.f));
  } else {
    // ragged rows: element by element (the last chunk may be short)
#pragma unroll
    for (int z = 0; z < kMaxSplits; ++z) {
      if (z < splits) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          v[z][j] = 0.0f;
          if (n + j < N) {
            v[z][j] = row[(int64_t)z * total + j];
            row[(int64_t)z * total + j] = 0.0f;
          }
        }
      }
    }
  }
  float acc[4] = {v[0][0], v[0][1], v[0][2], v[0][3]};
#pragma unroll
  for (int z = 1; z < kMaxSplits; ++z)
    if (z < splits)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[j] += v[z][j];
  __nv_bfloat16* const out = y + m * N + n;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if (n + j < N) {
      float o = acc[j];
      if (bias) o += __bfloat162float(bias[n + j]);
      out[j] = __float2bfloat16_rn(o);
    }
  }
}

// ------------------------------------------------------------------ host side
namespace {
// 256 x 256 tiles when they fill at least half the SMs; else 128 x 128 tiles (four times
// as many, no f32 partials through HBM), split along K only if even those are too few.
int gemm_tile(int64_t M, int64_t N, int num_sms) {
  const int64_t t256 = ((M + 255) / 256) * ((N + 255) / 256);
  return t256 * 2 > num_sms ? 256 : 128;
}
}  // namespace

int gemm_tc_splits(int64_t M, int64_t N, int64_t K, int num_sms) {
  const int tile = gemm_tile(M, N, num_sms);
  const int64_t tiles = ((M + tile - 1) / tile) * ((N + tile - 1) / tile);
  const int64_t nk = (K + kBK - 1) / kBK;
  if (tiles * 2 > num_sms) return 1;
  // as many k ranges as fill the SMs, each of at least 8 k steps, at most 8 ranges
  return (int)std::max<int64_t>(1, std::min<int64_t>({num_sms / tiles, nk / 8, (int64_t)kMaxSplits}));
}

size_t gemm_tc_ws_bytes(int64_t M, int64_t N, int64_t K, int num_sms) {
  const int s = gemm_tc_splits(M, N, K, num_sms);
  return s > 1 ? (size_t)s * (size_t)M * (size_t)N * 4 : 0;
}

bool gemm_tc_supported(int64_t M, int64_t N, int64_t K, int32_t group) {
  // The crossover, measured on GB300 on the 14336 x 4096 group-128 layer: the decode
  // kernel and this GEMM tie at M = 17 .. 32 (40 us either way), the GEMM is faster from
  // M = 48 on (45 us against 57 us); the default switches in between.
  const int64_t min_m = tuning(kKnobGemmMinM);  // tuning and test knob for the crossover
  if (M < (min_m >= 1 ? min_m : 40)) return false;
  return N >= 1 && K >= 32 && K % 32 == 0 && (group == 32 || group == 64 || group == 128 ||
                                               group == 256) &&
         K % group == 0 && M <= (int64_t(1) << 31) && N <= (int64_t(1) << 31);
}

namespace {
template <int kTile>
cudaError_t launch_gemm_tile(const GemmTcParams& p, int splits, cudaStream_t stream) {
  using C = TileCfg<kTile>;
  CUtensorMap xmap, pmap;
  if (!encode_tensor_map_2d(&xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                            const_cast<__nv_bfloat16*>(p.x), (uint64_t)p.K, (uint64_t)p.M,
                            (uint64_t)p.K * 2, kBK, kTile, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (!encode_tensor_map_2d(&pmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, const_cast<uint8_t*>(p.packed),
                            (uint64_t)p.K / 2, (uint64_t)p.N, (uint64_t)p.K / 2, kBK / 2, kTile,
                            CU_TENSOR_MAP_SWIZZLE_32B))
    return cudaErrorInvalidValue;
  const size_t smem = 1024 + (size_t)C::kStages * C::kStageBytes + sizeof(SharedTc);
  static_assert(1024 + (size_t)C::kStages * C::kStageBytes + sizeof(SharedTc) <= kSmemTcMax,
                "GEMM stages exceed shared memory");
  static std::atomic<uint64_t> attr_set{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_set.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(k_gemm_w4g_tc<false, kTile>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_gemm_w4g_tc<true, kTile>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    attr_set.fetch_or(bit, std::memory_order_release);
  }
  GemmTcParams q = p;
  if (splits == 1) q.part = nullptr;
  const dim3 grid((unsigned)((p.M + kTile - 1) / kTile), (unsigned)((p.N + kTile - 1) / kTile),
                  (unsigned)splits);
  note_launch("k_gemm_w4g_tc<%s,tile=%d> grid=%ux%ux%u%s", splits > 1 ? "split" : "unsplit", kTile, grid.x,
              grid.y, grid.z, splits > 1 ? " + k_splitk_reduce" : "");
  if (splits == 1)
    k_gemm_w4g_tc<false, kTile><<<grid, kThreadsTc, smem, stream>>>(xmap, pmap, q);
  else
    k_gemm_w4g_tc<true, kTile><<<grid, kThreadsTc, smem, stream>>>(xmap, pmap, q);
  e = cudaGetLastError();
  if (e != cudaSuccess || splits == 1) return e;
  // splits > 1 only with at most num_sms / 2 tiles, so M <= 256 * num_sms / 2 rows: within
  // the grid's y limit
  const dim3 rgrid((unsigned)((p.N + 1023) / 1024), (unsigned)p.M);
  k_splitk_reduce<<<rgrid, 256, 0, stream>>>(q.part, splits, p.M, p.N, p.bias, p.y);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_gemm_tc(const GemmTcParams& p, int num_sms, cudaStream_t stream) {
  const int splits = (p.part != nullptr) ? std::max(1, (int)p.splits) : 1;
  return gemm_tile(p.M, p.N, num_sms) == 256 ? launch_gemm_tile<256>(p, splits, stream)
                                             : launch_gemm_tile<128>(p, splits, stream);
}

}  // namespace wq
