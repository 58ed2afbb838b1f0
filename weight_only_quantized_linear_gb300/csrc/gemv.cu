// gemv.cu -- decode-regime (few activation rows) weight-only quantized linear.
//
// y[m, n] = sum_k x[m, k] * W-hat[n, k] with W-hat dequantized in registers from packed
// codes, for four storage formats:
//   I4G   group-wise asymmetric 4-bit ("Quantization" (Linnet docs): Int4GroupLinear,
//         dequantize_int4_groups "(q - zero) * scale per group")
//   I4R   per-row signed 4-bit (Int4Linear, dequantize_int4)
//   I8R   per-row int8 (Int8Linear, dequantize_int8 "q * scale in f32, cast to T")
//   MXFP4 E2M1 blocks of 32 with an E8M0 scale (dequantize_mxfp4), gathered per routed
//         expert (mxfp4_experts_shared)
//
// The regime is bound by HBM bandwidth ("Quantization: int8, int4 group (packed), fp8,
// KV quant", 1. Why now: decoding is limited by bytes moved).  Design on sm_103a:
//   * one thread block = a tile of 16 weight rows x a K range (split-K across blocks
//     when there are too few tiles to fill the 152 SMs);
//   * a producer warp streams the tile through a 4-stage shared-memory ring with TMA
//     (cp.async.bulk.tensor, 128-byte swizzle, evict-first L2 policy), each stage = 16
//     rows x 512 bytes, completion tracked by mbarriers;
//   * eight consumer warps each take one 64-byte column slice of every stage: a lane
//     reads 16 bytes of two rows, dequantizes them exactly (see dequant_nib8), and feeds
//     them as the A operand of mma.sync m16n8k16 with the activations as B;
//   * the k order inside an MMA is a permutation shared by A and B, so a lane's 16
//     contiguous bytes map straight onto its fragment slots (no shuffles);
//   * the eight warps' partial sums are added in shared memory in a fixed order, then
//     either written (bf16, + bias) or, under split-K, left as f32 partials that the
//     last-arriving block of the tile adds in split order (deterministic, wait-free).
#include <algorithm>
#include <atomic>
#include <cstdlib>

#include "common.cuh"
#include "launch.h"

namespace wq {

namespace {

constexpr int kRows = 16;              // weight rows per tile (one MMA M)
constexpr int kStageRowBytes = 512;    // bytes of a row per pipeline stage
constexpr int kBoxBytes = kRows * 128; // one TMA box: 16 rows x 128 bytes (swizzled)
constexpr int kStageBytes = kRows * kStageRowBytes;
constexpr int kStages = 4;
constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;

template <Fmt F>
struct FmtInfo {
  static constexpr int kPiece = (F == Fmt::I8R) ? 16 : 32;  // k per 16-byte lane piece
};
// 4-bit: 512 bytes a row = 1024 k a stage; int8: 512 k a stage.
template <Fmt F>
constexpr int stage_k() { return (F == Fmt::I8R) ? 512 : 1024; }

// Tile row held by MMA row g (0..7) and g + 8: rows differing by 4 share a shared-memory
// phase, which the 128-byte swizzle maps to disjoint banks.
__device__ __forceinline__ int tile_row_of(int g) { return ((g & 1) << 2) | (g >> 1); }

struct SharedTail {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  int xrow[16];
  int yrow[16];
  int nrows;
  int cursor;
  int abort;
  int last;
};

}  // namespace

template <Fmt F, int MT>
__global__ void __launch_bounds__(kThreads, 1)
    k_gemv(const __grid_constant__ CUtensorMap wmap, const GemvParams p) {
  constexpr int kPiece = FmtInfo<F>::kPiece;
  constexpr int kStageK = stage_k<F>();
  constexpr int kBatch = 8 * MT;

  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* stage_mem = smem;
  float* red = reinterpret_cast<float*>(smem + kStages * kStageBytes);  // [8][MT][16][8]
  SharedTail* sh = reinterpret_cast<SharedTail*>(red + kConsumerWarps * MT * 16 * 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tid = threadIdx.x;

  const int tile = blockIdx.x;
  const int split = blockIdx.y;
  const int expert = blockIdx.z;
  const int64_t N = p.N;
  const int64_t K = p.K;
  const int n0 = tile * kRows;
  const int64_t map_row0 = (F == Fmt::MXFP4 ? (int64_t)expert * N : 0) + n0;

  const int total_stages = (int)((K + kStageK - 1) / kStageK);
  const int st_begin = split * p.stages_per_split;
  const int st_end = min(total_stages, st_begin + p.stages_per_split);
  const int nst = st_end - st_begin;

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&sh->full[i], 1);
      mbar_init(&sh->empty[i], kConsumerWarps);
    }
    fence_mbar_init();
    sh->cursor = 0;
    sh->abort = 0;
  }
  if (warp == kConsumerWarps && lane == 0) tma_prefetch_desc(&wmap);
  __syncthreads();

  uint32_t it_base = 0;
  while (true) {
    // ---- next batch of activation rows (warp 0) ----
    if (warp == 0) {
      if constexpr (F != Fmt::MXFP4) {
        if (lane == 0) {
          const int start = sh->cursor;
          const int n = (int)imin64(kBatch, p.M - start);
          sh->nrows = n > 0 ? n : 0;
          for (int i = 0; i < kBatch; ++i) {
            sh->xrow[i] = start + i;
            sh->yrow[i] = start + i;
          }
          sh->cursor = start + sh->nrows;
        }
      } else {
        // rows routed to this expert, in (r, s) order, up to kBatch of them
        int cur = sh->cursor;
        int found = 0;
        const int64_t total = p.M * p.S;
        while (cur < total && found < kBatch) {
          const int idx = cur + lane;
          const bool hit = idx < total && p.experts[idx] == expert;
          const unsigned mask = __ballot_sync(0xffffffffu, hit);
          const int before = __popc(mask & ((1u << lane) - 1u));
          const int take = min(__popc(mask), kBatch - found);
          if (hit && before < take) {
            sh->xrow[found + before] = idx / (int)p.S;
            sh->yrow[found + before] = idx;
          }
          if (take < __popc(mask)) {
            // stop just after the last row taken
            int pos = 0, cnt = 0;
            for (int b = 0; b < 32; ++b)
              if ((mask >> b) & 1u) {
                if (++cnt == take) { pos = b; break; }
              }
            cur += pos + 1;
            found += take;
            break;
          }
          found += take;
          cur += 32;
        }
        if (lane == 0) {
          sh->nrows = found;
          sh->cursor = imin64(cur, total);
        }
      }
    }
    __syncthreads();
    const int nrows = sh->nrows;
    if (nrows == 0 || sh->abort) break;

    if (warp == kConsumerWarps) {
      // ================= producer =================
      if (lane == 0) {
        const uint64_t pol = l2_policy_evict_first();
        for (int t = 0; t < nst; ++t) {
          const uint32_t it = it_base + t;
          const int slot = it % kStages;
          if (*reinterpret_cast<volatile int*>(&sh->abort)) break;
          if (it >= (uint32_t)kStages) {
            if (!mbar_wait(&sh->empty[slot], ((it / kStages) - 1) & 1)) {
              set_dev_status(p.dev_status, WQ_DEV_TIMEOUT);
              atomicExch(&sh->abort, 1);
              break;
            }
          }
          mbar_arrive_expect_tx(&sh->full[slot], kStageBytes);
          uint8_t* dst = stage_mem + slot * kStageBytes;
          const int st = st_begin + t;
#pragma unroll
          for (int b = 0; b < 4; ++b)
            tma_load_2d(dst + b * kBoxBytes, &wmap, &sh->full[slot],
                        st * kStageRowBytes + b * 128, (int32_t)map_row0, pol);
        }
      }
    } else {
      // ================= consumers =================
      const int g = lane >> 2;
      const int c = lane & 3;
      const int r0 = tile_row_of(g);  // tile rows r0 and r0 + 8
      const int64_t nA = imin64(n0 + r0, N - 1);
      const int64_t nB = imin64(n0 + r0 + 8, N - 1);
      const int box = warp >> 1;
      const int piece = ((warp & 1) << 2) | c;
      const uint32_t offA = box * kBoxBytes + r0 * 128 + ((piece ^ (r0 & 7)) << 4);
      const uint32_t offB = offA + 8 * 128;
      const uint32_t stage_base = smem_u32(stage_mem);

      // x row pointers of this lane for each MMA column block
      const __nv_bfloat16* xp[MT];
#pragma unroll
      for (int t = 0; t < MT; ++t) {
        const int m = t * 8 + g;
        xp[t] = (m < nrows) ? p.x + (int64_t)sh->xrow[m] * K : nullptr;
      }

      // per-row constants of the row formats
      Nib8Consts rowA, rowB;
      float2 i8c, i8sA, i8sB;
      if constexpr (F == Fmt::I4R) {
        rowA = make_nib8_consts(p.scale[nA], 8.0f);
        rowB = make_nib8_consts(p.scale[nB], 8.0f);
      }
      if constexpr (F == Fmt::I8R) {
        i8c = make_float2(-8388736.0f, -8388736.0f);  // -(2^23 + 128)
        i8sA = make_float2(p.scale[nA], p.scale[nA]);
        i8sB = make_float2(p.scale[nB], p.scale[nB]);
      }

      float acc[MT][4];
#pragma unroll
      for (int t = 0; t < MT; ++t)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[t][i] = 0.0f;

      for (int t = 0; t < nst; ++t) {
        const uint32_t it = it_base + t;
        const int slot = it % kStages;
        const int64_t kp = (int64_t)(st_begin + t) * kStageK + (warp * 4 + c) * kPiece;
        const bool valid = kp < K;

        // activations first (independent of the stage)
        uint32_t xw[MT][kPiece / 2];
#pragma unroll
        for (int tt = 0; tt < MT; ++tt) {
#pragma unroll
          for (int q = 0; q < kPiece / 8; ++q) {
            uint4 v = make_uint4(0, 0, 0, 0);
            if (xp[tt] != nullptr && valid) v = ld_global_nc_v4(xp[tt] + kp + q * 8);
            xw[tt][4 * q + 0] = v.x;
            xw[tt][4 * q + 1] = v.y;
            xw[tt][4 * q + 2] = v.z;
            xw[tt][4 * q + 3] = v.w;
          }
        }
        // dequantization parameters of this piece
        Nib8Consts kA, kB;
        float2 XA, XB;
        if constexpr (F == Fmt::I4G) {
          const int64_t gpr = K / p.group;
          const int64_t gi = valid ? kp / p.group : 0;
          kA = make_nib8_consts(p.scale[nA * gpr + gi], (float)p.zero[nA * gpr + gi]);
          kB = make_nib8_consts(p.scale[nB * gpr + gi], (float)p.zero[nB * gpr + gi]);
        }
        if constexpr (F == Fmt::MXFP4) {
          const int64_t bpr = K / 32;
          const int64_t bi = valid ? kp / 32 : 0;
          const float xa = e8m0_to_f32(p.escale[((int64_t)expert * N + nA) * bpr + bi]);
          const float xb = e8m0_to_f32(p.escale[((int64_t)expert * N + nB) * bpr + bi]);
          XA = make_float2(xa, xa);
          XB = make_float2(xb, xb);
        }

        if (!mbar_wait(&sh->full[slot], (it / kStages) & 1)) {
          set_dev_status(p.dev_status, WQ_DEV_TIMEOUT);
          atomicExch(&sh->abort, 1);
          break;
        }
        uint4 wa = ld_shared_v4(stage_base + slot * kStageBytes + offA);
        uint4 wb = ld_shared_v4(stage_base + slot * kStageBytes + offB);
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->empty[slot]);
        if (!valid) {
          wa = make_uint4(0, 0, 0, 0);
          wb = make_uint4(0, 0, 0, 0);
        }
        const uint32_t wA[4] = {wa.x, wa.y, wa.z, wa.w};
        const uint32_t wB[4] = {wb.x, wb.y, wb.z, wb.w};

        if constexpr (F == Fmt::I8R) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint32_t ga[2], gb[2];
            dequant_i8x4(wA[i], i8c, i8sA, ga);
            dequant_i8x4(wB[i], i8c, i8sB, gb);
            if (!valid) ga[0] = ga[1] = gb[0] = gb[1] = 0u;
#pragma unroll
            for (int tt = 0; tt < MT; ++tt)
              mma_bf16_16816(acc[tt], ga[0], gb[0], ga[1], gb[1], xw[tt][2 * i],
                             xw[tt][2 * i + 1]);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint32_t ga[4], gb[4];
            if constexpr (F == Fmt::I4G) {
              dequant_nib8(wA[i], kA, ga);
              dequant_nib8(wB[i], kB, gb);
            } else if constexpr (F == Fmt::I4R) {
              dequant_nib8(wA[i] ^ 0x88888888u, rowA, ga);
              dequant_nib8(wB[i] ^ 0x88888888u, rowB, gb);
            } else {
              dequant_e2m1x8(wA[i], XA, ga);
              dequant_e2m1x8(wB[i], XB, gb);
            }
            if (!valid) {
#pragma unroll
              for (int q = 0; q < 4; ++q) ga[q] = gb[q] = 0u;
            }
#pragma unroll
            for (int tt = 0; tt < MT; ++tt) {
              mma_bf16_16816(acc[tt], ga[0], gb[0], ga[1], gb[1], xw[tt][4 * i],
                             xw[tt][4 * i + 1]);
              mma_bf16_16816(acc[tt], ga[2], gb[2], ga[3], gb[3], xw[tt][4 * i + 2],
                             xw[tt][4 * i + 3]);
            }
          }
        }
      }

      // ---- reduce the eight warps' partial sums ----
#pragma unroll
      for (int tt = 0; tt < MT; ++tt) {
        float* rb = red + ((warp * MT + tt) * 16) * 8;
        rb[g * 8 + 2 * c] = acc[tt][0];
        rb[g * 8 + 2 * c + 1] = acc[tt][1];
        rb[(g + 8) * 8 + 2 * c] = acc[tt][2];
        rb[(g + 8) * 8 + 2 * c + 1] = acc[tt][3];
      }
    }
    it_base += nst;
    __syncthreads();
    if (sh->abort) break;

    // thread -> (column block, MMA row, column); 256 consumer threads cover MT*128
    float sum = 0.0f;
    int out_m = -1;
    int64_t out_n = -1;
    if (tid < MT * 128) {
      const int tt = tid >> 7;
      const int row = (tid >> 3) & 15;
      const int col = tid & 7;
      for (int w = 0; w < kConsumerWarps; ++w) sum += red[((w * MT + tt) * 16 + row) * 8 + col];
      const int m = tt * 8 + col;
      const int trow = (row < 8) ? tile_row_of(row) : tile_row_of(row - 8) + 8;
      const int64_t n = n0 + trow;
      if (m < nrows && n < N) {
        out_m = m;
        out_n = n;
      }
    }
    if (p.ksplit == 1) {
      if (out_m >= 0) {
        float v = sum;
        if (p.bias) v += __bfloat162float(p.bias[out_n]);
        p.y[(int64_t)sh->yrow[out_m] * N + out_n] = __float2bfloat16_rn(v);
      }
    } else {
      const int64_t rows_total = p.M;  // split-K is only used with a single batch
      if (out_m >= 0)
        p.ws_part[((int64_t)split * rows_total + sh->yrow[out_m]) * N + out_n] = sum;
      __threadfence();
      __syncthreads();
      if (tid == 0) {
        const uint32_t prev = atomicAdd(&p.ws_cnt[tile], 1u);
        sh->last = (prev == (uint32_t)(p.ksplit - 1));
      }
      __syncthreads();
      if (sh->last) {
        __threadfence();
        if (out_m >= 0) {
          float v = 0.0f;
          for (int s = 0; s < p.ksplit; ++s)
            v += __ldcg(&p.ws_part[((int64_t)s * rows_total + sh->yrow[out_m]) * N + out_n]);
          if (p.bias) v += __bfloat162float(p.bias[out_n]);
          p.y[(int64_t)sh->yrow[out_m] * N + out_n] = __float2bfloat16_rn(v);
        }
        if (tid == 0) p.ws_cnt[tile] = 0u;
      }
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------ host side
namespace {

int tile_count(int64_t N) { return (int)((N + kRows - 1) / kRows); }

size_t smem_bytes(int MT) {
  return 1024 + (size_t)kStages * kStageBytes + (size_t)kConsumerWarps * MT * 16 * 8 * 4 +
         sizeof(SharedTail);
}

template <Fmt F, int MT>
cudaError_t launch_t(const CUtensorMap& map, const GemvParams& p, dim3 grid,
                     cudaStream_t stream) {
  auto kern = k_gemv<F, MT>;
  const size_t smem = smem_bytes(MT);
  static std::atomic<uint64_t> attr_set{0};  // one bit per device ordinal
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_set.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set.fetch_or(bit, std::memory_order_release);
  }
  kern<<<grid, kThreads, smem, stream>>>(map, p);
  return cudaGetLastError();
}

}  // namespace

GemvPlan plan_gemv(Fmt f, int64_t M, int64_t N, int64_t K, int num_sms) {
  GemvPlan pl;
  const int sk = (f == Fmt::I8R) ? 512 : 1024;
  const int total_stages = (int)((K + sk - 1) / sk);
  const int tiles = tile_count(N);
  int ksplit = 1;
  if (f != Fmt::MXFP4 && M <= 16) {
    const int target = 2 * num_sms;
    if (tiles < target) ksplit = std::min(total_stages, (target + tiles - 1) / tiles);
    if (const char* env = std::getenv("WQ_GEMV_KSPLIT")) {
      const int v = std::atoi(env);
      if (v >= 1) ksplit = std::min(total_stages, v);
    }
  }
  const int sps = (total_stages + ksplit - 1) / ksplit;
  ksplit = (total_stages + sps - 1) / sps;  // no empty splits
  pl.ksplit = ksplit;
  pl.stages_per_split = sps;
  pl.tiles = tiles;
  pl.ws_bytes = ksplit > 1 ? ws_counter_bytes(tiles) + (size_t)ksplit * M * N * 4 : 0;
  return pl;
}

cudaError_t launch_gemv(Fmt f, const CUtensorMap& map, GemvParams p, const GemvPlan& pl,
                        int64_t experts_grid, cudaStream_t stream) {
  p.ksplit = pl.ksplit;
  p.stages_per_split = pl.stages_per_split;
  const dim3 grid(pl.tiles, pl.ksplit, (unsigned)experts_grid);
  const bool wide = (f == Fmt::MXFP4) ? true : (p.M > 8);
  switch (f) {
    case Fmt::I4G:
      return wide ? launch_t<Fmt::I4G, 2>(map, p, grid, stream)
                  : launch_t<Fmt::I4G, 1>(map, p, grid, stream);
    case Fmt::I4R:
      return wide ? launch_t<Fmt::I4R, 2>(map, p, grid, stream)
                  : launch_t<Fmt::I4R, 1>(map, p, grid, stream);
    case Fmt::I8R:
      return wide ? launch_t<Fmt::I8R, 2>(map, p, grid, stream)
                  : launch_t<Fmt::I8R, 1>(map, p, grid, stream);
    case Fmt::MXFP4:
      return p.M * p.S > 8 ? launch_t<Fmt::MXFP4, 2>(map, p, grid, stream)
                           : launch_t<Fmt::MXFP4, 1>(map, p, grid, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace wq
