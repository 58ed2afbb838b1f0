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
//   * persistent: one thread block per SM walks a contiguous range of the flattened
//     (16-row tile x pipeline stage) work.  With a workspace the ranges are equal to
//     within one stage (stream-K); a tile cut by a range boundary is finished by the
//     block that contributes last, which adds the partials in block order
//     (deterministic, and no block ever waits for another);
//   * a producer warp streams 16 rows x 512 bytes a stage through an 8-deep shared-
//     memory ring with TMA (cp.async.bulk.tensor, 128-byte swizzle, evict-first), never
//     draining between tiles; completion is tracked by mbarriers (bounded waits);
//   * eight consumer warps each take one 64-byte column slice of every stage: a lane
//     reads 16 bytes of two rows, dequantizes them exactly (see dequant_nib8), and feeds
//     them as the A operand of mma.sync m16n8k16 with the activations as B.  The k order
//     inside an MMA is a permutation shared by A and B, so a lane's 16 contiguous bytes
//     map straight onto its fragment slots;
//   * scales and zero points are fetched into registers kPrefetch stages ahead and the
//     activations one stage ahead, so no global-memory latency sits on the critical path;
//   * the warps' partial sums are added in shared memory in a fixed order.
#include <algorithm>
#include <atomic>
#include <cstdlib>

#include "common.cuh"
#include "launch.h"

namespace wq {

namespace {

constexpr int kRows = 16;               // weight rows per tile (one MMA M)
constexpr int kStageRowBytes = 512;     // bytes of a row per pipeline stage
constexpr int kBoxBytes = kRows * 128;  // one TMA box: 16 rows x 128 bytes (swizzled)
constexpr int kStageBytes = kRows * kStageRowBytes;
constexpr int kStages = 8;
constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;  // + producer warp
constexpr int kPrefetch = 4;               // stages of scales / zeros fetched ahead
static_assert((kStages & (kStages - 1)) == 0, "ring depth must be a power of two");
constexpr int kMaxSlots = 4096;            // MXFP4: rows x slots handled by one launch
constexpr int kMaxExperts = 1024;
constexpr int kMaxPairs = kMaxExperts + kMaxSlots / 8;

template <Fmt F>
constexpr int piece_k() { return (F == Fmt::I8R) ? 16 : 32; }  // k per 16-byte lane piece
template <Fmt F>
constexpr int stage_k() { return (F == Fmt::I8R) ? 512 : 1024; }

// Tile row held by MMA row g (0..7) and g + 8: rows differing by 4 share a shared-memory
// phase, which the 128-byte swizzle maps to disjoint banks.
__device__ __forceinline__ int tile_row_of(int g) { return ((g & 1) << 2) | (g >> 1); }

struct Shared {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  int abort;
  int last[2];
  int npairs;
  // MXFP4 routing tables (identical in every block): slots sorted by expert, and
  // (expert, first sorted slot, count) for each batch of at most 8*MT slots.
  int pair_expert[kMaxPairs];
  int pair_start[kMaxPairs];
  int pair_count[kMaxPairs];
  int sorted[kMaxSlots];
  int ecount[kMaxExperts + 1];
};

// First flattened stage of block c: equal shares (stream-K) or whole items.
__device__ __forceinline__ int64_t block_begin(int64_t c, int64_t G, int64_t items, int spt,
                                               bool whole_items) {
  return whole_items ? (c * items / G) * spt : c * (items * spt) / G;
}

// The block whose range holds flattened stage s (stream-K split: c * W / G).
__device__ __forceinline__ int64_t owner_of(int64_t s, int64_t G, int64_t W) {
  int64_t cc = s * G / W;
  while (cc + 1 < G && (cc + 1) * W / G <= s) ++cc;
  while (cc > 0 && cc * W / G > s) --cc;
  return cc;
}

}  // namespace

template <Fmt F, int MT>
__global__ void __launch_bounds__(kThreads, 1)
    k_gemv(const __grid_constant__ CUtensorMap wmap, const GemvParams p) {
  constexpr int kPiece = piece_k<F>();
  constexpr int kStageK = stage_k<F>();
  constexpr int kBatch = 8 * MT;
  constexpr int kRedBuf = kConsumerWarps * MT * 16 * 8;

  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* ring = smem;
  float* red = reinterpret_cast<float*>(smem + kStages * kStageBytes);  // [2][8][MT][16][8]
  Shared* sh = reinterpret_cast<Shared*>(red + 2 * kRedBuf);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tid = threadIdx.x;
  const int64_t N = p.N;
  const int64_t K = p.K;
  const int tiles = (int)((N + kRows - 1) / kRows);
  const int spt = (int)((K + kStageK - 1) / kStageK);

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&sh->full[i], 1);
      mbar_init(&sh->empty[i], kConsumerWarps);
    }
    fence_mbar_init();
    sh->abort = 0;
  }

  // ---- work items: (tile, activation batch) or (tile, routed-expert batch) ----
  int64_t items;
  if constexpr (F == Fmt::MXFP4) {
    // stable counting sort of the R*S slots by expert, then batches of kBatch slots
    const int E = (int)p.E;
    const int slots = (int)(p.M * p.S);
    for (int e = tid; e <= E; e += kThreads) sh->ecount[e] = 0;
    __syncthreads();
    for (int i = tid; i < slots; i += kThreads) {
      const int e = p.experts[i];
      if (e >= 0 && e < E) atomicAdd(&sh->ecount[e], 1);
    }
    __syncthreads();
    if (tid == 0) {
      int run = 0, np = 0;
      for (int e = 0; e < E; ++e) {
        const int cnt = sh->ecount[e];
        sh->ecount[e] = run;
        for (int b = 0; b < cnt; b += kBatch) {
          sh->pair_expert[np] = e;
          sh->pair_start[np] = run + b;
          sh->pair_count[np] = min(kBatch, cnt - b);
          ++np;
        }
        run += cnt;
      }
      sh->npairs = np;
      for (int i = 0; i < slots; ++i) {  // ascending slot order within an expert
        const int e = p.experts[i];
        if (e >= 0 && e < E) sh->sorted[sh->ecount[e]++] = i;
      }
    }
    __syncthreads();
    items = (int64_t)sh->npairs * tiles;
  } else {
    const int nb = (int)((p.M + kBatch - 1) / kBatch);
    items = (int64_t)tiles * nb;
  }
  if (warp == kConsumerWarps && lane == 0) tma_prefetch_desc(&wmap);
  __syncthreads();

  const bool stream_k = (p.ws_cnt != nullptr);  // partial tiles allowed (one batch only)
  const int64_t G = gridDim.x;
  const int64_t c = blockIdx.x;
  const int64_t beg = block_begin(c, G, items, spt, !stream_k);
  const int64_t end = block_begin(c + 1, G, items, spt, !stream_k);
  if (beg >= end) return;

  auto item_tile = [&](int64_t item) -> int { return (int)(item % tiles); };
  auto item_group = [&](int64_t item) -> int { return (int)(item / tiles); };

  if (warp == kConsumerWarps) {
    // ================= producer =================
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      for (int64_t g = beg; g < end; ++g) {
        const uint32_t u = (uint32_t)(g - beg);
        const int slot = u % kStages;
        if (*reinterpret_cast<volatile int*>(&sh->abort)) break;
        if (u >= (uint32_t)kStages) {
          if (!mbar_wait(&sh->empty[slot], ((u / kStages) - 1) & 1)) {
            set_dev_status(p.dev_status, WQ_DEV_TIMEOUT);
            atomicExch(&sh->abort, 1);
            break;
          }
        }
        const int64_t item = g / spt;
        const int st = (int)(g % spt);
        int64_t row0 = (int64_t)item_tile(item) * kRows;
        if constexpr (F == Fmt::MXFP4) row0 += (int64_t)sh->pair_expert[item_group(item)] * N;
        mbar_arrive_expect_tx(&sh->full[slot], kStageBytes);
        uint8_t* dst = ring + slot * kStageBytes;
#pragma unroll
        for (int b = 0; b < 4; ++b)
          tma_load_2d(dst + b * kBoxBytes, &wmap, &sh->full[slot], st * kStageRowBytes + b * 128,
                      (int32_t)row0, pol);
      }
    }
    return;  // the producer takes no part in the reductions
  }

  // ================= consumers =================
  const int g8 = lane >> 2;
  const int cq = lane & 3;
  const int r0 = tile_row_of(g8);  // tile rows r0 and r0 + 8
  const int box = warp >> 1;
  const int piece = ((warp & 1) << 2) | cq;
  const uint32_t offA = box * kBoxBytes + r0 * 128 + ((piece ^ (r0 & 7)) << 4);
  const uint32_t offB = offA + 8 * 128;
  const uint32_t ring_base = smem_u32(ring);
  const int lane_k = (warp * 4 + cq) * kPiece;  // k offset of this lane inside a stage
  const int gshift = p.group_shift;             // I4G: log2(group)
  const int64_t gpr = (F == Fmt::I4G) ? (K >> gshift) : (K >> 5);  // scales a row

  // what this lane needs of an item: its two weight rows, and the expert's row offset
  struct Rows {
    const float* sA;    // scales of the two rows (row start)
    const float* sB;
    const uint8_t* zA;  // zero points, or E8M0 block scales (MXFP4), of the two rows
    const uint8_t* zB;
    int tile, grp;
  };
  auto rows_of = [&](int item) -> Rows {
    Rows r;
    r.tile = item % tiles;
    r.grp = item / tiles;
    const int64_t n0 = (int64_t)r.tile * kRows;
    const int64_t nA = imin64(n0 + r0, N - 1);
    const int64_t nB = imin64(n0 + r0 + 8, N - 1);
    if constexpr (F == Fmt::I4G) {
      r.sA = p.scale + nA * gpr;
      r.sB = p.scale + nB * gpr;
      r.zA = p.zero + nA * gpr;
      r.zB = p.zero + nB * gpr;
    } else if constexpr (F == Fmt::MXFP4) {
      const int64_t erow = (int64_t)sh->pair_expert[r.grp] * N;
      r.sA = r.sB = nullptr;
      r.zA = p.escale + (erow + nA) * gpr;
      r.zB = p.escale + (erow + nB) * gpr;
    } else {
      r.sA = p.scale + nA;
      r.sB = p.scale + nB;
      r.zA = r.zB = nullptr;
    }
    return r;
  };

  // scales / zero points (or E8M0 block scales) of this lane's piece
  struct Meta {
    float a, b;
    uint32_t z;
  };
  // A piece past the end of K gets scale 0 (and zero point 0 / block scale 0), so its
  // dequantized weights are exact zeros whatever bytes the zero-filled tile holds.
  auto load_meta = [&](const Rows& r, int st) -> Meta {
    Meta m{0.0f, 0.0f, 0u};
    const int kp = st * kStageK + lane_k;
    if (kp >= K) return m;
    if constexpr (F == Fmt::I4G) {
      const int gi = kp >> gshift;
      m.a = __ldg(r.sA + gi);
      m.b = __ldg(r.sB + gi);
      m.z = (uint32_t)__ldg(r.zA + gi) | ((uint32_t)__ldg(r.zB + gi) << 8);
    } else if constexpr (F == Fmt::MXFP4) {
      const int bi = kp >> 5;
      m.z = (uint32_t)__ldg(r.zA + bi) | ((uint32_t)__ldg(r.zB + bi) << 8) | 0x10000u;
    } else {
      m.a = __ldg(r.sA);
      m.b = __ldg(r.sB);
    }
    return m;
  };

  // activation row of MMA column m of an item (-1: none) and its output row
  auto xrow_of = [&](const Rows& r, int m, int* yrow) -> int {
    if constexpr (F == Fmt::MXFP4) {
      if (m >= sh->pair_count[r.grp]) return -1;
      const int slot = sh->sorted[sh->pair_start[r.grp] + m];
      *yrow = slot;
      return slot / (int)p.S;
    } else {
      const int64_t row = (int64_t)r.grp * kBatch + m;
      if (row >= p.M) return -1;
      *yrow = (int)row;
      return (int)row;
    }
  };

  // four independent accumulator sets per column block break the MMA dependency chain
  float acc[MT][4][4];
#pragma unroll
  for (int t = 0; t < MT; ++t)
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[t][a][i] = 0.0f;

  // main cursor: (item, stage) of flattened stage beg + u
  int item = (int)(beg / spt), st = (int)(beg % spt);
  Rows cr = rows_of(item);
  const __nv_bfloat16* xptr[MT];
  auto set_xptr = [&]() {
#pragma unroll
    for (int tt = 0; tt < MT; ++tt) {
      int yr;
      const int xr = xrow_of(cr, tt * 8 + g8, &yr);
      xptr[tt] = (xr >= 0) ? p.x + (int64_t)xr * K : nullptr;
    }
  };
  set_xptr();

  // prefetch cursor: kPrefetch stages ahead of the main one
  int pitem = item, pst = st;
  int64_t pg = beg;
  Rows pr = cr;
  auto next_meta = [&]() -> Meta {
    Meta m{0.0f, 0.0f, 0u};
    if (pg < end) m = load_meta(pr, pst);
    ++pg;
    if (++pst == spt) {
      pst = 0;
      ++pitem;
      if (pg < end) pr = rows_of(pitem);
    }
    return m;
  };
  Meta mring[kPrefetch];
#pragma unroll
  for (int j = 0; j < kPrefetch; ++j) mring[j] = next_meta();

  bool seg_first = true;           // the segment holds this block's first stage
  bool seg_from_start = (st == 0); // the segment began at stage 0 of its item
  int pend_tile[2] = {-1, -1};     // tiles cut by this block's range boundaries
  int npend = 0;
  int seg_count = 0;               // reductions done (selects the double-buffered scratch)

  const int64_t total = end - beg;
  for (int64_t u = 0; u < total; ++u) {
    const Meta m = mring[0];
#pragma unroll
    for (int j = 0; j + 1 < kPrefetch; ++j) mring[j] = mring[j + 1];
    mring[kPrefetch - 1] = next_meta();

    const int64_t kp = (int64_t)st * kStageK + lane_k;
    const bool valid = kp < K;
    // activations of this lane's piece (L1-resident; consumed after the dequant below)
    uint32_t xw[MT][kPiece / 2];
#pragma unroll
    for (int tt = 0; tt < MT; ++tt) {
#pragma unroll
      for (int q = 0; q < kPiece / 8; ++q) {
        uint4 v = make_uint4(0, 0, 0, 0);
        if (xptr[tt] != nullptr && valid) v = ld_global_nc_v4(xptr[tt] + kp + q * 8);
        xw[tt][4 * q + 0] = v.x;
        xw[tt][4 * q + 1] = v.y;
        xw[tt][4 * q + 2] = v.z;
        xw[tt][4 * q + 3] = v.w;
      }
    }
    const int slot = (int)(u & (kStages - 1));
    const uint32_t parity = (uint32_t)((u / kStages) & 1);

    // dequantization constants (independent of the stage's bytes)
    Nib8Consts kA, kB;
    float2 sA, sB;
    if constexpr (F == Fmt::I4G) {
      kA = make_nib8_consts_u(m.a, m.z & 0xFFu);
      kB = make_nib8_consts_u(m.b, (m.z >> 8) & 0xFFu);
    } else if constexpr (F == Fmt::I4R) {
      kA = make_nib8_consts(m.a, 8.0f);
      kB = make_nib8_consts(m.b, 8.0f);
    } else if constexpr (F == Fmt::I8R) {
      sA = make_float2(m.a, m.a);
      sB = make_float2(m.b, m.b);
    } else {
      const bool ok = (m.z >> 16) != 0u;
      const float xa = ok ? e8m0_to_f32(m.z & 0xFFu) : 0.0f;
      const float xb = ok ? e8m0_to_f32((m.z >> 8) & 0xFFu) : 0.0f;
      sA = make_float2(xa, xa);
      sB = make_float2(xb, xb);
    }

    if (!*reinterpret_cast<volatile int*>(&sh->abort) && !mbar_wait(&sh->full[slot], parity)) {
      set_dev_status(p.dev_status, WQ_DEV_TIMEOUT);
      atomicExch(&sh->abort, 1);
    }
    uint4 wa = ld_shared_v4(ring_base + slot * kStageBytes + offA);
    uint4 wb = ld_shared_v4(ring_base + slot * kStageBytes + offB);
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh->empty[slot]);
    const uint32_t wA[4] = {wa.x, wa.y, wa.z, wa.w};
    const uint32_t wB[4] = {wb.x, wb.y, wb.z, wb.w};

    if constexpr (F == Fmt::I8R) {
      const float2 i8c = make_float2(-8388736.0f, -8388736.0f);  // -(2^23 + 128)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t ga[2], gb[2];
        dequant_i8x4(wA[i], i8c, sA, ga);
        dequant_i8x4(wB[i], i8c, sB, gb);
#pragma unroll
        for (int tt = 0; tt < MT; ++tt)
          mma_bf16_16816(acc[tt][i], ga[0], gb[0], ga[1], gb[1], xw[tt][2 * i], xw[tt][2 * i + 1]);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t ga[4], gb[4];
        if constexpr (F == Fmt::I4G) {
          dequant_nib8(wA[i], kA, ga);
          dequant_nib8(wB[i], kB, gb);
        } else if constexpr (F == Fmt::I4R) {
          dequant_nib8(wA[i] ^ 0x88888888u, kA, ga);
          dequant_nib8(wB[i] ^ 0x88888888u, kB, gb);
        } else {
          dequant_e2m1x8(wA[i], sA, ga);
          dequant_e2m1x8(wB[i], sB, gb);
        }
#pragma unroll
        for (int tt = 0; tt < MT; ++tt) {
          mma_bf16_16816(acc[tt][(2 * i) & 3], ga[0], gb[0], ga[1], gb[1], xw[tt][4 * i],
                         xw[tt][4 * i + 1]);
          mma_bf16_16816(acc[tt][(2 * i + 1) & 3], ga[2], gb[2], ga[3], gb[3], xw[tt][4 * i + 2],
                         xw[tt][4 * i + 3]);
        }
      }
    }

    // ---- end of a segment: the item ends here, or this block's range does ----
    const bool item_end = (st == spt - 1);
    if (item_end || u + 1 == total) {
      float* rb = red + (seg_count & 1) * kRedBuf;
#pragma unroll
      for (int tt = 0; tt < MT; ++tt) {
        float v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          v[i] = (acc[tt][0][i] + acc[tt][1][i]) + (acc[tt][2][i] + acc[tt][3][i]);
#pragma unroll
          for (int a = 0; a < 4; ++a) acc[tt][a][i] = 0.0f;
        }
        float* w = rb + ((warp * MT + tt) * 16) * 8;
        w[g8 * 8 + 2 * cq] = v[0];
        w[g8 * 8 + 2 * cq + 1] = v[1];
        w[(g8 + 8) * 8 + 2 * cq] = v[2];
        w[(g8 + 8) * 8 + 2 * cq + 1] = v[3];
      }
      asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
      const bool full_tile = seg_from_start && item_end;
      if (tid < MT * 128) {
        const int tt = tid >> 7, row = (tid >> 3) & 15, col = tid & 7;
        float sum = 0.0f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) sum += rb[((w * MT + tt) * 16 + row) * 8 + col];
        const int trow = (row < 8) ? tile_row_of(row) : tile_row_of(row - 8) + 8;
        if (full_tile) {
          const int64_t n = (int64_t)cr.tile * kRows + trow;
          int yr = -1;
          const int xr = xrow_of(cr, tt * 8 + col, &yr);
          if (xr >= 0 && n < N) {
            if (p.bias) sum += __bfloat162float(p.bias[n]);
            p.y[(int64_t)yr * N + n] = __float2bfloat16_rn(sum);
          }
        } else {
          // slot 0: the segment holding this block's first stage; slot 1: its last
          const int s = seg_first ? 0 : 1;
          p.ws_part[((c * 2 + s) * 16 + (tt * 8 + col)) * kRows + trow] = sum;
        }
      }
      if (!full_tile) pend_tile[npend++] = cr.tile;
      ++seg_count;
      seg_first = false;
      seg_from_start = true;
    }

    // ---- advance the main cursor ----
    if (++st == spt) {
      st = 0;
      ++item;
      if (u + 1 < total) {
        cr = rows_of(item);
        set_xptr();
      }
    }
  }

  // ---- finish the tiles cut by a block boundary (stream-K only) ----
  // Each contributing block adds one to the tile's counter after its partial is out;
  // the one that brings it to the number of contributors adds the partials in block
  // order, writes y and clears the counter.  Nobody waits on anybody.
  const int64_t W = (int64_t)tiles * spt;
  for (int i = 0; i < npend; ++i) {
    const int tile = pend_tile[i];
    __threadfence();
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
    const int64_t t_beg = (int64_t)tile * spt, t_end = t_beg + spt;
    const int64_t c0 = owner_of(t_beg, G, W), c1 = owner_of(t_end - 1, G, W);
    if (tid == 0) {
      const uint32_t prev = atomicAdd(&p.ws_cnt[tile], 1u);
      sh->last[i] = (prev == (uint32_t)(c1 - c0));
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
    if (sh->last[i]) {
      __threadfence();
      const int m = tid >> 4, row = tid & 15;
      float sum = 0.0f;
      for (int64_t cc = c0; cc <= c1; ++cc) {
        const int s = (cc * W / G >= t_beg) ? 0 : 1;
        sum += __ldcg(&p.ws_part[((cc * 2 + s) * 16 + m) * kRows + row]);
      }
      const int64_t n = (int64_t)tile * kRows + row;
      if (m < p.M && n < N) {
        if (p.bias) sum += __bfloat162float(p.bias[n]);
        p.y[(int64_t)m * N + n] = __float2bfloat16_rn(sum);
      }
      if (tid == 0) p.ws_cnt[tile] = 0u;
    }
  }
}

// ------------------------------------------------------------------ host side
namespace {

size_t smem_bytes(int MT) {
  return 1024 + (size_t)kStages * kStageBytes + 2 * (size_t)kConsumerWarps * MT * 16 * 8 * 4 +
         sizeof(Shared);
}

template <Fmt F, int MT>
cudaError_t launch_t(const CUtensorMap& map, const GemvParams& p, int grid, cudaStream_t stream) {
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
  pl.spt = (int)((K + sk - 1) / sk);
  pl.tiles = (int)((N + kRows - 1) / kRows);
  const int64_t work = (int64_t)pl.tiles * pl.spt;
  pl.grid = (int)std::max<int64_t>(1, std::min<int64_t>(num_sms, work));
  if (const char* env = std::getenv("WQ_GEMV_GRID")) {  // tuning knob
    const int v = std::atoi(env);
    if (v >= 1) pl.grid = (int)std::min<int64_t>(v, work);
  }
  // equal stage shares need a workspace and a single activation batch; they only help
  // when whole tiles would not divide evenly among the blocks
  pl.stream_k = (f != Fmt::MXFP4) && M <= 16 && (pl.tiles % pl.grid) != 0;
  pl.ws_bytes = pl.stream_k ? ws_counter_bytes(pl.tiles) + ws_partial_bytes(pl.grid) : 0;
  return pl;
}

bool gemv_mxfp4_supported(int64_t R, int64_t S, int64_t E) {
  return R * S <= kMaxSlots && E <= kMaxExperts;
}

cudaError_t launch_gemv(Fmt f, const CUtensorMap& map, GemvParams p, const GemvPlan& pl,
                        cudaStream_t stream) {
  if (!pl.stream_k) {
    p.ws_cnt = nullptr;
    p.ws_part = nullptr;
  }
  const bool wide = (f == Fmt::MXFP4) ? (p.M * p.S > 8) : (p.M > 8);
  switch (f) {
    case Fmt::I4G:
      return wide ? launch_t<Fmt::I4G, 2>(map, p, pl.grid, stream)
                  : launch_t<Fmt::I4G, 1>(map, p, pl.grid, stream);
    case Fmt::I4R:
      return wide ? launch_t<Fmt::I4R, 2>(map, p, pl.grid, stream)
                  : launch_t<Fmt::I4R, 1>(map, p, pl.grid, stream);
    case Fmt::I8R:
      return wide ? launch_t<Fmt::I8R, 2>(map, p, pl.grid, stream)
                  : launch_t<Fmt::I8R, 1>(map, p, pl.grid, stream);
    case Fmt::MXFP4:
      return wide ? launch_t<Fmt::MXFP4, 2>(map, p, pl.grid, stream)
                  : launch_t<Fmt::MXFP4, 1>(map, p, pl.grid, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace wq
