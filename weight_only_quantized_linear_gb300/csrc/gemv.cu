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
//   * every warp works on its own: it owns a contiguous range of the flattened
//     (16-row tile x 64-byte column chunk) work and streams it with 16-byte loads kept
//     kDepth chunks deep in registers, together with the chunk's scales / zero points;
//     there is no shared memory, block barrier or cross-warp reduction on the way;
//   * with a workspace the ranges are equal to within one chunk (stream-K over all the
//     warps of the grid); a tile cut by a range boundary is finished by the warp that
//     contributes last, which adds the partials in warp order (deterministic, and no warp
//     ever waits for another).  Without one, each warp takes whole tiles;
//   * a lane reads 16 bytes of two rows a chunk, dequantizes them exactly (see
//     dequant_nib8) and feeds them as the A operand of mma.sync m16n8k16 with the
//     activations as B.  The k order inside an MMA is a permutation shared by A and B,
//     so a lane's 16 contiguous bytes map straight onto its fragment slots;
//   * the MMA accumulators of a warp hold whole output rows, written out in bf16.
#include <algorithm>
#include <atomic>
#include <cstdlib>
#include <type_traits>

#include "common.cuh"
#include "launch.h"

namespace wq {

namespace {

constexpr int kRows = 16;         // weight rows a tile (one MMA M)
constexpr int kChunkBytes = 64;   // bytes of a row a warp chunk (4 lanes x 16 bytes)
constexpr int kWarps = 8;         // warps a block
constexpr int kThreads = kWarps * 32;
constexpr int kBlocksPerSM = 2;
constexpr int kDepth = 3;         // chunks in flight a warp
constexpr int kAccSets = 2;       // independent accumulator sets (shorter MMA chains)
constexpr int kMinChunks = 8;     // fewest chunks a warp: bounds the contributors of a tile
constexpr int kMaxSlots = 2048;   // MXFP4: rows x slots handled by one launch
constexpr int kMaxExperts = 256;
constexpr int kMaxPairs = kMaxExperts + kMaxSlots / 8;

template <Fmt F>
constexpr int piece_k() { return (F == Fmt::I8R) ? 16 : 32; }  // k of a 16-byte lane piece
template <Fmt F>
constexpr int chunk_k() { return 4 * piece_k<F>(); }           // k of a 64-byte chunk

// MXFP4 routing tables (identical in every block): slots sorted by expert, and
// (expert, first sorted slot, count) for each batch of at most 8*MT slots.
struct Routing {
  int npairs;
  int pair_expert[kMaxPairs];
  int pair_start[kMaxPairs];
  int pair_count[kMaxPairs];
  int sorted[kMaxSlots];
  int ecount[kMaxExperts + 1];
};

// First flattened chunk of warp c: equal shares (stream-K) or whole items.
__device__ __forceinline__ int64_t warp_begin(int64_t c, int64_t G, int64_t items, int cpt,
                                              bool whole_items) {
  return whole_items ? (c * items / G) * cpt : c * (items * cpt) / G;
}

// Finish the tiles cut by warp-range boundaries (stream-K launches only).  Each
// contributing warp adds one to the tile's counter once its partial is out; the one that
// brings it to the number of contributors adds the partials in warp order, writes y and
// clears the counter.  Nobody waits on anybody.  W: chunks of the launch; G: warps.
__device__ __forceinline__ void finish_cut_tiles(const GemvParams& p, int64_t c, int64_t G,
                                                 int64_t W, int cpt, const int (&pend_tile)[2],
                                                 int npend, int lane) {
  const int64_t N = p.N;
  // range boundary c * W / G of warp c: 32-bit arithmetic when the product fits
  const bool narrow = (uint64_t)W * (uint64_t)G < (1ull << 32);
  auto bound = [&](int64_t cc) -> int64_t {
    return narrow ? (int64_t)((uint32_t)cc * (uint32_t)W / (uint32_t)G) : cc * W / G;
  };
  auto owner = [&](int64_t sidx) -> int64_t {
    int64_t cc = narrow ? (int64_t)((uint32_t)sidx * (uint32_t)G / (uint32_t)W) : sidx * G / W;
    while (cc + 1 < G && bound(cc + 1) <= sidx) ++cc;
    while (cc > 0 && bound(cc) > sidx) --cc;
    return cc;
  };
  for (int i = 0; i < npend; ++i) {
    const int tile = pend_tile[i];
    // the lanes' partial stores happen before lane 0's fence (warp barrier), and the
    // fence before its arrival on the counter
    __syncwarp();
    if (lane == 0) __threadfence();
    const int64_t t_beg = (int64_t)tile * cpt;
    const int64_t c0 = owner(t_beg), c1 = owner(t_beg + cpt - 1);
    // warps between c0 and c1 whose range is empty (fewer chunks than warps) take no part
    uint32_t contributors = 0;
    for (int64_t cc = c0; cc <= c1; ++cc)
      if (bound(cc) < bound(cc + 1)) ++contributors;
    int last = 0;
    if (lane == 0) last = (atomicAdd(&p.ws_cnt[tile], 1u) == contributors - 1u) ? 1 : 0;
    last = __shfl_sync(0xffffffffu, last, 0);
    if (last) {
      __threadfence();
      for (int idx = lane; idx < p.M * kRows; idx += 32) {
        const int m = idx / kRows, row = idx % kRows;
        // independent loads four at a time, added in warp order
        float v = 0.0f;
        for (int64_t cc0 = c0; cc0 <= c1; cc0 += 4) {
          float part[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int64_t cc = cc0 + q;
            part[q] = 0.0f;
            if (cc <= c1) {
              const int64_t b0 = bound(cc);
              if (b0 != bound(cc + 1)) {
                // read, then cleared: the call leaves the workspace zero-filled
                const int sid = (b0 >= t_beg) ? 0 : 1;
                float* src = &p.ws_part[((cc * 2 + sid) * p.M + m) * kRows + row];
                part[q] = __ldcg(src);
                __stcg(src, 0.0f);
              }
            }
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) v += part[q];
        }
        const int64_t n = (int64_t)tile * kRows + row;
        if (n < N) {
          if (p.bias) v += __bfloat162float(p.bias[n]);
          p.y[(int64_t)m * N + n] = __float2bfloat16_rn(v);
        }
      }
      __syncwarp();
      if (lane == 0) p.ws_cnt[tile] = 0u;
    }
  }
}

}  // namespace

// MT: activation rows a batch, in groups of 8 (MMA path) or 1..2 rows (FMA path).
// kFMA: multiply on the FMA pipe (mixed-precision bf16 x bf16 -> f32) instead of the
// warp MMA, for one or two activation rows.
template <Fmt F, int MT, bool kFMA>
__global__ void __launch_bounds__(kThreads, kBlocksPerSM) k_gemv(const GemvParams p) {
  constexpr int kPiece = piece_k<F>();
  constexpr int kChunkK = chunk_k<F>();
  constexpr int kBatch = kFMA ? MT : 8 * MT;
  extern __shared__ __align__(16) uint8_t smem_dyn[];
  Routing* rt = reinterpret_cast<Routing*>(smem_dyn);  // MXFP4 only

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tid = threadIdx.x;
  const int64_t N = p.N;
  const int64_t K = p.K;
  const int tiles = (int)((N + kRows - 1) / kRows);
  const int cpt = (int)((K + kChunkK - 1) / kChunkK);  // chunks a tile
  const int64_t row_bytes = (F == Fmt::I8R) ? K : K / 2;

  // ---- work items: (tile, activation batch) or (tile, routed-expert batch) ----
  int64_t items;
  if constexpr (F == Fmt::MXFP4) {
    // stable counting sort of the R*S slots by expert, then batches of kBatch slots
    const int E = (int)p.E;
    const int slots = (int)(p.M * p.S);
    for (int e = tid; e <= E; e += kThreads) rt->ecount[e] = 0;
    __syncthreads();
    for (int i = tid; i < slots; i += kThreads) {
      const int e = p.experts[i];
      if (e >= 0 && e < E) atomicAdd(&rt->ecount[e], 1);
    }
    __syncthreads();
    if (tid == 0) {
      int run = 0, np = 0;
      for (int e = 0; e < E; ++e) {
        const int cnt = rt->ecount[e];
        rt->ecount[e] = run;
        for (int b = 0; b < cnt; b += kBatch) {
          rt->pair_expert[np] = e;
          rt->pair_start[np] = run + b;
          rt->pair_count[np] = min(kBatch, cnt - b);
          ++np;
        }
        run += cnt;
      }
      rt->npairs = np;
      for (int i = 0; i < slots; ++i) {  // ascending slot order within an expert
        const int e = p.experts[i];
        if (e >= 0 && e < E) rt->sorted[rt->ecount[e]++] = i;
      }
    }
    __syncthreads();
    items = (int64_t)rt->npairs * tiles;
  } else {
    items = (int64_t)tiles * ((p.M + kBatch - 1) / kBatch);
  }

  const bool stream_k = (p.ws_cnt != nullptr);  // partial tiles allowed (one batch only)
  const int64_t G = (int64_t)gridDim.x * kWarps;
  const int64_t c = (int64_t)blockIdx.x * kWarps + warp;
  const int64_t beg = warp_begin(c, G, items, cpt, !stream_k);
  const int64_t end = warp_begin(c + 1, G, items, cpt, !stream_k);
  if (beg >= end) return;  // no block-wide synchronization after this point

  const int g8 = lane >> 2;  // MMA row group: tile rows g8 and g8 + 8
  const int cq = lane & 3;   // 16-byte piece of the chunk
  const int gshift = p.group_shift;
  const int64_t gpr = (F == Fmt::I4G) ? (K >> gshift) : (K >> 5);  // scales a row

  // this lane's two weight rows of an item: row A (tile row g8) and row B, 8 rows
  // further; a row past the end of the matrix loads nothing
  struct Rows {
    const uint8_t* w;   // row A's packed bytes at this lane's 16-byte piece
    const float* s;     // row A's scales
    const uint8_t* z;   // row A's zero points, or E8M0 block scales (MXFP4)
    uint32_t valid;     // bit 0: row A exists, bit 1: row B exists
  };
  auto rows_of = [&](int64_t item) -> Rows {
    Rows r;
    const int tile = (int)(item % tiles);
    const int64_t nA = (int64_t)tile * kRows + g8;
    r.valid = (nA < N ? 1u : 0u) | (nA + 8 < N ? 2u : 0u);
    int64_t erow = 0;
    if constexpr (F == Fmt::MXFP4) erow = (int64_t)rt->pair_expert[item / tiles] * N;
    r.w = p.w + (erow + nA) * row_bytes + cq * 16;
    if constexpr (F == Fmt::I4G) {
      r.s = p.scale + nA * gpr;
      r.z = p.zero + nA * gpr;
    } else if constexpr (F == Fmt::MXFP4) {
      r.s = nullptr;
      r.z = p.escale + (erow + nA) * gpr;
    } else {
      r.s = p.scale + nA;
      r.z = nullptr;
    }
    return r;
  };

  // one chunk in flight: 16 bytes of each row and the dequantization parameters.  A
  // piece past the end of K loads nothing and gets scale 0, so it dequantizes to zeros.
  struct Slot {
    uint4 a, b;
    float sa, sb;
    // zero points (I4G) or E8M0 block scales (MXFP4) of rows A and B, each loaded into a
    // register of its own: combining them here would wait for the loads
    uint32_t za, zb;
  };
  auto load_slot = [&](const Rows& r, int ch) -> Slot {
    Slot s;
    s.a = s.b = make_uint4(0, 0, 0, 0);
    s.sa = s.sb = 0.0f;  // MXFP4: sa = 1 marks a piece inside K
    s.za = s.zb = 0u;
    const int kp = ch * kChunkK + cq * kPiece;
    if (kp < K) {
      const int64_t wstep = 8 * row_bytes, mstep = 8 * gpr;
      if (r.valid & 1u) s.a = ld_global_stream_v4(r.w + ch * kChunkBytes);
      if (r.valid & 2u) s.b = ld_global_stream_v4(r.w + wstep + ch * kChunkBytes);
      if constexpr (F == Fmt::I4G) {
        const int gi = kp >> gshift;
        if (r.valid & 1u) {
          s.sa = __ldg(r.s + gi);
          s.za = (uint32_t)__ldg(r.z + gi);
        }
        if (r.valid & 2u) {
          s.sb = __ldg(r.s + mstep + gi);
          s.zb = (uint32_t)__ldg(r.z + mstep + gi);
        }
      } else if constexpr (F == Fmt::MXFP4) {
        const int bi = kp >> 5;
        s.sa = 1.0f;
        if (r.valid & 1u) s.za = (uint32_t)__ldg(r.z + bi);
        if (r.valid & 2u) s.zb = (uint32_t)__ldg(r.z + mstep + bi);
      } else {
        if (r.valid & 1u) s.sa = __ldg(r.s);
        if (r.valid & 2u) s.sb = __ldg(r.s + 8);
      }
    }
    return s;
  };

  // activation row of MMA column m of an item (-1: none) and its output row
  auto xrow_of = [&](int64_t item, int m, int* yrow) -> int {
    if constexpr (F == Fmt::MXFP4) {
      const int pr = (int)(item / tiles);
      if (m >= rt->pair_count[pr]) return -1;
      const int slot = rt->sorted[rt->pair_start[pr] + m];
      *yrow = slot;
      return p.x_per_slot ? slot : slot / (int)p.S;
    } else {
      const int64_t row = (item / tiles) * kBatch + m;
      if (row >= p.M) return -1;
      *yrow = (int)row;
      return (int)row;
    }
  };

  // prefetch cursor: kDepth chunks ahead of the main one
  int64_t pg = beg;
  int64_t pitem = beg / cpt;
  int pch = (int)(beg % cpt);
  Rows prow = rows_of(pitem);
  auto next_slot = [&]() -> Slot {
    Slot s;
    if (pg < end) {
      s = load_slot(prow, pch);
    } else {
      s.a = s.b = make_uint4(0, 0, 0, 0);
      s.sa = s.sb = 0.0f;
      s.za = s.zb = 0u;
    }
    ++pg;
    if (++pch == cpt) {
      pch = 0;
      ++pitem;
      if (pg < end) prow = rows_of(pitem);
    }
    return s;
  };
  Slot ring[kDepth];
#pragma unroll
  for (int j = 0; j < kDepth; ++j) ring[j] = next_slot();

  // main cursor
  int64_t item = beg / cpt;
  int ch = (int)(beg % cpt);
  const __nv_bfloat16* xptr[MT];
  auto set_xptr = [&]() {
#pragma unroll
    for (int tt = 0; tt < MT; ++tt) {
      int yr;
      const int xr = xrow_of(item, kFMA ? tt : tt * 8 + g8, &yr);
      xptr[tt] = (xr >= 0) ? p.x + (int64_t)xr * K : nullptr;
    }
  };
  set_xptr();

  float acc[MT][kAccSets][4];  // MMA path: D fragments; FMA path: [tt][set][row A lo, A hi, B lo, B hi]
#pragma unroll
  for (int t = 0; t < MT; ++t)
#pragma unroll
    for (int a = 0; a < kAccSets; ++a)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[t][a][i] = 0.0f;

  bool seg_first = true;            // the segment holds this warp's first chunk
  bool seg_from_start = (ch == 0);  // the segment began at chunk 0 of its tile
  int pend_tile[2] = {-1, -1};      // tiles cut by this warp's range boundaries
  int npend = 0;

  const int64_t total = end - beg;
  for (int64_t u0 = 0; u0 < total; u0 += kDepth) {
#pragma unroll
    for (int j = 0; j < kDepth; ++j) {
      if (u0 + j < total) {
        const Slot s = ring[j];
        ring[j] = next_slot();

        // activations of this lane's piece (L1-resident), consumed after the dequant
        const int64_t kp = (int64_t)ch * kChunkK + cq * kPiece;
        uint32_t xw[MT][kPiece / 2];
#pragma unroll
        for (int tt = 0; tt < MT; ++tt) {
#pragma unroll
          for (int q = 0; q < kPiece / 8; ++q) {
            uint4 v = make_uint4(0, 0, 0, 0);
            if (xptr[tt] != nullptr && kp < K) v = ld_global_nc_v4(xptr[tt] + kp + q * 8);
            xw[tt][4 * q + 0] = v.x;
            xw[tt][4 * q + 1] = v.y;
            xw[tt][4 * q + 2] = v.z;
            xw[tt][4 * q + 3] = v.w;
          }
        }

        const uint32_t wA[4] = {s.a.x, s.a.y, s.a.z, s.a.w};
        const uint32_t wB[4] = {s.b.x, s.b.y, s.b.z, s.b.w};
        if constexpr (F == Fmt::I8R) {
          const float2 i8c = make_float2(-8388736.0f, -8388736.0f);  // -(2^23 + 128)
          const float2 sA = make_float2(s.sa, s.sa), sB = make_float2(s.sb, s.sb);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint32_t ga[2], gb[2];
            dequant_i8x4(wA[i], i8c, sA, ga);
            dequant_i8x4(wB[i], i8c, sB, gb);
#pragma unroll
            for (int tt = 0; tt < MT; ++tt) {
              if constexpr (kFMA) {
                fma_bf16x2_f32(ga[0], xw[tt][2 * i], acc[tt][i % kAccSets][0], acc[tt][i % kAccSets][1]);
                fma_bf16x2_f32(ga[1], xw[tt][2 * i + 1], acc[tt][i % kAccSets][0], acc[tt][i % kAccSets][1]);
                fma_bf16x2_f32(gb[0], xw[tt][2 * i], acc[tt][i % kAccSets][2], acc[tt][i % kAccSets][3]);
                fma_bf16x2_f32(gb[1], xw[tt][2 * i + 1], acc[tt][i % kAccSets][2], acc[tt][i % kAccSets][3]);
              } else {
                mma_bf16_16816(acc[tt][i % kAccSets], ga[0], gb[0], ga[1], gb[1], xw[tt][2 * i],
                               xw[tt][2 * i + 1]);
              }
            }
          }
        } else {
          Nib8Consts kA, kB;
          float2 XA, XB;
          if constexpr (F == Fmt::I4G) {
            kA = make_nib8_consts_u(s.sa, s.za);
            kB = make_nib8_consts_u(s.sb, s.zb);
          } else if constexpr (F == Fmt::I4R) {
            kA = make_nib8_consts(s.sa, 8.0f);
            kB = make_nib8_consts(s.sb, 8.0f);
          } else {
            const bool ok = s.sa != 0.0f;
            const float xa = ok ? e8m0_to_f32(s.za) : 0.0f;
            const float xb = ok ? e8m0_to_f32(s.zb) : 0.0f;
            XA = make_float2(xa, xa);
            XB = make_float2(xb, xb);
          }
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
              dequant_e2m1x8(wA[i], XA, ga);
              dequant_e2m1x8(wB[i], XB, gb);
            }
#pragma unroll
            for (int tt = 0; tt < MT; ++tt) {
              if constexpr (kFMA) {
                // natural k order: x pair 4i + q holds elements (8i + 2q, 8i + 2q + 1)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  float* a = acc[tt][q % kAccSets];
                  fma_bf16x2_f32(ga[q], xw[tt][4 * i + q], a[0], a[1]);
                  fma_bf16x2_f32(gb[q], xw[tt][4 * i + q], a[2], a[3]);
                }
              } else {
                mma_bf16_16816(acc[tt][(2 * i) % kAccSets], ga[0], gb[0], ga[1], gb[1],
                               xw[tt][4 * i], xw[tt][4 * i + 1]);
                mma_bf16_16816(acc[tt][(2 * i + 1) % kAccSets], ga[2], gb[2], ga[3], gb[3],
                               xw[tt][4 * i + 2], xw[tt][4 * i + 3]);
              }
            }
          }
        }

        // ---- end of a segment: the tile ends here, or this warp's range does ----
        const bool tile_end = (ch == cpt - 1);
        if (tile_end || u0 + j + 1 == total) {
          const bool full_tile = seg_from_start && tile_end;
          const int tile = (int)(item % tiles);
          const int slot_id = seg_first ? 0 : 1;
          // one output value: full tiles go to y, cut tiles to this warp's partial slot
          auto emit = [&](int m, int row, float v) {
            const int64_t n = (int64_t)tile * kRows + row;
            if (full_tile) {
              int yr = -1;
              if (xrow_of(item, m, &yr) >= 0 && n < N) {
                if (p.bias) v += __bfloat162float(p.bias[n]);
                if (F == Fmt::MXFP4 && p.y32 != nullptr)
                  p.y32[(int64_t)yr * N + n] = p.sw ? v * __ldg(p.sw + yr) : v;
                else
                  p.y[(int64_t)yr * N + n] = __float2bfloat16_rn(v);
              }
            } else if (m < p.M) {
              p.ws_part[((c * 2 + slot_id) * p.M + m) * kRows + row] = v;
            }
          };
#pragma unroll
          for (int tt = 0; tt < MT; ++tt) {
            if constexpr (kFMA) {
              // [set][A lo, A hi, B lo, B hi]; add the halves, the sets and the four lanes
              // (cq) that share the row; lane cq == 0 writes rows g8 and g8 + 8
              float vA = 0.0f, vB = 0.0f;
#pragma unroll
              for (int a = 0; a < kAccSets; ++a) {
                vA += acc[tt][a][0] + acc[tt][a][1];
                vB += acc[tt][a][2] + acc[tt][a][3];
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[tt][a][i] = 0.0f;
              }
              vA += __shfl_xor_sync(0xffffffffu, vA, 1);
              vA += __shfl_xor_sync(0xffffffffu, vA, 2);
              vB += __shfl_xor_sync(0xffffffffu, vB, 1);
              vB += __shfl_xor_sync(0xffffffffu, vB, 2);
              if (cq == 0) {
                emit(tt, g8, vA);
                emit(tt, g8 + 8, vB);
              }
            } else {
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                float v = 0.0f;
#pragma unroll
                for (int a = 0; a < kAccSets; ++a) {
                  v += acc[tt][a][i];
                  acc[tt][a][i] = 0.0f;
                }
                // D fragment: i = 0, 1 -> row g8, columns 2cq, 2cq+1; i = 2, 3 -> row g8 + 8
                emit(tt * 8 + 2 * cq + (i & 1), g8 + ((i >> 1) << 3), v);
              }
            }
          }
          if (!full_tile) pend_tile[npend++] = tile;
          seg_first = false;
          seg_from_start = true;
        }

        // ---- advance the main cursor ----
        if (++ch == cpt) {
          ch = 0;
          ++item;
          if (u0 + j + 1 < total) set_xptr();
        }
      }
    }
  }

  finish_cut_tiles(p, c, G, items * cpt, cpt, pend_tile, npend, lane);
}

// ------------------------------------------------------------------ factored decode
// Formats I4G with a group of at least 128 codes, I4R and I8R; any number of activation
// rows (batches of 8 * MT).
//
// Within one 64-byte chunk of a row (128 4-bit codes, or 64 int8 codes) the scale s and
// the zero point z are constant, so the chunk's share of the dot product is
//     sum_k x[k] * ((q[k] - z) * s)  =  s * sum_k x[k] * (q[k] - z):
// the per-element product of the definition, reassociated ("Quantization" (Linnet docs):
// dequantize_int4_groups forms (q - zero) * scale per element in f32 and casts it to
// bf16; here that product is not rounded to bf16 and s is applied once a chunk).  q - z
// is a small integer and is formed exactly in bf16x2:
//   * 4-bit: the nibble q in the low mantissa bits of the bf16 128.0 (one logic op) is
//     128 + q; subtracting the bf16 128 + z (exact for z <= 127) leaves q - z.  Larger
//     zero points take a second exact subtraction (a warp-uniform slow path);
//   * int8: the byte q + 128 in the mantissa of the f32 2^23, minus 2^23 + 128, is q,
//     exact in bf16 since |q| <= 128.
// The chunk's sum then runs on the warp MMA (m16n8k16, bf16 in, f32 accumulate): the
// products x * (q - z) are exact and only the f32 sums round, as in any f32 dot product.
// A word of eight 4-bit codes costs four logic ops, three shifts, four packed
// subtractions and a quarter of an MMA a lane, against an f32 multiply and a conversion
// to bf16 for every element when the weights are dequantized first.
//
// Lane layout, work split and stream-K fixup are those of k_gemv.  The k order inside an
// MMA is a permutation shared by A and B: the nibble extraction yields the pairs
// (k, k + 4) of a word, so each lane permutes its activations into the same pairs once a
// chunk (shared by both rows and every MMA of the chunk).

namespace {

// The factored kernel runs in clusters of kCl CTAs (kCl * kWarps warps), as many as
// fit two blocks on every SM: the main loop is bound by instruction issue, so every SM
// should hold the same two CTAs.  Two CTAs a cluster, four for group-wise rows of 32 or
// more steps (K >= 8192 at one batch); clusters of eight fit only 34 to a launch on GB300
// (272 CTAs on 152 SMs, a fifth of the SMs with one CTA whose warps finish early).
// Measured on the Llama-3.1-8B decode layer (clusters of 8 / 4 / 2): 64.1 / 62.4 / 61.6 us
// a layer; down (4096 x 14336) 13.87 / 13.4 / 13.85 us.
template <int kCl>
struct ClusterShape {
  static constexpr int kWarpsC = kCl * kWarps;
  static constexpr int kLog2 = kCl == 2 ? 4 : (kCl == 4 ? 5 : 6);
  static_assert((1 << kLog2) == kWarpsC, "warps a cluster: a power of two");
};
__host__ __device__ constexpr int cluster_warps_log2(int cl) { return cl == 2 ? 4 : (cl == 4 ? 5 : 6); }

// Write a finished tile's D fragments (rows g8 / g8 + 8, columns 2cq, 2cq + 1 of each
// group of 8 activation rows) to y, adding the bias.
template <int MT>
__device__ __forceinline__ void emit_tile(const GemvParams& p, int64_t item, int tiles, int batch,
                                          const float (&tot)[MT][4], int g8, int cq) {
  const int64_t tile = item % tiles;
  const int64_t b0 = (item / tiles) * batch;
#pragma unroll
  for (int tt = 0; tt < MT; ++tt) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t m = b0 + tt * 8 + 2 * cq + (i & 1);
      const int64_t n = tile * kRows + g8 + ((i >> 1) << 3);
      if (m < p.M && n < p.N) {
        const float bias = p.bias ? __bfloat162float(p.bias[n]) : 0.0f;
        p.y[m * p.N + n] = __float2bfloat16_rn(tot[tt][i] + bias);
      }
    }
  }
}

}  // namespace

// Work split: launched in clusters of CTAs (thread-block clusters).  Each cluster takes
// a contiguous range of whole items (a 16-row tile and a batch of activation rows); the
// cluster's warps split its (item, step) units evenly, a step being two chunks, i.e. 128
// contiguous bytes of each of the tile's 16 rows.  A tile whose units fall to one warp is
// written to y by that warp; a tile cut between warps is finished inside the cluster:
// each contributor leaves its partial D fragment in its own shared-memory slot, and
// after a cluster barrier the warp that holds the tile's last step adds the
// contributors' slots in warp order (deterministic), reading the other CTAs' slots
// through distributed shared memory.  No workspace, atomics or memory fences.
//
// Loads: every warp streams its steps through its own ring of kFactStages shared-memory
// stages filled by TMA (a {128 bytes, 16 rows} box of codes with the 128-byte swizzle,
// and the step's scales and zero points), one mbarrier a stage; kFactStages - 1 steps
// are in flight while one is computed, independent of the register budget.  Rows past N
// arrive as zeros (TMA fills out-of-bounds boxes) and are never stored.  Activation rows
// past M are clamped to the last one (those MMA columns are never stored).
// kPush: tiles cut between warps are finished without cluster-wide barriers.  Every
// contributing warp stores its partial D fragment (16 rows x M columns) straight into a
// receive slot of the closing warp (the one holding the tile's last step) through
// distributed shared memory and arrives on that warp's mbarrier; only the closing warp
// waits, then adds the slots in warp order (deterministic) and its own partial last.
// geo.cmax: receive slots a warp (the most warps any tile of the launch meets).
struct FactGeom {
  uint32_t xstride;  // bytes between staged activation rows
  uint32_t cmax;     // receive slots a warp (push fixup)
};

struct FactMaps {
  CUtensorMap w;  // codes [N rows, row_bytes], box {128, 16}, 128-byte swizzle
  CUtensorMap s;  // I4G: scales [N, K/G] f32, box {4, 16}; I4R / I8R: scales [N] f32, box {16, 1}
  CUtensorMap z;  // I4G: zero points [N, K/G] u8, box {16, 16}
};

constexpr int kFactStageW = 2048;  // code bytes a stage (16 rows x 128)
constexpr int kFactStageS = 256;   // scale bytes a stage (I4G: 16 rows x 4 groups)
constexpr int kFactStageZ = 256;   // zero-point bytes a stage (16 rows x 16 groups)
constexpr int kFactXPad = 64;      // bytes between staged activation rows (banks)
// dynamic shared memory: codes (1024-byte aligned for the swizzle), scales, zero points,
// barriers of kSD stages a warp; then the staged activations; plus slack for the alignment
__host__ __device__ constexpr int fact_ring_bytes(int kSD) {
  return kWarps * kSD * (kFactStageW + kFactStageS + kFactStageZ + 8);
}

// kSD: ring stages a warp.  kXS: activations staged once a block in shared memory, in the
// order of the MMA fragments ([row][k / 128][(k / 8) % 4][(k / 32) % 4] 16-byte pieces
// holding (x0, x4) (x1, x5) (x2, x6) (x3, x7)), so that a lane's B fragments are four
// 16-byte shared loads a chunk, with no shuffles and no global-memory latency in the loop.
template <Fmt F, int MT, int kSD, bool kXS, bool kPush, int kCl>
__global__ void __launch_bounds__(kThreads, kBlocksPerSM)
    k_gemv_fact(const GemvParams p, const __grid_constant__ FactMaps maps, const FactGeom geo) {
  constexpr int kFactWarps = ClusterShape<kCl>::kWarpsC;
  constexpr int kFactWarpsLog2 = ClusterShape<kCl>::kLog2;
  const uint32_t xstride = geo.xstride;
  static_assert(F == Fmt::I4G || F == Fmt::I4R || F == Fmt::I8R, "affine formats only");
  constexpr int kPiece = piece_k<F>();   // k of a lane's 16 bytes
  constexpr int kChunkK = chunk_k<F>();  // k of a 64-byte chunk
  constexpr int kXR = kPiece / 2;        // bf16x2 registers of x a piece
  constexpr int kBatch = 8 * MT;         // activation rows an item
  constexpr int kS = kSD;
  static_assert(!kXS || (F != Fmt::I8R && MT == 1), "staged activations: 4-bit formats, one batch");
  constexpr uint32_t kStageTx =
      kFactStageW + ((F == Fmt::I4G) ? kFactStageS + kFactStageZ : 16 * 4);
  // partial D fragments of cut tiles: [warp][first / last segment][lane][4 * MT]
  __shared__ __align__(16) float s_part[kWarps][2][32][4 * MT];
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));

  // the next kernel of the stream may be scheduled as our CTAs retire; its own
  // grid_dep_wait() orders it after this grid
  grid_dep_launch_dependents();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g8 = lane >> 2;  // MMA row group: tile rows g8 and g8 + 8
  const int cq = lane & 3;   // 16-byte piece of a chunk
  const int64_t K = p.K;
  const int64_t M = p.M;
  const uint32_t tiles = (uint32_t)((p.N + kRows - 1) / kRows);
  const int64_t row_bytes = (F == Fmt::I8R) ? K : K / 2;
  const uint32_t spt = (uint32_t)(row_bytes / (2 * kChunkBytes));  // steps a tile
  // items * spt < 2^31 (checked by the host): unit and item indices are 32-bit
  const uint32_t items = tiles * (uint32_t)((M + kBatch - 1) / kBatch);

  // this warp's ring
  uint8_t* wst = smem + warp * kS * kFactStageW;
  uint8_t* sst = smem + kWarps * kS * kFactStageW + warp * kS * kFactStageS;
  uint8_t* zst = smem + kWarps * kS * (kFactStageW + kFactStageS) + warp * kS * kFactStageZ;
  uint64_t* bars = reinterpret_cast<uint64_t*>(
      smem + kWarps * kS * (kFactStageW + kFactStageS + kFactStageZ) + warp * kS * 8);

  // this cluster's items and units, and the first unit of warp w of the cluster (this
  // warp is warp wc of kFactWarps); recomputed after the main loop rather than kept in
  // registers.  Cluster c takes q or q + 1 items, q = items / clusters.
  struct Split {
    uint32_t u0, U, wc;
    __device__ uint32_t bound(uint32_t w) const {
      return u0 + (uint32_t)(((uint64_t)w * U) >> kFactWarpsLog2);
    }
  };
  auto split = [&]() -> Split {
    const uint32_t ncl = cluster_count_x(), cid = cluster_id_x();
    const uint32_t q = items / ncl, r = items - q * ncl;
    const uint32_t ibeg = cid * q + min(cid, r), icnt = q + (cid < r ? 1u : 0u);
    return Split{ibeg * spt, icnt * spt, cluster_ctarank() * kWarps + warp};
  };
  uint32_t beg, end;
  {
    const Split sp = split();
    beg = sp.bound(sp.wc);
    end = sp.bound(sp.wc + 1);
  }
  const int gshift = p.group_shift;
  // bf16x2 (128, 128), derived from a kernel argument so that it stays in a register
  const uint32_t magic = 0x43004300u | (uint32_t)(p.K >> 62);
  int close_item = -1;  // the cut tile this warp finishes after the cluster barrier
  float ctot[MT][4];    // push fixup: the partial of the tile this warp closes
#pragma unroll
  for (int tt = 0; tt < MT; ++tt) ctot[tt][0] = ctot[tt][1] = ctot[tt][2] = ctot[tt][3] = 0.0f;

  const int total = beg < end ? (int)(end - beg) : 0;
  // ---- producer side: lane 0 fills stage (u mod kS) with the data of unit beg + u; its
  // cursor (tile row, step) advances one unit an issue ----
  const uint64_t pol_stream = l2_policy_evict_first();
  const uint64_t pol_keep = l2_policy_evict_last();
  uint32_t i_st = beg % spt;
  uint32_t i_tile = (beg / spt) % tiles;
  auto issue = [&](int u) {
    const uint32_t st = i_st;
    const int32_t row0 = (int32_t)(i_tile * kRows);
    if (++i_st == spt) {
      i_st = 0;
      if (++i_tile == tiles) i_tile = 0;
    }
    const int stage = u % kS;
    uint64_t* bar = bars + stage;
    mbar_arrive_expect_tx(bar, kStageTx);
    tma_load_2d(wst + stage * kFactStageW, &maps.w, bar, (int32_t)(st * 2 * kChunkBytes), row0,
                pol_stream);
    if constexpr (F == Fmt::I4G) {
      const int32_t g0 = (int32_t)((st * 2 * kChunkK) >> gshift);
      tma_load_2d(sst + stage * kFactStageS, &maps.s, bar, g0 & ~3, row0, pol_keep);
      tma_load_2d(zst + stage * kFactStageZ, &maps.z, bar, g0 & ~15, row0, pol_keep);
    } else {
      tma_load_2d(sst + stage * kFactStageS, &maps.s, bar, row0, 0, pol_keep);
    }
  };
  // push fixup: receive slots [warp][cmax][16 rows][M] f32 and one mbarrier a warp, after
  // the staged activations
  uint8_t* const xs = smem + fact_ring_bytes(kS);
  float* const recv = reinterpret_cast<float*>(
      xs + (kXS ? (((uint32_t)M * xstride + 15u) & ~15u) : 0u));
  uint64_t* const recvbar = reinterpret_cast<uint64_t*>(recv + (size_t)kWarps * geo.cmax * 16 * M);
  // the tile this warp closes in the push fixup: its first segment, cut (the range starts
  // inside the tile) and ending inside the range; and how many lanes arrive for it
  uint32_t push_arrivals = 0;
  if constexpr (kPush) {
    if (beg < end && beg % spt != 0 && (beg / spt + 1) * spt <= end) {
      close_item = (int)(beg / spt);
      const Split sp = split();
      const uint32_t t0 = (uint32_t)close_item * spt;
      uint32_t w0 = sp.wc;
      while (w0 > 0 && sp.bound(w0) > t0) --w0;
      for (uint32_t w = w0; w < sp.wc; ++w)
        if (sp.bound(w) < sp.bound(w + 1) && sp.bound(w + 1) > t0) push_arrivals += 32;
    }
  }
  if (lane == 0) {
    for (int i = 0; i < kS; ++i) mbar_init(bars + i, 1);
    if constexpr (kPush) mbar_init(recvbar + warp, push_arrivals > 0 ? push_arrivals : 1u);
    fence_mbar_init();
  }
  bool cl_waited = false;  // this warp has passed the cluster barrier's wait
  if constexpr (kPush) {
    // every CTA's receive barriers are initialized before any warp of the cluster arrives
    // on them: arrive now, wait just before the first push (or at the end)
    __syncwarp();
    cluster_arrive_release();
  }
  // everything above overlaps the previous kernel (programmatic dependent launch).  Before
  // the wait, only the weights (codes, scales, zero points) may be read, and only when the
  // caller has declared them immutable; activations, outputs and everything else wait.
  if (p.weights_static && lane == 0) {
    for (int u = 0; u < kS - 1 && u < total; ++u) issue(u);
  }
  grid_dep_wait();
  if (!p.weights_static && lane == 0) {
    for (int u = 0; u < kS - 1 && u < total; ++u) issue(u);
  }
  __syncwarp();

  if constexpr (kXS) {
    // every thread of the block stages activations: eight independent 16-byte loads in
    // flight a thread, then their permuted stores
    const uint32_t k8n = (uint32_t)(K / 8);
    const uint32_t xtotal = (uint32_t)M * k8n;
    const uint32_t xbase = smem_u32(xs);
    bool bad_order = false;
    for (uint32_t base = 0; base < xtotal; base += 8 * kThreads) {
      uint4 v[8];
      if (p.order == nullptr) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint32_t idx = base + q * kThreads + threadIdx.x;
          if (idx < xtotal) {
            const uint32_t m = idx / k8n, k8 = idx - m * k8n;
            v[q] = ld_global_nc_v4(p.x + (int64_t)m * K + (int64_t)k8 * 8);
          }
        }
      } else {
        // activation order: stored column j multiplies input order[j] ("Quantization"
        // (Linnet docs), "Importing GPTQ and AWQ": the layer gathers its inputs first);
        // an entry outside [0, K) reads as 0 and is reported
        const unsigned short* xh = reinterpret_cast<const unsigned short*>(p.x);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint32_t idx = base + q * kThreads + threadIdx.x;
          if (idx < xtotal) {
            const uint32_t m = idx / k8n, k8 = idx - m * k8n;
            const int4 o0 = __ldg(reinterpret_cast<const int4*>(p.order + (int64_t)k8 * 8));
            const int4 o1 = __ldg(reinterpret_cast<const int4*>(p.order + (int64_t)k8 * 8 + 4));
            const int oi[8] = {o0.x, o0.y, o0.z, o0.w, o1.x, o1.y, o1.z, o1.w};
            uint32_t h[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const bool ok = (uint32_t)oi[j] < (uint32_t)K;
              bad_order |= !ok;
              h[j] = ok ? (uint32_t)__ldg(xh + (int64_t)m * K + oi[j]) : 0u;
            }
            v[q] = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16),
                              h[6] | (h[7] << 16));
          }
        }
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const uint32_t idx = base + q * kThreads + threadIdx.x;
        if (idx < xtotal) {
          const uint32_t m = idx / k8n, k8 = idx - m * k8n;
          const uint32_t o0 = __byte_perm(v[q].x, v[q].z, 0x5410), o1 = __byte_perm(v[q].x, v[q].z, 0x7632);
          const uint32_t o2 = __byte_perm(v[q].y, v[q].w, 0x5410), o3 = __byte_perm(v[q].y, v[q].w, 0x7632);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                           xbase + m * xstride + (k8 >> 4) * 256 + (k8 & 3) * 64 + ((k8 >> 2) & 3) * 16),
                       "r"(o0), "r"(o1), "r"(o2), "r"(o3)
                       : "memory");
        }
      }
    }
    if (bad_order) set_dev_status(p.dev_status, WQ_DEV_BAD_ORDER);
    __syncthreads();
  }

  if (beg < end) {
  // ---- consumer side ----
  uint32_t item = beg / spt;
  uint32_t st = beg - item * spt;
  const __nv_bfloat16* xrow[MT];  // activation row tt * 8 + g8 of the item's batch (clamped)
  auto set_xrow = [&]() {
    const int64_t b0 = (int64_t)(item / tiles) * kBatch;
#pragma unroll
    for (int tt = 0; tt < MT; ++tt) xrow[tt] = p.x + imin64(b0 + tt * 8 + g8, M - 1) * K + cq * kPiece;
  };
  set_xrow();
  float tot[MT][4];  // D fragments of the segment, scaled: rows g8 / g8 + 8, columns 2cq, 2cq+1
#pragma unroll
  for (int tt = 0; tt < MT; ++tt) tot[tt][0] = tot[tt][1] = tot[tt][2] = tot[tt][3] = 0.0f;
  bool seg_first = true;            // the segment holds this warp's first step
  bool seg_from_start = (st == 0);  // the segment began at step 0 of its tile

  // one chunk: tot += s (.) (W-chunk - z) x-chunk on the MMA
  auto chunk = [&](const uint4& wa, const uint4& wb, float sa, float sb, uint32_t za, uint32_t zb,
                   int kx) {
    const __nv_bfloat16* xb[MT];
#pragma unroll
    for (int tt = 0; tt < MT; ++tt) xb[tt] = xrow[tt] + kx;
    uint32_t xr[MT][kXR];
    if constexpr (kXS) {
      // row min(g8, M - 1), chunk kx / 128, this lane's 16 bytes of each word
      const uint32_t xa = smem_u32(xs) + (uint32_t)imin64(g8, M - 1) * xstride + (uint32_t)cq * 16 +
                          (uint32_t)(kx / kChunkK) * 256;
#pragma unroll
      for (int q = 0; q < kXR / 4; ++q) {
        const uint4 v = ld_shared_v4(xa + q * 64);
        xr[0][4 * q + 0] = v.x;
        xr[0][4 * q + 1] = v.y;
        xr[0][4 * q + 2] = v.z;
        xr[0][4 * q + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int tt = 0; tt < MT; ++tt) {
#pragma unroll
        for (int q = 0; q < kXR / 4; ++q) {
          const uint4 v = ld_global_nc_v4(xb[tt] + q * 8);
          if constexpr (F == Fmt::I8R) {
            xr[tt][4 * q + 0] = v.x;
            xr[tt][4 * q + 1] = v.y;
            xr[tt][4 * q + 2] = v.z;
            xr[tt][4 * q + 3] = v.w;
          } else {
            // word q of the piece holds elements 8q..8q+7: pairs (8q + j, 8q + j + 4)
            xr[tt][4 * q + 0] = __byte_perm(v.x, v.z, 0x5410);
            xr[tt][4 * q + 1] = __byte_perm(v.x, v.z, 0x7632);
            xr[tt][4 * q + 2] = __byte_perm(v.y, v.w, 0x5410);
            xr[tt][4 * q + 3] = __byte_perm(v.y, v.w, 0x7632);
          }
        }
      }
    }
    float acc[MT][2][4];
#pragma unroll
    for (int tt = 0; tt < MT; ++tt)
#pragma unroll
      for (int a = 0; a < 2; ++a) acc[tt][a][0] = acc[tt][a][1] = acc[tt][a][2] = acc[tt][a][3] = 0.0f;
    const uint32_t wA[4] = {wa.x, wa.y, wa.z, wa.w};
    const uint32_t wB[4] = {wb.x, wb.y, wb.z, wb.w};
    if constexpr (F == Fmt::I8R) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t ga[2], gb[2];
        i8x4_to_bf16x2(wA[i], ga);
        i8x4_to_bf16x2(wB[i], gb);
#pragma unroll
        for (int tt = 0; tt < MT; ++tt)
          mma_bf16_16816(acc[tt][i & 1], ga[0], gb[0], ga[1], gb[1], xr[tt][2 * i],
                         xr[tt][2 * i + 1]);
      }
    } else {
      auto mac = [&](auto big_tag, uint32_t zcA, uint32_t zcB, uint32_t zc2A, uint32_t zc2B) {
        constexpr bool kBig = decltype(big_tag)::value;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint32_t da[4], db[4];
          const uint32_t a = (F == Fmt::I4R) ? (wA[i] ^ 0x88888888u) : wA[i];
          const uint32_t b = (F == Fmt::I4R) ? (wB[i] ^ 0x88888888u) : wB[i];
          nib8_minus_zero<kBig>(a, zcA, zc2A, magic, da);
          nib8_minus_zero<kBig>(b, zcB, zc2B, magic, db);
#pragma unroll
          for (int tt = 0; tt < MT; ++tt) {
            mma_bf16_16816(acc[tt][0], da[0], db[0], da[1], db[1], xr[tt][4 * i],
                           xr[tt][4 * i + 1]);
            mma_bf16_16816(acc[tt][1], da[2], db[2], da[3], db[3], xr[tt][4 * i + 2],
                           xr[tt][4 * i + 3]);
          }
        }
      };
      if constexpr (F == Fmt::I4R) {
        // signed nibble v: (v ^ 8) = v + 8 in 0..15, zero point 8 (bf16 136)
        mac(std::false_type{}, 0x43084308u, 0x43084308u, 0u, 0u);
      } else if (__all_sync(0xffffffffu, ((za | zb) & 0x80u) == 0u)) {
        mac(std::false_type{}, 0x43004300u | (za * 0x00010001u), 0x43004300u | (zb * 0x00010001u),
            0u, 0u);
      } else {
        // zero points above 127: subtract 128 + min(z, 127), then max(z - 127, 0)
        const uint32_t zA1 = min(za, 127u), zB1 = min(zb, 127u);
        const uint32_t hA = __bfloat16_as_ushort(__float2bfloat16_rn((float)(za - zA1)));
        const uint32_t hB = __bfloat16_as_ushort(__float2bfloat16_rn((float)(zb - zB1)));
        mac(std::true_type{}, 0x43004300u | (zA1 * 0x00010001u), 0x43004300u | (zB1 * 0x00010001u),
            hA * 0x00010001u, hB * 0x00010001u);
      }
    }
#pragma unroll
    for (int tt = 0; tt < MT; ++tt) {
      tot[tt][0] = fmaf(sa, acc[tt][0][0] + acc[tt][1][0], tot[tt][0]);
      tot[tt][1] = fmaf(sa, acc[tt][0][1] + acc[tt][1][1], tot[tt][1]);
      tot[tt][2] = fmaf(sb, acc[tt][0][2] + acc[tt][1][2], tot[tt][2]);
      tot[tt][3] = fmaf(sb, acc[tt][0][3] + acc[tt][1][3], tot[tt][3]);
    }
  };

  // lane-constant offsets inside a stage: rows A / B, 16-byte units cq and 4 + cq, stored
  // at unit ^ (row mod 8) by the swizzle
  const uint32_t swz = (uint32_t)(g8 & 7);
  const uint32_t offA0 = g8 * 128 + (((uint32_t)cq ^ swz) << 4);
  const uint32_t offA1 = g8 * 128 + (((uint32_t)(4 + cq) ^ swz) << 4);
  const uint32_t w_base = smem_u32(wst), s_base = smem_u32(sst), z_base = smem_u32(zst);
  int stage = 0;
  uint32_t phase = 0;
  for (int u = 0; u < total; ++u) {
    if (!mbar_wait(bars + stage, phase)) {
      // the copy never completed: record it and give up on the warp's range (the
      // cluster barriers below are still reached by every thread).  Before leaving, wait
      // again (bounded) for every copy the warp has in flight: units u .. u + kS - 2,
      // the one that timed out included, so that no copy lands in shared memory after
      // the block may have exited.
      if (lane == 0) {
        set_dev_status(p.dev_status, WQ_DEV_TIMEOUT);
        for (int v = u; v < total && v <= u + kS - 2; ++v)
          (void)mbar_wait(bars + v % kS, (uint32_t)(v / kS) & 1u);
      }
      __syncwarp();
      break;
    }
    // codes of rows A (g8) and B (g8 + 8 = 1024 bytes further)
    const uint32_t wb = w_base + stage * kFactStageW;
    const uint4 a0 = ld_shared_v4(wb + offA0);
    const uint4 a1 = ld_shared_v4(wb + offA1);
    const uint4 b0 = ld_shared_v4(wb + offA0 + 8 * 128);
    const uint4 b1 = ld_shared_v4(wb + offA1 + 8 * 128);
    float sa0, sa1, sb0, sb1;
    uint32_t za0 = 0, za1 = 0, zb0 = 0, zb1 = 0;
    const uint32_t sv = s_base + stage * kFactStageS;
    if constexpr (F == Fmt::I4G) {
      const int g0 = (int)((st * 2 * kChunkK) >> gshift), g1 = (int)(((st * 2 + 1) * kChunkK) >> gshift);
      const uint32_t zv = z_base + stage * kFactStageZ;
      const uint32_t s0 = (uint32_t)(g0 & 3) * 4, s1 = (uint32_t)(g1 - (g0 & ~3)) * 4;
      const uint32_t z0 = (uint32_t)(g0 & 15), z1 = (uint32_t)(g1 - (g0 & ~15));
      sa0 = ld_shared_f32(sv + g8 * 16 + s0);
      sa1 = ld_shared_f32(sv + g8 * 16 + s1);
      sb0 = ld_shared_f32(sv + (g8 + 8) * 16 + s0);
      sb1 = ld_shared_f32(sv + (g8 + 8) * 16 + s1);
      za0 = ld_shared_u8(zv + g8 * 16 + z0);
      za1 = ld_shared_u8(zv + g8 * 16 + z1);
      zb0 = ld_shared_u8(zv + (g8 + 8) * 16 + z0);
      zb1 = ld_shared_u8(zv + (g8 + 8) * 16 + z1);
    } else {
      sa0 = sa1 = ld_shared_f32(sv + g8 * 4);
      sb0 = sb1 = ld_shared_f32(sv + (g8 + 8) * 4);
    }
    // every lane has its data: the stage consumed in the previous step is free again
    __syncwarp();
    if (lane == 0 && u + kS - 1 < total) issue(u + kS - 1);
    if (++stage == kS) {
      stage = 0;
      phase ^= 1u;
    }

    const int kx = (int)st * 2 * kChunkK;
    chunk(a0, b0, sa0, sb0, za0, zb0, kx);
    chunk(a1, b1, sa1, sb1, za1, zb1, kx + kChunkK);

    // ---- end of a segment: the tile ends here, or this warp's range does ----
    const bool tile_end = (st == spt - 1);
    if (tile_end || u + 1 == total) {
      if (seg_from_start && tile_end) {
        emit_tile(p, item, tiles, kBatch, tot, g8, cq);
      } else if (kPush && tile_end) {
        // this warp closes the tile: keep its own partial until the others' have arrived
#pragma unroll
        for (int tt = 0; tt < MT; ++tt)
#pragma unroll
          for (int i = 0; i < 4; ++i) ctot[tt][i] = tot[tt][i];
      } else if (kPush) {
        // a contributor: store the partial into the closing warp's receive slot
        if (!cl_waited) {
          cluster_wait_acquire();
          cl_waited = true;
        }
        const Split sp = split();
        const uint32_t t0 = item * spt, tl = t0 + spt - 1;
        uint32_t w0 = sp.wc;
        while (w0 > 0 && sp.bound(w0) > t0) --w0;
        uint32_t wcl = sp.wc;
        while (wcl + 1 < (uint32_t)kFactWarps && sp.bound(wcl + 1) <= tl) ++wcl;
        const uint32_t rank = wcl / kWarps, wl = wcl % kWarps;
        const uint32_t slot =
            smem_u32(recv) + ((wl * geo.cmax + (sp.wc - w0)) * 16u * (uint32_t)M) * 4u;
#pragma unroll
        for (int tt = 0; tt < MT; ++tt)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int col = tt * 8 + 2 * cq + (i & 1), row = g8 + ((i >> 1) << 3);
            if (col < M)
              st_shared_cluster_f32(map_shared_rank(slot + (uint32_t)(row * M + col) * 4u, rank),
                                    tot[tt][i]);
          }
        // every lane arrives (release, cluster scope) after its own stores: one arrival a
        // lane orders exactly that lane's stores, with no fence (measured cheaper than a
        // cluster fence a lane and one arrival a warp)
        mbar_arrive_remote(map_shared_rank(smem_u32(recvbar + wl), rank));
      } else {
        // a cut tile: park the partial; the warp holding the tile's last step (this
        // one, if the tile ends here) adds the partials up later
#pragma unroll
        for (int tt = 0; tt < MT; ++tt)
          *reinterpret_cast<float4*>(&s_part[warp][seg_first ? 0 : 1][lane][4 * tt]) =
              make_float4(tot[tt][0], tot[tt][1], tot[tt][2], tot[tt][3]);
        if (tile_end) close_item = (int)item;
      }
#pragma unroll
      for (int tt = 0; tt < MT; ++tt) tot[tt][0] = tot[tt][1] = tot[tt][2] = tot[tt][3] = 0.0f;
      seg_first = false;
      seg_from_start = true;
    }

    // ---- advance the main cursor ----
    if (++st == spt) {
      st = 0;
      ++item;
      if (u + 1 < total) set_xrow();
    }
  }
  }  // beg < end

  // ---- finish the cut tiles of the cluster ----
  if constexpr (kPush) {
    if (!cl_waited) cluster_wait_acquire();  // every thread passes the barrier once
    if (close_item >= 0) {
      // contributors w0 .. wc - 1 (in warp order; empty ranges add nothing), then this warp
      if (!mbar_wait_cluster(recvbar + warp, 0)) {
        set_dev_status(p.dev_status, WQ_DEV_TIMEOUT);
        return;
      }
      const Split sp = split();
      const uint32_t t0 = (uint32_t)close_item * spt;
      uint32_t w0 = sp.wc;
      while (w0 > 0 && sp.bound(w0) > t0) --w0;
      float tot[MT][4];
#pragma unroll
      for (int tt = 0; tt < MT; ++tt) tot[tt][0] = tot[tt][1] = tot[tt][2] = tot[tt][3] = 0.0f;
      const float* base = recv + (size_t)warp * geo.cmax * 16 * M;
      for (uint32_t w = w0; w < sp.wc; ++w) {
        if (!(sp.bound(w) < sp.bound(w + 1) && sp.bound(w + 1) > t0)) continue;
        const float* sl = base + (size_t)(w - w0) * 16 * M;
#pragma unroll
        for (int tt = 0; tt < MT; ++tt)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int col = tt * 8 + 2 * cq + (i & 1), row = g8 + ((i >> 1) << 3);
            if (col < M) tot[tt][i] += sl[row * M + col];
          }
      }
#pragma unroll
      for (int tt = 0; tt < MT; ++tt)
#pragma unroll
        for (int i = 0; i < 4; ++i) tot[tt][i] += ctot[tt][i];
      emit_tile(p, close_item, tiles, kBatch, tot, g8, cq);
    }
    return;
  }
  cluster_sync_all();
  if (close_item >= 0) {
    // contributors: the consecutive warps whose ranges meet the tile's units [t0, t1)
    const Split sp = split();
    const uint32_t t0 = (uint32_t)close_item * spt, t1 = t0 + spt;
    uint32_t w0 = sp.wc;
    while (w0 > 0 && sp.bound(w0) > t0) --w0;  // first warp whose range starts at or before t0
    float tot[MT][4];
#pragma unroll
    for (int tt = 0; tt < MT; ++tt) tot[tt][0] = tot[tt][1] = tot[tt][2] = tot[tt][3] = 0.0f;
    // four contributors at a time: their slots are read together, then added in order
    uint32_t bw = sp.bound(w0);
    for (uint32_t wb = w0; wb <= sp.wc; wb += 4) {
      float4 v[4][MT];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t w = wb + q;
        const uint32_t b0 = bw, b1 = (w <= sp.wc) ? sp.bound(w + 1) : b0;
        bw = b1;
        // empty ranges, and warps past the closer, add nothing
        const bool on = (w <= sp.wc) && b0 < b1 && b1 > t0 && b0 < t1;
        const int sid = (b0 >= t0) ? 0 : 1;  // the tile was the contributor's first segment?
        const uint32_t rank = w / kWarps, ww = w % kWarps;
#pragma unroll
        for (int tt = 0; tt < MT; ++tt)
          v[q][tt] = on ? ld_shared_cluster_f4(
                              map_shared_rank(smem_u32(&s_part[ww][sid][lane][4 * tt]), rank))
                        : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int tt = 0; tt < MT; ++tt) {
          tot[tt][0] += v[q][tt].x;
          tot[tt][1] += v[q][tt].y;
          tot[tt][2] += v[q][tt].z;
          tot[tt][3] += v[q][tt].w;
        }
    }
    emit_tile(p, close_item, tiles, kBatch, tot, g8, cq);
  }
  // no CTA leaves while another may still read its slots
  cluster_sync_all();
}

// The factored kernel takes I4G with a group of at least 128 codes, I4R and I8R when
// rows hold whole steps (two 64-byte chunks), there are at least 16 rows, the (item,
// step) units count in 31 bits, and the tensor maps' rules hold: 16-byte aligned bases,
// row strides a multiple of 16 bytes (for I4G zero points: K / G a multiple of 16).
bool fact_ok(Fmt f, const GemvParams& p) {
  const int64_t row_bytes = (f == Fmt::I8R) ? p.K : p.K / 2;
  if (row_bytes % (2 * kChunkBytes) != 0 || p.N < kRows) return false;
  const int64_t batch = (p.M <= 8) ? 8 : 16;
  const int64_t items = ((p.N + kRows - 1) / kRows) * ((p.M + batch - 1) / batch);
  if (items * (row_bytes / (2 * kChunkBytes)) >= (int64_t(1) << 31)) return false;
  if ((reinterpret_cast<uintptr_t>(p.w) | reinterpret_cast<uintptr_t>(p.scale)) % 16 != 0)
    return false;
  if (f == Fmt::I4G) {
    if (p.group < 128 || (p.K / p.group) % 16 != 0) return false;
    if (reinterpret_cast<uintptr_t>(p.zero) % 16 != 0) return false;
  }
  return true;
}

// ------------------------------------------------------------------ host side
namespace {

template <Fmt F, int MT, bool FMA>
cudaError_t launch_t(const GemvParams& p, int grid, cudaStream_t stream) {
  const size_t smem = (F == Fmt::MXFP4) ? sizeof(Routing) : 0;
  note_launch("k_gemv<%s,MT=%d,%s> grid=%d%s", fmt_name(F), MT, FMA ? "FMA" : "MMA", grid,
              p.ws_cnt ? " stream-K" : "");
  k_gemv<F, MT, FMA><<<grid, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

// The factored kernel runs in clusters of kFactCluster CTAs, as many clusters as fit on
// the GPU at once (one wave), never more than there are items.
template <Fmt F>
constexpr int kChunkK() { return chunk_k<F>(); }
constexpr int kFactMinSteps = 2;
constexpr int kMaxDevicesGemv = 64;

// Shared memory an SM offers blocks (sm_103a), and what the static partial slots of one
// block of the factored kernel take.
constexpr size_t kSmemPerSMFact = 228 * 1024;
constexpr size_t kFactStaticBytes = (size_t)kWarps * 2 * 32 * 4 * sizeof(float);

template <Fmt F, int MT, int kSD, bool kXS, bool kPush, int kCl>
cudaError_t launch_fact_t(const GemvParams& p, const FactMaps& maps, const FactGeom& geo,
                          size_t smem, int64_t clusters, int num_sms, cudaStream_t stream) {
  constexpr int kFactCluster = kCl;
  // co-resident clusters a device for the last dynamic shared-memory size (0: unknown)
  static int active[kMaxDevicesGemv] = {0};
  static size_t active_smem[kMaxDevicesGemv] = {0};
  static std::atomic<uint64_t> smem_set{0};  // devices whose limit is raised
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevicesGemv) dev = 0;
  const uint64_t bit = 1ull << dev;
  if (!(smem_set.load(std::memory_order_acquire) & bit)) {
    const cudaError_t e = cudaFuncSetAttribute(k_gemv_fact<F, MT, kSD, kXS, kPush, kCl>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)(kSmemPerSMFact / 2));
    if (e != cudaSuccess) return e;
    smem_set.fetch_or(bit, std::memory_order_acq_rel);
  }
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kFactCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // programmatic dependent launch: the prologue overlaps the previous kernel's tail; the
  // kernel waits for it (griddepcontrol.wait) before touching activations or outputs
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (active[dev] == 0 || active_smem[dev] != smem) {
    cfg.gridDim = dim3(kFactCluster * (unsigned)num_sms);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, k_gemv_fact<F, MT, kSD, kXS, kPush, kCl>, &cfg) != cudaSuccess ||
        n <= 0) {
      (void)cudaGetLastError();
      n = num_sms * kBlocksPerSM / kFactCluster;
    }
    active[dev] = n;
    active_smem[dev] = smem;
  }
  if (clusters > active[dev]) clusters = active[dev];  // one wave (the caller sized it)
  cfg.gridDim = dim3((unsigned)(std::max<int64_t>(1, clusters) * kFactCluster));
  cfg.numAttrs = 2;
  note_launch("k_gemv_fact<%s,MT=%d,stages=%d,%s,%s> grid=%u (%lld clusters of %d) smem=%zu",
              fmt_name(F), MT, kSD, kXS ? "x staged" : "x global", kPush ? "push fixup" : "barrier fixup",
              cfg.gridDim.x, (long long)std::max<int64_t>(1, clusters), kFactCluster, smem);
  return cudaLaunchKernelEx(&cfg, k_gemv_fact<F, MT, kSD, kXS, kPush, kCl>, p, maps, geo);
}

// Clusters of four for group-wise 4-bit at one batch with long rows, else two (the host
// split above was computed for the same size).
template <Fmt F, int MT, int kSD, bool kXS, bool kPush>
cudaError_t launch_fact_c(int cl, const GemvParams& p, const FactMaps& maps, const FactGeom& geo,
                          size_t smem, int64_t clusters, int num_sms, cudaStream_t stream) {
  if constexpr (F == Fmt::I4G && MT == 1) {
    if (cl == 4)
      return launch_fact_t<F, MT, kSD, kXS, kPush, 4>(p, maps, geo, smem, clusters, num_sms, stream);
  }
  return launch_fact_t<F, MT, kSD, kXS, kPush, 2>(p, maps, geo, smem, clusters, num_sms, stream);
}

// Ring depth and activation staging: four stages a warp; activations staged in shared
// memory (4-bit formats, up to 8 rows) when two blocks an SM still fit, with the ring cut
// to three stages if that is what makes them fit (K = 14336 at one row).
template <Fmt F, int MT>
cudaError_t launch_fact(const GemvParams& p, int num_sms, cudaStream_t stream) {
  // tensor maps of codes, scales and zero points
  FactMaps maps;
  const int64_t row_bytes = (F == Fmt::I8R) ? p.K : p.K / 2;
  if (!encode_tensor_map_2d(&maps.w, CU_TENSOR_MAP_DATA_TYPE_UINT8, const_cast<uint8_t*>(p.w),
                            (uint64_t)row_bytes, (uint64_t)p.N, (uint64_t)row_bytes, 2 * kChunkBytes,
                            kRows, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if constexpr (F == Fmt::I4G) {
    const uint64_t gpr = (uint64_t)(p.K / p.group);
    if (!encode_tensor_map_2d(&maps.s, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, const_cast<float*>(p.scale),
                              gpr, (uint64_t)p.N, gpr * 4, 4, kRows, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_tensor_map_2d(&maps.z, CU_TENSOR_MAP_DATA_TYPE_UINT8, const_cast<uint8_t*>(p.zero),
                              gpr, (uint64_t)p.N, gpr, 16, kRows, CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
  } else {
    const uint64_t stride = ((uint64_t)p.N * 4 + 15) & ~uint64_t(15);
    if (!encode_tensor_map_2d(&maps.s, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, const_cast<float*>(p.scale),
                              (uint64_t)p.N, 1, stride, kRows, 1, CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
    maps.z = maps.s;  // unused
  }
  // clusters: every co-resident one (two blocks an SM; the launch clamps to the figure the
  // occupancy query gives), but at least kFactMinSteps steps a warp on average (fewer,
  // fuller warps beat many idle ones), never more than there are items
  constexpr int64_t kBatch = 8 * MT;
  const int64_t items = ((p.N + kRows - 1) / kRows) * ((p.M + kBatch - 1) / kBatch);
  const int64_t spt = row_bytes / (2 * kChunkBytes);
  const int cl = (F == Fmt::I4G && MT == 1 && spt >= 32) ? 4 : 2;  // CTAs a cluster
  const int cl_log2 = cluster_warps_log2(cl);
  const int64_t cl_warps = (int64_t)cl * kWarps;
  int64_t cap = std::min<int64_t>((int64_t)num_sms * kBlocksPerSM / cl,
                                  std::max<int64_t>(1, items * spt / (cl_warps * kFactMinSteps)));
  if (const int64_t v = tuning(kKnobGemvClusters); v >= 1) cap = v;  // tuning and test knob
  const int64_t clusters = std::max<int64_t>(1, std::min<int64_t>(cap, items));
  // push fixup: receive slots a warp = the most warps any cut tile meets, from the same
  // split as the kernel (cluster c takes q or q + 1 items; warp w of a cluster starts at
  // unit (w * U) >> log2(warps a cluster))
  uint32_t cmax = 1;
  {
    const int64_t q = items / clusters;
    for (int64_t icnt = std::max<int64_t>(q, 1); icnt <= q + 1; ++icnt) {
      const uint64_t U = (uint64_t)(icnt * spt);
      auto bound = [&](uint64_t w) { return (w * U) >> cl_log2; };
      auto owner = [&](uint64_t u) {
        uint64_t w = 0;
        while (w + 1 < (uint64_t)cl_warps && bound(w + 1) <= u) ++w;
        return w;
      };
      for (int64_t t = 0; t < icnt; ++t) {
        const uint64_t w0 = owner((uint64_t)(t * spt)), w1 = owner((uint64_t)(t * spt + spt - 1));
        cmax = std::max<uint32_t>(cmax, (uint32_t)(w1 - w0 + 1));
      }
    }
  }
  const size_t ring4 = 1024 + (size_t)fact_ring_bytes(4), ring3 = 1024 + (size_t)fact_ring_bytes(3);
  const size_t recv = (size_t)kWarps * cmax * 16 * (size_t)p.M * 4 + kWarps * 8;
  // the push fixup pays where few warps share a tile (the closing warp waits for each in
  // turn); with many (long rows or small N) the cluster barriers do better, as measured
  const int64_t push_knob = tuning(kKnobGemvPush);  // test knob: 1 forces it, 2 disables it
  const bool push_ok = push_knob == 1 ? cmax <= 32 : (push_knob == 2 ? false : cmax <= 4);
  // two blocks an SM: (dynamic + static + the 1 KB the driver reserves) twice
  auto fits = [&](size_t dyn) { return 2 * (dyn + kFactStaticBytes + 1024) <= kSmemPerSMFact; };
  if constexpr (F != Fmt::I8R && MT == 1) {
    const bool x_ok = tuning(kKnobGemvXsmem) != 1 && p.K % kChunkK<F>() == 0 &&
                      (reinterpret_cast<uintptr_t>(p.x) % 16) == 0;
    const uint32_t xstride = (uint32_t)(p.M > 1 ? p.K * 2 + kFactXPad : p.K * 2);
    const size_t xbytes = ((size_t)p.M * xstride + 15) & ~size_t(15);
    const FactGeom geo{xstride, cmax};
    if (x_ok && push_ok && fits(ring4 + xbytes + recv))
      return launch_fact_c<F, MT, 4, true, true>(cl, p, maps, geo, ring4 + xbytes + recv, clusters, num_sms, stream);
    if (x_ok && push_ok && fits(ring3 + xbytes + recv))
      return launch_fact_c<F, MT, 3, true, true>(cl, p, maps, geo, ring3 + xbytes + recv, clusters, num_sms, stream);
    if (x_ok && fits(ring4 + xbytes))
      return launch_fact_c<F, MT, 4, true, false>(cl, p, maps, geo, ring4 + xbytes, clusters, num_sms, stream);
    if (x_ok && fits(ring3 + xbytes))
      return launch_fact_c<F, MT, 3, true, false>(cl, p, maps, geo, ring3 + xbytes, clusters, num_sms, stream);
  }
  const FactGeom geo{0, cmax};
  // activations read from global memory: an activation order is gathered first
  GemvParams q = p;
  if (q.order != nullptr) {
    if (q.xg == nullptr) return cudaErrorInvalidValue;
    const cudaError_t e = launch_gather_cols(q.x, q.order, q.M, q.K, q.xg, q.dev_status, stream);
    if (e != cudaSuccess) return e;
    q.x = q.xg;
    q.order = nullptr;
  }
  if (push_ok && fits(ring4 + recv))
    return launch_fact_c<F, MT, 4, false, true>(cl, q, maps, geo, ring4 + recv, clusters, num_sms, stream);
  return launch_fact_c<F, MT, 4, false, false>(cl, q, maps, geo, ring4, clusters, num_sms, stream);
}

// I4G with a group of at least 128 codes, I4R, I8R: the factored kernel (warp MMA,
// batches of 8 or 16 activation rows).  I4G with smaller groups and MXFP4: the exact
// kernel, on the FMA pipe for one or two rows and on the warp MMA for more.
template <Fmt F>
cudaError_t launch_f(const GemvParams& p, int64_t rows, int grid, int num_sms, cudaStream_t stream) {
  if constexpr (F != Fmt::MXFP4) {
    if (fact_ok(F, p) && tuning(kKnobDecode) != 2)
      return rows <= 8 ? launch_fact<F, 1>(p, num_sms, stream) : launch_fact<F, 2>(p, num_sms, stream);
  } else {
    // MXFP4: the TMA-ring cluster kernel (gemv_mx.cu) where its shape rules hold; it
    // writes the zero rows of out-of-range slots itself
    if (gemv_mx_ok(p) && tuning(kKnobDecode) != 2) {
      const cudaError_t e = launch_gemv_mx(p, num_sms, stream);
      if (e != cudaErrorNotSupported) return e;
    }
    // the exact kernel leaves them to a small kernel (y NULL in the combine form: only
    // the status bit)
    const cudaError_t e = launch_zero_bad_slots(p.experts, p.M * p.S, p.E, p.N, p.y, p.dev_status, stream);
    if (e != cudaSuccess) return e;
  }
  GemvParams q = p;
  if (q.order != nullptr) {  // the exact kernel reads activations from global memory
    if (q.xg == nullptr) return cudaErrorInvalidValue;
    const cudaError_t e = launch_gather_cols(q.x, q.order, q.M, q.K, q.xg, q.dev_status, stream);
    if (e != cudaSuccess) return e;
    q.x = q.xg;
    q.order = nullptr;
  }
  if (rows <= 1) return launch_t<F, 1, true>(q, grid, stream);
  if (rows <= 2) return launch_t<F, 2, true>(q, grid, stream);
  if (rows <= 8) return launch_t<F, 1, false>(q, grid, stream);
  return launch_t<F, 2, false>(q, grid, stream);
}

}  // namespace

namespace {
std::atomic<int> g_static_weights{0};
std::atomic<int64_t> g_tuning[kKnobCount] = {};
}  // namespace

int64_t tuning(int knob) {
  return (knob >= 0 && knob < kKnobCount) ? g_tuning[knob].load(std::memory_order_relaxed) : 0;
}
bool set_tuning(int knob, int64_t value) {
  if (knob < 0 || knob >= kKnobCount || value < 0) return false;
  g_tuning[knob].store(value, std::memory_order_relaxed);
  return true;
}

void set_static_weights(int on) { g_static_weights.store(on ? 1 : 0, std::memory_order_relaxed); }
int static_weights() { return g_static_weights.load(std::memory_order_relaxed); }

GemvPlan plan_gemv(Fmt f, int64_t M, int64_t N, int64_t K, int num_sms, int64_t batches) {
  GemvPlan pl;
  pl.num_sms = num_sms;
  const int ck = (f == Fmt::I8R) ? 64 : 128;
  pl.spt = (int)((K + ck - 1) / ck);  // chunks a tile
  pl.tiles = (int)((N + kRows - 1) / kRows);
  // MXFP4: every tile is streamed once for each routed-expert batch
  const int64_t work = (int64_t)pl.tiles * pl.spt * std::max<int64_t>(1, batches);
  int64_t blocks = (int64_t)num_sms * kBlocksPerSM;
  if (const int64_t v = tuning(kKnobGemvBlocks); v >= 1) blocks = v;  // tuning and test knob
  blocks = std::min<int64_t>(blocks, (work + kWarps * kMinChunks - 1) / (kWarps * kMinChunks));
  pl.grid = (int)std::max<int64_t>(1, blocks);
  // equal chunk shares need a workspace and a single activation batch
  pl.stream_k = (f != Fmt::MXFP4) && M <= 16;
  pl.ws_bytes = pl.stream_k ? ws_counter_bytes(pl.tiles) +
                                  (size_t)pl.grid * kWarps * 2 * (size_t)M * kRows * 4
                            : 0;
  return pl;
}

bool gemv_mxfp4_supported(int64_t R, int64_t S, int64_t E) {
  return R * S <= kMaxSlots && E <= kMaxExperts;
}

cudaError_t launch_gemv(Fmt f, GemvParams p, const GemvPlan& pl, cudaStream_t stream) {
  p.weights_static = static_weights();
  if (!pl.stream_k) {
    p.ws_cnt = nullptr;
    p.ws_part = nullptr;
  }
  // MXFP4: the rows of one expert batch are gathered, at most R*S of them
  const int64_t rows = (f == Fmt::MXFP4) ? std::min<int64_t>(p.M * p.S, 16) : p.M;
  switch (f) {
    case Fmt::I4G: return launch_f<Fmt::I4G>(p, rows, pl.grid, pl.num_sms, stream);
    case Fmt::I4R: return launch_f<Fmt::I4R>(p, rows, pl.grid, pl.num_sms, stream);
    case Fmt::I8R: return launch_f<Fmt::I8R>(p, rows, pl.grid, pl.num_sms, stream);
    case Fmt::MXFP4: return launch_f<Fmt::MXFP4>(p, rows, pl.grid, pl.num_sms, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace wq
