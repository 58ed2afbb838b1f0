// gemv_mx.cu -- MXFP4 mixture-of-experts decode on per-warp TMA rings in thread-block
// clusters.
//
// "Quantization" (Linnet docs), format table: mxfp4_experts_shared(x, blocks, scales,
// experts) multiplies each routed row by the experts its `experts` row names,
// mxfp4_experts gives every slot its own input row, mxfp4_combine_experts adds the slot
// results with their routing weights; "MXFP4 experts": E2M1 codes in blocks of 32 along
// K with one E8M0 scale byte a block, and the work grouped by expert.  The same page's
// "2. Principles" (MXFP4) gives the element: E2M1 value times 2^(scale - 127).
//
// Work: the routed slots are sorted by expert (stable) and cut into batches of at most
// eight (the eight MMA columns); an item is a batch and one 16-row tile of its expert's
// weights, a step 128 bytes of each of the tile's rows (256 codes).  As in the cluster
// kernel of the affine formats (gemv.cu), a cluster takes a contiguous range of items,
// its warps split the range's (item, step) units evenly, and tiles cut between warps are
// finished inside the cluster through distributed shared memory.  One CTA of 16 warps an
// SM, in clusters of two: with two CTAs of 8 warps an SM, the warps of one CTA ran ahead
// of the other's (by 15 us of a 79 us launch at eight routed rows, measured on GB300), and
// the SM finished the slower CTA's work with half its warps.
//
// Loads: each warp streams its units through its own ring of stages filled by TMA (a
// {128 bytes, 16 rows} box of the experts' codes stacked as [E * N rows, K / 2 bytes],
// 128-byte swizzle).  The E8M0 scale rows (K / 32 bytes, not a multiple of 16 in general)
// have no tensor map: a tile's 16 rows of scales are contiguous, so one bulk copy brings
// them into one of two tile buffers of the warp, on the barrier of the tile's first
// stage.  Activation rows are staged once a block in shared memory in the MMA fragment
// order, zero past K, when they fit; otherwise read from global memory.
//
// Dequantization, exact: a code (s, e1 e0, m) with its sign in bf16 bit 15 and e1 e0 m in
// bits 8..6 is the bf16 E2M1 * 2^-126 (the subnormal codes included); one packed bf16
// multiply by 2^(scale - 1) gives E2M1 * 2^(scale - 127), exactly the f32 product rounded
// once to bf16 as the definition does.  Scales above 128 (2^(scale - 1) past the bf16
// range) and the NaN scale 255 take two multiplies (by 2^126, then by the E8M0 value).
// Codes j and j + 4 of a word form one bf16x2 pair, the pairing of the group-wise kernels,
// so activations are staged in the same permuted order.
//
// Slots whose expert index lies outside [0, E) are left out of the routing tables; the
// grid writes their rows of y as zeros and sets WQ_DEV_BAD_EXPERT.

#include <algorithm>
#include <atomic>

#include "common.cuh"
#include "launch.h"

namespace wq {
namespace {

constexpr int kMxWarps = 16;
constexpr int kMxThreads = kMxWarps * 32;
constexpr int kMxCluster = 2;     // CTAs a cluster
constexpr int kMxClWarpsLog2 = 5; // log2(warps a cluster)
static_assert(kMxCluster * kMxWarps == (1 << kMxClWarpsLog2), "warps a cluster: a power of two");
constexpr int kMxRows = 16;        // weight rows a tile
constexpr int kMxStepBytes = 128;  // code bytes of a row a step (256 codes)
constexpr int kMxStageW = kMxRows * kMxStepBytes;
constexpr int kMxBatch = 8;        // routed slots an item (MMA columns)
constexpr int64_t kMxMaxSlots = 1024;
constexpr int64_t kMxMaxExperts = 256;
constexpr int64_t kMxMaxK = 8192;

struct MxGeom {
  uint32_t tiles;      // N / 16
  uint32_t spt;        // steps a tile: ceil(K / 256)
  uint32_t kb;         // scale bytes a row: K / 32
  uint32_t sbuf;       // bytes of a tile's scales: 16 * K / 32
  uint32_t xrows;      // activation rows staged (kXS)
  uint32_t xstride;    // bytes between staged activation rows
  uint32_t pairs_max;  // capacity of the batch tables
  uint32_t off_sbuf, off_bars, off_x, off_route;  // offsets in dynamic shared memory
};

template <int kS, bool kXS>
__global__ void __launch_bounds__(kMxThreads, 1)
    k_gemv_mx(const GemvParams p, const __grid_constant__ CUtensorMap wmap, const MxGeom g) {
  // partial D fragments of cut tiles: [warp][first / last segment][lane][4]
  __shared__ __align__(16) float s_part[kMxWarps][2][32][4];
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  grid_dep_launch_dependents();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tid = threadIdx.x;
  const int g8 = lane >> 2;  // MMA row group: tile rows g8 and g8 + 8
  const int cq = lane & 3;   // 16-byte piece of a 64-byte chunk: one MXFP4 block
  const int64_t N = p.N, K = p.K;
  const int E = (int)p.E;
  const int RS = (int)(p.M * p.S);
  const uint32_t spt = g.spt, tiles = g.tiles, kb = g.kb;

  uint8_t* const wst = smem + warp * kS * kMxStageW;
  const uint32_t sbuf0 = smem_u32(smem + g.off_sbuf) + (uint32_t)warp * 2u * g.sbuf;
  uint64_t* const bars = reinterpret_cast<uint64_t*>(smem + g.off_bars) + warp * kS;
  uint8_t* const xs = smem + g.off_x;
  int* const route = reinterpret_cast<int*>(smem + g.off_route);
  // routing tables: npairs; slot counts, first sorted slot and first batch of each expert;
  // expert, first sorted slot and count of each batch; expert of each slot; sorted slots
  int* const ecnt = route + 1;
  int* const ebase = ecnt + (E + 1);
  int* const pbase = ebase + (E + 1);
  int* const pexp = pbase + (E + 1);
  int* const pstart = pexp + g.pairs_max;
  int* const pcnt = pstart + g.pairs_max;
  int* const eidx = pcnt + g.pairs_max;
  int* const sorted = eidx + RS;

  if (lane == 0) {
    for (int i = 0; i < kS; ++i) mbar_init(bars + i, 1);
    fence_mbar_init();
  }
  for (int e = tid; e <= E; e += kMxThreads) ecnt[e] = 0;

  // activation rows in the MMA fragment order ([row][k / 128][(k / 8) % 4][(k / 32) % 4]
  // 16-byte pieces of pairs (x0, x4) (x1, x5) (x2, x6) (x3, x7)), zero from K to the end
  // of the last step: pieces base + q * kMxThreads + tid, loaded, then stored
  const uint32_t k8n = (uint32_t)(K / 8), k8p = spt * 32u;
  const uint32_t xtotal = kXS ? g.xrows * k8p : 0u;
  auto x_load = [&](uint32_t base, uint4 (&v)[8]) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const uint32_t idx = base + q * kMxThreads + tid;
      v[q] = make_uint4(0, 0, 0, 0);
      if (idx < xtotal) {
        const uint32_t m = idx / k8p, k8 = idx - m * k8p;
        if (k8 < k8n) v[q] = ld_global_nc_v4(p.x + (int64_t)m * K + (int64_t)k8 * 8);
      }
    }
  };
  auto x_store = [&](uint32_t base, const uint4 (&v)[8]) {
    const uint32_t xbase = smem_u32(xs);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const uint32_t idx = base + q * kMxThreads + tid;
      if (idx < xtotal) {
        const uint32_t m = idx / k8p, k8 = idx - m * k8p;
        const uint32_t o0 = __byte_perm(v[q].x, v[q].z, 0x5410), o1 = __byte_perm(v[q].x, v[q].z, 0x7632);
        const uint32_t o2 = __byte_perm(v[q].y, v[q].w, 0x5410), o3 = __byte_perm(v[q].y, v[q].w, 0x7632);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                         xbase + m * g.xstride + (k8 >> 4) * 256 + (k8 & 3) * 64 + ((k8 >> 2) & 3) * 16),
                     "r"(o0), "r"(o1), "r"(o2), "r"(o3)
                     : "memory");
      }
    }
  };

  // expert indices and activations come from earlier kernels: the first activation
  // pieces are in flight while the routing is built
  grid_dep_wait();
  uint4 xv0[8];
  if constexpr (kXS) x_load(0, xv0);
  __syncthreads();

  // ---- routing: a stable sort of the slots by expert, batches of kMxBatch ----
  for (int i = tid; i < RS; i += kMxThreads) {
    const int e = __ldg(p.experts + i);
    eidx[i] = e;
    if (e >= 0 && e < E) atomicAdd(&ecnt[e], 1);
  }
  __syncthreads();
  if (warp == 0) {
    // exclusive prefix sums over the experts of slot and batch counts; lane l takes
    // experts [l * per, (l + 1) * per)
    const int per = (E + 31) / 32;
    int s_sum = 0, p_sum = 0;
    for (int j = 0; j < per; ++j) {
      const int e = lane * per + j;
      if (e < E) {
        s_sum += ecnt[e];
        p_sum += (ecnt[e] + kMxBatch - 1) / kMxBatch;
      }
    }
    int s_inc = s_sum, p_inc = p_sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a = __shfl_up_sync(0xffffffffu, s_inc, o), b = __shfl_up_sync(0xffffffffu, p_inc, o);
      if (lane >= o) {
        s_inc += a;
        p_inc += b;
      }
    }
    int s_run = s_inc - s_sum, p_run = p_inc - p_sum;
    for (int j = 0; j < per; ++j) {
      const int e = lane * per + j;
      if (e < E) {
        ebase[e] = s_run;
        pbase[e] = p_run;
        s_run += ecnt[e];
        p_run += (ecnt[e] + kMxBatch - 1) / kMxBatch;
      }
    }
    if (lane == 31) route[0] = p_inc;
  }
  __syncthreads();
  for (int i = tid; i < RS; i += kMxThreads) {
    const int e = eidx[i];
    if (e >= 0 && e < E) {
      int rank = 0;  // slots of the same expert before slot i
      for (int j = 0; j < i; ++j) rank += (eidx[j] == e) ? 1 : 0;
      sorted[ebase[e] + rank] = i;
    }
  }
  for (int e = tid; e < E; e += kMxThreads) {
    const int cnt = ecnt[e];
    for (int b = 0; b * kMxBatch < cnt; ++b) {
      const int pi = pbase[e] + b;
      pexp[pi] = e;
      pstart[pi] = ebase[e] + b * kMxBatch;
      pcnt[pi] = min(kMxBatch, cnt - b * kMxBatch);
    }
  }

  if constexpr (kXS) {
    x_store(0, xv0);
    for (uint32_t base = 8 * kMxThreads; base < xtotal; base += 8 * kMxThreads) {
      uint4 v[8];
      x_load(base, v);
      x_store(base, v);
    }
  }
  __syncthreads();

  // slots whose expert index lies outside [0, E): the status bit, and zero rows of y
  // (the combine form only skips them), spread over the grid
  if (ebase[E - 1] + ecnt[E - 1] < RS) {
    if (blockIdx.x == 0 && tid == 0) set_dev_status(p.dev_status, WQ_DEV_BAD_EXPERT);
    if (p.y != nullptr) {
      const int64_t total = (int64_t)RS * N;
      for (int64_t i = (int64_t)blockIdx.x * kMxThreads + tid; i < total; i += (int64_t)gridDim.x * kMxThreads) {
        const int e = eidx[i / N];
        if (e < 0 || e >= E) p.y[i] = __float2bfloat16_rn(0.0f);
      }
    }
  }

  const uint32_t npairs = (uint32_t)route[0];
  const uint32_t items = npairs * tiles;
  if (items == 0) return;  // every slot's expert out of range (the same in every CTA)

  // this cluster's items and units; warp wc of the cluster's 64 takes units
  // [bound(wc), bound(wc + 1))
  const uint32_t ncl = cluster_count_x(), cid = cluster_id_x();
  const uint32_t qi = items / ncl, ri = items - qi * ncl;
  const uint32_t ibeg = cid * qi + min(cid, ri), icnt = qi + (cid < ri ? 1u : 0u);
  const uint32_t u0 = ibeg * spt, U = icnt * spt;
  const uint32_t wc = cluster_ctarank() * kMxWarps + warp;
  auto bound = [&](uint32_t w) -> uint32_t {
    return u0 + (uint32_t)(((uint64_t)w * U) >> kMxClWarpsLog2);
  };
  const uint32_t beg = bound(wc), end = bound(wc + 1);
  const int total = beg < end ? (int)(end - beg) : 0;

  // ---- producer side: lane 0 fills stage (u mod kS) with unit beg + u ----
  const uint64_t pol = l2_policy_evict_first();
  uint32_t i_item = beg / spt;
  uint32_t i_st = beg - i_item * spt;
  uint32_t i_tiles = 0;  // tiles whose scales this warp has requested
  auto issue = [&](int u) {
    const uint32_t pr = i_item / tiles, tile = i_item - pr * tiles;
    const int32_t row0 = pexp[pr] * (int32_t)N + (int32_t)(tile * kMxRows);
    const bool new_tile = (i_st == 0) || (u == 0);
    const int stage = u % kS;
    uint64_t* bar = bars + stage;
    mbar_arrive_expect_tx(bar, kMxStageW + (new_tile ? g.sbuf : 0u));
    tma_load_2d(wst + stage * kMxStageW, &wmap, bar, (int32_t)(i_st * kMxStepBytes), row0, pol);
    if (new_tile) {
      bulk_g2s(sbuf0 + (i_tiles & 1u) * g.sbuf, p.escale + (int64_t)row0 * kb, g.sbuf, bar, pol);
      ++i_tiles;
    }
    if (++i_st == spt) {
      i_st = 0;
      ++i_item;
    }
  };
  if (lane == 0) {
    tma_prefetch_desc(&wmap);
    for (int u = 0; u < kS - 1 && u < total; ++u) issue(u);
  }
  __syncwarp();

  int close_item = -1;  // the cut tile this warp finishes after the cluster barrier
  if (total > 0) {
    uint32_t item = beg / spt;
    uint32_t st = beg - item * spt;
    uint32_t c_tiles = 0;  // tiles whose scales this warp has consumed
    uint32_t sb = sbuf0;   // scale rows of the current tile
    // the activation row of this lane's MMA column (g8) in the current item; a column
    // past the batch reads the batch's first row (its results are not stored)
    uint32_t xa = 0;
    const __nv_bfloat16* xg = nullptr;
    auto set_item = [&]() {
      const uint32_t pr = item / tiles;
      const int m = (g8 < pcnt[pr]) ? g8 : 0;
      const int slot = sorted[pstart[pr] + m];
      const int xrow = p.x_per_slot ? slot : slot / (int)p.S;
      if constexpr (kXS)
        xa = smem_u32(xs) + (uint32_t)xrow * g.xstride + (uint32_t)cq * 16;
      else
        xg = p.x + (int64_t)xrow * K;
    };
    set_item();
    float acc[2][4];
#pragma unroll
    for (int a = 0; a < 2; ++a) acc[a][0] = acc[a][1] = acc[a][2] = acc[a][3] = 0.0f;
    bool seg_first = true;            // the segment holds this warp's first unit
    bool seg_from_start = (st == 0);  // the segment began at step 0 of its tile

    // one output tile's D fragment: rows g8, g8 + 8; columns 2 cq, 2 cq + 1 (slots)
    auto emit = [&](uint32_t it, const float (&t)[4]) {
      const uint32_t pr = it / tiles, tile = it - pr * tiles;
      const int cnt = pcnt[pr], s0 = pstart[pr];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int m = 2 * cq + (i & 1);
        const int64_t n = (int64_t)tile * kMxRows + g8 + ((i >> 1) << 3);
        if (m < cnt) {
          const int slot = sorted[s0 + m];
          if (p.y32 != nullptr)
            p.y32[(int64_t)slot * N + n] = p.sw ? t[i] * __ldg(p.sw + slot) : t[i];
          else
            p.y[(int64_t)slot * N + n] = __float2bfloat16_rn(t[i]);
        }
      }
    };

    const uint32_t swz = (uint32_t)(g8 & 7);
    const uint32_t offA0 = g8 * 128 + (((uint32_t)cq ^ swz) << 4);
    const uint32_t offA1 = g8 * 128 + (((uint32_t)(4 + cq) ^ swz) << 4);
    const uint32_t w_base = smem_u32(wst);
    int stage = 0;
    uint32_t phase = 0;
    for (int u = 0; u < total; ++u) {
      if (!mbar_wait(bars + stage, phase)) {
        // the copy never completed: record it and give up on the warp's range; first wait
        // (bounded) for the copies still in flight, units u .. u + kS - 2, so that none
        // lands in shared memory after the block may have exited
        if (lane == 0) {
          set_dev_status(p.dev_status, WQ_DEV_TIMEOUT);
          for (int v = u; v < total && v <= u + kS - 2; ++v)
            (void)mbar_wait(bars + v % kS, (uint32_t)(v / kS) & 1u);
        }
        __syncwarp();
        break;
      }
      if (st == 0 || u == 0) {
        sb = sbuf0 + (c_tiles & 1u) * g.sbuf;
        ++c_tiles;
      }
      const uint32_t wb = w_base + stage * kMxStageW;
      const uint4 a0 = ld_shared_v4(wb + offA0);
      const uint4 a1 = ld_shared_v4(wb + offA1);
      const uint4 b0 = ld_shared_v4(wb + offA0 + 8 * 128);
      const uint4 b1 = ld_shared_v4(wb + offA1 + 8 * 128);
      // this lane's blocks: cq of chunk 2 st and of chunk 2 st + 1; a block past K (zero
      // codes from the zero-filled box) takes scale byte 127
      const uint32_t j0 = st * 8u + (uint32_t)cq, j1 = j0 + 4u;
      const uint32_t ea0 = j0 < kb ? ld_shared_u8(sb + g8 * kb + j0) : 127u;
      const uint32_t ea1 = j1 < kb ? ld_shared_u8(sb + g8 * kb + j1) : 127u;
      const uint32_t eb0 = j0 < kb ? ld_shared_u8(sb + (g8 + 8) * kb + j0) : 127u;
      const uint32_t eb1 = j1 < kb ? ld_shared_u8(sb + (g8 + 8) * kb + j1) : 127u;
      // activations of the two chunks, pieces q = 0..3 (pairs of words 2q .. of the block)
      uint4 xv[2][4];
      if constexpr (kXS) {
        const uint32_t xo = xa + st * 512u;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          xv[0][q] = ld_shared_v4(xo + q * 64);
          xv[1][q] = ld_shared_v4(xo + 256 + q * 64);
        }
      } else {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int64_t k0 = (int64_t)(2 * st + c) * 128 + cq * 32;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 v = make_uint4(0, 0, 0, 0);
            if (k0 + q * 8 < K) v = ld_global_nc_v4(xg + k0 + q * 8);
            xv[c][q] = make_uint4(__byte_perm(v.x, v.z, 0x5410), __byte_perm(v.x, v.z, 0x7632),
                                  __byte_perm(v.y, v.w, 0x5410), __byte_perm(v.y, v.w, 0x7632));
          }
        }
      }
      // every lane has its data: the stage consumed in the previous step is free again
      __syncwarp();
      if (lane == 0 && u + kS - 1 < total) issue(u + kS - 1);
      if (++stage == kS) {
        stage = 0;
        phase ^= 1u;
      }

      auto mac = [&](auto two_tag, uint32_t sA0, uint32_t sA1, uint32_t sB0, uint32_t sB1, uint32_t tA0,
                     uint32_t tA1, uint32_t tB0, uint32_t tB1) {
        constexpr bool kTwo = decltype(two_tag)::value;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const uint4 wa = c ? a1 : a0, wbv = c ? b1 : b0;
          const uint32_t wA[4] = {wa.x, wa.y, wa.z, wa.w};
          const uint32_t wB[4] = {wbv.x, wbv.y, wbv.z, wbv.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint32_t da[4], db[4];
            e2m1x8_scaled<kTwo>(wA[i], c ? sA1 : sA0, c ? tA1 : tA0, da);
            e2m1x8_scaled<kTwo>(wB[i], c ? sB1 : sB0, c ? tB1 : tB0, db);
            mma_bf16_16816(acc[0], da[0], db[0], da[1], db[1], xv[c][i].x, xv[c][i].y);
            mma_bf16_16816(acc[1], da[2], db[2], da[3], db[3], xv[c][i].z, xv[c][i].w);
          }
        }
      };
      if (__all_sync(0xffffffffu, max(max(ea0, ea1), max(eb0, eb1)) <= 128u)) {
        mac(std::false_type{}, pow2_em1_bf16x2(ea0), pow2_em1_bf16x2(ea1), pow2_em1_bf16x2(eb0),
            pow2_em1_bf16x2(eb1), 0u, 0u, 0u, 0u);
      } else {
        const uint32_t c126 = 0x7E807E80u;  // bf16x2 (2^126, 2^126)
        mac(std::true_type{}, c126, c126, c126, c126, e8m0_bf16x2(ea0), e8m0_bf16x2(ea1),
            e8m0_bf16x2(eb0), e8m0_bf16x2(eb1));
      }

      // ---- end of a segment: the tile ends here, or this warp's range does ----
      const bool tile_end = (st == spt - 1);
      if (tile_end || u + 1 == total) {
        float t[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          t[i] = acc[0][i] + acc[1][i];
          acc[0][i] = acc[1][i] = 0.0f;
        }
        if (seg_from_start && tile_end) {
          emit(item, t);
        } else {
          // a cut tile: park the partial; the warp holding the tile's last step adds the
          // partials up after the cluster barrier
          *reinterpret_cast<float4*>(&s_part[warp][seg_first ? 0 : 1][lane][0]) =
              make_float4(t[0], t[1], t[2], t[3]);
          if (tile_end) close_item = (int)item;
        }
        seg_first = false;
        seg_from_start = true;
      }
      if (++st == spt) {
        st = 0;
        ++item;
        if (u + 1 < total) set_item();
      }
    }

    // ---- the cut tile this warp closes ----
    cluster_sync_all();
    if (close_item >= 0) {
      // contributors: the consecutive warps whose ranges meet the tile's units [t0, t1),
      // added in warp order (deterministic); a contributor's segment of the tile is its
      // first one when its range starts inside the tile
      const uint32_t t0 = (uint32_t)close_item * spt, t1 = t0 + spt;
      uint32_t w0 = wc;
      while (w0 > 0 && bound(w0) > t0) --w0;
      float t[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      for (uint32_t w = w0; w <= wc; ++w) {
        const uint32_t b0 = bound(w), b1 = bound(w + 1);
        if (!(b0 < b1 && b1 > t0 && b0 < t1)) continue;
        const int sid = (b0 >= t0) ? 0 : 1;
        const float4 v = ld_shared_cluster_f4(
            map_shared_rank(smem_u32(&s_part[w % kMxWarps][sid][lane][0]), w / kMxWarps));
        t[0] += v.x;
        t[1] += v.y;
        t[2] += v.z;
        t[3] += v.w;
      }
      emit((uint32_t)close_item, t);
    }
  } else {
    cluster_sync_all();
  }
  // no CTA leaves while another may still read its partials
  cluster_sync_all();
}

// Dynamic shared memory of one launch: the rings, the tile-scale buffers, the barriers,
// the staged activations and the routing tables (plus slack for the 1024-byte alignment).
struct MxLayout {
  MxGeom g;
  size_t bytes;
};
MxLayout mx_layout(const GemvParams& p, int kS, uint32_t xrows, uint32_t xstride) {
  MxLayout L{};
  MxGeom& g = L.g;
  g.tiles = (uint32_t)(p.N / kMxRows);
  g.spt = (uint32_t)((p.K + 255) / 256);
  g.kb = (uint32_t)(p.K / 32);
  g.sbuf = (uint32_t)(p.K / 2);
  g.xrows = xrows;
  g.xstride = xstride;
  const int64_t RS = p.M * p.S;
  g.pairs_max = (uint32_t)(std::min<int64_t>(p.E, RS) + RS / kMxBatch + 1);
  size_t off = (size_t)kMxWarps * kS * kMxStageW;
  g.off_sbuf = (uint32_t)off;
  off += (size_t)kMxWarps * 2 * g.sbuf;
  off = (off + 15) & ~size_t(15);
  g.off_bars = (uint32_t)off;
  off += (size_t)kMxWarps * kS * 8;
  off = (off + 15) & ~size_t(15);
  g.off_x = (uint32_t)off;
  off += (size_t)xrows * xstride;
  off = (off + 15) & ~size_t(15);
  g.off_route = (uint32_t)off;
  off += 4 * (1 + 3 * ((size_t)p.E + 1) + 3 * (size_t)g.pairs_max + 2 * (size_t)RS);
  L.bytes = 1024 + off;
  return L;
}

constexpr size_t kMxSmemPerSM = 228 * 1024;
constexpr size_t kMxSmemPerBlock = 227 * 1024;
constexpr size_t kMxStaticBytes = (size_t)kMxWarps * 2 * 32 * 4 * sizeof(float);
// one block an SM: dynamic + static + the 1 KB the driver reserves
bool mx_fits(size_t dyn) { return dyn + kMxStaticBytes + 1024 <= kMxSmemPerSM && dyn + kMxStaticBytes <= kMxSmemPerBlock; }

template <int kS, bool kXS>
cudaError_t launch_mx_t(const GemvParams& p, const CUtensorMap& wmap, const MxLayout& L, int num_sms,
                        cudaStream_t stream) {
  static std::atomic<uint64_t> smem_set{0};  // devices whose limit is raised
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  const uint64_t bit = 1ull << dev;
  if (!(smem_set.load(std::memory_order_acquire) & bit)) {
    const cudaError_t e = cudaFuncSetAttribute(k_gemv_mx<kS, kXS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)(kMxSmemPerBlock - kMxStaticBytes));
    if (e != cudaSuccess) return e;
    smem_set.fetch_or(bit, std::memory_order_acq_rel);
  }
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kMxCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kMxThreads);
  cfg.dynamicSmemBytes = L.bytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(kMxCluster * (unsigned)num_sms);
  int active = 0;
  if (cudaOccupancyMaxActiveClusters(&active, k_gemv_mx<kS, kXS>, &cfg) != cudaSuccess || active <= 0) {
    (void)cudaGetLastError();
    active = num_sms / kMxCluster;
  }
  // every co-resident cluster (one CTA on every SM), but at least two steps a warp on
  // average for the largest routing the launch can see
  const int64_t units_max = (int64_t)L.g.pairs_max * L.g.tiles * L.g.spt;
  int64_t clusters = std::min<int64_t>((int64_t)active,
                                       std::max<int64_t>(1, units_max / (kMxCluster * kMxWarps * 2)));
  if (const int64_t v = tuning(kKnobGemvClusters); v >= 1) clusters = std::min<int64_t>(v, active);
  clusters = std::max<int64_t>(1, clusters);
  cfg.gridDim = dim3((unsigned)(clusters * kMxCluster));
  cfg.numAttrs = 2;
  note_launch("k_gemv_mx<stages=%d,%s> grid=%u (%lld clusters of %d) smem=%zu", kS,
              kXS ? "x staged" : "x global", cfg.gridDim.x, (long long)clusters, kMxCluster, L.bytes);
  return cudaLaunchKernelEx(&cfg, k_gemv_mx<kS, kXS>, p, wmap, L.g);
}

}  // namespace

bool gemv_mx_ok(const GemvParams& p) {
  const int64_t RS = p.M * p.S;
  if (p.N % kMxRows != 0 || p.K % 32 != 0 || p.K < 3 * 256 || p.K > kMxMaxK) return false;
  if (RS > kMxMaxSlots || p.E > kMxMaxExperts || p.E * p.N >= (int64_t(1) << 30)) return false;
  if ((reinterpret_cast<uintptr_t>(p.w) | reinterpret_cast<uintptr_t>(p.escale) |
       reinterpret_cast<uintptr_t>(p.x)) % 16 != 0)
    return false;
  const int64_t pairs = std::min<int64_t>(p.E, RS) + RS / kMxBatch + 1;
  return pairs * (p.N / kMxRows) * ((p.K + 255) / 256) < (int64_t(1) << 31);
}

cudaError_t launch_gemv_mx(const GemvParams& p, int num_sms, cudaStream_t stream) {
  CUtensorMap wmap;
  if (!encode_tensor_map_2d(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, const_cast<uint8_t*>(p.w),
                            (uint64_t)(p.K / 2), (uint64_t)(p.E * p.N), (uint64_t)(p.K / 2),
                            kMxStepBytes, kMxRows, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  // activations staged when the block still fits (a four-, else three-stage ring)
  const uint32_t xrows = (uint32_t)(p.x_per_slot ? p.M * p.S : p.M);
  const uint32_t kpad = (uint32_t)(((p.K + 255) / 256) * 256);
  const uint32_t xstride = kpad * 2 + (xrows > 1 ? 64u : 0u);
  if (tuning(kKnobGemvXsmem) != 1) {
    const MxLayout L4 = mx_layout(p, 4, xrows, xstride);
    if (mx_fits(L4.bytes)) return launch_mx_t<4, true>(p, wmap, L4, num_sms, stream);
    const MxLayout L3 = mx_layout(p, 3, xrows, xstride);
    if (mx_fits(L3.bytes)) return launch_mx_t<3, true>(p, wmap, L3, num_sms, stream);
  }
  const MxLayout L = mx_layout(p, 4, 0, 0);
  if (!mx_fits(L.bytes)) return cudaErrorNotSupported;
  return launch_mx_t<4, false>(p, wmap, L, num_sms, stream);
}

}  // namespace wq
