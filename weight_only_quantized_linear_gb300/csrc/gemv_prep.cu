// gemv_prep.cu -- group-wise 4-bit weights repacked at load time ("Quantization" (Linnet
// docs), "Group-wise 4-bit weights": weights repacked at load, --prepare; "20.
// Quantization" (Inference Engineering book), "Speed needs a kernel": weight layouts
// pre-shuffled so that a 128-bit load fills a tensor-core fragment directly), and the
// decode kernel that streams that layout.
//
// The prepared copy holds the same codes, scales and zero points as the Int4GroupLinear
// layout, reordered so that everything one thread block consumes in one step is one
// contiguous run of bytes:
//   * stage (b, s) = rows 128b .. 128b + 127 and codes 256s .. 256s + 255 (b < ceil(N/128),
//     s < K/256): 16384 bytes of codes, then 1280 bytes of group parameters;
//   * codes: 128 rows x 8 units of 16 bytes.  Unit u = 4c + q of row r (chunk c of 128
//     codes, lane piece q) sits at unit position u ^ swz(r), swz(r) = 4 (r & 1) + ((r >> 1)
//     & 3): the 16-byte loads of one MMA row pair (rows r, r + 1 in the same quarter warp)
//     land on distinct banks.  Word i of unit (c, q) holds the codes 256s + 128c + 8(4i +
//     q) + j, j < 8, so that a lane's activation fragments are the consecutive 16-byte
//     units 16c + 4i + q of the activation slice; inside the word, nibble p holds code j =
//     2p for p < 4 and 2(p - 4) + 1 for p >= 4, so that the nibble unpack yields the pairs
//     (j, j + 1) in the order the MMA pairs activations;
//   * group parameters: 128 rows x (f32 scale of chunk 0, f32 scale of chunk 1), then 128
//     rows x (u8 zero point of chunk 0, u8 zero point of chunk 1);
//   * rows past N hold code 0, scale 0 and zero point 0 (they add nothing).
// One stage then arrives with two bulk copies (plus one 512-byte activation copy a row)
// instead of hundreds of tensor-map row requests, so the copy engine of an SM is never
// the bottleneck, also not while the next launch prefetches beside the running one.
//
// The decode kernel: thread blocks of one producer warp and eight consumer warps, sized
// for two blocks an SM; the producer fills a ring of stages with bulk copies (the weight
// stages before the dependency wait when the weights are declared immutable, the
// activation slices after it); the eight consumer warps take 16 rows each of every stage
// and compute the factored dot products of each 128-code chunk on the warp MMA,
// s * sum_k x[k] * (q[k] - z) with (q - z) exact in bf16x2; the (128-row block, k step)
// units are split into equal contiguous ranges (stream-K), and a row block cut between
// blocks is finished through the workspace by its last contributor, in block order.
#include <algorithm>
#include <atomic>
#include <type_traits>

#include "common.cuh"
#include "launch.h"

namespace wq {

namespace {

constexpr int kPW = 8;                    // consumer warps
constexpr int kPThreads = (kPW + 1) * 32; // and one producer warp
constexpr int kPRows = 128;               // weight rows a stage
constexpr int kPStepK = 256;              // codes a row a stage
constexpr uint32_t kPCode = 16384;        // code bytes a stage
constexpr uint32_t kPMeta = 1280;         // group-parameter bytes a stage
constexpr int kPMaxStages = 8;
constexpr uint32_t kPSmemHalf = 228u * 1024u / 2u - 1024u - 2u * kPMaxStages * 8u;
// bytes between the activation rows of a stage: 512 + 64, so that rows m and m + 1 sit
// four 16-byte units apart modulo 128 bytes (no bank conflicts between MMA columns)
constexpr uint32_t kPXPitch = 576;

__host__ __device__ __forceinline__ uint32_t prep_swz(uint32_t r) {
  return ((r & 1u) << 2) | ((r >> 1) & 3u);
}

struct PrepGeom {
  uint32_t ks;      // k steps a row block (K / 256)
  uint32_t rbs;     // row blocks
  uint32_t units;   // rbs * ks
  uint32_t whole;   // 1: ranges hold whole row blocks (no workspace)
  uint32_t stage;   // bytes a stage in shared memory
  uint32_t off_x;   // activation slice offset inside a stage
  uint32_t tx;      // bytes the copies of a stage complete
  uint32_t stages;
};

__device__ __forceinline__ uint32_t prep_bound(const PrepGeom& g, uint32_t c, uint32_t G) {
  return g.whole ? (uint32_t)((uint64_t)c * g.rbs / G) * g.ks : (uint32_t)((uint64_t)c * g.units / G);
}

__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// ------------------------------------------------------------------ the repack
// One thread a 16-byte unit of the prepared codes.
__global__ void k_prepare_codes(const uint8_t* __restrict__ packed, int64_t N, int64_t K,
                                uint32_t ks, uint8_t* __restrict__ out) {
  const int64_t unit = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t total = (int64_t)((N + kPRows - 1) / kPRows) * ks * kPRows * 8;
  if (unit >= total) return;
  const int64_t stage = unit / (kPRows * 8);
  const uint32_t r = (uint32_t)((unit / 8) % kPRows), pos = (uint32_t)(unit % 8);
  const uint32_t u = pos ^ prep_swz(r);  // logical unit stored at this position
  const uint32_t c = u >> 2, q = u & 3u;
  const int64_t rb = stage / ks, st = stage % ks;
  const int64_t n = rb * kPRows + r;
  uint32_t w[4] = {0u, 0u, 0u, 0u};
  if (n < N) {
    const uint8_t* row = packed + n * (K / 2);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t k0 = st * kPStepK + c * 128 + (int64_t)(4 * i + q) * 8;
      // codes k0 .. k0 + 7 in the public layout: four bytes, even code low
      const uint32_t src = *reinterpret_cast<const uint32_t*>(row + k0 / 2);
      uint32_t v = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t code = (src >> (4 * j)) & 0xFu;
        const int p = (j & 1) ? 4 + (j >> 1) : (j >> 1);  // nibble of code j
        v |= code << (4 * p);
      }
      w[i] = v;
    }
  }
  *reinterpret_cast<uint4*>(out + unit * 16) = make_uint4(w[0], w[1], w[2], w[3]);
}

// One thread a (stage, row): the two chunks' scales and zero points.
__global__ void k_prepare_meta(const float* __restrict__ scale, const uint8_t* __restrict__ zero,
                               int64_t N, int64_t K, int32_t gshift, uint32_t ks,
                               uint8_t* __restrict__ out) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t total = (int64_t)((N + kPRows - 1) / kPRows) * ks * kPRows;
  if (i >= total) return;
  const int64_t stage = i / kPRows;
  const uint32_t r = (uint32_t)(i % kPRows);
  const int64_t rb = stage / ks, st = stage % ks;
  const int64_t n = rb * kPRows + r;
  const int64_t gpr = K >> gshift;
  float s0 = 0.0f, s1 = 0.0f;
  uint32_t z0 = 0, z1 = 0;
  if (n < N) {
    const int64_t g0 = (st * kPStepK) >> gshift, g1 = (st * kPStepK + 128) >> gshift;
    s0 = scale[n * gpr + g0];
    s1 = scale[n * gpr + g1];
    z0 = zero[n * gpr + g0];
    z1 = zero[n * gpr + g1];
  }
  uint8_t* base = out + stage * kPMeta;
  *reinterpret_cast<float2*>(base + r * 8) = make_float2(s0, s1);
  *reinterpret_cast<uint16_t*>(base + 1024 + r * 2) = (uint16_t)(z0 | (z1 << 8));
}

}  // namespace

// ------------------------------------------------------------------ the decode kernel
// MT: groups of 8 activation rows; kX1: a single activation row.
template <int MT, bool kX1>
__global__ void __launch_bounds__(kPThreads, 2)
    k_gemv_prep(const GemvParams p, const uint8_t* __restrict__ prep, const PrepGeom g) {
  static_assert(!kX1 || MT == 1, "one activation row: one column group");
  extern __shared__ uint8_t ring_raw[];
  __shared__ uint64_t full[kPMaxStages], empty[kPMaxStages];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(ring_raw) + 127) &
                                             ~uintptr_t(127));
  // the next launch of the stream may start now: its blocks fit beside ours
  grid_dep_launch_dependents();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t G = gridDim.x, c = blockIdx.x;
  const uint32_t u0 = prep_bound(g, c, G), u1 = prep_bound(g, c + 1, G);
  const int n = (int)(u1 - u0);
  const int S = (int)g.stages;
  const int64_t M = p.M, N = p.N, K = p.K;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kPW);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kPW) {
    // ================= producer =================
    if (lane == 0 && n > 0) {
      const uint64_t pol_stream = l2_policy_evict_first();  // weights: read once
      const uint64_t pol_keep = l2_policy_evict_last();     // activations: reread
      const uint8_t* meta0 = prep + (size_t)g.units * kPCode;
      const uint8_t* xb = reinterpret_cast<const uint8_t*>(p.x);
      const uint32_t ring_s = smem_u32(ring);
      auto issue_w = [&](int t) {
        const int s = t % S;
        const size_t u = u0 + (uint32_t)t;  // stages are stored in unit order
        const uint32_t base = ring_s + (uint32_t)s * g.stage;
        mbar_arrive_expect_tx(&full[s], g.tx);
        bulk_g2s(base, prep + u * kPCode, kPCode, &full[s], pol_stream);
        bulk_g2s(base + kPCode, meta0 + u * kPMeta, kPMeta, &full[s], pol_stream);
      };
      auto issue_x = [&](int t) {
        const int s = t % S;
        const uint32_t st = (u0 + (uint32_t)t) % g.ks;
        const uint32_t dst = ring_s + (uint32_t)s * g.stage + g.off_x;
        for (int64_t m = 0; m < M; ++m)
          bulk_g2s(dst + (uint32_t)m * kPXPitch, xb + (m * K + (int64_t)st * kPStepK) * 2, kPStepK * 2,
                   &full[s], pol_keep);
      };
      const int pre = min(S, n);
      // the prepared weights only before the dependency wait, when declared immutable
      if (p.weights_static)
        for (int t = 0; t < pre; ++t) issue_w(t);
      grid_dep_wait();
      if (!p.weights_static)
        for (int t = 0; t < pre; ++t) issue_w(t);
      for (int t = 0; t < pre; ++t) issue_x(t);
      int t = pre;
      for (; t < n; ++t) {
        const int s = t % S;
        if (!mbar_wait(&empty[s], (uint32_t)((t / S) - 1) & 1u)) {
          set_dev_status(p.dev_status, WQ_DEV_TIMEOUT);
          break;
        }
        issue_w(t);
        issue_x(t);
      }
      // no copy may land after the block exits
      for (int v = max(0, t - S); v < t; ++v)
        (void)mbar_wait(&full[v % S], (uint32_t)(v / S) & 1u);
    }
    return;
  }

  // ================= consumers =================
  grid_dep_wait();
  const int g8 = lane >> 2, cq = lane & 3;
  const uint32_t magic = 0x43004300u | (uint32_t)(p.K >> 62);
  const uint32_t rowA = (uint32_t)(warp * 16 + g8);
  const uint32_t swz = prep_swz(rowA);  // rows A and A + 8 share it
  const uint32_t offA0 = rowA * 128 + ((((uint32_t)cq) ^ swz) << 4);
  const uint32_t offA1 = rowA * 128 + (((4u + (uint32_t)cq) ^ swz) << 4);
  const uint32_t ring_base = smem_u32(ring);
  // activation row of each MMA column group (rows past M are never stored)
  uint32_t xrow[MT];
#pragma unroll
  for (int tt = 0; tt < MT; ++tt)
    xrow[tt] = kX1 ? 0u : (uint32_t)min(tt * 8 + g8, (int)M - 1) * kPXPitch;

  float tot[MT][4];
#pragma unroll
  for (int tt = 0; tt < MT; ++tt) tot[tt][0] = tot[tt][1] = tot[tt][2] = tot[tt][3] = 0.0f;
  bool seg_first = true;
  uint32_t rb = u0 / g.ks, st = u0 - rb * g.ks;
  bool seg_from_start = (st == 0);
  int pend0 = -1, pend1 = -1;

  // chunk ch of a stage: tot += s (.) (W - z) x, four accumulator chains (one a word)
  auto chunk = [&](uint32_t xbase, int ch, const uint4& wa, const uint4& wb, float sa, float sb,
                   uint32_t za, uint32_t zb) {
    float acc[MT][4][4];
#pragma unroll
    for (int tt = 0; tt < MT; ++tt)
#pragma unroll
      for (int a = 0; a < 4; ++a) acc[tt][a][0] = acc[tt][a][1] = acc[tt][a][2] = acc[tt][a][3] = 0.0f;
    const uint32_t wA[4] = {wa.x, wa.y, wa.z, wa.w};
    const uint32_t wB[4] = {wb.x, wb.y, wb.z, wb.w};
    auto mac = [&](auto big_tag, uint32_t zcA, uint32_t zcB, uint32_t zc2A, uint32_t zc2B) {
      constexpr bool kBig = decltype(big_tag)::value;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t da[4], db[4];
        nib8_minus_zero<kBig>(wA[i], zcA, zc2A, magic, da);
        nib8_minus_zero<kBig>(wB[i], zcB, zc2B, magic, db);
#pragma unroll
        for (int tt = 0; tt < MT; ++tt) {
          // the activations of word i: 16-byte unit 16 ch + 4 i + cq of the slice
          const uint4 v = ld_shared_v4(xbase + xrow[tt] + (uint32_t)(16 * ch + 4 * i + cq) * 16u);
          mma_bf16_16816(acc[tt][i], da[0], db[0], da[1], db[1], v.x, v.y);
          mma_bf16_16816(acc[tt][i], da[2], db[2], da[3], db[3], v.z, v.w);
        }
      }
    };
    if (__all_sync(0xffffffffu, ((za | zb) & 0x80u) == 0u)) {
      mac(std::false_type{}, 0x43004300u | (za * 0x00010001u), 0x43004300u | (zb * 0x00010001u), 0u, 0u);
    } else {
      const uint32_t zA1 = min(za, 127u), zB1 = min(zb, 127u);
      const uint32_t hA = __bfloat16_as_ushort(__float2bfloat16_rn((float)(za - zA1)));
      const uint32_t hB = __bfloat16_as_ushort(__float2bfloat16_rn((float)(zb - zB1)));
      mac(std::true_type{}, 0x43004300u | (zA1 * 0x00010001u), 0x43004300u | (zB1 * 0x00010001u),
          hA * 0x00010001u, hB * 0x00010001u);
    }
#pragma unroll
    for (int tt = 0; tt < MT; ++tt)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float sum = (acc[tt][0][j] + acc[tt][1][j]) + (acc[tt][2][j] + acc[tt][3][j]);
        tot[tt][j] = fmaf(j < 2 ? sa : sb, sum, tot[tt][j]);
      }
  };

  auto emit = [&](uint32_t rbk) {
#pragma unroll
    for (int tt = 0; tt < MT; ++tt)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int64_t m = tt * 8 + 2 * cq + (i & 1);
        const int64_t nn = (int64_t)rbk * kPRows + warp * 16 + g8 + ((i >> 1) << 3);
        if (m < M && nn < N) {
          const float bias = p.bias ? __bfloat162float(p.bias[nn]) : 0.0f;
          p.y[m * N + nn] = __float2bfloat16_rn(tot[tt][i] + bias);
        }
      }
  };
  auto part_slot = [&](uint32_t cc, int slot) -> float* {
    return p.ws_part + ((size_t)(cc * 2 + slot) * kPW + warp) * (size_t)(M * 16);
  };

  bool aborted = false;
  for (int t = 0; t < n; ++t) {
    const int s = t % S;
    if (!mbar_wait(&full[s], (uint32_t)(t / S) & 1u)) {
      set_dev_status(p.dev_status, WQ_DEV_TIMEOUT);
      aborted = true;
      break;
    }
    const uint32_t base = ring_base + (uint32_t)s * g.stage;
    const uint4 a0 = ld_shared_v4(base + offA0);
    const uint4 a1 = ld_shared_v4(base + offA1);
    const uint4 b0 = ld_shared_v4(base + offA0 + 8 * 128);
    const uint4 b1 = ld_shared_v4(base + offA1 + 8 * 128);
    const float2 fa = ld_shared_f32x2(base + kPCode + rowA * 8);
    const float2 fb = ld_shared_f32x2(base + kPCode + (rowA + 8) * 8);
    const uint32_t ha = ld_shared_u16(base + kPCode + 1024 + rowA * 2);
    const uint32_t hb = ld_shared_u16(base + kPCode + 1024 + (rowA + 8) * 2);
    const uint32_t xbase = base + g.off_x;
    chunk(xbase, 0, a0, b0, fa.x, fb.x, ha & 0xFFu, hb & 0xFFu);
    chunk(xbase, 1, a1, b1, fa.y, fb.y, ha >> 8, hb >> 8);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);

    const bool last_step = (st == g.ks - 1);
    if (last_step || t == n - 1) {
      if (seg_from_start && last_step) {
        emit(rb);
      } else {
        float* dst = part_slot(c, seg_first ? 0 : 1);
#pragma unroll
        for (int tt = 0; tt < MT; ++tt)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int m = tt * 8 + 2 * cq + (i & 1);
            if (m < M) dst[m * 16 + g8 + ((i >> 1) << 3)] = tot[tt][i];
          }
        if (pend0 < 0) pend0 = (int)rb; else pend1 = (int)rb;
      }
#pragma unroll
      for (int tt = 0; tt < MT; ++tt) tot[tt][0] = tot[tt][1] = tot[tt][2] = tot[tt][3] = 0.0f;
      seg_first = false;
      seg_from_start = true;
    }
    if (++st == g.ks) {
      st = 0;
      ++rb;
    }
  }
  if (aborted) return;

  // ---- the cut row blocks: the last contributor adds the partials in block order ----
  for (int i = 0; i < 2; ++i) {
    const int pr = i == 0 ? pend0 : pend1;
    if (pr < 0) continue;
    const uint32_t rbk = (uint32_t)pr;
    const uint32_t tb = rbk * g.ks, te = tb + g.ks - 1;
    auto owner = [&](uint32_t u) {
      uint32_t cc = (uint32_t)((uint64_t)u * G / g.units);
      while (cc + 1 < G && prep_bound(g, cc + 1, G) <= u) ++cc;
      while (cc > 0 && prep_bound(g, cc, G) > u) --cc;
      return cc;
    };
    const uint32_t c0 = owner(tb), c1 = owner(te);
    const int slot0 = prep_bound(g, c0, G) < tb ? 1 : 0;
    const uint32_t tile = rbk * kPW + (uint32_t)warp;
    // the lanes' partial stores are ordered before lane 0's release by the warp barrier
    __syncwarp();
    int last = 0;
    if (lane == 0) last = (atom_add_acq_rel_gpu(&p.ws_cnt[tile], 1u) == c1 - c0) ? 1 : 0;
    last = __shfl_sync(0xffffffffu, last, 0);
    __syncwarp();  // the other lanes' reads below come after lane 0's acquire
    if (last) {
      for (int idx = lane; idx < M * 16; idx += 32) {
        const int m = idx >> 4, row = idx & 15;
        // each partial is cleared once read: the call leaves the workspace zero-filled
        float* src = part_slot(c0, slot0) + idx;
        float v = __ldcg(src);
        __stcg(src, 0.0f);
        for (uint32_t cc = c0 + 1; cc <= c1; ++cc) {
          src = part_slot(cc, 0) + idx;
          v += __ldcg(src);
          __stcg(src, 0.0f);
        }
        const int64_t nn = (int64_t)rbk * kPRows + warp * 16 + row;
        if (nn < N) {
          if (p.bias) v += __bfloat162float(p.bias[nn]);
          p.y[(int64_t)m * N + nn] = __float2bfloat16_rn(v);
        }
      }
      __syncwarp();
      if (lane == 0) p.ws_cnt[tile] = 0u;
    }
  }
}

// ------------------------------------------------------------------ host side
namespace {

struct PrepChoice {
  PrepGeom g{};
  int grid = 1;
  size_t smem = 0;
  size_t ws = 0;
};

PrepChoice prep_plan(int64_t M, int64_t N, int64_t K, int num_sms, bool split) {
  PrepChoice ch;
  PrepGeom& g = ch.g;
  g.ks = (uint32_t)(K / kPStepK);
  g.rbs = (uint32_t)((N + kPRows - 1) / kPRows);
  g.units = g.ks * g.rbs;
  g.whole = split ? 0u : 1u;
  g.off_x = kPCode + kPMeta;
  const uint32_t xbytes = M == 1 ? (uint32_t)kPStepK * 2u : (uint32_t)M * kPXPitch;
  g.stage = (g.off_x + xbytes + 127u) & ~127u;
  g.tx = kPCode + kPMeta + (uint32_t)M * kPStepK * 2u;
  g.stages = std::min<uint32_t>(kPMaxStages, (kPSmemHalf - 128u) / g.stage);
  ch.smem = 128 + (size_t)g.stages * g.stage;
  const int64_t items = split ? g.units : g.rbs;
  // two blocks an SM (every SM then gets the same share; with one an SM, two blocks of
  // the launch may still share an SM while another idles)
  const int64_t slots = (int64_t)num_sms * std::max<int64_t>(1, tuning(kKnobPrepBlocksPerSM) ?: 2);
  const int64_t per = (items + slots - 1) / slots;
  ch.grid = (int)std::max<int64_t>(1, (items + per - 1) / per);
  if (const int64_t v = tuning(kKnobGemvBlocks); v >= 1) ch.grid = (int)std::min<int64_t>(v, items);
  ch.ws = split ? ws_counter_bytes((int)(g.rbs * kPW)) + (size_t)ch.grid * 2 * kPW * (size_t)M * 16 * 4 : 0;
  return ch;
}

template <int MT, bool kX1>
cudaError_t launch_prep_t(const GemvParams& p, const uint8_t* prep, const PrepChoice& ch,
                          cudaStream_t stream) {
  static std::atomic<uint64_t> attr_set{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_set.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(k_gemv_prep<MT, kX1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kPSmemHalf);
    if (e != cudaSuccess) return e;
    attr_set.fetch_or(bit, std::memory_order_release);
  }
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ch.grid);
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = ch.smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = (tuning(kKnobPrep) & 1) ? 0 : 1;
  note_launch("k_gemv_prep<MT=%d%s> grid=%d stages=%u stage=%u B smem=%zu%s", MT, kX1 ? ",one row" : "",
              ch.grid, ch.g.stages, ch.g.stage, ch.smem, ch.g.whole ? " whole row blocks" : " stream-K");
  return cudaLaunchKernelEx(&cfg, k_gemv_prep<MT, kX1>, p, prep, ch.g);
}

}  // namespace

bool prep_shape_ok(int64_t M, int64_t N, int64_t K, int32_t group) {
  if (M < 1 || M > 16 || N < 1 || K < kPStepK || K % kPStepK != 0) return false;
  if (group < 128 || (group & (group - 1)) != 0 || K % group != 0) return false;
  return ((N + kPRows - 1) / kPRows) * (K / kPStepK) < (int64_t(1) << 30);
}

size_t prep_bytes(int64_t N, int64_t K) {
  const size_t stages = (size_t)((N + kPRows - 1) / kPRows) * (size_t)(K / kPStepK);
  return stages * (kPCode + kPMeta);
}

size_t prep_ws_bytes(int64_t M, int64_t N, int64_t K, int num_sms) {
  return prep_plan(M, N, K, num_sms, true).ws;
}

cudaError_t launch_prepare(const uint8_t* packed, const float* scale, const uint8_t* zero, int64_t N,
                           int64_t K, int32_t group, uint8_t* out, cudaStream_t s) {
  const uint32_t ks = (uint32_t)(K / kPStepK);
  const int64_t rbs = (N + kPRows - 1) / kPRows;
  const int64_t units = rbs * ks * kPRows * 8;
  k_prepare_codes<<<(unsigned)((units + 255) / 256), 256, 0, s>>>(packed, N, K, ks, out);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t rows = rbs * ks * kPRows;
  k_prepare_meta<<<(unsigned)((rows + 255) / 256), 256, 0, s>>>(scale, zero, N, K, __builtin_ctz(group), ks,
                                                               out + (size_t)rbs * ks * kPCode);
  return cudaGetLastError();
}

cudaError_t launch_prep(const GemvParams& p0, const uint8_t* prep, void* workspace, size_t ws_bytes,
                        int num_sms, cudaStream_t stream) {
  GemvParams p = p0;
  p.weights_static = (tuning(kKnobPrep) & 2) ? 0 : static_weights();
  const PrepChoice probe = prep_plan(p.M, p.N, p.K, num_sms, true);
  const bool split = workspace != nullptr && ws_bytes >= probe.ws &&
                     (reinterpret_cast<uintptr_t>(workspace) & 255) == 0;
  const PrepChoice ch = split ? probe : prep_plan(p.M, p.N, p.K, num_sms, false);
  p.ws_cnt = nullptr;
  p.ws_part = nullptr;
  if (split) {
    p.ws_cnt = static_cast<uint32_t*>(workspace);
    p.ws_part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                         ws_counter_bytes((int)(ch.g.rbs * kPW)));
  }
  if (p.M > 8) return launch_prep_t<2, false>(p, prep, ch, stream);
  if (p.M == 1) return launch_prep_t<1, true>(p, prep, ch, stream);
  return launch_prep_t<1, false>(p, prep, ch, stream);
}

}  // namespace wq
