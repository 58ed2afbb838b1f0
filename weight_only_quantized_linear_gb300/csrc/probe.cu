// probe.cu -- two small kernels that are not part of the method: a bounded-wait probe
// (the failure path every kernel of the library takes when a wait gives up, exercised
// without any copy in flight) and a pure HBM read stream (the per-launch bandwidth a
// kernel that does nothing but read can reach, the ceiling the decode kernels are
// compared with).
#include <algorithm>
#include <atomic>

#include "common.cuh"
#include "launch.h"

namespace wq {

namespace {

// One thread block, one warp: an mbarrier that expects one arrival.  With `arrive` the
// warp arrives first and the wait succeeds at once; without it nobody ever arrives, the
// bounded wait gives up after `limit_ns`, and WQ_DEV_TIMEOUT is recorded.  No bulk copy,
// no cluster peer and no other warp is involved, so giving up leaves nothing in flight.
__global__ void k_wait_probe(uint64_t limit_ns, int arrive, int32_t* dev_status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && arrive) mbar_arrive(&bar);
  __syncwarp();
  const bool ok = mbar_wait_limit(&bar, 0, limit_ns);
  if (threadIdx.x == 0 && !ok) set_dev_status(dev_status, WQ_DEV_TIMEOUT);
}

// ---- read stream, plain loads: every thread keeps kUnroll 16-byte loads in flight
// (read-once, no L1 allocation) and folds them into one word; the word reaches memory
// only if it equals a value no input of the benchmark produces, which keeps the loads.
constexpr int kUnroll = 8;
__global__ void __launch_bounds__(256) k_stream_plain(const uint4* __restrict__ p, int64_t n16,
                                                      uint32_t* sink) {
  uint32_t acc = 0;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + (kUnroll - 1) * stride < n16; i += kUnroll * stride) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) v[u] = ld_global_stream_v4(p + i + u * stride);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
  }
  for (; i < n16; i += stride) {
    const uint4 v = ld_global_stream_v4(p + i);
    acc ^= v.x ^ v.y ^ v.z ^ v.w;
  }
  if (acc == 0x9E3779B9u) sink[0] = acc;
}

// ---- read stream, bulk-copy ring: one block an SM, each streaming a contiguous share
// of the buffer through a ring of kRingStages shared-memory stages filled by
// cp.async.bulk (one elected thread issues, four warps consume a word of every 16 bytes
// and release the stage).  Launched with programmatic dependent launch: the ring is
// filled before the dependency wait, as a decode kernel with immutable weights does, so
// the stream of one launch overlaps the tail of the previous one; the block takes under
// half of an SM, so the next launch's block fits beside it.
constexpr int kRingStages = 6;
constexpr int kRingBytes = 16384;
constexpr int kRingConsumers = 4;
constexpr int kRingThreads = 32 * (kRingConsumers + 1);

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                          uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__global__ void __launch_bounds__(kRingThreads, 1)
    k_stream_ring(const uint8_t* __restrict__ p, int64_t bytes, uint32_t* sink) {
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ uint64_t full[kRingStages], empty[kRingStages];
  grid_dep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // this block's share, in whole 16-byte units
  const int64_t n16 = bytes / 16;
  const int64_t b0 = n16 * blockIdx.x / gridDim.x * 16, b1 = n16 * (blockIdx.x + 1) / gridDim.x * 16;
  const int nst = (int)((b1 - b0 + kRingBytes - 1) / kRingBytes);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRingStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kRingConsumers);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (warp == kRingConsumers) {
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      auto issue = [&](int t) {
        const int s = t % kRingStages;
        const int64_t off = b0 + (int64_t)t * kRingBytes;
        const uint32_t len = (uint32_t)std::min<int64_t>(kRingBytes, b1 - off);
        mbar_arrive_expect_tx(&full[s], len);
        bulk_load(ring + s * kRingBytes, p + off, len, &full[s], pol);
      };
      // the buffer is never written: fill the ring before the dependency wait
      int t = 0;
      for (; t < kRingStages && t < nst; ++t) issue(t);
      grid_dep_wait();
      for (; t < nst; ++t) {
        const int s = t % kRingStages;
        if (!mbar_wait(&empty[s], (uint32_t)((t / kRingStages) - 1) & 1u)) {
          set_dev_status(nullptr, WQ_DEV_TIMEOUT);
          break;
        }
        issue(t);
      }
      // every issued copy has landed before the block may exit
      for (int u = std::max(0, t - kRingStages); u < t; ++u)
        (void)mbar_wait(&full[u % kRingStages], (uint32_t)(u / kRingStages) & 1u);
    }
    return;
  }
  grid_dep_wait();
  uint32_t acc = 0;
  for (int t = 0; t < nst; ++t) {
    const int s = t % kRingStages;
    if (!mbar_wait(&full[s], (uint32_t)(t / kRingStages) & 1u)) break;
    const int64_t off = b0 + (int64_t)t * kRingBytes;
    const int len = (int)std::min<int64_t>(kRingBytes, b1 - off);
    const uint32_t base = smem_u32(ring + s * kRingBytes);
    for (int o = (warp * 32 + lane) * 16; o < len; o += kRingConsumers * 32 * 16) {
      const uint4 v = ld_shared_v4(base + o);
      acc ^= v.x ^ v.y ^ v.z ^ v.w;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  if (acc == 0x9E3779B9u) sink[0] = acc;
}

}  // namespace

cudaError_t launch_wait_probe(uint64_t limit_ns, int arrive, int32_t* dev_status, cudaStream_t s) {
  k_wait_probe<<<1, 32, 0, s>>>(limit_ns, arrive, dev_status);
  return cudaGetLastError();
}

cudaError_t launch_stream_read(const void* buf, int64_t bytes, int variant, uint32_t* sink,
                               int num_sms, cudaStream_t s) {
  if (variant == 0) {
    const int64_t n16 = bytes / 16;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((int64_t)num_sms * 8, (n16 + 255) / 256));
    k_stream_plain<<<grid, 256, 0, s>>>(static_cast<const uint4*>(buf), n16, sink);
    return cudaGetLastError();
  }
  static std::atomic<uint64_t> attr_set{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const size_t smem = (size_t)kRingStages * kRingBytes;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_set.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(k_stream_ring, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set.fetch_or(bit, std::memory_order_release);
  }
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)std::max<int64_t>(1, std::min<int64_t>(num_sms, bytes / kRingBytes + 1)));
  cfg.blockDim = dim3(kRingThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_stream_ring, static_cast<const uint8_t*>(buf), bytes, sink);
}

}  // namespace wq
