// api.cu -- the extern "C" entry points of libwq (declared in include/wq.h).
//
// Host side only: argument validation (before anything is launched), the choice of
// regime (decode GEMV for few activation rows, tcgen05 GEMM for many), TMA descriptor
// encoding, workspace layout, and the launches on the caller's stream.  No entry point
// synchronizes, allocates device memory or throws.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "../../include/wq.h"
#include "common.cuh"
#include "launch.h"

namespace wq {

namespace {

constexpr int kMaxDevices = 64;

int num_sms_current() {
  static int cache[kMaxDevices] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return kNumSMsFallback;
  if (dev < 0 || dev >= kMaxDevices) return kNumSMsFallback;
  if (cache[dev] == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
      return kNumSMsFallback;
    cache[dev] = v;
  }
  return cache[dev];
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}


int run_gemv(Fmt f, GemvParams p, void* workspace, size_t ws_bytes, cudaStream_t stream) {
  const int64_t batches = (f == Fmt::MXFP4) ? std::min<int64_t>(p.M * p.S, p.E) : 1;
  GemvPlan pl = plan_gemv(f, p.M, p.N, p.K, num_sms_current(), batches);
  if (pl.stream_k) {
    if (workspace == nullptr || ws_bytes == 0) {
      pl.stream_k = false;  // whole tiles a warp: correct, less evenly balanced
      pl.ws_bytes = 0;
    } else {
      if (ws_bytes < pl.ws_bytes) return WQ_EWORKSPACE;
      if (!aligned(workspace, 256)) return WQ_EALIGN;
      p.ws_cnt = static_cast<uint32_t*>(workspace);
      p.ws_part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                           ws_counter_bytes(pl.tiles));
    }
  }
  return launch_gemv(f, p, pl, stream) == cudaSuccess ? WQ_OK : WQ_ECUDA;
}

size_t gemv_ws_bytes(Fmt f, int64_t M, int64_t N, int64_t K, int32_t group) {
  (void)group;
  return plan_gemv(f, M, N, K, num_sms_current()).ws_bytes;
}

int check_rows_common(const void* x, int64_t M, int64_t K, const void* w, const float* scale,
                      const void* bias, int64_t N, const void* y) {
  if (!x || !w || !scale || !y) return WQ_EINVAL;
  if (M <= 0 || N <= 0 || K <= 0) return WQ_EINVAL;
  if (M > (1 << 20) || N > (1 << 28) || K > (1 << 28)) return WQ_EUNSUPPORTED;
  if (!aligned(x, 16) || !aligned(w, 16) || !aligned(scale, 4) || !aligned(y, 2) ||
      (bias && !aligned(bias, 2)))
    return WQ_EALIGN;
  return WQ_OK;
}

thread_local char t_last_launch[256] = "none";

}  // namespace

void note_launch(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_last_launch, sizeof(t_last_launch), fmt, ap);
  va_end(ap);
}
const char* last_launch() { return t_last_launch; }

bool encode_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, void* base,
                          uint64_t inner, uint64_t outer, uint64_t row_stride_bytes,
                          uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_stride_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, dtype, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace wq

using namespace wq;

extern "C" {

WQ_API const char* wq_status_string(int status) {
  switch (status) {
    case WQ_OK: return "WQ_OK";
    case WQ_EINVAL: return "WQ_EINVAL: null pointer, non-positive size or unknown mode";
    case WQ_ESHAPE: return "WQ_ESHAPE: sizes break a layout rule";
    case WQ_EALIGN: return "WQ_EALIGN: pointer not aligned";
    case WQ_ERANGE: return "WQ_ERANGE: value outside the format's range";
    case WQ_EUNSUPPORTED: return "WQ_EUNSUPPORTED: request not implemented";
    case WQ_ECUDA: return "WQ_ECUDA: CUDA runtime call failed";
    case WQ_EWORKSPACE: return "WQ_EWORKSPACE: workspace too small";
    default: return "unknown wq status";
  }
}

WQ_API int wq_version(void) { return 100; }

WQ_API const char* wq_last_launch(void) { return last_launch(); }

WQ_API int wq_set_static_weights(int on) {
  set_static_weights(on);
  return WQ_OK;
}

WQ_API int wq_set_tuning(int32_t knob, int64_t value) {
  return set_tuning(knob, value) ? WQ_OK : WQ_EINVAL;
}

WQ_API int wq_test_wait_timeout(uint64_t limit_ns, int32_t arrive, int32_t* dev_status,
                                wq_stream_t stream) {
  if (limit_ns == 0 || limit_ns > 100000000ull) return WQ_EINVAL;
  return launch_wait_probe(limit_ns, arrive, dev_status, reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? WQ_OK
             : WQ_ECUDA;
}

WQ_API int wq_bench_stream_read(const void* buf, size_t bytes, int32_t variant, uint32_t* sink,
                                wq_stream_t stream) {
  if (!buf || !sink || bytes < 16) return WQ_EINVAL;
  if (variant != 0 && variant != 1) return WQ_EINVAL;
  if (!aligned(buf, 16) || !aligned(sink, 4)) return WQ_EALIGN;
  return launch_stream_read(buf, (int64_t)(bytes & ~size_t(15)), variant, sink, num_sms_current(),
                            reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? WQ_OK
             : WQ_ECUDA;
}

// ------------------------------------------------------------------ group-wise 4-bit
WQ_API size_t wq_linear_int4_groups_workspace(int64_t M, int64_t N, int64_t K, int32_t group) {
  if (M <= 0 || N <= 0 || K <= 0 || group <= 0) return 0;
  if (M > 16 && gemm_tc_supported(M, N, K, group)) return gemm_tc_ws_bytes(M, N, K, num_sms_current());
  if (M > 16) return 0;
  return gemv_ws_bytes(Fmt::I4G, M, N, K, group);
}

namespace {
size_t gather_bytes(int64_t M, int64_t K) { return ((size_t)M * (size_t)K * 2 + 255) & ~size_t(255); }
}  // namespace

WQ_API size_t wq_linear_int4_groups_ordered_workspace(int64_t M, int64_t N, int64_t K,
                                                      int32_t group) {
  if (M <= 0 || N <= 0 || K <= 0 || group <= 0) return 0;
  return gather_bytes(M, K) + wq_linear_int4_groups_workspace(M, N, K, group);
}

WQ_API int wq_linear_int4_groups(const void* x, int64_t M, int64_t K, const uint8_t* packed,
                                 const float* scale, const uint8_t* zero, const int32_t* order,
                                 const void* bias, int64_t N, int32_t group, void* y,
                                 void* workspace, size_t ws_bytes, int32_t* dev_status,
                                 wq_stream_t stream) {
  if (!zero) return WQ_EINVAL;
  int st = check_rows_common(x, M, K, packed, scale, bias, N, y);
  if (st != WQ_OK) return st;
  if (group != 32 && group != 64 && group != 128 && group != 256) return WQ_ESHAPE;
  if (K % group != 0) return WQ_ESHAPE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // activation order: the gathered copy of x takes the head of the workspace
  __nv_bfloat16* xg = nullptr;
  if (order != nullptr) {
    const size_t gx = gather_bytes(M, K);
    if (!aligned(order, 16)) return WQ_EALIGN;
    if (workspace == nullptr || ws_bytes < gx) return WQ_EWORKSPACE;
    if (!aligned(workspace, 256)) return WQ_EALIGN;
    xg = static_cast<__nv_bfloat16*>(workspace);
    workspace = static_cast<uint8_t*>(workspace) + gx;
    ws_bytes -= gx;
    if (ws_bytes == 0) workspace = nullptr;
  }

  if (M > 16 && gemm_tc_supported(M, N, K, group)) {
    if (order != nullptr) {
      if (launch_gather_cols(static_cast<const __nv_bfloat16*>(x), order, M, K, xg, dev_status, s) !=
          cudaSuccess)
        return WQ_ECUDA;
      x = xg;
    }
    GemmTcParams gp{static_cast<const __nv_bfloat16*>(x), M, N, K, packed, scale, zero, group,
                    static_cast<const __nv_bfloat16*>(bias), static_cast<__nv_bfloat16*>(y),
                    dev_status, nullptr, 1};
    // split-K when the caller's workspace holds the partials (optional: without it the
    // tiles run unsplit, with the same result up to f32 summation order)
    const size_t need = gemm_tc_ws_bytes(M, N, K, num_sms_current());
    if (need > 0 && workspace != nullptr && ws_bytes >= need) {
      if (!aligned(workspace, 16)) return WQ_EALIGN;
      gp.part = static_cast<float*>(workspace);
      gp.splits = gemm_tc_splits(M, N, K, num_sms_current());
    }
    return launch_gemm_tc(gp, num_sms_current(), s) == cudaSuccess ? WQ_OK : WQ_ECUDA;
  }

  GemvParams p{};
  p.x = static_cast<const __nv_bfloat16*>(x);
  p.w = packed;
  p.M = M;
  p.K = K;
  p.N = N;
  p.scale = scale;
  p.zero = zero;
  p.group = group;
  p.group_shift = __builtin_ctz((unsigned)group);
  p.bias = static_cast<const __nv_bfloat16*>(bias);
  p.y = static_cast<__nv_bfloat16*>(y);
  p.dev_status = dev_status;
  p.order = order;
  p.xg = xg;
  return run_gemv(Fmt::I4G, p, M <= 16 ? workspace : nullptr, ws_bytes, s);
}

// ------------------------------------------------------------------ prepared layout
WQ_API size_t wq_prepared_int4_groups_bytes(int64_t N, int64_t K, int32_t group) {
  if (!prep_shape_ok(1, N, K, group)) return 0;
  return prep_bytes(N, K);
}

WQ_API int wq_prepare_int4_groups(const uint8_t* packed, const float* scale, const uint8_t* zero,
                                  int64_t N, int64_t K, int32_t group, void* prepared,
                                  size_t prepared_bytes, wq_stream_t stream) {
  if (!packed || !scale || !zero || !prepared) return WQ_EINVAL;
  if (N <= 0 || K <= 0 || group <= 0) return WQ_EINVAL;
  if (!prep_shape_ok(1, N, K, group)) return WQ_EUNSUPPORTED;
  if (prepared_bytes < prep_bytes(N, K)) return WQ_EWORKSPACE;
  if (!aligned(packed, 4) || !aligned(scale, 4) || !aligned(prepared, 16)) return WQ_EALIGN;
  return launch_prepare(packed, scale, zero, N, K, group, static_cast<uint8_t*>(prepared),
                        reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? WQ_OK
             : WQ_ECUDA;
}

WQ_API size_t wq_linear_int4_groups_prepared_workspace(int64_t M, int64_t N, int64_t K,
                                                       int32_t group) {
  if (!prep_shape_ok(M, N, K, group)) return 0;
  return prep_ws_bytes(M, N, K, num_sms_current());
}

WQ_API int wq_linear_int4_groups_prepared(const void* x, int64_t M, int64_t K, const void* prepared,
                                          const void* bias, int64_t N, int32_t group, void* y,
                                          void* workspace, size_t ws_bytes, int32_t* dev_status,
                                          wq_stream_t stream) {
  if (!x || !prepared || !y) return WQ_EINVAL;
  if (M <= 0 || N <= 0 || K <= 0 || group <= 0) return WQ_EINVAL;
  if (!prep_shape_ok(M, N, K, group)) return M > 16 ? WQ_EUNSUPPORTED : WQ_ESHAPE;
  if (!aligned(x, 16) || !aligned(prepared, 16) || !aligned(y, 2) || (bias && !aligned(bias, 2)))
    return WQ_EALIGN;
  GemvParams p{};
  p.x = static_cast<const __nv_bfloat16*>(x);
  p.M = M;
  p.K = K;
  p.N = N;
  p.group = group;
  p.group_shift = __builtin_ctz((unsigned)group);
  p.bias = static_cast<const __nv_bfloat16*>(bias);
  p.y = static_cast<__nv_bfloat16*>(y);
  p.dev_status = dev_status;
  return launch_prep(p, static_cast<const uint8_t*>(prepared), workspace, ws_bytes, num_sms_current(),
                     reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? WQ_OK
             : WQ_ECUDA;
}

// ------------------------------------------------------------------ allocation-free variant
// Scratch for callers that cannot allocate device memory (see wq.h): one static array a
// GPU, its device address looked up once per device with cudaGetSymbolAddress (the
// host-side name of the array is only a stand-in and must never reach a kernel).  The
// set-up also clears the array once on the caller's stream; from then on every launch
// leaves its arrival counters at zero, so no per-call clearing stands between the
// previous kernel and the next launch.
static __device__ __align__(256) uint8_t g_noalloc_scratch[WQ_NOALLOC_SCRATCH_BYTES];

namespace {
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {nullptr};

int noalloc_scratch(void** out, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return WQ_ECUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return WQ_ECUDA;
    if (cudaMemsetAsync(p, 0, WQ_NOALLOC_SCRATCH_BYTES, stream) != cudaSuccess) return WQ_ECUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return WQ_OK;
}
}  // namespace

WQ_API int wq_linear_int4_groups_noalloc(const void* x, int64_t M, int64_t K,
                                         const uint8_t* packed, const float* scale,
                                         const uint8_t* zero, const int32_t* order,
                                         const void* bias, int64_t N, int32_t group, void* y,
                                         int32_t* dev_status, wq_stream_t stream) {
  if (order != nullptr) return WQ_EUNSUPPORTED;  // the gathered copy of x needs a workspace
  if (!zero) return WQ_EINVAL;
  int st = check_rows_common(x, M, K, packed, scale, bias, N, y);
  if (st != WQ_OK) return st;
  if (group != 32 && group != 64 && group != 128 && group != 256) return WQ_ESHAPE;
  if (K % group != 0) return WQ_ESHAPE;
  // the tensor-core regime needs no scratch (split-K is only an option there)
  if (M > 16 && gemm_tc_supported(M, N, K, group))
    return wq_linear_int4_groups(x, M, K, packed, scale, zero, order, bias, N, group, y,
                                 nullptr, 0, dev_status, stream);
  const size_t need = wq_linear_int4_groups_workspace(M, N, K, group);
  // shapes that run without scratch, and shapes whose split-K scratch would not fit the
  // array, take the launch without cross-block split-K (same result up to f32 order)
  if (need == 0 || need > WQ_NOALLOC_SCRATCH_BYTES)
    return wq_linear_int4_groups(x, M, K, packed, scale, zero, order, bias, N, group, y,
                                 nullptr, 0, dev_status, stream);
  void* scratch = nullptr;
  st = noalloc_scratch(&scratch, reinterpret_cast<cudaStream_t>(stream));
  if (st != WQ_OK) return st;
  return wq_linear_int4_groups(x, M, K, packed, scale, zero, order, bias, N, group, y, scratch,
                               need, dev_status, stream);
}

// ------------------------------------------------------------------ per-row int8 / int4
WQ_API size_t wq_linear_rows_workspace(int64_t M, int64_t N, int64_t K, int32_t bits) {
  if (M <= 0 || N <= 0 || K <= 0 || M > 16) return 0;
  return gemv_ws_bytes(bits == 8 ? Fmt::I8R : Fmt::I4R, M, N, K, 0);
}

WQ_API int wq_linear_int8_rows(const void* x, int64_t M, int64_t K, const int8_t* q,
                               const float* scale, const void* bias, int64_t N, void* y,
                               void* workspace, size_t ws_bytes, int32_t* dev_status,
                               wq_stream_t stream) {
  int st = check_rows_common(x, M, K, q, scale, bias, N, y);
  if (st != WQ_OK) return st;
  if (K % 16 != 0) return WQ_ESHAPE;
  GemvParams p{};
  p.x = static_cast<const __nv_bfloat16*>(x);
  p.w = reinterpret_cast<const uint8_t*>(q);
  p.M = M;
  p.K = K;
  p.N = N;
  p.scale = scale;
  p.bias = static_cast<const __nv_bfloat16*>(bias);
  p.y = static_cast<__nv_bfloat16*>(y);
  p.dev_status = dev_status;
  return run_gemv(Fmt::I8R, p, M <= 16 ? workspace : nullptr, ws_bytes,
                  reinterpret_cast<cudaStream_t>(stream));
}

WQ_API int wq_linear_int4_rows(const void* x, int64_t M, int64_t K, const int8_t* packed,
                               const float* scale, const void* bias, int64_t N, void* y,
                               void* workspace, size_t ws_bytes, int32_t* dev_status,
                               wq_stream_t stream) {
  int st = check_rows_common(x, M, K, packed, scale, bias, N, y);
  if (st != WQ_OK) return st;
  if (K % 32 != 0) return WQ_ESHAPE;
  GemvParams p{};
  p.x = static_cast<const __nv_bfloat16*>(x);
  p.w = reinterpret_cast<const uint8_t*>(packed);
  p.M = M;
  p.K = K;
  p.N = N;
  p.scale = scale;
  p.bias = static_cast<const __nv_bfloat16*>(bias);
  p.y = static_cast<__nv_bfloat16*>(y);
  p.dev_status = dev_status;
  return run_gemv(Fmt::I4R, p, M <= 16 ? workspace : nullptr, ws_bytes,
                  reinterpret_cast<cudaStream_t>(stream));
}

// ------------------------------------------------------------------ MXFP4 experts
WQ_API size_t wq_mxfp4_experts_shared_workspace(int64_t R, int64_t S, int64_t E, int64_t N,
                                                int64_t K) {
  if (R <= 0 || S <= 0 || E <= 0 || N <= 0 || K <= 0) return 0;
  // the grouped GEMM's routing tables and gathered rows (many routed slots); else none
  return gemm_mx_ok(R, S, E, N, K, nullptr, nullptr, nullptr) ? gemm_mx_ws_bytes(R * S, E, K) : 0;
}

namespace {
size_t round256(size_t v) { return (v + 255) & ~size_t(255); }

// The three MXFP4 expert products share the decode kernels: x_per_slot selects one input
// row a slot; with y32 the slot results stay f32 (times sw) for the combine step.  With
// many routed slots and the grouped GEMM's workspace (gws) they take the grouped GEMM.
int run_mxfp4(const void* x, int64_t R, int64_t K, const uint8_t* blocks, const uint8_t* scales,
              int64_t E, int64_t N, const int32_t* experts, int64_t S, void* y, float* y32,
              const float* sw, int x_per_slot, void* gws, size_t gws_bytes, int32_t* dev_status,
              cudaStream_t s) {
  // a workspace too small for the grouped GEMM leaves the decode kernels (when they take
  // the slot count)
  if (gws != nullptr && gemm_mx_ok(R, S, E, N, K, x, blocks, scales) &&
      gws_bytes >= gemm_mx_ws_bytes(R * S, E, K)) {
    if (!aligned(gws, 16)) return WQ_EALIGN;
    return launch_gemm_mx(static_cast<const __nv_bfloat16*>(x), R, S, x_per_slot, blocks, scales, E, N, K,
                          experts, static_cast<__nv_bfloat16*>(y), y32, sw, gws, dev_status, s) == cudaSuccess
               ? WQ_OK
               : WQ_ECUDA;
  }
  // the decode kernels' routing tables hold a bounded number of slots
  if (!gemv_mxfp4_supported(R, S, E))
    return gemm_mx_ok(R, S, E, N, K, x, blocks, scales) ? WQ_EWORKSPACE : WQ_EUNSUPPORTED;
  // slots whose expert index is out of range get zero rows of y (the combine step skips
  // them: only the status bit) from the decode path itself
  GemvParams p{};
  p.x = static_cast<const __nv_bfloat16*>(x);
  p.w = blocks;
  p.M = R;
  p.K = K;
  p.N = N;
  p.escale = scales;
  p.experts = experts;
  p.S = S;
  p.E = E;
  p.y = static_cast<__nv_bfloat16*>(y);
  p.y32 = y32;
  p.sw = sw;
  p.x_per_slot = x_per_slot;
  p.dev_status = dev_status;
  return run_gemv(Fmt::MXFP4, p, nullptr, 0, s);
}

int check_mxfp4(const void* x, int64_t R, int64_t K, const uint8_t* blocks, const uint8_t* scales,
                int64_t E, int64_t N, const int32_t* experts, int64_t S, const void* y) {
  if (!x || !blocks || !scales || !experts || !y) return WQ_EINVAL;
  if (R <= 0 || K <= 0 || E <= 0 || N <= 0 || S <= 0) return WQ_EINVAL;
  if (K % 32 != 0) return WQ_ESHAPE;
  if (E > 256 || E * N > (1 << 30) || K > (1 << 24) || R > (1 << 24) || S > (1 << 24)) return WQ_EUNSUPPORTED;
  if (!aligned(x, 16) || !aligned(blocks, 16) || !aligned(experts, 4) || !aligned(y, 2))
    return WQ_EALIGN;
  return WQ_OK;
}
}  // namespace

WQ_API int wq_mxfp4_experts_shared(const void* x, int64_t R, int64_t K, const uint8_t* blocks,
                                   const uint8_t* scales, int64_t E, int64_t N,
                                   const int32_t* experts, int64_t S, void* y, void* workspace,
                                   size_t ws_bytes, int32_t* dev_status, wq_stream_t stream) {
  int st = check_mxfp4(x, R, K, blocks, scales, E, N, experts, S, y);
  if (st != WQ_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return run_mxfp4(x, R, K, blocks, scales, E, N, experts, S, y, nullptr, nullptr, 0, workspace, ws_bytes,
                   dev_status, s);
}

WQ_API int wq_mxfp4_linear_experts_shared(const void* x, int64_t R, int64_t K,
                                          const uint8_t* blocks, const uint8_t* scales, int64_t E,
                                          int64_t N, const int32_t* experts, int64_t S, void* y,
                                          void* workspace, size_t ws_bytes, int32_t* dev_status,
                                          wq_stream_t stream) {
  return wq_mxfp4_experts_shared(x, R, K, blocks, scales, E, N, experts, S, y, workspace, ws_bytes,
                                 dev_status, stream);
}

WQ_API size_t wq_mxfp4_experts_workspace(int64_t R, int64_t S, int64_t E, int64_t N, int64_t K) {
  return wq_mxfp4_experts_shared_workspace(R, S, E, N, K);
}

WQ_API int wq_mxfp4_experts(const void* x, int64_t R, int64_t K, const uint8_t* blocks,
                            const uint8_t* scales, int64_t E, int64_t N, const int32_t* experts,
                            int64_t S, void* y, void* workspace, size_t ws_bytes,
                            int32_t* dev_status, wq_stream_t stream) {
  int st = check_mxfp4(x, R, K, blocks, scales, E, N, experts, S, y);
  if (st != WQ_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return run_mxfp4(x, R, K, blocks, scales, E, N, experts, S, y, nullptr, nullptr, 1, workspace, ws_bytes,
                   dev_status, s);
}

WQ_API size_t wq_mxfp4_combine_experts_workspace(int64_t R, int64_t S, int64_t E, int64_t N,
                                                 int64_t K) {
  if (R <= 0 || S <= 0 || N <= 0) return 0;
  const size_t y32 = (size_t)R * (size_t)S * (size_t)N * 4;
  // many routed slots: the f32 slot results, then the grouped GEMM's workspace
  if (E > 0 && K > 0 && gemm_mx_ok(R, S, E, N, K, nullptr, nullptr, nullptr))
    return round256(y32) + gemm_mx_ws_bytes(R * S, E, K);
  return y32;
}

WQ_API int wq_mxfp4_combine_experts(const void* x, int64_t R, int64_t K, const uint8_t* blocks,
                                    const uint8_t* scales, int64_t E, int64_t N,
                                    const int32_t* experts, int64_t S, const float* weights,
                                    void* y, void* workspace, size_t ws_bytes,
                                    int32_t* dev_status, wq_stream_t stream) {
  int st = check_mxfp4(x, R, K, blocks, scales, E, N, experts, S, y);
  if (st != WQ_OK) return st;
  if (!weights || !workspace) return WQ_EINVAL;
  if (ws_bytes < (size_t)R * (size_t)S * (size_t)N * 4) return WQ_EWORKSPACE;
  if (!aligned(weights, 4) || !aligned(workspace, 16)) return WQ_EALIGN;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  float* y32 = static_cast<float*>(workspace);
  const size_t y32_bytes = round256((size_t)R * (size_t)S * (size_t)N * 4);
  const bool grouped = ws_bytes > y32_bytes && gemm_mx_ok(R, S, E, N, K, x, blocks, scales);
  st = run_mxfp4(x, R, K, blocks, scales, E, N, experts, S, nullptr, y32, weights, 0,
                 grouped ? static_cast<uint8_t*>(workspace) + y32_bytes : nullptr,
                 grouped ? ws_bytes - y32_bytes : 0, dev_status, s);
  if (st != WQ_OK) return st;
  return launch_combine_slots(y32, experts, R, S, E, N, static_cast<__nv_bfloat16*>(y), s) ==
                 cudaSuccess
             ? WQ_OK
             : WQ_ECUDA;
}

// ------------------------------------------------------------------ quantize / pack
WQ_API int wq_quantize_groups(const float* w, int64_t N, int64_t K, int32_t group, int32_t bits,
                              int32_t mode, void* codes, float* scale, uint8_t* zero,
                              int32_t* dev_status, wq_stream_t stream) {
  if (!w || !codes || !scale) return WQ_EINVAL;
  if (N <= 0 || K <= 0 || group <= 0) return WQ_EINVAL;
  if (mode != WQ_SYM && mode != WQ_SYM_U4 && mode != WQ_ASYM) return WQ_EINVAL;
  if (mode == WQ_SYM_U4 && bits != 4) return WQ_EINVAL;
  if (bits < 2 || bits > 8) return WQ_EINVAL;
  if (mode != WQ_SYM && !zero) return WQ_EINVAL;
  if (!aligned(w, 4) || !aligned(scale, 4)) return WQ_EALIGN;
  return launch_quantize(w, N, K, group, bits, mode, codes, scale, zero, dev_status,
                         reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? WQ_OK
             : WQ_ECUDA;
}

WQ_API int wq_pack_int4(const void* codes, int64_t rows, int64_t cols, int32_t is_unsigned,
                        uint8_t* packed, int32_t* dev_status, wq_stream_t stream) {
  if (!codes || !packed) return WQ_EINVAL;
  if (rows <= 0 || cols <= 0) return WQ_EINVAL;
  if (cols % 2 != 0) return WQ_ESHAPE;
  return launch_pack(codes, rows, cols, is_unsigned, packed, dev_status,
                     reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? WQ_OK
             : WQ_ECUDA;
}

WQ_API int wq_unpack_int4(const uint8_t* packed, int64_t rows, int64_t cols, int32_t is_unsigned,
                          void* codes, wq_stream_t stream) {
  if (!codes || !packed) return WQ_EINVAL;
  if (rows <= 0 || cols <= 0) return WQ_EINVAL;
  if (cols % 2 != 0) return WQ_ESHAPE;
  return launch_unpack(packed, rows, cols, is_unsigned, codes,
                       reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? WQ_OK
             : WQ_ECUDA;
}

// ------------------------------------------------------------------ dequantize exports
WQ_API int wq_dequantize_int4_groups(const uint8_t* packed, const float* scale,
                                     const uint8_t* zero, int64_t N, int64_t K, int32_t group,
                                     void* w, wq_stream_t stream) {
  if (!packed || !scale || !zero || !w) return WQ_EINVAL;
  if (N <= 0 || K <= 0 || group <= 0) return WQ_EINVAL;
  if (group % 2 != 0 || K % group != 0) return WQ_ESHAPE;
  if (!aligned(scale, 4) || !aligned(w, 2)) return WQ_EALIGN;
  return launch_dequant_i4g(packed, scale, zero, N, K, group, w,
                            reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? WQ_OK
             : WQ_ECUDA;
}

WQ_API int wq_dequantize_int8_rows(const int8_t* q, const float* scale, int64_t N, int64_t K,
                                   void* w, wq_stream_t stream) {
  if (!q || !scale || !w) return WQ_EINVAL;
  if (N <= 0 || K <= 0) return WQ_EINVAL;
  if (!aligned(scale, 4) || !aligned(w, 2)) return WQ_EALIGN;
  return launch_dequant_i8r(q, scale, N, K, w, reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? WQ_OK
             : WQ_ECUDA;
}

WQ_API int wq_dequantize_int4_rows(const int8_t* packed, const float* scale, int64_t N,
                                   int64_t K, void* w, wq_stream_t stream) {
  if (!packed || !scale || !w) return WQ_EINVAL;
  if (N <= 0 || K <= 0) return WQ_EINVAL;
  if (K % 2 != 0) return WQ_ESHAPE;
  if (!aligned(scale, 4) || !aligned(w, 2)) return WQ_EALIGN;
  return launch_dequant_i4r(packed, scale, N, K, w, reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? WQ_OK
             : WQ_ECUDA;
}

WQ_API int wq_dequantize_mxfp4(const uint8_t* blocks, const uint8_t* scales, int64_t E,
                               int64_t N, int64_t K, void* w, wq_stream_t stream) {
  if (!blocks || !scales || !w) return WQ_EINVAL;
  if (E <= 0 || N <= 0 || K <= 0) return WQ_EINVAL;
  if (K % 32 != 0) return WQ_ESHAPE;
  if (!aligned(w, 2)) return WQ_EALIGN;
  return launch_dequant_mxfp4(blocks, scales, E, N, K, w,
                              reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? WQ_OK
             : WQ_ECUDA;
}

}  // extern "C"
