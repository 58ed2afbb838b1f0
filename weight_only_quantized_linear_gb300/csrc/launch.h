// launch.h -- internal interface between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace wq {

// Storage formats of the decode GEMV.
enum class Fmt { I4G, I4R, I8R, MXFP4 };
constexpr const char* fmt_name(Fmt f) {
  return f == Fmt::I4G ? "I4G" : (f == Fmt::I4R ? "I4R" : (f == Fmt::I8R ? "I8R" : "MXFP4"));
}

struct GemvParams {
  const __nv_bfloat16* x;  // activations [M, K] (MXFP4: [R, K])
  const uint8_t* w;        // packed weights / codes, rows of K/2 (int8: K) bytes
  int64_t M;               // activation rows (MXFP4: R)
  int64_t K;
  int64_t N;               // output columns (rows of one weight matrix)
  const float* scale;      // I4G [N, K/G]; I4R / I8R [N]
  const uint8_t* zero;     // I4G [N, K/G]
  const uint8_t* escale;   // MXFP4 E8M0 scales [E, N, K/32]
  int32_t group;           // I4G group size
  int32_t group_shift;     // log2(group)
  const int32_t* experts;  // MXFP4 [R, S]
  int64_t S;               // MXFP4 slots per row
  int64_t E;               // MXFP4 experts
  const __nv_bfloat16* bias;
  __nv_bfloat16* y;        // [M, N] (MXFP4: [R * S, N])
  // MXFP4 only: x holds one row a slot ([R * S, K], mxfp4_experts) instead of one a
  // routed row ([R, K]); and, when y32 is set, every slot's f32 result times its weight
  // sw[slot] (1 without sw) goes to y32 [R * S, N] instead of y (mxfp4_combine_experts)
  int32_t x_per_slot;
  float* y32;
  const float* sw;
  // I4G activation order (i32 [K]) or NULL; xg: scratch of M * K bf16 for the gathered
  // activations of launches that do not gather while staging
  const int32_t* order;
  __nv_bfloat16* xg;
  float* ws_part;          // stream-K partial tiles [warps, 2, M, 16 rows]
  uint32_t* ws_cnt;        // stream-K arrival counters [tiles]
  int32_t* dev_status;
  int32_t weights_static;  // the caller promises the weights are not written meanwhile
};

struct GemvPlan {
  int num_sms = 152;      // SMs of the current device (queried)
  int grid = 1;           // thread blocks (a few an SM)
  int tiles = 1;          // 16-row weight tiles
  int spt = 1;            // 64-byte column chunks a tile
  bool stream_k = false;  // equal chunk ranges a warp; needs a workspace
  size_t ws_bytes = 0;
};

// Workspace layout of stream-K launches: arrival counters (one a tile, zero between
// calls) rounded up to 256 bytes, then the f32 partial tiles [warps, 2, M, 16].
inline size_t ws_counter_bytes(int tiles) { return ((size_t)tiles * 4 + 255) & ~size_t(255); }

// batches: MXFP4 routed-expert batches the launch streams each tile for (an estimate:
// min(R * S, E)); 1 for the other formats.
GemvPlan plan_gemv(Fmt f, int64_t M, int64_t N, int64_t K, int num_sms, int64_t batches = 1);
cudaError_t launch_gemv(Fmt f, GemvParams p, const GemvPlan& plan, cudaStream_t stream);
// Weights declared immutable by the caller (wq_set_static_weights): decode kernels may
// start reading them before the previous kernel of the stream has completed.
void set_static_weights(int on);
int static_weights();

// The prepared group-wise 4-bit layout (gemv_prep.cu): the load-time repack and its
// decode kernel (M <= 16, K % 256 == 0, groups of 128 codes or more).
bool prep_shape_ok(int64_t M, int64_t N, int64_t K, int32_t group);
size_t prep_bytes(int64_t N, int64_t K);
size_t prep_ws_bytes(int64_t M, int64_t N, int64_t K, int num_sms);
cudaError_t launch_prepare(const uint8_t* packed, const float* scale, const uint8_t* zero, int64_t N,
                           int64_t K, int32_t group, uint8_t* out, cudaStream_t s);
cudaError_t launch_prep(const GemvParams& p, const uint8_t* prep, void* workspace, size_t ws_bytes,
                        int num_sms, cudaStream_t stream);

// MXFP4 routing tables live in shared memory: bounded slot and expert counts.
bool gemv_mxfp4_supported(int64_t R, int64_t S, int64_t E);
// The MXFP4 TMA-ring cluster kernel (gemv_mx.cu): N a multiple of 16, 768 <= K <= 8192,
// at most 1024 slots and 256 experts, 16-byte aligned codes, scales and activations.
// launch_gemv_mx returns cudaErrorNotSupported when its shared memory does not fit.
bool gemv_mx_ok(const GemvParams& p);
cudaError_t launch_gemv_mx(const GemvParams& p, int num_sms, cudaStream_t stream);

// MXFP4 experts with many routed slots (gemm_mx.cu): the grouped tcgen05 GEMM.  gemm_mx_ok
// holds for R * S >= the crossover (WQ_TUNE_MX_GEMM_MIN_SLOTS, default 512), at most 256
// experts, K % 32 == 0 and 16-byte aligned x, codes and scales; the workspace
// (gemm_mx_ws_bytes, 256-byte aligned) holds the routing tables and the gathered rows.
// x: the shared input [R, K], or with x_per_slot one row a slot [R * S, K]; y: bf16
// [R * S, N]; or, with y32 set, f32 [R * S, N] slot results times sw[slot].
// Slots with an expert index outside [0, E) are not written.
bool gemm_mx_ok(int64_t R, int64_t S, int64_t E, int64_t N, int64_t K, const void* x, const void* blocks,
                const void* scales);
size_t gemm_mx_ws_bytes(int64_t RS, int64_t E, int64_t K);
cudaError_t launch_gemm_mx(const __nv_bfloat16* x, int64_t R, int64_t S, int x_per_slot, const uint8_t* blocks,
                           const uint8_t* scales, int64_t E, int64_t N, int64_t K, const int32_t* experts,
                           __nv_bfloat16* y, float* y32, const float* sw, void* workspace,
                           int32_t* dev_status, cudaStream_t stream);

// Load-time and test kernels (quant.cu).
cudaError_t launch_quantize(const float* w, int64_t N, int64_t K, int32_t G, int32_t bits,
                            int32_t mode, void* codes, float* scale, uint8_t* zero,
                            int32_t* dev_status, cudaStream_t s);
cudaError_t launch_pack(const void* codes, int64_t rows, int64_t cols, int32_t is_unsigned,
                        uint8_t* packed, int32_t* dev_status, cudaStream_t s);
cudaError_t launch_unpack(const uint8_t* packed, int64_t rows, int64_t cols,
                          int32_t is_unsigned, void* codes, cudaStream_t s);
cudaError_t launch_dequant_i4g(const uint8_t* packed, const float* scale, const uint8_t* zero,
                               int64_t N, int64_t K, int32_t G, void* w, cudaStream_t s);
cudaError_t launch_dequant_i8r(const int8_t* q, const float* scale, int64_t N, int64_t K,
                               void* w, cudaStream_t s);
cudaError_t launch_dequant_i4r(const int8_t* packed, const float* scale, int64_t N, int64_t K,
                               void* w, cudaStream_t s);
// Slots whose expert index is outside [0, E): their y rows are zeroed (y may be NULL:
// only the status bit is set).
cudaError_t launch_zero_bad_slots(const int32_t* experts, int64_t slots, int64_t E, int64_t N,
                                  __nv_bfloat16* y, int32_t* dev_status, cudaStream_t s);
// y[r, n] = bf16(sum over slots s of row r, in slot order, of y32[r * S + s, n]); slots
// with an expert index outside [0, E) add nothing.
cudaError_t launch_combine_slots(const float* y32, const int32_t* experts, int64_t R, int64_t S,
                                 int64_t E, int64_t N, __nv_bfloat16* y, cudaStream_t s);
cudaError_t launch_dequant_mxfp4(const uint8_t* blocks, const uint8_t* scales, int64_t E,
                                 int64_t N, int64_t K, void* w, cudaStream_t s);
// xg[m, j] = x[m, order[j]] (0 and WQ_DEV_BAD_ORDER for an entry outside [0, K)).
cudaError_t launch_gather_cols(const __nv_bfloat16* x, const int32_t* order, int64_t M, int64_t K,
                               __nv_bfloat16* xg, int32_t* dev_status, cudaStream_t s);

// Large-M tensor-core GEMM (gemm_tc.cu).  Returns cudaErrorNotSupported when the shape
// is outside what the kernel handles (the caller then uses the GEMV path).
struct GemmTcParams {
  const __nv_bfloat16* x;  // [M, K]
  int64_t M, N, K;
  const uint8_t* packed;   // [N, K/2]
  const float* scale;      // [N, K/G]
  const uint8_t* zero;     // [N, K/G]
  int32_t group;
  const __nv_bfloat16* bias;
  __nv_bfloat16* y;        // [M, N]
  int32_t* dev_status;
  float* part;             // split-K partials [splits, M, N] f32, or NULL (no split)
  int32_t splits;          // k ranges a tile is cut into (1: no split)
};
bool gemm_tc_supported(int64_t M, int64_t N, int64_t K, int32_t group);
// Split-K for shapes with fewer tiles than SMs: the number of k ranges, and the
// workspace (f32 partials) it needs; 1 and 0 when the shape has tiles enough.
int gemm_tc_splits(int64_t M, int64_t N, int64_t K, int num_sms);
size_t gemm_tc_ws_bytes(int64_t M, int64_t N, int64_t K, int num_sms);
cudaError_t launch_gemm_tc(const GemmTcParams& p, int num_sms, cudaStream_t stream);

// Tuning knobs (wq_set_tuning): set by an explicit call, read with one relaxed atomic
// load where a launch is planned; 0 means the library's own choice.
enum Knob { kKnobGemvBlocks = 0, kKnobGemvClusters, kKnobGemvPush, kKnobGemvXsmem, kKnobGemmMinM,
            kKnobDecode, kKnobPrep, kKnobPrepBlocksPerSM, kKnobMxGemmMinSlots, kKnobCount };
int64_t tuning(int knob);
bool set_tuning(int knob, int64_t value);

// Probes (probe.cu): the bounded-wait failure path, and a pure HBM read stream.
cudaError_t launch_wait_probe(uint64_t limit_ns, int arrive, int32_t* dev_status, cudaStream_t s);
cudaError_t launch_stream_read(const void* buf, int64_t bytes, int variant, uint32_t* sink,
                               int num_sms, cudaStream_t s);

// A description of the last kernel launch the calling thread made (wq_last_launch).
void note_launch(const char* fmt, ...);
const char* last_launch();

// Tensor-map encoding through the driver entry point (no link-time libcuda).
bool encode_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, void* base,
                          uint64_t inner, uint64_t outer, uint64_t row_stride_bytes,
                          uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz);

}  // namespace wq
