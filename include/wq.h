/*
 * wq.h -- C ABI of libwq: weight-only quantized linear layers y = x . W-hat^T on one
 * NVIDIA GB300 (sm_103a), with W-hat dequantized on the fly from packed codes and never
 * expanded to HBM.
 *
 * Sources (web pages, cited by title and section):
 *   [Linnet] "Quantization" (Linnet language docs, std.quant): the format table
 *            (Int8Linear, Int4Linear, Int4GroupLinear, dequantize_*, linear_int4_groups,
 *            mxfp4_experts_shared), "Group-wise 4-bit weights", "MXFP4 experts".
 *   [L8.5]   "Quantization: int8, int4 group (packed), fp8, KV quant" (OpenLearn TinyLLM
 *            module L8.5): "2. Principles", "3. Worked example by hand".
 *   [Ch20]   "20. Quantization" (Inference Engineering book): "Symmetric quantization,
 *            from scratch", "Granularity: who shares a scale", "Packing", "Speed needs
 *            a kernel".
 *
 * Conventions shared by every entry point
 *   - Every tensor argument is a DEVICE pointer owned by the caller (allocated with
 *     cudaMalloc / torch).  The library allocates no device memory; scratch space, where
 *     an operation wants it, is passed in as `workspace`.
 *   - Row-major, densely packed layouts.  bf16 tensors are passed as `void*` (IEEE
 *     bfloat16 bit patterns).  Device pointers must be 16-byte aligned.
 *   - Packed 4-bit data hold two values a byte, the even element in the low nibble
 *     ([Linnet] "Packed 4-bit formats hold two values a byte, the even element in the
 *     low nibble"; [L8.5] Packing).
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the legacy default
 *     stream) and returns a status: argument problems are detected on the host before
 *     anything is launched, and nothing is launched when the status is not WQ_OK.
 *   - `dev_status` (nullable, device int32): problems only the device can see are
 *     OR-ed into it as WQ_DEV_* bits; the caller reads it after synchronizing.  No call
 *     traps or asserts on the device.
 *   - No exception crosses this ABI.
 */
#ifndef WQ_H_
#define WQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define WQ_API __attribute__((visibility("default")))
#else
#define WQ_API
#endif

typedef struct CUstream_st* wq_stream_t; /* identical to cudaStream_t */

/* Host-side status codes. */
enum {
  WQ_OK = 0,
  WQ_EINVAL = 1,       /* null pointer, non-positive size, unknown mode */
  WQ_ESHAPE = 2,       /* sizes break a layout rule (odd width, K % G != 0, ...) */
  WQ_EALIGN = 3,       /* a pointer is not 16-byte aligned */
  WQ_ERANGE = 4,       /* a value outside the format's range */
  WQ_EUNSUPPORTED = 5, /* a valid request this build does not implement */
  WQ_ECUDA = 6,        /* a CUDA runtime call failed (launch, attribute query) */
  WQ_EWORKSPACE = 7    /* workspace too small for the chosen launch */
};

/* Device-side status bits (OR-ed into *dev_status). */
enum {
  WQ_DEV_NONFINITE = 1,   /* quantizer saw a non-finite weight or an overflowing range */
  WQ_DEV_BAD_EXPERT = 2,  /* an expert index outside [0, E); that slot's output is 0 */
  WQ_DEV_BAD_CODE = 4,    /* pack saw a code outside the 4-bit range; it packed code & 15 */
  WQ_DEV_TIMEOUT = 8,     /* a bounded device wait gave up (results invalid) */
  WQ_DEV_BAD_ORDER = 16   /* an activation-order entry outside [0, K); that input read as 0 */
};

/* Quantizer modes for wq_quantize_groups. */
enum {
  WQ_SYM = 0,    /* signed codes in [-Q, Q], Q = 2^(bits-1) - 1, one f32 scale per group */
  WQ_SYM_U4 = 1, /* as WQ_SYM at 4 bits, stored as code + 8 (u8) with zero = 8 */
  WQ_ASYM = 2    /* unsigned codes in [0, 2^bits - 1] with an f32 scale and u8 zero */
};

/* Human-readable name of a WQ_* status. */
WQ_API const char* wq_status_string(int status);

/* ABI version of this header (major * 100 + minor). */
WQ_API int wq_version(void);

/* A one-line description of the last compute kernel the calling thread launched through
 * this library (kernel, template instance, grid); "none" before the first.  The string
 * belongs to the library and stays valid until the thread's next launch. */
WQ_API const char* wq_last_launch(void);

/* ------------------------------------------------------------------------------------
 * Group-wise asymmetric 4-bit linear: [Linnet] linear_int4_groups(x, packed, scale,
 * zero, bias) over the Int4GroupLinear layout, "(q - zero) * scale per group"
 * (dequantize_int4_groups), "Group-wise 4-bit weights" (the GPTQ / AWQ scheme, 16
 * levels per group of Group consecutive inputs).
 *
 *   y[m, n] = bf16( sum_k x[m, k] * W-hat[n, k] + bias[n] ),
 *   W-hat[n, k] = bf16( f32(q[n, k] - zero[n, k/G]) * scale[n, k/G] )
 *
 *   x       bf16 [M, K]
 *   packed  u8   [N, K/G, G/2]  (= [N, K/2] row-major; code k of row n is nibble k%2 of
 *                                byte k/2, unsigned 0..15)
 *   scale   f32  [N, K/G]
 *   zero    u8   [N, K/G]       (values 0..15)
 *   order   i32 [K] or NULL: the activation order of a GPTQ checkpoint quantized in
 *           activation order ([Linnet] Int4GroupLinear "optional order: [In; i32]";
 *           "Importing GPTQ and AWQ": the layer gets an order and gathers its inputs
 *           first).  Stored column j multiplies input order[j]:
 *             y = x[:, order] . W-hat^T + bias
 *           Entries must lie in [0, K) (repeats allowed); an entry outside reads as 0 and
 *           sets WQ_DEV_BAD_ORDER.  The decode kernel gathers while it stages the
 *           activations in shared memory; the other launches first gather x[:, order]
 *           into the workspace (sized by wq_linear_int4_groups_ordered_workspace).
 *   bias    bf16 [N] or NULL
 *   y       bf16 [M, N]         (written; must not alias the inputs)
 *   group   G in {32, 64, 128, 256}; K % G == 0 (else WQ_ESHAPE)
 *   workspace / ws_bytes: optional scratch for splitting K across thread blocks (decode
 *           regime: arrival counters and partial tiles; tensor-core regime, M > 16, for
 *           shapes with fewer 256 x 256 output tiles than SMs: f32 partial sums of each
 *           k range).  Size it with wq_linear_int4_groups_workspace(); it must be
 *           zero-filled once when allocated (the kernels leave it zero-filled again on
 *           return), 16-byte aligned (256 in the decode regime).  Pass NULL / 0 to run
 *           without cross-block split-K (correct, slower at small N).  Calls that share
 *           one workspace must not run concurrently on the GPU.
 * The result is exact up to f32 accumulation order: |y - y_exact| <= 2e-3 *
 * sum_k |x_k W-hat_k| + 1 bf16 ulp.
 * ------------------------------------------------------------------------------------ */
WQ_API int wq_linear_int4_groups(const void* x, int64_t M, int64_t K,
                                 const uint8_t* packed, const float* scale,
                                 const uint8_t* zero, const int32_t* order,
                                 const void* bias, int64_t N, int32_t group, void* y,
                                 void* workspace, size_t ws_bytes, int32_t* dev_status,
                                 wq_stream_t stream);
/* Workspace bytes wq_linear_int4_groups wants for (M, N, K, group) on the current
 * device (0 if the launch needs none), with order == NULL. */
WQ_API size_t wq_linear_int4_groups_workspace(int64_t M, int64_t N, int64_t K,
                                              int32_t group);
/* The same with an activation order (order != NULL): room for the gathered activations
 * x[:, order] (M * K bf16, rounded up to 256 bytes) ahead of the split-K scratch.  With
 * order != NULL the workspace is required (WQ_EWORKSPACE if NULL or smaller than this). */
WQ_API size_t wq_linear_int4_groups_ordered_workspace(int64_t M, int64_t N, int64_t K,
                                                      int32_t group);

/* ------------------------------------------------------------------------------------
 * Prepared group-wise 4-bit weights: [Linnet] "Group-wise 4-bit weights" (weights
 * repacked at load, --prepare); [Ch20] "Speed needs a kernel" (weight layouts pre-shuffled
 * so that a 128-bit load fills a tensor-core fragment directly).
 *
 * wq_prepare_int4_groups copies an Int4GroupLinear layer (packed [N, K/2], scale and
 * zero [N, K/G], as for wq_linear_int4_groups) into one device buffer of
 * wq_prepared_int4_groups_bytes(N, K, group) bytes in the order the decode kernel
 * consumes it: for every block of 128 rows and every 256 codes, 16384 bytes of codes
 * (fragment-ordered, bank-swizzled, nibbles in pair order) followed by the 128 rows' two
 * scales and two zero points (1280 bytes); rows past N are padded with code 0, scale 0.
 * Same bytes a weight as the public layout (plus the row padding).  A load-time step:
 * asynchronous on `stream`, bit-exact (codes, scales and zero points are only moved).
 * Requires K % 256 == 0 and a power-of-two group of 128 or more (else
 * wq_prepared_int4_groups_bytes returns 0 and the call WQ_EUNSUPPORTED); prepared 16-byte
 * aligned; prepared_bytes too small: WQ_EWORKSPACE.
 *
 * wq_linear_int4_groups_prepared computes the product of wq_linear_int4_groups (the same
 * definition, result and tolerance) from the prepared copy, for the decode regime:
 * M <= 16 (WQ_EUNSUPPORTED above; the prefill regime reads the public layout).  No
 * activation order.  workspace: as wq_linear_int4_groups, sized by
 * wq_linear_int4_groups_prepared_workspace(); NULL runs whole 128-row blocks a thread
 * block.  Each step of the kernel arrives with two bulk copies of the prepared bytes and
 * one 512-byte copy of each activation row.
 * ------------------------------------------------------------------------------------ */
WQ_API size_t wq_prepared_int4_groups_bytes(int64_t N, int64_t K, int32_t group);
WQ_API int wq_prepare_int4_groups(const uint8_t* packed, const float* scale, const uint8_t* zero,
                                  int64_t N, int64_t K, int32_t group, void* prepared,
                                  size_t prepared_bytes, wq_stream_t stream);
WQ_API int wq_linear_int4_groups_prepared(const void* x, int64_t M, int64_t K,
                                          const void* prepared, const void* bias, int64_t N,
                                          int32_t group, void* y, void* workspace,
                                          size_t ws_bytes, int32_t* dev_status,
                                          wq_stream_t stream);
WQ_API size_t wq_linear_int4_groups_prepared_workspace(int64_t M, int64_t N, int64_t K,
                                                       int32_t group);

/* ------------------------------------------------------------------------------------
 * Declare the weights immutable (the source pages have no counterpart: a launch-order
 * promise made by the caller, not an operation of the method).
 *
 * on != 0: the caller promises that no GPU work writes the packed codes, scales or zero
 * points passed to the decode-regime linears (wq_linear_int4_groups and its _noalloc
 * variant with M <= 16, wq_linear_int8_rows, wq_linear_int4_rows) while a call that
 * reads them may run, in particular not the kernel issued just before the call on its
 * stream.  Weights loaded once and synchronized before serving satisfy it.  The decode
 * kernel then starts streaming its first weight stages while the previous kernel of the
 * stream is still running (programmatic dependent launch); activations, outputs and the
 * workspace are still read and written only after that kernel has completed.
 * on == 0 (the default): nothing is read before the previous kernel has completed.
 * Process-wide; applies to launches issued after the call.  Returns WQ_OK.
 * ------------------------------------------------------------------------------------ */
WQ_API int wq_set_static_weights(int on);

/* ------------------------------------------------------------------------------------
 * Allocation-free variant of wq_linear_int4_groups (the source pages have no
 * counterpart; it exists for callers of this library).
 *
 * Some callers cannot call cudaMalloc and so cannot hand in a workspace: for example a
 * serving loop that forbids device allocation once it has started, or a host program
 * that owns every byte of device memory through its own pool and exposes no allocator to
 * plugins.  This entry point takes the same arguments minus the workspace and allocates
 * nothing: the split-K scratch it needs lives in one static device array of
 * WQ_NOALLOC_SCRATCH_BYTES inside libwq, which every GPU that loads the library keeps
 * until the process exits.
 *   - Shapes whose split-K scratch would exceed that array run without cross-block
 *     split-K (the launch wq_linear_int4_groups makes with a NULL workspace: the same
 *     result up to f32 summation order, slower where N is small).  The decode kernel for
 *     groups of 128 codes or more needs no scratch at all.
 *   - The first call on a device looks up the array's device address (once per device,
 *     with that device current) and clears the array on the call's stream; make that
 *     first call before any stream capture.  The cached address outlives a
 *     cudaDeviceReset: do not reset the device between calls.
 *   - Every later launch leaves the array's arrival counters at zero again, so nothing
 *     else runs on the stream between the previous kernel and the launch (wq_set_static_
 *     weights applies as to wq_linear_int4_groups).  A call that reports WQ_DEV_TIMEOUT
 *     may leave them non-zero; later results of this entry point are then invalid.
 *   - Every call shares the one array: calls whose executions overlap on the GPU (two
 *     streams, or two host threads) race on it.  Serialize them.
 * Results are those of wq_linear_int4_groups.
 * ------------------------------------------------------------------------------------ */
#define WQ_NOALLOC_SCRATCH_BYTES (1024u * 1024u)
/* (order must be NULL here: WQ_EUNSUPPORTED otherwise.) */
WQ_API int wq_linear_int4_groups_noalloc(const void* x, int64_t M, int64_t K,
                                         const uint8_t* packed, const float* scale,
                                         const uint8_t* zero, const int32_t* order,
                                         const void* bias, int64_t N, int32_t group, void* y,
                                         int32_t* dev_status, wq_stream_t stream);

/* ------------------------------------------------------------------------------------
 * Tuning knobs (the source pages have no counterpart: launch-shape overrides for
 * measurement and for tests that force each code path).  value 0 restores the library's
 * own choice; a negative value or an unknown knob returns WQ_EINVAL.  Process-wide;
 * applies to launches issued after the call.
 *   WQ_TUNE_GEMV_BLOCKS    thread blocks of the exact decode kernel (groups < 128, MXFP4)
 *   WQ_TUNE_GEMV_CLUSTERS  thread-block clusters of the factored decode kernel
 *   WQ_TUNE_GEMV_PUSH      cut-tile fixup of the factored kernel: 1 push, 2 cluster barriers
 *   WQ_TUNE_GEMV_XSMEM     1: never stage activations in shared memory
 *   WQ_TUNE_GEMM_MIN_M     smallest M that takes the tensor-core GEMM (default 40)
 *   WQ_TUNE_DECODE         decode kernel for the affine formats: 0 (and 1) the cluster
 *                          kernel, 2 the exact kernel
 *   WQ_TUNE_PREP           prepared-layout kernel launch, bit mask: 1 without programmatic
 *                          dependent launch, 2 without streaming weights before the
 *                          dependency wait
 *   WQ_TUNE_PREP_BLOCKS_PER_SM  blocks an SM the prepared-layout kernel is sized for (2)
 *   WQ_TUNE_MX_GEMM_MIN_SLOTS   fewest routed slots (R * S) for which the MXFP4 expert
 *                          products take the grouped tensor-core GEMM when the caller
 *                          passes its workspace (default 512)
 * ------------------------------------------------------------------------------------ */
enum {
  WQ_TUNE_GEMV_BLOCKS = 0,
  WQ_TUNE_GEMV_CLUSTERS = 1,
  WQ_TUNE_GEMV_PUSH = 2,
  WQ_TUNE_GEMV_XSMEM = 3,
  WQ_TUNE_GEMM_MIN_M = 4,
  WQ_TUNE_DECODE = 5,
  WQ_TUNE_PREP = 6,
  WQ_TUNE_PREP_BLOCKS_PER_SM = 7,
  WQ_TUNE_MX_GEMM_MIN_SLOTS = 8
};
WQ_API int wq_set_tuning(int32_t knob, int64_t value);

/* ------------------------------------------------------------------------------------
 * Test and measurement exports (no counterpart in the source pages).
 *
 * wq_test_wait_timeout: launches one warp that waits on a shared-memory barrier with the
 * same bounded wait every kernel of the library uses, limited to limit_ns (1 ..
 * 100000000, else WQ_EINVAL).  arrive != 0: the warp arrives first and the wait succeeds;
 * arrive == 0: nobody arrives, the wait gives up after limit_ns, WQ_DEV_TIMEOUT is OR-ed
 * into *dev_status and the kernel returns.  Nothing else is in flight when it gives up,
 * so the context stays usable: it shows the failure path without a fault.
 *
 * wq_bench_stream_read: reads `bytes` (rounded down to a multiple of 16) of the device
 * buffer `buf` and does nothing else: the per-launch HBM read rate a kernel without any
 * arithmetic reaches.  variant 0: plain 16-byte loads, eight in flight a thread, 8 blocks
 * of 256 threads an SM; variant 1: one block an SM streaming its share through a
 * six-stage ring of 16 KB bulk copies, launched with programmatic dependent launch and
 * filling its ring before waiting for the previous kernel of the stream (buf must not be
 * written by that kernel).  *sink (device u32) is written only in the impossible case
 * that the folded words equal a fixed constant.
 * ------------------------------------------------------------------------------------ */
WQ_API int wq_test_wait_timeout(uint64_t limit_ns, int32_t arrive, int32_t* dev_status,
                                wq_stream_t stream);
WQ_API int wq_bench_stream_read(const void* buf, size_t bytes, int32_t variant, uint32_t* sink,
                                wq_stream_t stream);

/* ------------------------------------------------------------------------------------
 * Symmetric per-row int8 linear: [Linnet] Int8Linear<In, Out, T> (weight [Out, In; i8],
 * scale [Out; f32], optional bias) with dequantize_int8 "q * scale in f32, cast to T".
 *   q i8 [N, K]; scale f32 [N]; x bf16 [M, K]; bias bf16 [N] or NULL; y bf16 [M, N].
 *   K % 16 == 0 (rows start 16-byte aligned).  workspace as for wq_linear_int4_groups,
 *   sized by wq_linear_rows_workspace().
 * ------------------------------------------------------------------------------------ */
WQ_API int wq_linear_int8_rows(const void* x, int64_t M, int64_t K, const int8_t* q,
                               const float* scale, const void* bias, int64_t N, void* y,
                               void* workspace, size_t ws_bytes, int32_t* dev_status,
                               wq_stream_t stream);

/* ------------------------------------------------------------------------------------
 * Symmetric per-row signed int4 linear: [Linnet] Int4Linear<In, Out, T> (weight
 * [Out, In/2; i8], scale [Out; f32]) with dequantize_int4 "unpack, then dequantize";
 * nibbles are 4-bit two's complement ([L8.5] Packing: a nibble v >= 8 means v - 16).
 *   packed [N, K/2]; scale f32 [N]; K % 32 == 0.  Other arguments as above.
 * ------------------------------------------------------------------------------------ */
WQ_API int wq_linear_int4_rows(const void* x, int64_t M, int64_t K, const int8_t* packed,
                               const float* scale, const void* bias, int64_t N, void* y,
                               void* workspace, size_t ws_bytes, int32_t* dev_status,
                               wq_stream_t stream);
/* Workspace bytes for the two per-row linears (bits = 8 or 4). */
WQ_API size_t wq_linear_rows_workspace(int64_t M, int64_t N, int64_t K, int32_t bits);

/* ------------------------------------------------------------------------------------
 * MXFP4 experts, shared input: [Linnet] mxfp4_experts_shared(x, blocks, scales,
 * experts) -- "a mixture's chosen experts multiplied from MXFP4, each row's slots
 * sharing one input (x: [R, 1, In])"; dequantize_mxfp4: "E2M1 values in blocks of 32,
 * one E8M0 scale byte a block"; [L8.5] MXFP4 (element magnitudes 0, .5, 1, 1.5, 2, 3,
 * 4, 6 times the block's power-of-two scale).
 *
 *   y[r, s, n] = bf16( sum_k x[r, k] * W-hat_e[n, k] ),  e = experts[r, s]
 *   W-hat_e[n, k] = bf16( E2M1(code) * 2^(scales[e, n, k/32] - 127) )
 *
 *   x       bf16 [R, 1, K]
 *   blocks  u8 [E, N, K/32, 16]  (two E2M1 codes a byte, even element low)
 *   scales  u8 [E, N, K/32]      (E8M0; 255 = NaN)
 *   experts i32 [R, S]           (an index outside [0, E) gives a zero slot and sets
 *                                 WQ_DEV_BAD_EXPERT)
 *   y       bf16 [R, S, N]
 *   K % 32 == 0; at most 256 experts.
 *   Regimes: up to 2048 routed slots (R * S) the decode kernels run, with no workspace.
 *   From WQ_TUNE_MX_GEMM_MIN_SLOTS slots on (default 512) the grouped tensor-core GEMM
 *   runs when the workspace is given: wq_mxfp4_experts_shared_workspace() bytes (0 below
 *   the crossover), 16-byte aligned, holding the routing tables and the input rows
 *   gathered in expert order.  It needs no zero-fill and holds scratch on return: do not
 *   share it with the linears' split-K workspaces, which must stay zero-filled.  A
 *   smaller workspace leaves the decode kernels; more than 2048 slots without it give
 *   WQ_EWORKSPACE.
 * ------------------------------------------------------------------------------------ */
WQ_API int wq_mxfp4_experts_shared(const void* x, int64_t R, int64_t K,
                                   const uint8_t* blocks, const uint8_t* scales,
                                   int64_t E, int64_t N, const int32_t* experts,
                                   int64_t S, void* y, void* workspace, size_t ws_bytes,
                                   int32_t* dev_status, wq_stream_t stream);
WQ_API size_t wq_mxfp4_experts_shared_workspace(int64_t R, int64_t S, int64_t E,
                                                int64_t N, int64_t K);

/* ------------------------------------------------------------------------------------
 * [Linnet] mxfp4_linear_experts_shared(x, blocks, scales, experts): "std.nn.moe::
 * linear_experts_shared with MXFP4 experts, many rows (x: [R, In])".  The product is
 * that of wq_mxfp4_experts_shared, with x given as [R, K]:
 *   y[r, s, n] = bf16( sum_k x[r, k] * W-hat_e[n, k] ),  e = experts[r, s]
 * Arguments, layouts, limits and errors as wq_mxfp4_experts_shared.
 * ------------------------------------------------------------------------------------ */
WQ_API int wq_mxfp4_linear_experts_shared(const void* x, int64_t R, int64_t K,
                                          const uint8_t* blocks, const uint8_t* scales,
                                          int64_t E, int64_t N, const int32_t* experts,
                                          int64_t S, void* y, void* workspace, size_t ws_bytes,
                                          int32_t* dev_status, wq_stream_t stream);

/* ------------------------------------------------------------------------------------
 * [Linnet] mxfp4_experts(x, blocks, scales, experts): "a mixture's chosen experts
 * multiplied from MXFP4, each slot its own input".
 *   y[r, s, n] = bf16( sum_k x[r, s, k] * W-hat_e[n, k] ),  e = experts[r, s]
 *   x bf16 [R, S, K] (one input row a slot); the other arguments as
 *   wq_mxfp4_experts_shared, the workspace sized by wq_mxfp4_experts_workspace().  An
 *   expert index outside [0, E) gives a zero slot and sets WQ_DEV_BAD_EXPERT.
 * ------------------------------------------------------------------------------------ */
WQ_API int wq_mxfp4_experts(const void* x, int64_t R, int64_t K, const uint8_t* blocks,
                            const uint8_t* scales, int64_t E, int64_t N, const int32_t* experts,
                            int64_t S, void* y, void* workspace, size_t ws_bytes,
                            int32_t* dev_status, wq_stream_t stream);
WQ_API size_t wq_mxfp4_experts_workspace(int64_t R, int64_t S, int64_t E, int64_t N, int64_t K);

/* ------------------------------------------------------------------------------------
 * [Linnet] mxfp4_combine_experts(x, blocks, scales, experts, weights): "std.nn.moe::
 * combine_experts with MXFP4 experts".  The page gives the name and the arguments; the
 * reading taken is the weighted sum of the row's routed experts over the shared input:
 *   y[r, n] = bf16( sum_s weights[r, s] * sum_k x[r, k] * W-hat_e[n, k] ),  e = experts[r, s]
 * a slot whose expert index lies outside [0, E) adding nothing (WQ_DEV_BAD_EXPERT set).
 *   x bf16 [R, K] (or [R, 1, K]); weights f32 [R, S] (the combine weights, e.g. a softmax
 *   over the row's routing logits); y bf16 [R, N].
 *   workspace: R * S * N f32 slot results, then (from the grouped GEMM's crossover on)
 *   the grouped GEMM's scratch as for wq_mxfp4_experts_shared; sized by
 *   wq_mxfp4_combine_experts_workspace(), 16-byte aligned, required (WQ_EINVAL if NULL,
 *   WQ_EWORKSPACE if smaller than the slot results); no zero-fill needed.  Each slot's f32 result is multiplied by its weight in the product kernel's
 *   epilogue; a second small kernel adds a row's slots in slot order (deterministic) and
 *   rounds once to bf16.
 * ------------------------------------------------------------------------------------ */
WQ_API int wq_mxfp4_combine_experts(const void* x, int64_t R, int64_t K, const uint8_t* blocks,
                                    const uint8_t* scales, int64_t E, int64_t N,
                                    const int32_t* experts, int64_t S, const float* weights,
                                    void* y, void* workspace, size_t ws_bytes,
                                    int32_t* dev_status, wq_stream_t stream);
WQ_API size_t wq_mxfp4_combine_experts_workspace(int64_t R, int64_t S, int64_t E, int64_t N,
                                                 int64_t K);

/* ------------------------------------------------------------------------------------
 * Round-to-nearest quantizer, ties to even, one scale per group of `group` consecutive
 * inputs of a row; the last group of a row may be short ([Ch20] "Symmetric
 * quantization, from scratch" and "Granularity": scale = max|w| / Q, codes clamped to
 * [-Q, Q], an all-zero group gets scale 1, a short last group is padded for the
 * computation; [L8.5] "2. Principles": rint with ties to even, quotients in float32;
 * [Linnet] "Quantizing a checkpoint": each group rounded to the nearest level).
 *
 *   w      f32 [N, K]
 *   codes  [N, K] one byte a code: i8 for WQ_SYM; u8 for WQ_SYM_U4 and WQ_ASYM
 *   scale  f32 [N, ceil(K/G)]
 *   zero   u8  [N, ceil(K/G)] for WQ_SYM_U4 / WQ_ASYM; ignored (may be NULL) for WQ_SYM
 *   bits   2..8 for WQ_SYM and WQ_ASYM; 4 for WQ_SYM_U4
 * WQ_SYM: a = max|w|, s = f32(a / Q), code = clamp(rint(f32(w * f32(Q / a))), -Q, Q).
 * WQ_ASYM: lo = min(0, min w), hi = max(0, max w), L = 2^bits - 1,
 *   s = f32((hi - lo) / L), r = f32(L / (hi - lo)), zero = clamp(rint(f32(-lo * r)), 0,
 *   L), code = clamp(rint(f32(w * r)) + zero, 0, L); hi == lo gives s = 1 and
 *   zero = codes = 2^(bits-1).
 * When Q / a (or L / (hi - lo)) overflows f32 the codes use the quotient w / s instead.
 * A group holding a non-finite weight (or whose range overflows f32) is refused: it
 * gets scale 1 and the code of 0, and WQ_DEV_NONFINITE is set in *dev_status.
 * ------------------------------------------------------------------------------------ */
WQ_API int wq_quantize_groups(const float* w, int64_t N, int64_t K, int32_t group,
                              int32_t bits, int32_t mode, void* codes, float* scale,
                              uint8_t* zero, int32_t* dev_status, wq_stream_t stream);

/* ------------------------------------------------------------------------------------
 * Pack / unpack 4-bit codes, two a byte, even column low ([Ch20] Packing; [L8.5]
 * Packing).  codes [rows, cols] one byte a code (i8 in [-8, 7] when is_unsigned == 0,
 * u8 in [0, 15] otherwise); packed [rows, cols/2].  cols must be even (WQ_ESHAPE).  A
 * code outside the range sets WQ_DEV_BAD_CODE (its low nibble is packed).  Unpack
 * sign-extends when is_unsigned == 0 (a nibble v >= 8 gives v - 16).
 * ------------------------------------------------------------------------------------ */
WQ_API int wq_pack_int4(const void* codes, int64_t rows, int64_t cols, int32_t is_unsigned,
                        uint8_t* packed, int32_t* dev_status, wq_stream_t stream);
WQ_API int wq_unpack_int4(const uint8_t* packed, int64_t rows, int64_t cols,
                          int32_t is_unsigned, void* codes, wq_stream_t stream);

/* ------------------------------------------------------------------------------------
 * Dequantizers ([Linnet] format table: dequantize_int8 "q * scale in f32, cast to T",
 * dequantize_int4 "unpack, then dequantize", dequantize_int4_groups "(q - zero) *
 * scale per group", dequantize_mxfp4).  Output bf16, bit-identical to the definitions
 * above.  These expand W-hat to memory; the linear entry points never do.
 *   wq_dequantize_int4_groups: packed [N, K/2], scale/zero [N, K/G] -> w [N, K];
 *                              K % G == 0, G even.
 *   wq_dequantize_int8_rows:   q i8 [N, K], scale [N] -> w [N, K]
 *   wq_dequantize_int4_rows:   packed [N, K/2] signed nibbles, scale [N] -> w [N, K]
 *   wq_dequantize_mxfp4:       blocks [E, N, K/32, 16], scales [E, N, K/32] -> w [E, N, K]
 * ------------------------------------------------------------------------------------ */
WQ_API int wq_dequantize_int4_groups(const uint8_t* packed, const float* scale,
                                     const uint8_t* zero, int64_t N, int64_t K,
                                     int32_t group, void* w, wq_stream_t stream);
WQ_API int wq_dequantize_int8_rows(const int8_t* q, const float* scale, int64_t N,
                                   int64_t K, void* w, wq_stream_t stream);
WQ_API int wq_dequantize_int4_rows(const int8_t* packed, const float* scale, int64_t N,
                                   int64_t K, void* w, wq_stream_t stream);
WQ_API int wq_dequantize_mxfp4(const uint8_t* blocks, const uint8_t* scales, int64_t E,
                               int64_t N, int64_t K, void* w, wq_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* WQ_H_ */
