"""Python binding of libwq (weight-only quantized linear layers on one GB300).

Thin ctypes layer over the C ABI declared in ``include/wq.h``: the functions here have
the C names, take torch tensors that already live on the GPU, pass their device
pointers and the current CUDA stream, and raise ``WQError`` on a non-zero status.  All
arithmetic happens in the CUDA kernels of ``libwq.so``; there is no fallback of any kind:
if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libwq.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "wq.h")

WQ_OK, WQ_EINVAL, WQ_ESHAPE, WQ_EALIGN, WQ_ERANGE, WQ_EUNSUPPORTED, WQ_ECUDA, WQ_EWORKSPACE = range(8)
WQ_DEV_NONFINITE, WQ_DEV_BAD_EXPERT, WQ_DEV_BAD_CODE, WQ_DEV_TIMEOUT, WQ_DEV_BAD_ORDER = 1, 2, 4, 8, 16
WQ_SYM, WQ_SYM_U4, WQ_ASYM = 0, 1, 2
(WQ_TUNE_GEMV_BLOCKS, WQ_TUNE_GEMV_CLUSTERS, WQ_TUNE_GEMV_PUSH, WQ_TUNE_GEMV_XSMEM,
 WQ_TUNE_GEMM_MIN_M, WQ_TUNE_DECODE, WQ_TUNE_PREP, WQ_TUNE_PREP_BLOCKS_PER_SM,
 WQ_TUNE_MX_GEMM_MIN_SLOTS) = range(9)

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_SZ = ctypes.c_size_t

SIGNATURES = {
    "wq_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "wq_version": (ctypes.c_int, []),
    "wq_last_launch": (ctypes.c_char_p, []),
    "wq_linear_int4_groups": (ctypes.c_int, [_P, _I64, _I64, _P, _P, _P, _P, _P, _I64, _I32, _P, _P, _SZ,
                                             _P, _P]),
    "wq_linear_int4_groups_workspace": (_SZ, [_I64, _I64, _I64, _I32]),
    "wq_linear_int4_groups_ordered_workspace": (_SZ, [_I64, _I64, _I64, _I32]),
    "wq_prepared_int4_groups_bytes": (_SZ, [_I64, _I64, _I32]),
    "wq_prepare_int4_groups": (ctypes.c_int, [_P, _P, _P, _I64, _I64, _I32, _P, _SZ, _P]),
    "wq_linear_int4_groups_prepared": (ctypes.c_int, [_P, _I64, _I64, _P, _P, _I64, _I32, _P, _P, _SZ, _P,
                                                      _P]),
    "wq_linear_int4_groups_prepared_workspace": (_SZ, [_I64, _I64, _I64, _I32]),
    "wq_set_static_weights": (ctypes.c_int, [ctypes.c_int]),
    "wq_set_tuning": (ctypes.c_int, [_I32, _I64]),
    "wq_test_wait_timeout": (ctypes.c_int, [ctypes.c_uint64, _I32, _P, _P]),
    "wq_bench_stream_read": (ctypes.c_int, [_P, _SZ, _I32, _P, _P]),
    "wq_linear_int4_groups_noalloc": (ctypes.c_int, [_P, _I64, _I64, _P, _P, _P, _P, _P, _I64, _I32, _P,
                                                     _P, _P]),
    "wq_linear_int8_rows": (ctypes.c_int, [_P, _I64, _I64, _P, _P, _P, _I64, _P, _P, _SZ, _P, _P]),
    "wq_linear_int4_rows": (ctypes.c_int, [_P, _I64, _I64, _P, _P, _P, _I64, _P, _P, _SZ, _P, _P]),
    "wq_linear_rows_workspace": (_SZ, [_I64, _I64, _I64, _I32]),
    "wq_mxfp4_experts_shared": (ctypes.c_int, [_P, _I64, _I64, _P, _P, _I64, _I64, _P, _I64, _P, _P, _SZ,
                                               _P, _P]),
    "wq_mxfp4_experts_shared_workspace": (_SZ, [_I64, _I64, _I64, _I64, _I64]),
    "wq_mxfp4_linear_experts_shared": (ctypes.c_int, [_P, _I64, _I64, _P, _P, _I64, _I64, _P, _I64, _P, _P,
                                                      _SZ, _P, _P]),
    "wq_mxfp4_experts": (ctypes.c_int, [_P, _I64, _I64, _P, _P, _I64, _I64, _P, _I64, _P, _P, _SZ, _P, _P]),
    "wq_mxfp4_experts_workspace": (_SZ, [_I64, _I64, _I64, _I64, _I64]),
    "wq_mxfp4_combine_experts": (ctypes.c_int, [_P, _I64, _I64, _P, _P, _I64, _I64, _P, _I64, _P, _P, _P,
                                                _SZ, _P, _P]),
    "wq_mxfp4_combine_experts_workspace": (_SZ, [_I64, _I64, _I64, _I64, _I64]),
    "wq_quantize_groups": (ctypes.c_int, [_P, _I64, _I64, _I32, _I32, _I32, _P, _P, _P, _P, _P]),
    "wq_pack_int4": (ctypes.c_int, [_P, _I64, _I64, _I32, _P, _P, _P]),
    "wq_unpack_int4": (ctypes.c_int, [_P, _I64, _I64, _I32, _P, _P]),
    "wq_dequantize_int4_groups": (ctypes.c_int, [_P, _P, _P, _I64, _I64, _I32, _P, _P]),
    "wq_dequantize_int8_rows": (ctypes.c_int, [_P, _P, _I64, _I64, _P, _P]),
    "wq_dequantize_int4_rows": (ctypes.c_int, [_P, _P, _I64, _I64, _P, _P]),
    "wq_dequantize_mxfp4": (ctypes.c_int, [_P, _P, _I64, _I64, _I64, _P, _P]),
}

_lock = threading.Lock()
_lib = None


class WQError(RuntimeError):
    def __init__(self, status: int, fn: str):
        self.status = status
        super().__init__(f"{fn}: {status_string(status)}")


def build(force: bool = False) -> str:
    """Compile libwq.so in-tree (nvcc, sm_103a)."""
    from . import buildlib
    return buildlib.build(force=force)


def lib():
    """The loaded libwq.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libwq.so is not built ({LIB_PATH}); run "
                                   "weight_only_quantized_linear_gb300.build()")
            handle = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
        return _lib


def status_string(status: int) -> str:
    return lib().wq_status_string(int(status)).decode()


def wq_last_launch() -> str:
    """The last compute kernel this thread launched through the library (see wq.h)."""
    return lib().wq_last_launch().decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(st: int, fn: str):
    if st != WQ_OK:
        raise WQError(st, fn)


def _need(t, dtype, name, dims=None):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dims is not None and t.dim() != dims:
        raise ValueError(f"{name} must have {dims} dims")


# ------------------------------------------------------------------------ workspaces
def wq_linear_int4_groups_workspace(M: int, N: int, K: int, group: int) -> int:
    return int(lib().wq_linear_int4_groups_workspace(M, N, K, group))


def wq_linear_int4_groups_ordered_workspace(M: int, N: int, K: int, group: int) -> int:
    return int(lib().wq_linear_int4_groups_ordered_workspace(M, N, K, group))


def wq_linear_rows_workspace(M: int, N: int, K: int, bits: int) -> int:
    return int(lib().wq_linear_rows_workspace(M, N, K, bits))


def wq_mxfp4_experts_shared_workspace(R: int, S: int, E: int, N: int, K: int) -> int:
    return int(lib().wq_mxfp4_experts_shared_workspace(R, S, E, N, K))


def wq_set_static_weights(on: bool) -> None:
    """Promise that the weights passed to the decode-regime linears are not written by GPU
    work while calls read them (see wq.h): the decode kernel may then start streaming
    them before the previous kernel of the stream has completed."""
    _check(lib().wq_set_static_weights(1 if on else 0), "wq_set_static_weights")


def wq_set_tuning(knob: int, value: int) -> None:
    """Override one launch-shape choice (WQ_TUNE_*); 0 restores the library's own."""
    _check(lib().wq_set_tuning(int(knob), int(value)), "wq_set_tuning")


def wq_test_wait_timeout(limit_ns: int, arrive: bool, dev_status, stream=None) -> None:
    """One warp waits on a barrier with the library's bounded wait (see wq.h)."""
    _need(dev_status, torch.int32, "dev_status")
    _check(lib().wq_test_wait_timeout(int(limit_ns), 1 if arrive else 0, _ptr(dev_status), _stream(stream)),
           "wq_test_wait_timeout")


def wq_bench_stream_read(buf, variant: int, sink, stream=None, nbytes: int | None = None) -> None:
    """Read the device buffer and do nothing else (the per-launch read ceiling)."""
    n = buf.numel() * buf.element_size() if nbytes is None else int(nbytes)
    _check(lib().wq_bench_stream_read(_ptr(buf), n, int(variant), _ptr(sink), _stream(stream)),
           "wq_bench_stream_read")


def alloc_workspace(nbytes: int, device) -> torch.Tensor | None:
    """A zero-filled workspace buffer of at least ``nbytes`` (None when 0)."""
    if nbytes <= 0:
        return None
    return torch.zeros(nbytes, dtype=torch.uint8, device=device)


# ------------------------------------------------------------------------ linear layers
def wq_linear_int4_groups(x, packed, scale, zero, bias=None, group=128, y=None, workspace=None,
                          dev_status=None, stream=None, order=None):
    """y = x . W-hat^T (+ bias) over the group-wise asymmetric 4-bit layout.

    x bf16 [M, K]; packed u8 [N, K/G, G/2] (or [N, K/2]); scale f32 [N, K/G];
    zero u8 [N, K/G]; bias bf16 [N] or None.  Returns y bf16 [M, N]."""
    _need(x, torch.bfloat16, "x", 2)
    _need(packed, torch.uint8, "packed")
    _need(scale, torch.float32, "scale")
    _need(zero, torch.uint8, "zero")
    _need(bias, torch.bfloat16, "bias")
    _need(order, torch.int32, "order", 1)
    M, K = x.shape
    N = packed.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().wq_linear_int4_groups(_ptr(x), M, K, _ptr(packed), _ptr(scale), _ptr(zero), _ptr(order),
                                     _ptr(bias), N, group, _ptr(y), _ptr(workspace), ws_bytes,
                                     _ptr(dev_status), _stream(stream))
    _check(st, "wq_linear_int4_groups")
    return y


def wq_prepare_int4_groups(packed, scale, zero, group=128, stream=None):
    """The load-time repack of an Int4GroupLinear layer (see wq.h): returns the prepared
    u8 buffer the decode kernel streams."""
    _need(packed, torch.uint8, "packed")
    _need(scale, torch.float32, "scale")
    _need(zero, torch.uint8, "zero")
    N = packed.shape[0]
    K = scale.shape[1] * group
    nbytes = int(lib().wq_prepared_int4_groups_bytes(N, K, group))
    if nbytes == 0:
        raise WQError(WQ_EUNSUPPORTED, "wq_prepare_int4_groups")
    out = torch.empty(nbytes, dtype=torch.uint8, device=packed.device)
    _check(lib().wq_prepare_int4_groups(_ptr(packed), _ptr(scale), _ptr(zero), N, K, group, _ptr(out), nbytes,
                                        _stream(stream)), "wq_prepare_int4_groups")
    return out


def wq_linear_int4_groups_prepared_workspace(M: int, N: int, K: int, group: int) -> int:
    return int(lib().wq_linear_int4_groups_prepared_workspace(M, N, K, group))


def wq_linear_int4_groups_prepared(x, prepared, N, bias=None, group=128, y=None, workspace=None, dev_status=None,
                                   stream=None):
    """y = x . W-hat^T (+ bias) from the prepared copy of the layer (decode regime, M <= 16)."""
    _need(x, torch.bfloat16, "x", 2)
    _need(prepared, torch.uint8, "prepared")
    _need(bias, torch.bfloat16, "bias")
    M, K = x.shape
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().wq_linear_int4_groups_prepared(_ptr(x), M, K, _ptr(prepared), _ptr(bias), N, group, _ptr(y),
                                              _ptr(workspace), ws_bytes, _ptr(dev_status), _stream(stream))
    _check(st, "wq_linear_int4_groups_prepared")
    return y


def wq_linear_int4_groups_noalloc(x, packed, scale, zero, bias=None, group=128, y=None, dev_status=None,
                                  stream=None, order=None):
    """wq_linear_int4_groups for callers that cannot allocate device memory: no workspace
    argument; libwq's own static scratch array is used (shared by every call: do not run
    two of these concurrently on the GPU)."""
    _need(x, torch.bfloat16, "x", 2)
    _need(packed, torch.uint8, "packed")
    _need(scale, torch.float32, "scale")
    _need(zero, torch.uint8, "zero")
    _need(bias, torch.bfloat16, "bias")
    M, K = x.shape
    N = packed.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    st = lib().wq_linear_int4_groups_noalloc(_ptr(x), M, K, _ptr(packed), _ptr(scale), _ptr(zero),
                                             _ptr(order), _ptr(bias), N, group, _ptr(y), _ptr(dev_status),
                                             _stream(stream))
    _check(st, "wq_linear_int4_groups_noalloc")
    return y


def wq_linear_int8_rows(x, q, scale, bias=None, y=None, workspace=None, dev_status=None, stream=None):
    _need(x, torch.bfloat16, "x", 2)
    _need(q, torch.int8, "q", 2)
    _need(scale, torch.float32, "scale")
    _need(bias, torch.bfloat16, "bias")
    M, K = x.shape
    N = q.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().wq_linear_int8_rows(_ptr(x), M, K, _ptr(q), _ptr(scale), _ptr(bias), N, _ptr(y),
                                   _ptr(workspace), ws_bytes, _ptr(dev_status), _stream(stream))
    _check(st, "wq_linear_int8_rows")
    return y


def wq_linear_int4_rows(x, packed, scale, bias=None, y=None, workspace=None, dev_status=None,
                        stream=None):
    _need(x, torch.bfloat16, "x", 2)
    _need(packed, torch.int8, "packed", 2)
    _need(scale, torch.float32, "scale")
    _need(bias, torch.bfloat16, "bias")
    M, K = x.shape
    N = packed.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().wq_linear_int4_rows(_ptr(x), M, K, _ptr(packed), _ptr(scale), _ptr(bias), N, _ptr(y),
                                   _ptr(workspace), ws_bytes, _ptr(dev_status), _stream(stream))
    _check(st, "wq_linear_int4_rows")
    return y


def _mxfp4_workspace(R, S, E, N, K, device):
    # many routed slots: the grouped GEMM's scratch (routing tables and gathered rows)
    n = wq_mxfp4_experts_shared_workspace(R, S, E, N, K)
    return torch.empty(n, dtype=torch.uint8, device=device) if n else None


def wq_mxfp4_experts_shared(x, blocks, scales, experts, y=None, workspace=None, dev_status=None,
                            stream=None):
    """x bf16 [R, 1, K] (or [R, K]); blocks u8 [E, N, K/32, 16]; scales u8 [E, N, K/32];
    experts i32 [R, S].  Returns y bf16 [R, S, N]."""
    _need(x, torch.bfloat16, "x")
    _need(blocks, torch.uint8, "blocks", 4)
    _need(scales, torch.uint8, "scales", 3)
    _need(experts, torch.int32, "experts", 2)
    R, K = x.shape[0], x.shape[-1]
    E, N = blocks.shape[0], blocks.shape[1]
    S = experts.shape[1]
    if y is None:
        y = torch.empty((R, S, N), dtype=torch.bfloat16, device=x.device)
    if workspace is None:
        workspace = _mxfp4_workspace(R, S, E, N, K, x.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().wq_mxfp4_experts_shared(_ptr(x), R, K, _ptr(blocks), _ptr(scales), E, N, _ptr(experts), S,
                                       _ptr(y), _ptr(workspace), ws_bytes, _ptr(dev_status),
                                       _stream(stream))
    _check(st, "wq_mxfp4_experts_shared")
    return y


def wq_mxfp4_linear_experts_shared(x, blocks, scales, experts, y=None, workspace=None, dev_status=None,
                                   stream=None):
    """x bf16 [R, K]; blocks u8 [E, N, K/32, 16]; scales u8 [E, N, K/32]; experts i32
    [R, S].  Returns y bf16 [R, S, N]."""
    _need(x, torch.bfloat16, "x", 2)
    _need(blocks, torch.uint8, "blocks", 4)
    _need(scales, torch.uint8, "scales", 3)
    _need(experts, torch.int32, "experts", 2)
    R, K = x.shape
    E, N = blocks.shape[0], blocks.shape[1]
    S = experts.shape[1]
    if y is None:
        y = torch.empty((R, S, N), dtype=torch.bfloat16, device=x.device)
    if workspace is None:
        workspace = _mxfp4_workspace(R, S, E, N, K, x.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().wq_mxfp4_linear_experts_shared(_ptr(x), R, K, _ptr(blocks), _ptr(scales), E, N, _ptr(experts),
                                              S, _ptr(y), _ptr(workspace), ws_bytes, _ptr(dev_status),
                                              _stream(stream))
    _check(st, "wq_mxfp4_linear_experts_shared")
    return y


def wq_mxfp4_experts_workspace(R: int, S: int, E: int, N: int, K: int) -> int:
    return int(lib().wq_mxfp4_experts_workspace(R, S, E, N, K))


def wq_mxfp4_experts(x, blocks, scales, experts, y=None, workspace=None, dev_status=None, stream=None):
    """x bf16 [R, S, K] (one input a slot); blocks u8 [E, N, K/32, 16]; scales u8
    [E, N, K/32]; experts i32 [R, S].  Returns y bf16 [R, S, N]."""
    _need(x, torch.bfloat16, "x", 3)
    _need(blocks, torch.uint8, "blocks", 4)
    _need(scales, torch.uint8, "scales", 3)
    _need(experts, torch.int32, "experts", 2)
    R, S, K = x.shape
    E, N = blocks.shape[0], blocks.shape[1]
    if tuple(experts.shape) != (R, S):
        raise ValueError("experts must be [R, S] with x [R, S, K]")
    if y is None:
        y = torch.empty((R, S, N), dtype=torch.bfloat16, device=x.device)
    if workspace is None:
        workspace = _mxfp4_workspace(R, S, E, N, K, x.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().wq_mxfp4_experts(_ptr(x), R, K, _ptr(blocks), _ptr(scales), E, N, _ptr(experts), S, _ptr(y),
                                _ptr(workspace), ws_bytes, _ptr(dev_status), _stream(stream))
    _check(st, "wq_mxfp4_experts")
    return y


def wq_mxfp4_combine_experts_workspace(R: int, S: int, E: int, N: int, K: int) -> int:
    return int(lib().wq_mxfp4_combine_experts_workspace(R, S, E, N, K))


def wq_mxfp4_combine_experts(x, blocks, scales, experts, weights, y=None, workspace=None, dev_status=None,
                             stream=None):
    """x bf16 [R, K] (or [R, 1, K]); experts i32 [R, S]; weights f32 [R, S].  Returns
    y bf16 [R, N] = the rows' slot products weighted by `weights` and summed."""
    _need(x, torch.bfloat16, "x")
    _need(blocks, torch.uint8, "blocks", 4)
    _need(scales, torch.uint8, "scales", 3)
    _need(experts, torch.int32, "experts", 2)
    _need(weights, torch.float32, "weights", 2)
    R, K = x.shape[0], x.shape[-1]
    E, N = blocks.shape[0], blocks.shape[1]
    S = experts.shape[1]
    if y is None:
        y = torch.empty((R, N), dtype=torch.bfloat16, device=x.device)
    if workspace is None:
        workspace = torch.empty(wq_mxfp4_combine_experts_workspace(R, S, E, N, K), dtype=torch.uint8,
                                device=x.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    st = lib().wq_mxfp4_combine_experts(_ptr(x), R, K, _ptr(blocks), _ptr(scales), E, N, _ptr(experts), S,
                                        _ptr(weights), _ptr(y), _ptr(workspace), ws_bytes, _ptr(dev_status),
                                        _stream(stream))
    _check(st, "wq_mxfp4_combine_experts")
    return y


# ------------------------------------------------------------------------ load-time ops
def wq_quantize_groups(w, group, bits=4, mode=WQ_ASYM, dev_status=None, stream=None):
    """Round-to-nearest (ties to even) group quantizer.  w f32 [N, K].

    Returns (codes [N, K] (i8 for WQ_SYM, u8 otherwise), scale f32 [N, ceil(K/G)],
    zero u8 [N, ceil(K/G)] or None)."""
    _need(w, torch.float32, "w", 2)
    N, K = w.shape
    groups = -(-K // group)
    codes = torch.empty((N, K), dtype=torch.int8 if mode == WQ_SYM else torch.uint8, device=w.device)
    scale = torch.empty((N, groups), dtype=torch.float32, device=w.device)
    zero = None if mode == WQ_SYM else torch.empty((N, groups), dtype=torch.uint8, device=w.device)
    st = lib().wq_quantize_groups(_ptr(w), N, K, group, bits, mode, _ptr(codes), _ptr(scale), _ptr(zero),
                                  _ptr(dev_status), _stream(stream))
    _check(st, "wq_quantize_groups")
    return codes, scale, zero


def wq_pack_int4(codes, is_unsigned, dev_status=None, stream=None):
    if codes.dtype not in (torch.int8, torch.uint8):
        raise ValueError("codes must be int8 or uint8")
    _need(codes, codes.dtype, "codes", 2)
    rows, cols = codes.shape
    packed = torch.empty((rows, cols // 2), dtype=torch.uint8, device=codes.device)
    st = lib().wq_pack_int4(_ptr(codes), rows, cols, int(bool(is_unsigned)), _ptr(packed),
                            _ptr(dev_status), _stream(stream))
    _check(st, "wq_pack_int4")
    return packed


def wq_unpack_int4(packed, cols, is_unsigned, stream=None):
    _need(packed, packed.dtype, "packed", 2)
    rows = packed.shape[0]
    codes = torch.empty((rows, cols), dtype=torch.uint8 if is_unsigned else torch.int8, device=packed.device)
    st = lib().wq_unpack_int4(_ptr(packed), rows, cols, int(bool(is_unsigned)), _ptr(codes), _stream(stream))
    _check(st, "wq_unpack_int4")
    return codes


def wq_dequantize_int4_groups(packed, scale, zero, K, group, stream=None):
    N = packed.shape[0]
    w = torch.empty((N, K), dtype=torch.bfloat16, device=packed.device)
    st = lib().wq_dequantize_int4_groups(_ptr(packed), _ptr(scale), _ptr(zero), N, K, group, _ptr(w),
                                         _stream(stream))
    _check(st, "wq_dequantize_int4_groups")
    return w


def wq_dequantize_int8_rows(q, scale, stream=None):
    N, K = q.shape
    w = torch.empty((N, K), dtype=torch.bfloat16, device=q.device)
    st = lib().wq_dequantize_int8_rows(_ptr(q), _ptr(scale), N, K, _ptr(w), _stream(stream))
    _check(st, "wq_dequantize_int8_rows")
    return w


def wq_dequantize_int4_rows(packed, scale, K, stream=None):
    N = packed.shape[0]
    w = torch.empty((N, K), dtype=torch.bfloat16, device=packed.device)
    st = lib().wq_dequantize_int4_rows(_ptr(packed), _ptr(scale), N, K, _ptr(w), _stream(stream))
    _check(st, "wq_dequantize_int4_rows")
    return w


def wq_dequantize_mxfp4(blocks, scales, stream=None):
    E, N = blocks.shape[0], blocks.shape[1]
    K = blocks.shape[2] * 32
    w = torch.empty((E, N, K), dtype=torch.bfloat16, device=blocks.device)
    st = lib().wq_dequantize_mxfp4(_ptr(blocks), _ptr(scales), E, N, K, _ptr(w), _stream(stream))
    _check(st, "wq_dequantize_mxfp4")
    return w
