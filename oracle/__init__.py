"""CPU oracle for the weight-only quantized linear layer -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's ``cpu_baseline`` leg may
import this package.  The CUDA library (``weight_only_quantized_linear_gb300``) never
does, and the two share no code: this wrapper loads ``libwq_oracle.so`` compiled from
``wq_oracle.cpp`` (plain C++17, f32 quantizers, f64 linear sums), building it with g++
on first use.

bf16 arrays are passed as ``numpy.uint16`` bit patterns.

Pinning status of each function (what ties it to the pages rather than to itself) is
kept in ``tests/test_oracle_pins.py``; the asymmetric quantizer's tie rule is pinned by
invariants only (its formula is lost from the pages).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "wq_oracle.cpp")
_LIB = os.path.join(_HERE, "libwq_oracle.so")
_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int


def build(force: bool = False) -> str:
    """Compile ``libwq_oracle.so`` (plain g++, no CUDA).  Returns its path."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-fopenmp",
               "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB)
        sig = {
            "orc_quantize_sym": (_I64, [_P, _I64, _I64, _I64, _I32, _P, _P]),
            "orc_quantize_asym": (_I64, [_P, _I64, _I64, _I64, _I32, _P, _P, _P]),
            "orc_pack_int4": (_I32, [_P, _I64, _I64, _I32, _P]),
            "orc_unpack_int4": (_I32, [_P, _I64, _I64, _I32, _P]),
            "orc_dequant_int4_groups": (None, [_P, _P, _P, _I64, _I64, _I64, _P]),
            "orc_dequant_int8_rows": (None, [_P, _P, _I64, _I64, _P]),
            "orc_dequant_int4_rows": (None, [_P, _P, _I64, _I64, _P]),
            "orc_dequant_mxfp4": (None, [_P, _P, _I64, _I64, _I64, _P]),
            "orc_set_threads": (None, [_I32]),
            "orc_max_threads": (_I32, []),
            "orc_linear_bf16": (None, [_P, _I64, _I64, _P, _P, _I64, _P, _P]),
            "orc_linear_int4_groups": (None, [_P, _I64, _I64, _P, _P, _P, _P, _I64, _I64, _P, _P]),
            "orc_linear_int8_rows": (None, [_P, _I64, _I64, _P, _P, _P, _I64, _P, _P]),
            "orc_linear_int4_rows": (None, [_P, _I64, _I64, _P, _P, _P, _I64, _P, _P]),
            "orc_mxfp4_experts_shared": (_I64, [_P, _I64, _I64, _P, _P, _I64, _I64, _P, _I64,
                                                _I64, _I64, _P, _P]),
            "orc_bf16_from_f32": (ctypes.c_uint16, [ctypes.c_float]),
            "orc_e2m1_value": (ctypes.c_float, [_I32]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a):
    return None if a is None else a.ctypes.data


def set_threads(n: int) -> None:
    """Threads used by the linear functions (OpenMP over output rows)."""
    _load().orc_set_threads(int(n))


def max_threads() -> int:
    return int(_load().orc_max_threads())


# ----------------------------------------------------------------------------- quantize
def quantize_sym(w: np.ndarray, group: int, bits: int = 4):
    """Symmetric RTN per group.  Returns (codes i8 [N,K], scale f32 [N,ceil(K/G)], refused)."""
    w = _c(w, np.float32)
    n, k = w.shape
    groups = -(-k // group)
    codes = np.empty((n, k), np.int8)
    scale = np.empty((n, groups), np.float32)
    refused = _load().orc_quantize_sym(_ptr(w), n, k, group, bits, _ptr(codes), _ptr(scale))
    return codes, scale, int(refused)


def quantize_asym(w: np.ndarray, group: int, bits: int = 4):
    """Asymmetric RTN per group.  Returns (codes u8, scale f32, zero u8, refused)."""
    w = _c(w, np.float32)
    n, k = w.shape
    groups = -(-k // group)
    codes = np.empty((n, k), np.uint8)
    scale = np.empty((n, groups), np.float32)
    zero = np.empty((n, groups), np.uint8)
    refused = _load().orc_quantize_asym(_ptr(w), n, k, group, bits, _ptr(codes), _ptr(scale),
                                         _ptr(zero))
    return codes, scale, zero, int(refused)


def pack_int4(codes: np.ndarray, is_unsigned: bool):
    """Returns (status, packed u8 [rows, cols/2]); status 1 odd width, 2 out of range."""
    codes = _c(codes, np.uint8 if is_unsigned else np.int8)
    rows, cols = codes.shape
    packed = np.zeros((rows, max(cols // 2, 0)), np.uint8)
    st = _load().orc_pack_int4(_ptr(codes), rows, cols, int(is_unsigned), _ptr(packed))
    return int(st), packed


def unpack_int4(packed: np.ndarray, cols: int, is_unsigned: bool) -> np.ndarray:
    packed = _c(packed, np.uint8)
    rows = packed.shape[0]
    codes = np.empty((rows, cols), np.int8)
    st = _load().orc_unpack_int4(_ptr(packed), rows, cols, int(is_unsigned), _ptr(codes))
    if st:
        raise ValueError("odd width")
    return codes.view(np.uint8) if is_unsigned else codes


# ----------------------------------------------------------------------------- dequant
def dequant_int4_groups(packed, scale, zero, n: int, k: int, group: int) -> np.ndarray:
    packed = _c(packed, np.uint8)
    scale = _c(scale, np.float32)
    zero = _c(zero, np.uint8)
    out = np.empty((n, k), np.uint16)
    _load().orc_dequant_int4_groups(_ptr(packed), _ptr(scale), _ptr(zero), n, k, group, _ptr(out))
    return out


def dequant_int8_rows(q, scale) -> np.ndarray:
    q = _c(q, np.int8)
    scale = _c(scale, np.float32)
    n, k = q.shape
    out = np.empty((n, k), np.uint16)
    _load().orc_dequant_int8_rows(_ptr(q), _ptr(scale), n, k, _ptr(out))
    return out


def dequant_int4_rows(packed, scale, k: int) -> np.ndarray:
    packed = _c(packed, np.uint8)
    scale = _c(scale, np.float32)
    n = packed.shape[0]
    out = np.empty((n, k), np.uint16)
    _load().orc_dequant_int4_rows(_ptr(packed), _ptr(scale), n, k, _ptr(out))
    return out


def dequant_mxfp4(blocks, scales, e: int, n: int, k: int) -> np.ndarray:
    blocks = _c(blocks, np.uint8)
    scales = _c(scales, np.uint8)
    out = np.empty((e, n, k), np.uint16)
    _load().orc_dequant_mxfp4(_ptr(blocks), _ptr(scales), e, n, k, _ptr(out))
    return out


# ----------------------------------------------------------------------------- linear
def linear_bf16(x, w, bias=None):
    """y (f64, unrounded) and sum|x*w| for y = x . w^T + bias over bf16 bit arrays."""
    x = _c(x, np.uint16)
    w = _c(w, np.uint16)
    m, k = x.shape
    n = w.shape[0]
    b = None if bias is None else _c(bias, np.uint16)
    y = np.empty((m, n), np.float64)
    a = np.empty((m, n), np.float64)
    _load().orc_linear_bf16(_ptr(x), m, k, _ptr(w), _ptr(b), n, _ptr(y), _ptr(a))
    return y, a


def linear_int4_groups(x, packed, scale, zero, bias, n: int, group: int):
    x = _c(x, np.uint16)
    m, k = x.shape
    packed = _c(packed, np.uint8)
    scale = _c(scale, np.float32)
    zero = _c(zero, np.uint8)
    b = None if bias is None else _c(bias, np.uint16)
    y = np.empty((m, n), np.float64)
    a = np.empty((m, n), np.float64)
    _load().orc_linear_int4_groups(_ptr(x), m, k, _ptr(packed), _ptr(scale), _ptr(zero), _ptr(b),
                                   n, group, _ptr(y), _ptr(a))
    return y, a


def linear_int4_groups_ordered(x, order, packed, scale, zero, bias, n: int, group: int):
    """Int4GroupLinear with an activation order ("Quantization" (Linnet docs), format table
    "optional order: [In; i32]", and "Quantizing a checkpoint": a GPTQ checkpoint in
    activation order "gets an order and gathers its inputs first").  Stored column j of
    the weights multiplies input order[j]:  y = x[:, order] . W-hat^T + bias.

    Every entry of order must lie in [0, K) (ValueError otherwise).  Returns (y, absdot)
    as linear_int4_groups.
    """
    x = _c(x, np.uint16)
    order = np.asarray(order)
    if order.ndim != 1 or order.shape[0] != x.shape[1]:
        raise ValueError("order must have one entry per input")
    if (order < 0).any() or (order >= x.shape[1]).any():
        raise ValueError("order entries must lie in [0, K)")
    return linear_int4_groups(x[:, order.astype(np.int64)], packed, scale, zero, bias, n, group)


def linear_int8_rows(x, q, scale, bias=None):
    x = _c(x, np.uint16)
    m, k = x.shape
    q = _c(q, np.int8)
    n = q.shape[0]
    scale = _c(scale, np.float32)
    b = None if bias is None else _c(bias, np.uint16)
    y = np.empty((m, n), np.float64)
    a = np.empty((m, n), np.float64)
    _load().orc_linear_int8_rows(_ptr(x), m, k, _ptr(q), _ptr(scale), _ptr(b), n, _ptr(y), _ptr(a))
    return y, a


def linear_int4_rows(x, packed, scale, bias=None):
    x = _c(x, np.uint16)
    m, k = x.shape
    packed = _c(packed, np.uint8)
    n = packed.shape[0]
    scale = _c(scale, np.float32)
    b = None if bias is None else _c(bias, np.uint16)
    y = np.empty((m, n), np.float64)
    a = np.empty((m, n), np.float64)
    _load().orc_linear_int4_rows(_ptr(x), m, k, _ptr(packed), _ptr(scale), _ptr(b), n, _ptr(y),
                                 _ptr(a))
    return y, a


def mxfp4_experts_shared(x, blocks, scales, experts, n: int, n0: int = 0, n1: int | None = None):
    """x bf16 bits [R, K]; blocks [E, N, K/32, 16]; scales [E, N, K/32]; experts i32 [R, S].

    Returns (y f64 [R, S, N], absdot, bad_slots).  Only columns [n0, n1) are computed;
    the others are NaN.
    """
    x = _c(x, np.uint16)
    r, k = x.shape
    blocks = _c(blocks, np.uint8)
    scales = _c(scales, np.uint8)
    e = blocks.shape[0]
    experts = _c(experts, np.int32)
    s = experts.shape[1]
    n1 = n if n1 is None else n1
    y = np.full((r, s, n), np.nan)
    a = np.full((r, s, n), np.nan)
    bad = _load().orc_mxfp4_experts_shared(_ptr(x), r, k, _ptr(blocks), _ptr(scales), e, n,
                                           _ptr(experts), s, n0, n1, _ptr(y), _ptr(a))
    return y, a, int(bad)


def mxfp4_experts(x, blocks, scales, experts, n: int):
    """mxfp4_experts(x, blocks, scales, experts) ("Quantization" (Linnet docs), format
    table: "a mixture's chosen experts multiplied from MXFP4, each slot its own input"):
        y[r, s, n] = sum_k x[r, s, k] * W-hat[experts[r, s], n, k].
    Each slot is an experts-shared row with one slot.  x bf16 bits [R, S, K].  Returns
    (y f64 [R, S, N], absdot, bad_slots)."""
    x = _c(x, np.uint16)
    r, s, k = x.shape
    experts = _c(experts, np.int32)
    y, a, bad = mxfp4_experts_shared(x.reshape(r * s, k), blocks, scales, experts.reshape(r * s, 1), n)
    return y.reshape(r, s, n), a.reshape(r, s, n), bad


def mxfp4_combine_experts(x, blocks, scales, experts, weights, n: int):
    """mxfp4_combine_experts(x, blocks, scales, experts, weights) ("Quantization" (Linnet
    docs), format table: std.nn.moe::combine_experts with MXFP4 experts).  The page gives
    only the name and the arguments; the reading taken: each row's routed slots share the
    row's input, as in mxfp4_experts_shared, and the row's output is the weighted sum of
    its slots' outputs,
        y[r, n] = sum_s weights[r, s] * sum_k x[r, k] * W-hat[experts[r, s], n, k],
    a slot whose expert index lies outside [0, E) adding nothing.

    x bf16 bits [R, K]; weights f32 [R, S].  Returns (y f64 [R, N], absdot [R, N] =
    sum_s |weights[r, s]| * sum_k |x w|, bad_slots).
    """
    w = _c(weights, np.float32).astype(np.float64)
    ys, a, bad = mxfp4_experts_shared(x, blocks, scales, experts, n)
    y = np.einsum("rs,rsn->rn", w, ys)
    absdot = np.einsum("rs,rsn->rn", np.abs(w), a)
    return y, absdot, bad


def bf16_from_f32(v: float) -> int:
    return int(_load().orc_bf16_from_f32(float(v)))


def e2m1_value(nib: int) -> float:
    return float(_load().orc_e2m1_value(int(nib)))


# ----------------------------------------------------------------------------- tolerance
def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """One bf16 unit in the last place at |v| (for normal values: 2^(e-7))."""
    v = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.maximum(v, 2.0 ** -126)))
    return np.exp2(e - 7)


def within_tolerance(y_gpu: np.ndarray, y_ref: np.ndarray, absdot: np.ndarray,
                     rel: float = 2e-3) -> np.ndarray:
    """|y_gpu - y_ref| <= rel * sum|x*w| + 1 bf16 ulp(y_ref), elementwise."""
    return np.abs(y_gpu - y_ref) <= rel * absdot + bf16_ulp(y_ref)
