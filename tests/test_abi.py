"""The C-ABI library loads on a machine without a GPU and exports every entry point
that include/wq.h declares; argument checks that need no device answer correctly."""
import ctypes
import os
import re

import pytest

import weight_only_quantized_linear_gb300 as wq

HEADER = wq.HEADER_PATH


def declared_names():
    src = open(HEADER).read()
    return re.findall(r"WQ_API\s+[\w\s\*]+?\b(wq_\w+)\s*\(", src)


@pytest.fixture(scope="module")
def lib():
    wq.build()
    return wq.lib()


def test_header_declares_the_boundary():
    names = set(declared_names())
    for n in ("wq_linear_int4_groups", "wq_linear_int8_rows", "wq_linear_int4_rows",
              "wq_mxfp4_experts_shared", "wq_quantize_groups", "wq_pack_int4", "wq_unpack_int4",
              "wq_dequantize_int4_groups", "wq_dequantize_int8_rows", "wq_dequantize_int4_rows",
              "wq_dequantize_mxfp4"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(wq.LIB_PATH)
    for name in declared_names():
        assert hasattr(raw, name), f"{name} declared in wq.h but not exported"
    assert set(declared_names()) <= set(wq.SIGNATURES)


def test_status_strings_and_version(lib):
    assert wq.status_string(wq.WQ_OK) == "WQ_OK"
    for st in range(1, 8):
        assert wq.status_string(st).startswith("WQ_E")
    assert lib.wq_version() == 100


def test_host_validation_without_a_device(lib):
    fake = ctypes.c_void_p(0x10000)          # never dereferenced: checks fail first
    # null input
    assert lib.wq_linear_int4_groups(None, 1, 256, fake, fake, fake, None, None, 256, 128, fake, None, 0,
                                     None, None) == wq.WQ_EINVAL
    # an activation order needs room for the gathered activations in the workspace
    assert lib.wq_linear_int4_groups(fake, 1, 256, fake, fake, fake, fake, None, 256, 128, fake, None, 0,
                                     None, None) == wq.WQ_EWORKSPACE
    assert lib.wq_linear_int4_groups_ordered_workspace(1, 256, 256, 128) >= 512
    # ... and the allocation-free entry point has none
    assert lib.wq_linear_int4_groups_noalloc(fake, 1, 256, fake, fake, fake, fake, None, 256, 128, fake,
                                             None, None) == wq.WQ_EUNSUPPORTED
    # the combine form needs its slot workspace
    assert lib.wq_mxfp4_combine_experts(fake, 1, 64, fake, fake, 4, 8, fake, 2, fake, fake, None, 0, None,
                                        None) == wq.WQ_EINVAL
    assert lib.wq_mxfp4_combine_experts_workspace(3, 4, 32, 100, 64) == 3 * 4 * 100 * 4
    # knobs: unknown knob or negative value
    assert lib.wq_set_tuning(99, 1) == wq.WQ_EINVAL and lib.wq_set_tuning(0, -1) == wq.WQ_EINVAL
    assert lib.wq_set_tuning(0, 0) == wq.WQ_OK
    assert lib.wq_last_launch() is not None
    # group must divide K and be one of 32..256
    assert lib.wq_linear_int4_groups(fake, 1, 250, fake, fake, fake, None, None, 256, 128, fake, None, 0,
                                     None, None) == wq.WQ_ESHAPE
    assert lib.wq_linear_int4_groups(fake, 1, 256, fake, fake, fake, None, None, 256, 48, fake, None, 0,
                                     None, None) == wq.WQ_ESHAPE
    # misaligned activations
    assert lib.wq_linear_int4_groups(ctypes.c_void_p(0x10002), 1, 256, fake, fake, fake, None, None, 256,
                                     128, fake, None, 0, None, None) == wq.WQ_EALIGN
    # non-positive sizes
    assert lib.wq_linear_int8_rows(fake, 0, 256, fake, fake, None, 8, fake, None, 0, None, None) == wq.WQ_EINVAL
    assert lib.wq_linear_int8_rows(fake, 1, 40, fake, fake, None, 8, fake, None, 0, None, None) == wq.WQ_ESHAPE
    assert lib.wq_linear_int4_rows(fake, 1, 48, fake, fake, None, 8, fake, None, 0, None, None) == wq.WQ_ESHAPE
    # odd widths are refused by pack / unpack
    assert lib.wq_pack_int4(fake, 2, 3, 0, fake, None, None) == wq.WQ_ESHAPE
    assert lib.wq_unpack_int4(fake, 2, 3, 0, fake, None) == wq.WQ_ESHAPE
    # quantizer modes and widths
    assert lib.wq_quantize_groups(fake, 2, 8, 4, 4, 7, fake, fake, fake, None, None) == wq.WQ_EINVAL
    assert lib.wq_quantize_groups(fake, 2, 8, 4, 8, wq.WQ_SYM_U4, fake, fake, fake, None, None) == wq.WQ_EINVAL
    assert lib.wq_quantize_groups(fake, 2, 8, 4, 4, wq.WQ_ASYM, fake, fake, None, None, None) == wq.WQ_EINVAL
    # MXFP4 needs K in whole blocks of 32
    assert lib.wq_mxfp4_experts_shared(fake, 1, 48, fake, fake, 4, 8, fake, 2, fake, None, 0, None,
                                       None) == wq.WQ_ESHAPE
    assert lib.wq_dequantize_int4_groups(fake, fake, fake, 4, 96, 64, fake, None) == wq.WQ_ESHAPE


def test_mxfp4_workspace_queries_and_regimes(lib):
    """The MXFP4 workspace rules, on the host: no workspace below the grouped GEMM's
    crossover (512 routed rows by default), above it segment and tile starts
    [2, E + 2] i32, the sorted slots [R * S] i32 and the gathered rows [R * S, K] bf16,
    each rounded to 256 bytes; the combine form adds its f32 slot results in front."""
    al = lambda v: (v + 255) // 256 * 256
    gemm_ws = lambda RS, E, K: al(2 * 4 * (E + 2)) + al(4 * RS) + al(RS * K * 2)
    E, N, K, S = 32, 5760, 2880, 4
    assert lib.wq_mxfp4_experts_shared_workspace(127, S, E, N, K) == 0            # 508 slots
    assert lib.wq_mxfp4_combine_experts_workspace(127, S, E, N, K) == 127 * S * N * 4
    for R in (128, 2048):
        need = gemm_ws(R * S, E, K)
        assert lib.wq_mxfp4_experts_shared_workspace(R, S, E, N, K) == need
        assert lib.wq_mxfp4_experts_workspace(R, S, E, N, K) == need
        assert lib.wq_mxfp4_combine_experts_workspace(R, S, E, N, K) == al(R * S * N * 4) + need
    # outside the GEMM's rules: none (K not a multiple of 32, more than 256 experts)
    assert lib.wq_mxfp4_experts_shared_workspace(2048, S, E, N, 2880 + 16) == 0
    assert lib.wq_mxfp4_experts_shared_workspace(2048, S, 300, N, K) == 0
    # the crossover knob moves the regime, and 0 restores it
    try:
        assert lib.wq_set_tuning(wq.WQ_TUNE_MX_GEMM_MIN_SLOTS, 1) == wq.WQ_OK
        assert lib.wq_mxfp4_experts_shared_workspace(2, S, E, N, K) == gemm_ws(2 * S, E, K)
    finally:
        lib.wq_set_tuning(wq.WQ_TUNE_MX_GEMM_MIN_SLOTS, 0)
    assert lib.wq_mxfp4_experts_shared_workspace(2, S, E, N, K) == 0
    # more routed rows than the decode kernels' tables hold, and no workspace: refused
    # before any launch
    fake = ctypes.c_void_p(0x10000)
    assert lib.wq_mxfp4_experts_shared(fake, 1024, 64, fake, fake, 4, 16, fake, 4, fake, None, 0, None,
                                       None) == wq.WQ_EWORKSPACE
    assert lib.wq_mxfp4_experts(fake, 1024, 64, fake, fake, 4, 16, fake, 4, fake, None, 0, None,
                                None) == wq.WQ_EWORKSPACE
