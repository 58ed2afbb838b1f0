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
