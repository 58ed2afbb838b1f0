"""GPU quantize / pack / unpack / dequantize: bit-exact against the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle
import weight_only_quantized_linear_gb300 as wq
from weight_only_quantized_linear_gb300 import synth
from gpu_util import bf16_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    wq.build()


def _status(dev):
    return torch.zeros(1, dtype=torch.int32, device=dev)


@pytest.mark.parametrize("bits", [2, 3, 4, 8])
@pytest.mark.parametrize("group", [1, 7, 32, 128, 250])
def test_quantize_sym_and_asym_match_oracle(cuda_device, bits, group):
    w = synth.weight_f32(37, 500, seed=bits * 100 + group, outlier_frac=0.01)
    w_np = w.numpy()
    dev_w = w.to(cuda_device)
    st = _status(cuda_device)
    c, s, z = wq.wq_quantize_groups(dev_w, group, bits, wq.WQ_SYM, dev_status=st)
    oc, os_, ref = oracle.quantize_sym(w_np, group, bits)
    assert (c.cpu().numpy() == oc).all() and (s.cpu().numpy().view(np.uint32) == os_.view(np.uint32)).all()
    c, s, z = wq.wq_quantize_groups(dev_w, group, bits, wq.WQ_ASYM, dev_status=st)
    oc, os_, oz, _ = oracle.quantize_asym(w_np, group, bits)
    assert (c.cpu().numpy() == oc).all()
    assert (s.cpu().numpy().view(np.uint32) == os_.view(np.uint32)).all()
    assert (z.cpu().numpy() == oz).all()
    if bits == 4:
        c, s, z = wq.wq_quantize_groups(dev_w, group, 4, wq.WQ_SYM_U4, dev_status=st)
        oc, os_, _ = oracle.quantize_sym(w_np, group, 4)
        assert (c.cpu().numpy().astype(np.int16) - 8 == oc).all() and (z.cpu() == 8).all()
    assert int(st.item()) == 0


def test_quantize_llama_gate_shape_bit_exact(cuda_device):
    # the weights the decode benchmark uses: N(0, 0.02) with 0.1 % outliers x20, G = 128
    w = synth.weight_f32(14336, 4096, seed=0, outlier_frac=0.001)
    c, s, z = wq.wq_quantize_groups(w.to(cuda_device), 128, 4, wq.WQ_ASYM)
    oc, os_, oz, refused = oracle.quantize_asym(w.numpy(), 128, 4)
    assert refused == 0
    assert (c.cpu().numpy() == oc).all()
    assert (s.cpu().numpy().view(np.uint32) == os_.view(np.uint32)).all()
    assert (z.cpu().numpy() == oz).all()


def test_quantize_edge_groups(cuda_device):
    w = np.zeros((6, 64), np.float32)
    w[1, :32] = np.linspace(-1e-39, 1e-39, 32, dtype=np.float32)   # tiny: literal quotient path
    w[2, 5] = np.nan
    w[3, 40] = -np.inf
    w[4, :32] = 3e38
    w[4, 32:] = -3e38                                              # asym range overflow in no group
    w[5, :16] = 3e38
    w[5, 16:32] = -3e38                                            # asym range overflows here
    for mode in (wq.WQ_SYM, wq.WQ_ASYM):
        st = _status(cuda_device)
        c, s, z = wq.wq_quantize_groups(torch.from_numpy(w).to(cuda_device), 32, 4, mode, dev_status=st)
        if mode == wq.WQ_SYM:
            oc, os_, refused = oracle.quantize_sym(w, 32, 4)
        else:
            oc, os_, oz, refused = oracle.quantize_asym(w, 32, 4)
            assert (z.cpu().numpy() == oz).all()
        assert (c.cpu().numpy() == oc).all()
        assert (s.cpu().numpy().view(np.uint32) == os_.view(np.uint32)).all()
        assert refused > 0 and (int(st.item()) & wq.WQ_DEV_NONFINITE)


def test_pack_unpack_roundtrip_and_bad_codes(cuda_device):
    allb = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(1, 256).to(cuda_device)
    for uns in (False, True):
        codes = wq.wq_unpack_int4(allb, 512, uns)
        ref = oracle.unpack_int4(allb.cpu().numpy(), 512, uns)
        assert (codes.cpu().numpy() == ref).all()
        st = _status(cuda_device)
        assert (wq.wq_pack_int4(codes, uns, dev_status=st) == allb).all()
        assert int(st.item()) == 0
    rng = np.random.default_rng(0)
    codes = rng.integers(-8, 8, (33, 130)).astype(np.int8)
    got = wq.wq_pack_int4(torch.from_numpy(codes).to(cuda_device), False)
    assert (got.cpu().numpy() == oracle.pack_int4(codes, False)[1]).all()
    st = _status(cuda_device)
    bad = torch.tensor([[9, 0, 1, -9]], dtype=torch.int8, device=cuda_device)
    wq.wq_pack_int4(bad, False, dev_status=st)
    assert int(st.item()) & wq.WQ_DEV_BAD_CODE


def test_dequant_int4_groups_bit_exact(cuda_device):
    rng = np.random.default_rng(1)
    n, k, g = 512, 512, 32
    scale = (rng.standard_normal((n, k // g)) * 10.0 ** rng.integers(-30, 30, (n, k // g))).astype(np.float32)
    scale[0, :4] = [0.0, -0.0, 1e-45, 3e38]
    zero = rng.integers(0, 16, (n, k // g)).astype(np.uint8)
    packed = rng.integers(0, 256, (n, k // 2)).astype(np.uint8)
    d = lambda a: torch.from_numpy(a).to(cuda_device)
    got = wq.wq_dequantize_int4_groups(d(packed), d(scale), d(zero), k, g)
    assert (bf16_bits(got) == oracle.dequant_int4_groups(packed, scale, zero, n, k, g)).all()


def test_dequant_rows_bit_exact(cuda_device):
    rng = np.random.default_rng(2)
    q = rng.integers(-128, 128, (300, 96)).astype(np.int8)
    s = (rng.random(300) * 10.0 ** rng.integers(-20, 20, 300)).astype(np.float32)
    d = lambda a: torch.from_numpy(a).to(cuda_device)
    assert (bf16_bits(wq.wq_dequantize_int8_rows(d(q), d(s))) == oracle.dequant_int8_rows(q, s)).all()
    p = rng.integers(0, 256, (300, 48)).astype(np.uint8)
    got = wq.wq_dequantize_int4_rows(d(p.view(np.int8)), d(s), 96)
    assert (bf16_bits(got) == oracle.dequant_int4_rows(p, s, 96)).all()


def test_dequant_mxfp4_every_code_and_scale(cuda_device):
    # every (code, scale byte) pair: 256 scale bytes x 32 elements covering the 16 codes twice
    e, n, k = 1, 256, 32
    nibs = np.arange(32) % 16
    blocks = np.tile((nibs[0::2] | (nibs[1::2] << 4)).astype(np.uint8), (e, n, 1, 1))
    scales = np.arange(256, dtype=np.uint8).reshape(e, n, 1)
    d = lambda a: torch.from_numpy(a).to(cuda_device)
    got = bf16_bits(wq.wq_dequantize_mxfp4(d(blocks), d(scales)))
    ref = oracle.dequant_mxfp4(blocks, scales, e, n, k)
    nan = ((ref & 0x7F80) == 0x7F80) & ((ref & 0x7F) != 0)
    assert (got[~nan] == ref[~nan]).all()
    assert (((got[nan] & 0x7F80) == 0x7F80) & ((got[nan] & 0x7F) != 0)).all()
    # random blocks at the gpt-oss scale range
    bl, sc = synth.mxfp4_experts(4, 64, 2880, seed=3)
    got = bf16_bits(wq.wq_dequantize_mxfp4(bl.to(cuda_device), sc.to(cuda_device)))
    assert (got == oracle.dequant_mxfp4(bl.numpy(), sc.numpy(), 4, 64, 2880)).all()
