"""Planted mistakes must fail the pins (no GPU).

The mistakes are the pitfalls listed in "Quantization: int8, int4 group (packed), fp8,
KV quant" (OpenLearn TinyLLM module L8.5), section "5. Pitfalls".  Each mutant wraps the
oracle with one planted mistake, on the CPU; the same checks that the real oracle passes
(printed examples, invariants) must reject it.
"""
import numpy as np
import pytest

import oracle
from golden import floats, ints, load


# ------------------------------------------------------------------ checks (shared)
def check_l85_int4(quantize, pack, unpack) -> bool:
    g = load("openlearn_l85_int4_example.txt")
    w = np.array([floats(g["w_row0"]), floats(g["w_row1"])], np.float32)
    codes, scale = quantize(w, 4, 4)
    if codes[0].tolist() != ints(g["codes_row0"]) or codes[1].tolist() != ints(g["codes_row1"]):
        return False
    if scale[:, 0].tolist() != floats(g["scale"]):
        return False
    packed = pack(codes)
    if packed.reshape(-1).tolist() != [int(h, 16) for h in g["bytes_hex"]]:
        return False
    return (unpack(packed, 4) == codes).all()


def check_ch20(quantize) -> bool:
    g = load("inference_ch20_symmetric_example.txt")
    codes, _ = quantize(np.array([floats(g["w"])], np.float32), 5, 4)
    return codes[0].tolist() == ints(g["codes"])


def check_int8(quantize) -> bool:
    g = load("openlearn_l85_int8_example.txt")
    w = np.array([floats(g["w"])], np.float32)
    codes, scale = quantize(w, 4, 8)
    if codes[0].tolist() != ints(g["codes"]):
        return False
    # the row amax maps to +-127 on random rows too
    rng = np.random.default_rng(1)
    w = rng.standard_normal((8, 64)).astype(np.float32)
    codes, _ = quantize(w, 64, 8)
    return (np.abs(codes).max(1) == 127).all()


def check_half_step(quantize) -> bool:
    rng = np.random.default_rng(2)
    w = (rng.standard_normal((16, 128)) * 0.3).astype(np.float32)
    codes, scale = quantize(w, 32, 4)
    s = np.repeat(scale.astype(np.float64), 32, 1)
    return bool((np.abs(w - codes * s) <= s / 2 * (1 + 2.0 ** -18)).all())


def check_nibble_roundtrip(pack, unpack) -> bool:
    lo, hi = np.meshgrid(np.arange(-8, 8), np.arange(-8, 8), indexing="ij")
    pairs = np.stack([lo.ravel(), hi.ravel()], 1).reshape(1, -1).astype(np.int8)
    p = pack(pairs)
    if len(set(p.ravel().tolist())) != 256:
        return False
    if pack(np.array([[-1, 0, -8, 7]], np.int8)).tolist() != [[0x0F, 0x78]]:
        return False
    return (unpack(p, pairs.shape[1]) == pairs).all()


def check_dequant_groups(dequant) -> bool:
    # scale and zero differ along the group axis; the first two groups of one row
    packed = np.full((2, 8), 0x99, np.uint8)                 # every code 9
    scale = np.array([[1.0, 2.0], [4.0, 8.0]], np.float32)
    zero = np.array([[8, 7], [6, 5]], np.uint8)
    w = dequant(packed, scale, zero, 2, 16, 8)
    from test_oracle_pins import bf16_bits_to_f64
    v = bf16_bits_to_f64(w)
    return v[0, :8].tolist() == [1.0] * 8 and v[0, 8:].tolist() == [4.0] * 8 and \
        v[1, :8].tolist() == [12.0] * 8 and v[1, 8:].tolist() == [32.0] * 8


def check_linear(linear) -> bool:
    rng = np.random.default_rng(4)
    from test_oracle_pins import _rand_bf16, bf16_bits_to_f64
    x = _rand_bf16(rng, (2, 64))
    packed = rng.integers(0, 256, (24, 32)).astype(np.uint8)
    scale = (rng.random((24, 2)) * 0.02 + 0.002).astype(np.float32)
    zero = rng.integers(6, 10, (24, 2)).astype(np.uint8)
    bias = _rand_bf16(rng, (24,))
    y = linear(x, packed, scale, zero, bias, 24, 32)
    if y.shape != (2, 24):
        return False
    wdq = bf16_bits_to_f64(oracle.dequant_int4_groups(packed, scale, zero, 24, 64, 32))
    ref = bf16_bits_to_f64(x) @ wdq.T + bf16_bits_to_f64(bias)
    return np.allclose(y, ref, rtol=0, atol=1e-12)


# ------------------------------------------------------------------ the real oracle
def real_quantize(w, group, bits):
    c, s, _ = oracle.quantize_sym(w, group, bits)
    return c, s


def real_pack(codes):
    st, p = oracle.pack_int4(codes, False)
    assert st == 0
    return p


def real_unpack(p, cols):
    return oracle.unpack_int4(p, cols, False)


def real_linear(x, packed, scale, zero, bias, n, group):
    return oracle.linear_int4_groups(x, packed, scale, zero, bias, n, group)[0]


def test_real_oracle_passes_every_check():
    from test_oracle_pins import check_dequant_mxfp4
    assert check_l85_int4(real_quantize, real_pack, real_unpack)
    assert check_ch20(real_quantize)
    assert check_int8(real_quantize)
    assert check_half_step(real_quantize)
    assert check_nibble_roundtrip(real_pack, real_unpack)
    assert check_dequant_groups(oracle.dequant_int4_groups)
    assert check_linear(real_linear)
    assert check_dequant_mxfp4(oracle.dequant_mxfp4)


def _check_mx(dequant) -> bool:
    from test_oracle_pins import check_dequant_mxfp4
    return check_dequant_mxfp4(dequant)


def mut_mx_scale_per_16(blocks, scales, e, n, k):       # one scale byte per 16 elements
    s = np.repeat(scales, 2, -1)[..., : k // 32]
    return oracle.dequant_mxfp4(blocks, np.ascontiguousarray(s), e, n, k)


def mut_mx_scales_transposed(blocks, scales, e, n, k):   # scales stored [E, K/32, N]
    s = np.ascontiguousarray(scales.reshape(e, k // 32, n).transpose(0, 2, 1))
    return oracle.dequant_mxfp4(blocks, s, e, n, k)


def mut_mx_swapped_nibbles(blocks, scales, e, n, k):     # even element in the high nibble
    return oracle.dequant_mxfp4(_swap_nibbles(blocks), scales, e, n, k)


def mut_mx_bias_128(blocks, scales, e, n, k):            # E8M0 bias 128
    s = np.where(scales == 255, 255, np.maximum(scales.astype(np.int16) - 1, 0)).astype(np.uint8)
    return oracle.dequant_mxfp4(blocks, s, e, n, k)


def mut_mx_expert_stride(blocks, scales, e, n, k):       # every expert reads expert 0's scales
    s = np.ascontiguousarray(np.broadcast_to(scales[:1], scales.shape))
    return oracle.dequant_mxfp4(blocks, s, e, n, k)


# ------------------------------------------------------------------ mutants
def _swap_nibbles(p):
    return ((p >> 4) | (p << 4)).astype(np.uint8)


def mut_s01_pack(codes):                       # even column in the high nibble
    return _swap_nibbles(real_pack(codes))


def mut_s01_unpack(p, cols):
    return real_unpack(_swap_nibbles(p), cols)


def mut_s02_pack(codes):                       # offset binary instead of two's complement
    c = (codes.astype(np.int16) + 8).astype(np.uint8)
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


def mut_s03_unpack(p, cols):                   # no sign extension
    return oracle.unpack_int4(p, cols, True).astype(np.int16)


def mut_s04_quantize(w, group, bits):          # truncation instead of rint
    q = 2 ** (bits - 1) - 1
    n, k = w.shape
    blocks = w.reshape(n, -1, group).astype(np.float32)
    a = np.abs(blocks).max(-1, keepdims=True)
    s = np.where(a > 0, a / np.float32(q), np.float32(1)).astype(np.float32)
    r = np.where(a > 0, np.float32(q) / a, np.float32(1)).astype(np.float32)
    codes = np.clip(np.trunc(blocks * r), -q, q).astype(np.int8)
    return codes.reshape(n, k), s[..., 0]


def _scaled(divisor_of_amax):
    def quantize(w, group, bits):
        q = 2 ** (bits - 1) - 1
        d = divisor_of_amax(q)
        n, k = w.shape
        blocks = w.reshape(n, -1, group).astype(np.float32)
        a = np.abs(blocks).max(-1, keepdims=True)
        s = np.where(a > 0, a / np.float32(d), np.float32(1)).astype(np.float32)
        codes = np.clip(np.rint(blocks / s), -q, q).astype(np.int8)
        return codes.reshape(n, k), s[..., 0]
    return quantize


mut_s06_quantize = _scaled(lambda q: 128 if q == 127 else q)     # int8 scale amax/128
mut_s08_quantize = _scaled(lambda q: q + 1)                      # int4 scale amax/8


def mut_s05_quantize(w, group, bits):          # int8 codes cast without rounding
    c, s = real_quantize(w, group, bits)
    if bits == 8:
        n, k = w.shape
        sr = np.repeat(s, group, 1)
        c = np.clip((w / sr).astype(np.int8), -127, 127).astype(np.int8)
    return c, s


def mut_s11_quantize(w, group, bits):          # one scale per tensor
    q = 2 ** (bits - 1) - 1
    a = np.float32(np.abs(w).max())
    s = a / np.float32(q)
    codes = np.clip(np.rint(w / s), -q, q).astype(np.int8)
    return codes, np.full((w.shape[0], -(-w.shape[1] // group)), s, np.float32)


def mut_m01_dequant(packed, scale, zero, n, k, group):   # scales along the wrong axis
    return oracle.dequant_int4_groups(packed, np.ascontiguousarray(scale.T).reshape(scale.shape),
                                      np.ascontiguousarray(zero.T).reshape(zero.shape), n, k, group)


def mut_s16_linear(x, packed, scale, zero, bias, n, group):   # bias dropped
    return oracle.linear_int4_groups(x, packed, scale, zero, None, n, group)[0]


def mut_s17_linear(x, packed, scale, zero, bias, n, group):   # W read as [K, N], not W^T
    from test_oracle_pins import bf16_bits_to_f64
    k = x.shape[1]
    wdq = bf16_bits_to_f64(oracle.dequant_int4_groups(packed, scale, zero, n, k, group))
    return bf16_bits_to_f64(x) @ wdq.reshape(k, n) + bf16_bits_to_f64(bias)


@pytest.mark.parametrize("name,check", [
    ("s01 swapped nibbles", lambda: check_l85_int4(real_quantize, mut_s01_pack, mut_s01_unpack)
     and check_nibble_roundtrip(mut_s01_pack, mut_s01_unpack)),
    ("s02 offset binary", lambda: check_l85_int4(real_quantize, mut_s02_pack, real_unpack)
     and check_nibble_roundtrip(mut_s02_pack, real_unpack)),
    ("s03 no sign extension", lambda: check_l85_int4(real_quantize, real_pack, mut_s03_unpack)
     and check_nibble_roundtrip(real_pack, mut_s03_unpack)),
    ("s04 truncation", lambda: check_ch20(mut_s04_quantize) and check_half_step(mut_s04_quantize)
     and check_l85_int4(mut_s04_quantize, real_pack, real_unpack)),
    ("s05 int8 cast without rounding", lambda: check_int8(mut_s05_quantize)),
    ("s06 int8 amax/128", lambda: check_int8(mut_s06_quantize)),
    ("s08 int4 amax/8", lambda: check_half_step(mut_s08_quantize)
     and check_l85_int4(mut_s08_quantize, real_pack, real_unpack)),
    ("s11 per-tensor scale", lambda: check_int8(mut_s11_quantize)
     and check_l85_int4(mut_s11_quantize, real_pack, real_unpack)),
    ("m01 scales along the wrong axis", lambda: check_dequant_groups(mut_m01_dequant)),
    ("s16 bias dropped", lambda: check_linear(mut_s16_linear)),
    ("s17 W instead of W^T", lambda: check_linear(mut_s17_linear)),
    ("mx one scale per 16", lambda: _check_mx(mut_mx_scale_per_16)),
    ("mx scales transposed over N", lambda: _check_mx(mut_mx_scales_transposed)),
    ("mx swapped nibbles", lambda: _check_mx(mut_mx_swapped_nibbles)),
    ("mx E8M0 bias 128", lambda: _check_mx(mut_mx_bias_128)),
    ("mx expert stride dropped", lambda: _check_mx(mut_mx_expert_stride)),
])
def test_mutant_is_caught(name, check):
    assert not check(), f"planted mistake not caught: {name}"


def test_literal_f32_division_misses_the_printed_example():
    """The literal f32 quotient w / fl32(a / Q) gives -3 / 3 on the printed example
    (the reading that rounds fl32(w * fl32(Q / a)) reproduces the page)."""
    assert not check_ch20(_scaled(lambda q: q))
