"""Pins of the CPU oracle against what the pages and mathematics fix (no GPU).

Each test ties an oracle function to something other than itself: a value the pages
print (fixtures under tests/golden/, each citing its page and section), a closed form,
an invariant the pages state, a library routine of torch, or brute force on tiny
inputs.  ``test_oracle_mutants.py`` checks that these pins catch planted mistakes.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from golden import floats, ints, load


def bf16_bits_to_f64(b):
    return torch.from_numpy(np.asarray(b, np.uint16).view(np.int16).copy()).view(torch.bfloat16).double().numpy()


def f32_to_bf16_bits_torch(a):
    t = torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


# ------------------------------------------------------------------ printed examples
def test_ch20_symmetric_worked_example():
    g = load("inference_ch20_symmetric_example.txt")
    w = np.array([floats(g["w"])], np.float32)
    codes, scale, refused = oracle.quantize_sym(w, int(g["group"][0]), int(g["bits"][0]))
    assert refused == 0
    assert codes[0].tolist() == ints(g["codes"])
    what = codes[0].astype(np.float32) * scale[0, 0]
    assert np.allclose(what, floats(g["what_printed"]), atol=5e-4)
    # the page: the error on +-1 is exactly s/2
    s = float(scale[0, 0])
    assert abs(abs(float(what[1]) - (-1.0)) - s / 2) < 1e-6


def test_l85_int4_worked_example():
    g = load("openlearn_l85_int4_example.txt")
    w = np.array([floats(g["w_row0"]), floats(g["w_row1"])], np.float32)
    codes, scale, refused = oracle.quantize_sym(w, int(g["group"][0]), int(g["bits"][0]))
    assert refused == 0
    assert scale[:, 0].tolist() == floats(g["scale"])
    assert codes[0].tolist() == ints(g["codes_row0"])
    assert codes[1].tolist() == ints(g["codes_row1"])
    st, packed = oracle.pack_int4(codes, is_unsigned=False)
    assert st == 0
    assert packed.reshape(-1).tolist() == [int(h, 16) for h in g["bytes_hex"]]
    back = oracle.unpack_int4(packed, 4, is_unsigned=False)
    assert (back == codes).all()
    what = codes.astype(np.float32) * scale
    assert what[0].tolist() == floats(g["what_row0"])
    assert what[1].tolist() == floats(g["what_row1"])
    assert np.abs(what - w).max() <= float(g["max_error"][0])
    # the same values through the group-wise asymmetric layout: codes + 8, zero 8
    ucodes = (codes.astype(np.int16) + 8).astype(np.uint8)
    st, upacked = oracle.pack_int4(ucodes, is_unsigned=True)
    assert st == 0
    deq = oracle.dequant_int4_groups(upacked, scale, np.full((2, 1), 8, np.uint8), 2, 4, 4)
    assert bf16_bits_to_f64(deq).tolist() == what.astype(np.float64).tolist()


def test_l85_int8_worked_example():
    g = load("openlearn_l85_int8_example.txt")
    w = np.array([floats(g["w"])], np.float32)
    codes, scale, _ = oracle.quantize_sym(w, w.shape[1], int(g["bits"][0]))
    assert scale[0, 0] == float(g["scale"][0])
    assert codes[0].tolist() == ints(g["codes"])


def test_mxfp4_value_table_and_scale():
    g = load("openlearn_l85_mxfp4_values.txt")
    mags = floats(g["magnitudes"])
    for nib in range(16):
        v = oracle.e2m1_value(nib)
        expect = mags[nib & 7] * (-1.0 if nib & 8 else 1.0)
        assert v == expect and math.copysign(1.0, v) == (-1.0 if nib & 8 else 1.0)
    # one block of 32 at scale byte 127 (X = 1) reproduces the table; 128 doubles it;
    # 120 multiplies by 2^-7 (torch.ldexp as the independent routine)
    k = 32
    nibs = np.arange(32) % 16
    blocks = (nibs[0::2] | (nibs[1::2] << 4)).astype(np.uint8).reshape(1, 1, 1, 16)
    for sc in (127, 128, 120, 118, 124):
        deq = oracle.dequant_mxfp4(blocks, np.array([[[sc]]], np.uint8), 1, 1, k)
        table = torch.tensor([mags[n & 7] * (-1.0 if n & 8 else 1.0) for n in nibs], dtype=torch.float64)
        expect = torch.ldexp(table, torch.tensor(sc - 127, dtype=torch.float64))
        assert bf16_bits_to_f64(deq[0, 0]).tolist() == expect.tolist()
    # 4.25 bits per weight: 16 code bytes + 1 scale byte per block of 32
    assert (16 + 1) * 8 / int(g["block"][0]) == float(g["bits_per_weight"][0])


def mxfp4_torch_restatement(blocks: np.ndarray, scales: np.ndarray) -> torch.Tensor:
    """dequantize_mxfp4 written again with torch alone ("Quantization" (Linnet docs),
    format table: E2M1 values in blocks of 32 along K, one E8M0 scale byte a block;
    "Quantization: int8, int4 group (packed), fp8, KV quant", 2. Principles, MXFP4: the
    printed magnitudes times the block's power of two): nibbles by torch bit ops (even
    element low), the printed table by indexing, the block scale by repeat_interleave
    and torch.ldexp, bias 127, scale byte 255 giving NaN.  Returns f64 [E, N, K]."""
    g = load("openlearn_l85_mxfp4_values.txt")
    mags = torch.tensor(floats(g["magnitudes"]), dtype=torch.float64)
    b = torch.from_numpy(np.ascontiguousarray(blocks)).to(torch.int64)
    e, n, nb, _ = b.shape
    nib = torch.stack([b & 15, b >> 4], dim=-1).reshape(e, n, nb * 32)
    val = mags[nib & 7] * torch.where((nib & 8) != 0, -1.0, 1.0).to(torch.float64)
    sc = torch.from_numpy(np.ascontiguousarray(scales)).to(torch.int64).repeat_interleave(32, dim=-1)
    out = torch.ldexp(val, (sc - 127).to(torch.float64))
    return torch.where(sc == 255, torch.full_like(out, float("nan")), out)


def check_dequant_mxfp4(dequant) -> bool:
    """A dequantizer over several experts, rows and blocks (E = 2, N = 3, K = 128: every
    scale byte distinct along each axis, codes covering all 16 values in every block) and
    over the whole E8M0 range 0..255 equals the torch restatement bit for bit (NaN where
    the scale byte is 255)."""
    rng = np.random.default_rng(17)
    e, n, k = 2, 3, 128
    nibs = np.stack([rng.permutation(16) for _ in range(e * n * (k // 16))]).reshape(e, n, k)
    blocks = (nibs[..., 0::2] | (nibs[..., 1::2] << 4)).astype(np.uint8).reshape(e, n, k // 32, 16)
    scales = rng.choice(np.arange(110, 135), size=(e, n, k // 32), replace=False).astype(np.uint8)
    for sc in (scales, np.arange(256, dtype=np.uint8).reshape(2, 4, 32)):
        ee, nn, kk = sc.shape[0], sc.shape[1], sc.shape[2] * 32
        bl = blocks if sc is scales else rng.integers(0, 256, (ee, nn, kk // 32, 16)).astype(np.uint8)
        got = bf16_bits_to_f64(dequant(bl, sc, ee, nn, kk))
        want = mxfp4_torch_restatement(bl, sc)
        want_bf16 = want.to(torch.bfloat16).double().numpy()   # the products are bf16 values
        if not np.array_equal(got, want_bf16, equal_nan=True):
            return False
        if not np.array_equal(np.isnan(got), (np.repeat(sc, 32, -1) == 255)):
            return False
    return True


def test_dequant_mxfp4_across_experts_rows_and_blocks():
    """orc_dequant_mxfp4 past one block: the block-scale index (row * K/32 + k/32 over
    experts and rows) and the nibble order against an independent torch restatement, and
    the E8M0 reading (bias 127, 255 = NaN) over every scale byte."""
    assert check_dequant_mxfp4(oracle.dequant_mxfp4)
    # the E8M0 end points on their own: byte 0 is 2^-127, byte 254 is 2^127, 255 is NaN
    one = np.full((1, 1, 1, 16), 0x22, np.uint8)            # every code 2: magnitude 1.0
    for byte, want in ((0, 2.0 ** -127), (127, 1.0), (254, 2.0 ** 127)):
        v = bf16_bits_to_f64(oracle.dequant_mxfp4(one, np.array([[[byte]]], np.uint8), 1, 1, 32))
        assert (v == want).all()
    v = bf16_bits_to_f64(oracle.dequant_mxfp4(one, np.array([[[255]]], np.uint8), 1, 1, 32))
    assert np.isnan(v).all()


# ------------------------------------------------------------------ symmetric quantizer
def test_zero_group_gets_scale_one():
    w = np.zeros((3, 64), np.float32)
    w[1, 40:] = 0.5                       # group 1 of row 1 nonzero
    codes, scale, _ = oracle.quantize_sym(w, 32, 4)
    assert scale[0].tolist() == [1.0, 1.0] and scale[2].tolist() == [1.0, 1.0]
    assert scale[1, 0] == 1.0 and scale[1, 1] == np.float32(0.5) / np.float32(7)
    assert (codes[0] == 0).all() and (codes[1, :32] == 0).all()


def test_short_last_group_equals_padded():
    rng = np.random.default_rng(7)
    w = (rng.standard_normal((5, 250)) * 0.02).astype(np.float32)
    pad = np.zeros((5, 256), np.float32)
    pad[:, :250] = w
    for bits in (2, 3, 4, 8):
        c1, s1, _ = oracle.quantize_sym(w, 32, bits)
        c2, s2, _ = oracle.quantize_sym(pad, 32, bits)
        assert (c1 == c2[:, :250]).all() and (s1 == s2).all()
    c1, s1, z1, _ = oracle.quantize_asym(w, 32, 4)
    c2, s2, z2, _ = oracle.quantize_asym(pad, 32, 4)
    assert (c1 == c2[:, :250]).all() and (s1 == s2).all() and (z1 == z2).all()


@pytest.mark.parametrize("bits", [2, 3, 4, 8])
def test_half_step_bound_and_amax_maps_to_q(bits):
    rng = np.random.default_rng(bits)
    q = 2 ** (bits - 1) - 1
    for group in (16, 32, 64):
        for mag in (1e-3, 1.0, 100.0):
            w = (rng.standard_normal((16, 4 * group)) * mag).astype(np.float32)
            codes, scale, _ = oracle.quantize_sym(w, group, bits)
            assert np.abs(codes).max() <= q
            s = np.repeat(scale.astype(np.float64), group, axis=1)
            what = codes.astype(np.float64) * s
            assert (np.abs(w - what) <= s / 2 * (1 + 2.0 ** -18)).all()
            blocks = np.abs(w).reshape(16, 4, group)
            arg = blocks.argmax(-1)
            cb = codes.reshape(16, 4, group)
            top = np.take_along_axis(cb, arg[..., None], -1)[..., 0]
            assert (np.abs(top) == q).all()


def test_ties_go_to_even():
    # scale 1 (amax 7 at 4 bits): halves must round to the even code
    w = np.array([[7.0, 0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 3.5]], np.float32)
    codes, scale, _ = oracle.quantize_sym(w, 8, 4)
    assert scale[0, 0] == 1.0
    assert codes[0].tolist() == [7, 0, 2, 2, 0, -2, -2, 4]


def test_non_finite_group_is_refused():
    w = np.ones((2, 64), np.float32)
    w[1, 3] = np.nan
    w[0, 40] = np.inf
    codes, scale, refused = oracle.quantize_sym(w, 32, 4)
    assert refused == 2
    assert scale[1, 0] == 1.0 and (codes[1, :32] == 0).all()
    assert scale[0, 1] == 1.0 and (codes[0, 32:] == 0).all()
    assert (codes[0, :32] == 7).all()
    c, s, z, refused = oracle.quantize_asym(w, 32, 4)
    assert refused == 2 and (c[1, :32] == 8).all() and z[1, 0] == 8


def test_tiny_groups_use_the_literal_quotient():
    # amax so small that Q / amax overflows f32: codes still follow rint(w / s)
    w = np.array([[1e-39, -5e-40, 0.0, 2.5e-40]], np.float32)
    codes, scale, refused = oracle.quantize_sym(w, 4, 4)
    assert refused == 0 and np.isfinite(scale).all()
    s = np.float32(scale[0, 0])
    expect = np.clip(np.rint(w / s), -7, 7).astype(np.int8)
    assert (codes == expect).all() and codes[0, 0] == 7


# ------------------------------------------------------------------ asymmetric quantizer
def test_asym_invariants():
    rng = np.random.default_rng(11)
    for group in (32, 128):
        w = (rng.standard_normal((64, 4 * group)) * 0.02).astype(np.float32)
        w[0, :group] = np.abs(w[0, :group])          # all-positive group -> zero = 0
        w[1, :group] = -np.abs(w[1, :group])         # all-negative group -> zero = 15
        w[2, :group] = 0.0                           # zero group
        w[3, 5] = 0.0
        codes, scale, zero, refused = oracle.quantize_asym(w, group, 4)
        assert refused == 0
        assert codes.max() <= 15 and zero.max() <= 15
        assert zero[0, 0] == 0 and zero[1, 0] == 15
        assert scale[2, 0] == 1.0 and zero[2, 0] == 8 and (codes[2, :group] == 8).all()
        z = np.repeat(zero.astype(np.float64), group, axis=1)
        s = np.repeat(scale.astype(np.float64), group, axis=1)
        what = (codes.astype(np.float64) - z) * s
        assert (np.abs(w - what) <= s / 2 * (1 + 2.0 ** -18)).all()
        assert (what[w == 0.0] == 0.0).all()         # zero maps to zero exactly


# ------------------------------------------------------------------ pack / unpack
def test_pack_unpack_every_byte_and_pair():
    allb = np.arange(256, dtype=np.uint8).reshape(1, 256)
    for uns in (False, True):
        codes = oracle.unpack_int4(allb, 512, is_unsigned=uns)
        st, packed = oracle.pack_int4(codes, is_unsigned=uns)
        assert st == 0 and (packed == allb).all()
    lo, hi = np.meshgrid(np.arange(-8, 8), np.arange(-8, 8), indexing="ij")
    pairs = np.stack([lo.ravel(), hi.ravel()], 1).reshape(1, -1).astype(np.int8)
    st, packed = oracle.pack_int4(pairs, is_unsigned=False)
    assert st == 0 and len(set(packed.ravel().tolist())) == 256
    # two's complement nibbles: -1 -> 0xF, -8 -> 0x8, even column low
    st, p = oracle.pack_int4(np.array([[-1, 0, -8, 7]], np.int8), is_unsigned=False)
    assert p.tolist() == [[0x0F, 0x78]]


def test_pack_refuses_odd_width_and_out_of_range():
    assert oracle.pack_int4(np.zeros((2, 3), np.int8), False)[0] == 1
    assert oracle.pack_int4(np.array([[8, 0]], np.int8), False)[0] == 2
    assert oracle.pack_int4(np.array([[-9, 0]], np.int8), False)[0] == 2
    assert oracle.pack_int4(np.array([[16, 0]], np.uint8), True)[0] == 2
    assert oracle.pack_int4(np.array([[15, 0]], np.uint8), True)[0] == 0


# ------------------------------------------------------------------ dequant vs torch
def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(3)
    vals = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(10.0) ** rng.integers(-40, 38, 20000),
        np.array([0.0, -0.0, np.inf, -np.inf, 1e-45, 3e38, 3.4e38, 1.00390625, 1.01171875,
                  -1.00390625, 2.0 ** -133, 2.0 ** -127], np.float32),
    ]).astype(np.float32)
    # exact ties: low 16 bits 0x8000 with both parities of the kept part
    ties = (rng.integers(0, 2 ** 15, 4000, dtype=np.uint32) << 16 | 0x8000).astype(np.uint32).view(np.float32)
    vals = np.concatenate([vals, ties])
    ours = np.array([oracle.bf16_from_f32(v) for v in vals], np.uint16)
    nan = np.isnan(vals)
    assert (ours[~nan] == f32_to_bf16_bits_torch(vals)[~nan]).all()
    # NaN payloads differ between libraries; NaN must stay NaN (exponent all ones,
    # mantissa nonzero)
    assert ((ours[nan] & 0x7F80) == 0x7F80).all() and ((ours[nan] & 0x7F) != 0).all()


def test_dequant_int4_groups_all_codes_and_zeros_vs_torch():
    rng = np.random.default_rng(5)
    n, k, gsz = 625, 256, 16                     # 10^4 (row, group) scales
    scale = (rng.standard_normal((n, k // gsz)) * 10.0 ** rng.integers(-6, 4, (n, k // gsz))).astype(np.float32)
    zero = rng.integers(0, 16, (n, k // gsz)).astype(np.uint8)
    codes = np.tile(np.arange(16, dtype=np.uint8), (n, k // 16))   # every code in every group
    st, packed = oracle.pack_int4(codes, is_unsigned=True)
    deq = oracle.dequant_int4_groups(packed, scale, zero, n, k, gsz)
    qz = torch.from_numpy(codes.astype(np.int32)) - torch.from_numpy(zero.astype(np.int32)).repeat_interleave(gsz, 1)
    ref = (qz.float() * torch.from_numpy(scale).repeat_interleave(gsz, 1)).to(torch.bfloat16)
    assert (deq == ref.view(torch.int16).numpy().view(np.uint16)).all()


def test_dequant_rows_vs_torch():
    rng = np.random.default_rng(6)
    q8 = rng.integers(-127, 128, (33, 64)).astype(np.int8)
    s = (rng.random(33) * 0.05 + 1e-4).astype(np.float32)
    ref = (torch.from_numpy(q8).float() * torch.from_numpy(s)[:, None]).to(torch.bfloat16)
    assert (oracle.dequant_int8_rows(q8, s) == ref.view(torch.int16).numpy().view(np.uint16)).all()
    q4 = rng.integers(-8, 8, (33, 64)).astype(np.int8)
    st, p = oracle.pack_int4(q4, is_unsigned=False)
    ref = (torch.from_numpy(q4).float() * torch.from_numpy(s)[:, None]).to(torch.bfloat16)
    assert (oracle.dequant_int4_rows(p, s, 64) == ref.view(torch.int16).numpy().view(np.uint16)).all()


# ------------------------------------------------------------------ linear
def _rand_bf16(rng, shape, scale=1.0):
    return f32_to_bf16_bits_torch((rng.standard_normal(shape) * scale).astype(np.float32))


def test_linear_brute_force_tiny():
    rng = np.random.default_rng(8)
    x = _rand_bf16(rng, (2, 8))
    w = _rand_bf16(rng, (3, 8))
    b = _rand_bf16(rng, (3,))
    y, a = oracle.linear_bf16(x, w, b)
    xf, wf, bf = bf16_bits_to_f64(x), bf16_bits_to_f64(w), bf16_bits_to_f64(b)
    for m in range(2):
        for n in range(3):
            terms = [xf[m, k] * wf[n, k] for k in range(8)]
            assert y[m, n] == pytest.approx(math.fsum(terms) + bf[n], rel=0, abs=1e-14)
            assert a[m, n] == pytest.approx(math.fsum(abs(t) for t in terms), rel=1e-15)


def test_linear_int4_groups_vs_torch_and_one_hot():
    rng = np.random.default_rng(9)
    m, n, k, gsz = 3, 40, 256, 32
    x = _rand_bf16(rng, (m, k))
    packed = rng.integers(0, 256, (n, k // 2)).astype(np.uint8)
    scale = (rng.random((n, k // gsz)) * 0.018 + 0.002).astype(np.float32)
    zero = rng.integers(6, 10, (n, k // gsz)).astype(np.uint8)
    bias = _rand_bf16(rng, (n,))
    y, a = oracle.linear_int4_groups(x, packed, scale, zero, bias, n, gsz)
    wdq = oracle.dequant_int4_groups(packed, scale, zero, n, k, gsz)
    ref = torch.nn.functional.linear(torch.from_numpy(bf16_bits_to_f64(x)), torch.from_numpy(bf16_bits_to_f64(wdq)),
                                     torch.from_numpy(bf16_bits_to_f64(bias)))
    assert np.allclose(y, ref.numpy(), rtol=0, atol=1e-12)
    # one-hot input picks one dequantized column exactly
    for kk in (0, 1, 77, 255):
        e = np.zeros((1, k), np.uint16)
        e[0, kk] = 0x3F80                         # bf16 1.0
        y1, _ = oracle.linear_int4_groups(e, packed, scale, zero, None, n, gsz)
        assert (y1[0] == bf16_bits_to_f64(wdq[:, kk])).all()
    # W^T, not W: a non-square layer has output width N
    assert y.shape == (m, n)


def test_linear_rows_vs_torch():
    rng = np.random.default_rng(10)
    m, n, k = 2, 24, 96
    x = _rand_bf16(rng, (m, k))
    q8 = rng.integers(-127, 128, (n, k)).astype(np.int8)
    s = (rng.random(n) * 0.01 + 1e-4).astype(np.float32)
    y, _ = oracle.linear_int8_rows(x, q8, s)
    ref = bf16_bits_to_f64(x) @ bf16_bits_to_f64(oracle.dequant_int8_rows(q8, s)).T
    assert np.allclose(y, ref, rtol=0, atol=1e-12)
    q4 = rng.integers(-8, 8, (n, k)).astype(np.int8)
    _, p = oracle.pack_int4(q4, False)
    y, _ = oracle.linear_int4_rows(x, p, s)
    ref = bf16_bits_to_f64(x) @ bf16_bits_to_f64(oracle.dequant_int4_rows(p, s, k)).T
    assert np.allclose(y, ref, rtol=0, atol=1e-12)


def test_mxfp4_experts_shared_brute_force():
    rng = np.random.default_rng(12)
    r, e, n, k, s = 3, 5, 7, 64, 2
    x = _rand_bf16(rng, (r, k))
    blocks = rng.integers(0, 256, (e, n, k // 32, 16)).astype(np.uint8)
    scales = rng.integers(118, 125, (e, n, k // 32)).astype(np.uint8)
    experts = np.array([[0, 4], [2, 2], [1, 9]], np.int32)    # 9 is out of range
    y, a, bad = oracle.mxfp4_experts_shared(x, blocks, scales, experts, n)
    assert bad == 1 and (y[2, 1] == 0).all()
    wdq = bf16_bits_to_f64(oracle.dequant_mxfp4(blocks, scales, e, n, k))
    xf = bf16_bits_to_f64(x)
    for rr in range(r):
        for ss in range(s):
            ex = experts[rr, ss]
            if ex < e:
                assert np.allclose(y[rr, ss], wdq[ex] @ xf[rr], rtol=0, atol=1e-12)


def test_mxfp4_combine_experts_reduces_to_single_slots():
    """mxfp4_combine_experts (a reading: the weighted sum of the row's slot outputs) against
    what it must reduce to: one-hot weights pick exactly one slot of mxfp4_experts_shared;
    a row routed S times to one expert with weights summing to one gives that expert's
    product (checked against the separately written dequantizer and a plain matmul); an
    out-of-range slot adds nothing whatever its weight."""
    rng = np.random.default_rng(21)
    r, e, n, k, s = 3, 6, 9, 96, 4
    x = _rand_bf16(rng, (r, k))
    blocks = rng.integers(0, 256, (e, n, k // 32, 16)).astype(np.uint8)
    scales = rng.integers(118, 125, (e, n, k // 32)).astype(np.uint8)
    experts = np.array([[0, 3, 5, 1], [2, 2, 2, 2], [4, 7, 1, 0]], np.int32)  # 7: out of range
    ys, _, _ = oracle.mxfp4_experts_shared(x, blocks, scales, experts, n)
    wdq = bf16_bits_to_f64(oracle.dequant_mxfp4(blocks, scales, e, n, k))
    xf = bf16_bits_to_f64(x)
    # one-hot weights: slot j of each row (rows of different j: a transposed index fails)
    pick = np.array([2, 0, 3])
    onehot = np.zeros((r, s), np.float32)
    onehot[np.arange(r), pick] = 1.0
    y1, a1, bad = oracle.mxfp4_combine_experts(x, blocks, scales, experts, onehot, n)
    assert bad == 1
    for rr in range(r):
        assert np.array_equal(y1[rr], ys[rr, pick[rr]])
    # softmax weights (sum 1) on a row routed four times to expert 2
    logits = rng.standard_normal((r, s))
    wsm = (np.exp(logits) / np.exp(logits).sum(axis=1, keepdims=True)).astype(np.float32)
    y2, a2, _ = oracle.mxfp4_combine_experts(x, blocks, scales, experts, wsm, n)
    ref = wdq[2] @ xf[1] * float(wsm[1].astype(np.float64).sum())
    assert np.allclose(y2[1], ref, rtol=1e-12, atol=1e-12)
    assert (a2[1] > 0).all() and (a2[1] >= np.abs(y2[1]) - 1e-12).all()
    # the out-of-range slot (row 2, slot 1) carries weight but adds nothing
    w3 = np.zeros((r, s), np.float32)
    w3[2, 1] = 5.0
    y3, a3, _ = oracle.mxfp4_combine_experts(x, blocks, scales, experts, w3, n)
    assert (y3 == 0).all() and (a3 == 0).all()


def test_ordered_linear_gathers_inputs_like_scattered_weights():
    """Int4GroupLinear with an activation order (next row f3): gathering the inputs by
    `order` must equal scattering the dequantized stored columns back to input positions
    (stored column j belongs to input order[j]) and multiplying in plain f64, the other
    way round; identity order gives the plain layer bit for bit; repeated indices add
    their columns; out-of-range entries are refused."""
    rng = np.random.default_rng(22)
    m, n, k, g = 3, 10, 256, 64
    x = _rand_bf16(rng, (m, k))
    codes = rng.integers(0, 16, (n, k)).astype(np.uint8)
    _, packed = oracle.pack_int4(codes, True)
    scale = (rng.random((n, k // g)) * 0.02 + 0.002).astype(np.float32)
    zero = rng.integers(0, 16, (n, k // g)).astype(np.uint8)
    bias = _rand_bf16(rng, (n,))
    wst = bf16_bits_to_f64(oracle.dequant_int4_groups(packed, scale, zero, n, k, g))
    xf = bf16_bits_to_f64(x)
    bf = bf16_bits_to_f64(bias)
    y0, a0 = oracle.linear_int4_groups(x, packed, scale, zero, bias, n, g)
    y1, a1 = oracle.linear_int4_groups_ordered(x, np.arange(k), packed, scale, zero, bias, n, g)
    assert np.array_equal(y0, y1) and np.array_equal(a0, a1)
    for order in (rng.permutation(k), rng.integers(0, k, k)):  # a permutation, then repeats
        y, _ = oracle.linear_int4_groups_ordered(x, order, packed, scale, zero, bias, n, g)
        wnat = np.zeros((n, k))
        np.add.at(wnat.T, order, wst.T)  # stored column j added to input position order[j]
        assert np.allclose(y, xf @ wnat.T + bf, rtol=1e-12, atol=1e-12)
    for bad in (np.full(k, k), np.full(k, -1)):
        with pytest.raises(ValueError):
            oracle.linear_int4_groups_ordered(x, bad, packed, scale, zero, bias, n, g)


def test_mxfp4_experts_per_slot_inputs():
    """mxfp4_experts (next row f2, each slot its own input) reduces to
    mxfp4_experts_shared when every slot of a row gets the row's input, and otherwise
    to a plain matmul of each slot's input with its expert's dequantized weights."""
    rng = np.random.default_rng(23)
    r, e, n, k, s = 2, 5, 6, 64, 3
    blocks = rng.integers(0, 256, (e, n, k // 32, 16)).astype(np.uint8)
    scales = rng.integers(118, 125, (e, n, k // 32)).astype(np.uint8)
    experts = np.array([[4, 0, 2], [1, 1, 3]], np.int32)
    xr = _rand_bf16(rng, (r, k))
    ys, _, _ = oracle.mxfp4_experts_shared(xr, blocks, scales, experts, n)
    yp, _, _ = oracle.mxfp4_experts(np.repeat(xr[:, None, :], s, axis=1), blocks, scales, experts, n)
    assert np.array_equal(ys, yp)
    xs = _rand_bf16(rng, (r, s, k))
    y, _, bad = oracle.mxfp4_experts(xs, blocks, scales, experts, n)
    assert bad == 0
    wdq = bf16_bits_to_f64(oracle.dequant_mxfp4(blocks, scales, e, n, k))
    xf = bf16_bits_to_f64(xs)
    for rr in range(r):
        for ss in range(s):
            assert np.allclose(y[rr, ss], wdq[experts[rr, ss]] @ xf[rr, ss], rtol=0, atol=1e-12)


def test_quantization_error_budget():
    """Sanity (not parity): the quantized layer's output stays within the error budget
    of the quantization step (Delta = s/2 plus the bf16 rounding of W-hat) plus f64
    rounding, and that budget is not rounding-only."""
    rng = np.random.default_rng(13)
    m, n, k, gsz = 4, 32, 512, 32
    w = (rng.standard_normal((n, k)) * 0.02).astype(np.float32)
    x = _rand_bf16(rng, (m, k))
    codes, scale, zero, _ = oracle.quantize_asym(w, gsz, 4)
    _, packed = oracle.pack_int4(codes, True)
    yq, _ = oracle.linear_int4_groups(x, packed, scale, zero, None, n, gsz)
    xf = bf16_bits_to_f64(x)
    y = xf @ w.astype(np.float64).T
    wdq = bf16_bits_to_f64(oracle.dequant_int4_groups(packed, scale, zero, n, k, gsz))
    delta = np.repeat(scale.astype(np.float64), gsz, 1) / 2 * (1 + 2.0 ** -18) + np.abs(wdq) * 2.0 ** -8
    bound = np.abs(xf) @ delta.T + 1e-12
    err = np.abs(yq - y)
    assert (err <= bound).all()
    assert err.max() > 1e3 * 2.0 ** -24 * (np.abs(xf) @ np.abs(w.astype(np.float64)).T).max() * 1e-3
