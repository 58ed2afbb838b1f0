"""GPU linear layers against the CPU oracle, element by element, within the stated
tolerance |y_gpu - y_ref| <= 2e-3 * sum_k |x_k * w_k| + 1 bf16 ulp(y_ref)."""
import numpy as np
import pytest
import torch

import oracle
import weight_only_quantized_linear_gb300 as wq
from weight_only_quantized_linear_gb300 import synth
from gpu_util import assert_within, bf16_bits, guarded, guards_intact

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    wq.build()
    oracle.set_threads(oracle.max_threads())


def dev(a, d):
    return torch.from_numpy(np.ascontiguousarray(a)).to(d) if isinstance(a, np.ndarray) else a.to(d)


def make_i4g(n, k, g, seed):
    rng = np.random.default_rng(seed)
    packed = rng.integers(0, 256, (n, k // 2)).astype(np.uint8)
    scale = (rng.random((n, k // g)) * 0.018 + 0.002).astype(np.float32)
    zero = rng.integers(6, 10, (n, k // g)).astype(np.uint8)
    return packed, scale, zero


def run_i4g(d, x, packed, scale, zero, bias, g, use_ws=True):
    M, K = x.shape
    N = packed.shape[0]
    ws = wq.alloc_workspace(wq.wq_linear_int4_groups_workspace(M, N, K, g), d) if use_ws else None
    buf, y = guarded((M, N), torch.bfloat16, d)
    st = torch.zeros(1, dtype=torch.int32, device=d)
    wq.wq_linear_int4_groups(x, packed, scale, zero, bias, g, y=y, workspace=ws, dev_status=st)
    torch.cuda.synchronize()
    assert guards_intact(buf), "write outside y"
    assert int(st.item()) == 0
    if ws is not None:
        assert int(ws.view(torch.int32)[:64].abs().sum().item()) == 0, "split-K counters not reset"
    return y


def test_tiny_config(cuda_device):
    """x [1, 256]; packed [256, 8, 16]; scale U[0.002, 0.02]; zero U{6..9}; G = 32."""
    t = synth.tiny_int4_groups(seed=0)
    x, packed, scale, zero = t["x"], t["packed"], t["scale"], t["zero"]
    y = run_i4g(cuda_device, dev(x, cuda_device), dev(packed, cuda_device), dev(scale, cuda_device),
                dev(zero, cuda_device), None, 32)
    yr, ad = oracle.linear_int4_groups(bf16_bits(x), packed.numpy().reshape(256, 128), scale.numpy(),
                                       zero.numpy(), None, 256, 32)
    assert_within(y, yr, ad, "tiny")
    # the same weights quantized from W on both sides: codes bit-exact, then linear
    w = t["w"]
    c, s, z = wq.wq_quantize_groups(w.to(cuda_device), 32, 4, wq.WQ_ASYM)
    oc, os_, oz, _ = oracle.quantize_asym(w.numpy(), 32, 4)
    assert (c.cpu().numpy() == oc).all() and (z.cpu().numpy() == oz).all()
    p = wq.wq_pack_int4(c, True)
    assert (p.cpu().numpy() == oracle.pack_int4(oc, True)[1]).all()


CASES = [
    # M, N, K, G, bias
    (1, 256, 256, 32, False),
    (1, 1000, 4096 + 128, 128, True),     # ragged N, K tail inside a stage
    (1, 37, 3072, 64, False),
    (2, 300, 1024, 256, True),
    (5, 129, 2048, 128, False),
    (8, 512, 4096, 128, True),
    (9, 64, 1024, 32, False),
    (16, 1024, 4096, 128, True),
    (17, 100, 512, 128, False),           # multiple activation batches
    (1, 1000, 2048, 128, True),           # factored kernel: ragged N, TMA boxes past N
    (3, 48, 4096, 256, False),
    (24, 200, 4096, 128, True),           # factored kernel, two batches of 16
    (40, 48, 1024, 64, True),             # tensor-core regime from here on
    (32, 256, 256, 32, False),
    (256, 512, 4096, 128, True),
    (300, 300, 1056, 32, True),           # K % 64 == 32, ragged M and N
    (513, 1000, 2048, 256, False),
]


@pytest.mark.parametrize("M,N,K,G,bias", CASES)
@pytest.mark.parametrize("use_ws", [True, False])
def test_int4_groups_shapes(cuda_device, M, N, K, G, bias, use_ws):
    d = cuda_device
    packed, scale, zero = make_i4g(N, K, G, seed=M * 1000 + N)
    x = synth.normal_bf16((M, K), seed=M + N)
    b = synth.normal_bf16((N,), seed=7) if bias else None
    y = run_i4g(d, dev(x, d), dev(packed, d), dev(scale, d), dev(zero, d), None if b is None else dev(b, d),
                G, use_ws)
    yr, ad = oracle.linear_int4_groups(bf16_bits(x), packed, scale, zero, None if b is None else bf16_bits(b),
                                       N, G)
    assert_within(y, yr, ad, f"M={M} N={N} K={K} G={G}")


@pytest.mark.parametrize("M,G", [(1, 128), (5, 128), (1, 256), (13, 64), (2, 32)])
def test_int4_groups_zero_points_over_full_byte_range(cuda_device, M, G):
    """The layout stores zero points as u8: codes minus any zero point 0..255 (above 127
    the factored kernel takes its two-subtraction path) match the oracle."""
    d = cuda_device
    N, K = 200, 2048
    rng = np.random.default_rng(M * 7 + G)
    packed = rng.integers(0, 256, (N, K // 2)).astype(np.uint8)
    scale = (rng.random((N, K // G)) * 0.018 + 0.002).astype(np.float32)
    zero = rng.integers(0, 256, (N, K // G)).astype(np.uint8)
    zero[:8] = 255           # whole tiles of large zero points, and mixed warps elsewhere
    x = synth.normal_bf16((M, K), seed=M + 11)
    y = run_i4g(d, dev(x, d), dev(packed, d), dev(scale, d), dev(zero, d), None, G)
    yr, ad = oracle.linear_int4_groups(bf16_bits(x), packed, scale, zero, None, N, G)
    assert_within(y, yr, ad, f"full-range zero points M={M} G={G}")


def test_int4_groups_deterministic_and_split_invariant(cuda_device):
    d = cuda_device
    M, N, K, G = 1, 1024, 4096, 128
    packed, scale, zero = make_i4g(N, K, G, seed=3)
    x = dev(synth.normal_bf16((M, K), seed=4), d)
    args = (dev(packed, d), dev(scale, d), dev(zero, d))
    y1 = run_i4g(d, x, *args, None, G)
    y2 = run_i4g(d, x, *args, None, G)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


@pytest.mark.parametrize("name", synth.LLAMA_ORDER)
def test_llama_decode_full_size_sampled(cuda_device, name):
    """Full Llama-3.1-8B projection sizes at M = 1, G = 128, in the launch the benchmark
    times (workspace on); weights quantized by the oracle; 384 sampled rows checked."""
    d = cuda_device
    N, K = synth.LLAMA_PROJ[name]
    w = synth.weight_f32(N, K, seed=11, outlier_frac=0.001)
    codes, scale, zero, _ = oracle.quantize_asym(w.numpy(), 128, 4)
    _, packed = oracle.pack_int4(codes, True)
    x = synth.normal_bf16((1, K), seed=12)
    y = run_i4g(d, dev(x, d), dev(packed, d), dev(scale, d), dev(zero, d), None, 128)
    rows = np.unique(np.concatenate([np.arange(16), np.arange(N - 16, N),
                                     np.random.default_rng(13).choice(N, 352, replace=False)]))
    yr, ad = oracle.linear_int4_groups(bf16_bits(x), packed[rows], scale[rows], zero[rows], None, len(rows), 128)
    assert_within(y[:, torch.from_numpy(rows).to(d)], yr, ad, name)


@pytest.mark.parametrize("M", [1, 4, 16, 64, 128])
def test_m_sweep_gate_sampled(cuda_device, M):
    d = cuda_device
    N, K = synth.LLAMA_PROJ["gate"]
    w = synth.weight_f32(N, K, seed=21, outlier_frac=0.001)
    c, s, z = wq.wq_quantize_groups(w.to(d), 128, 4, wq.WQ_ASYM)
    p = wq.wq_pack_int4(c, True)
    x = synth.normal_bf16((M, K), seed=22)
    y = run_i4g(d, dev(x, d), p, s, z, None, 128)
    rows = np.random.default_rng(M).choice(N, 96, replace=False)
    rows.sort()
    ms = np.random.default_rng(M + 1).choice(M, min(M, 8), replace=False)
    ms.sort()
    # inputs for the oracle come from the oracle's own quantizer (bit-identical, checked)
    oc, os_, oz, _ = oracle.quantize_asym(w.numpy()[rows], 128, 4)
    assert (c.cpu().numpy()[rows] == oc).all()
    _, op = oracle.pack_int4(oc, True)
    yr, ad = oracle.linear_int4_groups(bf16_bits(x)[ms], op, os_, oz, None, len(rows), 128)
    ysel = y[torch.from_numpy(ms).to(d)][:, torch.from_numpy(rows).to(d)]
    assert_within(ysel, yr, ad, f"M={M}")


# ------------------------------------------------------------------ per-row formats
ROW_CASES = [(1, 256, 4096), (3, 100, 512), (8, 1000, 4096 + 64), (16, 64, 1024), (20, 40, 256)]


@pytest.mark.parametrize("M,N,K", ROW_CASES)
def test_int8_rows(cuda_device, M, N, K):
    d = cuda_device
    w = synth.weight_f32(N, K, seed=N)
    q, s, _ = oracle.quantize_sym(w.numpy(), K, 8)
    x = synth.normal_bf16((M, K), seed=M)
    b = synth.normal_bf16((N,), seed=5)
    ws = wq.alloc_workspace(wq.wq_linear_rows_workspace(M, N, K, 8), d)
    buf, y = guarded((M, N), torch.bfloat16, d)
    wq.wq_linear_int8_rows(dev(x, d), dev(q, d), dev(s[:, 0].copy(), d), dev(b, d), y=y, workspace=ws)
    torch.cuda.synchronize()
    assert guards_intact(buf)
    yr, ad = oracle.linear_int8_rows(bf16_bits(x), q, s[:, 0].copy(), bf16_bits(b))
    assert_within(y, yr, ad, f"int8 M={M} N={N} K={K}")


@pytest.mark.parametrize("M,N,K", ROW_CASES)
def test_int4_rows(cuda_device, M, N, K):
    d = cuda_device
    w = synth.weight_f32(N, K, seed=N + 1)
    q, s, _ = oracle.quantize_sym(w.numpy(), K, 4)
    _, p = oracle.pack_int4(q, False)
    x = synth.normal_bf16((M, K), seed=M + 1)
    ws = wq.alloc_workspace(wq.wq_linear_rows_workspace(M, N, K, 4), d)
    buf, y = guarded((M, N), torch.bfloat16, d)
    wq.wq_linear_int4_rows(dev(x, d), dev(p.view(np.int8), d), dev(s[:, 0].copy(), d), None, y=y, workspace=ws)
    torch.cuda.synchronize()
    assert guards_intact(buf)
    yr, ad = oracle.linear_int4_rows(bf16_bits(x), p, s[:, 0].copy())
    assert_within(y, yr, ad, f"int4 rows M={M} N={N} K={K}")


@pytest.mark.parametrize("N,K", [(14336, 4096), (4096, 14336)])
@pytest.mark.parametrize("M", [1, 8, 16])
def test_rows_full_size_sampled(cuda_device, N, K, M):
    d = cuda_device
    w = synth.weight_f32(N, K, seed=31)
    x = synth.normal_bf16((M, K), seed=32)
    rows = np.random.default_rng(N + M).choice(N, 128, replace=False)
    rows.sort()
    ridx = torch.from_numpy(rows).to(d)
    q8, s8, _ = oracle.quantize_sym(w.numpy(), K, 8)
    ws = wq.alloc_workspace(wq.wq_linear_rows_workspace(M, N, K, 8), d)
    y = wq.wq_linear_int8_rows(dev(x, d), dev(q8, d), dev(s8[:, 0].copy(), d), workspace=ws)
    yr, ad = oracle.linear_int8_rows(bf16_bits(x), q8[rows], s8[rows, 0].copy())
    assert_within(y[:, ridx], yr, ad, "int8 rows full size")
    q4, s4, _ = oracle.quantize_sym(w.numpy(), K, 4)
    _, p4 = oracle.pack_int4(q4, False)
    ws = wq.alloc_workspace(wq.wq_linear_rows_workspace(M, N, K, 4), d)
    y = wq.wq_linear_int4_rows(dev(x, d), dev(p4.view(np.int8), d), dev(s4[:, 0].copy(), d), workspace=ws)
    yr, ad = oracle.linear_int4_rows(bf16_bits(x), p4[rows], s4[rows, 0].copy())
    assert_within(y[:, ridx], yr, ad, "int4 rows full size")


# ------------------------------------------------------------------ MXFP4 experts
@pytest.mark.parametrize("R", [1, 8, 64])
@pytest.mark.parametrize("N", [5760, 2880])
def test_mxfp4_experts_shared_gptoss_sampled(cuda_device, R, N):
    d = cuda_device
    E, K, S = 32, 2880, 4
    blocks, scales = synth.mxfp4_experts(E, N, K, seed=41)
    experts, _ = synth.routing_topk(R, E, S, seed=42)
    x = synth.normal_bf16((R, 1, K), seed=43)
    st = torch.zeros(1, dtype=torch.int32, device=d)
    buf, y = guarded((R, S, N), torch.bfloat16, d)
    wq.wq_mxfp4_experts_shared(dev(x, d), dev(blocks, d), dev(scales, d), dev(experts, d), y=y, dev_status=st)
    torch.cuda.synchronize()
    assert guards_intact(buf) and int(st.item()) == 0
    n0 = int(np.random.default_rng(R).integers(0, N - 64))
    for a, b in ((0, 32), (n0, n0 + 64), (N - 32, N)):
        yr, ad, bad = oracle.mxfp4_experts_shared(bf16_bits(x).reshape(R, K), blocks.numpy(), scales.numpy(),
                                                  experts.numpy(), N, a, b)
        assert bad == 0
        assert_within(y[:, :, a:b], yr[:, :, a:b], ad[:, :, a:b], f"mxfp4 R={R} N={N} [{a},{b})")


def test_mxfp4_many_rows_per_expert_and_bad_index(cuda_device):
    d = cuda_device
    E, N, K, R, S = 3, 200, 320, 30, 2
    blocks, scales = synth.mxfp4_experts(E, N, K, seed=51)
    rng = np.random.default_rng(52)
    experts = rng.integers(0, E, (R, S)).astype(np.int32)
    experts[3, 1] = E          # out of range
    experts[7, 0] = -1
    x = synth.normal_bf16((R, 1, K), seed=53)
    st = torch.zeros(1, dtype=torch.int32, device=d)
    y = wq.wq_mxfp4_experts_shared(dev(x, d), dev(blocks, d), dev(scales, d), dev(experts, d), dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & wq.WQ_DEV_BAD_EXPERT
    yr, ad, bad = oracle.mxfp4_experts_shared(bf16_bits(x).reshape(R, K), blocks.numpy(), scales.numpy(),
                                              experts, N)
    assert bad == 2
    assert (y[3, 1].float() == 0).all() and (y[7, 0].float() == 0).all()
    assert_within(y, yr, ad, "mxfp4 many rows")


@pytest.mark.parametrize("grid", [1, 3, 7, 64, 151])
@pytest.mark.parametrize("M", [1, 13])
def test_stream_k_partitions(cuda_device, tune, grid, M):
    """Every block (exact kernel) or cluster (factored kernel) count gives the same
    answer: tiles cut anywhere by the equal-share ranges are finished from their partials
    (deterministically)."""
    d = cuda_device
    tune(wq.WQ_TUNE_GEMV_BLOCKS, grid)
    tune(wq.WQ_TUNE_GEMV_CLUSTERS, grid)
    N, K, G = 1000, 4096 + 1024, 128
    packed, scale, zero = make_i4g(N, K, G, seed=grid)
    x = synth.normal_bf16((M, K), seed=grid + 1)
    b = synth.normal_bf16((N,), seed=3)
    y = run_i4g(d, dev(x, d), dev(packed, d), dev(scale, d), dev(zero, d), dev(b, d), G)
    yr, ad = oracle.linear_int4_groups(bf16_bits(x), packed, scale, zero, bf16_bits(b), N, G)
    assert_within(y, yr, ad, f"grid={grid} M={M}")
    y2 = run_i4g(d, dev(x, d), dev(packed, d), dev(scale, d), dev(zero, d), dev(b, d), G)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


def test_gemm_matches_gemv_path(cuda_device, tune):
    """The tensor-core regime and the decode regime agree (both within the oracle's
    tolerance); the crossover moves with the WQ_TUNE_GEMM_MIN_M knob."""
    d = cuda_device
    M, N, K, G = 48, 512, 2048, 128
    packed, scale, zero = make_i4g(N, K, G, seed=77)
    x = dev(synth.normal_bf16((M, K), seed=78), d)
    args = (dev(packed, d), dev(scale, d), dev(zero, d))
    y_tc = run_i4g(d, x, *args, None, G)
    tune(wq.WQ_TUNE_GEMM_MIN_M, 100000)
    y_gemv = run_i4g(d, x, *args, None, G)
    yr, ad = oracle.linear_int4_groups(bf16_bits(x.cpu()), packed, scale, zero, None, N, G)
    assert_within(y_tc, yr, ad, "tcgen05")
    assert_within(y_gemv, yr, ad, "gemv")


@pytest.mark.parametrize("M,N,K,G", [(256, 256, 4096, 128), (300, 1000, 3072, 64), (64, 520, 2048, 32)])
def test_gemm_split_k(cuda_device, M, N, K, G):
    """Tensor-core shapes with fewer tiles than SMs split K across blocks through the
    workspace; the split result matches the oracle and the unsplit launch, and the
    workspace is left zero-filled."""
    d = cuda_device
    packed, scale, zero = make_i4g(N, K, G, seed=M + N)
    x = synth.normal_bf16((M, K), seed=M)
    b = synth.normal_bf16((N,), seed=N)
    nbytes = wq.wq_linear_int4_groups_workspace(M, N, K, G)
    assert nbytes > 0, "expected a split-K workspace for a shape with few tiles"
    args = (dev(x, d), dev(packed, d), dev(scale, d), dev(zero, d), dev(b, d), G)
    y_split = run_i4g(d, *args, use_ws=True)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=d)
    y2 = torch.empty((M, N), dtype=torch.bfloat16, device=d)
    wq.wq_linear_int4_groups(*args[:4], args[4], G, y=y2, workspace=ws)
    torch.cuda.synchronize()
    assert int(ws.view(torch.int32).abs().sum().item()) == 0, "partials not cleared"
    y_whole = run_i4g(d, *args, use_ws=False)
    yr, ad = oracle.linear_int4_groups(bf16_bits(x), packed, scale, zero, bf16_bits(b), N, G)
    assert_within(y_split, yr, ad, f"split M={M} N={N} K={K}")
    assert_within(y_whole, yr, ad, f"unsplit M={M} N={N} K={K}")
    assert torch.equal(y_split.view(torch.int16), y2.view(torch.int16))


@pytest.mark.parametrize("M,N,K", [(1, 4096, 4096), (5, 1000, 2048)])
def test_static_weights_same_result(cuda_device, M, N, K):
    """Streaming the weights before the previous kernel completes changes no bit of the
    result: back-to-back calls on one stream, each right after a kernel that rewrites the
    activations (which are read only after that kernel has completed)."""
    d = cuda_device
    G = 128
    packed, scale, zero = make_i4g(N, K, G, seed=31)
    x0 = dev(synth.normal_bf16((M, K), seed=32), d)
    args = (dev(packed, d), dev(scale, d), dev(zero, d))
    ws = wq.alloc_workspace(wq.wq_linear_int4_groups_workspace(M, N, K, G), d)
    outs = []
    for on in (False, True):
        wq.wq_set_static_weights(on)
        try:
            x = x0.clone()
            ys = []
            for i in range(4):
                x.copy_(x0 * float(i + 1))  # a kernel that writes the activations just before the call
                y = torch.empty((M, N), dtype=torch.bfloat16, device=d)
                wq.wq_linear_int4_groups(x, *args, None, G, y=y, workspace=ws)
                ys.append(y)
            torch.cuda.synchronize()
            outs.append(torch.stack(ys))
        finally:
            wq.wq_set_static_weights(False)
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    x3 = (x0 * 4.0).cpu()
    yr, ad = oracle.linear_int4_groups(bf16_bits(x3), packed, scale, zero, None, N, G)
    assert_within(outs[1][3], yr, ad, "static weights, last call")


@pytest.mark.parametrize("xsmem", ["1", "0"])
@pytest.mark.parametrize("M,N,K", [(1, 4096, 14336), (3, 1000, 4096), (8, 300, 2048)])
def test_factored_activation_paths(cuda_device, tune, xsmem, M, N, K):
    """Activations staged in shared memory (the default where two blocks an SM still fit,
    with a three-stage ring at K = 14336) and read from global memory give results
    within the tolerance."""
    tune(wq.WQ_TUNE_GEMV_XSMEM, 0 if xsmem == "1" else 1)
    d = cuda_device
    G = 128
    packed, scale, zero = make_i4g(N, K, G, seed=K + M)
    x = synth.normal_bf16((M, K), seed=M + 40)
    y = run_i4g(d, dev(x, d), dev(packed, d), dev(scale, d), dev(zero, d), None, G)
    yr, ad = oracle.linear_int4_groups(bf16_bits(x), packed, scale, zero, None, N, G)
    assert_within(y, yr, ad, f"xsmem={xsmem} M={M} N={N} K={K}")


@pytest.mark.parametrize("fmt", ["groups", "rows"])
@pytest.mark.parametrize("M", [1, 3, 8])
def test_decode_offset_activations_full_range_zero_points(cuda_device, M, fmt):
    """Activations with a large common offset (mean 6, so that the sums of x_k * (q_k - z)
    are small differences of large terms) and zero points over the whole byte range
    (signed per-row codes: the fixed offset 8) match the oracle, column by column (M = 3
    leaves MMA columns past M)."""
    d = cuda_device
    N, K = 600, 4096
    x = (synth.normal_bf16((M, K), seed=M + 71).float() + 6.0).to(torch.bfloat16)
    if fmt == "groups":
        G = 128
        rng = np.random.default_rng(M + 70)
        packed = rng.integers(0, 256, (N, K // 2)).astype(np.uint8)
        scale = (rng.random((N, K // G)) * 0.018 + 0.002).astype(np.float32)
        zero = rng.integers(0, 256, (N, K // G)).astype(np.uint8)
        y = run_i4g(d, dev(x, d), dev(packed, d), dev(scale, d), dev(zero, d), None, G)
        yr, ad = oracle.linear_int4_groups(bf16_bits(x), packed, scale, zero, None, N, G)
    else:
        w = synth.weight_f32(N, K, seed=N + 72)
        q, s, _ = oracle.quantize_sym(w.numpy(), K, 4)
        _, p = oracle.pack_int4(q, False)
        ws = wq.alloc_workspace(wq.wq_linear_rows_workspace(M, N, K, 4), d)
        buf, y = guarded((M, N), torch.bfloat16, d)
        wq.wq_linear_int4_rows(dev(x, d), dev(p.view(np.int8), d), dev(s[:, 0].copy(), d), None, y=y, workspace=ws)
        torch.cuda.synchronize()
        assert guards_intact(buf)
        yr, ad = oracle.linear_int4_rows(bf16_bits(x), p, s[:, 0].copy())
    assert_within(y, yr, ad, f"offset activations {fmt} M={M}")


@pytest.mark.parametrize("mode", ["push", "barrier", "default"])
@pytest.mark.parametrize("M,N,K,clusters", [(1, 14336, 4096, None), (1, 4096, 14336, None), (1, 1024, 4096, None),
                                            (1, 4096, 4096, None), (4, 1000, 6144, 5), (12, 700, 4096, None),
                                            (1, 256, 2048, 3), (1, 1000, 8192, 7), (2, 600, 16384, None),
                                            (3, 4100, 8192, 200)])
def test_factored_cut_tile_fixup(cuda_device, tune, mode, M, N, K, clusters):
    """Tiles cut between warps are finished either by pushes into the closing warp's
    shared memory (no cluster-wide barrier) or by the closing warp reading the parked
    partials after cluster barriers (forced each way, and the launch's own choice), with
    clusters of two CTAs and, for rows of 32 or more steps (K >= 8192), of four; all match
    the oracle and are deterministic."""
    if mode == "push":
        tune(wq.WQ_TUNE_GEMV_PUSH, 1)
    elif mode == "barrier":
        tune(wq.WQ_TUNE_GEMV_PUSH, 2)
    if clusters is not None:
        tune(wq.WQ_TUNE_GEMV_CLUSTERS, clusters)
    d = cuda_device
    G = 128
    packed, scale, zero = make_i4g(N, K, G, seed=N + M)
    x = synth.normal_bf16((M, K), seed=M + 50)
    b = synth.normal_bf16((N,), seed=51)
    args = (dev(x, d), dev(packed, d), dev(scale, d), dev(zero, d), dev(b, d), G)
    y = run_i4g(d, *args)
    rows = np.unique(np.concatenate([np.arange(min(N, 64)), np.arange(max(0, N - 64), N),
                                     np.random.default_rng(5).choice(N, min(N, 256), replace=False)]))
    yr, ad = oracle.linear_int4_groups(bf16_bits(x), packed[rows], scale[rows], zero[rows], bf16_bits(b)[rows],
                                       len(rows), G)
    assert_within(y[:, torch.from_numpy(rows).to(d)], yr, ad, f"{mode} M={M} N={N} K={K}")
    y2 = run_i4g(d, *args)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


def test_one_workspace_shared_by_shapes_in_turn(cuda_device):
    """Calls of different shapes and kernels that share one workspace in turn (never
    concurrently) all stay correct: every call leaves the whole workspace zero-filled."""
    d = cuda_device
    shapes = [(2, 300, 2048, 64), (1, 4096, 4096, 128), (5, 1000, 6144, 128), (1, 300, 2048, 64),
              (13, 4096, 4096, 128), (1, 1000, 4096 + 1024, 128), (64, 256, 4096, 128)]
    need = max(wq.wq_linear_int4_groups_workspace(M, N, K, G) for M, N, K, G in shapes)
    ws = torch.zeros(need, dtype=torch.uint8, device=d)
    for i, (M, N, K, G) in enumerate(shapes):
        packed, scale, zero = make_i4g(N, K, G, seed=i)
        x = synth.normal_bf16((M, K), seed=i + 50)
        y = wq.wq_linear_int4_groups(dev(x, d), dev(packed, d), dev(scale, d), dev(zero, d), None, G, workspace=ws)
        torch.cuda.synchronize()
        assert int(ws.view(torch.int32).abs().sum().item()) == 0, f"workspace dirty after {M, N, K, G}"
        rows = np.random.default_rng(i).choice(N, min(N, 128), replace=False)
        yr, ad = oracle.linear_int4_groups(bf16_bits(x), packed[rows], scale[rows], zero[rows], None, len(rows), G)
        assert_within(y[:, torch.from_numpy(rows).to(d)], yr, ad, f"shared workspace {M, N, K, G}")
