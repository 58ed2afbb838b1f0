"""The grouped tcgen05 GEMM for MXFP4 experts with many routed slots (k_gemm_mx_tc) against
the CPU oracle ("Quantization" (Linnet docs), format table: mxfp4_experts_shared,
mxfp4_linear_experts_shared "many rows (x: [R, In])", mxfp4_combine_experts).

Cases: a slot count past the decode kernels' routing tables (4096), the gpt-oss gate/up
shape at 2048 slots (sampled column ranges: the first and the last 256-wide tiles), a
ragged N (not a multiple of 8) with K % 64 == 32, scales above 128 (two multiplies),
every slot on one expert (many tiles of one segment; last tiles of 128 and 129 rows,
one and two 128-row halves) and a skewed routing (one-row segments), out-of-range expert
indices, the per-slot and combine forms, the crossover knob, and the workspace rules.  Tolerance: |y_gpu - y_ref| <= 2e-3 * sum_k |x_k w_k| + 1 bf16 ulp(y_ref)."""
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


def _experts(E, N, K, seed, elo=118, ehi=124):
    rng = np.random.default_rng(seed)
    blocks = torch.from_numpy(rng.integers(0, 256, (E, N, K // 32, 16), dtype=np.uint8))
    scales = torch.from_numpy(rng.integers(elo, ehi + 1, (E, N, K // 32), dtype=np.uint8))
    return blocks, scales


def _route(R, S, E, seed, kind="topk"):
    rng = np.random.default_rng(seed)
    if kind == "topk":
        e = np.stack([rng.choice(E, S, replace=False) for _ in range(R)])
    elif kind == "one":  # every slot on expert E - 1
        e = np.full((R, S), E - 1)
    else:  # skewed: most slots on expert 0, a few on each of the others
        e = np.zeros((R, S), dtype=np.int64)
        flat = e.reshape(-1)
        idx = rng.choice(flat.size, size=min(flat.size, 3 * E), replace=False)
        flat[idx] = rng.integers(1, E, idx.size)
    return torch.from_numpy(e.astype(np.int32))


def _run_shared(d, x, blocks, scales, experts, N, workspace=None):
    R, S = experts.shape
    st = torch.zeros(1, dtype=torch.int32, device=d)
    buf, y = guarded((R, S, N), torch.bfloat16, d)
    wq.wq_mxfp4_linear_experts_shared(x.to(d), blocks.to(d), scales.to(d), experts.to(d), y=y,
                                      workspace=workspace, dev_status=st)
    torch.cuda.synchronize()
    assert guards_intact(buf), "write outside y"
    return y, int(st.item())


def _check_cols(y, x, blocks, scales, experts, N, n0, n1, what):
    R = x.shape[0]
    yr, ad, bad = oracle.mxfp4_experts_shared(bf16_bits(x).reshape(R, -1), blocks.numpy(), scales.numpy(),
                                              experts.numpy(), N, n0, n1)
    assert_within(y[..., n0:n1], yr[..., n0:n1], ad[..., n0:n1], what)
    return bad


@pytest.mark.parametrize("E,N,K,R,S,elo,ehi,kind,cols", [
    (8, 512, 1024, 256, 4, 118, 124, "topk", None),      # 1024 slots, 16 tiles of 256 rows
    (16, 256, 768, 1024, 4, 118, 124, "topk", None),     # 4096 slots: past the decode kernels' tables
    (5, 200, 992, 300, 3, 110, 130, "topk", None),       # N ragged (scalar stores), K % 64 == 32
    (4, 640, 1536, 160, 4, 100, 200, "topk", None),      # scales above 128: two multiplies
    (6, 384, 1024, 700, 1, 118, 124, "one", None),       # one segment of 700 rows (3 tiles)
    (6, 384, 1024, 640, 1, 118, 124, "one", None),       # last tile 128 rows: its first half only
    (6, 384, 1024, 641, 1, 118, 124, "one", None),       # last tile 129 rows: both halves
    (12, 320, 1024, 600, 2, 118, 124, "skew", None),     # one large segment, one-row segments
    (32, 5760, 2880, 512, 4, 118, 124, "topk", ((0, 256), (5504, 5760))),  # gpt-oss gate/up
    (32, 2880, 2880, 2048, 4, 118, 124, "topk", ((0, 256), (2816, 2880))),  # gpt-oss down, 8192 slots
    (32, 200, 992, 100, 6, 100, 200, "topk", None),      # 32 experts: ragged N, K % 64 == 32, scales > 128
])
def test_grouped_gemm_matches_oracle(cuda_device, E, N, K, R, S, elo, ehi, kind, cols):
    d = cuda_device
    blocks, scales = _experts(E, N, K, seed=E * 7 + N + K, elo=elo, ehi=ehi)
    experts = _route(R, S, E, seed=R + S, kind=kind)
    x = synth.normal_bf16((R, K), seed=K + R)
    y, st = _run_shared(d, x, blocks, scales, experts, N)
    assert st == 0
    assert "k_gemm_mx_tc" in wq.wq_last_launch(), wq.wq_last_launch()
    for n0, n1 in (cols or ((0, N),)):
        bad = _check_cols(y, x, blocks, scales, experts, N, n0, n1, f"E={E} N={N} K={K} R={R} S={S} {kind}")
        assert bad == 0
    # the order of a segment's rows depends on atomics; every row's result does not
    y2, _ = _run_shared(d, x, blocks, scales, experts, N)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16)), "not deterministic"


def test_grouped_gemm_bad_experts(cuda_device):
    d = cuda_device
    E, N, K, R, S = 8, 256, 1024, 200, 4
    blocks, scales = _experts(E, N, K, seed=31)
    experts = _route(R, S, E, seed=32)
    experts[3, 0] = -1
    experts[77, 2] = E
    experts[199, 3] = 1 << 20
    x = synth.normal_bf16((R, K), seed=33)
    y, st = _run_shared(d, x, blocks, scales, experts, N)
    assert "k_gemm_mx_tc" in wq.wq_last_launch()
    assert st & wq.WQ_DEV_BAD_EXPERT
    for r, s in ((3, 0), (77, 2), (199, 3)):
        assert (y[r, s].float() == 0).all()
    assert _check_cols(y, x, blocks, scales, experts, N, 0, N, "bad experts") == 3
    # no valid slot at all: only the zero-row tiles run
    y0, st0 = _run_shared(d, x, blocks, scales, torch.full((R, S), -2, dtype=torch.int32), N)
    assert "k_gemm_mx_tc" in wq.wq_last_launch()
    assert st0 & wq.WQ_DEV_BAD_EXPERT
    assert (y0.float() == 0).all()


def test_grouped_gemm_combine(cuda_device):
    d = cuda_device
    E, N, K, R, S = 16, 640, 1024, 300, 4
    blocks, scales = _experts(E, N, K, seed=41)
    experts = _route(R, S, E, seed=42)
    experts[5, 1] = -7
    x = synth.normal_bf16((R, K), seed=43)
    wts = torch.softmax(torch.from_numpy(np.random.default_rng(44).normal(size=(R, S))).float(), -1)
    need = wq.wq_mxfp4_combine_experts_workspace(R, S, E, N, K)
    assert need > R * S * N * 4  # the f32 slot results and the grouped GEMM's scratch
    ws = wq.alloc_workspace(need, d)
    st = torch.zeros(1, dtype=torch.int32, device=d)
    buf, y = guarded((R, N), torch.bfloat16, d)
    wq.wq_mxfp4_combine_experts(x.to(d), blocks.to(d), scales.to(d), experts.to(d), wts.to(d), y=y, workspace=ws,
                                dev_status=st)
    torch.cuda.synchronize()
    assert guards_intact(buf)
    assert "k_gemm_mx_tc" in wq.wq_last_launch(), wq.wq_last_launch()
    assert int(st.item()) & wq.WQ_DEV_BAD_EXPERT
    yr, ad, bad = oracle.mxfp4_combine_experts(bf16_bits(x), blocks.numpy(), scales.numpy(), experts.numpy(),
                                               wts.numpy(), N)
    assert bad == 1
    assert_within(y, yr, ad, "combine")


def test_grouped_gemm_crossover_knob(cuda_device, tune):
    """Below the default crossover the decode kernel runs; the knob moves the crossover
    and both kernels meet the same oracle."""
    d = cuda_device
    E, N, K, R, S = 8, 512, 1536, 20, 3
    blocks, scales = _experts(E, N, K, seed=51)
    experts = _route(R, S, E, seed=52)
    x = synth.normal_bf16((R, K), seed=53)
    assert wq.wq_mxfp4_experts_shared_workspace(R, S, E, N, K) == 0
    y0, _ = _run_shared(d, x, blocks, scales, experts, N)
    assert "k_gemv_mx" in wq.wq_last_launch(), wq.wq_last_launch()
    tune(wq.WQ_TUNE_MX_GEMM_MIN_SLOTS, 1)
    assert wq.wq_mxfp4_experts_shared_workspace(R, S, E, N, K) > 0
    y1, st = _run_shared(d, x, blocks, scales, experts, N)
    assert st == 0 and "k_gemm_mx_tc" in wq.wq_last_launch(), wq.wq_last_launch()
    _check_cols(y0, x, blocks, scales, experts, N, 0, N, "decode kernel")
    _check_cols(y1, x, blocks, scales, experts, N, 0, N, "grouped GEMM")


def test_grouped_gemm_workspace_rules(cuda_device):
    d = cuda_device
    E, N, K = 8, 256, 1024
    blocks, scales = _experts(E, N, K, seed=61)
    # 1024 slots with a workspace too small for the GEMM: the decode kernel takes them
    R, S = 256, 4
    experts = _route(R, S, E, seed=62)
    x = synth.normal_bf16((R, K), seed=63)
    small = wq.alloc_workspace(256, d)
    y, st = _run_shared(d, x, blocks, scales, experts, N, workspace=small)
    assert st == 0 and "k_gemv_mx" in wq.wq_last_launch(), wq.wq_last_launch()
    _check_cols(y, x, blocks, scales, experts, N, 0, N, "decode fallback")
    # 4096 slots (past the decode kernels' tables) without the GEMM's workspace: refused
    R2 = 1024
    e2 = _route(R2, S, E, seed=64)
    x2 = synth.normal_bf16((R2, K), seed=65)
    with pytest.raises(wq.WQError) as err:
        _run_shared(d, x2, blocks, scales, e2, N, workspace=small)
    assert err.value.status == wq.WQ_EWORKSPACE


@pytest.mark.parametrize("E,N,K,R,S", [(8, 384, 1024, 300, 4), (16, 256, 768, 1024, 4)])
def test_grouped_gemm_per_slot(cuda_device, E, N, K, R, S):
    """mxfp4_experts: one input row a slot (x [R, S, K]), 1200 and 4096 slots."""
    d = cuda_device
    blocks, scales = _experts(E, N, K, seed=71 + R)
    experts = _route(R, S, E, seed=72 + R)
    experts[1, 2] = E + 3
    x = synth.normal_bf16((R, S, K), seed=73 + R)
    st = torch.zeros(1, dtype=torch.int32, device=d)
    buf, y = guarded((R, S, N), torch.bfloat16, d)
    ws = wq.alloc_workspace(wq.wq_mxfp4_experts_workspace(R, S, E, N, K), d)
    wq.wq_mxfp4_experts(x.to(d), blocks.to(d), scales.to(d), experts.to(d), y=y, workspace=ws, dev_status=st)
    torch.cuda.synchronize()
    assert guards_intact(buf)
    assert "k_gemm_mx_tc" in wq.wq_last_launch(), wq.wq_last_launch()
    assert int(st.item()) & wq.WQ_DEV_BAD_EXPERT
    assert (y[1, 2].float() == 0).all()
    yr, ad, bad = oracle.mxfp4_experts(bf16_bits(x), blocks.numpy(), scales.numpy(), experts.numpy(), N)
    assert bad == 1
    assert_within(y, yr, ad, f"per slot R={R} S={S}")


@pytest.mark.parametrize("E,N,K,R,S", [(3, 16, 64, 40, 2), (2, 24, 96, 30, 2), (4, 8, 32, 50, 3)])
def test_grouped_gemm_small_shapes(cuda_device, tune, E, N, K, R, S):
    """Shapes smaller than a TMA box (K of one or two blocks, E * N under 256 rows, fewer
    routed rows than a half tile), forced onto the grouped GEMM by the crossover knob."""
    d = cuda_device
    tune(wq.WQ_TUNE_MX_GEMM_MIN_SLOTS, 1)
    blocks, scales = _experts(E, N, K, seed=81 + K)
    experts = _route(R, S, E, seed=82 + K)
    x = synth.normal_bf16((R, K), seed=83 + K)
    y, st = _run_shared(d, x, blocks, scales, experts, N)
    assert st == 0 and "k_gemm_mx_tc" in wq.wq_last_launch(), wq.wq_last_launch()
    assert _check_cols(y, x, blocks, scales, experts, N, 0, N, f"E={E} N={N} K={K}") == 0


def test_grouped_gemm_in_cuda_graph(cuda_device):
    """Captured once in a CUDA graph, replayed with new routings and inputs written into
    the same buffers: the launch shape does not depend on the routing (the grid is sized
    for the worst case), so every replay matches the oracle."""
    d = cuda_device
    E, N, K, R, S = 16, 512, 1024, 256, 4
    blocks, scales = _experts(E, N, K, seed=91)
    bd, sd = blocks.to(d), scales.to(d)
    x_buf = torch.empty((R, K), dtype=torch.bfloat16, device=d)
    e_buf = torch.empty((R, S), dtype=torch.int32, device=d)
    y = torch.empty((R, S, N), dtype=torch.bfloat16, device=d)
    ws = wq.alloc_workspace(wq.wq_mxfp4_experts_shared_workspace(R, S, E, N, K), d)
    routes = [_route(R, S, E, seed=92), _route(R, S, E, seed=93, kind="skew"), _route(R, S, E, seed=94, kind="one")]
    xs = [synth.normal_bf16((R, K), seed=95 + i) for i in range(3)]
    x_buf.copy_(xs[0])
    e_buf.copy_(routes[0])
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        wq.wq_mxfp4_linear_experts_shared(x_buf, bd, sd, e_buf, y=y, workspace=ws, stream=stream)  # warm-up
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            wq.wq_mxfp4_linear_experts_shared(x_buf, bd, sd, e_buf, y=y, workspace=ws, stream=stream)
    assert "k_gemm_mx_tc" in wq.wq_last_launch()
    for i in (1, 2, 0):
        x_buf.copy_(xs[i])
        e_buf.copy_(routes[i])
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert _check_cols(y, xs[i], blocks, scales, routes[i], N, 0, N, f"replay {i}") == 0
