"""The MXFP4 TMA-ring cluster kernel (k_gemv_mx) against the CPU oracle: shapes at the
edges of its rules (K = 768, a last step cut by K, several batches of eight slots for one
expert, N a multiple of 16), scales above 128 (the two-multiply dequantization), every
cluster count, bad and all-bad expert indices, and the shared, per-slot and combine forms
("Quantization" (Linnet docs), format table: mxfp4_experts_shared, mxfp4_experts,
mxfp4_combine_experts).  Tolerance: |y_gpu - y_ref| <= 2e-3 * sum_k |x_k w_k| + 1 bf16
ulp(y_ref); the exact kernel (WQ_TUNE_DECODE = 2) is held to the same oracle."""
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


def _route(R, S, E, seed):
    rng = np.random.default_rng(seed)
    return torch.from_numpy(np.stack([rng.choice(E, S, replace=False) for _ in range(R)]).astype(np.int32))


def _shared(d, x, blocks, scales, experts, N):
    R, S = experts.shape
    st = torch.zeros(1, dtype=torch.int32, device=d)
    buf, y = guarded((R, S, N), torch.bfloat16, d)
    wq.wq_mxfp4_experts_shared(x.to(d), blocks.to(d), scales.to(d), experts.to(d), y=y, dev_status=st)
    torch.cuda.synchronize()
    assert guards_intact(buf), "write outside y"
    return y, int(st.item())


@pytest.mark.parametrize("E,N,K,R,S,elo,ehi", [
    (32, 5760, 2880, 1, 4, 118, 124),   # gpt-oss gate/up, one routed row
    (8, 256, 768, 3, 2, 118, 124),      # three steps a tile: the ring's tile-buffer edge
    (5, 160, 1056, 20, 3, 110, 130),    # K/2 = 528: last step cut by K; 12 slots an expert
    (4, 2880, 2880, 2, 4, 100, 200),    # scales above 128 in most units (two multiplies)
    (16, 512, 4096, 8, 4, 118, 124),
])
def test_ring_kernel_matches_oracle(cuda_device, tune, E, N, K, R, S, elo, ehi):
    d = cuda_device
    blocks, scales = _experts(E, N, K, seed=E + N + K, elo=elo, ehi=ehi)
    experts = _route(R, S, E, seed=R + S)
    x = synth.normal_bf16((R, 1, K), seed=K + R)
    y, st = _shared(d, x, blocks, scales, experts, N)
    assert st == 0
    assert "k_gemv_mx" in wq.wq_last_launch(), wq.wq_last_launch()
    yr, ad, bad = oracle.mxfp4_experts_shared(bf16_bits(x).reshape(R, K), blocks.numpy(), scales.numpy(),
                                              experts.numpy(), N)
    assert bad == 0
    assert_within(y, yr, ad, f"ring E={E} N={N} K={K} R={R} S={S}")
    y2, _ = _shared(d, x, blocks, scales, experts, N)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16)), "not deterministic"
    tune(wq.WQ_TUNE_DECODE, 2)  # the exact kernel, same oracle
    y3, _ = _shared(d, x, blocks, scales, experts, N)
    assert "k_gemv<MXFP4" in wq.wq_last_launch(), wq.wq_last_launch()
    assert_within(y3, yr, ad, "exact kernel")


@pytest.mark.parametrize("clusters", [1, 2, 5, 13, 1000])
def test_ring_kernel_every_cluster_count(cuda_device, tune, clusters):
    """Every split of the items between clusters gives the same bits (tiles cut between
    warps anywhere are finished from their partials in warp order)."""
    d = cuda_device
    E, N, K, R, S = 6, 480, 1536, 5, 3
    blocks, scales = _experts(E, N, K, seed=7)
    experts = _route(R, S, E, seed=8)
    x = synth.normal_bf16((R, 1, K), seed=9)
    tune(wq.WQ_TUNE_GEMV_CLUSTERS, clusters)
    y, st = _shared(d, x, blocks, scales, experts, N)
    assert st == 0 and "k_gemv_mx" in wq.wq_last_launch()
    yr, ad, _ = oracle.mxfp4_experts_shared(bf16_bits(x).reshape(R, K), blocks.numpy(), scales.numpy(),
                                            experts.numpy(), N)
    assert_within(y, yr, ad, f"clusters={clusters}")
    y2, _ = _shared(d, x, blocks, scales, experts, N)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


def test_ring_kernel_bad_and_all_bad_experts(cuda_device):
    d = cuda_device
    E, N, K, R, S = 8, 256, 1024, 4, 2
    blocks, scales = _experts(E, N, K, seed=11)
    experts = _route(R, S, E, seed=12)
    experts[1, 0] = -3
    experts[2, 1] = E
    x = synth.normal_bf16((R, 1, K), seed=13)
    y, st = _shared(d, x, blocks, scales, experts, N)
    assert "k_gemv_mx" in wq.wq_last_launch()
    assert st & wq.WQ_DEV_BAD_EXPERT
    yr, ad, bad = oracle.mxfp4_experts_shared(bf16_bits(x).reshape(R, K), blocks.numpy(), scales.numpy(),
                                              experts.numpy(), N)
    assert bad == 2
    assert (y[1, 0].float() == 0).all() and (y[2, 1].float() == 0).all()
    assert_within(y, yr, ad, "bad experts")
    # no valid slot at all: every output row is zero and the launch still completes
    y0, st0 = _shared(d, x, blocks, scales, torch.full((R, S), -1, dtype=torch.int32), N)
    assert st0 & wq.WQ_DEV_BAD_EXPERT
    assert (y0.float() == 0).all()


@pytest.mark.parametrize("form", ["per_slot", "combine"])
def test_ring_kernel_per_slot_and_combine(cuda_device, form):
    d = cuda_device
    E, N, K, R, S = 32, 2880, 2880, 2, 4
    blocks, scales = _experts(E, N, K, seed=21)
    experts = _route(R, S, E, seed=22)
    if form == "per_slot":
        x = synth.normal_bf16((R, S, K), seed=23)
        st = torch.zeros(1, dtype=torch.int32, device=d)
        buf, y = guarded((R, S, N), torch.bfloat16, d)
        wq.wq_mxfp4_experts(x.to(d), blocks.to(d), scales.to(d), experts.to(d), y=y, dev_status=st)
        torch.cuda.synchronize()
        assert guards_intact(buf) and int(st.item()) == 0
        assert "k_gemv_mx" in wq.wq_last_launch()
        yr, ad, bad = oracle.mxfp4_experts(bf16_bits(x), blocks.numpy(), scales.numpy(), experts.numpy(), N)
        assert_within(y, yr, ad, "per slot")
    else:
        x = synth.normal_bf16((R, 1, K), seed=24)
        wts = torch.softmax(torch.from_numpy(np.random.default_rng(25).normal(size=(R, S))).float(), -1)
        st = torch.zeros(1, dtype=torch.int32, device=d)
        ws = wq.alloc_workspace(wq.wq_mxfp4_combine_experts_workspace(R, S, E, N, K), d)
        buf, y = guarded((R, N), torch.bfloat16, d)
        wq.wq_mxfp4_combine_experts(x.to(d), blocks.to(d), scales.to(d), experts.to(d), wts.to(d), y=y,
                                    workspace=ws, dev_status=st)
        torch.cuda.synchronize()
        assert guards_intact(buf) and int(st.item()) == 0
        yr, ad, bad = oracle.mxfp4_combine_experts(bf16_bits(x).reshape(R, K), blocks.numpy(), scales.numpy(),
                                                   experts.numpy(), wts.numpy(), N)
        assert_within(y, yr, ad, "combine")
