"""MXFP4 experts on the GPU against the CPU oracle at the gpt-oss-20b configuration (32
experts, K = 2880, N = 5760 and 2880, top-4 routing, R = 1, 8, 64): the shared-input,
per-slot-input, linear (x: [R, K]) and combine forms ("Quantization" (Linnet docs),
format table: mxfp4_experts_shared, mxfp4_experts, mxfp4_linear_experts_shared,
mxfp4_combine_experts).

Every 16-row output tile of every launch is checked: one sampled column in each tile,
plus the first and last 32 columns, against the oracle on the same columns of the
experts' weights, within |y_gpu - y_ref| <= 2e-3 * sum_k |x_k w_k| + 1 bf16 ulp(y_ref).
"""
import numpy as np
import pytest
import torch

import oracle
import weight_only_quantized_linear_gb300 as wq
from weight_only_quantized_linear_gb300 import synth
from gpu_util import assert_within, bf16_bits, guarded, guards_intact

pytestmark = pytest.mark.gpu

E, K, S = 32, 2880, 4


@pytest.fixture(scope="module", autouse=True)
def _built():
    wq.build()
    oracle.set_threads(oracle.max_threads())


def cols_every_tile(n, seed):
    """One column in every 16-row tile (its row inside the tile drawn from the seed), and
    the first and last 32 columns."""
    rng = np.random.default_rng(seed)
    tiles = (n + 15) // 16
    inside = np.minimum(np.arange(tiles) * 16 + rng.integers(0, 16, tiles), n - 1)
    return np.unique(np.concatenate([inside, np.arange(32), np.arange(n - 32, n)]))


@pytest.fixture(scope="module")
def experts_5760():
    return synth.mxfp4_experts(E, 5760, K, seed=41)


@pytest.fixture(scope="module")
def experts_2880():
    return synth.mxfp4_experts(E, 2880, K, seed=42)


def _weights(N, experts_5760, experts_2880):
    return experts_5760 if N == 5760 else experts_2880


def _sub(blocks, scales, cols):
    return (np.ascontiguousarray(blocks.numpy()[:, cols]), np.ascontiguousarray(scales.numpy()[:, cols]))


@pytest.mark.parametrize("R", [1, 8, 64])
@pytest.mark.parametrize("N", [5760, 2880])
def test_experts_shared_every_tile(cuda_device, experts_5760, experts_2880, R, N):
    d = cuda_device
    blocks, scales = _weights(N, experts_5760, experts_2880)
    experts, _ = synth.routing_topk(R, E, S, seed=100 + R)
    x = synth.normal_bf16((R, 1, K), seed=101 + R)
    st = torch.zeros(1, dtype=torch.int32, device=d)
    buf, y = guarded((R, S, N), torch.bfloat16, d)
    wq.wq_mxfp4_experts_shared(x.to(d), blocks.to(d), scales.to(d), experts.to(d), y=y, dev_status=st)
    torch.cuda.synchronize()
    assert guards_intact(buf) and int(st.item()) == 0
    cols = cols_every_tile(N, seed=R + N)
    b_s, s_s = _sub(blocks, scales, cols)
    yr, ad, bad = oracle.mxfp4_experts_shared(bf16_bits(x).reshape(R, K), b_s, s_s, experts.numpy(), len(cols))
    assert bad == 0
    assert_within(y[:, :, torch.from_numpy(cols).to(d)], yr, ad, f"shared R={R} N={N}")


@pytest.mark.parametrize("R", [1, 8, 64])
@pytest.mark.parametrize("N", [5760, 2880])
def test_experts_per_slot_every_tile(cuda_device, experts_5760, experts_2880, R, N):
    """mxfp4_experts: each slot its own input row, x [R, S, K]."""
    d = cuda_device
    blocks, scales = _weights(N, experts_5760, experts_2880)
    experts, _ = synth.routing_topk(R, E, S, seed=200 + R)
    x = synth.normal_bf16((R, S, K), seed=201 + R)
    st = torch.zeros(1, dtype=torch.int32, device=d)
    buf, y = guarded((R, S, N), torch.bfloat16, d)
    wq.wq_mxfp4_experts(x.to(d), blocks.to(d), scales.to(d), experts.to(d), y=y, dev_status=st)
    torch.cuda.synchronize()
    assert guards_intact(buf) and int(st.item()) == 0
    cols = cols_every_tile(N, seed=R + N + 1)
    b_s, s_s = _sub(blocks, scales, cols)
    yr, ad, bad = oracle.mxfp4_experts(bf16_bits(x), b_s, s_s, experts.numpy(), len(cols))
    assert bad == 0
    assert_within(y[:, :, torch.from_numpy(cols).to(d)], yr, ad, f"per-slot R={R} N={N}")


@pytest.mark.parametrize("R", [1, 8, 64])
@pytest.mark.parametrize("N", [5760, 2880])
def test_combine_experts_every_tile(cuda_device, experts_5760, experts_2880, R, N):
    """mxfp4_combine_experts with the configured combine weights: a softmax over each
    row's four routing logits."""
    d = cuda_device
    blocks, scales = _weights(N, experts_5760, experts_2880)
    experts, logits = synth.routing_topk(R, E, S, seed=300 + R)
    weights = torch.softmax(logits, dim=-1).contiguous()
    x = synth.normal_bf16((R, 1, K), seed=301 + R)
    st = torch.zeros(1, dtype=torch.int32, device=d)
    buf, y = guarded((R, N), torch.bfloat16, d)
    wq.wq_mxfp4_combine_experts(x.to(d), blocks.to(d), scales.to(d), experts.to(d), weights.to(d), y=y,
                                dev_status=st)
    torch.cuda.synchronize()
    assert guards_intact(buf) and int(st.item()) == 0
    cols = cols_every_tile(N, seed=R + N + 2)
    b_s, s_s = _sub(blocks, scales, cols)
    yr, ad, bad = oracle.mxfp4_combine_experts(bf16_bits(x).reshape(R, K), b_s, s_s, experts.numpy(),
                                               weights.numpy(), len(cols))
    assert bad == 0
    assert_within(y[:, torch.from_numpy(cols).to(d)], yr, ad, f"combine R={R} N={N}")


def test_combine_skips_bad_slots_and_is_deterministic(cuda_device):
    d = cuda_device
    e, n, k, r, s = 5, 200, 320, 12, 3
    blocks, scales = synth.mxfp4_experts(e, n, k, seed=61)
    rng = np.random.default_rng(62)
    experts = rng.integers(0, e, (r, s)).astype(np.int32)
    experts[2, 1] = e          # out of range: adds nothing
    experts[5, 0] = -3
    experts[7, :] = 99         # a row with no valid slot: zeros
    weights = rng.random((r, s)).astype(np.float32)
    x = synth.normal_bf16((r, k), seed=63)
    args = (x.to(d), blocks.to(d), scales.to(d), torch.from_numpy(experts).to(d), torch.from_numpy(weights).to(d))
    st = torch.zeros(1, dtype=torch.int32, device=d)
    y1 = wq.wq_mxfp4_combine_experts(*args, dev_status=st)
    y2 = wq.wq_mxfp4_combine_experts(*args)
    torch.cuda.synchronize()
    assert int(st.item()) & wq.WQ_DEV_BAD_EXPERT
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    assert (y1[7].float() == 0).all()
    yr, ad, bad = oracle.mxfp4_combine_experts(bf16_bits(x), blocks.numpy(), scales.numpy(), experts, weights, n)
    assert bad == 5
    assert_within(y1, yr, ad, "combine with bad slots")


def test_linear_experts_shared_many_rows(cuda_device, experts_2880):
    """mxfp4_linear_experts_shared, x [R, K] with many rows (R = 300, 1200 routed slots):
    the oracle on every tile, and the same bits as the shared-input entry point."""
    d = cuda_device
    R, N = 300, 2880
    blocks, scales = experts_2880
    experts, _ = synth.routing_topk(R, E, S, seed=400)
    x = synth.normal_bf16((R, K), seed=401)
    st = torch.zeros(1, dtype=torch.int32, device=d)
    y = wq.wq_mxfp4_linear_experts_shared(x.to(d), blocks.to(d), scales.to(d), experts.to(d), dev_status=st)
    y_sh = wq.wq_mxfp4_experts_shared(x.view(R, 1, K).to(d), blocks.to(d), scales.to(d), experts.to(d))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(y.view(torch.int16), y_sh.view(torch.int16))
    cols = cols_every_tile(N, seed=5)
    b_s, s_s = _sub(blocks, scales, cols)
    rows = np.unique(np.concatenate([np.arange(4), np.arange(R - 4, R),
                                     np.random.default_rng(6).choice(R, 24, replace=False)]))
    yr, ad, bad = oracle.mxfp4_experts_shared(bf16_bits(x)[rows], b_s, s_s, experts.numpy()[rows], len(cols))
    ysel = y[torch.from_numpy(rows).to(d)][:, :, torch.from_numpy(cols).to(d)]
    assert_within(ysel, yr, ad, "linear experts shared")


def test_per_slot_bad_index(cuda_device):
    d = cuda_device
    e, n, k, r, s = 3, 100, 256, 6, 2
    blocks, scales = synth.mxfp4_experts(e, n, k, seed=71)
    experts = np.array([[0, 1], [2, 3], [1, 1], [-1, 0], [2, 2], [0, 2]], np.int32)
    x = synth.normal_bf16((r, s, k), seed=72)
    st = torch.zeros(1, dtype=torch.int32, device=d)
    y = wq.wq_mxfp4_experts(x.to(d), blocks.to(d), scales.to(d), torch.from_numpy(experts).to(d), dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & wq.WQ_DEV_BAD_EXPERT
    assert (y[1, 1].float() == 0).all() and (y[3, 0].float() == 0).all()
    yr, ad, bad = oracle.mxfp4_experts(bf16_bits(x), blocks.numpy(), scales.numpy(), experts, n)
    assert bad == 2
    assert_within(y, yr, ad, "per-slot with bad indices")
