"""Activation order on the GPU against the oracle ("Quantization" (Linnet docs):
Int4GroupLinear "optional order: [In; i32]"; "Importing GPTQ and AWQ": a checkpoint in
activation order gets an order and gathers its inputs first).

Stored column j of the weights multiplies input order[j]: y = x[:, order] . W-hat^T + b.
Covered: the decode kernel that gathers while staging activations (M = 1, 4), the decode
launches that gather into the workspace first (M = 12, group 64), and the tensor-core
GEMM after a gather pass (M = 256); permutations and repeated entries; an entry outside
[0, K) reads as 0 and sets WQ_DEV_BAD_ORDER.
"""
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


def _layer(n, k, g, seed):
    rng = np.random.default_rng(seed)
    packed = rng.integers(0, 256, (n, k // 2), dtype=np.uint8)
    scale = (rng.random((n, k // g)) * 0.018 + 0.002).astype(np.float32)
    zero = rng.integers(0, 16, (n, k // g), dtype=np.uint8)
    return packed, scale, zero


def _run(d, x, order, packed, scale, zero, bias, g):
    M, K = x.shape
    N = packed.shape[0]
    ws = wq.alloc_workspace(wq.wq_linear_int4_groups_ordered_workspace(M, N, K, g), d)
    buf, y = guarded((M, N), torch.bfloat16, d)
    st = torch.zeros(1, dtype=torch.int32, device=d)
    wq.wq_linear_int4_groups(x.to(d), torch.from_numpy(packed).to(d), torch.from_numpy(scale).to(d),
                             torch.from_numpy(zero).to(d), None if bias is None else bias.to(d), g, y=y,
                             workspace=ws, dev_status=st, order=torch.from_numpy(order).to(d))
    torch.cuda.synchronize()
    assert guards_intact(buf), "write outside y"
    return y, int(st.item())


@pytest.mark.parametrize("kind", ["permutation", "repeats"])
@pytest.mark.parametrize("M,N,K,G", [(1, 1000, 4096, 128), (4, 600, 14336, 128), (12, 500, 4096, 128),
                                     (1, 300, 2048, 64), (256, 520, 2048, 128), (40, 256, 1024, 32)])
def test_ordered_linear_matches_oracle(cuda_device, kind, M, N, K, G):
    d = cuda_device
    packed, scale, zero = _layer(N, K, G, seed=M + N + K)
    rng = np.random.default_rng(K + M)
    order = rng.permutation(K).astype(np.int32) if kind == "permutation" else \
        rng.integers(0, K, K).astype(np.int32)
    x = synth.normal_bf16((M, K), seed=M + 5)
    bias = synth.normal_bf16((N,), seed=N)
    y, st = _run(d, x, order, packed, scale, zero, bias, G)
    assert st == 0
    rows = np.unique(np.concatenate([np.arange(min(N, 32)), np.arange(max(0, N - 32), N),
                                     rng.choice(N, min(N, 128), replace=False)]))
    ms = np.unique(np.concatenate([[0, M - 1], rng.choice(M, min(M, 6), replace=False)]))
    yr, ad = oracle.linear_int4_groups_ordered(bf16_bits(x)[ms], order, packed[rows], scale[rows], zero[rows],
                                               bf16_bits(bias)[rows], len(rows), G)
    ysel = y[torch.from_numpy(ms).to(d)][:, torch.from_numpy(rows).to(d)]
    assert_within(ysel, yr, ad, f"order {kind} M={M} N={N} K={K} G={G}")


def test_identity_order_equals_plain_layer(cuda_device):
    d = cuda_device
    M, N, K, G = 1, 512, 4096, 128
    packed, scale, zero = _layer(N, K, G, seed=3)
    x = synth.normal_bf16((M, K), seed=4)
    y, st = _run(d, x, np.arange(K, dtype=np.int32), packed, scale, zero, None, G)
    y0 = wq.wq_linear_int4_groups(x.to(d), torch.from_numpy(packed).to(d), torch.from_numpy(scale).to(d),
                                  torch.from_numpy(zero).to(d), None, G)
    torch.cuda.synchronize()
    assert st == 0 and torch.equal(y.view(torch.int16), y0.view(torch.int16))


@pytest.mark.parametrize("M", [1, 256])
def test_out_of_range_entry_reads_zero(cuda_device, M):
    d = cuda_device
    N, K, G = 300, 2048, 128
    packed, scale, zero = _layer(N, K, G, seed=M + 9)
    rng = np.random.default_rng(M)
    order = rng.permutation(K).astype(np.int32)
    order[5] = K + 3
    order[K - 1] = -1
    x = synth.normal_bf16((M, K), seed=M + 10)
    y, st = _run(d, x, order, packed, scale, zero, None, G)
    assert st & wq.WQ_DEV_BAD_ORDER
    # the expected result: the gathered inputs with the two bad columns read as 0
    xb = bf16_bits(x)
    xg = xb[:, np.clip(order, 0, K - 1)]
    xg[:, [5, K - 1]] = 0
    ms = np.array([0, M - 1])
    yr, ad = oracle.linear_int4_groups(xg[ms], packed, scale, zero, None, N, G)
    assert_within(y[torch.from_numpy(ms).to(d)], yr, ad, f"bad order entries M={M}")


def test_ordered_call_needs_workspace(cuda_device):
    d = cuda_device
    N, K, G = 64, 256, 128
    packed, scale, zero = _layer(N, K, G, seed=1)
    x = synth.normal_bf16((1, K), seed=2).to(d)
    with pytest.raises(wq.WQError) as e:
        wq.wq_linear_int4_groups(x, torch.from_numpy(packed).to(d), torch.from_numpy(scale).to(d),
                                 torch.from_numpy(zero).to(d), None, G,
                                 order=torch.arange(K, dtype=torch.int32, device=d))
    assert e.value.status == wq.WQ_EWORKSPACE
