"""The allocation-free entry point (for callers that cannot call cudaMalloc and so
cannot pass a workspace) gives the results of wq_linear_int4_groups.

It keeps its split-K scratch in a static device array inside libwq, shared by every
call, so this file is collected last and checks two calls in a row on the same array;
it must pass alone in a fresh process and after the other tests.
"""
import numpy as np
import pytest
import torch

import oracle
import weight_only_quantized_linear_gb300 as wq
from weight_only_quantized_linear_gb300 import synth
from gpu_util import assert_within, bf16_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    wq.build()


def _inputs(M, N, K, G, seed, d):
    rng = np.random.default_rng(seed)
    packed = torch.from_numpy(rng.integers(0, 256, (N, K // 2)).astype(np.uint8)).to(d)
    scale = torch.from_numpy((rng.random((N, K // G)) * 0.018 + 0.002).astype(np.float32)).to(d)
    zero = torch.from_numpy(rng.integers(6, 10, (N, K // G)).astype(np.uint8)).to(d)
    x = synth.normal_bf16((M, K), seed=seed + 1).to(d)
    bias = synth.normal_bf16((N,), seed=seed + 2).to(d)
    return x, packed, scale, zero, bias


@pytest.mark.parametrize("M,N,K,G", [(1, 1000, 4096 + 1024, 128), (2, 300, 2048, 64), (1, 4096, 4096, 128)])
def test_noalloc_matches_workspace_entry_point_twice(cuda_device, M, N, K, G):
    d = cuda_device
    x, packed, scale, zero, bias = _inputs(M, N, K, G, seed=M + N, d=d)
    ws = wq.alloc_workspace(wq.wq_linear_int4_groups_workspace(M, N, K, G), d)
    y_ref = wq.wq_linear_int4_groups(x, packed, scale, zero, bias, G, workspace=ws)
    st = torch.zeros(1, dtype=torch.int32, device=d)
    y1 = wq.wq_linear_int4_groups_noalloc(x, packed, scale, zero, bias, G, dev_status=st)
    y2 = wq.wq_linear_int4_groups_noalloc(x, packed, scale, zero, bias, G, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    yr, ad = oracle.linear_int4_groups(bf16_bits(x), packed.cpu().numpy(), scale.cpu().numpy(),
                                       zero.cpu().numpy(), bf16_bits(bias), N, G)
    for y in (y_ref, y1, y2):
        assert_within(y, yr, ad, "noalloc")
    # same launch configuration and summation order: identical to the workspace path
    assert torch.equal(y1.view(torch.int16), y_ref.view(torch.int16))
    assert torch.equal(y2.view(torch.int16), y_ref.view(torch.int16))


def test_noalloc_refuses_shapes_beyond_its_scratch(cuda_device):
    d = cuda_device
    M, N, K, G = 1, 6_000_000, 32, 32       # 375000 tiles: counters alone exceed the array
    x, packed, scale, zero, _ = _inputs(1, 16, K, G, seed=5, d=d)
    big_packed = torch.zeros((N, K // 2), dtype=torch.uint8, device=d)
    big_scale = torch.ones((N, K // G), dtype=torch.float32, device=d)
    big_zero = torch.zeros((N, K // G), dtype=torch.uint8, device=d)
    assert wq.wq_linear_int4_groups_workspace(M, N, K, G) > 1024 * 1024
    with pytest.raises(wq.WQError) as e:
        wq.wq_linear_int4_groups_noalloc(x, big_packed, big_scale, big_zero, None, G)
    assert e.value.status == wq.WQ_EWORKSPACE
