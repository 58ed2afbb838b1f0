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


@pytest.mark.parametrize("M,N,K,G", [(16, 14336, 4096, 128), (16, 14336, 4096, 64)])
def test_noalloc_large_decode_shapes_run_without_split(cuda_device, M, N, K, G):
    """The Llama gate shape at M = 16.  Group 128 takes the decode kernel that needs no
    scratch; group 64 takes the exact kernel, whose split-K scratch for this shape is
    larger than the static array, so the call runs it without cross-block split-K (as
    wq_linear_int4_groups does with a NULL workspace) instead of refusing."""
    d = cuda_device
    x, packed, scale, zero, bias = _inputs(M, N, K, G, seed=M + N + G, d=d)
    y1 = wq.wq_linear_int4_groups_noalloc(x, packed, scale, zero, bias, G)
    y2 = wq.wq_linear_int4_groups_noalloc(x, packed, scale, zero, bias, G)
    y_nows = wq.wq_linear_int4_groups(x, packed, scale, zero, bias, G)
    torch.cuda.synchronize()
    if G == 64:
        assert wq.wq_linear_int4_groups_workspace(M, N, K, G) > 1024 * 1024
    assert torch.equal(y1.view(torch.int16), y_nows.view(torch.int16))
    assert torch.equal(y2.view(torch.int16), y_nows.view(torch.int16))
    rows = np.random.default_rng(G).choice(N, 256, replace=False)
    rows.sort()
    yr, ad = oracle.linear_int4_groups(bf16_bits(x), packed.cpu().numpy()[rows], scale.cpu().numpy()[rows],
                                       zero.cpu().numpy()[rows], bf16_bits(bias)[rows], len(rows), G)
    assert_within(y1[:, torch.from_numpy(rows).to(d)], yr, ad, f"noalloc M={M} G={G}")


def test_noalloc_allocates_no_device_memory(cuda_device):
    """After a first call (which sets up the static array), further calls with a
    preallocated output change neither torch's allocator nor the device's free bytes."""
    d = cuda_device
    M, N, K, G = 2, 1000, 4096, 64                  # the exact kernel, split-K through the array
    x, packed, scale, zero, bias = _inputs(M, N, K, G, seed=9, d=d)
    assert 0 < wq.wq_linear_int4_groups_workspace(M, N, K, G) <= 1024 * 1024
    y = torch.empty((M, N), dtype=torch.bfloat16, device=d)
    wq.wq_linear_int4_groups_noalloc(x, packed, scale, zero, bias, G, y=y)
    torch.cuda.synchronize()
    y_first = y.clone()
    torch.cuda.synchronize()
    alloc0 = torch.cuda.memory_allocated(d)
    free0, _ = torch.cuda.mem_get_info(d)
    for _ in range(3):
        wq.wq_linear_int4_groups_noalloc(x, packed, scale, zero, bias, G, y=y)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info(d)
    assert torch.cuda.memory_allocated(d) == alloc0
    assert free1 == free0
    assert torch.equal(y.view(torch.int16), y_first.view(torch.int16))
