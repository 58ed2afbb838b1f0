"""The tensor-core regime at the benchmark's prefill sizes, against the CPU oracle.

Llama-3.1-8B projection shapes at M = 2048 (gate 14336 x 4096; down 4096 x 14336, i.e.
K = 14336 and 224 k steps; k and v 1024 x 4096 on the 128 x 128 tiles) and
M = 512 (gate), group 128, in the launch configuration the benchmark times (workspace
sized by wq_linear_int4_groups_workspace).  The oracle computes sampled rows of x times
sampled output columns that include the first and the last 256-wide column tiles and
the first and last 256-row tiles of x; each element must lie within
|y_gpu - y_ref| <= 2e-3 * sum_k |x_k w_k| + 1 bf16 ulp(y_ref).
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


def _weights(n, k, g, seed):
    rng = np.random.default_rng(seed)
    packed = rng.integers(0, 256, (n, k // 2), dtype=np.uint8)
    scale = (rng.random((n, k // g)) * 0.018 + 0.002).astype(np.float32)
    zero = rng.integers(0, 16, (n, k // g), dtype=np.uint8)
    return packed, scale, zero


def _sample(total, edge, count, seed):
    """Indices: the first and last `edge`, plus `count` others drawn from the seed."""
    rng = np.random.default_rng(seed)
    pick = np.concatenate([np.arange(min(edge, total)), np.arange(max(0, total - edge), total),
                           rng.choice(total, min(count, total), replace=False)])
    return np.unique(pick)


@pytest.mark.parametrize("name,M", [("gate", 2048), ("down", 2048), ("gate", 512), ("k", 2048),
                                    ("v", 2048), ("q", 2048)])
def test_prefill_full_size_sampled(cuda_device, name, M):
    d = cuda_device
    G = 128
    N, K = synth.LLAMA_PROJ[name]
    packed, scale, zero = _weights(N, K, G, seed=N + K + M)
    x = synth.normal_bf16((M, K), seed=M + K)
    bias = synth.normal_bf16((N,), seed=N + 3)
    nbytes = wq.wq_linear_int4_groups_workspace(M, N, K, G)
    ws = wq.alloc_workspace(nbytes, d)
    buf, y = guarded((M, N), torch.bfloat16, d)
    st = torch.zeros(1, dtype=torch.int32, device=d)
    wq.wq_linear_int4_groups(x.to(d), torch.from_numpy(packed).to(d), torch.from_numpy(scale).to(d),
                             torch.from_numpy(zero).to(d), bias.to(d), G, y=y, workspace=ws, dev_status=st)
    torch.cuda.synchronize()
    if name in ("k", "v"):
        # fewer 256 x 256 tiles than SMs: the 128 x 128 tiles, whole K, no partials
        assert "tile=128" in wq.wq_last_launch() and nbytes == 0, wq.wq_last_launch()
    assert guards_intact(buf), "write outside y"
    assert int(st.item()) == 0
    if ws is not None:
        assert int(ws.view(torch.int32).abs().sum().item()) == 0, "split-K partials not cleared"
    rows = _sample(M, 2, 6, seed=M)                 # rows of x: both 256-row tile ends
    cols = _sample(N, 256, 192, seed=N)             # first and last 256-wide column tiles
    yr, ad = oracle.linear_int4_groups(bf16_bits(x)[rows], packed[cols], scale[cols], zero[cols],
                                       bf16_bits(bias)[cols], len(cols), G)
    ysel = y[torch.from_numpy(rows).to(d)][:, torch.from_numpy(cols).to(d)]
    assert_within(ysel, yr, ad, f"prefill {name} M={M} N={N} K={K}")
    # and the tile edges inside x: rows 255/256 (a 256-row tile boundary) on a few columns
    if M > 256:
        r2 = np.array([255, 256, M - 257, M - 256])
        c2 = cols[:32]
        yr2, ad2 = oracle.linear_int4_groups(bf16_bits(x)[r2], packed[c2], scale[c2], zero[c2],
                                             bf16_bits(bias)[c2], len(c2), G)
        y2 = y[torch.from_numpy(r2).to(d)][:, torch.from_numpy(c2).to(d)]
        assert_within(y2, yr2, ad2, f"prefill {name} M={M} tile-edge rows")
