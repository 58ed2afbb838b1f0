"""The prepared (load-time repacked) group-wise 4-bit layout ("Quantization" (Linnet docs),
"Group-wise 4-bit weights": weights repacked at load, --prepare) and its decode kernel.

The repack is checked byte for byte against a numpy restatement of the layout documented
in include/wq.h; the linear against the CPU oracle (the same definition and tolerance as
wq_linear_int4_groups) at ragged and full Llama-3.1-8B sizes, every split of the work
into thread-block ranges, with and without a workspace.
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


def _layer(n, k, g, seed, zlo=0, zhi=16):
    rng = np.random.default_rng(seed)
    return (rng.integers(0, 256, (n, k // 2), dtype=np.uint8),
            (rng.random((n, k // g)) * 0.018 + 0.002).astype(np.float32),
            rng.integers(zlo, zhi, (n, k // g), dtype=np.uint8))


def prepared_reference(packed, scale, zero, n, k, g):
    """The documented prepared layout, built in numpy from the public one."""
    rbs, ks = -(-n // 128), k // 256
    codes = np.zeros((rbs * 128, k), np.uint8)
    codes[:n, 0::2] = packed & 15
    codes[:n, 1::2] = packed >> 4
    swz = ((np.arange(128) & 1) << 2) | ((np.arange(128) >> 1) & 3)
    nib_of = np.array([0, 4, 1, 5, 2, 6, 3, 7])       # nibble holding code j of a word
    out_codes = np.zeros((rbs, ks, 128, 8, 4), np.uint32)
    for rb in range(rbs):
        for st in range(ks):
            blk = codes[rb * 128:(rb + 1) * 128, st * 256:(st + 1) * 256].astype(np.uint32)
            for u in range(8):
                c, q = u >> 2, u & 3
                for i in range(4):
                    k0 = c * 128 + (4 * i + q) * 8
                    word = np.zeros(128, np.uint32)
                    for j in range(8):
                        word |= blk[:, k0 + j] << np.uint32(4 * nib_of[j])
                    pos = u ^ swz
                    out_codes[rb, st, np.arange(128), pos, i] = word
    gpr = k // g
    s_pad = np.zeros((rbs * 128, gpr), np.float32)
    z_pad = np.zeros((rbs * 128, gpr), np.uint8)
    s_pad[:n], z_pad[:n] = scale, zero
    meta = np.zeros((rbs, ks, 1280), np.uint8)
    for st in range(ks):
        g0, g1 = (st * 256) // g, (st * 256 + 128) // g
        for rb in range(rbs):
            rows = slice(rb * 128, (rb + 1) * 128)
            sc = np.stack([s_pad[rows, g0], s_pad[rows, g1]], 1).astype(np.float32)
            zc = np.stack([z_pad[rows, g0], z_pad[rows, g1]], 1).astype(np.uint8)
            meta[rb, st, :1024] = sc.view(np.uint8).reshape(-1)
            meta[rb, st, 1024:] = zc.reshape(-1)
    return np.concatenate([out_codes.view(np.uint8).reshape(-1), meta.reshape(-1)])


@pytest.mark.parametrize("N,K,G", [(128, 256, 128), (300, 512, 128), (129, 1024, 256), (1000, 2048, 512)])
def test_prepare_matches_documented_layout(cuda_device, N, K, G):
    d = cuda_device
    p, s, z = _layer(N, K, G, seed=N + K)
    prep = wq.wq_prepare_int4_groups(torch.from_numpy(p).to(d), torch.from_numpy(s).to(d),
                                     torch.from_numpy(z).to(d), G)
    torch.cuda.synchronize()
    ref = prepared_reference(p, s, z, N, K, G)
    assert prep.numel() == ref.size == wq.lib().wq_prepared_int4_groups_bytes(N, K, G)
    assert np.array_equal(prep.cpu().numpy(), ref)


def _run(d, x, prep, N, bias, G, use_ws=True):
    M, K = x.shape
    ws = wq.alloc_workspace(wq.wq_linear_int4_groups_prepared_workspace(M, N, K, G), d) if use_ws else None
    buf, y = guarded((M, N), torch.bfloat16, d)
    st = torch.zeros(1, dtype=torch.int32, device=d)
    wq.wq_linear_int4_groups_prepared(x, prep, N, bias, G, y=y, workspace=ws, dev_status=st)
    torch.cuda.synchronize()
    assert guards_intact(buf), "write outside y"
    assert int(st.item()) == 0
    assert "k_gemv_prep" in wq.wq_last_launch()
    if ws is not None:
        assert int(ws.view(torch.int32).abs().sum().item()) == 0, "workspace not left zero-filled"
    return y


@pytest.mark.parametrize("M,N,K,G,zrange", [(1, 1000, 4096, 128, (0, 16)), (1, 64, 2048, 256, (0, 16)),
                                            (2, 300, 4096, 128, (0, 256)), (5, 129, 2048, 128, (6, 10)),
                                            (8, 4096, 4096, 128, (0, 16)), (9, 200, 2048, 128, (0, 256)),
                                            (16, 1100, 4096, 128, (0, 16)), (3, 14336, 4096, 128, (0, 16))])
def test_prepared_linear_matches_oracle(cuda_device, M, N, K, G, zrange):
    d = cuda_device
    p, s, z = _layer(N, K, G, seed=M + N, zlo=zrange[0], zhi=zrange[1])
    prep = wq.wq_prepare_int4_groups(torch.from_numpy(p).to(d), torch.from_numpy(s).to(d),
                                     torch.from_numpy(z).to(d), G)
    x = synth.normal_bf16((M, K), seed=M + K)
    b = synth.normal_bf16((N,), seed=N)
    y = _run(d, x.to(d), prep, N, b.to(d), G)
    rows = np.unique(np.concatenate([np.arange(min(N, 64)), np.arange(max(0, N - 64), N),
                                     np.random.default_rng(N).choice(N, min(N, 256), replace=False)]))
    yr, ad = oracle.linear_int4_groups(bf16_bits(x), p[rows], s[rows], z[rows], bf16_bits(b)[rows], len(rows), G)
    assert_within(y[:, torch.from_numpy(rows).to(d)], yr, ad, f"prepared M={M} N={N} K={K} G={G}")
    y2 = _run(d, x.to(d), prep, N, b.to(d), G, use_ws=False)
    assert_within(y2[:, torch.from_numpy(rows).to(d)], yr, ad, f"prepared whole blocks M={M} N={N} K={K}")


@pytest.mark.parametrize("blocks", [1, 2, 5, 17, 64, 150, 10000])
@pytest.mark.parametrize("M", [1, 6])
def test_prepared_partitions(cuda_device, tune, blocks, M):
    d = cuda_device
    tune(wq.WQ_TUNE_GEMV_BLOCKS, blocks)
    N, K, G = 1000, 6144, 128
    p, s, z = _layer(N, K, G, seed=blocks)
    prep = wq.wq_prepare_int4_groups(torch.from_numpy(p).to(d), torch.from_numpy(s).to(d),
                                     torch.from_numpy(z).to(d), G)
    x = synth.normal_bf16((M, K), seed=M)
    y = _run(d, x.to(d), prep, N, None, G)
    yr, ad = oracle.linear_int4_groups(bf16_bits(x), p, s, z, None, N, G)
    assert_within(y, yr, ad, f"prepared blocks={blocks} M={M}")
    y2 = _run(d, x.to(d), prep, N, None, G)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


@pytest.mark.parametrize("name", synth.LLAMA_ORDER)
def test_prepared_llama_full_size_sampled(cuda_device, name):
    """Full Llama-3.1-8B projections at M = 1, group 128, weights quantized by the oracle,
    in the launch configuration the benchmark times (workspace on, static weights)."""
    d = cuda_device
    N, K = synth.LLAMA_PROJ[name]
    w = synth.weight_f32(N, K, seed=61, outlier_frac=0.001)
    codes, scale, zero, _ = oracle.quantize_asym(w.numpy(), 128, 4)
    _, packed = oracle.pack_int4(codes, True)
    prep = wq.wq_prepare_int4_groups(torch.from_numpy(packed).to(d), torch.from_numpy(scale).to(d),
                                     torch.from_numpy(zero).to(d), 128)
    x = synth.normal_bf16((1, K), seed=62)
    wq.wq_set_static_weights(True)
    try:
        y = _run(d, x.to(d), prep, N, None, 128)
    finally:
        wq.wq_set_static_weights(False)
    rows = np.unique(np.concatenate([np.arange(16), np.arange(N - 16, N),
                                     np.random.default_rng(63).choice(N, 352, replace=False)]))
    yr, ad = oracle.linear_int4_groups(bf16_bits(x), packed[rows], scale[rows], zero[rows], None, len(rows), 128)
    assert_within(y[:, torch.from_numpy(rows).to(d)], yr, ad, f"prepared {name}")


def test_prepared_refuses_unsupported(cuda_device):
    d = cuda_device
    p, s, z = _layer(64, 384, 128, seed=1)     # K % 256 != 0
    assert wq.lib().wq_prepared_int4_groups_bytes(64, 384, 128) == 0
    with pytest.raises(wq.WQError) as e:
        wq.wq_prepare_int4_groups(torch.from_numpy(p).to(d), torch.from_numpy(s).to(d), torch.from_numpy(z).to(d),
                                  128)
    assert e.value.status == wq.WQ_EUNSUPPORTED
    p, s, z = _layer(64, 512, 128, seed=2)
    prep = wq.wq_prepare_int4_groups(torch.from_numpy(p).to(d), torch.from_numpy(s).to(d),
                                     torch.from_numpy(z).to(d), 128)
    with pytest.raises(wq.WQError) as e:       # the prefill regime reads the public layout
        wq.wq_linear_int4_groups_prepared(synth.normal_bf16((17, 512), seed=3).to(d), prep, 64, None, 128)
    assert e.value.status == wq.WQ_EUNSUPPORTED
