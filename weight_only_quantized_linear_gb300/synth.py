"""Seeded synthetic inputs for the weight-only quantized linear layer.

This module draws random numbers and nothing else: no quantization, packing or
dequantization happens here, so both the CUDA library and the CPU oracle can be fed
from it without sharing any of the method's arithmetic.  Every function takes explicit
seeds and returns torch tensors on ``device`` (CPU by default).

Workloads (shapes and distributions follow the layer shapes the pages measure on; the
Llama-3.1-8B and gpt-oss-20b weights themselves are not available, so seeded tensors of
their shapes stand in for them):

* tiny group-wise W4A16 layer: x [1, 256], 256 x 256 weight, group 32, uniform codes
* Llama-3.1-8B decode projections (N x K): q/o 4096x4096, k/v 1024x4096,
  gate/up 14336x4096, down 4096x14336; W ~ N(0, 0.02) with 0.1 % of entries x20
* per-row int8 / int4: W ~ N(0, 0.02)
* MXFP4 experts: 32 experts, K = 2880, N in {5760, 2880}, top-4 routing
"""
from __future__ import annotations

import torch

LLAMA_PROJ = {
    "q": (4096, 4096),
    "k": (1024, 4096),
    "v": (1024, 4096),
    "o": (4096, 4096),
    "gate": (14336, 4096),
    "up": (14336, 4096),
    "down": (4096, 14336),
}
LLAMA_ORDER = ("q", "k", "v", "o", "gate", "up", "down")


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal_bf16(shape, seed: int, device="cpu") -> torch.Tensor:
    """x ~ N(0, 1) drawn in f32 and stored as bf16."""
    g = _gen(seed, device)
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def weight_f32(n: int, k: int, seed: int, std: float = 0.02, outlier_frac: float = 0.0,
               outlier_mult: float = 20.0, device="cpu") -> torch.Tensor:
    """W ~ N(0, std) in f32; a fraction of entries, chosen uniformly without replacement,
    multiplied by ``outlier_mult``."""
    g = _gen(seed, device)
    w = torch.randn((n, k), generator=g, device=device, dtype=torch.float32) * std
    count = int(round(outlier_frac * n * k))
    if count:
        idx = torch.randperm(n * k, generator=g, device=device)[:count]
        flat = w.view(-1)
        flat[idx] = flat[idx] * outlier_mult
    return w


def uniform_bytes(shape, seed: int, device="cpu") -> torch.Tensor:
    """Bytes uniform over 0..255 (= two independent uniform 4-bit codes a byte)."""
    g = _gen(seed, device)
    return torch.randint(0, 256, shape, generator=g, device=device, dtype=torch.int32).to(torch.uint8)


def uniform_f32(shape, lo: float, hi: float, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    return torch.rand(shape, generator=g, device=device, dtype=torch.float32) * (hi - lo) + lo


def uniform_int(shape, lo: int, hi_inclusive: int, seed: int, dtype=torch.uint8,
                device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    return torch.randint(lo, hi_inclusive + 1, shape, generator=g, device=device,
                         dtype=torch.int32).to(dtype)


def tiny_int4_groups(seed: int = 0):
    """The tiny group-wise layer: x bf16 [1, 256]; packed u8 [256, 8, 16]; scale f32
    [256, 8] ~ U[0.002, 0.02]; zero u8 [256, 8] ~ U{6..9}; W f32 [256, 256] ~ N(0, 0.02)
    for the quantizer."""
    return {
        "x": normal_bf16((1, 256), seed + 1),
        "packed": uniform_bytes((256, 8, 16), seed + 2),
        "scale": uniform_f32((256, 8), 0.002, 0.02, seed + 3),
        "zero": uniform_int((256, 8), 6, 9, seed + 4),
        "w": weight_f32(256, 256, seed + 5),
        "N": 256, "K": 256, "G": 32,
    }


def routing_topk(r: int, e: int, s: int, seed: int, device="cpu"):
    """experts i32 [R, S]: S distinct experts per row, uniformly without replacement;
    combine logits f32 [R, S] ~ N(0, 1)."""
    g = _gen(seed, "cpu")
    ex = torch.stack([torch.randperm(e, generator=g)[:s] for _ in range(r)]).to(torch.int32)
    logits = torch.randn((r, s), generator=g, dtype=torch.float32)
    return ex.to(device), logits.to(device)


def mxfp4_experts(e: int, n: int, k: int, seed: int, device="cpu"):
    """blocks u8 [E, N, K/32, 16] (uniform E2M1 codes), scales u8 [E, N, K/32] ~ U{118..124}."""
    return (uniform_bytes((e, n, k // 32, 16), seed, device),
            uniform_int((e, n, k // 32), 118, 124, seed + 1, device=device))
