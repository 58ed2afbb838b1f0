"""Helpers for the GPU parity tests: bf16 <-> bit arrays, guarded outputs, tolerance."""
import numpy as np
import torch

import oracle


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor (any device) -> numpy uint16 bit patterns."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().double().numpy()


def from_bits(b: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).to(device)


GUARD = 512
SENTINEL = 0x7FAB  # a NaN pattern no kernel writes


def guarded(shape, dtype, device):
    """An output buffer with GUARD sentinel elements on both sides of the view."""
    n = int(np.prod(shape))
    buf = torch.empty(n + 2 * GUARD, dtype=torch.int16, device=device)
    buf.fill_(SENTINEL)
    view = buf[GUARD:GUARD + n].view(dtype).view(shape)
    return buf, view


def guards_intact(buf) -> bool:
    b = buf.cpu()
    return bool((b[:GUARD] == SENTINEL).all() and (b[-GUARD:] == SENTINEL).all())


def assert_within(y_gpu: torch.Tensor, y_ref: np.ndarray, absdot: np.ndarray, what: str = ""):
    y = bf16_to_f64(y_gpu).reshape(y_ref.shape)
    ok = oracle.within_tolerance(y, y_ref, absdot)
    if not ok.all():
        idx = np.argwhere(~ok)[:5]
        msg = [f"{tuple(i)}: gpu={y[tuple(i)]!r} ref={y_ref[tuple(i)]!r} absdot={absdot[tuple(i)]!r}"
               for i in idx]
        raise AssertionError(f"{what}: {int((~ok).sum())} of {ok.size} outside tolerance\n" + "\n".join(msg))
    # the bound must not be vacuous: errors stay far inside it on random data
    err = np.abs(y - y_ref)
    bound = 2e-3 * absdot + oracle.bf16_ulp(y_ref)
    return float((err / np.maximum(bound, 1e-300)).max())
