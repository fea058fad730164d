"""Helpers shared by the GPU parity tests (not collected as tests).

Tolerance for bf16 outputs (fp32 arithmetic on both sides, one rounding to
bf16 each, SiLU through different exp implementations): an element passes
when |gpu - oracle| <= 1e-2 * |oracle| + 2e-5.  One bf16 ulp is 2^-8 (0.39%)
relative, so this admits a one-ulp rounding flip with margin and nothing
larger.  conv_state, the paged cache, untouched output regions and all
index outputs are compared bit for bit.
"""
from __future__ import annotations

import torch

RTOL = 1e-2
ATOL = 2e-5
SENTINEL = -12345


def to_device(kwargs: dict, dev) -> dict:
    return {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in kwargs.items()}


def sentinel_like(x: torch.Tensor, device=None) -> torch.Tensor:
    out = torch.empty_strided(x.shape, x.stride(), dtype=x.dtype,
                              device=x.device if device is None else device)
    out.view(torch.int16).fill_(SENTINEL)
    return out


def assert_close(got: torch.Tensor, ref: torch.Tensor, what: str = "") -> None:
    g = got.detach().float().cpu()
    r = ref.detach().float().cpu()
    assert g.shape == r.shape, (what, g.shape, r.shape)
    err = (g - r).abs()
    bound = RTOL * r.abs() + ATOL
    bad = ~(err <= bound)  # NaN counts as bad
    if bool(bad.any()):
        idx = int(bad.flatten().nonzero()[0])
        raise AssertionError(
            f"{what}: {int(bad.sum())}/{bad.numel()} elements outside tolerance; first at flat "
            f"index {idx}: gpu {float(g.flatten()[idx]):.6e} oracle {float(r.flatten()[idx]):.6e}")


def assert_bits(got: torch.Tensor, ref: torch.Tensor, what: str = "") -> None:
    g = got.detach().cpu()
    r = ref.detach().cpu()
    assert g.shape == r.shape, (what, g.shape, r.shape)
    if g.dtype == torch.bfloat16:
        g, r = g.view(torch.int16), r.view(torch.int16)
    neq = g != r
    if bool(neq.any()):
        idx = int(neq.flatten().nonzero()[0])
        raise AssertionError(f"{what}: {int(neq.sum())}/{neq.numel()} elements differ; first at "
                             f"flat index {idx}: {int(g.flatten()[idx])} vs {int(r.flatten()[idx])}")
