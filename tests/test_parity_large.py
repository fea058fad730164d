"""GPU parity past 2^31 elements: one sequence of 270,000 tokens at dim 8192
(2.2 G elements, 4.4 GB per tensor) in both layouts, so every element offset
above 2^31 must be computed in 64 bits.  The inputs follow a cheap closed
formula evaluated on the device; the CPU oracle gets the same values for a
sample of channels (first, last, and some in between, at both ends of each
channel tile) and checks those outputs and their state columns.
"""
from __future__ import annotations

import pytest
import torch

import oracle
import causal_depthwise_conv1d_fwd_gb300 as ccv
from parity_util import assert_bits, assert_close

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
DEV = torch.device("cuda", 0)

T, DIM, W = 270_000, 8192, 4
CHANNELS = [0, 1, 7, 8, 255, 256, 4095, 4096, 8183, 8191]


def x_values(c: torch.Tensor, t: torch.Tensor) -> torch.Tensor:
    """x[c, t] as fp32: small values that vary along both axes."""
    v = ((c * 131 + t * 7) % 193).to(torch.float32) - 96.0
    return v * (1.0 / 1024.0)


def make_x(layout: str):
    t = torch.arange(T, device=DEV, dtype=torch.int64)
    if layout == "dim_tokens":
        x = torch.empty(DIM, T, dtype=torch.bfloat16, device=DEV)
        for c0 in range(0, DIM, 512):  # a slab at a time keeps temporaries small
            c = torch.arange(c0, c0 + 512, device=DEV, dtype=torch.int64)[:, None]
            x[c0:c0 + 512] = x_values(c, t[None, :]).to(torch.bfloat16)
        return x
    x = torch.empty(T, DIM, dtype=torch.bfloat16, device=DEV)
    c = torch.arange(DIM, device=DEV, dtype=torch.int64)[None, :]
    for t0 in range(0, T, 16384):
        tt = t[t0:t0 + 16384][:, None]
        x[t0:t0 + 16384] = x_values(c, tt).to(torch.bfloat16)
    return x.t()


@pytest.mark.parametrize("layout", ["tokens_dim", "dim_tokens"])
def test_beyond_2_pow_31_elements(layout):
    assert T * DIM > 2 ** 31
    g = torch.Generator().manual_seed(1009)
    weight = (torch.randn(DIM, W, generator=g) * 0.02).to(torch.bfloat16)
    bias = (torch.randn(DIM, generator=g) * 0.02).to(torch.bfloat16)
    states = (torch.randn(1, W - 1, DIM, generator=g) * 0.02).to(torch.bfloat16).transpose(1, 2)
    qsl = torch.tensor([0, T], dtype=torch.int32)
    has_init = torch.ones(1, dtype=torch.bool)

    x = make_x(layout)
    out = torch.empty_strided(x.shape, x.stride(), dtype=torch.bfloat16, device=DEV)
    d_states = torch.empty_strided(states.shape, states.stride(), dtype=torch.bfloat16,
                                   device=DEV).copy_(states)
    ccv.ccv_fwd(x, weight.to(DEV), bias.to(DEV), d_states, qsl.to(DEV), None,
                has_init.to(DEV), "silu", out=out)
    torch.cuda.synchronize()

    cs = torch.tensor(CHANNELS, dtype=torch.int64)
    xs = x_values(cs[:, None], torch.arange(T, dtype=torch.int64)[None, :]).to(torch.bfloat16)
    ref_states = states[:, CHANNELS].clone()
    ref_out, err = oracle.ccv_fwd(xs, weight[CHANNELS], bias[CHANNELS], ref_states, qsl, None,
                                  has_init, "silu")
    assert err == 0
    got = out[CHANNELS].cpu()
    assert_close(got, ref_out, f"{layout} sampled channels")
    assert_bits(d_states[:, CHANNELS].cpu(), ref_states, f"{layout} sampled state columns")
    del x, out
    torch.cuda.empty_cache()
