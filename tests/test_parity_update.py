"""GPU parity of ccv_update (decode) against the CPU oracle.

Outputs within 1e-2*|ref| + 2e-5; the conv_state pool bit-exact (every line,
including untouched ones); pad rows untouched; graph replay equals eager.
"""
from __future__ import annotations

import pytest
import torch

import oracle
import causal_depthwise_conv1d_fwd_gb300 as ccv
from causal_depthwise_conv1d_fwd_gb300 import workloads as wl
from parity_util import assert_bits, assert_close, to_device

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


def run_both(case, separate_out=False, err=False):
    ref_state = case.conv_state.clone()
    x_cpu = case.x.clone()
    ref_out_buf = torch.full_like(case.x, -3.0) if separate_out else None
    ref_out, _ = oracle.ccv_update(x_cpu, ref_state, case.weight, case.bias, case.activation,
                                   case.conv_state_indices, case.pad_slot_id, out=ref_out_buf)
    d = to_device(case.kwargs(), DEV)
    out_buf = torch.full_like(d["x"], -3.0) if separate_out else None
    err_t = torch.zeros(1, dtype=torch.int32, device=DEV) if err else None
    out = ccv.ccv_update(**d, out=out_buf, err_count=err_t)
    torch.cuda.synchronize()
    return ref_out, ref_state, out, d["conv_state"], d["x"], x_cpu, err_t


def check(case, separate_out=False):
    ref_out, ref_state, out, state, x_dev, x_cpu, _ = run_both(case, separate_out)
    assert_close(out, ref_out, f"{case.name} out")
    assert_bits(state, ref_state, f"{case.name} conv_state")
    if separate_out:
        assert_bits(x_dev, case.x, f"{case.name} x must be unchanged")


def test_config_decode_full_size():
    check(wl.config_decode())


@pytest.mark.parametrize("width", [2, 3, 4, 5])
@pytest.mark.parametrize("state_layout", ["dim_contiguous", "tok_contiguous"])
def test_widths_and_state_layouts(width, state_layout):
    check(wl.decode(2000 + width, 37, 2056, width, num_lines=80, state_layout=state_layout,
                    pad_positions=(0, 5)))


@pytest.mark.parametrize("dim", [1, 13, 100, 1000, 1032])
def test_dims(dim):
    check(wl.decode(2100 + dim, 9, dim, 4, num_lines=11, pad_positions=(3,)))


def test_separate_out_and_no_indices():
    check(wl.decode(2201, 16, 512, 4, num_lines=16, with_indices=False), separate_out=True)
    check(wl.decode(2202, 16, 512, 4, num_lines=20, use_bias=False, activation=None),
          separate_out=True)


@pytest.mark.parametrize("seqlen", [2, 3, 5])
@pytest.mark.parametrize("width", [2, 4])
def test_multi_token_keeps_history(seqlen, width):
    """seqlen > 1: the state holds W-2+seqlen columns after the call."""
    check(wl.decode(2300 + seqlen, 10, 256, width, num_lines=12, seqlen=seqlen, squeeze=False))
    check(wl.decode(2310 + seqlen, 10, 256, width, num_lines=12, seqlen=seqlen, squeeze=False,
                    state_layout="tok_contiguous"), separate_out=True)


def test_state_too_narrow_is_rejected():
    case = wl.decode(2401, 4, 64, 4, num_lines=4, seqlen=3, state_len=3, squeeze=False)
    d = to_device(case.kwargs(), DEV)
    with pytest.raises(ccv.CcvError):
        ccv.ccv_update(**d)


def test_invalid_line_counted_not_faulting():
    case = wl.decode(2501, 6, 128, 4, num_lines=8)
    case.conv_state_indices[2] = 8  # one past the pool
    ref_out, ref_state, out, state, x_dev, x_cpu, err = run_both(case, err=True)
    assert int(err.item()) > 0
    assert_close(out, ref_out, "invalid out")
    assert_bits(state, ref_state, "invalid state")


def test_graph_replay_matches_eager():
    c1 = wl.config_decode(2601)
    c2 = wl.config_decode(2602)
    d = to_device(c1.kwargs(), DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        ccv.ccv_update(**d)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ccv.ccv_update(**d)
    d2 = to_device(c2.kwargs(), DEV)
    for k in ("x", "weight", "bias", "conv_state", "conv_state_indices"):
        d[k].copy_(d2[k])
    for step in range(3):  # replay three decode steps, oracle alongside
        x_next = torch.randn(c2.x.shape, generator=torch.Generator().manual_seed(step)) * 0.02
        x_next = x_next.to(torch.bfloat16)
        c2.x.copy_(x_next)
        d["x"].copy_(x_next.to(DEV))
        g.replay()
        oracle.ccv_update(c2.x, c2.conv_state, c2.weight, c2.bias, c2.activation,
                          c2.conv_state_indices, -1)
        torch.cuda.synchronize()
        assert_close(d["x"], c2.x, f"graph step {step} out")
        assert_bits(d["conv_state"], c2.conv_state, f"graph step {step} state")
