"""GPU parity of ccv_update_spec (speculative verify / decode with the
spec-decoding extras) against the CPU oracle.

Outputs within 1e-2*|ref| + 2e-5; the whole state pool and the whole
intermediate buffer bit-exact (entries the call must not write included);
invalid offsets and output lines counted.
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


def run_both(case):
    ref_pool = case.conv_state.clone()
    ref_inter = None if case.intermediate_conv_window is None else case.intermediate_conv_window.clone()
    x_cpu = case.x.clone()
    ref_out, ref_err = oracle.ccv_update_spec(
        x_cpu, ref_pool, case.weight, case.bias, case.activation, case.conv_state_indices,
        case.num_accepted_tokens, ref_inter, case.output_state_indices, case.pad_slot_id)
    d = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in case.kwargs().items()}
    if case.intermediate_conv_window is not None:
        # keep the generator's strides on the device
        src = case.intermediate_conv_window
        dev = torch.empty_strided(src.shape, src.stride(), dtype=src.dtype, device=DEV)
        dev.copy_(src)
        d["intermediate_conv_window"] = dev
    err_t = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = ccv.ccv_update_spec(**d, err_count=err_t)
    torch.cuda.synchronize()
    return (ref_out, ref_pool, ref_inter, ref_err), (out, d["conv_state"],
                                                      d["intermediate_conv_window"], int(err_t))


def check(case, expect_err=False):
    (ro, rp, ri, re), (go, gp, gi, ge) = run_both(case)
    assert_close(go, ro, f"{case.name} out")
    assert_bits(gp, rp, f"{case.name} conv_state pool")
    if ri is not None:
        assert_bits(gi, ri, f"{case.name} intermediate_conv_window")
    assert (ge > 0) == (re > 0) == expect_err, (ge, re)


def test_config_spec_verify_full_size():
    """64 rows x 4 drafts, dim 8192: every output, state line and window."""
    check(wl.config_spec_decode())


@pytest.mark.parametrize("width", [2, 3, 4, 5])
@pytest.mark.parametrize("extras", ["accepted", "intermediate", "output_lines", "all"])
def test_widths_and_extras(width, extras):
    case = wl.spec_decode(3000 + width, 23, 1032, width, 3, history=3,
                          with_accepted=extras in ("accepted", "all"),
                          with_intermediate=extras in ("intermediate", "all"),
                          with_output_indices=extras in ("output_lines", "all"),
                          steps=5, pad_positions=(4,), name=f"spec_w{width}_{extras}")
    check(case)


def test_intermediate_in_the_pages_contiguous_layout():
    """(batch, steps, dim, width-1) contiguous: window entries are not
    contiguous over channels, so the per-element store path runs."""
    case = wl.spec_decode(3101, 9, 256, 4, 4, with_intermediate=True)
    case.intermediate_conv_window = case.intermediate_conv_window.contiguous()
    check(case)


@pytest.mark.parametrize("dim", [1, 13, 100])
def test_odd_dims(dim):
    check(wl.spec_decode(3200 + dim, 7, dim, 4, 2, with_intermediate=True,
                         with_output_indices=True))


def test_no_bias_no_activation_single_token():
    check(wl.spec_decode(3301, 16, 512, 4, 1, use_bias=False, activation=None,
                         with_intermediate=True))


def test_without_extras_equals_ccv_update():
    case = wl.spec_decode(3401, 12, 1024, 4, 3, with_accepted=False, history=1)
    d = to_device(case.kwargs(), DEV)
    pool_a = d["conv_state"].clone()
    out_a = ccv.ccv_update_spec(d["x"].clone(), pool_a, d["weight"], d["bias"], "silu",
                                d["conv_state_indices"])
    pool_b = d["conv_state"].clone()
    out_b = ccv.ccv_update(d["x"].clone(), pool_b, d["weight"], d["bias"], "silu",
                           d["conv_state_indices"])
    torch.cuda.synchronize()
    assert_bits(out_a, out_b, "out")
    assert_bits(pool_a, pool_b, "pool")


def test_invalid_offsets_and_output_lines_are_counted():
    case = wl.spec_decode(3501, 6, 64, 4, 2, history=1, with_output_indices=True,
                          skip_frac=0.0)
    case.num_accepted_tokens[1] = 0
    case.num_accepted_tokens[2] = 3
    case.output_state_indices[4, 1] = case.conv_state.shape[0] + 5
    check(case, expect_err=True)


def test_graph_replay_matches_eager():
    case = wl.spec_decode(3601, 32, 2048, 4, 4, with_intermediate=True, with_output_indices=True)
    d = to_device(case.kwargs(), DEV)
    src = case.intermediate_conv_window
    inter = torch.empty_strided(src.shape, src.stride(), dtype=src.dtype, device=DEV)
    inter.copy_(src)
    x0, pool0, inter0 = d["x"].clone(), d["conv_state"].clone(), inter.clone()
    launch = ccv.prepare_ccv_update_spec(d["x"], d["conv_state"], d["weight"], d["bias"], "silu",
                                         d["conv_state_indices"], d["num_accepted_tokens"],
                                         inter, d["output_state_indices"])
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        launch(s)  # warm-up on the capture stream
    torch.cuda.synchronize()
    eager = (d["x"].clone(), d["conv_state"].clone(), inter.clone())
    d["x"].copy_(x0)
    d["conv_state"].copy_(pool0)
    inter.copy_(inter0)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        launch(s)
    g.replay()
    torch.cuda.synchronize()
    assert_bits(d["x"], eager[0], "out (in place)")
    assert_bits(d["conv_state"], eager[1], "pool")
    assert_bits(inter, eager[2], "intermediate")


def test_golden_spec_window_after_acceptance_on_gpu():
    """The page's rolling example (tests/golden/spec_rolling.txt) through the
    CUDA path: unit filters read the window at num_accepted_tokens = k back
    column by column, on 8 channels (the vector kernel)."""
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "spec_rolling.txt")
    rows = [ln for ln in open(path) if ln.strip() and not ln.startswith("#")]
    for row in rows:
        head, after_s, tail = [p.strip() for p in row.split("|")]
        M, N = (int(v) for v in head.split())
        W = M + 1
        k_s, window_s = [p.strip() for p in tail.split("->")]
        names = [f"h{i}" for i in range(1, M + 1)] + [f"d{j}" for j in range(1, N + 1)]
        code = {n: float(i + 1) for i, n in enumerate(names)}
        cols = [code[n] for n in after_s.split()]
        got = []
        for p in range(W - 1):
            state = torch.tensor(cols, dtype=torch.bfloat16, device=DEV).repeat(8, 1)
            state = state.t().contiguous().t().unsqueeze(0)   # (1, 8, L) channels contiguous
            weight = torch.zeros(8, W, dtype=torch.bfloat16, device=DEV)
            weight[:, p] = 1.0
            x = torch.zeros(1, 8, 1, dtype=torch.bfloat16, device=DEV)
            out = ccv.ccv_update_spec(x, state, weight, None, None, None,
                                      torch.tensor([int(k_s)], dtype=torch.int32, device=DEV))
            torch.cuda.synchronize()
            got.append(float(out[0, 0, 0]))
        assert got == [code[n] for n in window_s.split()], (row, got)
