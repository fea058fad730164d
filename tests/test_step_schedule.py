"""The step's parts under the schedules the bench times them in.

The step runs a streaming-size prefill in both layouts, a short varlen
prefill, the paged conv (metadata, then conv) and a decode update.  They
share no buffer, so the order of the launches and the stream each runs on
change nothing: one stream in step order, one stream in the reverse order
and two streams at once (prefill on one; paged and decode on the other) must
give bit-identical outputs, conv states and cache.  The two-stream run is
also compared with the oracle, part by part.
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


def _cases():
    # 4 x 1100 tokens at dim 2048 is above 2^23 elements: the streaming kernels.
    big = [1100, 1100, 1100, 1100]
    return {
        "prefill_tokens_dim": wl.varlen_prefill(3101, big, 2048, layout="tokens_dim", has_init="all"),
        "prefill_dim_tokens": wl.varlen_prefill(3102, big, 2048, layout="dim_tokens", has_init="all"),
        "varlen": wl.config_varlen(3103),
        "paged": wl.paged(3104, [300, 1, 1, 4, 1, 57], [0, 40, 17, 200, 3, 999], H=4, ws=64, N=16,
                          D=256, num_blocks=160, off_s=64, width=4, interior_pad_frac=0.02,
                          pad_rows=5, pad_multiple=8),
        "decode": wl.decode(3105, 96, 2048),
    }


class Step:
    """Device copies of every part's inputs, reset from the host cases before
    each schedule, and each part's launch on a given stream."""

    def __init__(self, cases):
        self.cases = cases
        self.dev = {}
        self.outs = {}
        for name, c in cases.items():
            self.dev[name] = to_device(c.kwargs(), DEV)
        for name in ("prefill_tokens_dim", "prefill_dim_tokens", "varlen"):
            x = self.dev[name]["x"]
            self.outs[name] = torch.empty_strided(x.shape, x.stride(), dtype=x.dtype, device=DEV)
        p = cases["paged"]
        self.outs["paged"] = torch.empty_like(self.dev["paged"]["x"])
        self.seq = torch.empty(p.T, dtype=torch.int32, device=DEV)
        self.qs = torch.empty(p.T, dtype=torch.int32, device=DEV)
        self.qsl = p.query_start_loc.to(DEV)

    def reset(self):
        for name, c in self.cases.items():
            for k, v in c.kwargs().items():
                if isinstance(v, torch.Tensor):
                    self.dev[name][k].copy_(v)
        for o in self.outs.values():
            o.zero_()

    def run(self, name, stream):
        with torch.cuda.stream(stream):
            if name == "decode":
                ccv.ccv_update(**self.dev[name])
            elif name == "paged":
                p = self.cases["paged"]
                d = {k: v for k, v in self.dev[name].items() if k not in ("seq_idx", "query_start")}
                ccv.paged_sconv_seq_metadata(self.qsl, len(p.req_lengths), p.num_actual_tokens,
                                             self.seq, self.qs, p.T)
                ccv.paged_sconv_fwd(**d, seq_idx=self.seq, query_start=self.qs,
                                    out=self.outs[name])
            else:
                ccv.ccv_fwd(**self.dev[name], out=self.outs[name])

    def snapshot(self):
        torch.cuda.synchronize()
        snap = {f"out/{k}": v.clone() for k, v in self.outs.items()}
        for name in ("prefill_tokens_dim", "prefill_dim_tokens", "varlen"):
            snap[f"states/{name}"] = self.dev[name]["conv_states"].clone()
        snap["decode/x"] = self.dev["decode"]["x"].clone()
        snap["decode/state"] = self.dev["decode"]["conv_state"].clone()
        snap["paged/cache"] = self.dev["paged"]["cache"].clone()
        return snap


ORDER = ["prefill_tokens_dim", "prefill_dim_tokens", "varlen", "paged", "decode"]


def _sequential(step, order):
    step.reset()
    s = torch.cuda.current_stream()
    for name in order:
        step.run(name, s)
    return step.snapshot()


def _two_streams(step):
    step.reset()
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    side.wait_stream(main)
    for name in ORDER:
        step.run(name, main if name.startswith(("prefill", "varlen")) else side)
    main.wait_stream(side)
    return step.snapshot()


def test_schedules_agree_bit_for_bit():
    step = Step(_cases())
    ref = _sequential(step, ORDER)
    for what, got in (("reverse order", _sequential(step, ORDER[::-1])),
                      ("two streams", _two_streams(step))):
        for k in ref:
            assert_bits(got[k], ref[k], f"{what}: {k}")


def test_two_streams_match_the_oracle():
    cases = _cases()
    step = Step(cases)
    got = _two_streams(step)
    for name in ("prefill_tokens_dim", "prefill_dim_tokens", "varlen"):
        c = cases[name]
        states = c.conv_states.clone()
        ref_out = torch.zeros_like(c.x)  # rows of a PAD sequence stay as the GPU run left them: 0
        oracle.ccv_fwd(c.x, c.weight, c.bias, states, c.query_start_loc, c.cache_indices,
                       c.has_initial_state, c.activation, out=ref_out)
        assert_close(got[f"out/{name}"], ref_out, f"{name} out")
        assert_bits(got[f"states/{name}"], states, f"{name} states")
    d = cases["decode"]
    state = d.conv_state.clone()
    ref_out, _ = oracle.ccv_update(d.x.clone(), state, d.weight, d.bias, d.activation,
                                   d.conv_state_indices)
    assert_close(got["decode/x"], ref_out, "decode out")
    assert_bits(got["decode/state"], state, "decode state")
    p = cases["paged"]
    cache = p.cache.clone()
    ref_out, _ = oracle.paged_sconv_fwd(p.x, p.weight, cache, p.positions, p.block_table,
                                        p.seq_idx, p.slot_mapping, p.query_start, p.off_s, p.ws,
                                        p.block_size, p.activation, p.use_residual)
    assert_close(got["out/paged"], ref_out, "paged out")
    assert_bits(got["paged/cache"], cache, "paged cache")
