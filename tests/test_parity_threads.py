"""Several host threads call the library at once, each on its own CUDA stream
with its own buffers (the first calls fill the library's per-kernel caches
concurrently); every result must still match the oracle."""
from __future__ import annotations

import threading

import pytest
import torch

import oracle
import causal_depthwise_conv1d_fwd_gb300 as ccv
from causal_depthwise_conv1d_fwd_gb300 import workloads as wl
from parity_util import assert_bits, assert_close, sentinel_like, to_device

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


def test_concurrent_host_threads():
    cases = [wl.varlen_prefill(9000 + i, [300, 1, 77, 0, 1000], 264, 2 + i % 4, num_cache_lines=6,
                               layout=("tokens_dim", "dim_tokens")[i % 2], has_init="bernoulli",
                               name=f"thread_{i}") for i in range(8)]
    refs = []
    for c in cases:
        st = c.conv_states.clone()
        out = sentinel_like(c.x)
        oracle.ccv_fwd(c.x, c.weight, c.bias, st, c.query_start_loc, c.cache_indices,
                       c.has_initial_state, c.activation, c.pad_slot_id, out=out)
        refs.append((out, st))
    devs = [to_device(c.kwargs(), DEV) for c in cases]
    outs = [sentinel_like(d["x"]) for d in devs]
    errors = []
    barrier = threading.Barrier(len(cases))

    def work(i):
        try:
            s = torch.cuda.Stream(device=DEV)
            barrier.wait()
            with torch.cuda.stream(s):
                for _ in range(3):  # the state is written back each call: restore it first
                    devs[i]["conv_states"].copy_(cases[i].conv_states)
                    ccv.ccv_fwd(**devs[i], out=outs[i])
            s.synchronize()
        except Exception as e:  # surfaced below
            errors.append((i, e))

    threads = [threading.Thread(target=work, args=(i,)) for i in range(len(cases))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    torch.cuda.synchronize()
    for c, d, out, (ref_out, ref_st) in zip(cases, devs, outs, refs):
        assert_close(out, ref_out, c.name)
        assert_bits(d["conv_states"], ref_st, f"{c.name} states")
