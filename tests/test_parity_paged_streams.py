"""GPU parity of paged_sconv_fwd_streams (several conv streams of a layer
sharing one paged cache, one launch) against the oracle.

Every stream's output within 1e-2*|ref| + 2e-5; the whole cache bit-exact;
the fused call equals one paged_sconv_fwd per stream bit for bit.
"""
from __future__ import annotations

import pytest
import torch

import oracle
import causal_depthwise_conv1d_fwd_gb300 as ccv
from causal_depthwise_conv1d_fwd_gb300 import workloads as wl
from parity_util import assert_bits, assert_close

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)

META = ("positions", "block_table", "seq_idx", "slot_mapping", "query_start")


def run_both(base, streams):
    ref_cache = base.cache.clone()
    ref_outs, _ = oracle.paged_sconv_fwd_streams(
        streams, ref_cache, base.positions, base.block_table, base.seq_idx, base.slot_mapping,
        base.query_start, base.block_size, base.activation, base.use_residual)
    cache = base.cache.to(DEV)
    dstreams = [{"x": st["x"].to(DEV), "weight": st["weight"].to(DEV), "off_s": st["off_s"],
                 "ws": st["ws"]} for st in streams]
    meta = {k: getattr(base, k).to(DEV) for k in META}
    outs = ccv.paged_sconv_fwd_streams(dstreams, cache, block_size=base.block_size,
                                       activation=base.activation,
                                       use_residual=base.use_residual, **meta)
    torch.cuda.synchronize()
    return ref_outs, ref_cache, outs, cache


def check(base, streams):
    ref_outs, ref_cache, outs, cache = run_both(base, streams)
    for i, (o, r) in enumerate(zip(outs, ref_outs)):
        assert_close(o, r, f"{base.name} stream {i} out")
    assert_bits(cache, ref_cache, f"{base.name} cache")


def test_config_four_streams_full_size():
    """A layer's K, V, attn-output and mlp-output streams: 3800 tokens each."""
    check(*wl.config_paged_streams())


@pytest.mark.parametrize("width", [2, 3, 4, 5])
def test_widths(width):
    base = wl.paged(5000 + width, [40, 1, 4, 77, 1], [0, 30, 2, 500, 9], H=4, ws=32, N=16,
                    D=160, num_blocks=128, off_s=0, width=width, interior_pad_frac=0.05,
                    pad_rows=3, pad_multiple=8)
    check(base, wl.paged_streams(base, 5100 + width, (0, 32, 96, 128), 32))


def test_streams_of_different_widths():
    """ws 32 for the base, 64 and 16 for the others: channel tiles differ per stream."""
    base = wl.paged(5201, [33, 1, 70], [5, 0, 300], H=4, ws=32, N=16, D=256, num_blocks=128,
                    off_s=0, width=4)
    g = torch.Generator().manual_seed(5202)
    T = base.x.shape[0]
    streams = [{"x": base.x, "weight": base.weight, "off_s": 0, "ws": 32}]
    for off, ws in ((64, 64), (200, 16)):
        streams.append({"x": (torch.randn(T, 4 * ws, generator=g) * 0.02).to(torch.bfloat16),
                        "weight": (torch.randn(4 * ws, 4, generator=g) * 0.02).to(torch.bfloat16),
                        "off_s": off, "ws": ws})
    check(base, streams)


def test_unaligned_stream_falls_back_per_stream():
    """A stream width that is not a multiple of 8 cannot use 16-byte vectors:
    the call runs stream by stream with the same results."""
    base = wl.paged(5301, [20, 1, 9], [0, 40, 3], H=2, ws=12, N=8, D=64, num_blocks=64,
                    off_s=0, width=4)
    streams = wl.paged_streams(base, 5302, (0, 16, 40), 12)
    check(base, streams)


def test_fused_equals_separate_calls():
    base, streams = wl.config_paged_streams(5401)
    meta = {k: getattr(base, k).to(DEV) for k in META}
    dstreams = [{"x": st["x"].to(DEV), "weight": st["weight"].to(DEV), "off_s": st["off_s"],
                 "ws": st["ws"]} for st in streams]
    cache_a = base.cache.to(DEV)
    outs_a = ccv.paged_sconv_fwd_streams(dstreams, cache_a, block_size=base.block_size,
                                         activation="silu", use_residual=True, **meta)
    cache_b = base.cache.to(DEV)
    outs_b = [ccv.paged_sconv_fwd(st["x"], st["weight"], cache_b, off_s=st["off_s"],
                                  ws=st["ws"], block_size=base.block_size, activation="silu",
                                  use_residual=True, **meta) for st in dstreams]
    torch.cuda.synchronize()
    for a, b in zip(outs_a, outs_b):
        assert_bits(a, b, "fused vs separate out")
    assert_bits(cache_a, cache_b, "fused vs separate cache")


def test_graph_replay_matches_eager():
    base, streams = wl.config_paged_streams(5501)
    meta = {k: getattr(base, k).to(DEV) for k in META}
    dstreams = [{"x": st["x"].to(DEV), "weight": st["weight"].to(DEV), "off_s": st["off_s"],
                 "ws": st["ws"]} for st in streams]
    cache = base.cache.to(DEV)
    launch = ccv.prepare_paged_sconv_fwd_streams(dstreams, cache, block_size=base.block_size,
                                                 activation="silu", use_residual=True, **meta)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        launch(s)
    torch.cuda.synchronize()
    eager = [o.clone() for o in launch.result]
    cache_eager = cache.clone()
    cache.copy_(base.cache.to(DEV))
    for o in launch.result:
        o.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        launch(s)
    g.replay()
    torch.cuda.synchronize()
    for o, e in zip(launch.result, eager):
        assert_bits(o, e, "graph out")
    assert_bits(cache, cache_eager, "graph cache")
