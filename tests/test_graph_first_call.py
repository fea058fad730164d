"""Every entry point can be captured in a CUDA graph even as the first call
in a process (when the library still sets kernel attributes and computes
occupancy).  A fresh interpreter captures one call of each, replays the
graph, and compares with the same calls run eagerly afterwards."""
from __future__ import annotations

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r'''
import torch
import causal_depthwise_conv1d_fwd_gb300 as ccv
from causal_depthwise_conv1d_fwd_gb300 import workloads as wl

dev = torch.device("cuda", 0)
torch.cuda.set_device(dev)

def to_dev(c):
    return {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in c.kwargs().items()}

pre = [wl.varlen_prefill(1, [300, 2, 900], 512, 4, num_cache_lines=4, layout=l, has_init="all")
       for l in ("tokens_dim", "dim_tokens")]
dec = wl.decode(2, 64, 1024, 4)
spec = wl.spec_decode(3, 16, 1024, 4, 3, with_intermediate=True, with_output_indices=True)
pg = wl.paged(4, [40, 1, 9], [0, 33, 2], H=4, ws=32, N=16, D=128, num_blocks=64, off_s=32)
streams = wl.paged_streams(pg, 5, (0, 64), 32)
meta = ("positions", "block_table", "seq_idx", "slot_mapping", "query_start")

def fresh():
    st = {}
    st["pre"] = [to_dev(c) for c in pre]
    st["pre_out"] = [torch.empty_strided(d["x"].shape, d["x"].stride(), dtype=torch.bfloat16,
                                         device=dev) for d in st["pre"]]
    st["dec"] = to_dev(dec)
    st["spec"] = to_dev(spec)
    src = spec.intermediate_conv_window
    st["spec"]["intermediate_conv_window"] = torch.empty_strided(
        src.shape, src.stride(), dtype=src.dtype, device=dev).copy_(src)
    st["pg"] = to_dev(pg)
    st["pg_out"] = torch.empty_like(st["pg"]["x"])
    st["cache2"] = pg.cache.to(dev)
    st["meta"] = {k: getattr(pg, k).to(dev) for k in meta}
    st["streams"] = [{"x": s["x"].to(dev), "weight": s["weight"].to(dev), "off_s": s["off_s"],
                      "ws": s["ws"]} for s in streams]
    st["qsl"] = pg.query_start_loc.to(dev)
    st["seq"] = torch.zeros(pg.T, dtype=torch.int32, device=dev)
    st["qs"] = torch.zeros(pg.T, dtype=torch.int32, device=dev)
    st["pg3"] = {k: v for k, v in to_dev(pg).items() if k not in ("seq_idx", "query_start")}
    st["pg3_out"] = torch.empty_like(st["pg3"]["x"])
    st["seq3"] = torch.zeros(pg.T, dtype=torch.int32, device=dev)
    st["qs3"] = torch.zeros(pg.T, dtype=torch.int32, device=dev)
    return st

def run(st, s=None):
    for d, o in zip(st["pre"], st["pre_out"]):
        ccv.ccv_fwd(**d, out=o, stream=s)
    ccv.ccv_update(**st["dec"], stream=s)
    ccv.ccv_update_spec(**st["spec"], stream=s)
    ccv.paged_sconv_seq_metadata(st["qsl"], len(pg.req_lengths), pg.num_actual_tokens,
                                 st["seq"], st["qs"], pg.T, stream=s)
    ccv.paged_sconv_fwd(**st["pg"], out=st["pg_out"], stream=s)
    ccv.paged_sconv_fwd_with_metadata(query_start_loc=st["qsl"], num_reqs=len(pg.req_lengths),
                                      num_actual_tokens=pg.num_actual_tokens,
                                      seq_idx_out=st["seq3"], query_start_out=st["qs3"],
                                      out=st["pg3_out"], stream=s, **st["pg3"])
    return ccv.paged_sconv_fwd_streams(st["streams"], st["cache2"], block_size=pg.block_size,
                                       activation="silu", use_residual=True, stream=s,
                                       **st["meta"])

g_state = fresh()
s = torch.cuda.Stream()
g = torch.cuda.CUDAGraph()
with torch.cuda.graph(g, stream=s):
    g_outs = run(g_state, s)          # the very first calls of every kernel
g.replay()
torch.cuda.synchronize()

e_state = fresh()
e_outs = run(e_state)
torch.cuda.synchronize()

def same(a, b, what):
    if not torch.equal(a.view(torch.int16), b.view(torch.int16)):
        raise SystemExit(f"graph vs eager differ: {what}")

for i in range(2):
    same(g_state["pre_out"][i], e_state["pre_out"][i], f"prefill {i} out")
    same(g_state["pre"][i]["conv_states"], e_state["pre"][i]["conv_states"], f"prefill {i} states")
same(g_state["dec"]["x"], e_state["dec"]["x"], "decode out")
same(g_state["dec"]["conv_state"], e_state["dec"]["conv_state"], "decode state")
same(g_state["spec"]["x"], e_state["spec"]["x"], "spec out")
same(g_state["spec"]["conv_state"], e_state["spec"]["conv_state"], "spec pool")
same(g_state["spec"]["intermediate_conv_window"], e_state["spec"]["intermediate_conv_window"], "spec windows")
same(g_state["pg_out"], e_state["pg_out"], "paged out")
same(g_state["pg"]["cache"], e_state["pg"]["cache"], "paged cache")
same(g_state["pg3_out"], e_state["pg3_out"], "single-launch paged out")
same(g_state["pg3"]["cache"], e_state["pg3"]["cache"], "single-launch paged cache")
if not (torch.equal(g_state["seq3"], e_state["seq3"]) and torch.equal(g_state["qs3"], e_state["qs3"])):
    raise SystemExit("graph vs eager differ: single-launch metadata")
for i in range(2):
    same(g_outs[i], e_outs[i], f"stream {i} out")
same(g_state["cache2"], e_state["cache2"], "streams cache")
print("graph-first-call: ok")
'''


def test_every_entry_point_captures_as_first_call():
    proc = subprocess.run([sys.executable, "-c", SCRIPT], cwd=ROOT, capture_output=True,
                          text=True, timeout=600)
    assert proc.returncode == 0, proc.stdout[-2000:] + proc.stderr[-4000:]
    assert "graph-first-call: ok" in proc.stdout
