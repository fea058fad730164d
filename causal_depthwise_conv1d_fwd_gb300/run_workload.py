"""Run one entry point on one of the named benchmark workloads a few times.

Used to give a profiler a small, self-contained program:

    python -m causal_depthwise_conv1d_fwd_gb300.run_workload --part prefill_tokens_dim --reps 3

Parts: prefill_tokens_dim, prefill_dim_tokens (4 x 4096 tokens, dim 8192),
decode (256 x 8192; prefill parts take --width), paged (H16 x ws128, 32 requests; metadata + conv),
spec (speculative verify, 64 rows x 4 drafts, dim 8192), atrex (one
channel-first sequence of --tokens x --dim, the atrex-bench #003 shapes),
paged_streams (a layer's four conv streams on one paged cache, one launch),
varlen (8 sequences of 1..512 tokens, dim 4096, channel-last), paged_single
(the paged workload as one paged_sconv_fwd_with_metadata launch), many (--batch
channel-first sequences of --tokens tokens each at --dim, all with initial state).
The process exits 0 after a device synchronize; it times nothing.
"""
from __future__ import annotations

import argparse

import torch

from . import api
from . import workloads as wl

PARTS = ("prefill_tokens_dim", "prefill_dim_tokens", "decode", "paged", "spec", "atrex",
         "paged_streams", "varlen", "paged_single", "many")


def _dev(kwargs, dev):
    return {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in kwargs.items()}


def make_launch(part: str, dev, tokens: int = 1024, dim: int = 4096, width: int = 4, batch: int = 64):
    if part.startswith("prefill"):
        layout = "tokens_dim" if part.endswith("tokens_dim") else "dim_tokens"
        c = wl.config_large_prefill(layout=layout)
        if width != 4:
            g = torch.Generator().manual_seed(1008)
            c.weight = (torch.randn(c.dim, width, generator=g) * 0.02).to(torch.bfloat16)
            if c.conv_states.shape[2] < width - 1:
                c.conv_states = wl.make_states(c.conv_states.shape[0], c.dim, width - 1,
                                               "dim_contiguous", g)
        d = _dev(c.kwargs(), dev)
        out = torch.empty_strided(d["x"].shape, d["x"].stride(), dtype=torch.bfloat16,
                                  device=dev)
        launch = api.prepare_ccv_fwd(**d, out=out)
        return lambda: launch()
    if part == "decode":
        launch = api.prepare_ccv_update(**_dev(wl.config_decode().kwargs(), dev))
        return lambda: launch()
    if part == "paged":
        c = wl.config_paged()
        d = _dev(c.kwargs(), dev)
        seq = torch.empty(c.T, dtype=torch.int32, device=dev)
        qs = torch.empty(c.T, dtype=torch.int32, device=dev)
        d["seq_idx"], d["query_start"] = seq, qs
        meta = api.prepare_paged_sconv_seq_metadata(c.query_start_loc.to(dev),
                                                    len(c.req_lengths), c.num_actual_tokens,
                                                    seq, qs, c.T)
        conv = api.prepare_paged_sconv_fwd(**d)

        def run():
            meta()
            conv()
        return run
    if part == "paged_single":
        c = wl.config_paged()
        d = {k: v for k, v in _dev(c.kwargs(), dev).items() if k not in ("seq_idx", "query_start")}
        seq = torch.empty(c.T, dtype=torch.int32, device=dev)
        qs = torch.empty(c.T, dtype=torch.int32, device=dev)
        launch = api.prepare_paged_sconv_fwd_with_metadata(
            query_start_loc=c.query_start_loc.to(dev), num_reqs=len(c.req_lengths),
            num_actual_tokens=c.num_actual_tokens, seq_idx_out=seq, query_start_out=qs, **d)
        return lambda: launch()
    if part == "spec":
        c = wl.config_spec_decode()
        d = _dev(c.kwargs(), dev)
        src = c.intermediate_conv_window
        inter = torch.empty_strided(src.shape, src.stride(), dtype=src.dtype, device=dev)
        inter.copy_(src)
        d["intermediate_conv_window"] = inter
        launch = api.prepare_ccv_update_spec(**d)
        return lambda: launch()
    if part == "atrex":
        d = _dev(wl.config_atrex(tokens, dim).kwargs(), dev)
        out = torch.empty_strided(d["x"].shape, d["x"].stride(), dtype=torch.bfloat16,
                                  device=dev)
        launch = api.prepare_ccv_fwd(**d, out=out)
        return lambda: launch()
    if part == "many":
        c = wl.varlen_prefill(1010, [tokens] * batch, dim, width, layout="dim_tokens",
                              has_init="all")
        d = _dev(c.kwargs(), dev)
        out = torch.empty_strided(d["x"].shape, d["x"].stride(), dtype=torch.bfloat16,
                                  device=dev)
        launch = api.prepare_ccv_fwd(**d, out=out)
        return lambda: launch()
    if part == "varlen":
        d = _dev(wl.config_varlen().kwargs(), dev)
        out = torch.empty_strided(d["x"].shape, d["x"].stride(), dtype=torch.bfloat16,
                                  device=dev)
        launch = api.prepare_ccv_fwd(**d, out=out)
        return lambda: launch()
    if part == "paged_streams":
        base, streams = wl.config_paged_streams()
        cache = base.cache.to(dev)
        meta = {k: getattr(base, k).to(dev) for k in
                ("positions", "block_table", "seq_idx", "slot_mapping", "query_start")}
        ds = [{"x": st["x"].to(dev), "weight": st["weight"].to(dev), "off_s": st["off_s"],
               "ws": st["ws"]} for st in streams]
        launch = api.prepare_paged_sconv_fwd_streams(ds, cache, block_size=base.block_size,
                                                     activation="silu", use_residual=True, **meta)
        return lambda: launch()
    raise ValueError(f"unknown part {part!r}; choose from {PARTS}")


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--part", choices=PARTS, required=True)
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--tokens", type=int, default=1024, help="atrex and many parts only")
    ap.add_argument("--dim", type=int, default=4096, help="atrex and many parts only")
    ap.add_argument("--batch", type=int, default=64, help="many part only")
    ap.add_argument("--width", type=int, default=4, help="prefill parts only: conv width 2..5")
    args = ap.parse_args(argv)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    run = make_launch(args.part, dev, args.tokens, args.dim, args.width, args.batch)
    for _ in range(args.reps):
        run()
    torch.cuda.synchronize()
    print(f"run_workload: {args.part} x{args.reps} ok")


if __name__ == "__main__":
    main()
