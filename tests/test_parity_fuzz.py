"""Seeded random sweeps against the oracle: many small configurations per
entry point, drawn from every option the generators offer (lengths including
0 and 1, widths 2..5, both x layouts, both state layouts, wider states, pad
entries, has_initial_state patterns, bias and SiLU on or off, odd and vector
dims, paged request mixes and block sizes, spec-decode extras).  Each case
is checked like the hand-written ones: outputs within 1e-2*|ref| + 2e-5,
states, caches and windows bit-exact.
"""
from __future__ import annotations

import random

import pytest
import torch

import oracle
import causal_depthwise_conv1d_fwd_gb300 as ccv
from causal_depthwise_conv1d_fwd_gb300 import workloads as wl
from parity_util import assert_bits, assert_close, sentinel_like, to_device

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


@pytest.mark.parametrize("seed", range(120))
def test_fwd_random(seed, monkeypatch):
    # even seeds through the streaming prefill kernels, odd ones through the
    # short-problem kernels
    monkeypatch.setenv("CCV_PREFILL_PATH", "stream" if seed % 2 == 0 else "short")
    r = random.Random(7000 + seed)
    width = r.randint(2, 5)
    batch = r.randint(1, 6)
    lengths = [r.choice([0, 1, 2, 3, r.randint(1, 40), r.randint(100, 700)]) for _ in range(batch)]
    dim = r.choice([8, 16, 24, 40, 64, 136, 256, 264, 7, 13, 100])
    lines = batch + r.randint(0, 4)
    pads = tuple(i for i in range(batch) if r.random() < 0.2)
    case = wl.varlen_prefill(8000 + seed, lengths, dim, width, num_cache_lines=lines,
                             layout=r.choice(["tokens_dim", "dim_tokens"]),
                             state_layout=r.choice(["dim_contiguous", "tok_contiguous"]),
                             state_len=width - 1 + r.choice([0, 0, 1, 3]), pad_positions=pads,
                             has_init=r.choice(["bernoulli", "all", "none", "null"]),
                             use_bias=r.random() < 0.7,
                             activation=r.choice(["silu", None]),
                             with_cache_indices=r.random() < 0.8,
                             extra_tokens=r.choice([0, 0, 5]), name=f"fuzz_fwd_{seed}")
    ref_states = None if case.conv_states is None else case.conv_states.clone()
    ref_out = sentinel_like(case.x)
    oracle.ccv_fwd(case.x, case.weight, case.bias, ref_states, case.query_start_loc,
                   case.cache_indices, case.has_initial_state, case.activation,
                   case.pad_slot_id, out=ref_out)
    d = to_device(case.kwargs(), DEV)
    out = sentinel_like(d["x"])
    ccv.ccv_fwd(**d, out=out)
    torch.cuda.synchronize()
    assert_close(out, ref_out, case.name)
    if ref_states is not None:
        assert_bits(d["conv_states"], ref_states, f"{case.name} states")


@pytest.mark.parametrize("seed", range(60))
def test_decode_random(seed):
    """ccv_update without the spec extras: one or more tokens per row, both
    state layouts, wider states, PAD rows, no index vector, in place or into
    a separate out, bias and SiLU on or off, odd and vector dims."""
    r = random.Random(7300 + seed)
    width = r.randint(2, 5)
    batch = r.randint(1, 40)
    seqlen = r.choice([1, 1, 1, 2, 3])
    dim = r.choice([8, 16, 64, 1024, 1032, 13, 100, 8192])
    extra = r.choice([0, 0, 1, 3])
    with_indices = r.random() < 0.8
    case = wl.decode(9100 + seed, batch, dim, width, seqlen=seqlen,
                     state_len=width - 2 + seqlen + extra,
                     state_layout=r.choice(["dim_contiguous", "tok_contiguous"]),
                     pad_positions=(tuple(i for i in range(batch) if r.random() < 0.15)
                                    if with_indices else ()),
                     use_bias=r.random() < 0.7, activation=r.choice(["silu", None]),
                     with_indices=with_indices, squeeze=r.random() < 0.7,
                     name=f"fuzz_decode_{seed}")
    separate = r.random() < 0.3
    ref_state = case.conv_state.clone()
    ref_buf = torch.full_like(case.x, -3.0) if separate else None
    ref_out, _ = oracle.ccv_update(case.x.clone(), ref_state, case.weight, case.bias,
                                   case.activation, case.conv_state_indices, case.pad_slot_id,
                                   out=ref_buf)
    d = to_device(case.kwargs(), DEV)
    buf = torch.full_like(d["x"], -3.0) if separate else None
    out = ccv.ccv_update(**d, out=buf)
    torch.cuda.synchronize()
    assert_close(out, ref_out, case.name)
    assert_bits(d["conv_state"], ref_state, f"{case.name} conv_state")
    if separate:
        assert_bits(d["x"], case.x, f"{case.name} x unchanged")


@pytest.mark.parametrize("seed", range(80))
def test_update_random(seed):
    r = random.Random(7100 + seed)
    width = r.randint(2, 5)
    batch = r.randint(1, 12)
    seqlen = r.choice([1, 1, 2, 3, 5])
    dim = r.choice([8, 64, 1024, 1032, 13, 100])
    case = wl.spec_decode(8100 + seed, batch, dim, width, seqlen, history=r.randint(1, 4),
                          with_accepted=r.random() < 0.6,
                          with_intermediate=r.random() < 0.5,
                          with_output_indices=r.random() < 0.5,
                          steps=seqlen + r.choice([0, 2]),
                          pad_positions=tuple(i for i in range(batch) if r.random() < 0.15),
                          use_bias=r.random() < 0.7, activation=r.choice(["silu", None]),
                          name=f"fuzz_spec_{seed}")
    ref_pool = case.conv_state.clone()
    ref_inter = (None if case.intermediate_conv_window is None
                 else case.intermediate_conv_window.clone())
    ref_out, _ = oracle.ccv_update_spec(case.x.clone(), ref_pool, case.weight, case.bias,
                                        case.activation, case.conv_state_indices,
                                        case.num_accepted_tokens, ref_inter,
                                        case.output_state_indices, case.pad_slot_id)
    d = to_device(case.kwargs(), DEV)
    if ref_inter is not None:
        src = case.intermediate_conv_window
        d["intermediate_conv_window"] = torch.empty_strided(src.shape, src.stride(),
                                                            dtype=src.dtype, device=DEV).copy_(src)
    out = ccv.ccv_update_spec(**d)
    torch.cuda.synchronize()
    assert_close(out, ref_out, case.name)
    assert_bits(d["conv_state"], ref_pool, f"{case.name} pool")
    if ref_inter is not None:
        assert_bits(d["intermediate_conv_window"], ref_inter, f"{case.name} windows")


@pytest.mark.parametrize("seed", range(80))
def test_paged_random(seed):
    r = random.Random(7200 + seed)
    width = r.randint(2, 5)
    N = r.choice([4, 8, 16, 12])
    H = r.choice([1, 2, 4])
    ws = r.choice([8, 16, 32, 12])
    nreq = r.randint(1, 6)
    lengths = [r.choice([1, 1, 4, r.randint(2, 60)]) for _ in range(nreq)]
    starts = [r.choice([0, 1, 2, r.randint(0, 120)]) for _ in range(nreq)]
    D = r.choice([ws, ws + 16, 4 * ws])
    off_s = r.choice([0, D - ws, ((D - ws) // 8) * 8])
    case = wl.paged(8200 + seed, lengths, starts, H=H, ws=ws, N=N, D=D, num_blocks=256,
                    off_s=off_s, width=width, interior_pad_frac=r.choice([0.0, 0.1]),
                    pad_rows=r.choice([0, 3]), pad_multiple=r.choice([1, 8]),
                    activation=r.choice(["silu", None]), use_residual=r.random() < 0.6,
                    name=f"fuzz_paged_{seed}")
    ref_cache = case.cache.clone()
    ref_out, _ = oracle.paged_sconv_fwd(case.x, case.weight, ref_cache, case.positions,
                                        case.block_table, case.seq_idx, case.slot_mapping,
                                        case.query_start, case.off_s, case.ws, case.block_size,
                                        case.activation, case.use_residual)
    d = to_device(case.kwargs(), DEV)
    out = ccv.paged_sconv_fwd(**d)
    torch.cuda.synchronize()
    assert_close(out, ref_out, case.name)
    assert_bits(d["cache"], ref_cache, f"{case.name} cache")


@pytest.mark.parametrize("seed", range(40))
def test_paged_streams_random(seed):
    r = random.Random(7300 + seed)
    width = r.randint(2, 5)
    H = r.choice([1, 2, 4])
    N = r.choice([8, 16])
    nreq = r.randint(1, 5)
    lengths = [r.choice([1, 1, 4, r.randint(2, 50)]) for _ in range(nreq)]
    starts = [r.choice([0, 2, r.randint(0, 100)]) for _ in range(nreq)]
    # disjoint D-ranges of random widths, in a random order
    widths = [r.choice([8, 16, 24, 12]) for _ in range(r.randint(1, 4))]
    offs, pos = [], 0
    for w in widths:
        pos += r.choice([0, 8])
        offs.append(pos)
        pos += w
    D = pos + r.choice([0, 8])
    order = list(range(len(widths)))
    r.shuffle(order)
    base = wl.paged(8300 + seed, lengths, starts, H=H, ws=widths[0], N=N, D=D, num_blocks=128,
                    off_s=offs[0], width=width, interior_pad_frac=r.choice([0.0, 0.1]),
                    pad_rows=r.choice([0, 2]), pad_multiple=8,
                    activation=r.choice(["silu", None]), use_residual=r.random() < 0.6,
                    name=f"fuzz_streams_{seed}")
    g = torch.Generator().manual_seed(8400 + seed)
    T = base.x.shape[0]
    streams = []
    for i in order:
        ws = widths[i]
        x = base.x if i == 0 else (torch.randn(T, H * ws, generator=g) * 0.02).to(torch.bfloat16)
        w = (base.weight if i == 0 else
             (torch.randn(H * ws, width, generator=g) * 0.02).to(torch.bfloat16))
        streams.append({"x": x, "weight": w, "off_s": offs[i], "ws": ws})
    ref_cache = base.cache.clone()
    ref_outs, _ = oracle.paged_sconv_fwd_streams(
        streams, ref_cache, base.positions, base.block_table, base.seq_idx, base.slot_mapping,
        base.query_start, base.block_size, base.activation, base.use_residual)
    cache = base.cache.to(DEV)
    meta = {k: getattr(base, k).to(DEV) for k in
            ("positions", "block_table", "seq_idx", "slot_mapping", "query_start")}
    outs = ccv.paged_sconv_fwd_streams(
        [{"x": st["x"].to(DEV), "weight": st["weight"].to(DEV), "off_s": st["off_s"],
          "ws": st["ws"]} for st in streams], cache, block_size=base.block_size,
        activation=base.activation, use_residual=base.use_residual, **meta)
    torch.cuda.synchronize()
    for i, (o, ref) in enumerate(zip(outs, ref_outs)):
        assert_close(o, ref, f"{base.name} stream {i}")
    assert_bits(cache, ref_cache, f"{base.name} cache")


@pytest.mark.parametrize("seed", range(40))
def test_metadata_random(seed):
    r = random.Random(7400 + seed)
    num_reqs = r.randint(1, 40)
    lengths = [r.choice([0, 1, 1, 4, r.randint(1, 300)]) for _ in range(num_reqs)]
    qsl = torch.tensor([0] + list(torch.tensor(lengths).cumsum(0)), dtype=torch.int32)
    actual = int(qsl[-1])
    padded = actual + r.choice([0, 1, 7, 64])
    cap = padded + r.choice([0, 5])
    ref_seq = torch.full((cap,), 77, dtype=torch.int32)
    ref_qs = ref_seq.clone()
    oracle.paged_sconv_seq_metadata(qsl, num_reqs, actual, ref_seq, ref_qs, padded)
    seq = torch.full((cap,), 77, dtype=torch.int32, device=DEV)
    qs = seq.clone()
    ccv.paged_sconv_seq_metadata(qsl.to(DEV), num_reqs, actual, seq, qs, padded)
    torch.cuda.synchronize()
    assert_bits(seq.cpu(), ref_seq, "seq_idx")
    assert_bits(qs.cpu(), ref_qs, "query_start")
