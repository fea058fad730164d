"""GPU parity of paged_sconv_seq_metadata and paged_sconv_fwd against the oracle.

Metadata exact; outputs within 1e-2*|ref| + 2e-5; the whole paged cache
bit-exact after the insert (every block, every D column, including other
streams' slices); repeated launches and graph replay deterministic.
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


def run_both(case, err=False):
    ref_cache = case.cache.clone()
    ref_out, _ = oracle.paged_sconv_fwd(case.x, case.weight, ref_cache, case.positions,
                                        case.block_table, case.seq_idx, case.slot_mapping,
                                        case.query_start, case.off_s, case.ws, case.block_size,
                                        case.activation, case.use_residual)
    d = to_device(case.kwargs(), DEV)
    err_t = torch.zeros(1, dtype=torch.int32, device=DEV) if err else None
    out = ccv.paged_sconv_fwd(**d, err_count=err_t)
    torch.cuda.synchronize()
    return ref_out, ref_cache, out, d["cache"], err_t


def check(case):
    ref_out, ref_cache, out, cache, _ = run_both(case)
    assert_close(out, ref_out, f"{case.name} out")
    assert_bits(cache, ref_cache, f"{case.name} cache")


def small(seed, lengths, starts, **kw):
    args = dict(H=4, ws=32, N=16, D=160, num_blocks=96, off_s=64, width=4)
    args.update(kw)
    return wl.paged(seed, lengths, starts, **args)


def test_config_paged_full_size():
    check(wl.config_paged())


def test_taps_past_the_block_table_are_clamped():
    """Cached taps whose logical block lies past the table read its last column."""
    check(wl.paged_past_table(161))


def test_config_paged_metadata_full_size():
    case = wl.config_paged()
    seq = torch.full((case.T + 8,), 77, dtype=torch.int32, device=DEV)
    qs = torch.full((case.T + 8,), 77, dtype=torch.int32, device=DEV)
    ccv.paged_sconv_seq_metadata(case.query_start_loc.to(DEV), len(case.req_lengths),
                                 case.num_actual_tokens, seq, qs, case.T)
    ref_seq = torch.full((case.T + 8,), 77, dtype=torch.int32)
    ref_qs = ref_seq.clone()
    oracle.paged_sconv_seq_metadata(case.query_start_loc, len(case.req_lengths),
                                    case.num_actual_tokens, ref_seq, ref_qs, case.T)
    torch.cuda.synchronize()
    assert_bits(seq, ref_seq, "seq_idx")
    assert_bits(qs, ref_qs, "query_start")
    assert_bits(seq[:case.T], case.seq_idx, "seq_idx vs construction")
    assert_bits(qs[:case.T], case.query_start, "query_start vs construction")


@pytest.mark.parametrize("width", [2, 3, 4, 5])
@pytest.mark.parametrize("silu,residual", [(True, True), (False, False), (True, False),
                                           (False, True)])
def test_widths_and_flags(width, silu, residual):
    check(small(3000 + width, [70, 1, 4, 1, 33, 2], [0, 40, 2, 300, 17, 1], width=width,
                interior_pad_frac=0.05, pad_rows=5, pad_multiple=8,
                activation="silu" if silu else None, use_residual=residual))


@pytest.mark.parametrize("ws,off_s", [(12, 4), (8, 3), (24, 8)])
def test_unaligned_streams_use_strided_kernel(ws, off_s):
    check(small(3100 + ws, [9, 1, 20], [5, 30, 0], H=3, ws=ws, D=40, off_s=off_s))


def test_single_token_and_tiny():
    check(small(3201, [1], [0]))
    check(small(3202, [1], [5]))
    check(small(3203, [3], [1], pad_rows=1))


def test_large_values():
    check(small(3301, [30, 1, 4], [3, 50, 0], std=20.0))


def test_invalid_block_counted_not_faulting():
    case = small(3401, [5, 1], [20, 40])
    case.block_table[1, :] = 100000
    ref_out, ref_cache, out, cache, err = run_both(case, err=True)
    assert int(err.item()) > 0
    assert_close(out, ref_out, "invalid out")
    assert_bits(cache, ref_cache, "invalid cache")


def test_zero_tokens():
    case = small(3501, [1], [0])
    d = to_device(case.kwargs(), DEV)
    for k in ("x", "positions", "seq_idx", "slot_mapping", "query_start"):
        d[k] = d[k][:0]
    out = ccv.paged_sconv_fwd(**d)
    assert out.shape[0] == 0


def test_rejects_bad_stream_range():
    case = small(3601, [3], [0])
    d = to_device(case.kwargs(), DEV)
    d["off_s"] = 140  # 140 + 32 > D = 160
    with pytest.raises(ccv.CcvError):
        ccv.paged_sconv_fwd(**d)


def test_repeat_launches_are_deterministic():
    case = small(3701, [200, 1, 4, 1, 90], [7, 300, 0, 2, 120])
    d = to_device(case.kwargs(), DEV)
    cache0 = d["cache"].clone()
    outs = []
    for _ in range(3):
        d["cache"].copy_(cache0)
        outs.append(ccv.paged_sconv_fwd(**d).clone())
    torch.cuda.synchronize()
    assert_bits(outs[1], outs[0], "repeat 1")
    assert_bits(outs[2], outs[0], "repeat 2")


def test_graph_replay_matches_eager():
    """Capture metadata + conv once; replay it; same as the oracle."""
    case = small(3801, [40, 1, 4, 1], [2, 60, 0, 9], pad_rows=4, pad_multiple=8)
    d = to_device(case.kwargs(), DEV)
    qsl = case.query_start_loc.to(DEV)
    n_req = len(case.req_lengths)
    seq = torch.zeros(case.T, dtype=torch.int32, device=DEV)
    qs = torch.zeros(case.T, dtype=torch.int32, device=DEV)
    d["seq_idx"], d["query_start"] = seq, qs
    out = torch.empty_like(d["x"])
    cache0 = d["cache"].clone()

    def step():
        ccv.paged_sconv_seq_metadata(qsl, n_req, case.num_actual_tokens, seq, qs, case.T)
        ccv.paged_sconv_fwd(**d, out=out)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    d["cache"].copy_(cache0)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    ref_cache = case.cache.clone()
    ref_out, _ = oracle.paged_sconv_fwd(case.x, case.weight, ref_cache, case.positions,
                                        case.block_table, case.seq_idx, case.slot_mapping,
                                        case.query_start, case.off_s, case.ws, case.block_size,
                                        case.activation, case.use_residual)
    assert_close(out, ref_out, "graph out")
    assert_bits(d["cache"], ref_cache, "graph cache")
