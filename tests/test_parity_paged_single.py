"""GPU parity of paged_sconv_fwd_with_metadata: the paged conv in one launch
that resolves each token's request and first x-row from query_start_loc.

Against the oracle's metadata followed by its paged conv: outputs within
1e-2*|ref| + 2e-5, the whole cache and the written metadata bit-exact.
Against the two-call GPU path (paged_sconv_seq_metadata, then
paged_sconv_fwd): outputs, cache and error count bit-identical.  Covers the
shuffle search (up to 32 requests), the per-lane search (more), zero-length
requests, trailing padded rows, a forward with no real token, graph replay
and a seeded sweep.
"""
from __future__ import annotations

import random

import pytest
import torch

import oracle
import causal_depthwise_conv1d_fwd_gb300 as ccv
from causal_depthwise_conv1d_fwd_gb300 import workloads as wl
from parity_util import assert_bits, assert_close, to_device

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


def _oracle(case):
    """The oracle's metadata, then its paged conv on a copy of the cache."""
    n_req = len(case.req_lengths)
    seq = torch.full((case.T,), 77, dtype=torch.int32)
    qs = torch.full((case.T,), 77, dtype=torch.int32)
    oracle.paged_sconv_seq_metadata(case.query_start_loc, n_req, case.num_actual_tokens, seq,
                                    qs, case.T)
    cache = case.cache.clone()
    out, _ = oracle.paged_sconv_fwd(case.x, case.weight, cache, case.positions,
                                    case.block_table, seq, case.slot_mapping, qs, case.off_s,
                                    case.ws, case.block_size, case.activation,
                                    case.use_residual)
    return out, cache, seq, qs


def _single(case, with_meta_out=True, err=False):
    d = to_device(case.kwargs(), DEV)
    for k in ("seq_idx", "query_start"):
        d.pop(k)
    seq = torch.full((case.T,), 77, dtype=torch.int32, device=DEV) if with_meta_out else None
    qs = torch.full((case.T,), 77, dtype=torch.int32, device=DEV) if with_meta_out else None
    err_t = torch.zeros(1, dtype=torch.int32, device=DEV) if err else None
    out = ccv.paged_sconv_fwd_with_metadata(
        query_start_loc=case.query_start_loc.to(DEV), num_reqs=len(case.req_lengths),
        num_actual_tokens=case.num_actual_tokens, seq_idx_out=seq, query_start_out=qs,
        err_count=err_t, **d)
    torch.cuda.synchronize()
    return out, d["cache"], seq, qs, err_t


def _two_calls(case, err=False):
    d = to_device(case.kwargs(), DEV)
    seq = torch.empty(case.T, dtype=torch.int32, device=DEV)
    qs = torch.empty(case.T, dtype=torch.int32, device=DEV)
    ccv.paged_sconv_seq_metadata(case.query_start_loc.to(DEV), len(case.req_lengths),
                                 case.num_actual_tokens, seq, qs, case.T)
    d["seq_idx"], d["query_start"] = seq, qs
    err_t = torch.zeros(1, dtype=torch.int32, device=DEV) if err else None
    out = ccv.paged_sconv_fwd(**d, err_count=err_t)
    torch.cuda.synchronize()
    return out, d["cache"], err_t


def check(case):
    ref_out, ref_cache, ref_seq, ref_qs = _oracle(case)
    out, cache, seq, qs, err = _single(case, err=True)
    assert_close(out, ref_out, f"{case.name} out")
    assert_bits(cache, ref_cache, f"{case.name} cache")
    assert_bits(seq, ref_seq, f"{case.name} seq_idx")
    assert_bits(qs, ref_qs, f"{case.name} query_start")
    out2, cache2, err2 = _two_calls(case, err=True)
    assert_bits(out, out2, f"{case.name} single launch == two calls (out)")
    assert_bits(cache, cache2, f"{case.name} single launch == two calls (cache)")
    assert int(err.item()) == int(err2.item())


def small(seed, lengths, starts, **kw):
    args = dict(H=4, ws=32, N=16, D=160, num_blocks=128, off_s=64, width=4)
    args.update(kw)
    return wl.paged(seed, lengths, starts, **args)


def test_config_paged_full_size():
    """The bench's paged workload (32 requests: the shuffle search)."""
    check(wl.config_paged())


def test_more_than_32_requests_search_per_lane():
    lengths = [1, 4, 1, 37, 2, 1, 1, 9, 4, 1] * 5
    starts = [(13 * i) % 90 for i in range(len(lengths))]
    check(small(3101, lengths, starts, pad_rows=5, pad_multiple=8))


@pytest.mark.parametrize("width", [2, 3, 4, 5])
def test_widths_with_padded_rows(width):
    check(small(3110 + width, [5, 1, 4, 60, 1], [0, 7, 2, 33, 1], width=width,
                interior_pad_frac=0.1, pad_rows=3, pad_multiple=8))


def test_exactly_32_requests_and_33():
    for n in (32, 33):
        lengths = [(i % 5) + 1 for i in range(n)]
        starts = [(7 * i) % 50 for i in range(n)]
        check(small(3120 + n, lengths, starts, pad_rows=2))


def test_no_metadata_outputs():
    case = small(3130, [3, 50, 1], [2, 0, 40], pad_rows=4)
    ref_out, ref_cache, _, _ = _oracle(case)
    out, cache, _, _, _ = _single(case, with_meta_out=False)
    assert_close(out, ref_out, "no metadata outputs")
    assert_bits(cache, ref_cache, "no metadata outputs cache")


def test_forward_with_only_padded_rows():
    """num_actual_tokens = 0: every row is a padded row (out = residual or 0),
    nothing is inserted, the metadata is all zero."""
    case = small(3140, [4, 2], [0, 3], pad_rows=6)
    case.num_actual_tokens = 0
    case.slot_mapping.fill_(-1)
    check(case)


def test_rejects_inconsistent_sizes():
    case = small(3150, [4], [0])
    d = to_device(case.kwargs(), DEV)
    for k in ("seq_idx", "query_start"):
        d.pop(k)
    with pytest.raises(ccv.CcvError):  # more real tokens than rows
        ccv.paged_sconv_fwd_with_metadata(query_start_loc=case.query_start_loc.to(DEV),
                                          num_reqs=1, num_actual_tokens=case.T + 1, **d)


def test_graph_replay_matches_eager():
    case = wl.config_paged()
    d = to_device(case.kwargs(), DEV)
    for k in ("seq_idx", "query_start"):
        d.pop(k)
    qsl = case.query_start_loc.to(DEV)
    cache0 = d["cache"].clone()
    launch = ccv.prepare_paged_sconv_fwd_with_metadata(
        query_start_loc=qsl, num_reqs=len(case.req_lengths),
        num_actual_tokens=case.num_actual_tokens, **d)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        eager = launch(s.cuda_stream).clone()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    eager_cache = d["cache"].clone()
    d["cache"].copy_(cache0)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        launch(torch.cuda.current_stream().cuda_stream)
    d["cache"].copy_(cache0)
    g.replay()
    torch.cuda.synchronize()
    assert_bits(launch.result, eager, "graph out")
    assert_bits(d["cache"], eager_cache, "graph cache")


@pytest.mark.parametrize("seed", range(30))
def test_random(seed):
    r = random.Random(7600 + seed)
    width = r.randint(2, 5)
    N = r.choice([8, 16])
    H = r.choice([1, 2, 4])
    ws = r.choice([8, 16, 32, 12])
    nreq = r.choice([1, 3, 6, 31, 32, 33, 45])
    lengths = [r.choice([0, 1, 1, 4, r.randint(2, 40)]) for _ in range(nreq)]
    if sum(lengths) == 0:
        lengths[0] = 1
    starts = [r.choice([0, 1, 2, r.randint(0, 120)]) for _ in range(nreq)]
    D = r.choice([ws, ws + 16, 4 * ws])
    off_s = r.choice([0, D - ws, ((D - ws) // 8) * 8])
    case = wl.paged(8600 + seed, lengths, starts, H=H, ws=ws, N=N, D=D, num_blocks=512,
                    off_s=off_s, width=width, interior_pad_frac=r.choice([0.0, 0.1]),
                    pad_rows=r.choice([0, 3]), pad_multiple=r.choice([1, 8]),
                    activation=r.choice(["silu", None]), use_residual=r.random() < 0.6,
                    name=f"fuzz_single_{seed}")
    check(case)
