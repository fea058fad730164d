"""GPU parity of ccv_fwd (varlen prefill) against the CPU oracle, through
both kernel families (forced by CCV_PREFILL_PATH) and through the automatic
choice on both sides of its size threshold.

Outputs within 1e-2*|ref| + 2e-5, conv_state bit-exact, untouched regions
(pad sequences, zero-length sequences, wider state columns, guard bands)
bit-exact.  Sizes span several chunks and ragged tails of both kernels
(channel-last chunks of 256 tokens; channel-first chunks of 32632 tokens for
aligned rows and 256 for the strided fallback).
"""
from __future__ import annotations

import os

import pytest
import torch

import oracle
import causal_depthwise_conv1d_fwd_gb300 as ccv
from causal_depthwise_conv1d_fwd_gb300 import workloads as wl
from parity_util import assert_bits, assert_close, sentinel_like, to_device
from test_kernel_tiling import K as TILING

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


@pytest.fixture(params=["short", "stream"], autouse=True)
def prefill_path(request, monkeypatch):
    """Every case runs through both prefill kernel families: the short-problem
    kernels (a warp per short chunk, inputs straight into registers) and the
    streaming ones (block chunks through shared-memory rings)."""
    monkeypatch.setenv("CCV_PREFILL_PATH", request.param)
    return request.param


def run_both(case, out_cpu=None, out_dev=None, err=False):
    """Run the oracle and the GPU on the same inputs; return both results."""
    ref_states = None if case.conv_states is None else case.conv_states.clone()
    ref_out = sentinel_like(case.x) if out_cpu is None else out_cpu
    oracle.ccv_fwd(case.x, case.weight, case.bias, ref_states, case.query_start_loc,
                   case.cache_indices, case.has_initial_state, case.activation,
                   case.pad_slot_id, out=ref_out)
    d = to_device(case.kwargs(), DEV)
    out = sentinel_like(d["x"]) if out_dev is None else out_dev
    err_t = torch.zeros(1, dtype=torch.int32, device=DEV) if err else None
    ccv.ccv_fwd(**d, out=out, err_count=err_t)
    torch.cuda.synchronize()
    return ref_out, ref_states, out, d["conv_states"], err_t


def check(case, **kw):
    ref_out, ref_states, out, states, _ = run_both(case, **kw)
    assert_close(out, ref_out, f"{case.name} out")
    assert_bits(out.isnan(), ref_out.isnan(), f"{case.name} nan pattern")
    if ref_states is not None:
        assert_bits(states, ref_states, f"{case.name} conv_states")


# ------------------------------------------------------------ the configs ----

def test_config_single_sequence():
    check(wl.config_single())


@pytest.mark.parametrize("layout", ["tokens_dim", "dim_tokens"])
def test_config_varlen_batch(layout):
    check(wl.config_varlen(layout=layout))


@pytest.mark.parametrize("layout", ["tokens_dim", "dim_tokens"])
def test_config_large_prefill_full_size(layout):
    """4 x 4096 tokens, dim 8192: every output element, as the bench launches it."""
    check(wl.config_large_prefill(layout=layout))


@pytest.mark.parametrize("tokens,dim", wl.ATREX_SHAPES)
def test_atrex_bench_shapes(tokens, dim):
    """The nine shapes of the atrex-bench #003 table: one channel-first
    sequence with initial state, bias and SiLU."""
    check(wl.config_atrex(tokens, dim))


# ------------------------------------------------------------- edge cases ----

def _bf16_sweep(lo: float, hi: float) -> torch.Tensor:
    """Every finite bf16 value in [lo, hi], as a 1-D bf16 tensor."""
    bits = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16)
    vals = bits.view(torch.bfloat16)
    f = vals.float()
    return vals[torch.isfinite(f) & (f >= lo) & (f <= hi)]


@pytest.mark.parametrize("layout", ["tokens_dim", "dim_tokens"])
def test_silu_over_every_bf16_value(layout):
    """A delta filter (last tap 1, no bias, zero prior) makes out = silu(x):
    x runs through every finite bf16 value in [-30, 30], so the activation
    is checked across its whole range, on both sides of every switch in its
    evaluation."""
    sweep = _bf16_sweep(-30.0, 30.0)
    dim = 64
    tokens = (sweep.numel() + dim - 1) // dim
    case = wl.varlen_prefill(90, [tokens], dim, 4, num_cache_lines=1, layout=layout,
                             has_init="none", use_bias=False, with_cache_indices=False,
                             name=f"silu_sweep_{layout}")
    flat = torch.zeros(dim * tokens, dtype=torch.bfloat16)
    flat[: sweep.numel()] = sweep
    case.x.copy_(flat.view(dim, tokens))
    case.weight.zero_()
    case.weight[:, -1] = 1.0
    check(case)


LENGTHS = [1, 2, 3, 4, 5, 127, 128, 129, 255, 0, 300, 31, 33]


@pytest.mark.parametrize("width", [2, 3, 4, 5])
@pytest.mark.parametrize("layout", ["tokens_dim", "dim_tokens"])
def test_widths_and_ragged_chunks(width, layout):
    case = wl.varlen_prefill(200 + width, LENGTHS, 40, width, num_cache_lines=20,
                             layout=layout, pad_positions=(4,), has_init="bernoulli")
    check(case)


@pytest.mark.parametrize("layout", ["tokens_dim", "dim_tokens"])
def test_long_sequences_span_many_chunks(layout):
    case = wl.varlen_prefill(301, [2500, 7, 4100, 1], 24, 4, num_cache_lines=4,
                             layout=layout, has_init="all")
    check(case)


@pytest.mark.parametrize("dim", [1, 7, 100, 264])
@pytest.mark.parametrize("layout", ["tokens_dim", "dim_tokens"])
def test_dims_not_multiple_of_eight(dim, layout):
    case = wl.varlen_prefill(400 + dim, [9, 130, 1, 45], dim, 4, num_cache_lines=5,
                             layout=layout, has_init="bernoulli")
    check(case)


@pytest.mark.parametrize("width", [2, 5])
@pytest.mark.parametrize("extra", [0, 3])
def test_channel_first_chunk_edges(width, extra):
    """Sequences one token short of, exactly at and one past the channel-first
    chunk length (kCfaChunk, read from the kernel source) and of two chunks,
    on rows at several 16-byte phases: the second chunk's halo and segment
    0's slack (up to 127 tokens before the first one needed) meet the
    previous chunk's last segment."""
    lengths = _lengths_around_cf_chunk()
    case = wl.varlen_prefill(520 + width + extra, lengths, 8, width,
                             num_cache_lines=6, layout="dim_tokens", has_init="all",
                             extra_tokens=extra)
    check(case)


def _kernel_constant(name):
    import re

    src = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                            "causal_depthwise_conv1d_fwd_gb300", "csrc", "ccv_fwd.cu")).read()
    return int(re.search(rf"constexpr int {name} = (\d+);", src).group(1))


def _cf_chunk_tokens(total, batch):
    """The host's choice of channel-first streaming kernel and chunk length
    (cf_short_rows and cf_long_chunks in the kernel source), with its
    constants read from the source: the multi-row kernel's kCfrChunk up to
    kCfrMaxAvg tokens per sequence on average, one kCfaChunk-token chunk per
    sequence up to kCfaOneChunk, kCfaChunkSplit-token chunks above."""
    import re

    src = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                            "causal_depthwise_conv1d_fwd_gb300", "csrc", "ccv_fwd.cu")).read()
    one = int(re.search(r"constexpr int kCfaOneChunk = (\d+);", src).group(1))
    rows_max = int(re.search(r"constexpr int kCfrMaxAvg = (\d+);", src).group(1))
    avg = -(-total // batch)
    if avg <= rows_max:
        return TILING["kCfrChunk"]
    return TILING["kCfaChunk"] if avg <= one else TILING["kCfaChunkSplit"]


def _lengths_around_cf_chunk():
    """Sequence lengths c-1, c, c+1, 2c+1 and 3 around the chunk length c the
    host picks for long sequences, plus a filler sequence that makes the
    average long enough for that choice."""
    c = _cf_chunk_tokens(1 << 20, 1)
    head = [c - 1, c, c + 1, 2 * c + 1, 3]
    return head + [70000]


def _lengths_around_rows_chunk(max_avg=None):
    """Sequence lengths c-1, c, c+1, 2c+1 and 3 around the multi-row
    kernel's chunk length c, then short fillers (1 to 60 tokens) until the
    average is at most max_avg (default: the multi-row kernel's limit)."""
    c = TILING["kCfrChunk"]
    max_avg = max_avg or _kernel_constant("kCfrMaxAvg")
    lengths = [c - 1, c, c + 1, 2 * c + 1, 3]
    fill = [1, 2, 3, 5, 60, 17]
    while -(-sum(lengths) // len(lengths)) > max_avg:
        lengths.append(fill[len(lengths) % len(fill)])
    return lengths


def test_chunk_edge_lengths_sit_on_the_chosen_chunk():
    """The chunk-edge cases straddle the chunk length the host picks: the
    split chunk of long sequences, and the multi-row kernel's chunk."""
    lengths = _lengths_around_cf_chunk()
    c = lengths[1]
    assert _cf_chunk_tokens(sum(lengths), len(lengths)) == c
    assert c == TILING["kCfaChunkSplit"] < TILING["kCfaChunk"]
    lengths = _lengths_around_rows_chunk()
    assert _cf_chunk_tokens(sum(lengths), len(lengths)) == lengths[1] == TILING["kCfrChunk"]


@pytest.mark.parametrize("width", [2, 4, 5])
@pytest.mark.parametrize("dim, extra", [(8, 0), (72, 3), (300, 1)])
@pytest.mark.parametrize("limit, above", [("kCfrMaxAvg", "kCfrMidAvg"), ("kCfrMidAvg", "kCfrShortAvg"),
                                          ("kCfrShortAvg", None)])
def test_channel_first_rows_chunk_edges(width, dim, extra, limit, above):
    """The multi-row kernel (blocks of 64, 128 or 256 channel rows by the
    average sequence length; one ring running across each warp's rows) on
    sequences one token short of, at and past its chunk length and of two
    chunks among short fillers; dims of one partial row group, of full
    groups plus a partial one, and rows at several 16-byte phases."""
    lengths = _lengths_around_rows_chunk(_kernel_constant(limit))
    if above is not None:  # the average picks this block size, not the next
        assert -(-sum(lengths) // len(lengths)) > _kernel_constant(above)
    case = wl.varlen_prefill(560 + width + dim + extra, lengths, dim, width,
                             num_cache_lines=len(lengths) + 2, layout="dim_tokens",
                             has_init="bernoulli", extra_tokens=extra)
    check(case)


@pytest.mark.parametrize("extra", [0, 1, 3, 5])
def test_channel_first_unaligned_rows(extra):
    """Channel-first x whose row length is not a multiple of 8 tokens: rows
    start at different 16-byte phases (and tokens past the last sequence are
    not processed)."""
    case = wl.varlen_prefill(500 + extra, [13, 2049, 6, 300], 16, 4, num_cache_lines=4,
                             layout="dim_tokens", has_init="all", extra_tokens=extra)
    check(case)


@pytest.mark.parametrize("shift", [1, 3])
def test_channel_first_misaligned_base(shift):
    """x and out start `shift` elements past a 16-byte boundary (same phase):
    the channel-first kernel that needs only equal phases handles them."""
    case = wl.varlen_prefill(551 + shift, [40, 2100, 5], 16, 4, num_cache_lines=3,
                             layout="dim_tokens", has_init="all")
    T = case.total_tokens

    def shifted(src, device, fill=None):
        buf = torch.zeros(case.dim * (T + 8) + 16, dtype=torch.bfloat16, device=device)
        view = buf[shift:shift + case.dim * (T + 8)].view(case.dim, T + 8)[:, :T]
        if fill is None:
            view.copy_(src.to(device))
        else:
            view.view(torch.int16).fill_(fill)
        return view

    x_cpu, out_cpu = shifted(case.x, "cpu"), shifted(None, "cpu", -12345)
    ref_states = case.conv_states.clone()
    oracle.ccv_fwd(x_cpu, case.weight, case.bias, ref_states, case.query_start_loc,
                   case.cache_indices, case.has_initial_state, case.activation, -1, out=out_cpu)
    d = to_device(case.kwargs(), DEV)
    d["x"] = shifted(case.x, DEV)
    out = shifted(None, DEV, -12345)
    assert d["x"].data_ptr() % 16 == 2 * shift and out.data_ptr() % 16 == 2 * shift
    ccv.ccv_fwd(**d, out=out)
    torch.cuda.synchronize()
    assert_close(out, out_cpu, "misaligned out")
    assert_bits(d["conv_states"], ref_states, "misaligned states")


def test_mixed_layouts_use_generic_path():
    case = wl.varlen_prefill(601, [17, 140, 3], 24, 4, num_cache_lines=3, layout="tokens_dim",
                             has_init="bernoulli")
    out_cpu = sentinel_like(case.x.t().contiguous().t().contiguous())  # (dim, T) channel-first
    out_dev = sentinel_like(out_cpu, DEV)
    ref_out, ref_states, out, states, _ = run_both(case, out_cpu=out_cpu, out_dev=out_dev)
    assert_close(out, ref_out, "mixed out")
    assert_bits(states, ref_states, "mixed states")


def test_strided_views():
    """x and out as every third row of wider buffers: stride over channels 1,
    stride over tokens 90 (not a multiple of 8), so the strided kernel runs."""
    base = wl.varlen_prefill(701, [11, 50, 4], 30, 4, num_cache_lines=3, layout="tokens_dim",
                             has_init="all")
    T = base.total_tokens

    def spread(t_dim_major, device):
        wide = torch.zeros(T * 3, 30, dtype=torch.bfloat16, device=device)
        wide.view(torch.int16).fill_(-99)
        wide[::3] = t_dim_major.t().to(device)
        return wide, wide[::3].t()

    _, x_cpu = spread(base.x, "cpu")
    wide_out_cpu, out_cpu = spread(base.x, "cpu")
    out_cpu.view(torch.int16).fill_(-12345)
    ref_states = base.conv_states.clone()
    oracle.ccv_fwd(x_cpu, base.weight, base.bias, ref_states, base.query_start_loc,
                   base.cache_indices, base.has_initial_state, base.activation, -1, out=out_cpu)
    d = to_device(base.kwargs(), DEV)
    _, d["x"] = spread(base.x, DEV)
    wide_out, out = spread(base.x, DEV)
    out.view(torch.int16).fill_(-12345)
    assert d["x"].stride() == (1, 90) and out.stride() == (1, 90)
    ccv.ccv_fwd(**d, out=out)
    torch.cuda.synchronize()
    assert_close(out, out_cpu, "strided out")
    assert_bits(wide_out, wide_out_cpu, "strided out incl. gaps")
    assert_bits(d["conv_states"], ref_states, "strided states")


@pytest.mark.parametrize("state_layout", ["dim_contiguous", "tok_contiguous"])
@pytest.mark.parametrize("layout", ["tokens_dim", "dim_tokens"])
def test_state_layouts_and_wider_state(state_layout, layout):
    case = wl.varlen_prefill(801, [1, 2, 9, 200], 64, 4, num_cache_lines=6, state_len=7,
                             layout=layout, state_layout=state_layout, has_init="bernoulli")
    check(case)


@pytest.mark.parametrize("layout", ["tokens_dim", "dim_tokens"])
def test_optional_inputs_absent(layout):
    base = dict(num_cache_lines=4, layout=layout)
    check(wl.varlen_prefill(901, [5, 77, 2], 32, 4, use_bias=False, activation=None, **base))
    check(wl.varlen_prefill(902, [5, 77, 2], 32, 4, has_init="null", **base))
    check(wl.varlen_prefill(903, [5, 77, 2], 32, 4, with_cache_indices=False, **base))
    check(wl.varlen_prefill(904, [5, 77, 2], 32, 4, with_states=False, has_init="null", **base))


@pytest.mark.parametrize("layout", ["tokens_dim", "dim_tokens"])
def test_invalid_indices_counted_not_faulting(layout):
    case = wl.varlen_prefill(1001, [6, 9, 3], 16, 4, num_cache_lines=3, layout=layout,
                             has_init="all")
    case.cache_indices[1] = 999  # outside the pool, not the pad id
    ref_out, ref_states, out, states, err = run_both(case, err=True)
    assert int(err.item()) > 0
    assert_close(out, ref_out, "invalid out")
    assert_bits(states, ref_states, "invalid states")


def test_large_values_and_saturation():
    """Inputs far from the benchmark's 0.02 scale: SiLU tails, exp overflow."""
    case = wl.varlen_prefill(1101, [40, 3], 48, 4, num_cache_lines=2, layout="tokens_dim",
                             has_init="all", std=20.0)
    check(case)


def test_guard_bands_untouched():
    """Outputs and states inside larger sentinel-filled buffers: nothing outside
    the logical views changes."""
    case = wl.varlen_prefill(1201, [7, 129, 2], 64, 4, num_cache_lines=4, layout="tokens_dim",
                             has_init="bernoulli")
    T, dim = case.total_tokens, case.dim
    d = to_device(case.kwargs(), DEV)
    big_out = torch.empty(T * dim + 4096, dtype=torch.bfloat16, device=DEV)
    big_out.view(torch.int16).fill_(-777)
    out = big_out[2048:2048 + T * dim].view(T, dim).t()
    st = case.conv_states
    big_st = torch.empty(st.numel() + 4096, dtype=torch.bfloat16, device=DEV)
    big_st.view(torch.int16).fill_(-555)
    st_view = big_st[2048:2048 + st.numel()].view(st.shape[0], st.shape[2], st.shape[1])
    st_view.copy_(st.transpose(1, 2))
    d["conv_states"] = st_view.transpose(1, 2)
    ccv.ccv_fwd(**d, out=out)
    torch.cuda.synchronize()
    assert bool((big_out[:2048].view(torch.int16) == -777).all())
    assert bool((big_out[2048 + T * dim:].view(torch.int16) == -777).all())
    assert bool((big_st[:2048].view(torch.int16) == -555).all())
    assert bool((big_st[2048 + st.numel():].view(torch.int16) == -555).all())
    ref_states = case.conv_states.clone()
    ref_out = sentinel_like(case.x)
    oracle.ccv_fwd(case.x, case.weight, case.bias, ref_states, case.query_start_loc,
                   case.cache_indices, case.has_initial_state, case.activation, -1, out=ref_out)
    assert_close(out, ref_out, "guard out")
    assert_bits(d["conv_states"], ref_states, "guard states")


def test_empty_inputs_launch_nothing():
    case = wl.varlen_prefill(1301, [0, 0], 16, 4, num_cache_lines=2)
    check(case)
    d = to_device(case.kwargs(), DEV)
    d["query_start_loc"] = torch.zeros(1, dtype=torch.int32, device=DEV)
    d["cache_indices"] = d["cache_indices"][:0]
    d["has_initial_state"] = d["has_initial_state"][:0]
    ccv.ccv_fwd(**d)  # batch 0


def test_rejects_cpu_tensors_and_aliasing():
    case = wl.varlen_prefill(1401, [4], 16, 4, num_cache_lines=1)
    with pytest.raises(TypeError):
        ccv.ccv_fwd(**case.kwargs())
    d = to_device(case.kwargs(), DEV)
    with pytest.raises(ccv.CcvError):
        ccv.ccv_fwd(**d, out=d["x"])


def test_cuda_graph_replay_matches_eager():
    """Capture one call, then replay it on fresh inputs copied into the same
    buffers: same results as an eager call on those inputs."""
    c1 = wl.varlen_prefill(1501, [100, 3, 260], 256, 4, num_cache_lines=4, layout="tokens_dim",
                           has_init="all")
    c2 = wl.varlen_prefill(1502, [100, 3, 260], 256, 4, num_cache_lines=4, layout="tokens_dim",
                           has_init="all")
    d = to_device(c1.kwargs(), DEV)
    out = sentinel_like(d["x"])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        ccv.ccv_fwd(**d, out=out)  # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ccv.ccv_fwd(**d, out=out)
    d2 = to_device(c2.kwargs(), DEV)
    for k in ("x", "weight", "bias", "conv_states", "query_start_loc", "cache_indices",
              "has_initial_state"):
        d[k].copy_(d2[k])
    g.replay()
    torch.cuda.synchronize()
    ref_states = c2.conv_states.clone()
    ref_out = sentinel_like(c2.x)
    oracle.ccv_fwd(c2.x, c2.weight, c2.bias, ref_states, c2.query_start_loc, c2.cache_indices,
                   c2.has_initial_state, c2.activation, -1, out=ref_out)
    assert_close(out, ref_out, "graph out")
    assert_bits(d["conv_states"], ref_states, "graph states")


def test_strided_bias_is_rejected():
    """bias is read as dim contiguous values: a strided view raises in the
    binding for prefill, decode and spec-verify alike (no silent misread)."""
    case = wl.varlen_prefill(1601, [5, 9], 64, 4, num_cache_lines=2)
    d = to_device(case.kwargs(), DEV)
    packed = torch.zeros(64, 2, dtype=torch.bfloat16, device=DEV)
    d["bias"] = packed[:, 1]
    with pytest.raises(ValueError, match="contiguous"):
        ccv.ccv_fwd(**d)
    dc = to_device(wl.decode(1602, 4, 64, 4, num_lines=4).kwargs(), DEV)
    dc["bias"] = packed[:, 0]
    with pytest.raises(ValueError, match="contiguous"):
        ccv.ccv_update(**dc)
    with pytest.raises(ValueError, match="contiguous"):
        ccv.ccv_update_spec(**dc)


def _kernel_names(fn):
    """Names of the CUDA kernels `fn` launches, or None when the profiler is
    unavailable or records no kernel launched outside torch."""
    try:
        from torch.profiler import ProfilerActivity, profile
        with profile(activities=[ProfilerActivity.CUDA]) as prof:
            fn()
            torch.cuda.synchronize()
        names = [e.name for e in prof.events() if e.device_type.name == "CUDA"]
    except Exception:  # no CUPTI in this build
        return None
    return names or None  # a profiler that saw no kernel at all tells nothing


@pytest.mark.parametrize("layout", ["tokens_dim", "dim_tokens"])
@pytest.mark.parametrize("tokens", [2048, 2049])
def test_automatic_choice_at_its_threshold(prefill_path, monkeypatch, layout, tokens):
    """Without CCV_PREFILL_PATH the size decides: total_tokens x dim up to 2^23
    elements takes the short kernels, more takes the streaming ones.  At dim
    4096, 2048 tokens is the last short problem and 2049 the first streaming
    one; both match the oracle."""
    if prefill_path == "stream":
        pytest.skip("the automatic choice is the same for both fixture values")
    monkeypatch.delenv("CCV_PREFILL_PATH")
    case = wl.varlen_prefill(1700 + tokens, [tokens - 700, 3, 697], 4096, 4, num_cache_lines=4,
                             layout=layout, pad_positions=(1,), has_init="bernoulli")
    ref_out, ref_states, out, states, _ = run_both(case)
    assert_close(out, ref_out, f"threshold {tokens} out")
    assert_bits(states, ref_states, f"threshold {tokens} states")
    d = to_device(case.kwargs(), DEV)
    names = _kernel_names(lambda: ccv.ccv_fwd(**d))
    if names is not None:
        # streaming: fwd_cl_async, fwd_cf_async or, for short sequences, fwd_cf_rows
        want = ("short",) if tokens * 4096 <= (1 << 23) else ("async", "rows")
        assert any(w in n for n in names for w in want), names


@pytest.mark.parametrize("avg, want, rows", [(512, "fwd_cf_rows_kernel", 256),
                                             (1024, "fwd_cf_rows_kernel", 128),
                                             (3072, "fwd_cf_rows_kernel", 64),
                                             (3073, "fwd_cf_async_kernel", None)])
def test_channel_first_streaming_choice(prefill_path, avg, want, rows):
    """The host picks the channel-first streaming kernel from the average
    sequence length: the multi-row kernel up to kCfrMaxAvg tokens (256, 128
    or 64 rows per block by kCfrShortAvg and kCfrMidAvg), the single-row one
    above.  Lengths with that average at dim 1024, streaming kernels forced,
    match the oracle and launch the expected kernel."""
    if prefill_path == "short":
        pytest.skip("the streaming choice only")
    assert _kernel_constant("kCfrMaxAvg") == 3072 and _kernel_constant("kCfrMidAvg") == 1024
    assert _kernel_constant("kCfrShortAvg") == 512
    batch = 4
    lengths = [avg - 7, avg + 3, avg + 7, avg - 3]  # mean avg; ceil(total / batch) == avg
    case = wl.varlen_prefill(1900 + avg, lengths, 1024, 4, num_cache_lines=batch,
                             layout="dim_tokens", has_init="bernoulli")
    check(case)
    d = to_device(case.kwargs(), DEV)
    names = _kernel_names(lambda: ccv.ccv_fwd(**d))
    if names is not None:
        assert any(want in n for n in names), names
        if rows is not None:
            assert any(f", {rows}>" in n for n in names), names


@pytest.mark.parametrize("layout", ["tokens_dim", "dim_tokens"])
@pytest.mark.parametrize("batch", [33, 100, 128, 129, 1100, 4200])
def test_many_sequences(layout, batch):
    """More than 32 sequences: the chunk search narrows the candidates in
    rounds before its final one (the short kernels and the channel-last
    streaming kernel take 32 candidates in the final round, the channel-first
    streaming kernel 128, four per lane: 128 and 129 sit on its edge, 4200
    takes it two narrowing rounds), with zero-length and pad sequences among
    them."""
    import random

    r = random.Random(1800 + batch)
    lengths = [r.choice([0, 1, 2, 3, 5, 9, 17, r.randint(1, 60)]) for _ in range(batch)]
    pads = tuple(i for i in range(batch) if r.random() < 0.1)
    case = wl.varlen_prefill(1800 + batch, lengths, 16, 4, num_cache_lines=batch + 3,
                             layout=layout, pad_positions=pads, has_init="bernoulli")
    check(case)
