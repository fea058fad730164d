"""Pins for the CPU oracle (``oracle/``), checked against things other than itself.

* the reference formulation of atrex-bench #003 ``causal_conv1d``
  (``Model.forward``: concatenate the state, grouped ``F.conv1d``, keep the last
  T outputs, SiLU), run here by torch in float64 -- a library routine the
  oracle does not use;
* exact small-integer arithmetic against ``numpy.correlate``;
* torch's own float -> bfloat16 cast and ``F.silu``;
* the worked examples the pages print (``tests/golden/``);
* invariants: split sequence == one sequence, decode == one-token prefill,
  delta filters, pad and zero-state behaviour.

All of this runs on the CPU.
"""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from causal_depthwise_conv1d_fwd_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
SENTINEL = -12345  # int16 bit pattern written into "must stay untouched" memory


def _f64(t):
    return None if t is None else t.to(torch.float64)


def r1_reference(x_seq, weight, bias, state, silu):
    """atrex-bench #003 reference formulation, float64, for one sequence.

    x_seq (dim, L), weight (dim, W), bias (dim,) or None, state (dim, >=W-1).
    """
    W = weight.shape[1]
    seq = _f64(x_seq).unsqueeze(0)
    st = _f64(state).unsqueeze(0)
    seq_with_state = torch.cat([st[:, :, -(W - 1):], seq], dim=-1)
    out = F.conv1d(seq_with_state, _f64(weight).unsqueeze(1), _f64(bias),
                   groups=weight.shape[0])
    out = out[:, :, -x_seq.shape[-1]:]
    if silu:
        out = F.silu(out)
    return out.squeeze(0)


def assert_bf16_close(got, ref, rtol=2.0 ** -8, atol=1e-6):
    got = got.to(torch.float64)
    ref = ref.to(torch.float64)
    err = (got - ref).abs()
    bound = rtol * ref.abs() + atol
    bad = err > bound
    assert not bool(bad.any()), (
        f"{int(bad.sum())} of {bad.numel()} outside tolerance; worst err "
        f"{float(err.max()):.3e} at ref {float(ref.flatten()[int(err.argmax())]):.3e}")


def prior_of(case, i):
    """The (dim, W-1) prior of batch entry i, per the pages' has_initial_state rule."""
    W = case.width
    line = int(case.cache_indices[i]) if case.cache_indices is not None else i
    use = (case.conv_states is not None and case.has_initial_state is not None
           and bool(case.has_initial_state[i]))
    if use:
        return case.conv_states[line, :, :W - 1].clone()
    return torch.zeros(case.dim, W - 1, dtype=torch.bfloat16)


def run_oracle_fwd(case, out=None):
    states = None if case.conv_states is None else case.conv_states.clone()
    if out is None:
        out = wl.empty_like_layout(case.x)
        out.view(torch.int16).fill_(SENTINEL)
    o, err = oracle.ccv_fwd(case.x, case.weight, case.bias, states, case.query_start_loc,
                            case.cache_indices, case.has_initial_state, case.activation,
                            case.pad_slot_id, out=out)
    return o, states, err


# ------------------------------------------------------------ primitives ----

def test_bf16_rounding_matches_torch_cast():
    g = torch.Generator().manual_seed(1)
    vals = torch.randn(200000, generator=g) * torch.exp(torch.randn(200000, generator=g) * 20)
    # exact ties, both parities, around 1.0 and a few binades
    base = torch.tensor([1.0, 2.0, 0.5, 3.0e-38, 1.0e30], dtype=torch.float32)
    ties = []
    for b in base:
        u = int(b.view(torch.int32))
        for lsb in (0, 1):
            ties.append((u & ~0xFFFF) | (lsb << 16) | 0x8000)
            ties.append((u & ~0xFFFF) | (lsb << 16) | 0x7FFF)
            ties.append((u & ~0xFFFF) | (lsb << 16) | 0x8001)
    specials = torch.tensor([0.0, -0.0, float("inf"), float("-inf"), 3.3895314e38,
                             -3.3895314e38, 1e-45, -1e-45, 1.17e-38], dtype=torch.float32)
    allv = torch.cat([vals.float(), torch.tensor(ties, dtype=torch.int32).view(torch.float32),
                      specials])
    mine = oracle.f32_to_bf16_bits(allv)
    ref = allv.to(torch.bfloat16).view(torch.int16)
    assert torch.equal(mine, ref)
    nan = oracle.f32_to_bf16_bits(torch.tensor([float("nan")]))
    assert torch.isnan(nan.view(torch.bfloat16).float()).all()


def test_silu_matches_torch_float64():
    v = torch.cat([torch.linspace(-120, 120, 20001), torch.randn(10000) * 0.05]).float()
    mine = oracle.silu_f32(v).to(torch.float64)
    ref = F.silu(v.to(torch.float64))
    ulp = torch.finfo(torch.float32).eps * ref.abs() + 1e-44
    assert bool(((mine - ref).abs() <= ulp).all())


# ------------------------------------------- reference formulation (R1) ----

@pytest.mark.parametrize("width", [2, 3, 4, 5])
@pytest.mark.parametrize("layout", ["tokens_dim", "dim_tokens"])
@pytest.mark.parametrize("silu", [True, False])
@pytest.mark.parametrize("T", [1, 2, 3, 7, 32])
def test_single_sequence_matches_reference_formulation(width, layout, silu, T):
    case = wl.varlen_prefill(11 + width * 100 + T, [T], 24, width, layout=layout,
                             has_init="all", with_cache_indices=False,
                             activation="silu" if silu else None)
    out, states, err = run_oracle_fwd(case)
    assert err == 0
    ref = r1_reference(case.x, case.weight, case.bias, prior_of(case, 0), silu)
    assert_bf16_close(out, ref)


@pytest.mark.parametrize("layout", ["tokens_dim", "dim_tokens"])
@pytest.mark.parametrize("state_layout", ["dim_contiguous", "tok_contiguous"])
def test_varlen_matches_reference_formulation_per_sequence(layout, state_layout):
    lengths = [5, 1, 9, 2, 33, 3, 17]
    case = wl.varlen_prefill(77, lengths, 40, 4, num_cache_lines=12, layout=layout,
                             state_layout=state_layout, has_init="bernoulli",
                             use_bias=True, activation="silu")
    out, states, err = run_oracle_fwd(case)
    assert err == 0
    q = case.query_start_loc
    for i in range(len(lengths)):
        s, e = int(q[i]), int(q[i + 1])
        ref = r1_reference(case.x[:, s:e], case.weight, case.bias, prior_of(case, i), True)
        assert_bf16_close(out[:, s:e], ref)


def test_exact_integer_arithmetic_matches_numpy_correlate():
    """Small integers keep every product, sum and result exact in fp32 and bf16,
    so the oracle must reproduce numpy's correlation bit for bit."""
    g = torch.Generator().manual_seed(5)
    for width in (2, 3, 4, 5):
        lengths = [1, 2, width - 1, width, 11]
        dim = 6
        case = wl.varlen_prefill(9, lengths, dim, width, num_cache_lines=8,
                                 layout="dim_tokens", has_init="bernoulli", activation=None)
        total = sum(lengths)
        case.x.copy_(torch.randint(-3, 4, (dim, total), generator=g).to(torch.bfloat16))
        case.weight.copy_(torch.randint(-2, 3, (dim, width), generator=g).to(torch.bfloat16))
        case.bias.copy_(torch.randint(-3, 4, (dim,), generator=g).to(torch.bfloat16))
        case.conv_states.copy_(torch.randint(-3, 4, case.conv_states.shape,
                                             generator=g).to(torch.bfloat16))
        out, states, err = run_oracle_fwd(case)
        q = case.query_start_loc.tolist()
        for i in range(len(lengths)):
            prior = prior_of(case, i).to(torch.int64).numpy()
            for c in range(dim):
                u = np.concatenate([prior[c], case.x[c, q[i]:q[i + 1]].to(torch.int64).numpy()])
                want = np.correlate(u, case.weight[c].to(torch.int64).numpy(), "valid")
                want = want + int(case.bias[c])
                got = out[c, q[i]:q[i + 1]].to(torch.int64).numpy()
                assert np.array_equal(got, want), (width, i, c, got, want)


# ------------------------------------------------------------ invariants ----

@pytest.mark.parametrize("width", [2, 3, 4, 5])
def test_split_sequence_equals_one_call(width):
    """Prefilling L tokens at once == prefilling L1 then L-L1 with the state
    carried in between (has_initial_state=1 on the second call), bit for bit,
    for every split point including those shorter than W-1."""
    L, dim = 13, 16
    full = wl.varlen_prefill(3 + width, [L], dim, width, layout="tokens_dim",
                             has_init="all", with_cache_indices=False)
    out_full, st_full, _ = run_oracle_fwd(full)
    for L1 in range(0, L + 1):
        st = full.conv_states.clone()
        pieces = []
        for s, e in ((0, L1), (L1, L)):
            part = wl.PrefillCase("part", full.x[:, s:e], full.weight, full.bias, st,
                                  torch.tensor([0, e - s], dtype=torch.int32), None,
                                  torch.ones(1, dtype=torch.bool), full.activation)
            o = wl.empty_like_layout(part.x)
            oracle.ccv_fwd(part.x, part.weight, part.bias, st, part.query_start_loc,
                           None, part.has_initial_state, part.activation, -1, out=o)
            pieces.append(o)
        joined = torch.cat(pieces, dim=1)
        assert torch.equal(joined.view(torch.int16), out_full.view(torch.int16)), L1
        assert torch.equal(st.view(torch.int16), st_full.view(torch.int16)), L1


@pytest.mark.parametrize("width", [2, 4, 5])
def test_delta_filters(width):
    """w = e_{W-1} gives x + bias; w = e_0 gives the input delayed by W-1 taps
    (the prior first).  SiLU off; the single fp32 add and the bf16 cast are
    done here by torch."""
    L, dim = 9, 8
    case = wl.varlen_prefill(21, [L], dim, width, layout="dim_tokens", has_init="all",
                             with_cache_indices=False, activation=None)
    prior = prior_of(case, 0)
    for tap in (width - 1, 0):
        case.weight.zero_()
        case.weight[:, tap] = 1.0
        out, _, _ = run_oracle_fwd(case)
        u = torch.cat([prior, case.x], dim=1).float()
        shifted = u[:, tap:tap + L]
        want = (shifted + case.bias.float()[:, None]).to(torch.bfloat16)
        assert torch.equal(out.view(torch.int16), want.view(torch.int16)), tap


@pytest.mark.parametrize("width", [2, 3, 4, 5])
@pytest.mark.parametrize("L", [1, 2, 3, 4, 8])
def test_state_writeback_is_last_inputs(width, L):
    """The new state is the last W-1 inputs of prior ++ x (shift-left for short
    sequences; zeros stand in for a missing initial state)."""
    for init in (True, False):
        case = wl.varlen_prefill(5 * L + width, [L], 8, width, layout="tokens_dim",
                                 has_init="all" if init else "none",
                                 with_cache_indices=False)
        before = case.conv_states.clone()
        _, states, _ = run_oracle_fwd(case)
        prior = before[0, :, :width - 1] if init else torch.zeros(8, width - 1, dtype=torch.bfloat16)
        u = torch.cat([prior, case.x], dim=1)
        assert torch.equal(states[0, :, :width - 1].view(torch.int16),
                           u[:, -(width - 1):].view(torch.int16))


def test_wider_state_columns_are_left_alone():
    case = wl.varlen_prefill(8, [6, 2], 8, 4, state_len=6, num_cache_lines=2,
                             has_init="all", with_cache_indices=False)
    before = case.conv_states.clone()
    _, states, _ = run_oracle_fwd(case)
    assert torch.equal(states[:, :, 3:].view(torch.int16), before[:, :, 3:].view(torch.int16))
    assert not torch.equal(states[:, :, :3].view(torch.int16), before[:, :, :3].view(torch.int16))


def test_pad_entries_and_zero_length_sequences_are_untouched():
    lengths = [4, 0, 3, 5]
    case = wl.varlen_prefill(31, lengths, 16, 4, num_cache_lines=6, pad_positions=(2,),
                             has_init="all")
    before = case.conv_states.clone()
    out, states, err = run_oracle_fwd(case)
    assert err == 0
    q = case.query_start_loc.tolist()
    # pad entry: its tokens stay as the sentinel, its line keeps its bits
    assert bool((out[:, q[2]:q[3]].view(torch.int16) == SENTINEL).all())
    pad_line_untouched = [l for l in range(6) if l not in case.cache_indices.tolist()]
    for l in pad_line_untouched:
        assert torch.equal(states[l].view(torch.int16), before[l].view(torch.int16))
    # zero-length entry: no output tokens exist, and its line is not rewritten
    line1 = int(case.cache_indices[1])
    assert torch.equal(states[line1].view(torch.int16), before[line1].view(torch.int16))
    # the others were processed
    for i in (0, 3):
        assert not bool((out[:, q[i]:q[i + 1]].view(torch.int16) == SENTINEL).any())


def test_zero_length_sequence_without_initial_state_keeps_its_line():
    """A zero-length sequence launches nothing in the pages' prefill, so even
    with has_initial_state = 0 its line is not zeroed."""
    case = wl.varlen_prefill(33, [3, 0, 2], 8, 4, num_cache_lines=3, has_init="none")
    before = case.conv_states.clone()
    _, states, _ = run_oracle_fwd(case)
    line1 = int(case.cache_indices[1])
    assert torch.equal(states[line1].view(torch.int16), before[line1].view(torch.int16))


def test_has_initial_state_false_equals_zero_state():
    case = wl.varlen_prefill(41, [7, 2], 16, 4, num_cache_lines=2, has_init="none",
                             with_cache_indices=False)
    out_a, st_a, _ = run_oracle_fwd(case)
    zero = case.conv_states.clone().zero_()
    case2 = wl.PrefillCase("z", case.x, case.weight, case.bias, zero, case.query_start_loc,
                           None, torch.ones(2, dtype=torch.bool), case.activation)
    out_b, st_b, _ = run_oracle_fwd(case2)
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))
    assert torch.equal(st_a.view(torch.int16), st_b.view(torch.int16))
    # a null has_initial_state and a null conv_states also mean a zero prior
    for hi, cs in ((None, case.conv_states), (None, None)):
        c3 = wl.PrefillCase("n", case.x, case.weight, case.bias, cs, case.query_start_loc,
                            None, hi, case.activation)
        out_c, _, _ = run_oracle_fwd(c3)
        assert torch.equal(out_c.view(torch.int16), out_a.view(torch.int16))


def test_invalid_indices_are_counted_and_skipped():
    case = wl.varlen_prefill(51, [3, 4], 8, 4, num_cache_lines=2, has_init="all")
    case.cache_indices[1] = 7  # outside the pool, not the pad id
    before = case.conv_states.clone()
    out, states, err = run_oracle_fwd(case)
    assert err == 1
    q = case.query_start_loc.tolist()
    assert bool((out[:, q[1]:q[2]].view(torch.int16) == SENTINEL).all())
    line0 = int(case.cache_indices[0])
    assert not torch.equal(states[line0].view(torch.int16), before[line0].view(torch.int16))
    bad_qsl = wl.PrefillCase("q", case.x, case.weight, case.bias, case.conv_states.clone(),
                             torch.tensor([0, 5, 3], dtype=torch.int32), None,
                             None, case.activation)
    _, _, err2 = run_oracle_fwd(bad_qsl)
    assert err2 == 1


# ------------------------------------------------------ worked examples ----

def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line)
    return rows


def test_golden_query_start_loc_examples():
    """The docstring's examples: lengths -> query_start_loc, and each sequence's
    outputs are exactly those of running it alone."""
    for row in _read_golden("qsl_examples.txt"):
        lens_s, qsl_s, total_s = [p.strip() for p in row.split("|")]
        lengths = [int(v) for v in lens_s.split()]
        want_qsl = [int(v) for v in qsl_s.split()]
        assert wl.cumulative(lengths).tolist() == want_qsl
        case = wl.varlen_prefill(61, lengths, 8, 4, has_init="bernoulli")
        assert case.total_tokens == int(total_s)
        out, _, err = run_oracle_fwd(case)
        assert err == 0
        for i in range(len(lengths)):
            s, e = want_qsl[i], want_qsl[i + 1]
            ref = r1_reference(case.x[:, s:e], case.weight, case.bias, prior_of(case, i), True)
            assert_bf16_close(out[:, s:e], ref)


def test_golden_pad_cache_indices_example():
    kv = {}
    for r in _read_golden("cache_indices_pad.txt"):
        k, v = r.split("=")
        kv[k.strip()] = [int(t) for t in v.split()]
    pad = kv["pad_slot_id"][0]
    idx = kv["cache_indices"]
    skipped = kv["not_processed"]
    case = wl.varlen_prefill(71, [2, 3, 1, 4], 8, 4, num_cache_lines=21, has_init="all")
    case.cache_indices.copy_(torch.tensor(idx, dtype=torch.int32))
    case.pad_slot_id = pad
    out, states, err = run_oracle_fwd(case)
    q = case.query_start_loc.tolist()
    for i in range(4):
        touched = not bool((out[:, q[i]:q[i + 1]].view(torch.int16) == SENTINEL).all())
        assert touched == (i not in skipped), i
    # decode: the same example through the update path
    dcase = wl.decode(72, 4, 8, 4, num_lines=21)
    dcase.conv_state_indices.copy_(torch.tensor(idx, dtype=torch.int32))
    x_before = dcase.x.clone()
    res, _ = oracle.ccv_update(dcase.x, dcase.conv_state, dcase.weight, dcase.bias,
                               dcase.activation, dcase.conv_state_indices, pad)
    for i in range(4):
        same = torch.equal(res[i].view(torch.int16), x_before[i].view(torch.int16))
        assert same == (i in skipped), i


def test_golden_rolling_after_forward():
    """Decode over N new tokens keeps history: [h1..hM] -> [h2..hM, d1..dN]."""
    for row in _read_golden("spec_rolling.txt"):
        head, after_s, _ = [p.strip() for p in row.split("|")]
        M, N = (int(v) for v in head.split())
        W = M + 1
        names = [f"h{i}" for i in range(1, M + 1)] + [f"d{j}" for j in range(1, N + 1)]
        code = {n: float(k + 1) for k, n in enumerate(names)}  # exact in bf16
        dcase = wl.decode(81, 1, 2, W, num_lines=1, seqlen=N, with_indices=False, squeeze=False)
        for c in range(2):
            for m in range(M):
                dcase.conv_state[0, c, m] = code[f"h{m + 1}"]
            for j in range(N):
                dcase.x[0, c, j] = code[f"d{j + 1}"]
        out = torch.empty_like(dcase.x)
        oracle.ccv_update(dcase.x, dcase.conv_state, dcase.weight, dcase.bias,
                          dcase.activation, None, -1, out=out)
        want = [code[n] for n in after_s.split()]
        for c in range(2):
            got = dcase.conv_state[0, c, :M - 1 + N].float().tolist()
            assert got == want, (row, got, want)


def test_golden_spec_window_after_acceptance():
    """The second half of the same example: after accepting k drafts, the next
    step reads the window [h(k+1) .. hM, d1 .. dk], i.e. num_accepted_tokens
    = k.  A unit filter (tap p = 1, no bias, no activation) makes the output
    equal window column p, so the window is read out column by column."""
    for row in _read_golden("spec_rolling.txt"):
        head, after_s, tail = [p.strip() for p in row.split("|")]
        M, N = (int(v) for v in head.split())
        W = M + 1
        k_s, window_s = [p.strip() for p in tail.split("->")]
        k = int(k_s)
        names = [f"h{i}" for i in range(1, M + 1)] + [f"d{j}" for j in range(1, N + 1)]
        code = {n: float(i + 1) for i, n in enumerate(names)}
        state = torch.tensor([[code[n] for n in after_s.split()]], dtype=torch.bfloat16)
        state = state.unsqueeze(0).repeat(1, 2, 1)           # (1 line, 2 channels, M-1+N)
        got = []
        for p in range(W - 1):
            weight = torch.zeros(2, W, dtype=torch.bfloat16)
            weight[:, p] = 1.0
            x = torch.zeros(1, 2, 1, dtype=torch.bfloat16)
            out, err = oracle.ccv_update_spec(x, state.clone(), weight, None, None, None,
                                              torch.tensor([k], dtype=torch.int32))
            assert err == 0
            got.append(float(out[0, 0, 0]))
        assert got == [code[n] for n in window_s.split()], (row, got)


# ---------------------------------------------------------------- decode ----

@pytest.mark.parametrize("width", [2, 3, 4, 5])
@pytest.mark.parametrize("state_layout", ["dim_contiguous", "tok_contiguous"])
def test_decode_equals_one_token_prefill(width, state_layout):
    dcase = wl.decode(91 + width, 6, 24, width, num_lines=9, state_layout=state_layout,
                      pad_positions=(3,))
    pool_a = dcase.conv_state.clone()
    pool_b = dcase.conv_state.clone()
    x = dcase.x.clone()
    out_dec, err = oracle.ccv_update(x, pool_a, dcase.weight, dcase.bias, "silu",
                                     dcase.conv_state_indices, -1)
    assert err == 0
    pre = wl.PrefillCase("p", dcase.x.t(), dcase.weight, dcase.bias, pool_b,
                         torch.arange(7, dtype=torch.int32), dcase.conv_state_indices,
                         torch.ones(6, dtype=torch.bool), "silu")
    out_pre = wl.empty_like_layout(pre.x)
    out_pre.view(torch.int16).fill_(SENTINEL)
    oracle.ccv_fwd(pre.x, pre.weight, pre.bias, pool_b, pre.query_start_loc,
                   pre.cache_indices, pre.has_initial_state, "silu", -1, out=out_pre)
    for b in range(6):
        if b == 3:
            assert torch.equal(out_dec[b].view(torch.int16), dcase.x[b].view(torch.int16))
            continue
        assert torch.equal(out_dec[b].view(torch.int16), out_pre[:, b].view(torch.int16))
    assert torch.equal(pool_a.view(torch.int16), pool_b.view(torch.int16))


def test_decode_matches_reference_formulation():
    dcase = wl.decode(101, 5, 32, 4, num_lines=7)
    before = dcase.conv_state.clone()
    x = dcase.x.clone()
    out, _ = oracle.ccv_update(x, dcase.conv_state, dcase.weight, dcase.bias, "silu",
                               dcase.conv_state_indices, -1)
    for b in range(5):
        line = int(dcase.conv_state_indices[b])
        ref = r1_reference(dcase.x[b][:, None], dcase.weight, dcase.bias, before[line], True)
        assert_bf16_close(out[b][:, None], ref)


# -------------------------------------------------------- spec decoding ----

def _spec_prior(case, b):
    """(dim, W-1) window row b starts from: state columns off .. off+W-2."""
    W = case.weight.shape[1]
    line = int(case.conv_state_indices[b])
    off = int(case.num_accepted_tokens[b]) - 1 if case.num_accepted_tokens is not None else 0
    return case.conv_state[line, :, off:off + W - 1].clone()


def _run_spec(case):
    pool = case.conv_state.clone()
    inter = None if case.intermediate_conv_window is None else case.intermediate_conv_window.clone()
    x = case.x.clone()
    out, err = oracle.ccv_update_spec(x, pool, case.weight, case.bias, case.activation,
                                      case.conv_state_indices, case.num_accepted_tokens,
                                      inter, case.output_state_indices, case.pad_slot_id)
    return out, pool, inter, err


@pytest.mark.parametrize("width", [2, 3, 4, 5])
def test_spec_without_extras_equals_plain_update(width):
    """No accepted-token offset and no buffers: the plain multi-token update."""
    case = wl.spec_decode(400 + width, 5, 24, width, 3, with_accepted=False, history=1,
                          pad_positions=(2,))
    out_s, pool_s, _, err_s = _run_spec(case)
    pool_p = case.conv_state.clone()
    out_p, err_p = oracle.ccv_update(case.x.clone(), pool_p, case.weight, case.bias,
                                     case.activation, case.conv_state_indices, -1)
    assert err_s == err_p == 0
    assert torch.equal(out_s.view(torch.int16), out_p.view(torch.int16))
    assert torch.equal(pool_s.view(torch.int16), pool_p.view(torch.int16))


@pytest.mark.parametrize("width", [2, 3, 4, 5])
def test_spec_outputs_match_reference_formulation(width):
    """Outputs against F.conv1d on the window at the accepted-token offset."""
    case = wl.spec_decode(410 + width, 6, 32, width, 4, history=3, with_intermediate=True,
                          with_output_indices=True)
    out, _, _, err = _run_spec(case)
    assert err == 0
    for b in range(6):
        ref = r1_reference(case.x[b], case.weight, case.bias, _spec_prior(case, b), True)
        assert_bf16_close(out[b], ref)


@pytest.mark.parametrize("width", [2, 3, 4, 5])
def test_spec_windows_and_output_lines_are_last_inputs(width):
    """After token t the window is the last W-1 inputs of prior ++ x[:t+1]:
    it lands in the intermediate buffer at (b, t) and in output line
    output_state_indices[b, t] (columns 0..W-2); nothing else changes."""
    seqlen, steps = 3, 5
    case = wl.spec_decode(420 + width, 4, 16, width, seqlen, history=2, steps=steps,
                          with_intermediate=True, with_output_indices=True, skip_frac=0.3)
    _, pool, inter, err = _run_spec(case)
    assert err == 0
    exp_pool = case.conv_state.clone()
    exp_inter = case.intermediate_conv_window.clone()
    for b in range(4):
        u = torch.cat([_spec_prior(case, b), case.x[b]], dim=1)
        for t in range(seqlen):
            win = u[:, t + 1:t + width]
            exp_inter[b, t] = win
            o = int(case.output_state_indices[b, t])
            if o >= 0:
                exp_pool[o, :, :width - 1] = win
    assert torch.equal(inter.view(torch.int16), exp_inter.view(torch.int16))
    assert torch.equal(pool.view(torch.int16), exp_pool.view(torch.int16))


@pytest.mark.parametrize("width", [2, 3, 4, 5])
def test_spec_verify_equals_successive_single_token_updates(width):
    """A verify step over N drafts gives the outputs and per-step windows of N
    single-token decode updates started from the offset window."""
    seqlen = 4
    case = wl.spec_decode(430 + width, 3, 16, width, seqlen, history=3,
                          with_intermediate=True)
    out, _, inter, err = _run_spec(case)
    assert err == 0
    for b in range(3):
        pool = _spec_prior(case, b).unsqueeze(0).contiguous()
        for t in range(seqlen):
            xt = case.x[b:b + 1, :, t].clone()
            o1, e1 = oracle.ccv_update(xt, pool, case.weight, case.bias, case.activation,
                                       None, -1)
            assert e1 == 0
            assert torch.equal(out[b, :, t].view(torch.int16), o1[0].view(torch.int16))
            assert torch.equal(inter[b, t].view(torch.int16), pool[0].view(torch.int16))


@pytest.mark.parametrize("width", [2, 4, 5])
def test_spec_shift_with_offset_is_closed_form(width):
    """Offset but no buffers: columns [0, W-2+seqlen) of the line become
    (window ++ x)[1:]; the other columns and lines stay."""
    seqlen = 3
    case = wl.spec_decode(440 + width, 4, 16, width, seqlen, history=3)
    _, pool, _, err = _run_spec(case)
    assert err == 0
    exp = case.conv_state.clone()
    for b in range(4):
        line = int(case.conv_state_indices[b])
        u = torch.cat([_spec_prior(case, b), case.x[b]], dim=1)
        exp[line, :, :width - 2 + seqlen] = u[:, 1:]
    assert torch.equal(pool.view(torch.int16), exp.view(torch.int16))


def test_spec_invalid_offsets_and_output_lines_are_counted():
    case = wl.spec_decode(450, 4, 16, 4, 2, history=1, with_output_indices=True,
                          skip_frac=0.0)
    case.num_accepted_tokens[1] = 0                   # offset -1
    case.num_accepted_tokens[2] = 3                   # offset 2: needs 5 columns, has 4
    case.output_state_indices[3, 1] = case.conv_state.shape[0]   # outside the pool
    out, pool, _, err = _run_spec(case)
    assert err > 0
    for b in (1, 2):                                  # skipped rows: out is still x
        assert torch.equal(out[b].view(torch.int16), case.x[b].view(torch.int16))
        for t in range(2):
            o = int(case.output_state_indices[b, t])
            assert torch.equal(pool[o].view(torch.int16), case.conv_state[o].view(torch.int16))
    o = int(case.output_state_indices[3, 0])          # the valid write of row 3 happened
    u = torch.cat([_spec_prior(case, 3), case.x[3]], dim=1)
    assert torch.equal(pool[o, :, :3].view(torch.int16), u[:, 1:4].view(torch.int16))


# ----------------------------------------------------------------- paged ----

def _small_paged(seed, lengths, starts, **kw):
    args = dict(H=2, ws=8, N=4, D=24, num_blocks=64, off_s=8, width=4)
    args.update(kw)
    return wl.paged(seed, lengths, starts, **args)


def _history(case, r, W):
    """The W-1 pre-forward inputs of request r, read from the cache through
    its block table (zeros before position 0), as (C, W-1)."""
    p0 = case.req_starts[r]
    H = case.cache.shape[1]
    ws, N = case.ws, case.block_size
    cols = []
    for src in range(p0 - (W - 1), p0):
        if src < 0:
            cols.append(torch.zeros(H * ws, dtype=torch.bfloat16))
            continue
        blk = int(case.block_table[r, src // N])
        cols.append(case.cache[blk, :, src % N, case.off_s:case.off_s + ws].reshape(-1))
    return torch.stack(cols, dim=1)


def _run_paged(case, cache=None):
    cache = case.cache.clone() if cache is None else cache
    out, err = oracle.paged_sconv_fwd(case.x, case.weight, cache, case.positions,
                                      case.block_table, case.seq_idx, case.slot_mapping,
                                      case.query_start, case.off_s, case.ws,
                                      case.block_size, case.activation, case.use_residual)
    return out, cache, err


@pytest.mark.parametrize("width", [2, 3, 4, 5])
@pytest.mark.parametrize("silu,residual", [(True, True), (False, False), (True, False)])
def test_paged_matches_reference_formulation_per_request(width, silu, residual):
    lengths, starts = [5, 1, 4, 9, 1], [0, 13, 2, 30, 1]
    case = _small_paged(111 + width, lengths, starts, width=width,
                        activation="silu" if silu else None, use_residual=residual)
    out, _, err = _run_paged(case)
    assert err == 0
    q = case.query_start_loc.tolist()
    for r in range(len(lengths)):
        xs = case.x[q[r]:q[r + 1]].t()
        ref = r1_reference(xs, case.weight, None, _history(case, r, width), silu)
        if residual:
            ref = ref + xs.to(torch.float64)
        assert_bf16_close(out[q[r]:q[r + 1]].t(), ref)


def test_paged_exact_integers_match_numpy_correlate():
    g = torch.Generator().manual_seed(9)
    lengths, starts = [6, 1, 4, 2], [0, 9, 1, 21]
    case = _small_paged(121, lengths, starts, activation=None, use_residual=False)
    case.x.copy_(torch.randint(-3, 4, case.x.shape, generator=g).to(torch.bfloat16))
    case.weight.copy_(torch.randint(-2, 3, case.weight.shape, generator=g).to(torch.bfloat16))
    case.cache.copy_(torch.randint(-3, 4, case.cache.shape, generator=g).to(torch.bfloat16))
    out, _, _ = _run_paged(case)
    q = case.query_start_loc.tolist()
    for r in range(len(lengths)):
        hist = _history(case, r, 4).to(torch.int64).numpy()
        for c in range(case.x.shape[1]):
            u = np.concatenate([hist[c], case.x[q[r]:q[r + 1], c].to(torch.int64).numpy()])
            want = np.correlate(u, case.weight[c].to(torch.int64).numpy(), "valid")
            got = out[q[r]:q[r + 1], c].to(torch.int64).numpy()
            assert np.array_equal(got, want), (r, c)


def test_paged_cache_insert_is_exact_scatter():
    case = _small_paged(131, [5, 1, 4, 3], [0, 6, 3, 17], interior_pad_frac=0.2, pad_rows=3,
                        pad_multiple=8)
    before = case.cache.clone()
    _, after, _ = _run_paged(case)
    want = before.clone()
    H, ws, N = case.cache.shape[1], case.ws, case.block_size
    for t in range(case.T):
        s = int(case.slot_mapping[t])
        if s < 0:
            continue
        want[s // N, :, s % N, case.off_s:case.off_s + ws] = case.x[t].reshape(H, ws)
    assert torch.equal(after.view(torch.int16), want.view(torch.int16))


def test_paged_pad_rows_are_residual_or_zero():
    case = _small_paged(141, [5, 2], [3, 7], interior_pad_frac=0.3, pad_rows=4)
    pads = (case.slot_mapping < 0).nonzero().flatten().tolist()
    assert len(pads) >= 4
    out, _, _ = _run_paged(case)
    for t in pads:
        assert torch.equal(out[t].view(torch.int16), case.x[t].view(torch.int16))
    case.use_residual = False
    out2, _, _ = _run_paged(case)
    for t in pads:
        assert bool((out2[t].float() == 0).all())


def test_paged_in_forward_taps_read_pad_rows_of_their_request():
    """An in-forward tap reads x even when that row is a PAD row (the tap rule
    of "sconv.py" decides by row >= query_start only); PAD rows themselves
    give the residual."""
    case = _small_paged(145, [9, 6, 3], [2, 11, 0], interior_pad_frac=0.3)
    pads = set((case.slot_mapping < 0).nonzero().flatten().tolist())
    assert pads, "the case must hold interior PAD rows"
    out, _, err = _run_paged(case)
    assert err == 0
    q = case.query_start_loc.tolist()
    hit = 0
    for r in range(len(case.req_lengths)):
        xs = case.x[q[r]:q[r + 1]].t()
        ref = r1_reference(xs, case.weight, None, _history(case, r, 4), True)
        ref = ref + xs.to(torch.float64)
        for i, t in enumerate(range(q[r], q[r + 1])):
            if t in pads:
                continue
            hit += any(row in pads for row in range(max(q[r], t - 3), t))
            assert_bf16_close(out[t:t + 1].t(), ref[:, i:i + 1])
    assert hit, "some real token must have a PAD row in its window"


def test_paged_split_requests_equal_one_forward():
    """Running each request's tokens as several consecutive forwards (cache
    carried between them) gives the same outputs and cache as one forward."""
    lengths, starts = [7, 1, 5], [2, 11, 0]
    one = _small_paged(151, lengths, starts)
    out_one, cache_one, _ = _run_paged(one)
    cache = one.cache.clone()
    outs = []
    for cut in ((0, 3), (3, 7)):
        parts = []
        for r, (L, p0) in enumerate(zip(lengths, starts)):
            a, b = cut[0], min(cut[1], L)
            if a < b:
                parts.append((r, a, b))
        rows, pos, sidx, slots, qs = [], [], [], [], []
        q = one.query_start_loc.tolist()
        row = 0
        for r, a, b in parts:
            for i in range(a, b):
                rows.append(q[r] + i)
                pos.append(starts[r] + i)
                sidx.append(r)
                slots.append(int(one.slot_mapping[q[r] + i]))
                qs.append(row)
            row += b - a
        x = one.x[rows].contiguous()
        out, err = oracle.paged_sconv_fwd(
            x, one.weight, cache, torch.tensor(pos), one.block_table,
            torch.tensor(sidx, dtype=torch.int32), torch.tensor(slots),
            torch.tensor(qs, dtype=torch.int32), one.off_s, one.ws, one.block_size,
            one.activation, one.use_residual)
        assert err == 0
        outs.append((rows, out))
    for rows, out in outs:
        assert torch.equal(out.view(torch.int16), out_one[rows].view(torch.int16))
    assert torch.equal(cache.view(torch.int16), cache_one.view(torch.int16))


def test_paged_equals_prefill_with_cached_history():
    """With no PAD rows and no residual, each request's paged output equals the
    varlen prefill with bias 0 and the cached history as its initial state."""
    lengths, starts = [6, 1, 4], [1, 20, 0]
    case = _small_paged(161, lengths, starts, use_residual=False)
    out, _, _ = _run_paged(case)
    q = case.query_start_loc.tolist()
    for r in range(3):
        hist = _history(case, r, 4)
        states = hist.unsqueeze(0).contiguous()
        xs = case.x[q[r]:q[r + 1]].t()
        o = wl.empty_like_layout(xs)
        oracle.ccv_fwd(xs, case.weight, None, states,
                       torch.tensor([0, q[r + 1] - q[r]], dtype=torch.int32), None,
                       torch.ones(1, dtype=torch.bool), "silu", -1, out=o)
        assert torch.equal(o.view(torch.int16), out[q[r]:q[r + 1]].t().view(torch.int16))


def test_paged_streams_with_equal_inputs_agree_slice_by_slice():
    """Streams that share inputs and histories but own different D-ranges
    give identical outputs, and the cache is the initial cache with every real token's x
    scattered into each stream's slice at its slot (nothing else changes)."""
    base = _small_paged(460, [5, 1, 9], [0, 7, 3], D=40, off_s=0)
    ws, N = base.ws, base.block_size
    H = base.cache.shape[1]
    offs = (0, ws, 3 * ws)
    for off in offs[1:]:  # equal histories: every stream's slice starts as stream 0's
        base.cache[..., off:off + ws] = base.cache[..., :ws]
    streams = [{"x": base.x, "weight": base.weight, "off_s": off, "ws": ws} for off in offs]
    cache = base.cache.clone()
    outs, err = oracle.paged_sconv_fwd_streams(
        streams, cache, base.positions, base.block_table, base.seq_idx, base.slot_mapping,
        base.query_start, base.block_size, base.activation, base.use_residual)
    assert err == 0
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))
    expected = base.cache.clone()
    for t in range(base.x.shape[0]):
        slot = int(base.slot_mapping[t])
        if slot < 0:
            continue
        for off in offs:
            expected[slot // N, :, slot % N, off:off + ws] = base.x[t].view(H, ws)
    assert torch.equal(cache.view(torch.int16), expected.view(torch.int16))


def test_paged_taps_past_the_block_table_use_its_last_column():
    """A cached tap whose logical block lies past the block table reads the
    table's last column at the same offset in the block ("sconv.py",
    `_fused_sconv_kernel`, the clamp to MAX_BLOCKS - 1)."""
    case = wl.paged_past_table(151)
    out, _, err = _run_paged(case)
    assert err == 0
    W, N, ws = case.weight.shape[1], case.block_size, case.ws
    last = case.block_table.shape[1] - 1
    for r in range(case.T):
        p0 = int(case.positions[r])
        cols = []
        for src in range(p0 - (W - 1), p0):
            assert src // N > last
            blk = int(case.block_table[r, last])
            cols.append(case.cache[blk, :, src % N, case.off_s:case.off_s + ws].reshape(-1))
        xs = case.x[r:r + 1].t()
        ref = r1_reference(xs, case.weight, None, torch.stack(cols, dim=1), True)
        assert_bf16_close(out[r:r + 1].t(), ref + xs.to(torch.float64))


def test_paged_invalid_block_is_counted():
    case = _small_paged(171, [2, 1], [5, 9])
    case.block_table[1, :] = 10_000
    _, _, err = _run_paged(case)
    assert err > 0


# --------------------------------------------------------------- metadata ----

@pytest.mark.parametrize("lengths", [[3, 0, 5, 1], [1], [7, 7, 7, 7, 7], [0, 0, 4], [2, 9, 0]])
@pytest.mark.parametrize("extra", [0, 5])
def test_metadata_matches_searchsorted(lengths, extra):
    qsl = wl.cumulative(lengths)
    n_req = len(lengths)
    n_act = int(qsl[-1])
    n_pad = n_act + extra
    seq = torch.full((n_pad + 3,), 99, dtype=torch.int32)
    qs = torch.full((n_pad + 3,), 99, dtype=torch.int32)
    oracle.paged_sconv_seq_metadata(qsl, n_req, n_act, seq, qs, n_pad)
    t = np.arange(n_act)
    want_seq = np.searchsorted(qsl[:n_req].numpy(), t, side="right") - 1
    assert seq[:n_act].tolist() == want_seq.tolist()
    assert qs[:n_act].tolist() == qsl.numpy()[want_seq].tolist()
    assert seq[n_act:n_pad].tolist() == [0] * extra
    assert qs[n_act:n_pad].tolist() == [0] * extra
    assert seq[n_pad:].tolist() == [99] * 3


def test_metadata_rejects_bad_padding():
    qsl = wl.cumulative([2, 3])
    buf = torch.zeros(8, dtype=torch.int32)
    with pytest.raises(ValueError):
        oracle.paged_sconv_seq_metadata(qsl, 2, 5, buf, buf.clone(), 4)
    with pytest.raises(ValueError):
        oracle.paged_sconv_seq_metadata(qsl, 2, 5, buf, buf.clone(), 9)
