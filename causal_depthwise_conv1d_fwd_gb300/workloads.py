"""Seeded synthetic workloads for the causal depthwise conv1d forward family.

This module only draws inputs; it holds none of the method's arithmetic, so
both the CUDA path and the CPU oracle can be fed the very same bits from it.
Every tensor is created on the CPU from a seeded ``torch.Generator``; callers
copy to the device themselves.

Value distribution: every bf16 tensor is N(0, 0.02^2), the recipe of the
atrex-bench #003 ``causal_conv1d`` input generator (x, weight, bias and the
initial state all ``randn * 0.02``).

Layouts:

* ``x`` for the varlen prefill is logically ``(dim, total_tokens)``.  The
  ``"tokens_dim"`` layout stores it channel-last (the tokenspeed wrapper's
  ``is_channel_last`` case, stride(0) == 1); ``"dim_tokens"`` stores it
  channel-first (stride(1) == 1, as the atrex-bench generator does).
* ``conv_states`` is logically ``(num_cache_lines, dim, state_len)`` with
  column 0 the oldest.  ``"dim_contiguous"`` (the default) gives stride(1) == 1,
  the layout the tokenspeed decode wrapper asserts; ``"tok_contiguous"`` is the
  plain contiguous tensor.

The named configurations mirror the five benchmark workloads: a single short
sequence, a varlen continuous-batching prefill, a decode step, a large
prefill, and the paged sliding-window short conv.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List, Optional

import torch

BF16 = torch.bfloat16
STD = 0.02
PAD_SLOT_ID = -1


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(int(seed))
    return g


def randn_bf16(shape, g: torch.Generator, std: float = STD) -> torch.Tensor:
    return (torch.randn(shape, generator=g, dtype=torch.float32) * std).to(BF16)


def make_x(dim: int, total_tokens: int, layout: str, g: torch.Generator,
           std: float = STD) -> torch.Tensor:
    """x of logical shape (dim, total_tokens) in the requested memory layout."""
    if layout == "tokens_dim":
        return randn_bf16((total_tokens, dim), g, std).t()
    if layout == "dim_tokens":
        return randn_bf16((dim, total_tokens), g, std)
    raise ValueError(f"unknown x layout {layout!r}")


def make_states(num_lines: int, dim: int, state_len: int, layout: str,
                g: torch.Generator, std: float = STD) -> torch.Tensor:
    """conv_state pool of logical shape (num_lines, dim, state_len)."""
    if layout == "dim_contiguous":
        return randn_bf16((num_lines, state_len, dim), g, std).transpose(1, 2)
    if layout == "tok_contiguous":
        return randn_bf16((num_lines, dim, state_len), g, std)
    raise ValueError(f"unknown state layout {layout!r}")


def empty_like_layout(x: torch.Tensor) -> torch.Tensor:
    return torch.empty_strided(x.shape, x.stride(), dtype=x.dtype, device=x.device)


def cumulative(lengths: List[int]) -> torch.Tensor:
    """query_start_loc: running offsets with a leading 0 (int32)."""
    offs = [0]
    for n in lengths:
        offs.append(offs[-1] + int(n))
    return torch.tensor(offs, dtype=torch.int32)


# --------------------------------------------------------------- prefill ----

@dataclass
class PrefillCase:
    name: str
    x: torch.Tensor
    weight: torch.Tensor
    bias: Optional[torch.Tensor]
    conv_states: Optional[torch.Tensor]
    query_start_loc: torch.Tensor
    cache_indices: Optional[torch.Tensor]
    has_initial_state: Optional[torch.Tensor]
    activation: Optional[str]
    pad_slot_id: int = PAD_SLOT_ID
    lengths: List[int] = field(default_factory=list)

    @property
    def dim(self) -> int:
        return self.x.shape[0]

    @property
    def total_tokens(self) -> int:
        return self.x.shape[1]

    @property
    def width(self) -> int:
        return self.weight.shape[1]

    def kwargs(self) -> Dict:
        return dict(x=self.x, weight=self.weight, bias=self.bias,
                    conv_states=self.conv_states,
                    query_start_loc=self.query_start_loc,
                    cache_indices=self.cache_indices,
                    has_initial_state=self.has_initial_state,
                    activation=self.activation, pad_slot_id=self.pad_slot_id)


def varlen_prefill(seed: int, lengths: List[int], dim: int, width: int = 4, *,
                   num_cache_lines: Optional[int] = None, layout: str = "tokens_dim",
                   state_layout: str = "dim_contiguous", state_len: Optional[int] = None,
                   pad_positions=(), has_init: str = "bernoulli", use_bias: bool = True,
                   activation: Optional[str] = "silu", with_states: bool = True,
                   with_cache_indices: bool = True, extra_tokens: int = 0,
                   std: float = STD, name: str = "varlen") -> PrefillCase:
    """A varlen continuous-batching prefill batch.

    ``has_init`` is ``"bernoulli"`` (each sequence 0/1 with p=0.5), ``"all"``,
    ``"none"`` (all False) or ``"null"`` (no has_initial_state tensor at all).
    ``pad_positions`` lists batch entries whose cache index is the pad id.
    ``extra_tokens`` appends unowned tokens after the last sequence.
    """
    g = _gen(seed)
    batch = len(lengths)
    total = sum(lengths) + extra_tokens
    state_len = width - 1 if state_len is None else state_len
    if num_cache_lines is None:
        num_cache_lines = max(batch, 1)
    x = make_x(dim, total, layout, g, std)
    weight = randn_bf16((dim, width), g, std)
    bias = randn_bf16((dim,), g, std) if use_bias else None
    conv_states = (make_states(num_cache_lines, dim, state_len, state_layout, g, std)
                   if with_states else None)
    if with_cache_indices:
        perm = torch.randperm(num_cache_lines, generator=g)[:batch].to(torch.int32)
        for p in pad_positions:
            perm[p] = PAD_SLOT_ID
        cache_indices = perm
    else:
        cache_indices = None
    if has_init == "bernoulli":
        hi = torch.rand(batch, generator=g) < 0.5
    elif has_init == "all":
        hi = torch.ones(batch, dtype=torch.bool)
    elif has_init == "none":
        hi = torch.zeros(batch, dtype=torch.bool)
    elif has_init == "null":
        hi = None
    else:
        raise ValueError(has_init)
    return PrefillCase(name=name, x=x, weight=weight, bias=bias, conv_states=conv_states,
                       query_start_loc=cumulative(lengths), cache_indices=cache_indices,
                       has_initial_state=hi, activation=activation, lengths=list(lengths))


def config_single(seed: int = 1000) -> PrefillCase:
    """One sequence, dim 64, W 4, 16 tokens, channel-first x, initial state (1,64,3)."""
    return varlen_prefill(seed, [16], 64, 4, num_cache_lines=1, layout="dim_tokens",
                          has_init="all", with_cache_indices=False, name="single_dim64_T16")


# (tokens, dim) of the atrex-bench #003 "causal_conv1d" shape table.
ATREX_SHAPES = ((1, 4096), (128, 4096), (256, 4096), (514, 4096), (1024, 4096),
                (1, 8192), (4195, 8192), (11027, 8192), (14807, 8192))


def config_atrex(tokens: int, dim: int, seed: int = 1006) -> PrefillCase:
    """One channel-first sequence as in the atrex-bench #003 generator: x
    (dim, tokens), weight (dim, 4), bias and initial state, all randn * 0.02,
    SiLU on."""
    return varlen_prefill(seed + tokens + dim, [tokens], dim, 4, num_cache_lines=1,
                          layout="dim_tokens", has_init="all", with_cache_indices=False,
                          name=f"atrex_T{tokens}_dim{dim}")


def varlen_lengths(seed: int, batch: int = 8, lo: int = 1, hi: int = 512) -> List[int]:
    g = _gen(seed + 7919)
    return [int(v) for v in torch.randint(lo, hi + 1, (batch,), generator=g)]


def config_varlen(seed: int = 1001, layout: str = "tokens_dim") -> PrefillCase:
    """8 sequences, lengths U[1,512], dim 4096, pool of 64 lines, one pad entry."""
    lengths = varlen_lengths(seed)
    g = _gen(seed + 104729)
    pad_at = int(torch.randint(0, len(lengths), (1,), generator=g))
    return varlen_prefill(seed, lengths, 4096, 4, num_cache_lines=64, layout=layout,
                          pad_positions=(pad_at,), has_init="bernoulli",
                          name="varlen_8seq_dim4096")


def config_large_prefill(seed: int = 1003, layout: str = "tokens_dim",
                         seqs: int = 4, seqlen: int = 4096, dim: int = 8192) -> PrefillCase:
    """4 sequences x 4096 tokens (16384 total), dim 8192, all with initial state."""
    return varlen_prefill(seed, [seqlen] * seqs, dim, 4, num_cache_lines=seqs, layout=layout,
                          has_init="all", name=f"prefill_{seqs}x{seqlen}_dim{dim}_{layout}")


# ---------------------------------------------------------------- decode ----

@dataclass
class DecodeCase:
    name: str
    x: torch.Tensor                 # (batch, dim) or (batch, dim, seqlen)
    weight: torch.Tensor
    bias: Optional[torch.Tensor]
    conv_state: torch.Tensor        # (num_lines, dim, state_len)
    conv_state_indices: Optional[torch.Tensor]
    activation: Optional[str]
    pad_slot_id: int = PAD_SLOT_ID

    def kwargs(self) -> Dict:
        return dict(x=self.x, conv_state=self.conv_state, weight=self.weight,
                    bias=self.bias, activation=self.activation,
                    conv_state_indices=self.conv_state_indices,
                    pad_slot_id=self.pad_slot_id)


def decode(seed: int, batch: int, dim: int, width: int = 4, *, num_lines: Optional[int] = None,
           seqlen: int = 1, state_len: Optional[int] = None,
           state_layout: str = "dim_contiguous", pad_positions=(), use_bias: bool = True,
           activation: Optional[str] = "silu", with_indices: bool = True,
           squeeze: bool = True, std: float = STD, name: str = "decode") -> DecodeCase:
    g = _gen(seed)
    num_lines = 2 * batch if num_lines is None else num_lines
    state_len = (width - 2 + seqlen) if state_len is None else state_len
    if squeeze and seqlen == 1:
        x = randn_bf16((batch, dim), g, std)
    else:
        x = randn_bf16((batch, dim, seqlen), g, std)
    weight = randn_bf16((dim, width), g, std)
    bias = randn_bf16((dim,), g, std) if use_bias else None
    conv_state = make_states(num_lines, dim, state_len, state_layout, g, std)
    if with_indices:
        idx = torch.randperm(num_lines, generator=g)[:batch].to(torch.int32)
        for p in pad_positions:
            idx[p] = PAD_SLOT_ID
    else:
        idx = None
    return DecodeCase(name=name, x=x, weight=weight, bias=bias, conv_state=conv_state,
                      conv_state_indices=idx, activation=activation)


def config_decode(seed: int = 1002) -> DecodeCase:
    """256 single-token rows, dim 8192, state pool (512, 8192, 3)."""
    return decode(seed, 256, 8192, 4, num_lines=512, name="decode_256x8192")


@dataclass
class SpecDecodeCase:
    """Speculative verify step: seqlen draft tokens per row, the state holding
    history columns, and the page's optional spec-decoding buffers."""
    name: str
    x: torch.Tensor                          # (batch, dim, seqlen)
    weight: torch.Tensor
    bias: Optional[torch.Tensor]
    conv_state: torch.Tensor                 # (num_lines, dim, state_len)
    conv_state_indices: Optional[torch.Tensor]
    num_accepted_tokens: Optional[torch.Tensor]      # int32 [batch], values >= 1
    intermediate_conv_window: Optional[torch.Tensor]  # bf16 (batch, steps, dim, width-1)
    output_state_indices: Optional[torch.Tensor]      # int32 (batch, steps)
    activation: Optional[str]
    pad_slot_id: int = PAD_SLOT_ID

    def kwargs(self) -> Dict:
        return dict(x=self.x, conv_state=self.conv_state, weight=self.weight,
                    bias=self.bias, activation=self.activation,
                    conv_state_indices=self.conv_state_indices,
                    num_accepted_tokens=self.num_accepted_tokens,
                    intermediate_conv_window=self.intermediate_conv_window,
                    output_state_indices=self.output_state_indices,
                    pad_slot_id=self.pad_slot_id)


def spec_decode(seed: int, batch: int, dim: int, width: int = 4, seqlen: int = 4, *,
                num_lines: Optional[int] = None, history: int = 4,
                with_accepted: bool = True, with_intermediate: bool = False,
                with_output_indices: bool = False, steps: Optional[int] = None,
                skip_frac: float = 0.25, pad_positions=(), use_bias: bool = True,
                activation: Optional[str] = "silu", std: float = STD,
                name: str = "spec_decode") -> SpecDecodeCase:
    """Random verify step.  The state keeps width-1+history columns, so up to
    history+1 accepted tokens can be addressed; without intermediate or
    output buffers it is widened to the width-2+seqlen columns the in-place
    shift writes.  Input lines are a random subset of the pool; output lines
    (when asked for) are drawn from the rest, about skip_frac of them -1.
    The intermediate buffer starts as random values, so untouched entries are
    recognisable."""
    g = _gen(seed)
    steps = seqlen if steps is None else steps
    if num_lines is None:  # room for the input lines and distinct output lines
        num_lines = max(3 * batch * max(1, seqlen), batch * (steps + 3))
    state_len = width - 1 + history
    if not (with_intermediate or with_output_indices):
        state_len = max(state_len, width - 2 + seqlen)
    # channels contiguous (x.stride(1) == 1), the layout the page's update
    # wrapper asserts
    x = randn_bf16((batch, seqlen, dim), g, std).transpose(1, 2)
    weight = randn_bf16((dim, width), g, std)
    bias = randn_bf16((dim,), g, std) if use_bias else None
    conv_state = make_states(num_lines, dim, state_len, "dim_contiguous", g, std)
    perm = torch.randperm(num_lines, generator=g).to(torch.int32)
    idx = perm[:batch].clone()
    for p in pad_positions:
        idx[p] = PAD_SLOT_ID
    nacc = None
    if with_accepted:
        nacc = torch.randint(1, history + 2, (batch,), generator=g, dtype=torch.int32)
    inter = None
    if with_intermediate:
        inter = randn_bf16((batch, width - 1, steps, dim), g, std).permute(0, 2, 3, 1)
    oidx = None
    if with_output_indices:
        pool = perm[batch:]
        if pool.numel() < batch * steps:
            raise ValueError("num_lines too small for distinct output lines")
        oidx = pool[: batch * steps].reshape(batch, steps).clone()
        drop = torch.rand((batch, steps), generator=g) < skip_frac
        oidx[drop] = -1
    return SpecDecodeCase(name=name, x=x, weight=weight, bias=bias, conv_state=conv_state,
                          conv_state_indices=idx, num_accepted_tokens=nacc,
                          intermediate_conv_window=inter, output_state_indices=oidx,
                          activation=activation)


def config_spec_decode(seed: int = 1005) -> SpecDecodeCase:
    """Speculative verify: 64 rows x 4 draft tokens, dim 8192, W 4, history of
    4 columns, num_accepted_tokens in [1, 5], per-step windows written to an
    intermediate buffer and scattered to output state lines."""
    return spec_decode(seed, 64, 8192, 4, 4, num_lines=768, history=4, with_accepted=True,
                       with_intermediate=True, with_output_indices=True,
                       name="spec_verify_64x4_dim8192")


# ----------------------------------------------------------------- paged ----

@dataclass
class PagedCase:
    name: str
    x: torch.Tensor                 # [T_padded, C]
    weight: torch.Tensor            # [C, W]
    cache: torch.Tensor             # [num_blocks, H, N, D]
    positions: torch.Tensor         # int64 [T_padded]
    block_table: torch.Tensor       # int32 [num_reqs, max_blocks]
    seq_idx: torch.Tensor           # int32 [T_padded], by construction
    slot_mapping: torch.Tensor      # int64 [T_padded], -1 = PAD
    query_start: torch.Tensor       # int32 [T_padded], by construction
    query_start_loc: torch.Tensor   # int32 [num_reqs + 1]
    num_actual_tokens: int
    off_s: int
    ws: int
    block_size: int
    activation: Optional[str]
    use_residual: bool
    req_lengths: List[int] = field(default_factory=list)
    req_starts: List[int] = field(default_factory=list)

    @property
    def T(self) -> int:
        return self.x.shape[0]

    def kwargs(self) -> Dict:
        return dict(x=self.x, weight=self.weight, cache=self.cache,
                    positions=self.positions, block_table=self.block_table,
                    seq_idx=self.seq_idx, slot_mapping=self.slot_mapping,
                    query_start=self.query_start, off_s=self.off_s, ws=self.ws,
                    block_size=self.block_size, activation=self.activation,
                    use_residual=self.use_residual)


def paged(seed: int, req_lengths: List[int], req_starts: List[int], *, H: int, ws: int,
          N: int, D: int, num_blocks: int, off_s: int, width: int = 4,
          max_blocks: Optional[int] = None, interior_pad_frac: float = 0.0,
          pad_rows: int = 0, pad_multiple: int = 1, activation: Optional[str] = "silu",
          use_residual: bool = True, std: float = STD, name: str = "paged") -> PagedCase:
    """A paged short-conv forward over requests laid out back to back.

    Request r holds ``req_lengths[r]`` tokens at absolute positions
    ``req_starts[r] ..``.  Every (request, logical block) pair that the forward
    writes or reads gets its own physical block, drawn without replacement from
    one permutation, so no slot written by this forward is a pre-forward tap of
    another token.  Unused block-table entries hold random (in-range) ids.
    ``interior_pad_frac`` turns that fraction of real tokens into PAD rows
    (slot -1); ``pad_rows`` appends trailing padded rows (slot -1, seq_idx 0,
    query_start 0), and the padded count is rounded up to ``pad_multiple``.
    """
    g = _gen(seed)
    num_reqs = len(req_lengths)
    C = H * ws
    need = []
    for L, p0 in zip(req_lengths, req_starts):
        lo = max(p0 - (width - 1), 0) // N
        hi = (p0 + L - 1) // N
        need.append((lo, hi))
    top = max(hi for _, hi in need) if need else 0
    if max_blocks is None:
        max_blocks = top + 1
    if max_blocks <= top:
        raise ValueError("max_blocks too small for the requested positions")
    total_needed = sum(hi - lo + 1 for lo, hi in need)
    if total_needed > num_blocks:
        raise ValueError(f"workload needs {total_needed} blocks > {num_blocks}")
    block_table = torch.randint(0, num_blocks, (max(num_reqs, 1), max_blocks),
                                generator=g, dtype=torch.int32)
    perm = torch.randperm(num_blocks, generator=g).to(torch.int32)
    k = 0
    for r, (lo, hi) in enumerate(need):
        for lb in range(lo, hi + 1):
            block_table[r, lb] = perm[k]
            k += 1

    positions, seq_idx, slots, qstart = [], [], [], []
    row = 0
    for r, (L, p0) in enumerate(zip(req_lengths, req_starts)):
        for i in range(L):
            pos = p0 + i
            positions.append(pos)
            seq_idx.append(r)
            slots.append(int(block_table[r, pos // N]) * N + pos % N)
            qstart.append(row)
        row += L
    T_actual = row
    T_padded = T_actual + pad_rows
    if pad_multiple > 1:
        T_padded = -(-T_padded // pad_multiple) * pad_multiple
    for _ in range(T_padded - T_actual):
        positions.append(0)
        seq_idx.append(0)
        slots.append(PAD_SLOT_ID)
        qstart.append(0)
    slots_t = torch.tensor(slots, dtype=torch.int64)
    if interior_pad_frac > 0 and T_actual > 0:
        n_pad = max(1, int(round(interior_pad_frac * T_actual)))
        which = torch.randperm(T_actual, generator=g)[:n_pad]
        slots_t[which] = PAD_SLOT_ID

    x = randn_bf16((T_padded, C), g, std)
    weight = randn_bf16((C, width), g, std)
    cache = randn_bf16((num_blocks, H, N, D), g, std)
    return PagedCase(
        name=name, x=x, weight=weight, cache=cache,
        positions=torch.tensor(positions, dtype=torch.int64),
        block_table=block_table, seq_idx=torch.tensor(seq_idx, dtype=torch.int32),
        slot_mapping=slots_t, query_start=torch.tensor(qstart, dtype=torch.int32),
        query_start_loc=cumulative(req_lengths), num_actual_tokens=T_actual,
        off_s=off_s, ws=ws, block_size=N, activation=activation,
        use_residual=use_residual, req_lengths=list(req_lengths),
        req_starts=list(req_starts))


def paged_past_table(seed: int, *, H: int = 2, ws: int = 128, N: int = 16, D: int = 256,
                     num_blocks: int = 16, off_s: int = 128, width: int = 4, top: int = 5,
                     num_reqs: int = 3) -> PagedCase:
    """Decode requests whose cached window lies in logical block ``top`` while
    the block table has only ``top`` columns, so every cached tap's logical
    block is past the table (the conv clamps it to the last column).

    Request r is one token at position top*N + (width-1) + r, so its earlier
    taps sit in block ``top``.  The table's last column points each request
    at a physical block that no insert of the call writes, so the clamped
    taps read data that is stable during the call.
    """
    if N < width - 1 + num_reqs:
        raise ValueError("block too small for the requested positions")
    starts = [top * N + (width - 1) + r for r in range(num_reqs)]
    case = paged(seed, [1] * num_reqs, starts, H=H, ws=ws, N=N, D=D, num_blocks=num_blocks,
                 off_s=off_s, width=width, name="paged_past_table")
    written = {int(s) // N for s in case.slot_mapping.tolist() if s >= 0}
    free = [b for b in range(num_blocks) if b not in written]
    table = case.block_table[:, :top].clone().contiguous()
    for r in range(num_reqs):
        table[r, top - 1] = free[r]
    case.block_table = table
    return case


def paged_mix(seed: int, num_reqs: int = 32, prefill_lo: int = 64, prefill_hi: int = 1024,
              max_start: int = 2048, N: int = 16, num_blocks: int = 1024,
              width: int = 4):
    """Request lengths and start positions for the mixed paged workload.

    About a quarter prefill (length U[prefill_lo, prefill_hi]), half decode
    (1 token) and a quarter speculative (4 tokens), at random absolute start
    positions in [0, max_start]; three requests are forced to start at 0, 1
    and 2 so that taps before position 0 occur.  Prefill lengths are redrawn
    until the touched blocks fit in ``num_blocks``.
    """
    g = _gen(seed + 31337)
    n_pre = num_reqs // 4
    n_spec = num_reqs // 4
    kinds = ["prefill"] * n_pre + ["spec"] * n_spec + ["decode"] * (num_reqs - n_pre - n_spec)
    order = torch.randperm(num_reqs, generator=g).tolist()
    kinds = [kinds[i] for i in order]
    for _ in range(100):
        lengths, starts = [], []
        for kind in kinds:
            if kind == "prefill":
                lengths.append(int(torch.randint(prefill_lo, prefill_hi + 1, (1,), generator=g)))
            elif kind == "spec":
                lengths.append(4)
            else:
                lengths.append(1)
            starts.append(int(torch.randint(0, max_start + 1, (1,), generator=g)))
        for r, p in zip(range(min(3, num_reqs)), (0, 1, 2)):
            starts[r] = p
        blocks = sum((p + L - 1) // N - max(p - (width - 1), 0) // N + 1
                     for L, p in zip(lengths, starts))
        if blocks <= num_blocks:
            return lengths, starts
    raise RuntimeError("could not fit the paged workload into the block budget")


def config_paged(seed: int = 1004, num_blocks: int = 1024) -> PagedCase:
    """H=16 x ws=128 (C=2048), W=4, cache [1024,16,16,512], stream offset 128,
    32 mixed requests, ~2% PAD rows (half interior, half trailing), T padded to 8."""
    lengths, starts = paged_mix(seed, num_blocks=num_blocks)
    T_actual = sum(lengths)
    n_pad = max(2, int(round(0.02 * T_actual)))
    trailing = n_pad // 2
    interior = (n_pad - trailing) / max(T_actual, 1)
    return paged(seed, lengths, starts, H=16, ws=128, N=16, D=512, num_blocks=num_blocks,
                 off_s=128, width=4, max_blocks=(2048 + 1024) // 16 + 8,
                 interior_pad_frac=interior, pad_rows=trailing, pad_multiple=8,
                 activation="silu", use_residual=True, name="paged_H16_ws128_32req")


def paged_streams(base: PagedCase, seed: int, offsets, ws: int, std: float = STD):
    """Conv streams sharing base's cache and token metadata: stream i owns
    D-range [offsets[i], offsets[i] + ws).  Stream 0 reuses base's x and
    weight; the others draw their own."""
    g = _gen(seed)
    T, C = base.x.shape
    H = base.cache.shape[1]
    if C != H * ws:
        raise ValueError("base channels must equal H * ws")
    streams = []
    for i, off in enumerate(offsets):
        if i == 0:
            x, w = base.x, base.weight
        else:
            x = randn_bf16((T, C), g, std)
            w = randn_bf16((C, base.weight.shape[1]), g, std)
        streams.append({"x": x, "weight": w, "off_s": int(off), "ws": ws})
    return streams


def config_paged_streams(seed: int = 1007):
    """A layer's four conv streams (K, V, attn-output, mlp-output): the paged
    workload's requests and cache [1024, 16, 16, 512], each stream 128
    channels per head at D offsets 0, 128, 256, 384.  Returns (base case,
    streams)."""
    lengths, starts = paged_mix(seed, num_blocks=1024)
    T_actual = sum(lengths)
    n_pad = max(2, int(round(0.02 * T_actual)))
    trailing = n_pad // 2
    base = paged(seed, lengths, starts, H=16, ws=128, N=16, D=512, num_blocks=1024, off_s=0,
                 width=4, max_blocks=(2048 + 1024) // 16 + 8,
                 interior_pad_frac=(n_pad - trailing) / max(T_actual, 1), pad_rows=trailing,
                 pad_multiple=8, activation="silu", use_residual=True,
                 name="paged_4streams_H16_ws128_32req")
    return base, paged_streams(base, seed + 7, (0, 128, 256, 384), 128)
