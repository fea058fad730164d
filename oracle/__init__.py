"""CPU oracle for the causal depthwise conv1d forward family.

TEST INFRASTRUCTURE ONLY.  The library's product path never imports this
package; only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline / reference leg may use it.

The arithmetic lives in ``ccv_oracle.c`` (plain scalar loops, fp32 accumulation
as the pages fix it, one round-to-nearest-even to bf16).  This module only
marshals torch CPU tensors into that library through ctypes: it does no
arithmetic of its own.  The pages it follows:

* tokenspeed ``causal_conv1d.py``: ``causal_conv1d_fn`` (varlen prefill with
  conv_state) and ``causal_conv1d_update`` (decode);
* vLLM Inkling ``sconv.py``: ``fused_sconv`` (paged sliding-window short conv)
  and ``sconv_seq_metadata``;
* atrex-bench #003 ``causal_conv1d``: the reference formulation.

Functions mutate ``conv_states`` / ``cache`` in place exactly as the device
entry points do; callers that need the original must clone first.
"""
from __future__ import annotations

import ctypes
from typing import Optional

import torch

from . import build as _build

_LIB = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int


def _lib():
    global _LIB
    if _LIB is None:
        lib = ctypes.CDLL(_build.build())
        lib.oracle_ccv_fwd.argtypes = [
            _P, _I64, _I64, _P, _I64, _I64, _P, _I64, _I64, _P,
            _P, _I64, _I64, _I64, _I32, _P, _I32, _P, _P,
            _I32, _I32, _I32, _I32, _I32, _P]
        lib.oracle_ccv_update.argtypes = [
            _P, _I64, _I64, _I64, _P, _I64, _I64, _I64, _P, _I64, _I64, _P,
            _P, _I64, _I64, _I64, _I32, _P, _I32, _I32, _I32,
            _I32, _I32, _I32, _P]
        lib.oracle_ccv_update_spec.argtypes = [
            _P, _I64, _I64, _I64, _P, _I64, _I64, _I64, _P, _I64, _I64, _P,
            _P, _I64, _I64, _I64, _I32, _I32, _P, _P,
            _P, _I64, _I64, _I64, _I64, _P, _I64, _I64,
            _I32, _I32, _I32, _I32, _I32, _I32, _P]
        lib.oracle_paged_sconv_seq_metadata.argtypes = [_P, _I32, _I32, _I32, _P, _P]
        lib.oracle_paged_sconv_fwd.argtypes = [
            _P, _I64, _P, _I64, _I64, _I64, _I32, _I32, _I32, _I32,
            _P, _I64, _I64, _P, _I64, _P, _P, _P, _P, _I64, _I32, _I32,
            _P, _I32, _I32, _I32, _I32, _I32, _I32, _P]
        lib.oracle_f32_to_bf16.argtypes = [_P, _P, _I64]
        lib.oracle_silu_f32.argtypes = [_P, _P, _I64]
        for name in ("oracle_ccv_fwd", "oracle_ccv_update", "oracle_ccv_update_spec",
                     "oracle_paged_sconv_seq_metadata", "oracle_paged_sconv_fwd"):
            getattr(lib, name).restype = ctypes.c_int
        _LIB = lib
    return _LIB


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    assert t.device.type == "cpu", "the oracle runs on CPU tensors only"
    return ctypes.c_void_p(t.data_ptr())


def _check(t: torch.Tensor, dtype, name):
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")


def _silu_flag(activation) -> int:
    if activation is None or activation is False:
        return 0
    if activation is True or activation in ("silu", "swish"):
        return 1
    raise ValueError(f"unsupported activation: {activation!r}")


def f32_to_bf16_bits(values: torch.Tensor) -> torch.Tensor:
    """Round fp32 values to bf16 with the oracle's own rounding; int16 bit patterns."""
    src = values.contiguous().to(torch.float32)
    dst = torch.empty(src.shape, dtype=torch.int16)
    _lib().oracle_f32_to_bf16(_ptr(src), _ptr(dst), src.numel())
    return dst


def silu_f32(values: torch.Tensor) -> torch.Tensor:
    src = values.contiguous().to(torch.float32)
    dst = torch.empty_like(src)
    _lib().oracle_silu_f32(_ptr(src), _ptr(dst), src.numel())
    return dst


def ccv_fwd(x, weight, bias, conv_states, query_start_loc, cache_indices=None,
            has_initial_state=None, activation="silu", pad_slot_id=-1, out=None):
    """Varlen prefill; x is logically (dim, total_tokens), any strides.

    Returns (out, err_count).  ``out`` defaults to a fresh tensor with x's
    strides whose untouched elements are left as allocated (callers that
    compare skipped rows should pass a sentinel-filled ``out``).
    """
    _check(x, torch.bfloat16, "x")
    dim, total = x.shape
    width = weight.shape[1]
    if out is None:
        out = torch.empty_strided(x.shape, x.stride(), dtype=x.dtype)
    silu = _silu_flag(activation)
    qsl = query_start_loc.to(torch.int32).contiguous()
    batch = qsl.numel() - 1
    ci = None if cache_indices is None else cache_indices.to(torch.int32).contiguous()
    hi = None if has_initial_state is None else has_initial_state.to(torch.uint8).contiguous()
    if conv_states is not None:
        ss = conv_states.stride()
        nl = conv_states.shape[0]
    else:
        ss, nl = (0, 0, 0), 0
    err = ctypes.c_int(0)
    _lib().oracle_ccv_fwd(
        _ptr(x), x.stride(0), x.stride(1), _ptr(out), out.stride(0), out.stride(1),
        _ptr(weight), weight.stride(0), weight.stride(1), _ptr(bias),
        _ptr(conv_states), ss[0], ss[1], ss[2], nl,
        _ptr(qsl), batch, _ptr(ci), _ptr(hi), dim, total, width, pad_slot_id, silu,
        ctypes.byref(err))
    return out, err.value


def ccv_update(x, conv_state, weight, bias=None, activation=None,
               conv_state_indices=None, pad_slot_id=-1, out=None):
    """Decode update; x is (batch, dim) or (batch, dim, seqlen).  out defaults to x.

    Returns (out, err_count).
    """
    _check(x, torch.bfloat16, "x")
    squeeze = x.dim() == 2
    x3 = x.unsqueeze(-1) if squeeze else x
    if out is None:
        out3 = x3
    else:
        out3 = out.unsqueeze(-1) if out.dim() == 2 else out
    batch, dim, seqlen = x3.shape
    width = weight.shape[1]
    silu = _silu_flag(activation)
    idx = None if conv_state_indices is None else conv_state_indices.to(torch.int32).contiguous()
    ss = conv_state.stride()
    err = ctypes.c_int(0)
    _lib().oracle_ccv_update(
        _ptr(x3), *x3.stride(), _ptr(out3), *out3.stride(),
        _ptr(weight), weight.stride(0), weight.stride(1), _ptr(bias),
        _ptr(conv_state), ss[0], ss[1], ss[2], conv_state.shape[0],
        _ptr(idx), batch, dim, seqlen, width, pad_slot_id, silu, ctypes.byref(err))
    res = out3.squeeze(-1) if squeeze else out3
    return res, err.value


def ccv_update_spec(x, conv_state, weight, bias=None, activation=None,
                    conv_state_indices=None, num_accepted_tokens=None,
                    intermediate_conv_window=None, output_state_indices=None,
                    pad_slot_id=-1, out=None):
    """Decode / speculative-verify update with the page's spec-decoding extras.

    x is (batch, dim, seqlen) (or (batch, dim)); out defaults to x.
    num_accepted_tokens: int32 [batch] or None; intermediate_conv_window:
    bf16 (batch, >= seqlen, dim, width-1) or None, written; output_state_indices:
    int32 (batch, >= seqlen) or None.  Returns (out, err_count).
    """
    _check(x, torch.bfloat16, "x")
    squeeze = x.dim() == 2
    x3 = x.unsqueeze(-1) if squeeze else x
    if out is None:
        out3 = x3
    else:
        out3 = out.unsqueeze(-1) if out.dim() == 2 else out
    batch, dim, seqlen = x3.shape
    width = weight.shape[1]
    silu = _silu_flag(activation)
    # keep converted index tensors alive until the call returns
    idx = None if conv_state_indices is None else conv_state_indices.to(torch.int32).contiguous()
    nacc = None if num_accepted_tokens is None else num_accepted_tokens.to(torch.int32).contiguous()
    oidx = None if output_state_indices is None else output_state_indices.to(torch.int32)
    inter = intermediate_conv_window
    if inter is not None:
        _check(inter, torch.bfloat16, "intermediate_conv_window")
    ist = inter.stride() if inter is not None else (0, 0, 0, 0)
    ost = oidx.stride() if oidx is not None else (0, 0)
    ss = conv_state.stride()
    err = ctypes.c_int(0)
    _lib().oracle_ccv_update_spec(
        _ptr(x3), *x3.stride(), _ptr(out3), *out3.stride(),
        _ptr(weight), weight.stride(0), weight.stride(1), _ptr(bias),
        _ptr(conv_state), ss[0], ss[1], ss[2], conv_state.shape[0], conv_state.shape[2],
        _ptr(idx), _ptr(nacc), _ptr(inter), *ist, _ptr(oidx), *ost,
        batch, dim, seqlen, width, pad_slot_id, silu, ctypes.byref(err))
    res = out3.squeeze(-1) if squeeze else out3
    return res, err.value


def paged_sconv_seq_metadata(query_start_loc, num_reqs, num_actual_tokens,
                             seq_idx_out, query_start_out, num_padded_tokens=None):
    if num_padded_tokens is None:
        num_padded_tokens = num_actual_tokens
    if num_padded_tokens < num_actual_tokens:
        raise ValueError("num_padded_tokens must cover all actual tokens")
    if num_padded_tokens > seq_idx_out.shape[0] or num_padded_tokens > query_start_out.shape[0]:
        raise ValueError("output buffers are too small for the padded token count")
    qsl = query_start_loc.to(torch.int32).contiguous()
    _check(seq_idx_out, torch.int32, "seq_idx_out")
    _check(query_start_out, torch.int32, "query_start_out")
    _lib().oracle_paged_sconv_seq_metadata(
        _ptr(qsl), num_reqs, num_actual_tokens, num_padded_tokens,
        _ptr(seq_idx_out), _ptr(query_start_out))


def paged_sconv_fwd(x, weight, cache, positions, block_table, seq_idx, slot_mapping,
                    query_start, off_s, ws, block_size, activation=None,
                    use_residual=True, out=None):
    """Paged sliding-window short conv.  Returns (out, err_count); cache is updated."""
    _check(x, torch.bfloat16, "x")
    T = x.shape[0]
    if out is None:
        out = torch.empty_like(x)
    num_blocks, H, N, D = cache.shape
    assert N == block_size
    assert cache.stride(3) == 1
    width = weight.shape[1]
    _check(block_table, torch.int32, "block_table")
    # keep converted index tensors alive until the call returns
    pos = positions.to(torch.int64).contiguous()
    sidx = seq_idx.to(torch.int32).contiguous()
    slots = slot_mapping.to(torch.int64).contiguous()
    qs = query_start.to(torch.int32).contiguous()
    err = ctypes.c_int(0)
    _lib().oracle_paged_sconv_fwd(
        _ptr(x), x.stride(0), _ptr(cache), cache.stride(0), cache.stride(1), cache.stride(2),
        num_blocks, H, N, D, _ptr(weight), weight.stride(0), weight.stride(1),
        _ptr(out), out.stride(0), _ptr(pos), _ptr(sidx), _ptr(slots),
        _ptr(block_table), block_table.stride(0), block_table.shape[0], block_table.shape[1],
        _ptr(qs), T, off_s, ws, width,
        _silu_flag(activation), int(bool(use_residual)), ctypes.byref(err))
    return out, err.value


def paged_sconv_fwd_streams(streams, cache, positions, block_table, seq_idx, slot_mapping,
                            query_start, block_size, activation=None, use_residual=True):
    """Several conv streams sharing one paged cache (vLLM Inkling sconv.py,
    module docstring): each stream is one fused_sconv call on its own
    D-range, so the definition is the single-stream routine applied to each
    stream in turn.  streams: list of dicts with x, weight, off_s, ws.
    Returns (list of outputs, total err_count); the cache is updated."""
    outs, errs = [], 0
    for st in streams:
        out, err = paged_sconv_fwd(st["x"], st["weight"], cache, positions, block_table,
                                   seq_idx, slot_mapping, query_start, st["off_s"], st["ws"],
                                   block_size, activation, use_residual)
        outs.append(out)
        errs += err
    return outs, errs
