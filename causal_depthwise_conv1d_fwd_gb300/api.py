"""Python binding of the C ABI: argument marshalling only.

Every function takes CUDA tensors, reads their pointers and strides, and
calls the entry point of the same name in libccv.so on the current (or given)
stream.  No arithmetic of the method happens here and there is no CPU path:
CPU tensors are rejected.
"""
from __future__ import annotations

import ctypes
from typing import Optional

import torch

from . import _lib

PAD_SLOT_ID = -1


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need_cuda(t: Optional[torch.Tensor], name: str, dtype=None):
    if t is None:
        return
    if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
        raise TypeError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def _index_vector(t: Optional[torch.Tensor], name: str, dtype, length: Optional[int] = None):
    if t is None:
        return None
    _need_cuda(t, name)
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != 1 or t.stride(0) != 1:
        raise ValueError(f"{name} must be a contiguous 1-D tensor")
    if length is not None and t.numel() < length:
        raise ValueError(f"{name} has {t.numel()} entries, needs {length}")
    return t


def _bias_vector(bias: Optional[torch.Tensor], dim: int):
    """The C ABI reads bias as `dim` contiguous values: reject any other
    shape or a strided view (a column of a packed parameter, say)."""
    if bias is None:
        return None
    if bias.shape != (dim,):
        raise ValueError(f"bias must have shape ({dim},), got {tuple(bias.shape)}")
    if dim > 1 and bias.stride(0) != 1:
        raise ValueError(f"bias must be contiguous (stride 1), got stride {bias.stride(0)}")
    return bias


def _device_of(tensors) -> torch.device:
    """The one device that every given tensor lives on (other items skipped)."""
    devs = {t.device for t in tensors if isinstance(t, torch.Tensor)}
    if len(devs) != 1:
        raise ValueError("all tensors of a call must be on one device, got "
                         + ", ".join(sorted(str(d) for d in devs)))
    return devs.pop()


def _stream(stream, device: int) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    return ctypes.c_void_p(handle)


def _silu_flag(activation) -> int:
    if activation is None or activation is False:
        return 0
    if activation is True or activation in ("silu", "swish"):
        return 1
    raise ValueError(f"unsupported activation: {activation!r}")


def _check(status: int, where: str):
    if status != 0:
        raise _lib.CcvError(status, where)


class Launch:
    """A pre-marshalled call of one entry point: the tensors' pointers, strides
    and sizes are converted once, so each call costs one ctypes call.  The
    tensors must stay alive and keep their storage while the plan is used.
    The call runs on the tensors' device (made current for the call if it is
    not) and, by default, on that device's current stream."""

    def __init__(self, name: str, args: tuple, result, keep: tuple):
        self.name = name
        self._fn = getattr(_lib.load(), name)
        self._args = args
        self.result = result
        self._keep = keep
        self.device = _device_of(keep).index

    def __call__(self, stream=None):
        if torch.cuda.current_device() != self.device:
            with torch.cuda.device(self.device):
                return self._launch(stream)
        return self._launch(stream)

    def _launch(self, stream):
        _check(self._fn(*self._args, _stream(stream, self.device)), self.name)
        return self.result


def ccv_fwd(x: torch.Tensor, weight: torch.Tensor, bias: Optional[torch.Tensor],
            conv_states: Optional[torch.Tensor], query_start_loc: torch.Tensor,
            cache_indices: Optional[torch.Tensor] = None,
            has_initial_state: Optional[torch.Tensor] = None, activation="silu",
            pad_slot_id: int = PAD_SLOT_ID, out: Optional[torch.Tensor] = None,
            err_count: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Varlen causal depthwise conv1d prefill with conv_state (continuous batching).

    x is logically (dim, total_tokens) bf16 in either layout; out defaults to
    an empty tensor with x's strides.  conv_states (num_lines, dim, >= W-1) is
    updated in place.  Returns out.
    """
    return prepare_ccv_fwd(x, weight, bias, conv_states, query_start_loc, cache_indices,
                           has_initial_state, activation, pad_slot_id, out, err_count)(stream)


def prepare_ccv_fwd(x, weight, bias, conv_states, query_start_loc, cache_indices=None,
                    has_initial_state=None, activation="silu", pad_slot_id=PAD_SLOT_ID,
                    out=None, err_count=None) -> Launch:
    """Validate and marshal a ccv_fwd call once; returns a reusable Launch."""
    _need_cuda(x, "x", torch.bfloat16)
    _need_cuda(weight, "weight", torch.bfloat16)
    _need_cuda(bias, "bias", torch.bfloat16)
    _need_cuda(conv_states, "conv_states", torch.bfloat16)
    if x.dim() != 2 or weight.dim() != 2:
        raise ValueError("x must be (dim, total_tokens) and weight (dim, width)")
    dim, total = x.shape
    width = weight.shape[1]
    if weight.shape[0] != dim:
        raise ValueError("weight does not match dim")
    bias = _bias_vector(bias, dim)
    qsl = _index_vector(query_start_loc, "query_start_loc", torch.int32)
    batch = qsl.numel() - 1
    ci = _index_vector(cache_indices, "cache_indices", torch.int32, batch)
    hi = has_initial_state
    if hi is not None:
        if hi.dtype not in (torch.bool, torch.uint8):
            raise TypeError("has_initial_state must be bool or uint8")
        hi = _index_vector(hi, "has_initial_state", hi.dtype, batch)
    if conv_states is not None:
        if conv_states.dim() != 3 or conv_states.shape[1] != dim:
            raise ValueError("conv_states must be (num_cache_lines, dim, state_len)")
        ss = conv_states.stride()
        nl, sl = conv_states.shape[0], conv_states.shape[2]
    else:
        ss, nl, sl = (0, 0, 0), 0, 0
    if out is None:
        out = torch.empty_strided(x.shape, x.stride(), dtype=x.dtype, device=x.device)
    else:
        _need_cuda(out, "out", torch.bfloat16)
        if out.shape != x.shape:
            raise ValueError("out must have x's shape")
    _need_cuda(err_count, "err_count", torch.int32)
    args = (_ptr(x), x.stride(0), x.stride(1), _ptr(out), out.stride(0), out.stride(1),
            _ptr(weight), weight.stride(0), weight.stride(1), _ptr(bias),
            _ptr(conv_states), ss[0], ss[1], ss[2], nl, sl,
            _ptr(qsl), batch, _ptr(ci), _ptr(hi), dim, total, width, pad_slot_id,
            _silu_flag(activation), _ptr(err_count))
    return Launch("ccv_fwd", args, out,
                  (x, weight, bias, conv_states, qsl, ci, hi, out, err_count))


def ccv_update(x: torch.Tensor, conv_state: torch.Tensor, weight: torch.Tensor,
               bias: Optional[torch.Tensor] = None, activation=None,
               conv_state_indices: Optional[torch.Tensor] = None,
               pad_slot_id: int = PAD_SLOT_ID, out: Optional[torch.Tensor] = None,
               err_count: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Decode step.  x is (batch, dim) or (batch, dim, seqlen); out defaults to
    x itself (in place).  conv_state (num_lines, dim, state_len) is shifted in
    place.  Returns out with x's rank."""
    return prepare_ccv_update(x, conv_state, weight, bias, activation, conv_state_indices,
                              pad_slot_id, out, err_count)(stream)


def prepare_ccv_update(x, conv_state, weight, bias=None, activation=None,
                       conv_state_indices=None, pad_slot_id=PAD_SLOT_ID, out=None,
                       err_count=None) -> Launch:
    """Validate and marshal a ccv_update call once; returns a reusable Launch."""
    _need_cuda(x, "x", torch.bfloat16)
    _need_cuda(conv_state, "conv_state", torch.bfloat16)
    _need_cuda(weight, "weight", torch.bfloat16)
    _need_cuda(bias, "bias", torch.bfloat16)
    squeeze = x.dim() == 2
    x3 = x.unsqueeze(-1) if squeeze else x
    if x3.dim() != 3:
        raise ValueError("x must be (batch, dim) or (batch, dim, seqlen)")
    batch, dim, seqlen = x3.shape
    width = weight.shape[1]
    if weight.shape[0] != dim or conv_state.dim() != 3 or conv_state.shape[1] != dim:
        raise ValueError("weight / conv_state do not match dim")
    bias = _bias_vector(bias, dim)
    if out is None:
        out3 = x3
    else:
        _need_cuda(out, "out", torch.bfloat16)
        out3 = out.unsqueeze(-1) if out.dim() == 2 else out
        if out3.shape != x3.shape:
            raise ValueError("out must have x's shape")
    idx = _index_vector(conv_state_indices, "conv_state_indices", torch.int32, batch)
    _need_cuda(err_count, "err_count", torch.int32)
    ss = conv_state.stride()
    args = (_ptr(x3), *x3.stride(), _ptr(out3), *out3.stride(),
            _ptr(weight), weight.stride(0), weight.stride(1), _ptr(bias),
            _ptr(conv_state), ss[0], ss[1], ss[2], conv_state.shape[0], conv_state.shape[2],
            _ptr(idx), batch, dim, seqlen, width, pad_slot_id, _silu_flag(activation),
            _ptr(err_count))
    result = out3.squeeze(-1) if squeeze else out3
    return Launch("ccv_update", args, result,
                  (x3, out3, weight, bias, conv_state, idx, err_count))


def ccv_update_spec(x: torch.Tensor, conv_state: torch.Tensor, weight: torch.Tensor,
                    bias: Optional[torch.Tensor] = None, activation=None,
                    conv_state_indices: Optional[torch.Tensor] = None,
                    num_accepted_tokens: Optional[torch.Tensor] = None,
                    intermediate_conv_window: Optional[torch.Tensor] = None,
                    output_state_indices: Optional[torch.Tensor] = None,
                    pad_slot_id: int = PAD_SLOT_ID, out: Optional[torch.Tensor] = None,
                    err_count: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Decode / speculative-verify step with the spec-decoding extras.

    num_accepted_tokens: int32 [batch] (window read at column value-1);
    intermediate_conv_window: bf16 (batch, steps >= seqlen, dim, width-1),
    receives the window after every token; output_state_indices: int32
    (batch, steps >= seqlen), the state line each step's window is written
    to (-1: none).  With either buffer the state is not shifted in place.
    """
    return prepare_ccv_update_spec(x, conv_state, weight, bias, activation, conv_state_indices,
                                   num_accepted_tokens, intermediate_conv_window,
                                   output_state_indices, pad_slot_id, out, err_count)(stream)


def prepare_ccv_update_spec(x, conv_state, weight, bias=None, activation=None,
                            conv_state_indices=None, num_accepted_tokens=None,
                            intermediate_conv_window=None, output_state_indices=None,
                            pad_slot_id=PAD_SLOT_ID, out=None, err_count=None) -> Launch:
    """Validate and marshal a ccv_update_spec call once; returns a reusable Launch."""
    _need_cuda(x, "x", torch.bfloat16)
    _need_cuda(conv_state, "conv_state", torch.bfloat16)
    _need_cuda(weight, "weight", torch.bfloat16)
    _need_cuda(bias, "bias", torch.bfloat16)
    squeeze = x.dim() == 2
    x3 = x.unsqueeze(-1) if squeeze else x
    if x3.dim() != 3:
        raise ValueError("x must be (batch, dim) or (batch, dim, seqlen)")
    batch, dim, seqlen = x3.shape
    width = weight.shape[1]
    if weight.shape[0] != dim or conv_state.dim() != 3 or conv_state.shape[1] != dim:
        raise ValueError("weight / conv_state do not match dim")
    bias = _bias_vector(bias, dim)
    if out is None:
        out3 = x3
    else:
        _need_cuda(out, "out", torch.bfloat16)
        out3 = out.unsqueeze(-1) if out.dim() == 2 else out
        if out3.shape != x3.shape:
            raise ValueError("out must have x's shape")
    idx = _index_vector(conv_state_indices, "conv_state_indices", torch.int32, batch)
    nacc = _index_vector(num_accepted_tokens, "num_accepted_tokens", torch.int32, batch)
    inter = intermediate_conv_window
    _need_cuda(inter, "intermediate_conv_window", torch.bfloat16)
    if inter is not None and (inter.dim() != 4 or inter.shape[0] != batch or
                              inter.shape[2] != dim or inter.shape[3] != width - 1):
        raise ValueError("intermediate_conv_window must be (batch, steps, dim, width-1)")
    oidx = output_state_indices
    _need_cuda(oidx, "output_state_indices", torch.int32)
    if oidx is not None and (oidx.dim() != 2 or oidx.shape[0] != batch):
        raise ValueError("output_state_indices must be (batch, steps)")
    _need_cuda(err_count, "err_count", torch.int32)
    ss = conv_state.stride()
    ist = inter.stride() if inter is not None else (0, 0, 0, 0)
    ost = oidx.stride() if oidx is not None else (0, 0)
    args = (_ptr(x3), *x3.stride(), _ptr(out3), *out3.stride(),
            _ptr(weight), weight.stride(0), weight.stride(1), _ptr(bias),
            _ptr(conv_state), ss[0], ss[1], ss[2], conv_state.shape[0], conv_state.shape[2],
            _ptr(idx), _ptr(nacc),
            _ptr(inter), *ist, inter.shape[1] if inter is not None else 0,
            _ptr(oidx), *ost, oidx.shape[1] if oidx is not None else 0,
            batch, dim, seqlen, width, pad_slot_id, _silu_flag(activation), _ptr(err_count))
    result = out3.squeeze(-1) if squeeze else out3
    return Launch("ccv_update_spec", args, result,
                  (x3, out3, weight, bias, conv_state, idx, nacc, inter, oidx, err_count))


def paged_sconv_seq_metadata(query_start_loc: torch.Tensor, num_reqs: int,
                             num_actual_tokens: int, seq_idx_out: torch.Tensor,
                             query_start_out: torch.Tensor,
                             num_padded_tokens: Optional[int] = None, stream=None) -> None:
    """Fill the per-token request id and first x-row buffers in one launch."""
    prepare_paged_sconv_seq_metadata(query_start_loc, num_reqs, num_actual_tokens,
                                     seq_idx_out, query_start_out, num_padded_tokens)(stream)


def prepare_paged_sconv_seq_metadata(query_start_loc, num_reqs, num_actual_tokens,
                                     seq_idx_out, query_start_out,
                                     num_padded_tokens=None) -> Launch:
    """Validate and marshal a paged_sconv_seq_metadata call once."""
    if num_padded_tokens is None:
        num_padded_tokens = num_actual_tokens
    qsl = _index_vector(query_start_loc, "query_start_loc", torch.int32, num_reqs)
    seq = _index_vector(seq_idx_out, "seq_idx_out", torch.int32)
    qs = _index_vector(query_start_out, "query_start_out", torch.int32)
    cap = min(seq.numel(), qs.numel())
    args = (_ptr(qsl), num_reqs, num_actual_tokens, num_padded_tokens, _ptr(seq), _ptr(qs), cap)
    return Launch("paged_sconv_seq_metadata", args, None, (qsl, seq, qs))


def paged_sconv_fwd(x: torch.Tensor, weight: torch.Tensor, cache: torch.Tensor,
                    positions: torch.Tensor, block_table: torch.Tensor, seq_idx: torch.Tensor,
                    slot_mapping: torch.Tensor, query_start: torch.Tensor, off_s: int, ws: int,
                    block_size: int, activation=None, use_residual: bool = True,
                    out: Optional[torch.Tensor] = None,
                    err_count: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Single-launch paged insert + depthwise causal conv.  Returns out [T, H*ws]."""
    return prepare_paged_sconv_fwd(x, weight, cache, positions, block_table, seq_idx,
                                   slot_mapping, query_start, off_s, ws, block_size,
                                   activation, use_residual, out, err_count)(stream)


def prepare_paged_sconv_fwd(x, weight, cache, positions, block_table, seq_idx, slot_mapping,
                            query_start, off_s, ws, block_size, activation=None,
                            use_residual=True, out=None, err_count=None) -> Launch:
    """Validate and marshal a paged_sconv_fwd call once; returns a reusable Launch."""
    _need_cuda(x, "x", torch.bfloat16)
    _need_cuda(weight, "weight", torch.bfloat16)
    _need_cuda(cache, "cache", torch.bfloat16)
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be [T, C] with channel stride 1")
    if cache.dim() != 4 or cache.stride(3) != 1:
        raise ValueError("cache must be [num_blocks, H, N, D] with D stride 1")
    num_blocks, H, N, D = cache.shape
    if N != block_size:
        raise ValueError("block_size does not match the cache's N")
    T, C = x.shape
    if C != H * ws or weight.dim() != 2 or weight.shape[0] != C:
        raise ValueError("x / weight channels must equal H * ws")
    width = weight.shape[1]
    pos = _index_vector(positions, "positions", torch.int64, T)
    sidx = _index_vector(seq_idx, "seq_idx", torch.int32, T)
    slots = _index_vector(slot_mapping, "slot_mapping", torch.int64, T)
    qs = _index_vector(query_start, "query_start", torch.int32, T)
    _need_cuda(block_table, "block_table", torch.int32)
    if block_table.dim() != 2 or block_table.stride(1) != 1:
        raise ValueError("block_table must be [num_reqs, max_blocks] with stride 1 along blocks")
    if out is None:
        out = torch.empty_like(x)
    else:
        _need_cuda(out, "out", torch.bfloat16)
        if out.shape != x.shape or out.stride(1) != 1:
            raise ValueError("out must be [T, C] with channel stride 1")
    _need_cuda(err_count, "err_count", torch.int32)
    cs = cache.stride()
    args = (_ptr(x), x.stride(0), _ptr(cache), cs[0], cs[1], cs[2], num_blocks, H, N, D,
            _ptr(weight), weight.stride(0), weight.stride(1), _ptr(out), out.stride(0),
            _ptr(pos), _ptr(sidx), _ptr(slots), _ptr(block_table), block_table.stride(0),
            block_table.shape[0], block_table.shape[1], _ptr(qs), T, off_s, ws, width,
            _silu_flag(activation), int(bool(use_residual)), _ptr(err_count))
    return Launch("paged_sconv_fwd", args, out,
                  (x, weight, cache, pos, sidx, slots, block_table, qs, out, err_count))


def paged_sconv_fwd_with_metadata(x: torch.Tensor, weight: torch.Tensor, cache: torch.Tensor,
                                  positions: torch.Tensor, block_table: torch.Tensor,
                                  query_start_loc: torch.Tensor, num_reqs: int,
                                  num_actual_tokens: int, slot_mapping: torch.Tensor,
                                  off_s: int, ws: int, block_size: int, activation=None,
                                  use_residual: bool = True, out: Optional[torch.Tensor] = None,
                                  seq_idx_out: Optional[torch.Tensor] = None,
                                  query_start_out: Optional[torch.Tensor] = None,
                                  err_count: Optional[torch.Tensor] = None,
                                  stream=None) -> torch.Tensor:
    """paged_sconv_fwd in one launch that resolves each token's request and
    first x-row from query_start_loc itself (and writes them to seq_idx_out
    / query_start_out when given).  Returns out [T, H*ws]."""
    return prepare_paged_sconv_fwd_with_metadata(
        x, weight, cache, positions, block_table, query_start_loc, num_reqs, num_actual_tokens,
        slot_mapping, off_s, ws, block_size, activation, use_residual, out, seq_idx_out,
        query_start_out, err_count)(stream)


def prepare_paged_sconv_fwd_with_metadata(x, weight, cache, positions, block_table,
                                          query_start_loc, num_reqs, num_actual_tokens,
                                          slot_mapping, off_s, ws, block_size, activation=None,
                                          use_residual=True, out=None, seq_idx_out=None,
                                          query_start_out=None, err_count=None) -> Launch:
    """Validate and marshal a paged_sconv_fwd_with_metadata call once."""
    _need_cuda(x, "x", torch.bfloat16)
    _need_cuda(weight, "weight", torch.bfloat16)
    _need_cuda(cache, "cache", torch.bfloat16)
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be [T, C] with channel stride 1")
    if cache.dim() != 4 or cache.stride(3) != 1:
        raise ValueError("cache must be [num_blocks, H, N, D] with D stride 1")
    num_blocks, H, N, D = cache.shape
    if N != block_size:
        raise ValueError("block_size does not match the cache's N")
    T, C = x.shape
    if C != H * ws or weight.dim() != 2 or weight.shape[0] != C:
        raise ValueError("x / weight channels must equal H * ws")
    width = weight.shape[1]
    pos = _index_vector(positions, "positions", torch.int64, T)
    slots = _index_vector(slot_mapping, "slot_mapping", torch.int64, T)
    qsl = _index_vector(query_start_loc, "query_start_loc", torch.int32, num_reqs)
    seq_o = _index_vector(seq_idx_out, "seq_idx_out", torch.int32, T)
    qs_o = _index_vector(query_start_out, "query_start_out", torch.int32, T)
    _need_cuda(block_table, "block_table", torch.int32)
    if block_table.dim() != 2 or block_table.stride(1) != 1:
        raise ValueError("block_table must be [num_reqs, max_blocks] with stride 1 along blocks")
    if out is None:
        out = torch.empty_like(x)
    else:
        _need_cuda(out, "out", torch.bfloat16)
        if out.shape != x.shape or out.stride(1) != 1:
            raise ValueError("out must be [T, C] with channel stride 1")
    _need_cuda(err_count, "err_count", torch.int32)
    cs = cache.stride()
    args = (_ptr(x), x.stride(0), _ptr(cache), cs[0], cs[1], cs[2], num_blocks, H, N, D,
            _ptr(weight), weight.stride(0), weight.stride(1), _ptr(out), out.stride(0),
            _ptr(pos), _ptr(qsl), num_reqs, num_actual_tokens, _ptr(seq_o), _ptr(qs_o),
            _ptr(slots), _ptr(block_table), block_table.stride(0), block_table.shape[0],
            block_table.shape[1], T, off_s, ws, width, _silu_flag(activation),
            int(bool(use_residual)), _ptr(err_count))
    return Launch("paged_sconv_fwd_with_metadata", args, out,
                  (x, weight, cache, pos, qsl, seq_o, qs_o, slots, block_table, out, err_count))


def paged_sconv_fwd_streams(streams, cache: torch.Tensor, positions: torch.Tensor,
                            block_table: torch.Tensor, seq_idx: torch.Tensor,
                            slot_mapping: torch.Tensor, query_start: torch.Tensor,
                            block_size: int, activation=None, use_residual: bool = True,
                            err_count: Optional[torch.Tensor] = None, stream=None):
    """paged_sconv_fwd for several conv streams of one layer in one launch.

    streams: list of dicts with keys x, weight, off_s, ws and optionally out
    (created when missing).  Returns the list of outputs."""
    return prepare_paged_sconv_fwd_streams(streams, cache, positions, block_table, seq_idx,
                                           slot_mapping, query_start, block_size, activation,
                                           use_residual, err_count)(stream)


def prepare_paged_sconv_fwd_streams(streams, cache, positions, block_table, seq_idx,
                                    slot_mapping, query_start, block_size, activation=None,
                                    use_residual=True, err_count=None) -> Launch:
    """Validate and marshal a paged_sconv_fwd_streams call once."""
    _need_cuda(cache, "cache", torch.bfloat16)
    if cache.dim() != 4 or cache.stride(3) != 1:
        raise ValueError("cache must be [num_blocks, H, N, D] with D stride 1")
    num_blocks, H, N, D = cache.shape
    if N != block_size:
        raise ValueError("block_size does not match the cache's N")
    if not 1 <= len(streams) <= 8:
        raise ValueError("between 1 and 8 streams")
    T = streams[0]["x"].shape[0]
    width = streams[0]["weight"].shape[1]
    descs = (_lib.PagedStream * len(streams))()
    outs, keep = [], []
    for i, st in enumerate(streams):
        x, w, ws = st["x"], st["weight"], int(st["ws"])
        _need_cuda(x, f"streams[{i}].x", torch.bfloat16)
        _need_cuda(w, f"streams[{i}].weight", torch.bfloat16)
        if x.dim() != 2 or x.stride(1) != 1 or x.shape[0] != T:
            raise ValueError(f"streams[{i}].x must be [T, C] with channel stride 1")
        if x.shape[1] != H * ws or w.dim() != 2 or w.shape[0] != H * ws or w.shape[1] != width:
            raise ValueError(f"streams[{i}]: x / weight channels must equal H * ws, same width")
        out = st.get("out")
        if out is None:
            out = torch.empty_like(x)
        else:
            _need_cuda(out, f"streams[{i}].out", torch.bfloat16)
            if out.shape != x.shape or out.stride(1) != 1:
                raise ValueError(f"streams[{i}].out must be [T, C] with channel stride 1")
        descs[i] = _lib.PagedStream(x.data_ptr(), x.stride(0), w.data_ptr(), w.stride(0),
                                    w.stride(1), out.data_ptr(), out.stride(0),
                                    int(st["off_s"]), ws)
        outs.append(out)
        keep += [x, w, out]
    pos = _index_vector(positions, "positions", torch.int64, T)
    sidx = _index_vector(seq_idx, "seq_idx", torch.int32, T)
    slots = _index_vector(slot_mapping, "slot_mapping", torch.int64, T)
    qs = _index_vector(query_start, "query_start", torch.int32, T)
    _need_cuda(block_table, "block_table", torch.int32)
    if block_table.dim() != 2 or block_table.stride(1) != 1:
        raise ValueError("block_table must be [num_reqs, max_blocks] with stride 1 along blocks")
    _need_cuda(err_count, "err_count", torch.int32)
    cs = cache.stride()
    args = (ctypes.cast(descs, ctypes.c_void_p), len(streams), _ptr(cache), cs[0], cs[1], cs[2],
            num_blocks, H, N, D, _ptr(pos), _ptr(sidx), _ptr(slots), _ptr(block_table),
            block_table.stride(0), block_table.shape[0], block_table.shape[1], _ptr(qs), T,
            width, _silu_flag(activation), int(bool(use_residual)), _ptr(err_count))
    return Launch("paged_sconv_fwd_streams", args, outs,
                  (descs, cache, pos, sidx, slots, block_table, qs, err_count, *keep))
