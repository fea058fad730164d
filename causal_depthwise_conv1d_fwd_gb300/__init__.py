"""GB300-native causal depthwise conv1d forward: varlen prefill with conv_state,
decode update (with the speculative-decoding extras), and the paged
sliding-window short conv.

The compute path is the hand-written CUDA library ``libccv.so`` (C ABI in
``include/ccv.h``); :mod:`.api` is a thin ctypes binding over it with the same
entry-point names.  Nothing here computes on the CPU: the binding rejects CPU
tensors and raises if the library has not been built.
"""
from .api import (PAD_SLOT_ID, Launch, ccv_fwd, ccv_update, ccv_update_spec,  # noqa: F401
                  paged_sconv_fwd, paged_sconv_fwd_streams, paged_sconv_fwd_with_metadata,
                  paged_sconv_seq_metadata, prepare_ccv_fwd, prepare_ccv_update,
                  prepare_ccv_update_spec, prepare_paged_sconv_fwd,
                  prepare_paged_sconv_fwd_streams, prepare_paged_sconv_fwd_with_metadata,
                  prepare_paged_sconv_seq_metadata)
from ._lib import CcvError  # noqa: F401

__all__ = ["PAD_SLOT_ID", "ccv_fwd", "ccv_update", "ccv_update_spec", "paged_sconv_seq_metadata",
           "paged_sconv_fwd", "paged_sconv_fwd_with_metadata", "paged_sconv_fwd_streams",
           "prepare_paged_sconv_fwd_with_metadata", "prepare_paged_sconv_fwd_streams",
           "prepare_ccv_fwd", "prepare_ccv_update", "prepare_ccv_update_spec",
           "prepare_paged_sconv_seq_metadata", "prepare_paged_sconv_fwd", "Launch",
           "CcvError"]
