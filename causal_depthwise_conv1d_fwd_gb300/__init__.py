"""GB300-native causal depthwise conv1d forward: varlen prefill with conv_state,
single-token decode update, and the paged sliding-window short conv.

The compute path is the hand-written CUDA library ``libccv.so`` (C ABI in
``include/ccv.h``); this package is a thin ctypes binding over it.
"""
