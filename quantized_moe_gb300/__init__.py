"""ds4moe: forward pass of a quantized Mixture-of-Experts layer on one GB300 (sm_103a).

The compute lives in the C-ABI library ``lib/libds4moe.so`` (hand-written CUDA, built by
``quantized_moe_gb300.build``); ``quantized_moe_gb300.ds4moe`` is its ctypes binding.
"""
from . import ds4moe  # noqa: F401
from .ds4moe import (DS4MOE_FMT_Q2_K, DS4MOE_FMT_Q8_0, Ds4MoeError, ds4moe_create, ds4moe_destroy,  # noqa: F401
                     ds4moe_forward, ds4moe_forward_ex, ds4moe_forward_host, ds4moe_get_route,
                     ds4moe_get_stats, ds4moe_last_error, make_shapes, make_weights)
