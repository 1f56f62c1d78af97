"""Longformer sparse self-attention for one B300 GPU.

The compute path is the CUDA library ``liblfattn.so`` (hand-written sm_103a
kernels behind a C ABI, declared in include/lfattn.h); this package holds
its ctypes binding, the build script and the seeded workload generators.

Calls (one Python function per C entry, same name, argument marshalling only):
  lf_attn_fwd / attention / prepare_fwd   the forward (window, dilation, globals)
  lf_attn_fwd_f32, lf_attn_fwd_host, lf_attn_fwd_noalloc   its fp32, host-buffer
                                          and allocation-free forms
  lf_attn_pairs                           the attended key lists
  lf_attn_fwd_lse, lf_attn_bwd            forward with log-sum-exp, and the backward
  lf_layer_fwd                            one Longformer layer forward
  lf_attn_fwd_bias                        forward with a relative position bias
  lf_attn_fwd_blocks                      forward with extra (random / strided) key blocks
"""
from ._binding import (  # noqa: F401
    LfError, attention, lf_attn_bwd, lf_attn_fwd, lf_attn_fwd_f32, lf_attn_fwd_host,
    lf_attn_fwd_bias, lf_attn_fwd_blocks, lf_attn_fwd_lse, lf_attn_fwd_noalloc,
    lf_attn_get_status, lf_attn_pairs, lf_last_error, lf_launch_count, lf_layer_fwd,
    lf_selftest_wait_timeout,
    lf_plan_cache_clear, lf_profile_enable, lf_profile_only, lf_profile_query, lf_profile_reset,
    lf_version, load_library, LIB_PATH, PreparedFwd, prepare_fwd,
)
