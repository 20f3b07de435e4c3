"""Bitwise-reproducible int8 QAT linear layer (forward, backward) and its
fixed-order gradient reduction, for one GB300 (sm_103a).

The product is the C-ABI library ``librepro.so`` (declared in
``include/repro.h``); ``repro`` is its thin Python binding with the same
names.  ``inputs`` draws the seeded synthetic workloads.
"""
from .repro import (  # noqa: F401
    REPRO_BWD_DW_ACCUMULATE, REPRO_OK, REPRO_QMAX, REPRO_SCALE_ACT_AMAX,
    REPRO_SCALE_WEIGHT_MEANABS, ReproError, lib, repro_device_check, repro_grad_accum,
    repro_launch_count, repro_linear_bwd, repro_linear_bwd_ws_bytes, repro_linear_fwd,
    repro_linear_fwd_ws_bytes, repro_running_sum, repro_sumsq, repro_sumsq_ws_bytes,
    repro_adamw_step, repro_attn_bwd, repro_attn_bwd_ws_bytes, repro_attn_fwd, repro_attn_fwd_ws_bytes,
    repro_quant_i8, repro_quant_i8_multi, repro_wscale_multi, repro_wscale_multi_ws_bytes,
    repro_selftest, repro_set_launch_cfg, repro_state_hash, repro_state_hash_ws_bytes, repro_status_str,
    repro_treefold, repro_version, repro_wait_probe, repro_wscale, repro_wscale_ws_bytes,
    REPRO_HASH_LEAF_BYTES, REPRO_DEBUG_CHECK_FINITE, REPRO_ERR_NONFINITE, REPRO_ERR_TIMEOUT,
    repro_set_debug,
)
