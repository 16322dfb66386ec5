"""GB300-native ZeRO partitioned optimizer step (one data-parallel rank).

The compute path is ``libzero.so`` (CUDA kernels for sm_103a behind the C ABI
of ``include/zero.h``); ``_abi`` binds it with the same function names and
``step`` drives it with the global skip/commit rule.  There is no CPU
fallback: without the built library every entry point raises.
"""
from ._abi import (  # noqa: F401
    ZERO_BF16, ZERO_ERR_ALIGNMENT, ZERO_ERR_CUDA, ZERO_ERR_INVALID_ARG, ZERO_ERR_IO,
    ZERO_ERR_TIMEOUT, ZERO_ERR_UNSUPPORTED, ZERO_F16, ZERO_FUSED_WINDOW_ELEMS,
    ZERO_GATHER_SEGMENTS_PER_LAUNCH, ZERO_OK, ZERO_STATIC_CB_ELEMS, ZERO_STATIC_CB_MAX_BUCKET,
    AdamW, CkptHeader, Grads, Layout, State, ZeroError, adamw, exported_names,
    fused_launch_count, gather_launch_count, grads, streamed_launch_count,
    unfused_launch_count, lib, state, zero_adam_step_shard,
    zero_check_nonfinite, zero_checkpoint_load, zero_checkpoint_read_header,
    zero_checkpoint_save, zero_comm_volume_elems, zero_feed_buckets, zero_gather_params_shard,
    zero_gather_range, zero_model_state_bytes, zero_model_state_bytes_mp,
    zero_partition_layout, zero_reduce_scatter_bucket, zero_status_string, zero_step_shard,
    zero_step_shard_streamed, zero_step_shard_unfused, zero_step_shard_unfused_static)
