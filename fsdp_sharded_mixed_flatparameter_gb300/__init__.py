"""GB300-native flat-shard optimizer step (ZeRO-1/2/3, FSDP FlatParameter).

The compute path is libzeroshard (hand-written sm_103a CUDA kernels behind a
C ABI, include/zero_shard.h); this package is its ctypes binding plus a small
orchestrator.  Build the library with ``__graft_entry__.build()`` (or
``python -m fsdp_sharded_mixed_flatparameter_gb300.build``).
"""
from .zero_shard import (  # noqa: F401
    DeviceLossScale, DynamicLossScale, ZERO_BF16, ZERO_EINVAL, ZERO_ECUDA, ZERO_F16, ZERO_F32, ZERO_OK, NormResult, ZeroError, decode_norm_result,
    device_table, lib, new_norm_result, zero_accum, zero_reduce_chunks, zero_adamw_step, zero_adamw_step_tensors, zero_flatten_cast, zero_grad_sqnorm,
    zero_grad_sqnorm_combine, zero_grad_sqnorm_finalize, zero_grad_sqnorm_noalloc, zero_grad_sqnorm_workspace_bytes, zero_shard_range, zero_tensor_table, sqnorm_view,
    AdamwDeviceState, decode_adamw_device_state, device_hparams, new_adamw_device_state, zero_adamw_prepare_device,
    zero_adamw_scalars, zero_adamw_step_device, zero_adamw_step_tensors_device, zero_loss_scale_update_device)
from .optimizer import FlatShardAdamW, gather_sqnorms, torch_stream  # noqa: F401
from .dataplane import ZeroDataPlane, ZeroUnits, chunk_layout, exchange_chunks, gather_shards  # noqa: F401
