"""GB300-native ZeRO partitioned mixed-precision Adam step over a flat,
padded parameter buffer.

The compute path is libzero (hand-written CUDA for sm_103a behind the C ABI
of include/zero.h); this package only marshals arguments to it.  PyTorch is
used for device memory and streams.
"""
from ._abi import (  # noqa: F401
    LIB_PATH, SIGNATURES, STATUS_NAMES, ZERO_BF16, ZERO_EALIGN, ZERO_ECUDA, ZERO_EINVAL,
    ZERO_ENOMEM, ZERO_ESTATE, ZERO_ETIMEOUT, ZERO_FP16, ZERO_MAX_RANKS, ZERO_NORM_TILE, ZERO_OK,
    ZeroError,
    load, zero_adam_step, zero_adam_step_range, zero_allgather_params, zero_gather_layer,
    zero_last_error,
    zero_memory_report, zero_partition_stats, zero_plan_check, zero_plan_create,
    zero_plan_destroy, zero_plan_fragments, zero_plan_query, zero_plan_set_loss_scaler,
    zero_plan_unit_shards,
    zero_plan_set_spin_limit, zero_plan_set_state, zero_plan_set_reduce_precision,
    zero_plan_units, zero_reduce_partition, zero_reduce_units, zero_step_result,
    zero_reduce_partitions, zero_adam_step_partitions,
    zero_step_set_global_stats, zero_reduce_partition_noalloc, ZERO_NOALLOC_MAX_ELEMS,
    zero_quantize_shard, zero_gather_layer_quantized, ZERO_QUANT_BLOCK,
    zero_plan_set_gather_quantization, ZERO_QUANT_INT8, ZERO_QUANT_FP8_E4M3,
)
from .plan import ZeroPlan  # noqa: F401
