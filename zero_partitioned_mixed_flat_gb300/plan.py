"""ZeroPlan: an owning handle around a libzero plan (marshalling only)."""
from typing import Optional, Sequence

from . import _abi as A


class ZeroPlan:
    """Owns one `zero_plan *`.  Methods map one-to-one onto the C calls."""

    def __init__(self, psi: int, n_ranks: int, tensor_sizes: Optional[Sequence[int]] = None,
                 align: int = 128, stage: int = 1, unit_of_tensor=None, lp: int = A.ZERO_FP16,
                 growth_interval: Optional[int] = None):
        self.handle = A.zero_plan_create(psi, n_ranks, tensor_sizes, align, stage,
                                         unit_of_tensor, lp)
        self.n_ranks, self.stage, self.lp, self.align = n_ranks, stage, lp, align
        self.n_tensors = 0 if tensor_sizes is None else len(tensor_sizes)
        self.psi_padded, self.part_len, self.tensor_offsets = A.zero_plan_query(
            self.handle, self.n_tensors)
        self.n_units, self.unit_offsets, self.unit_padded = A.zero_plan_units(self.handle)
        self.shard_lens, self.shard_offsets = A.zero_plan_unit_shards(self.handle, self.n_units)
        if growth_interval is not None:
            A.zero_plan_set_loss_scaler(self.handle, growth_interval)

    # lifetime
    def close(self):
        if self.handle:
            A.zero_plan_destroy(self.handle)
            self.handle = 0

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # layout
    def fragments(self, rank: int):
        return A.zero_plan_fragments(self.handle, rank)

    def keep_ranges(self, rank: int):
        """(partition offset, length) of every non-padding run of rank's partition."""
        return [(int(f[2]), int(f[3])) for f in self.fragments(rank)]

    def shard_len(self, unit: int) -> int:
        return int(self.shard_lens[unit])

    def unit_shard_offset(self, unit: int) -> int:
        return int(self.shard_offsets[unit])

    # the step
    def reduce(self, rank, grad_slices, grad_out, loss_scale, bucket_elems=0, stream=None):
        A.zero_reduce_partition(self.handle, rank, grad_slices, grad_out, loss_scale,
                                bucket_elems, stream)

    def reduce_many(self, ranks, grad_slices, grad_out, loss_scale, bucket_elems=0, stream=None):
        A.zero_reduce_partitions(self.handle, ranks, grad_slices, grad_out, loss_scale, bucket_elems,
                                 stream)

    def adam_many(self, ranks, grad, master, m, v, param_out, lr, beta1, beta2, eps, wd, adamw,
                  loss_scale, clip, remote_sumsq=0.0, remote_overflow=0, stream=None):
        A.zero_adam_step_partitions(self.handle, ranks, grad, master, m, v, param_out, lr, beta1,
                                    beta2, eps, wd, adamw, loss_scale, clip, remote_sumsq,
                                    remote_overflow, stream)

    def reduce_units(self, rank, first_unit, n_units, grad_slices, grad_out, loss_scale, stream=None):
        A.zero_reduce_units(self.handle, rank, first_unit, n_units, grad_slices, grad_out, loss_scale,
                            stream)

    def partition_stats(self, stats, stream=None):
        """Write this step's per-partition statistics (2*N float64) into `stats`."""
        A.zero_partition_stats(self.handle, stats, stream)

    def set_global_stats(self, stats):
        """Decide this step from the all-reduced statistics vector `stats`."""
        A.zero_step_set_global_stats(self.handle, stats)

    def adam(self, rank, grad, master, m, v, param_out, lr, beta1, beta2, eps, wd, adamw,
             loss_scale, clip, remote_sumsq=0.0, remote_overflow=0, stream=None):
        A.zero_adam_step(self.handle, rank, grad, master, m, v, param_out, lr, beta1, beta2,
                         eps, wd, adamw, loss_scale, clip, remote_sumsq, remote_overflow, stream)

    def adam_range(self, rank, begin, length, grad, master, m, v, param_out, lr, beta1, beta2,
                   eps, wd, adamw, loss_scale, clip, remote_sumsq=0.0, remote_overflow=0,
                   stream=None):
        A.zero_adam_step_range(self.handle, rank, begin, length, grad, master, m, v, param_out,
                               lr, beta1, beta2, eps, wd, adamw, loss_scale, clip, remote_sumsq,
                               remote_overflow, stream)

    def result(self):
        return A.zero_step_result(self.handle)

    def check(self):
        A.zero_plan_check(self.handle)

    def gather(self, unit, shards, out, stream=None):
        A.zero_gather_layer(self.handle, unit, shards, out, stream)

    def allgather(self, partitions, out, bucket_elems=0, stream=None):
        A.zero_allgather_params(self.handle, partitions, out, bucket_elems, stream)

    def quantize(self, shard, codes, scales, stream=None):
        A.zero_quantize_shard(self.handle, shard, codes, scales, stream)

    def gather_quantized(self, unit, codes, scales, out, stream=None):
        A.zero_gather_layer_quantized(self.handle, unit, codes, scales, out, stream)

    def set_state(self, step, good_steps=0):
        A.zero_plan_set_state(self.handle, step, good_steps)

    def set_gather_quantization(self, fmt):
        A.zero_plan_set_gather_quantization(self.handle, fmt)

    def set_reduce_precision(self, accumulate_in_lp):
        A.zero_plan_set_reduce_precision(self.handle, accumulate_in_lp)

    def set_spin_limit(self, polls):
        A.zero_plan_set_spin_limit(self.handle, polls)
