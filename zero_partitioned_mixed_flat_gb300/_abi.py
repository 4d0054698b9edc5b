"""Thin ctypes binding of libzero (include/zero.h): argument marshalling only.

Every function keeps the C name.  Device buffers may be passed as torch
tensors (their data_ptr() is used) or as raw integer addresses; `stream` may
be None (the current torch stream), a torch.cuda.Stream, or a raw
cudaStream_t integer.  Failures raise ZeroError with the library's message.
There is no fallback: if libzero.so is missing the import of any entry point
fails loudly.
"""
import ctypes as C
import os
from typing import Optional, Sequence

import numpy as np

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libzero.so")

ZERO_OK, ZERO_EINVAL, ZERO_EALIGN, ZERO_ENOMEM, ZERO_ECUDA, ZERO_ETIMEOUT, ZERO_ESTATE = range(7)
STATUS_NAMES = ["ZERO_OK", "ZERO_EINVAL", "ZERO_EALIGN", "ZERO_ENOMEM", "ZERO_ECUDA",
                "ZERO_ETIMEOUT", "ZERO_ESTATE"]
ZERO_FP16, ZERO_BF16 = 0, 1
ZERO_MAX_RANKS = 1024
ZERO_NORM_TILE = 4096
ZERO_QUANT_INT8, ZERO_QUANT_FP8_E4M3 = 0, 1

# every exported entry point of include/zero.h, with its ctypes signature
_i32, _i64, _f32, _f64, _vp = C.c_int32, C.c_int64, C.c_float, C.c_double, C.c_void_p
SIGNATURES = {
    "zero_plan_create": (_i32, [_i64, _i32, _vp, _i32, _i32, _i32, _vp, _i32, _vp]),
    "zero_plan_query": (_i32, [_vp, _vp, _vp, _vp]),
    "zero_plan_units": (_i32, [_vp, _vp, _vp, _vp]),
    "zero_plan_fragments": (_i32, [_vp, _i32, _i64, _vp, _vp]),
    "zero_plan_unit_shards": (_i32, [_vp, _vp, _vp]),
    "zero_plan_set_loss_scaler": (_i32, [_vp, _i32]),
    "zero_plan_set_state": (_i32, [_vp, _i64, _i32]),
    "zero_plan_set_spin_limit": (_i32, [_vp, _i64]),
    "zero_plan_set_reduce_precision": (_i32, [_vp, _i32]),
    "zero_plan_set_gather_quantization": (_i32, [_vp, _i32]),
    "zero_reduce_partition": (_i32, [_vp, _i32, _vp, _vp, _f32, _i64, _vp]),
    "zero_reduce_units": (_i32, [_vp, _i32, _i32, _i32, _vp, _vp, _f32, _vp]),
    "zero_reduce_partitions": (_i32, [_vp, _i32, _vp, _vp, _vp, _f32, _i64, _vp]),
    "zero_adam_step_partitions": (_i32, [_vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _f32, _f32, _f32,
                                         _f32, _f32, _i32, _f32, _f32, _f64, _i32, _vp]),
    "zero_partition_stats": (_i32, [_vp, _vp, _vp]),
    "zero_step_set_global_stats": (_i32, [_vp, _vp]),
    "zero_adam_step": (_i32, [_vp, _i32, _vp, _vp, _vp, _vp, _vp, _f32, _f32, _f32, _f32,
                              _f32, _i32, _f32, _f32, _f64, _i32, _vp]),
    "zero_adam_step_range": (_i32, [_vp, _i32, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _f32, _f32,
                                    _f32, _f32, _f32, _i32, _f32, _f32, _f64, _i32, _vp]),
    "zero_step_result": (_i32, [_vp, _vp, _vp, _vp, _vp]),
    "zero_plan_check": (_i32, [_vp]),
    "zero_gather_layer": (_i32, [_vp, _i32, _vp, _vp, _vp]),
    "zero_allgather_params": (_i32, [_vp, _vp, _vp, _i64, _vp]),
    "zero_quantize_shard": (_i32, [_vp, _vp, _vp, _vp, _vp]),
    "zero_gather_layer_quantized": (_i32, [_vp, _i32, _vp, _vp, _vp, _vp]),
    "zero_reduce_partition_noalloc": (_i32, [_i32, _i32, _vp, _i64, _f32, _vp, _vp, _vp, _vp]),
    "zero_memory_report": (_i32, [_i64, _i32, _i32, _vp, _vp, _vp]),
    "zero_plan_destroy": (None, [_vp]),
    "zero_last_error": (C.c_char_p, []),
}

_LIB = None


class ZeroError(RuntimeError):
    def __init__(self, code: int, where: str, message: str):
        self.code = code
        self.status = STATUS_NAMES[code] if 0 <= code < len(STATUS_NAMES) else str(code)
        super().__init__("%s: %s (%s)" % (where, self.status, message))


def load():
    """Load libzero.so (built in-tree by build()).  Raises if it is missing."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError("libzero.so is not built (%s): run "
                              "`python -m zero_partitioned_mixed_flat_gb300.build`" % LIB_PATH)
        lib = C.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
    return _LIB


def _check(code: int, where: str):
    if code != ZERO_OK:
        msg = load().zero_last_error()
        raise ZeroError(code, where, msg.decode() if msg else "")


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return int(x.data_ptr())
    if isinstance(x, np.ndarray):
        return int(x.ctypes.data)
    raise TypeError("cannot take the address of %r" % type(x))


def _ptr_array(xs: Sequence):
    return (_vp * len(xs))(*[_ptr(x) for x in xs])


def _stream(s) -> Optional[int]:
    if s is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)


# ---- plan -----------------------------------------------------------------

def zero_plan_create(psi: int, n_ranks: int, tensor_sizes=None, align: int = 128,
                     stage: int = 1, unit_of_tensor=None, lp: int = ZERO_FP16) -> int:
    out = _vp()
    sizes = None if tensor_sizes is None else np.ascontiguousarray(tensor_sizes, np.int64)
    units = None if unit_of_tensor is None else np.ascontiguousarray(unit_of_tensor, np.int32)
    n = 0 if sizes is None else sizes.size
    _check(load().zero_plan_create(psi, n_ranks, _ptr(sizes), n, align, stage, _ptr(units),
                                   lp, C.byref(out)), "zero_plan_create")
    return out.value


def zero_plan_query(plan: int, n_tensors: int = 0):
    psi_p, part = _i64(), _i64()
    offs = np.zeros(max(n_tensors, 1), np.int64)
    _check(load().zero_plan_query(plan, C.byref(psi_p), C.byref(part),
                                  _ptr(offs) if n_tensors else None), "zero_plan_query")
    return psi_p.value, part.value, offs[:n_tensors]


def zero_plan_units(plan: int):
    n = _i32()
    _check(load().zero_plan_units(plan, C.byref(n), None, None), "zero_plan_units")
    offs = np.zeros(n.value + 1, np.int64)
    pads = np.zeros(n.value, np.int64)
    _check(load().zero_plan_units(plan, C.byref(n), _ptr(offs), _ptr(pads)), "zero_plan_units")
    return n.value, offs, pads


def zero_plan_unit_shards(plan: int, n_units: int):
    """(shard length, shard offset in the partition) of every unit."""
    ln = np.zeros(max(n_units, 1), np.int64)
    off = np.zeros(max(n_units, 1), np.int64)
    _check(load().zero_plan_unit_shards(plan, _ptr(ln), _ptr(off)), "zero_plan_unit_shards")
    return ln[:n_units], off[:n_units]


def zero_plan_fragments(plan: int, rank: int) -> np.ndarray:
    cnt = _i64()
    _check(load().zero_plan_fragments(plan, rank, 0, None, C.byref(cnt)), "zero_plan_fragments")
    out = np.zeros((max(cnt.value, 1), 4), np.int64)
    _check(load().zero_plan_fragments(plan, rank, cnt.value, _ptr(out), C.byref(cnt)),
           "zero_plan_fragments")
    return out[:cnt.value]


def zero_plan_set_loss_scaler(plan: int, growth_interval: int):
    _check(load().zero_plan_set_loss_scaler(plan, growth_interval), "zero_plan_set_loss_scaler")


def zero_plan_set_state(plan: int, step: int, good_steps: int = 0):
    _check(load().zero_plan_set_state(plan, step, good_steps), "zero_plan_set_state")


def zero_plan_set_spin_limit(plan: int, polls: int):
    _check(load().zero_plan_set_spin_limit(plan, polls), "zero_plan_set_spin_limit")


def zero_plan_set_reduce_precision(plan: int, accumulate_in_lp: int):
    _check(load().zero_plan_set_reduce_precision(plan, int(accumulate_in_lp)),
           "zero_plan_set_reduce_precision")


def zero_plan_set_gather_quantization(plan: int, fmt: int):
    _check(load().zero_plan_set_gather_quantization(plan, fmt), "zero_plan_set_gather_quantization")


def zero_plan_destroy(plan: int):
    if plan:
        load().zero_plan_destroy(plan)


def zero_last_error() -> str:
    msg = load().zero_last_error()
    return msg.decode() if msg else ""


# ---- the step ---------------------------------------------------------------

def zero_reduce_partition(plan: int, rank: int, grad_slices: Sequence, grad_out,
                          loss_scale: float, bucket_elems: int = 0, stream=None):
    _check(load().zero_reduce_partition(plan, rank, C.cast(_ptr_array(grad_slices), _vp),
                                        _ptr(grad_out), loss_scale, bucket_elems,
                                        _stream(stream)), "zero_reduce_partition")


def zero_reduce_units(plan: int, rank: int, first_unit: int, n_units: int, grad_slices: Sequence,
                      grad_out, loss_scale: float, stream=None):
    _check(load().zero_reduce_units(plan, rank, first_unit, n_units,
                                    C.cast(_ptr_array(grad_slices), _vp), _ptr(grad_out), loss_scale,
                                    _stream(stream)), "zero_reduce_units")


def zero_reduce_partitions(plan: int, ranks: Sequence[int], grad_slices: Sequence[Sequence],
                           grad_out: Sequence, loss_scale: float, bucket_elems: int = 0, stream=None):
    """grad_slices[i]: the N slices of partition ranks[i]; grad_out[i]: its output."""
    rk = np.ascontiguousarray(ranks, np.int32)
    flat = [x for sl in grad_slices for x in sl]
    _check(load().zero_reduce_partitions(plan, int(rk.size), _ptr(rk), C.cast(_ptr_array(flat), _vp),
                                         C.cast(_ptr_array(grad_out), _vp), loss_scale,
                                         int(bucket_elems), _stream(stream)), "zero_reduce_partitions")


def zero_adam_step_partitions(plan: int, ranks: Sequence[int], grad: Sequence, master: Sequence,
                              m: Sequence, v: Sequence, param_out: Sequence, lr: float, beta1: float,
                              beta2: float, eps: float, wd: float, adamw: int, loss_scale: float,
                              clip: float, remote_sumsq: float = 0.0, remote_overflow: int = 0,
                              stream=None):
    rk = np.ascontiguousarray(ranks, np.int32)
    arrs = [C.cast(_ptr_array(x), _vp) for x in (grad, master, m, v, param_out)]
    _check(load().zero_adam_step_partitions(plan, int(rk.size), _ptr(rk), *arrs, lr, beta1, beta2,
                                            eps, wd, int(adamw), loss_scale, clip, remote_sumsq,
                                            int(remote_overflow), _stream(stream)),
           "zero_adam_step_partitions")


def zero_partition_stats(plan: int, stats, stream=None):
    """stats: 2*N float64 (device, managed or pinned host), written on stream."""
    _check(load().zero_partition_stats(plan, _ptr(stats), _stream(stream)), "zero_partition_stats")


def zero_step_set_global_stats(plan: int, stats):
    """stats: the all-reduced 2*N float64 vector (read by the step's decision)."""
    _check(load().zero_step_set_global_stats(plan, _ptr(stats)), "zero_step_set_global_stats")


def zero_adam_step(plan: int, rank: int, grad, master, m, v, param_out, lr: float,
                   beta1: float, beta2: float, eps: float, wd: float, adamw: int,
                   loss_scale: float, clip: float, remote_sumsq: float = 0.0,
                   remote_overflow: int = 0, stream=None):
    _check(load().zero_adam_step(plan, rank, _ptr(grad), _ptr(master), _ptr(m), _ptr(v),
                                 _ptr(param_out), lr, beta1, beta2, eps, wd, int(adamw),
                                 loss_scale, clip, remote_sumsq, int(remote_overflow),
                                 _stream(stream)), "zero_adam_step")


def zero_adam_step_range(plan: int, rank: int, begin: int, length: int, grad, master, m, v,
                         param_out, lr: float, beta1: float, beta2: float, eps: float, wd: float,
                         adamw: int, loss_scale: float, clip: float, remote_sumsq: float = 0.0,
                         remote_overflow: int = 0, stream=None):
    _check(load().zero_adam_step_range(plan, rank, begin, length, _ptr(grad), _ptr(master), _ptr(m),
                                       _ptr(v), _ptr(param_out), lr, beta1, beta2, eps, wd,
                                       int(adamw), loss_scale, clip, remote_sumsq,
                                       int(remote_overflow), _stream(stream)), "zero_adam_step_range")


def zero_step_result(plan: int) -> dict:
    norm, skipped, scale, step = _f64(), _i32(), _f32(), _i64()
    _check(load().zero_step_result(plan, C.byref(norm), C.byref(skipped), C.byref(scale),
                                   C.byref(step)), "zero_step_result")
    return {"norm": norm.value, "skipped": skipped.value, "loss_scale": scale.value,
            "step": step.value}


def zero_plan_check(plan: int):
    _check(load().zero_plan_check(plan), "zero_plan_check")


def zero_gather_layer(plan: int, unit: int, shards: Sequence, out, stream=None):
    _check(load().zero_gather_layer(plan, unit, C.cast(_ptr_array(shards), _vp), _ptr(out),
                                    _stream(stream)), "zero_gather_layer")


def zero_allgather_params(plan: int, partitions: Sequence, out, bucket_elems: int = 0,
                          stream=None):
    _check(load().zero_allgather_params(plan, C.cast(_ptr_array(partitions), _vp), _ptr(out),
                                        int(bucket_elems), _stream(stream)),
           "zero_allgather_params")


ZERO_QUANT_BLOCK = 128


def zero_quantize_shard(plan: int, shard, codes, scales, stream=None):
    _check(load().zero_quantize_shard(plan, _ptr(shard), _ptr(codes), _ptr(scales),
                                      _stream(stream)), "zero_quantize_shard")


def zero_gather_layer_quantized(plan: int, unit: int, codes: Sequence, scales: Sequence, out,
                                stream=None):
    _check(load().zero_gather_layer_quantized(plan, unit, C.cast(_ptr_array(codes), _vp),
                                              C.cast(_ptr_array(scales), _vp), _ptr(out),
                                              _stream(stream)), "zero_gather_layer_quantized")


ZERO_NOALLOC_MAX_ELEMS = 65536 * ZERO_NORM_TILE


def zero_reduce_partition_noalloc(n_ranks: int, lp: int, grad_slices: Sequence, length: int,
                                  loss_scale: float, grad_out, sumsq_out, overflow_out,
                                  stream=None):
    """Allocation-free reduce of one partition (see include/zero.h): for callers
    that cannot allocate device memory.  sumsq_out: device float64[1];
    overflow_out: device int32[1]."""
    _check(load().zero_reduce_partition_noalloc(n_ranks, lp, C.cast(_ptr_array(grad_slices), _vp),
                                                length, loss_scale, _ptr(grad_out),
                                                _ptr(sumsq_out), _ptr(overflow_out),
                                                _stream(stream)), "zero_reduce_partition_noalloc")


def zero_memory_report(psi: int, n_ranks: int, align: int = 1):
    formula = np.zeros(4, np.float64)
    actual = np.zeros(4, np.int64)
    comm = np.zeros(4, np.int64)
    _check(load().zero_memory_report(psi, n_ranks, align, _ptr(formula), _ptr(actual),
                                     _ptr(comm)), "zero_memory_report")
    return formula, actual, comm
