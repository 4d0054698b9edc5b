"""ctypes front end of the CPU oracle (test infrastructure only).

Only the tests, the smoke check and the benchmark's CPU-baseline leg may
import this package.  It wraps oracle/liboracle_zero.so (plain C, built by
oracle/build.py) with numpy arrays; it performs no arithmetic of its own.
"""
import ctypes as C
import os

import numpy as np

from . import build as _build

_LIB = None

_i32, _i64, _f32, _f64 = C.c_int32, C.c_int64, C.c_float, C.c_double
_vp = C.c_void_p


class Decision(C.Structure):
    _fields_ = [("norm", _f64), ("coef", _f32), ("skip", _i32),
                ("new_scale", _f32), ("good_steps", _i32), ("step", _i64),
                ("bc1", _f32), ("bc2", _f32)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


def lib():
    """Load (building first if needed) the oracle library."""
    global _LIB
    if _LIB is None:
        # ZERO_ORACLE_LIB lets the mutation test load a deliberately broken copy
        path = os.environ.get("ZERO_ORACLE_LIB") or _build.build()
        L = C.CDLL(path)
        L.orc_half_to_float.argtypes = [C.c_uint16]
        L.orc_half_to_float.restype = _f32
        L.orc_float_to_half.argtypes = [_f32]
        L.orc_float_to_half.restype = C.c_uint16
        L.orc_bf16_to_float.argtypes = [C.c_uint16]
        L.orc_bf16_to_float.restype = _f32
        L.orc_float_to_bf16.argtypes = [_f32]
        L.orc_float_to_bf16.restype = C.c_uint16
        L.orc_lp_array_to_float.argtypes = [_i64, _vp, _i32, _vp]
        L.orc_lp_array_to_float.restype = None
        L.orc_float_array_to_lp.argtypes = [_i64, _vp, _i32, _vp]
        L.orc_float_array_to_lp.restype = None
        L.orc_layout.argtypes = [_i32, _vp, _vp, _i32, _i32, _i32, _vp, _vp, _vp,
                                 _vp, _vp, _vp, _vp]
        L.orc_layout.restype = _i32
        L.orc_partition_to_flat.argtypes = [_i32, _vp, _vp, _i32, _i32, _i32, _i64]
        L.orc_partition_to_flat.restype = _i64
        L.orc_fragments.argtypes = [_i32, _vp, _vp, _i32, _i32, _i32, _i32, _i64, _vp]
        L.orc_fragments.restype = _i64
        L.orc_memory.argtypes = [_i64, _i32, _i32, _vp, _vp, _vp]
        L.orc_memory.restype = _i32
        L.orc_reduce.argtypes = [_i32, _vp, _i32, _i64, _f32, _vp, _vp, _vp]
        L.orc_reduce.restype = None
        L.orc_reduce_lp_accum.argtypes = [_i32, _vp, _i32, _i64, _f32, _vp, _vp, _vp]
        L.orc_reduce_lp_accum.restype = None
        L.orc_decide.argtypes = [_f64, _f64, _i32, _i32, _f32, _f32, _i64, _i32,
                                 _i32, _f32, _f32, C.POINTER(Decision)]
        L.orc_decide.restype = None
        L.orc_adam.argtypes = [_i64, _vp, _vp, _vp, _vp, _vp, _i32, _f32, _i32,
                               _f32, _f32, _f32, _f32, _f32, _i32, _f32, _f32]
        L.orc_adam.restype = None
        L.orc_quantize_blocks.argtypes = [_i64, _vp, _i32, _i32, _vp, _vp]
        L.orc_quantize_blocks.restype = None
        L.orc_dequant_gather.argtypes = [_i32, _vp, _vp, _i64, _i32, _i32, _vp]
        L.orc_dequant_gather.restype = None
        L.orc_gather.argtypes = [_i32, _vp, _i64, _vp]
        L.orc_gather.restype = None
        L.orc_e4m3_decode_array.argtypes = [_i64, _vp, _vp]
        L.orc_e4m3_decode_array.restype = None
        L.orc_e4m3_encode_array.argtypes = [_i64, _vp, _vp]
        L.orc_e4m3_encode_array.restype = None
        L.orc_quantize_blocks_fp8.argtypes = [_i64, _vp, _i32, _i32, _vp, _vp]
        L.orc_quantize_blocks_fp8.restype = None
        L.orc_dequant_gather_fp8.argtypes = [_i32, _vp, _vp, _i64, _i32, _i32, _vp]
        L.orc_dequant_gather_fp8.restype = None
        _LIB = L
    return _LIB


def _ptr(a):
    return a.ctypes.data if a is not None else None


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def _ptr_array(arrays):
    arr = (_vp * len(arrays))(*[a.ctypes.data for a in arrays])
    return arr


# ---- number formats -------------------------------------------------------

def lp_to_float(codes, lp):
    codes = _c(codes, np.uint16)
    out = np.empty(codes.shape, np.float32)
    lib().orc_lp_array_to_float(codes.size, _ptr(codes), lp, _ptr(out))
    return out


def float_to_lp(x, lp):
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().orc_float_array_to_lp(x.size, _ptr(x), lp, _ptr(out))
    return out


# ---- layout ---------------------------------------------------------------

def layout(sizes, n_ranks, align=128, stage=1, unit_of_tensor=None):
    sizes = _c(sizes, np.int64)
    n = sizes.size
    units = None if unit_of_tensor is None else _c(unit_of_tensor, np.int32)
    psi, psi_p, part = _i64(), _i64(), _i64()
    nu = _i32()
    toff = np.zeros(max(n, 1), np.int64)
    uoff = np.zeros(max(n, 1) + 2, np.int64)
    upad = np.zeros(max(n, 1) + 1, np.int64)
    rc = lib().orc_layout(n, _ptr(sizes), _ptr(units), n_ranks, align, stage,
                          C.byref(psi), C.byref(psi_p), C.byref(part), C.byref(nu),
                          _ptr(toff), _ptr(uoff), _ptr(upad))
    if rc != 0:
        raise ValueError("oracle layout rejected the arguments")
    k = nu.value
    return {"psi": psi.value, "psi_padded": psi_p.value, "part_len": part.value,
            "n_units": k, "tensor_offsets": toff[:n].copy(),
            "unit_offsets": uoff[:k + 1].copy(), "unit_padded": upad[:k].copy(),
            "n_ranks": n_ranks, "stage": stage}


def partition_to_flat(lay, rank, k):
    return lib().orc_partition_to_flat(lay["n_units"], _ptr(lay["unit_offsets"]),
                                       _ptr(lay["unit_padded"]), lay["n_ranks"],
                                       lay["stage"], rank, k)


def fragments(sizes, n_ranks, align, stage, rank, unit_of_tensor=None):
    sizes = _c(sizes, np.int64)
    units = None if unit_of_tensor is None else _c(unit_of_tensor, np.int32)
    cnt = lib().orc_fragments(sizes.size, _ptr(sizes), _ptr(units), n_ranks, align,
                              stage, rank, 0, None)
    if cnt < 0:
        raise ValueError("oracle fragments rejected the arguments")
    out = np.zeros((max(cnt, 1), 4), np.int64)
    lib().orc_fragments(sizes.size, _ptr(sizes), _ptr(units), n_ranks, align, stage,
                        rank, cnt, _ptr(out))
    return out[:cnt]


def memory(psi, n_ranks, align=1):
    formula = np.zeros(4, np.float64)
    actual = np.zeros(4, np.int64)
    comm = np.zeros(4, np.int64)
    if lib().orc_memory(psi, n_ranks, align, _ptr(formula), _ptr(actual), _ptr(comm)) != 0:
        raise ValueError("oracle memory rejected the arguments")
    return formula, actual, comm


# ---- the step ---------------------------------------------------------------

def reduce(slices, lp, loss_scale, sumsq=0.0, overflow=0, out=None):
    """slices: list of N equal-length uint16 code arrays.  Returns (g, sumsq, overflow)."""
    slices = [_c(s, np.uint16) for s in slices]
    n = len(slices)
    length = slices[0].size
    g = np.empty(length, np.float32) if out is None else out
    acc = _f64(sumsq)
    of = _i32(overflow)
    lib().orc_reduce(n, C.cast(_ptr_array(slices), _vp), lp, length, loss_scale,
                     _ptr(g), C.byref(acc), C.byref(of))
    return g, acc.value, of.value


def reduce_lp_accum(slices, lp, loss_scale, sumsq=0.0, overflow=0, out=None):
    """Like reduce(), with every partial sum rounded to the lp type."""
    slices = [_c(s, np.uint16) for s in slices]
    n = len(slices)
    length = slices[0].size
    g = np.empty(length, np.float32) if out is None else out
    acc = _f64(sumsq)
    of = _i32(overflow)
    lib().orc_reduce_lp_accum(n, C.cast(_ptr_array(slices), _vp), lp, length, loss_scale,
                              _ptr(g), C.byref(acc), C.byref(of))
    return g, acc.value, of.value


def decide(sumsq, overflow, clip, loss_scale, step, good_steps=0, growth_interval=1000,
           beta1=0.9, beta2=0.999, remote_sumsq=0.0, remote_overflow=0):
    d = Decision()
    lib().orc_decide(sumsq, remote_sumsq, int(overflow), int(remote_overflow), clip,
                     loss_scale, step, good_steps, growth_interval, beta1, beta2,
                     C.byref(d))
    return d.as_dict()


def adam(g, master, m, v, lp, coef, skip, lr, beta1, beta2, eps, wd, adamw, bc1, bc2,
         param=True):
    """Update master, m, v in place (float32 arrays); return the lp codes (or None)."""
    for a in (master, m, v):
        assert a.dtype == np.float32 and a.flags.c_contiguous
    g = _c(g, np.float32)
    out = np.empty(g.size, np.uint16) if param else None
    lib().orc_adam(g.size, _ptr(g), _ptr(master), _ptr(m), _ptr(v), _ptr(out), lp,
                   coef, int(skip), lr, beta1, beta2, eps, wd, int(adamw), bc1, bc2)
    return out


def gather(shards):
    shards = [_c(s, np.uint16) for s in shards]
    length = shards[0].size
    out = np.empty(length * len(shards), np.uint16)
    lib().orc_gather(len(shards), C.cast(_ptr_array(shards), _vp), length, _ptr(out))
    return out


def quantize_blocks(x_codes, lp, block=128):
    x = _c(x_codes, np.uint16)
    assert x.size % block == 0
    q = np.empty(x.size, np.int8)
    sc = np.empty(x.size // block, np.float32)
    lib().orc_quantize_blocks(x.size, _ptr(x), lp, block, _ptr(q), _ptr(sc))
    return q, sc


def dequant_gather(qs, scales, lp, block=128):
    qs = [_c(q, np.int8) for q in qs]
    scales = [_c(s, np.float32) for s in scales]
    length = qs[0].size
    out = np.empty(length * len(qs), np.uint16)
    lib().orc_dequant_gather(len(qs), C.cast(_ptr_array(qs), _vp), C.cast(_ptr_array(scales), _vp),
                             length, block, lp, _ptr(out))
    return out


def e4m3_decode(codes):
    c = _c(codes, np.uint8)
    out = np.empty(c.shape, np.float32)
    lib().orc_e4m3_decode_array(c.size, _ptr(c), _ptr(out))
    return out


def e4m3_encode(x):
    v = _c(x, np.float32)
    out = np.empty(v.shape, np.uint8)
    lib().orc_e4m3_encode_array(v.size, _ptr(v), _ptr(out))
    return out


def quantize_blocks_fp8(x_codes, lp, block=128):
    x = _c(x_codes, np.uint16)
    assert x.size % block == 0
    q = np.empty(x.size, np.uint8)
    sc = np.empty(x.size // block, np.float32)
    lib().orc_quantize_blocks_fp8(x.size, _ptr(x), lp, block, _ptr(q), _ptr(sc))
    return q, sc


def dequant_gather_fp8(qs, scales, lp, block=128):
    qs = [_c(q, np.uint8) for q in qs]
    scales = [_c(s, np.float32) for s in scales]
    length = qs[0].size
    out = np.empty(length * len(qs), np.uint16)
    lib().orc_dequant_gather_fp8(len(qs), C.cast(_ptr_array(qs), _vp),
                                 C.cast(_ptr_array(scales), _vp), length, block, lp, _ptr(out))
    return out


LIB_PATH = _build.LIB
__all__ = ["lib", "lp_to_float", "float_to_lp", "layout", "partition_to_flat",
           "fragments", "memory", "reduce", "reduce_lp_accum", "decide", "quantize_blocks",
           "dequant_gather", "e4m3_decode", "e4m3_encode", "quantize_blocks_fp8",
           "dequant_gather_fp8", "adam", "gather", "LIB_PATH",
           "Decision"]
