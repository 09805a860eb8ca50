"""CPU oracle for fused residual-add + RMSNorm + dynamic FP8 / NVFP4 / MXFP4 quantisation.

TEST INFRASTRUCTURE. Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg may import this package. The product path (the CUDA library and its binding) never
does, and this package never imports the product.

The arithmetic lives in ``rmsq_oracle.c`` (plain C, double precision, no fast-math, no FMA
contraction). This module only compiles it with gcc, loads it with ctypes and splits rows over
threads. Rows are independent, so running row ranges on several threads changes no result.

Sources: Modular's "rms_norm_fused_fp8" and "allreduce_residual_rmsnorm_fp8" API pages, and
FlashInfer's "cute_dsl/rmsnorm_fp4quant.py" (RMSNormFP4QuantKernel, phases 2 and 3). Each C
function names the passage it follows.
"""
from __future__ import annotations

import ctypes
import functools
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rmsq_oracle.c")
_LIB_PATH = os.path.join(_HERE, "librmsq_oracle.so")

BF16, FP16, F32 = 0, 1, 2
E4M3_MAX = 448.0
E2M1_MAX = 6.0

_lib = None


def build(force: bool = False) -> str:
    """Compile rmsq_oracle.c into librmsq_oracle.so next to it (gcc, -O2, strict ISO C)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".%d.tmp" % os.getpid()
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P, I64, I, F, D = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_double
    lib.oracle_format_round.argtypes = [D, I, I]
    lib.oracle_format_round.restype = D
    lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_decode.restype = D
    lib.oracle_e2m1_decode.argtypes = [ctypes.c_uint8]
    lib.oracle_e2m1_decode.restype = D
    lib.oracle_e4m3_encode.argtypes = [D]
    lib.oracle_e4m3_encode.restype = ctypes.c_uint8
    lib.oracle_e2m1_encode.argtypes = [D]
    lib.oracle_e2m1_encode.restype = ctypes.c_uint8
    lib.oracle_ue8m0_code.argtypes = [D]
    lib.oracle_ue8m0_code.restype = I
    lib.oracle_fp16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_fp16_to_double.restype = D
    lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_double.restype = D
    lib.oracle_scale_offset.argtypes = [I64, I64, I64, I]
    lib.oracle_scale_offset.restype = I64
    for name in ("oracle_e4m3_encode_f64_array", "oracle_e4m3_encode_f32_array",
                 "oracle_e2m1_encode_f64_array", "oracle_e2m1_encode_f32_array",
                 "oracle_bf16_round_array", "oracle_fp16_round_array", "oracle_ue8m0_code_array"):
        getattr(lib, name).argtypes = [P, P, I64]
        getattr(lib, name).restype = None
    lib.oracle_quant_fp8.argtypes = [P, P, I, P, I64, I64, F, F, F, I, P, P, P, P, P, P]
    lib.oracle_quant_nvfp4.argtypes = [P, P, I, P, I64, I64, F, F, F, I, P, P, P, P, P, P, P]
    lib.oracle_quant_mxfp4.argtypes = [P, P, I, P, I64, I64, F, F, I, P, P, P, P, P, P, P]
    lib.oracle_rmsnorm.argtypes = [P, P, I, P, I64, I64, F, F, P, P, P]
    for name in ("oracle_quant_fp8", "oracle_quant_nvfp4", "oracle_quant_mxfp4", "oracle_rmsnorm"):
        getattr(lib, name).restype = I
    _lib = lib
    return lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


# ---------------------------------------------------------------------------------------------
# Scalar / array format helpers
# ---------------------------------------------------------------------------------------------

def format_round(v: float, mant_bits: int, emin: int) -> float:
    return _load().oracle_format_round(float(v), mant_bits, emin)


def e4m3_decode(code: int) -> float:
    return _load().oracle_e4m3_decode(code)


def e2m1_decode(code: int) -> float:
    return _load().oracle_e2m1_decode(code)


def e4m3_encode(v) -> np.ndarray:
    """RNE + satfinite E4M3 codes of an array of float32 or float64 values."""
    v = np.ascontiguousarray(v)
    out = np.empty(v.shape, np.uint8)
    if v.dtype == np.float32:
        _load().oracle_e4m3_encode_f32_array(_ptr(v), _ptr(out), v.size)
    else:
        v = np.ascontiguousarray(v, np.float64)
        _load().oracle_e4m3_encode_f64_array(_ptr(v), _ptr(out), v.size)
    return out


def e2m1_encode(v) -> np.ndarray:
    """RNE + satfinite E2M1 codes (low nibble) of an array of float32 or float64 values."""
    v = np.ascontiguousarray(v)
    out = np.empty(v.shape, np.uint8)
    if v.dtype == np.float32:
        _load().oracle_e2m1_encode_f32_array(_ptr(v), _ptr(out), v.size)
    else:
        v = np.ascontiguousarray(v, np.float64)
        _load().oracle_e2m1_encode_f64_array(_ptr(v), _ptr(out), v.size)
    return out


def round_to_dtype(v, dtype: int) -> np.ndarray:
    """Correctly rounded double -> bf16 / fp16 bit patterns."""
    v = np.ascontiguousarray(v, np.float64)
    out = np.empty(v.shape, np.uint16)
    fn = _load().oracle_bf16_round_array if dtype == BF16 else _load().oracle_fp16_round_array
    fn(_ptr(v), _ptr(out), v.size)
    return out


def ue8m0_code(a) -> np.ndarray:
    a = np.ascontiguousarray(a, np.float64)
    out = np.empty(a.shape, np.uint8)
    _load().oracle_ue8m0_code_array(_ptr(a), _ptr(out), a.size)
    return out


def scale_offset(row: int, sf: int, num_sf: int, swizzled: bool) -> int:
    return _load().oracle_scale_offset(row, sf, num_sf, int(swizzled))


def swizzled_scale_size(rows: int, num_sf: int) -> int:
    """Bytes of a swizzled 128x4 scale tensor: whole 128-row by 4-scale tiles of 512 bytes."""
    return ((rows + 127) // 128) * ((num_sf + 3) // 4) * 512


def e4m3_values() -> np.ndarray:
    return np.array([e4m3_decode(c) for c in range(256)])


def e2m1_values() -> np.ndarray:
    return np.array([e2m1_decode(c) for c in range(16)])


@functools.lru_cache(maxsize=None)
def _fp16_table() -> np.ndarray:
    lib = _load()
    return np.array([lib.oracle_fp16_to_double(c) for c in range(65536)])


def decode_bits(bits: np.ndarray, dtype: int) -> np.ndarray:
    """bf16 / fp16 bit patterns -> float64 values (software decode, for the tests)."""
    bits = np.asarray(bits, np.uint16)
    if dtype == BF16:
        with np.errstate(invalid="ignore"):
            return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return _fp16_table()[bits]


# ---------------------------------------------------------------------------------------------
# The row math
# ---------------------------------------------------------------------------------------------

def _as_input(a, dtype):
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    want = np.float32 if dtype == F32 else np.uint16
    if a.dtype != want:
        raise TypeError("oracle input must be %s bits, got %s" % (want, a.dtype))
    return a


def _run_rows(fn_rows, rows: int, threads: int | None):
    """Run fn_rows(r0, r1) over row ranges on a thread pool (ctypes releases the GIL)."""
    threads = max(1, min(threads or _cores(), rows))
    if threads == 1:
        fn_rows(0, rows)
        return 1
    bounds = np.linspace(0, rows, threads + 1).astype(np.int64)
    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(lambda i: fn_rows(int(bounds[i]), int(bounds[i + 1])), range(threads)))
    return threads


class _Rows:
    """Row-offset pointer helper for row-major [rows, cols] numpy arrays."""

    def __init__(self, a):
        self.a = a

    def at(self, r):
        if self.a is None:
            return None
        return self.a.ctypes.data + r * self.a.strides[0]


def quant_fp8(x, residual, gamma, *, dtype=BF16, eps=1e-6, weight_offset=0.0, scale_ub=1200.0,
              scale_dtype=F32, want_y=False, want_pre=False, threads=None):
    """FP8 E4M3 with a per-row dynamic scale. Inputs are bit arrays [rows, H] (uint16 for bf16 /
    fp16, float32 for fp32). Returns a dict with q [rows, H] uint8, scale [rows] float32 (the
    stored scale, rounded to scale_dtype and widened), residual_output (or None), and optionally
    y (float32) and pre (float64, y / scale)."""
    lib = _load()
    x, residual, gamma = _as_input(x, dtype), _as_input(residual, dtype), _as_input(gamma, dtype)
    rows, H = x.shape
    q = np.zeros((rows, H), np.uint8)
    scale = np.zeros(rows, np.float32)
    res_out = np.zeros_like(x) if residual is not None else None
    y = np.zeros((rows, H), np.float32) if want_y else None
    pre = np.zeros((rows, H), np.float64) if want_pre else None
    R = [_Rows(a) for a in (x, residual, res_out, q, y, pre)]
    scale_rows = _Rows(scale.reshape(rows, 1))

    def run(r0, r1):
        if r1 <= r0:
            return
        tmp = np.zeros(H, np.float32)
        lib.oracle_quant_fp8(R[0].at(r0), R[1].at(r0), dtype, _ptr(gamma), r1 - r0, H, eps,
                             weight_offset, scale_ub, scale_dtype, R[2].at(r0), R[3].at(r0),
                             scale_rows.at(r0),
                             R[4].at(r0), R[5].at(r0), _ptr(tmp))

    _run_rows(run, rows, threads)
    return dict(q=q, scale=scale, residual_output=res_out, y=y, pre=pre)


def quant_nvfp4(x, residual, gamma, global_scale, *, dtype=BF16, eps=1e-6, weight_offset=0.0,
                swizzled=False, want_y=False, want_pre=False, threads=None):
    """NVFP4: packed E2M1 [rows, H/2] with an E4M3 scale per 16 elements under an fp32 global
    scale. Returns q (packed), block_scale (row-major [rows, H/16], or the flat swizzled tensor),
    residual_output, and optionally y, pre (y * gs / dec(s)) and t (pre-rounding block scale)."""
    lib = _load()
    x, residual, gamma = _as_input(x, dtype), _as_input(residual, dtype), _as_input(gamma, dtype)
    rows, H = x.shape
    nsf = H // 16
    q = np.zeros((rows, H // 2), np.uint8)
    res_out = np.zeros_like(x) if residual is not None else None
    y = np.zeros((rows, H), np.float32) if want_y else None
    pre = np.zeros((rows, H), np.float64) if want_pre else None
    t = np.zeros((rows, nsf), np.float64) if want_pre else None
    if swizzled:
        # swizzled tiles interleave rows, so the whole tensor is written by one call
        bs = np.zeros(swizzled_scale_size(rows, nsf), np.uint8)
        tmp = np.zeros(H, np.float32)
        lib.oracle_quant_nvfp4(_ptr(x), _ptr(residual), dtype, _ptr(gamma), rows, H, eps,
                               weight_offset, float(global_scale), 1, _ptr(res_out), _ptr(q),
                               _ptr(bs), _ptr(y), _ptr(pre), _ptr(t), _ptr(tmp))
        return dict(q=q, block_scale=bs, residual_output=res_out, y=y, pre=pre, t=t)
    bs = np.zeros((rows, nsf), np.uint8)
    R = [_Rows(a) for a in (x, residual, res_out, q, bs, y, pre, t)]

    def run(r0, r1):
        if r1 <= r0:
            return
        tmp = np.zeros(H, np.float32)
        lib.oracle_quant_nvfp4(R[0].at(r0), R[1].at(r0), dtype, _ptr(gamma), r1 - r0, H, eps,
                               weight_offset, float(global_scale), 0, R[2].at(r0), R[3].at(r0),
                               R[4].at(r0), R[5].at(r0), R[6].at(r0), R[7].at(r0), _ptr(tmp))

    _run_rows(run, rows, threads)
    return dict(q=q, block_scale=bs, residual_output=res_out, y=y, pre=pre, t=t)


def quant_mxfp4(x, residual, gamma, *, dtype=BF16, eps=1e-6, weight_offset=0.0, swizzled=False,
                want_y=False, want_pre=False, threads=None):
    """MXFP4: packed E2M1 [rows, H/2] with a UE8M0 scale per 32 elements. Returns q, block_scale,
    residual_output, and optionally y, pre (y * 2^(127 - code)) and a (block max |y|)."""
    lib = _load()
    x, residual, gamma = _as_input(x, dtype), _as_input(residual, dtype), _as_input(gamma, dtype)
    rows, H = x.shape
    nsf = H // 32
    q = np.zeros((rows, H // 2), np.uint8)
    res_out = np.zeros_like(x) if residual is not None else None
    y = np.zeros((rows, H), np.float32) if want_y else None
    pre = np.zeros((rows, H), np.float64) if want_pre else None
    amax = np.zeros((rows, nsf), np.float64) if want_pre else None
    if swizzled:
        bs = np.zeros(swizzled_scale_size(rows, nsf), np.uint8)
        tmp = np.zeros(H, np.float32)
        lib.oracle_quant_mxfp4(_ptr(x), _ptr(residual), dtype, _ptr(gamma), rows, H, eps,
                               weight_offset, 1, _ptr(res_out), _ptr(q), _ptr(bs), _ptr(y),
                               _ptr(pre), _ptr(amax), _ptr(tmp))
        return dict(q=q, block_scale=bs, residual_output=res_out, y=y, pre=pre, a=amax)
    bs = np.zeros((rows, nsf), np.uint8)
    R = [_Rows(a) for a in (x, residual, res_out, q, bs, y, pre, amax)]

    def run(r0, r1):
        if r1 <= r0:
            return
        tmp = np.zeros(H, np.float32)
        lib.oracle_quant_mxfp4(R[0].at(r0), R[1].at(r0), dtype, _ptr(gamma), r1 - r0, H, eps,
                               weight_offset, 0, R[2].at(r0), R[3].at(r0), R[4].at(r0),
                               R[5].at(r0), R[6].at(r0), R[7].at(r0), _ptr(tmp))

    _run_rows(run, rows, threads)
    return dict(q=q, block_scale=bs, residual_output=res_out, y=y, pre=pre, a=amax)


def rmsnorm(x, residual, gamma, *, dtype=BF16, eps=1e-6, weight_offset=0.0, threads=None):
    """y = RN_fp32(s * rstd * (gamma + offset)) and rstd per row, with s the rounded residual
    sum. Returns dict(y, rstd, residual_output)."""
    lib = _load()
    x, residual, gamma = _as_input(x, dtype), _as_input(residual, dtype), _as_input(gamma, dtype)
    rows, H = x.shape
    y = np.zeros((rows, H), np.float32)
    rstd = np.zeros(rows, np.float32)
    res_out = np.zeros_like(x) if residual is not None else None
    R = [_Rows(a) for a in (x, residual, res_out, y)]
    rstd_rows = _Rows(rstd.reshape(rows, 1))

    def run(r0, r1):
        if r1 <= r0:
            return
        lib.oracle_rmsnorm(R[0].at(r0), R[1].at(r0), dtype, _ptr(gamma), r1 - r0, H, eps,
                           weight_offset, R[2].at(r0), R[3].at(r0), rstd_rows.at(r0))

    _run_rows(run, rows, threads)
    return dict(y=y, rstd=rstd, residual_output=res_out)


def nvfp4_global_scale(amax_y: float) -> np.float32:
    """gs = 448 * 6 / amax(y) in fp32: the global scale that maps the tensor's largest |y| onto
    the largest E4M3 block scale times the largest E2M1 value."""
    return np.float32(np.float32(E4M3_MAX * E2M1_MAX) / np.float32(amax_y))


def cores() -> int:
    return _cores()
