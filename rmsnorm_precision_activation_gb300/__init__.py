"""GB300 (sm_103a) fused residual-add + RMSNorm + dynamic FP8 / NVFP4 / MXFP4 quantisation.

Python binding of librmsq.so (C ABI in include/rmsq.h). The functions here only marshal
arguments: they check shapes and dtypes, allocate outputs the caller did not pass, and call the
C entry point of the same name on the current CUDA stream. Every step of the computation runs in
the library's CUDA kernels; there is no fallback. If librmsq.so has not been built, every call
raises.

    out, scale, res_out = rmsnorm_quant_fp8(x, gamma, residual=r, scale_ub=1200.0)
    q, block_scale, res_out = rmsnorm_quant_nvfp4(x, gamma, global_scale=gs)
    q, block_scale, res_out = rmsnorm_quant_mxfp4(x, gamma, residual=r)
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "librmsq.so")

RMSQ_BF16, RMSQ_FP16, RMSQ_F32 = 0, 1, 2
SCALE_ROW_MAJOR, SCALE_SWIZZLED_128x4 = 0, 1
SCHED_AUTO, SCHED_PIPE, SCHED_REG, SCHED_WARP, SCHED_CLUSTER = 0, 1, 2, 3, 4
# Widest row accepted, in elements (fp32 input: half). Rows wider than ONE_CTA_HIDDEN (fp32:
# half) run on a thread-block cluster and must be a multiple of 256 elements.
MAX_HIDDEN, ONE_CTA_HIDDEN = 131072, 32768

STATUS = {0: "RMSQ_OK", 1: "RMSQ_ERR_NULL", 2: "RMSQ_ERR_SHAPE", 3: "RMSQ_ERR_ALIGN",
          4: "RMSQ_ERR_DTYPE", 5: "RMSQ_ERR_LAUNCH", 6: "RMSQ_ERR_VALUE", 7: "RMSQ_ERR_DEVICE",
          8: "RMSQ_ERR_TIMEOUT"}

_DT = {torch.bfloat16: RMSQ_BF16, torch.float16: RMSQ_FP16, torch.float32: RMSQ_F32}

# Exported C symbols and their ctypes signatures.
_P, _I64, _I, _F, _U64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_uint64
SIGNATURES = {
    "rmsnorm_quant_fp8": ([_P, _P, _P, _P, _I64, _I64, _I, _F, _F, _F, _P, _P, _I, _P], _I),
    "rmsnorm_quant_fp8_static_scratch": ([_P, _P, _P, _P, _I64, _I64, _I, _F, _F, _F, _P, _P, _I, _P], _I),
    "rmsnorm_quant_nvfp4": ([_P, _P, _P, _P, _I64, _I64, _I, _F, _F, _P, _P, _P, _I, _P], _I),
    "rmsnorm_quant_mxfp4": ([_P, _P, _P, _P, _I64, _I64, _I, _F, _F, _P, _P, _I, _P], _I),
    "rmsnorm_nvfp4_global_scale": ([_P, _P, _P, _I64, _I64, _I, _F, _F, _P, _P], _I),
    "rmsq_status_string": ([_I], ctypes.c_char_p),
    "rmsq_device_status": ([], _I),
    "rmsq_set_schedule": ([_I], _I),
    "rmsq_set_tuning": ([_I, _I, _I], _I),
    "rmsq_set_row_warps": ([_I], _I),
    "rmsq_set_cluster_size": ([_I], _I),
    "rmsq_set_dynamic_rows": ([_I], _I),
    "rmsq_set_pdl": ([_I], _I),
    "rmsq_set_wait_timeout_ns": ([_U64], None),
    "rmsq_selftest_wait_timeout": ([_U64, _P], _I),
    "rmsq_debug_convert": ([_I, _P, _P, _I64, _P], _I),
    "rmsq_launch_count": ([], _U64),
    "rmsq_plan": ([_I, _I, _I, _F, _I64, _I, _I, _I, _P], _I),
}

# rmsq_plan's modes, and GB300's shared-memory limits in bytes (opt-in per CTA, per SM, reserved
# per CTA), which let it plan without a GPU.
MODES = {"fp8": 0, "nvfp4": 1, "mxfp4": 2, "global_scale": 3}
GB300_SMEM = (232448, 233472, 1024)


class PlanInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("schedule", "vectors_per_thread", "threads", "stages",
                                            "cluster", "smem_bytes", "ctas_per_sm", "w16")]

_lib = None


class RmsqError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s: %s" % (where, STATUS.get(status, "status %d" % status)))


def lib() -> ctypes.CDLL:
    """The loaded librmsq.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("librmsq.so is not built (%s); run "
                               "rmsnorm_precision_activation_gb300.build.build()" % LIB_PATH)
        handle = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.argtypes = args
            fn.restype = res
        _lib = handle
    return _lib


def _check(status: int, where: str):
    if status != 0:
        raise RmsqError(status, where)


def _stream(device, stream):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _flat(t, H):
    return t.reshape(-1, H) if t.dim() != 2 else t


def _prepare(input, gamma, residual, residual_output):
    if not input.is_cuda:
        raise ValueError("input must be a CUDA tensor")
    if input.dtype not in _DT:
        raise TypeError("input dtype must be bfloat16, float16 or float32")
    H = input.shape[-1]
    x = _flat(input, H)
    for name, t in (("input", x), ("gamma", gamma), ("residual", residual)):
        if t is not None and (not t.is_contiguous() or t.dtype != input.dtype or t.device != input.device):
            raise ValueError("%s must be a contiguous %s tensor on %s" % (name, input.dtype, input.device))
    if gamma.shape != (H,):
        raise ValueError("gamma must have shape (%d,)" % H)
    r = None
    if residual is not None:
        r = _flat(residual, H)
        if r.shape != x.shape:
            raise ValueError("residual must have the input's shape")
        if residual_output is None:
            residual_output = torch.empty_like(input)
        if residual_output.shape != input.shape or not residual_output.is_contiguous():
            raise ValueError("residual_output must be a contiguous tensor of the input's shape")
    elif residual_output is not None:
        raise ValueError("residual_output given without residual")
    ro = None if residual_output is None else _flat(residual_output, H)
    return x, r, ro, residual_output, H


def rmsnorm_quant_fp8(input, gamma, *, residual=None, residual_output=None, epsilon=1e-6,
                      weight_offset=0.0, scale_ub=1200.0, output=None, scale_output=None,
                      scale_dtype=torch.float32, stream=None):
    """Residual add + RMSNorm + FP8 E4M3 with a per-row dynamic scale.

    Returns (output float8_e4m3fn [..., H], scale_output [...] of scale_dtype, residual_output)."""
    x, r, ro, residual_output, H = _prepare(input, gamma, residual, residual_output)
    lead = input.shape[:-1]
    if output is None:
        output = torch.empty(input.shape, dtype=torch.float8_e4m3fn, device=input.device)
    if scale_output is None:
        scale_output = torch.empty(lead, dtype=scale_dtype, device=input.device)
    with torch.cuda.device(input.device):
        st = lib().rmsnorm_quant_fp8(_ptr(x), _ptr(r), _ptr(ro), _ptr(gamma), x.shape[0], H,
                                     _DT[input.dtype], float(epsilon), float(weight_offset),
                                     float(scale_ub), _ptr(output), _ptr(scale_output),
                                     _DT[scale_output.dtype], _stream(input.device, stream))
    _check(st, "rmsnorm_quant_fp8")
    return output, scale_output, residual_output


def swizzled_scale_numel(rows: int, hidden: int, block: int) -> int:
    """Bytes of a swizzled 128x4 block-scale tensor (whole 128 x 4 tiles of 512 bytes)."""
    return ((rows + 127) // 128) * ((hidden // block + 3) // 4) * 512


def _fp4_outputs(input, H, block, output, block_scale, swizzled, scale_torch_dtype):
    rows = input.numel() // H
    if output is None:
        output = torch.empty(tuple(input.shape[:-1]) + (H // 2,), dtype=torch.uint8, device=input.device)
    if block_scale is None:
        if swizzled:
            block_scale = torch.empty(swizzled_scale_numel(rows, H, block), dtype=scale_torch_dtype,
                                      device=input.device)
        else:
            block_scale = torch.empty(tuple(input.shape[:-1]) + (H // block,), dtype=scale_torch_dtype,
                                      device=input.device)
    return output, block_scale


def rmsnorm_quant_nvfp4(input, gamma, *, global_scale=None, residual=None, residual_output=None,
                        epsilon=1e-6, weight_offset=0.0, output=None, block_scale=None,
                        swizzled=False, stream=None):
    """Residual add + RMSNorm + NVFP4 (packed E2M1, E4M3 scale per 16 elements, fp32 global
    scale read on the device). global_scale: a CUDA float32 tensor of one element (default 1.0).

    Returns (output uint8 [..., H/2], block_scale float8_e4m3fn, residual_output)."""
    x, r, ro, residual_output, H = _prepare(input, gamma, residual, residual_output)
    if global_scale is None:
        global_scale = torch.ones(1, dtype=torch.float32, device=input.device)
    if global_scale.dtype != torch.float32 or global_scale.numel() != 1 or not global_scale.is_cuda:
        raise ValueError("global_scale must be a CUDA float32 tensor with one element")
    output, block_scale = _fp4_outputs(input, H, 16, output, block_scale, swizzled, torch.float8_e4m3fn)
    with torch.cuda.device(input.device):
        st = lib().rmsnorm_quant_nvfp4(_ptr(x), _ptr(r), _ptr(ro), _ptr(gamma), x.shape[0], H,
                                       _DT[input.dtype], float(epsilon), float(weight_offset),
                                       _ptr(global_scale), _ptr(output), _ptr(block_scale),
                                       SCALE_SWIZZLED_128x4 if swizzled else SCALE_ROW_MAJOR,
                                       _stream(input.device, stream))
    _check(st, "rmsnorm_quant_nvfp4")
    return output, block_scale, residual_output


def rmsnorm_quant_mxfp4(input, gamma, *, residual=None, residual_output=None, epsilon=1e-6,
                        weight_offset=0.0, output=None, block_scale=None, swizzled=False,
                        stream=None):
    """Residual add + RMSNorm + MXFP4 (packed E2M1, UE8M0 scale per 32 elements).

    Returns (output uint8 [..., H/2], block_scale uint8 (UE8M0 codes), residual_output)."""
    x, r, ro, residual_output, H = _prepare(input, gamma, residual, residual_output)
    output, block_scale = _fp4_outputs(input, H, 32, output, block_scale, swizzled, torch.uint8)
    with torch.cuda.device(input.device):
        st = lib().rmsnorm_quant_mxfp4(_ptr(x), _ptr(r), _ptr(ro), _ptr(gamma), x.shape[0], H,
                                       _DT[input.dtype], float(epsilon), float(weight_offset),
                                       _ptr(output), _ptr(block_scale),
                                       SCALE_SWIZZLED_128x4 if swizzled else SCALE_ROW_MAJOR,
                                       _stream(input.device, stream))
    _check(st, "rmsnorm_quant_mxfp4")
    return output, block_scale, residual_output


def rmsnorm_nvfp4_global_scale(input, gamma, *, residual=None, epsilon=1e-6, weight_offset=0.0,
                               out=None, stream=None):
    """gs = 448 * 6 / max |y| over the whole tensor, computed on the device (one extra read of
    input and residual). Returns a CUDA float32 tensor of one element."""
    H = input.shape[-1]
    x = _flat(input, H)
    r = None if residual is None else _flat(residual, H)
    if out is None:
        out = torch.empty(1, dtype=torch.float32, device=input.device)
    with torch.cuda.device(input.device):
        st = lib().rmsnorm_nvfp4_global_scale(_ptr(x), _ptr(r), _ptr(gamma), x.shape[0], H,
                                              _DT[input.dtype], float(epsilon),
                                              float(weight_offset), _ptr(out),
                                              _stream(input.device, stream))
    _check(st, "rmsnorm_nvfp4_global_scale")
    return out


def rmsq_device_status() -> int:
    return lib().rmsq_device_status()


def rmsq_set_schedule(schedule: int) -> int:
    return lib().rmsq_set_schedule(int(schedule))


def rmsq_set_tuning(stages: int = 0, ctas_per_sm: int = 0, vectors_per_thread: int = 0):
    _check(lib().rmsq_set_tuning(stages, ctas_per_sm, vectors_per_thread), "rmsq_set_tuning")


def rmsq_set_cluster_size(ctas_per_cluster: int = 0):
    _check(lib().rmsq_set_cluster_size(int(ctas_per_cluster)), "rmsq_set_cluster_size")


def rmsq_set_row_warps(warps_per_cta: int = 0):
    _check(lib().rmsq_set_row_warps(int(warps_per_cta)), "rmsq_set_row_warps")


def rmsq_set_dynamic_rows(enable: bool) -> bool:
    return bool(lib().rmsq_set_dynamic_rows(int(bool(enable))))


def rmsq_set_pdl(enable: bool) -> bool:
    return bool(lib().rmsq_set_pdl(int(bool(enable))))


def rmsq_set_wait_timeout_ns(ns: int):
    lib().rmsq_set_wait_timeout_ns(int(ns))


def rmsq_selftest_wait_timeout(timeout_ns: int, stream=None):
    dev = torch.device("cuda", torch.cuda.current_device())
    _check(lib().rmsq_selftest_wait_timeout(int(timeout_ns), _stream(dev, stream)),
           "rmsq_selftest_wait_timeout")


def rmsq_debug_convert(fmt: int, values: torch.Tensor, stream=None) -> torch.Tensor:
    """Convert fp32 values on the device with the kernels' conversion instructions.
    fmt 0: E4M3 codes; fmt 1: E2M1 codes (low nibble). Returns uint8 codes."""
    out = torch.empty(values.shape, dtype=torch.uint8, device=values.device)
    with torch.cuda.device(values.device):
        _check(lib().rmsq_debug_convert(int(fmt), _ptr(values), _ptr(out), values.numel(),
                                        _stream(values.device, stream)), "rmsq_debug_convert")
    return out


def rmsq_launch_count() -> int:
    return lib().rmsq_launch_count()


def rmsq_plan(mode: str, dtype, hidden: int, residual: bool = False, weight_offset: float = 0.0,
              smem=GB300_SMEM) -> dict:
    """The launch plan the entry point of `mode` ("fp8", "nvfp4", "mxfp4", "global_scale") would
    choose now for rows of `hidden` elements, tuning settings included (rmsq_plan in
    include/rmsq.h). smem: the (opt-in per CTA, per SM, reserved per CTA) shared-memory limits in
    bytes, GB300's by default; None takes the current device's."""
    dt = _DT[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    optin, per_sm, reserved = smem if smem is not None else (0, 0, 0)
    info = PlanInfo()
    _check(lib().rmsq_plan(MODES[mode], dt, int(bool(residual)), float(weight_offset), int(hidden),
                           optin, per_sm, reserved, ctypes.byref(info)), "rmsq_plan")
    return {n: getattr(info, n) for n, _ in PlanInfo._fields_}
