"""The C ABI library on a machine without a GPU: it builds, loads, exports every function that
include/rmsq.h declares, and rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from rmsnorm_precision_activation_gb300 import build
    build.build()
    import rmsnorm_precision_activation_gb300 as rq
    return rq.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "rmsq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w]+\s*\*?\s*(\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("rmsnorm_quant_fp8", "rmsnorm_quant_nvfp4", "rmsnorm_quant_mxfp4",
              "rmsnorm_nvfp4_global_scale", "rmsq_status_string", "rmsq_device_status"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    import rmsnorm_precision_activation_gb300 as rq
    for n in _declared():
        assert hasattr(lib, n), n
        assert n in rq.SIGNATURES, n


def test_python_constants_match_the_header():
    import rmsnorm_precision_activation_gb300 as rq
    src = open(os.path.join(ROOT, "include", "rmsq.h")).read()
    define = lambda n: int(re.search(r"#define %s (\d+)" % n, src).group(1))
    assert rq.MAX_HIDDEN == define("RMSQ_MAX_HIDDEN")
    assert rq.ONE_CTA_HIDDEN == define("RMSQ_ONE_CTA_HIDDEN")
    for code, name in rq.STATUS.items():
        assert re.search(r"\b%s = %d\b" % (name, code), src), name
    for name in ("RMSQ_BF16", "RMSQ_FP16", "RMSQ_F32"):
        assert re.search(r"\b%s = %d\b" % (name, getattr(rq, name)), src), name


def test_status_strings(lib):
    for code, name in [(0, "RMSQ_OK"), (2, "RMSQ_ERR_SHAPE"), (8, "RMSQ_ERR_TIMEOUT")]:
        assert lib.rmsq_status_string(code).decode().startswith(name)
    assert lib.rmsq_status_string(99).decode() == "RMSQ_UNKNOWN_STATUS"


def test_host_side_validation_without_gpu(lib):
    A = 1 << 20    # fake, 16-byte aligned "device" addresses: never dereferenced on these paths
    f = lib.rmsnorm_quant_fp8
    assert f(None, None, None, A, 4, 64, 0, 1e-6, 0.0, 1.0, A, A, 2, None) == 1
    assert f(A, A, None, A, 4, 64, 0, 1e-6, 0.0, 1.0, A, A, 2, None) == 1
    assert f(A + 8, None, None, A, 4, 64, 0, 1e-6, 0.0, 1.0, A, A, 2, None) == 3
    assert f(A, None, None, A, 4, 60, 0, 1e-6, 0.0, 1.0, A, A, 2, None) == 2
    assert f(A, None, None, A, 4, 131072 + 256, 0, 1e-6, 0.0, 1.0, A, A, 2, None) == 2  # > max
    assert f(A, None, None, A, 4, 65536 + 256, 2, 1e-6, 0.0, 1.0, A, A, 2, None) == 2   # fp32 > max
    assert f(A, None, None, A, 4, 32768 + 8, 0, 1e-6, 0.0, 1.0, A, A, 2, None) == 2     # wide, not /256
    assert f(A, None, None, A, 4, 64, 3, 1e-6, 0.0, 1.0, A, A, 2, None) == 4
    assert f(A, None, None, A, 4, 64, 0, float("nan"), 0.0, 1.0, A, A, 2, None) == 6
    assert f(A, None, None, A, 4, 64, 0, 1e-6, 0.0, -1.0, A, A, 2, None) == 6
    assert f(A, None, None, A, 0, 64, 0, 1e-6, 0.0, 1.0, A, A, 2, None) == 0      # empty call
    assert lib.rmsnorm_quant_nvfp4(A, None, None, A, 4, 64, 0, 1e-6, 0.0, None, A, A, 0, None) == 1
    assert lib.rmsnorm_quant_mxfp4(A, None, None, A, 4, 48, 0, 1e-6, 0.0, A, A, 0, None) == 2
    assert lib.rmsnorm_quant_mxfp4(A, None, None, A, 4, 64, 0, 1e-6, 0.0, A, A, 2, None) == 4
    assert lib.rmsq_set_tuning(9, 0, 0) == 6 and lib.rmsq_set_tuning(0, 0, 3) == 6
    assert lib.rmsq_set_tuning(-1, 0, 0) == 6 and lib.rmsq_set_tuning(0, 33, 0) == 6
    assert lib.rmsq_set_tuning(0, 0, 0) == 0


def test_valid_call_without_gpu_reports_no_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    A = 1 << 20
    assert lib.rmsnorm_quant_fp8(A, None, None, A, 4, 64, 0, 1e-6, 0.0, 1.0, A, A, 2, None) == 7
