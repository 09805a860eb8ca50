"""rmsnorm_quant_fp8_static_scratch, the FP8 call for callers that cannot let a library allocate
or hand out device memory for them (a runtime that reserves all device memory itself before it
serves, a host thread that may not call the CUDA allocator). Its only scratch, the counter that
hands out a launch's last rows, sits in a fixed 256-byte array of the library's device memory,
cleared on the caller's stream before each launch.

The GPU test calls it through the C ABI, twice in a row, and checks each result against
rmsnorm_quant_fp8 on the same inputs. The two calls run the same kernel, so the outputs must
match bit for bit, which is inside the parity tolerance the other tests use. The file is named
to be collected last."""
import ctypes

import pytest
import torch

import workloads as W
from gpu_common import inputs, rq

RMSQ_F32 = 2


def _call(name, d, w, out):
    import rmsnorm_precision_activation_gb300 as pkg
    x, r, g = d["input"], d["residual"], d["gamma"]
    q, sc, ro = out
    fn = getattr(rq().lib(), name)
    st = fn(x.data_ptr(), None if r is None else r.data_ptr(), None if ro is None else ro.data_ptr(),
            g.data_ptr(), x.shape[0], x.shape[1], pkg._DT[x.dtype], w.eps, w.weight_offset,
            w.scale_ub, q.data_ptr(), sc.data_ptr(), RMSQ_F32,
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, (name, st)


def _outputs(d):
    x, r = d["input"], d["residual"]
    return (torch.empty(x.shape, dtype=torch.uint8, device=x.device),
            torch.empty(x.shape[0], dtype=torch.float32, device=x.device),
            None if r is None else torch.empty_like(x))


CASES = [
    # a CTA per row, where the kernel uses the row counter
    W.config("fp8_residual"),
    # weight offset and fp16: the other FP8 kernel
    W.Workload("custom", "fp8", 3000, 8192, "fp16", True, weight_offset=1.0, scale_ub=10.0),
    # short rows: a row per warp, no counter
    W.Workload("custom", "fp8", 5000, 1024, "bf16", False, scale_ub=1200.0),
]


@pytest.mark.gpu
@pytest.mark.parametrize("w", CASES, ids=["fp8_residual", "offset_fp16", "short_rows"])
def test_static_scratch_matches_regular_entry_point_twice(w):
    d = inputs(w, seed=77)
    ref = _outputs(d)
    _call("rmsnorm_quant_fp8", d, w, ref)
    for _ in range(2):                   # two calls in a row share the scratch array
        got = _outputs(d)
        _call("rmsnorm_quant_fp8_static_scratch", d, w, got)
        torch.cuda.synchronize()
        assert torch.equal(got[0], ref[0])
        assert torch.equal(got[1], ref[1])
        if ref[2] is not None:
            assert torch.equal(got[2], ref[2])
    assert rq().rmsq_device_status() == 0


def test_static_scratch_rejects_rows_beyond_the_counter():
    # checked on the host before any device work, so no GPU is needed
    lib = rq().lib()
    A = 1 << 20      # fake 16-byte aligned addresses: never dereferenced on this path
    st = lib.rmsnorm_quant_fp8_static_scratch(A, None, None, A, (1 << 31), 64, 0, 1e-6, 0.0, 1.0,
                                              A, A, RMSQ_F32, None)
    assert st == 2   # RMSQ_ERR_SHAPE
