"""rmsnorm_quant_fp8_static_scratch, the FP8 call for callers that cannot let a library allocate
or hand out device memory for them (a runtime that reserves all device memory itself before it
serves, a host thread that may not call the CUDA allocator). Its only scratch, the counter that
hands out a launch's last rows, sits in a fixed 256-byte array of the library's device memory,
cleared on the caller's stream before each launch.

The GPU test calls it through the C ABI, twice in a row, and checks each result two ways:
against the oracle, element by element under the parity rules the other tests use, and against
rmsnorm_quant_fp8 on the same inputs, which runs the same kernel and so must match bit for bit.
The first two cases force the CTA-per-row ring schedule, whose launches on these shapes take
their last rows from the counter in the array; the third runs a short-row shape whose schedule
uses no counter.

The clear before each launch matters only after a launch that a timed-out wait stopped: a
launch that runs to the end leaves the counter at zero itself (the thread holding its last
ticket resets it). That case is argued from the code, not tested, since no test here makes a
wait run out inside a quantisation kernel. The file is named to be collected last."""
import ctypes

import pytest
import torch

import oracle
import parity as P
import workloads as W
from gpu_common import ODT, host_bits, inputs, rq, schedule

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
    # a CTA per row (forced), where the kernel takes its last rows from the counter
    (W.config("fp8_residual"), 1),
    # weight offset and fp16: the other FP8 kernel, also a CTA per row (forced)
    (W.Workload("custom", "fp8", 3000, 8192, "fp16", True, weight_offset=1.0, scale_ub=10.0), 1),
    # short rows: a row per warp (the planner's choice), no counter
    (W.Workload("custom", "fp8", 5000, 1024, "bf16", False, scale_ub=1200.0), 0),
]


def _oracle(d, w):
    x, r, g = d["input"], d["residual"], d["gamma"]
    return oracle.quant_fp8(host_bits(x), None if r is None else host_bits(r), host_bits(g),
                            dtype=ODT[x.dtype], eps=w.eps, weight_offset=w.weight_offset,
                            scale_ub=w.scale_ub, want_pre=True)


@pytest.mark.gpu
@pytest.mark.parametrize("w,sched", CASES, ids=["fp8_residual", "offset_fp16", "short_rows"])
def test_static_scratch_matches_oracle_and_regular_entry_point_twice(w, sched):
    d = inputs(w, seed=77)
    ora = _oracle(d, w)
    with schedule(sched):
        ref = _outputs(d)
        _call("rmsnorm_quant_fp8", d, w, ref)
        for _ in range(2):                   # two calls in a row share the scratch array
            got = _outputs(d)
            _call("rmsnorm_quant_fp8_static_scratch", d, w, got)
            torch.cuda.synchronize()
            rep = P.compare_fp8(got[0].cpu().numpy(), got[1].cpu().numpy(),
                                None if got[2] is None else host_bits(got[2]), ora).check()
            assert rep["bad"] == 0
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
