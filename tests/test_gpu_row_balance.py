"""GPU tests of the dynamic row tail of the CTA-per-row schedule.

After an equal round-robin share, CTAs take their last rows one at a time from a per-launch
counter in the library's device memory. Which CTA handles a row must not change any output
bit. The counters are reused from a pool of 4096 slots and must come back clean, also when
launches overlap on two streams and after a timed-out wait has been reported."""
import pytest
import torch

import workloads as W
from gpu_common import check_fp8, inputs, rq

pytestmark = pytest.mark.gpu


def _fp8(d, w, stream=None):
    return rq().rmsnorm_quant_fp8(d["input"], d["gamma"], residual=d["residual"], epsilon=w.eps,
                                  scale_ub=w.scale_ub, stream=stream)


def _outputs_equal(a, b):
    return all(torch.equal(x.view(torch.uint8) if x.dtype == torch.float8_e4m3fn else x,
                           y.view(torch.uint8) if y.dtype == torch.float8_e4m3fn else y)
               for x, y in zip(a, b))


@pytest.mark.parametrize("mode", ["fp8", "nvfp4", "mxfp4"])
def test_dynamic_and_round_robin_rows_give_identical_bits(mode):
    w = W.Workload("custom", mode, 6000, 5120, "bf16", True, scale_ub=1200.0)
    d = inputs(w, seed=41)

    def run():
        if mode == "fp8":
            return _fp8(d, w)
        if mode == "nvfp4":
            gs = torch.full((1,), 2.5, device="cuda")
            return rq().rmsnorm_quant_nvfp4(d["input"], d["gamma"], global_scale=gs,
                                            residual=d["residual"])
        return rq().rmsnorm_quant_mxfp4(d["input"], d["gamma"], residual=d["residual"])

    prev = rq().rmsq_set_dynamic_rows(True)
    try:
        dyn = run()
        rq().rmsq_set_dynamic_rows(False)
        static = run()
    finally:
        rq().rmsq_set_dynamic_rows(prev)
    torch.cuda.synchronize()
    assert _outputs_equal(dyn, static)


def test_counter_pool_wraps_around_cleanly():
    # more launches than counter slots, back to back: every launch must see a clean counter
    w = W.config("fp8_residual", rows=1500)
    d = inputs(w, seed=42)
    ref = _fp8(d, w)
    for _ in range(4200):
        out = _fp8(d, w)
    torch.cuda.synchronize()
    assert _outputs_equal(ref, out)
    assert rq().rmsq_device_status() == 0
    check_fp8(w, d)


def test_launches_on_two_streams():
    w = W.config("fp8_residual", rows=3000)
    d1, d2 = inputs(w, seed=43), inputs(w, seed=44)
    ref1, ref2 = _fp8(d1, w), _fp8(d2, w)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    for _ in range(50):
        with torch.cuda.stream(s1):
            o1 = _fp8(d1, w, stream=s1)
        with torch.cuda.stream(s2):
            o2 = _fp8(d2, w, stream=s2)
        outs.append((o1, o2))
    torch.cuda.synchronize()
    for o1, o2 in outs:
        assert _outputs_equal(o1, ref1) and _outputs_equal(o2, ref2)


def test_rows_after_a_reported_timeout():
    assert rq().rmsq_device_status() == 0
    rq().rmsq_selftest_wait_timeout(2_000_000)
    assert rq().rmsq_device_status() == 8
    w = W.config("fp8_residual", rows=2000)
    check_fp8(w, inputs(w, seed=45))
