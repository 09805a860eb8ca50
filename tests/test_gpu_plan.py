"""The planner with the device's own shared-memory limits.

The CPU tests of the planner use GB300's limits (opt-in per CTA, per SM, reserved per CTA); here
rmsq_plan reads them from the current device, and every plan must be the one those tests
checked."""
import pytest
import torch

from gpu_common import rq

pytestmark = pytest.mark.gpu


def test_device_limits_are_gb300s():
    m = rq()
    cases = [("fp8", torch.float16, 8192, True, 1.0), ("nvfp4", torch.bfloat16, 7168, False, 0.0),
             ("mxfp4", torch.bfloat16, 2048, True, 0.0), ("mxfp4", torch.bfloat16, 16384, True, 0.0),
             ("fp8", torch.bfloat16, 4096, True, 0.0), ("fp8", torch.bfloat16, 1024, False, 0.0),
             ("fp8", torch.bfloat16, 65536, True, 0.0), ("nvfp4", torch.bfloat16, 131072, True, 0.0),
             ("global_scale", torch.bfloat16, 7168, False, 0.0),
             ("fp8", torch.float32, 65536, True, 0.0)]
    for mode, dt, h, res, off in cases:
        dev = m.rmsq_plan(mode, dt, h, residual=res, weight_offset=off, smem=None)
        ref = m.rmsq_plan(mode, dt, h, residual=res, weight_offset=off)
        assert dev == ref, (mode, dt, h, res, off, dev, ref)
    props = torch.cuda.get_device_properties(0)
    optin = getattr(props, "shared_memory_per_block_optin", None)
    if optin is not None:
        assert optin == m.GB300_SMEM[0]
