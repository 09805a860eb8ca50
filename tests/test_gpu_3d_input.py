"""3-D input through the three Python entry points.

FlashInfer's rmsnorm_fp4quant accepts a [B, T, H] activation and treats it as B*T rows of H (its
input validation folds the leading dimensions). The binding does the same: it views a
contiguous [..., H] tensor as rows and returns outputs with the input's leading dimensions. These
tests pass [B, T, H] input (with and without a residual) to rmsnorm_quant_fp8, _nvfp4 and
_mxfp4, check that every output keeps the leading dimensions, compare the flattened rows element
by element with the oracle under the parity rules, and check that the results are bit-identical
to the same call on the [B*T, H] view."""
import numpy as np
import pytest
import torch

import oracle
import parity as P
import workloads as W
from gpu_common import ODT, host_bits, inputs, oracle_global_scale, rq

pytestmark = pytest.mark.gpu

B, T = 3, 45


def _pair(d, residual):
    x = d["input"]
    H = x.shape[-1]
    x3 = x.reshape(B, T, H)
    r3 = d["residual"].reshape(B, T, H) if residual else None
    return x3, r3


@pytest.mark.parametrize("residual", [False, True])
@pytest.mark.parametrize("hidden", [2048, 7168])
def test_fp8_3d(hidden, residual):
    w = W.Workload("custom", "fp8", B * T, hidden, "bf16", residual, scale_ub=1200.0)
    d = inputs(w, seed=hidden + residual)
    x3, r3 = _pair(d, residual)
    q3, s3, ro3 = rq().rmsnorm_quant_fp8(x3, d["gamma"], residual=r3, epsilon=w.eps,
                                         scale_ub=w.scale_ub)
    q2, s2, ro2 = rq().rmsnorm_quant_fp8(d["input"], d["gamma"], residual=d["residual"],
                                         epsilon=w.eps, scale_ub=w.scale_ub)
    torch.cuda.synchronize()
    assert q3.shape == (B, T, hidden) and s3.shape == (B, T)
    assert torch.equal(q3.view(torch.uint8).reshape(-1, hidden), q2.view(torch.uint8))
    assert torch.equal(s3.reshape(-1), s2)
    if residual:
        assert ro3.shape == (B, T, hidden)
        assert torch.equal(ro3.reshape(-1, hidden), ro2)
    else:
        assert ro3 is None
    ora = oracle.quant_fp8(host_bits(d["input"]), host_bits(d["residual"]) if residual else None,
                           host_bits(d["gamma"]), dtype=ODT[torch.bfloat16], eps=w.eps,
                           scale_ub=w.scale_ub, want_pre=True)
    P.compare_fp8(q3.view(torch.uint8).reshape(-1, hidden).cpu().numpy(),
                  s3.reshape(-1).cpu().numpy(),
                  host_bits(ro3.reshape(-1, hidden)) if residual else None, ora).check()


@pytest.mark.parametrize("residual", [False, True])
def test_nvfp4_3d(residual):
    hidden = 7168
    w = W.Workload("custom", "nvfp4", B * T, hidden, "bf16", residual)
    d = inputs(w, seed=31 + residual)
    x3, r3 = _pair(d, residual)
    # the device pre-pass takes the 3-D tensor too and agrees with the oracle's global scale
    gs3 = rq().rmsnorm_nvfp4_global_scale(x3, d["gamma"], residual=r3, epsilon=w.eps)
    gs2 = rq().rmsnorm_nvfp4_global_scale(d["input"], d["gamma"], residual=d["residual"],
                                          epsilon=w.eps)
    gs_ora = float(oracle_global_scale(w, d))
    assert torch.equal(gs3, gs2)
    assert abs(float(gs3.cpu()[0]) - gs_ora) <= 2e-6 * gs_ora
    gst = torch.tensor([gs_ora], dtype=torch.float32, device="cuda")
    q3, b3, ro3 = rq().rmsnorm_quant_nvfp4(x3, d["gamma"], global_scale=gst, residual=r3,
                                           epsilon=w.eps)
    q2, b2, ro2 = rq().rmsnorm_quant_nvfp4(d["input"], d["gamma"], global_scale=gst,
                                           residual=d["residual"], epsilon=w.eps)
    torch.cuda.synchronize()
    assert q3.shape == (B, T, hidden // 2) and b3.shape == (B, T, hidden // 16)
    assert torch.equal(q3.reshape(-1, hidden // 2), q2)
    assert torch.equal(b3.view(torch.uint8).reshape(-1, hidden // 16), b2.view(torch.uint8))
    if residual:
        assert torch.equal(ro3.reshape(-1, hidden), ro2)
    ora = oracle.quant_nvfp4(host_bits(d["input"]), host_bits(d["residual"]) if residual else None,
                             host_bits(d["gamma"]), gs_ora, dtype=ODT[torch.bfloat16], eps=w.eps,
                             want_y=True, want_pre=True)
    P.compare_nvfp4(q3.reshape(-1, hidden // 2).cpu().numpy(),
                    b3.view(torch.uint8).reshape(-1, hidden // 16).cpu().numpy(),
                    host_bits(ro3.reshape(-1, hidden)) if residual else None, ora, gs_ora).check()


@pytest.mark.parametrize("residual", [False, True])
@pytest.mark.parametrize("hidden", [2048, 5120])
def test_mxfp4_3d(hidden, residual):
    w = W.Workload("custom", "mxfp4", B * T, hidden, "bf16", residual)
    d = inputs(w, seed=53 + hidden + residual)
    x3, r3 = _pair(d, residual)
    q3, b3, ro3 = rq().rmsnorm_quant_mxfp4(x3, d["gamma"], residual=r3, epsilon=w.eps)
    q2, b2, ro2 = rq().rmsnorm_quant_mxfp4(d["input"], d["gamma"], residual=d["residual"],
                                           epsilon=w.eps)
    torch.cuda.synchronize()
    assert q3.shape == (B, T, hidden // 2) and b3.shape == (B, T, hidden // 32)
    assert torch.equal(q3.reshape(-1, hidden // 2), q2)
    assert torch.equal(b3.reshape(-1, hidden // 32), b2)
    if residual:
        assert torch.equal(ro3.reshape(-1, hidden), ro2)
    ora = oracle.quant_mxfp4(host_bits(d["input"]), host_bits(d["residual"]) if residual else None,
                             host_bits(d["gamma"]), dtype=ODT[torch.bfloat16], eps=w.eps,
                             want_y=True, want_pre=True)
    P.compare_mxfp4(q3.reshape(-1, hidden // 2).cpu().numpy(),
                    b3.reshape(-1, hidden // 32).cpu().numpy(),
                    host_bits(ro3.reshape(-1, hidden)) if residual else None, ora).check()
    assert np.all(b3.cpu().numpy() <= 254)
