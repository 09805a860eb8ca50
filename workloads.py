"""Seeded synthetic inputs for the fused residual-add + RMSNorm + FP8 / NVFP4 / MXFP4 op.

This module holds no arithmetic of the method: it only draws the inputs (activation, residual,
gamma) with the shapes and value distributions of the five benchmark workloads, from a seeded
torch generator. Both the CUDA path's callers and the oracle's callers take their inputs from here.

Distributions (the pages name no dataset; every input is synthetic):
  fp8_small       64 x 4096 bf16, x ~ N(0,1); gamma ~ N(1,0.1); eps 1e-6; offset 0; ub 1200
  fp8_residual    8192 x 4096 bf16, x ~ N(0,0.5) with Bernoulli(0.001) elements multiplied by 50;
                  residual ~ N(0,1); gamma ~ N(1,0.1); ub 1200
  fp8_gemma       16384 x 8192 fp16, x, residual ~ N(0,1); 1 % of rows (Bernoulli per row) have
                  x * 200; gamma ~ N(0,0.05); offset 1.0; ub 10
  fp8_gemma_spike as fp8_gemma, but a chosen row gets one element * 200 instead of the whole row,
                  which drives amax(y) above ub = 10 (RMSNorm removes a whole-row scale)
  nvfp4           32768 x 7168 bf16, x ~ N(0,1) with Bernoulli(0.005) elements replaced by
                  Laplace(0, 10); gamma ~ N(1,0.1); no residual; gs = 448 * 6 / amax(y)
  mxfp4_residual  rows in {1,16,128,4096,65536} x hidden in {2048,5120,8192,16384} bf16,
                  x, residual ~ N(0,1); gamma ~ N(1,0.1)
Laplace samples are drawn by inverse CDF from a uniform; outlier masks are i.i.d. Bernoulli.
"""
from __future__ import annotations

import dataclasses

import torch

MXFP4_ROWS = (1, 16, 128, 4096, 65536)
MXFP4_HIDDEN = (2048, 5120, 8192, 16384)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    mode: str            # "fp8" | "nvfp4" | "mxfp4"
    rows: int
    hidden: int
    dtype: str           # "bf16" | "fp16"
    residual: bool
    eps: float = 1e-6
    weight_offset: float = 0.0
    scale_ub: float = 1200.0

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float16

    def with_rows(self, rows: int) -> "Workload":
        return dataclasses.replace(self, rows=rows)

    def algorithmic_bytes(self) -> int:
        """Bytes the op must move once: inputs read, outputs written, gamma once per launch."""
        e = 2
        n = self.rows * self.hidden
        read = n * e * (2 if self.residual else 1) + self.hidden * e
        write = n * e if self.residual else 0
        if self.mode == "fp8":
            write += n + 4 * self.rows
        elif self.mode == "nvfp4":
            read += 4                      # the fp32 global scale
            write += n // 2 + n // 16
        else:
            write += n // 2 + n // 32
        return read + write


CONFIGS = {
    "fp8_small": Workload("fp8_small", "fp8", 64, 4096, "bf16", False),
    "fp8_residual": Workload("fp8_residual", "fp8", 8192, 4096, "bf16", True),
    "fp8_gemma": Workload("fp8_gemma", "fp8", 16384, 8192, "fp16", True, weight_offset=1.0,
                          scale_ub=10.0),
    "fp8_gemma_spike": Workload("fp8_gemma_spike", "fp8", 16384, 8192, "fp16", True,
                                weight_offset=1.0, scale_ub=10.0),
    "nvfp4": Workload("nvfp4", "nvfp4", 32768, 7168, "bf16", False),
    "mxfp4_residual": Workload("mxfp4_residual", "mxfp4", 65536, 16384, "bf16", True),
}


def config(name: str, rows: int | None = None, hidden: int | None = None) -> Workload:
    w = CONFIGS[name]
    if rows is not None:
        w = dataclasses.replace(w, rows=rows)
    if hidden is not None:
        w = dataclasses.replace(w, hidden=hidden)
    return w


def _normal(shape, mean, std, g, device):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std + mean


def _laplace(shape, b, g, device):
    u = torch.rand(shape, generator=g, device=device, dtype=torch.float32) - 0.5
    u = u.clamp(-0.4999999, 0.4999999)
    return -b * torch.sign(u) * torch.log1p(-2.0 * u.abs())


def generate(w: Workload, seed: int = 0, device: str | torch.device = "cpu") -> dict:
    """Draw (input, residual or None, gamma) for workload w. Returns tensors of w's dtype.

    The draw order is fixed (gamma, then input, then residual), so a given seed and device give
    the same bits on any machine of the same torch build."""
    device = torch.device(device)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    R, H = w.rows, w.hidden
    dt = w.torch_dtype
    if w.name.startswith("fp8_gemma"):
        gamma = _normal((H,), 0.0, 0.05, g, device)
    else:
        gamma = _normal((H,), 1.0, 0.1, g, device)

    if w.name == "fp8_residual":
        x = _normal((R, H), 0.0, 0.5, g, device)
        mask = torch.rand((R, H), generator=g, device=device) < 0.001
        x = torch.where(mask, x * 50.0, x)
    elif w.name == "fp8_gemma":
        x = _normal((R, H), 0.0, 1.0, g, device)
        rowmask = torch.rand((R, 1), generator=g, device=device) < 0.01
        x = torch.where(rowmask, x * 200.0, x)
    elif w.name == "fp8_gemma_spike":
        x = _normal((R, H), 0.0, 1.0, g, device)
        rowmask = torch.rand((R,), generator=g, device=device) < 0.01
        col = torch.randint(0, H, (R,), generator=g, device=device)
        rows = torch.nonzero(rowmask).flatten()
        x[rows, col[rows]] *= 200.0
    elif w.name == "nvfp4":
        x = _normal((R, H), 0.0, 1.0, g, device)
        mask = torch.rand((R, H), generator=g, device=device) < 0.005
        x = torch.where(mask, _laplace((R, H), 10.0, g, device), x)
    else:  # fp8_small, mxfp4_residual and any custom shape: x ~ N(0,1)
        x = _normal((R, H), 0.0, 1.0, g, device)

    residual = _normal((R, H), 0.0, 1.0, g, device).to(dt) if w.residual else None
    return dict(input=x.to(dt), residual=residual, gamma=gamma.to(dt))


def bits(t: torch.Tensor):
    """bf16 / fp16 tensor -> numpy uint16 bit patterns (CPU copy)."""
    import numpy as np
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def ideal_us(w: Workload, gbs: float) -> float:
    return w.algorithmic_bytes() / (gbs * 1e9) * 1e6


def describe(w: Workload) -> str:
    return "%s %dx%d %s%s" % (w.mode, w.rows, w.hidden, w.dtype, " +residual" if w.residual else "")


