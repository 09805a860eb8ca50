"""Helpers for the GPU parity tests: run the CUDA path through the C ABI binding, run the oracle on
the same input bits (all rows, or a sample of rows at full sizes), and compare under the parity
rules of tests/parity.py."""
from __future__ import annotations

import contextlib

import numpy as np
import torch

import oracle
import parity as P
import workloads as W

ODT = {torch.bfloat16: oracle.BF16, torch.float16: oracle.FP16, torch.float32: oracle.F32}


def rq():
    import rmsnorm_precision_activation_gb300 as m
    return m


def host_bits(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.float32:
        return t.numpy()
    return t.view(torch.int16).numpy().view(np.uint16)


def sample_rows(rows: int, n: int = 64, seed: int = 0, extra=()) -> np.ndarray:
    if rows <= n + 2:
        return np.arange(rows)
    rng = np.random.default_rng(seed)
    idx = {0, rows - 1} | {int(i) for i in extra} | {int(i) for i in rng.choice(rows, n, replace=False)}
    return np.array(sorted(idx))


@contextlib.contextmanager
def schedule(s: int):
    prev = rq().rmsq_set_schedule(s)
    try:
        yield
    finally:
        rq().rmsq_set_schedule(prev)


def inputs(w: W.Workload, seed: int = 0, device="cuda", dtype=None):
    d = W.generate(w, seed=seed, device=device)
    if dtype is not None:
        d = {k: (None if v is None else v.to(dtype)) for k, v in d.items()}
    return d


def _rows(t, idx):
    return None if t is None else t[torch.as_tensor(idx, device=t.device)]


def check_fp8(w: W.Workload, d: dict, idx=None, scale_dtype=torch.float32):
    x, r, g = d["input"], d["residual"], d["gamma"]
    q, sc, ro = rq().rmsnorm_quant_fp8(x, g, residual=r, epsilon=w.eps,
                                       weight_offset=w.weight_offset, scale_ub=w.scale_ub,
                                       scale_dtype=scale_dtype)
    torch.cuda.synchronize()
    idx = np.arange(x.shape[0]) if idx is None else idx
    gq = _rows(q.view(torch.uint8), idx).cpu().numpy()
    gs_ = _rows(sc, idx).float().cpu().numpy()
    gro = None if r is None else host_bits(_rows(ro, idx))
    ora = oracle.quant_fp8(host_bits(_rows(x, idx)), None if r is None else host_bits(_rows(r, idx)),
                           host_bits(g), dtype=ODT[x.dtype], eps=w.eps,
                           weight_offset=w.weight_offset, scale_ub=w.scale_ub,
                           scale_dtype=ODT[scale_dtype], want_pre=True)
    rep = P.compare_fp8(gq, gs_, gro, ora)
    rep["clamped_rows"] = int((ora["scale"] >= np.float32(w.scale_ub / 448.0) * (1 - 1e-6)).sum())
    return rep.check(), ora


def oracle_global_scale(w: W.Workload, d: dict) -> np.float32:
    x, r, g = d["input"], d["residual"], d["gamma"]
    y = oracle.rmsnorm(host_bits(x), None if r is None else host_bits(r), host_bits(g),
                       dtype=ODT[x.dtype], eps=w.eps, weight_offset=w.weight_offset)["y"]
    return oracle.nvfp4_global_scale(np.abs(y).max())


def check_nvfp4(w: W.Workload, d: dict, gs: float, idx=None, swizzled=False):
    x, r, g = d["input"], d["residual"], d["gamma"]
    gst = torch.tensor([gs], dtype=torch.float32, device=x.device)
    q, bs, ro = rq().rmsnorm_quant_nvfp4(x, g, global_scale=gst, residual=r, epsilon=w.eps,
                                         weight_offset=w.weight_offset, swizzled=swizzled)
    torch.cuda.synchronize()
    rows, H = x.shape
    idx = np.arange(rows) if idx is None else idx
    gq = _rows(q, idx).cpu().numpy()
    if swizzled:
        gbs = P.unswizzle(bs.view(torch.uint8).cpu().numpy(), rows, H // 16)[idx]
    else:
        gbs = _rows(bs.view(torch.uint8), idx).cpu().numpy()
    gro = None if r is None else host_bits(_rows(ro, idx))
    ora = oracle.quant_nvfp4(host_bits(_rows(x, idx)), None if r is None else host_bits(_rows(r, idx)),
                             host_bits(g), float(gs), dtype=ODT[x.dtype], eps=w.eps,
                             weight_offset=w.weight_offset, want_y=True, want_pre=True)
    return P.compare_nvfp4(gq, gbs, gro, ora, gs).check(), (q, bs, ro)


def check_mxfp4(w: W.Workload, d: dict, idx=None, swizzled=False):
    x, r, g = d["input"], d["residual"], d["gamma"]
    q, bs, ro = rq().rmsnorm_quant_mxfp4(x, g, residual=r, epsilon=w.eps,
                                         weight_offset=w.weight_offset, swizzled=swizzled)
    torch.cuda.synchronize()
    rows, H = x.shape
    idx = np.arange(rows) if idx is None else idx
    gq = _rows(q, idx).cpu().numpy()
    if swizzled:
        gbs = P.unswizzle(bs.cpu().numpy(), rows, H // 32)[idx]
    else:
        gbs = _rows(bs, idx).cpu().numpy()
    gro = None if r is None else host_bits(_rows(ro, idx))
    ora = oracle.quant_mxfp4(host_bits(_rows(x, idx)), None if r is None else host_bits(_rows(r, idx)),
                             host_bits(g), dtype=ODT[x.dtype], eps=w.eps,
                             weight_offset=w.weight_offset, want_y=True, want_pre=True)
    return P.compare_mxfp4(gq, gbs, gro, ora).check(), (q, bs, ro)


GUARD = 4096       # canary bytes after every guarded output
GUARD_FILL = 0x5A


def guarded(n, dtype):
    """An output of n elements of dtype followed by GUARD canary bytes; returns (view, raw). A
    kernel that writes past the output changes raw[-GUARD:]."""
    itemsize = torch.empty(0, dtype=dtype).element_size()
    raw = torch.full((n * itemsize + GUARD,), GUARD_FILL, dtype=torch.uint8, device="cuda")
    return raw[: n * itemsize].view(dtype), raw


def guards_intact(raws) -> bool:
    return all(bool(torch.all(raw[-GUARD:] == GUARD_FILL)) for raw in raws)
