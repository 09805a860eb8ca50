"""The entry points inside a captured CUDA graph.

Every argument the kernels read at run time lives in device memory (inputs, gamma, the NVFP4
global scale), and the scratch a launch uses (the row counter of the dynamic row tail, the
pre-pass's running maximum) starts and ends each launch at zero. So a graph captured once can be
replayed on new inputs copied into the captured buffers. This test captures the global-scale
pre-pass followed by the NVFP4 quantiser that reads its result, the FP8 quantiser (with and
without a weight offset) and the MXFP4 quantiser, replays the graph three times on fresh inputs,
and compares every output bit for bit with eager calls on the same inputs."""
import pytest
import torch

import workloads as W
from gpu_common import rq

pytestmark = pytest.mark.gpu


def _fill(bufs, seed):
    for k, (w, d) in enumerate(bufs):
        fresh = W.generate(w, seed=seed + k, device="cuda")
        for name, t in d.items():
            if t is not None and name != "gamma":
                t.copy_(fresh[name])


def test_graph_replay_matches_eager_calls():
    m = rq()
    fp8 = W.config("fp8_residual")                                              # W16, row tail
    fp8o = W.Workload("custom", "fp8", 4096, 8192, "fp16", True, weight_offset=1.0, scale_ub=10.0)
    nv = W.Workload("custom", "nvfp4", 8192, 2048, "bf16", False)
    mx = W.Workload("custom", "mxfp4", 8192, 4096, "bf16", True)
    bufs = [(w, W.generate(w, seed=3, device="cuda")) for w in (fp8, fp8o, nv, mx)]

    def outputs():
        o = {}
        for w, d in bufs:
            x = d["input"]
            if w.mode == "fp8":
                o[w] = (torch.empty(x.shape, dtype=torch.float8_e4m3fn, device="cuda"),
                        torch.empty(x.shape[0], dtype=torch.float32, device="cuda"),
                        torch.empty_like(x) if w.residual else None)
            else:
                blk = 16 if w.mode == "nvfp4" else 32
                o[w] = (torch.empty(x.shape[0], x.shape[1] // 2, dtype=torch.uint8, device="cuda"),
                        torch.empty(x.shape[0], x.shape[1] // blk, dtype=torch.uint8, device="cuda"),
                        torch.empty_like(x) if w.residual else None)
        o["gs"] = torch.empty(1, dtype=torch.float32, device="cuda")
        return o

    def run(o):
        for w, d in bufs:
            x, r, g = d["input"], d["residual"], d["gamma"]
            q, sc, ro = o[w]
            if w.mode == "fp8":
                m.rmsnorm_quant_fp8(x, g, residual=r, residual_output=ro, epsilon=w.eps,
                                    weight_offset=w.weight_offset, scale_ub=w.scale_ub,
                                    output=q, scale_output=sc)
            elif w.mode == "nvfp4":
                m.rmsnorm_nvfp4_global_scale(x, g, residual=r, epsilon=w.eps, out=o["gs"])
                m.rmsnorm_quant_nvfp4(x, g, global_scale=o["gs"], residual=r, residual_output=ro,
                                      epsilon=w.eps, output=q, block_scale=sc.view(torch.float8_e4m3fn))
            else:
                m.rmsnorm_quant_mxfp4(x, g, residual=r, residual_output=ro, epsilon=w.eps,
                                      output=q, block_scale=sc)

    graph_out, eager_out = outputs(), outputs()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        run(graph_out)                       # warm-up: function attributes, occupancy
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run(graph_out)
    for rep in range(3):
        _fill(bufs, seed=100 + 10 * rep)
        graph.replay()
        run(eager_out)
        torch.cuda.synchronize()
        assert torch.equal(graph_out["gs"], eager_out["gs"])
        for w, _ in bufs:
            for a, b in zip(graph_out[w], eager_out[w]):
                if a is not None:
                    assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), (rep, w.mode)
    assert m.rmsq_device_status() == 0
