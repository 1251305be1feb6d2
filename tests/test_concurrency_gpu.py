"""GPU tests of the claims the header makes about calling the library:
thread-safe calls from several host threads on their own streams, and calls
captured into a CUDA graph (the benchmark's launch method) giving the same
bits as eager calls.
"""
from __future__ import annotations

import threading

import numpy as np
import pytest
import torch

from memory_bound_normalization_fwd_gb300 import binding as B
from memory_bound_normalization_fwd_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_calls_from_several_threads_on_their_own_streams():
    # Eight host threads, each with its own stream and inputs, each mixing the
    # device forward, the host-buffer forward and the backward; every result
    # must equal the same call made alone.
    shapes = [(3000, 512, "bf16"), (1000, 4096, "fp16"), (700, 1000, "fp32"), (2000, 8192, "bf16"),
              (5000, 256, "bf16"), (500, 32768, "bf16"), (800, 777, "fp16"), (1200, 2048, "fp32")]
    inputs = []
    for i, (M, N, dt) in enumerate(shapes):
        x, w = W.generate(W.custom(M, N, dt, seed=i + 1))
        dy, _ = W.generate(W.custom(M, N, dt, seed=i + 100))
        inputs.append((W.to_torch(x, dt).cuda(), W.to_torch(w, dt).cuda(), W.to_torch(dy, dt).cuda(),
                       W.to_torch(x, dt).pin_memory()))

    def work(i, out):
        xd, wd, gd, xh = inputs[i]
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            for _ in range(5):
                y, r = B.fwd(xd, wd, eps=1e-6, offset=float(i % 2), stream=s)
                yh, rh = B.fwd_host(xh, wd, eps=1e-6, offset=float(i % 2), stream=s)
                dx, dw = B.bwd(xd, wd, r, gd, offset=float(i % 2), stream=s)
                res = (y, r, yh, rh, dx, dw)
        s.synchronize()
        out[i] = [t.cpu().clone() for t in res]

    out = {}
    threads = [threading.Thread(target=work, args=(i, out)) for i in range(len(shapes))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    alone = {}
    for i in range(len(shapes)):
        work(i, alone)
    for i in range(len(shapes)):
        for a, b in zip(out[i], alone[i]):
            if a.dtype in (torch.bfloat16, torch.float16):
                assert torch.equal(a.view(torch.int16), b.view(torch.int16)), i
            else:
                assert torch.equal(a.view(torch.int32), b.view(torch.int32)), i


@pytest.mark.parametrize("opts", [{}, {"early_loads": True}, {"early_weights": True},
                                  {"variant": "cluster"}, {"variant": "generic"}])
def test_graph_captured_calls_equal_eager_calls(opts):
    N = 65536 if opts.get("variant") == "cluster" else 1024
    M = 64 if N == 65536 else 4000
    xs = [W.to_torch(W.generate(W.custom(M, N, "bf16", seed=k))[0], "bf16").cuda() for k in range(4)]
    w = W.to_torch(W.generate(W.custom(M, N, "bf16", seed=9))[1], "bf16").cuda()
    o = B.make_options(**opts)
    s = torch.cuda.Stream()
    eager_y = [torch.empty_like(xs[0]) for _ in xs]
    eager_r = [torch.empty(M, device="cuda") for _ in xs]
    graph_y = [torch.full_like(xs[0], 7.0) for _ in xs]
    graph_r = [torch.full((M,), -1.0, device="cuda") for _ in xs]

    def calls(ys, rs):
        for x, y, r in zip(xs, ys, rs):
            assert B.rmsnorm_fwd_ex(x.data_ptr(), w.data_ptr(), y.data_ptr(), r.data_ptr(), M, N,
                                    1e-6, 1.0, B.BF16, o, s.cuda_stream) == 0, B.rmsnorm_last_error()

    with torch.cuda.stream(s):
        calls(eager_y, eager_r)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        calls(graph_y, graph_r)
    with torch.cuda.stream(s):
        g.replay()
    s.synchronize()
    for a, b, ra, rb in zip(eager_y, graph_y, eager_r, graph_r):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
        assert torch.equal(ra, rb)
