"""GPU: the pipelined schedule (quantisation of step i+1 on one stream while
the GEMM of step i runs on another, codes and scales double-buffered) gives
the same results, bit for bit, as running the steps one after another.

Each step uses different inputs, so a step that read the other buffer, or
a quantisation that overwrote codes still being read, would show up."""

import numpy as np
import pytest

from _helpers import lib, to_dev
from precision_linear_algebra_gb300 import workloads

pytestmark = pytest.mark.gpu


def test_two_stream_pipeline_matches_serial():
    import torch
    fl = lib()
    n, steps = 1024, 6
    A_np, B_np = workloads.square(n, seed=3)
    A0, B0 = to_dev(A_np), to_dev(B_np)
    # step i multiplies A by (i + 1) and B by 1 / (i + 2): new codes and scales
    As = [A0 * (i + 1) for i in range(steps)]
    Bs = [B0 / (i + 2) for i in range(steps)]

    # serial reference
    ref = []
    for i in range(steps):
        qa, _, sa = fl.quantize_pertensor(As[i])
        qb, _, sb = fl.quantize_pertensor(Bs[i])
        ref.append(fl.gemm(qa, qb, sa, sb).clone())
    torch.cuda.synchronize()

    main = torch.cuda.current_stream()
    sq, sg = torch.cuda.Stream(), torch.cuda.Stream()
    qa2 = [torch.empty((n, n), dtype=torch.uint8, device="cuda") for _ in range(2)]
    qb2 = [torch.empty((n, n), dtype=torch.uint8, device="cuda") for _ in range(2)]
    amax = torch.empty(4, dtype=torch.float32, device="cuda")
    scale = torch.empty(4, dtype=torch.float32, device="cuda")
    outs = [torch.empty((n, n), dtype=torch.bfloat16, device="cuda") for _ in range(steps)]
    qdone = [torch.cuda.Event(), torch.cuda.Event()]
    gdone = [torch.cuda.Event(), torch.cuda.Event()]
    for e in qdone + gdone:
        e.record(main)
    sq.wait_stream(main)
    sg.wait_stream(main)
    P = lambda t, i=0: t.data_ptr() + i * t.element_size()
    for i in range(steps):
        b = i & 1
        sq.wait_event(gdone[b])
        fl.fp8_quantize_pertensor(P(As[i]), n, n, n, P(qa2[b]), n, P(amax, 2 * b),
                                  P(scale, 2 * b), sq.cuda_stream)
        fl.fp8_quantize_pertensor(P(Bs[i]), n, n, n, P(qb2[b]), n, P(amax, 2 * b + 1),
                                  P(scale, 2 * b + 1), sq.cuda_stream)
        qdone[b].record(sq)
        sg.wait_event(qdone[b])
        fl.fp8_gemm(P(qa2[b]), n, P(qb2[b]), n, P(outs[i]), n, n, n, n,
                    P(scale, 2 * b), P(scale, 2 * b + 1), sg.cuda_stream)
        gdone[b].record(sg)
    main.wait_stream(sq)
    main.wait_stream(sg)
    torch.cuda.synchronize()
    assert fl.device_status() == 0
    for i in range(steps):
        assert torch.equal(outs[i].view(torch.int16), ref[i].view(torch.int16)), i
    # the steps really differ from each other
    assert not torch.equal(ref[0], ref[1])


def test_cuda_graph_capture_and_replay():
    """A quantize -> quantize -> GEMM step captured into a CUDA graph and
    replayed gives the eager result; replays see updated inputs."""
    import torch
    fl = lib()
    n = 512
    A_np, B_np = workloads.square(n, seed=4)
    A, B = to_dev(A_np), to_dev(B_np)
    qa = torch.empty((n, n), dtype=torch.uint8, device="cuda")
    qb = torch.empty_like(qa)
    amax = torch.empty(2, dtype=torch.float32, device="cuda")
    scale = torch.empty(2, dtype=torch.float32, device="cuda")
    C = torch.empty((n, n), dtype=torch.bfloat16, device="cuda")
    P = lambda t, i=0: t.data_ptr() + i * t.element_size()

    def launches(s):
        fl.fp8_quantize_pertensor(P(A), n, n, n, P(qa), n, P(amax, 0), P(scale, 0), s)
        fl.fp8_quantize_pertensor(P(B), n, n, n, P(qb), n, P(amax, 1), P(scale, 1), s)
        fl.fp8_gemm(P(qa), n, P(qb), n, P(C), n, n, n, n, P(scale, 0), P(scale, 1), s)

    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        launches(cap.cuda_stream)            # eager warm-up: one-time set-up
    torch.cuda.current_stream().wait_stream(cap)
    torch.cuda.synchronize()
    eager = C.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        launches(cap.cuda_stream)
    C.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(C.view(torch.int16), eager.view(torch.int16))
    # new inputs through the same graph
    A.mul_(3.0)
    B.mul_(0.5)
    g.replay()
    torch.cuda.synchronize()
    ref_qa, _, _ = fl.quantize_pertensor(A)
    ref_qb, _, _ = fl.quantize_pertensor(B)
    torch.cuda.synchronize()
    assert torch.equal(qa, ref_qa) and torch.equal(qb, ref_qb)
    assert fl.device_status() == 0
