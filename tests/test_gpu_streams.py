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


def test_moe_two_stream_pipeline_matches_serial():
    """The MoE step pipelined the same way: step i+1's grouped activation
    quantisation and one-pass (carried-amax) weight quantisation on one
    stream while step i's grouped GEMM runs on another, with the routing
    offsets on the device.  Same results as the serial steps, bit for bit;
    every step has new activations and new routing."""
    import torch
    fl = lib()
    E, N, K, steps = 4, 256, 192, 5
    rng = np.random.default_rng(31)
    W = to_dev((rng.standard_normal((E, N, K)) * 0.02).astype(np.float32))
    offs = []
    Xs = []
    for i in range(steps):
        counts = rng.integers(0, 160, E) * (rng.random(E) > 0.2)
        offs.append(to_dev(np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)))
        Xs.append(to_dev(rng.standard_normal((640, K)).astype(np.float32)))
    P = lambda t, i=0: t.data_ptr() + i * t.element_size()

    def quant(x, off, qx, ax, sx, qw, hist, parity, sw, s):
        fl.fp8_quantize_pertensor_grouped(P(x), E, P(off), 640, K, K, P(qx), K, P(ax), P(sx), s)
        for e in range(E):
            fl.fp8_quantize_pertensor_delayed(P(W) + e * N * K * 4, N, K, K, P(qw) + e * N * K,
                                              K, P(hist[parity ^ 1], e), P(hist[parity], e),
                                              P(sw, e), 0, s)

    def gemm(off, qx, sx, qw, sw, out, s):
        fl.fp8_grouped_gemm(E, P(off), 640, P(qx), K, P(qw), K, N * K, P(out), N, N, K,
                            P(sx), P(sw), s)

    def seed_history():
        hist = torch.empty((2, E), dtype=torch.float32, device="cuda")
        sw = torch.empty(E, dtype=torch.float32, device="cuda")
        q = torch.empty((E, N, K), dtype=torch.uint8, device="cuda")
        for e in range(E):
            for parity in (0, 1):
                fl.fp8_quantize_pertensor(P(W) + e * N * K * 4, N, K, K, P(q) + e * N * K, K,
                                          P(hist[parity], e), P(sw, e),
                                          torch.cuda.current_stream().cuda_stream)
        return hist

    def buffers():
        return (torch.empty((640, K), dtype=torch.uint8, device="cuda"),
                torch.empty(E, dtype=torch.float32, device="cuda"),
                torch.empty(E, dtype=torch.float32, device="cuda"),
                torch.empty((E, N, K), dtype=torch.uint8, device="cuda"),
                torch.empty(E, dtype=torch.float32, device="cuda"))

    # serial reference
    cur = torch.cuda.current_stream().cuda_stream
    hist = seed_history()
    qx, ax, sx, qw, sw = buffers()
    ref = []
    for i in range(steps):
        out = torch.full((640, N), 9.0, dtype=torch.bfloat16, device="cuda")
        quant(Xs[i], offs[i], qx, ax, sx, qw, hist, i & 1, sw, cur)
        gemm(offs[i], qx, sx, qw, sw, out, cur)
        ref.append(out)
    torch.cuda.synchronize()

    # pipelined
    hist = seed_history()
    bufs = [buffers(), buffers()]
    outs = [torch.full((640, N), 9.0, dtype=torch.bfloat16, device="cuda") for _ in range(steps)]
    main = torch.cuda.current_stream()
    sq, sg = torch.cuda.Stream(), torch.cuda.Stream()
    qdone = [torch.cuda.Event(), torch.cuda.Event()]
    gdone = [torch.cuda.Event(), torch.cuda.Event()]
    for ev in qdone + gdone:
        ev.record(main)
    sq.wait_stream(main)
    sg.wait_stream(main)
    for i in range(steps):
        b = i & 1
        qx, ax, sx, qw, sw = bufs[b]
        sq.wait_event(gdone[b])
        quant(Xs[i], offs[i], qx, ax, sx, qw, hist, i & 1, sw, sq.cuda_stream)
        qdone[b].record(sq)
        sg.wait_event(qdone[b])
        gemm(offs[i], qx, sx, qw, sw, outs[i], sg.cuda_stream)
        gdone[b].record(sg)
    main.wait_stream(sq)
    main.wait_stream(sg)
    torch.cuda.synchronize()
    assert fl.device_status() == 0
    for i in range(steps):
        assert torch.equal(outs[i].view(torch.int16), ref[i].view(torch.int16)), i
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


def test_blockscaled_linears_pipeline_matches_serial():
    """Several linears in a row, pipelined per linear: linear k+1's block
    quantisation (activations and weights) on one stream while linear k's
    block-scaled GEMM runs on another, across step boundaries, each linear
    with its own code and scale buffers.  Same results as the serial steps,
    bit for bit; every step has new activations."""
    import torch
    fl = lib()
    rng = np.random.default_rng(41)
    shapes = [(96, 160, 256), (96, 64, 320), (96, 224, 96)]      # (M, N, K) per linear
    steps = 4
    Ws = [to_dev((rng.standard_normal((N, K)) * 0.02).astype(np.float32)) for _, N, K in shapes]
    Xs = [[to_dev(rng.standard_normal((M, K)).astype(np.float32)) for M, _, K in shapes]
          for _ in range(steps)]

    def buffers(M, N, K):
        kb = (K + 31) // 32
        sc = lambda r: torch.zeros((r, (kb + 3) // 4 * 4), dtype=torch.float32,
                                   device="cuda")[:, :kb]
        return (torch.empty((M, K), dtype=torch.uint8, device="cuda"),
                torch.empty((N, K), dtype=torch.uint8, device="cuda"),
                sc((M + 31) // 32), sc((N + 31) // 32))

    def quant(k, x, buf, s):
        M, N, K = shapes[k]
        qx, qw, sx, sw = buf
        fl.fp8_quantize_blockwise_32x32(x.data_ptr(), M, K, K, qx.data_ptr(), K,
                                        sx.data_ptr(), sx.stride(0), s)
        fl.fp8_quantize_blockwise_32x32(Ws[k].data_ptr(), N, K, K, qw.data_ptr(), K,
                                        sw.data_ptr(), sw.stride(0), s)

    def gemm(k, buf, out, s):
        M, N, K = shapes[k]
        qx, qw, sx, sw = buf
        fl.fp8_gemm_blockscaled_32x32(qx.data_ptr(), K, qw.data_ptr(), K, out.data_ptr(), N,
                                      M, N, K, sx.data_ptr(), sx.stride(0), sw.data_ptr(),
                                      sw.stride(0), s)

    def outputs():
        return [[torch.full((M, N), 9.0, dtype=torch.bfloat16, device="cuda")
                 for M, N, _ in shapes] for _ in range(steps)]

    cur = torch.cuda.current_stream().cuda_stream
    bufs = [buffers(*sh) for sh in shapes]
    ref = outputs()
    for i in range(steps):
        for k in range(len(shapes)):
            quant(k, Xs[i][k], bufs[k], cur)
            gemm(k, bufs[k], ref[i][k], cur)
    torch.cuda.synchronize()

    bufs = [buffers(*sh) for sh in shapes]
    got = outputs()
    main = torch.cuda.current_stream()
    sq, sg = torch.cuda.Stream(), torch.cuda.Stream()
    qdone = [torch.cuda.Event() for _ in shapes]
    gdone = [torch.cuda.Event() for _ in shapes]
    for ev in qdone + gdone:
        ev.record(main)
    sq.wait_stream(main)
    sg.wait_stream(main)
    for i in range(steps):
        for k in range(len(shapes)):
            sq.wait_event(gdone[k])
            quant(k, Xs[i][k], bufs[k], sq.cuda_stream)
            qdone[k].record(sq)
            sg.wait_event(qdone[k])
            gemm(k, bufs[k], got[i][k], sg.cuda_stream)
            gdone[k].record(sg)
    main.wait_stream(sq)
    main.wait_stream(sg)
    torch.cuda.synchronize()
    assert fl.device_status() == 0
    for i in range(steps):
        for k in range(len(shapes)):
            assert torch.equal(got[i][k].view(torch.int16), ref[i][k].view(torch.int16)), (i, k)
    assert not torch.equal(ref[0][0], ref[1][0])
