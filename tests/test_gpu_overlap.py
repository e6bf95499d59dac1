"""Launch overlap (programmatic dependent launch) changes no result.

A chain of GEMVs where each one reads the previous one's output (y of one is x of
the next, across kernel families: streaming, warp per row, batched ring, row pair,
split-K, tensor cores), run eagerly and from a CUDA graph with every overlap mode:
bit-identical to plain launches.  With "weights" the weights are written before the
chain starts, never inside it.
"""
from __future__ import annotations

import pytest
import torch

import decode_linear_layers_gb300 as g

pytestmark = pytest.mark.gpu

# (rows, vectors) per link: every link's K is the previous link's rows
CHAIN = [(4096, 1), (4096, 1), (65536, 1), (4096, 4), (2048, 16), (512, 3), (8, 2), (4096, 32), (1024, 1)]


def _weights(K0):
    gen = torch.Generator().manual_seed(11)
    ws, K = [], K0
    for M, _ in CHAIN:
        ws.append((torch.randn(M, K, generator=gen) / K ** 0.5).to(torch.bfloat16).cuda())
        K = M
    return ws


def _run_chain(ws, x0):
    ys = []
    x = x0
    for (M, B), A in zip(CHAIN, ws):
        K = A.shape[1]
        xin = x[:1].expand(B, K).contiguous() if x.shape[0] != B else x
        y = torch.empty(B, M, dtype=torch.bfloat16, device="cuda")
        g.gemv_bf16(A, xin, None, y, M, K, B)
        ys.append(y)
        x = y
    return ys


@pytest.mark.parametrize("mode", ["launch", "weights"])
def test_overlap_chain_bitwise(mode):
    K0 = 4096
    ws = _weights(K0)
    x0 = torch.randn(1, K0, generator=torch.Generator().manual_seed(12)).to(torch.bfloat16).cuda()
    g.set_launch_overlap("off")
    ref = _run_chain(ws, x0)
    torch.cuda.synchronize()
    try:
        g.set_launch_overlap(mode)
        got = _run_chain(ws, x0)
        torch.cuda.synchronize()
        for i, (a, b) in enumerate(zip(ref, got)):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16)), f"link {i} differs with overlap {mode}"
        # the same chain captured in a CUDA graph and replayed
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            _run_chain(ws, x0)
        torch.cuda.current_stream().wait_stream(s)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            out = _run_chain(ws, x0)
        for y in out:
            y.zero_()
        graph.replay()
        torch.cuda.synchronize()
        for i, (a, b) in enumerate(zip(ref, out)):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16)), f"graph link {i} differs ({mode})"
    finally:
        g.set_launch_overlap("launch")  # the default

