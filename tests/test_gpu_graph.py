"""libgemv calls captured into a CUDA graph and replayed.

A decode step issues the same GEMVs every token; capturing them once into a CUDA
graph removes the per-launch host cost (the glossary page's note that CUDA graphs
separate kernel time from launch overhead).  The entry points only enqueue work
on the caller's stream, and split-K takes its scratch from the stream-ordered
pool, so the whole sequence can be captured.  Replays must give bit-identical
results to eager calls on the same data, including after the inputs change in
place.
"""
from __future__ import annotations

import pytest
import torch

import decode_linear_layers_gb300 as g
import workloads as W
from tests import gpu_util as U

pytestmark = pytest.mark.gpu

# one shape per kernel family the dispatcher picks, plus a forced split-K
STEP = [
    ("bf16", 6144, 4096, 1, False, "auto"),       # stream
    ("bf16", 256, 65536, 1, True, "auto"),        # split-K (few long rows)
    ("f16", 2048, 4096, 16, False, "auto"),       # batched, B > 4
    ("w8", 1024, 8192, 4, True, "auto"),          # batched, B <= 4
    ("f32", 16384, 32, 1, True, "auto"),          # rows per warp
    ("bf16", 1000, 2048, 2, True, "split_k"),     # forced split-K with B = 2
    ("bf16", 4096, 4096, 4, True, "xsplit"),      # K split over a CTA, cp.async ring
]


def _setup(seed0=900):
    items = []
    for i, (dt, M, K, B, bias, kern) in enumerate(STEP):
        w = W.small(dt, M, K, B, bias, seed=seed0 + i)
        d = U.to_device(W.make_inputs(w))
        y = torch.empty((B, M), dtype=U.out_dtype(dt), device="cuda")
        items.append((dt, M, K, B, kern, d, y))
    return items


def _run_all(items):
    for (dt, M, K, B, kern, d, y) in items:
        g.force_kernel(kern)
        U.call(dt, d, y, M, K, B)
    g.force_kernel("auto")


def test_capture_and_replay_match_eager():
    items = _setup()
    torch.cuda.synchronize()
    # eager reference
    _run_all(items)
    torch.cuda.synchronize()
    eager = [y.clone() for (*_, y) in items]
    # capture (a warm-up pass outside capture first, as torch recommends)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _run_all(items)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    for (*_, y) in items:
        y.zero_()
    with torch.cuda.graph(graph):
        _run_all(items)
    graph.replay()
    torch.cuda.synchronize()
    for (dt, M, K, B, kern, d, y), ye in zip(items, eager):
        assert torch.equal(y, ye), (dt, M, K, B, kern)


def test_replay_follows_new_inputs():
    items = _setup(seed0=950)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _run_all(items)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        _run_all(items)
    # new activations written in place into the captured buffers
    gen = torch.Generator(device="cpu").manual_seed(7)
    for (dt, M, K, B, kern, d, y) in items:
        d["x"].copy_(torch.randn(d["x"].shape, generator=gen).to(d["x"].dtype))
    graph.replay()
    torch.cuda.synchronize()
    got = [y.clone() for (*_, y) in items]
    _run_all(items)
    torch.cuda.synchronize()
    for (dt, M, K, B, kern, d, y), yg in zip(items, got):
        assert torch.equal(y, yg), (dt, M, K, B, kern)
        # and the replayed result is right, not just repeatable
        inp = {k: (None if v is None else v.cpu()) for k, v in d.items()}
        y_ref, absdot = U.oracle_for(dt, inp)
        U.assert_close(dt, yg, y_ref, absdot, with_rounding=True, what=f"graph {dt} {M}x{K} B={B}")
