"""Host-side check of the persistent kernels' row walks (no GPU).

The streaming kernel deals rows to warps round-robin and, in SwiGLU mode, walks
(gate row p, up row p + I) pairs.  These loops mirror its index arithmetic for
the shapes it runs on and check that every row or pair is visited by exactly one
warp and that every walk ends.
"""
import pytest


def stream_walk(M, G, W, b, w):
    row, out, steps = b + G * w, [], 0
    while row < M:
        out.append(row)
        row += G * W
        steps += 1
        assert steps <= M
    return out


def swiglu_walk(half, G, W, b, w):
    M, rstride = 2 * half, G * W

    def nxt(r):
        if r < half:
            return r + half
        np_ = r - half + rstride
        return np_ if np_ < half else M

    row = b + G * w
    if row >= half:
        row = M
    out, steps = [], 0
    while row < M:
        out.append(row)
        row = nxt(row)
        steps += 1
        assert steps <= M, "walk does not end"
    return out


@pytest.mark.parametrize("M,G,W", [(16384, 608, 16), (4096, 304, 16), (7, 304, 16), (128256, 304, 16)])
def test_stream_rows_once(M, G, W):
    seen = []
    for b in range(G):
        for w in range(W):
            seen += stream_walk(M, G, W, b, w)
    assert sorted(seen) == list(range(M))


@pytest.mark.parametrize("half,G,W", [(14336, 304, 16), (777, 304, 16), (777, 608, 16), (5, 304, 16),
                                      (4864, 304, 16), (4865, 304, 16), (30000, 608, 16)])
def test_swiglu_pairs_once(half, G, W):
    gates = []
    for b in range(G):
        for w in range(W):
            s = swiglu_walk(half, G, W, b, w)
            assert len(s) % 2 == 0
            for i in range(0, len(s), 2):
                assert s[i] < half and s[i + 1] == s[i] + half
                gates.append(s[i])
    assert sorted(gates) == list(range(half))
