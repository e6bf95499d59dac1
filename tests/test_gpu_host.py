"""gemv_host: the GEMV with its operands in host memory (copies inside the call).

* every storage type: y from host buffers equals, bit for bit, y from the device call
  on the same values, and matches the oracle;
* weights (and scales) resident on the device: h_A = NULL skips their copy;
* argument errors come back before any copy.
"""
from __future__ import annotations

import pytest
import torch

import decode_linear_layers_gb300 as g
import workloads as W
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


def _pinned(t):
    return None if t is None else t.contiguous().pin_memory()


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16", "w8", "w4"])
@pytest.mark.parametrize("B", [1, 3, 16])
def test_host_matches_device_call(dtype, B):
    M, K = 1000, 1024
    w = W.small(dtype, M, K, B, True, seed=5000 + B)
    inp = W.make_inputs(w)
    y_ref, absdot = U.oracle_for(dtype, inp)
    d = U.to_device(inp)
    y_dev = U.run_gpu(dtype, d, M, K, B)
    h = {k: _pinned(v) for k, v in inp.items()}
    hy = torch.empty(B, M, dtype=U.out_dtype(dtype)).pin_memory()
    dd = {k: (None if v is None else torch.empty_like(v, device="cuda")) for k, v in inp.items()}
    dy = torch.empty(B, M, dtype=U.out_dtype(dtype), device="cuda")
    g.gemv_host(dtype, h["A"], h["scale"], h["x"], h["bias"], hy, dd["A"], dd["scale"], dd["x"], dd["bias"], dy,
                M, K, B)
    torch.cuda.synchronize()
    assert torch.equal(hy, y_dev.cpu()), "host-buffer call differs from the device call"
    U.assert_close(dtype, hy, y_ref, absdot, with_rounding=True, what=f"{dtype} host B={B}")
    # resident weights and scales: only x (and bias) are copied
    dy.zero_()
    hy2 = torch.zeros_like(hy).pin_memory()
    g.gemv_host(dtype, None, None, h["x"], h["bias"], hy2, dd["A"], dd["scale"], dd["x"], dd["bias"], dy, M, K, B)
    torch.cuda.synchronize()
    assert torch.equal(hy2, hy)


def test_host_argument_errors():
    M, K, B = 64, 256, 2
    hA = torch.zeros(M, K, dtype=torch.bfloat16).pin_memory()
    hx = torch.zeros(B, K, dtype=torch.bfloat16).pin_memory()
    hy = torch.zeros(B, M, dtype=torch.bfloat16).pin_memory()
    dA = torch.zeros(M, K, dtype=torch.bfloat16, device="cuda")
    dx = torch.zeros(B, K, dtype=torch.bfloat16, device="cuda")
    dy = torch.zeros(B, M, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(g.GemvError) as e:       # a host A but no device buffer for it
        g.gemv_host("bf16", hA, None, hx, None, hy, None, None, dx, None, dy, M, K, B)
    assert e.value.status == g.ERR_INVALID_VALUE
    with pytest.raises(g.GemvError) as e:       # no host y
        g.gemv_host("bf16", hA, None, hx, None, None, dA, None, dx, None, dy, M, K, B)
    assert e.value.status == g.ERR_INVALID_VALUE
    # 17 vectors of int8: beyond its limit (raw C call: sizes are the library's to check)
    st = g.lib().gemv_host(g.DTYPE_CODES["w8"], hA.data_ptr(), None, hx.data_ptr(), None, hy.data_ptr(),
                           dA.data_ptr(), None, dx.data_ptr(), None, dy.data_ptr(), M, K, 17, None)
    assert st == g.ERR_UNSUPPORTED
    with pytest.raises(ValueError):             # a device tensor where a host one belongs
        g.gemv_host("bf16", dA, None, hx, None, hy, dA, None, dx, None, dy, M, K, B)
