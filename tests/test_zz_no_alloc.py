"""gsi_forward_noalloc: one token of the gated map with no handle and no
allocation, for callers that cannot call cudaMalloc (code inside a framework
or server whose allocator owns all device memory, or fixed-memory
deployments).  Its scratch is a fixed array inside the library.

Checked through the C ABI against the handle-based gsi_forward on the same
inputs, within the parity tolerances (gates equal, rho within 1e-4, y within
2e-3 of max|y|), on two calls in a row.  This file is collected last so that a
run stopping at the first failure has already run every other test; it also
passes alone in a fresh process.
"""
import numpy as np
import pytest

import gsi_inputs as gi
from gsi_testlib import RHO2_TOL, RHO_TOL, Y_REL_TOL, GpuLinear, to_dev


NOALLOC_SHAPES = [(2304, 768, 256), (200, 512, 128), (4096, 16384, 256)]


@pytest.mark.gpu
@pytest.mark.parametrize("d_out,d,k", NOALLOC_SHAPES)
def test_noalloc_matches_oracle(gsi, orc, d_out, d, k):
    """The entry point on its own against the fp64 oracle (gates exact outside
    the 1e-4 band, rho within 1e-4, y within 2e-3 of max|y| per token), two
    calls in a row on each token."""
    import torch
    from gsi_testlib import check_against_oracle
    eps = 0.1
    spec = gi.LinearSpec("noalloc", d_out, d, k, eps, 0.05, 0.3)
    inp = gi.make_linear_inputs(spec, 4, 2, seed=91 + k)
    lin = GpuLinear(gsi, orc, inp.W, inp.V_bits, eps)
    x = to_dev(inp.X_bits)
    stream = torch.cuda.current_stream()
    for call in range(2):
        y = torch.full((4, d_out), float("nan"), dtype=torch.float32, device="cuda")
        g = torch.full((4,), 7, dtype=torch.uint8, device="cuda")
        r = torch.full((4,), -1.0, dtype=torch.float32, device="cuda")
        for t in range(4):
            gsi.gsi_forward_noalloc(lin.W_dev, lin.V_dev, lin.M_dev, eps, x[t:t + 1],
                                    y[t:t + 1], g[t:t + 1], r[t:t + 1], stream)
        stream.synchronize()
        rep = check_against_oracle(orc, lin, inp.X_bits, y.cpu().numpy(), g.cpu().numpy(),
                                   r.cpu().numpy(), what=f"noalloc call {call}")
        assert rep["n_slow"] == 2
    lin.close()


@pytest.mark.gpu
@pytest.mark.parametrize("d_out,d,k", NOALLOC_SHAPES)
def test_noalloc_matches_handle_path(gsi, orc, d_out, d, k):
    import torch
    eps = 0.1
    spec = gi.LinearSpec("noalloc", d_out, d, k, eps, 0.05, 0.3)
    inp = gi.make_linear_inputs(spec, 4, 2, seed=77 + k)
    lin = GpuLinear(gsi, orc, inp.W, inp.V_bits, eps)
    y_ref, g_ref, r_ref = lin.forward(inp.X_bits, one_by_one=True)
    x = to_dev(inp.X_bits)
    stream = torch.cuda.current_stream()
    for call in range(2):              # two calls in a row on each token
        for t in range(4):
            y = torch.full((1, d_out), float("nan"), dtype=torch.float32, device="cuda")
            g = torch.full((1,), 7, dtype=torch.uint8, device="cuda")
            r = torch.full((1,), -1.0, dtype=torch.float32, device="cuda")
            gsi.gsi_forward_noalloc(lin.W_dev, lin.V_dev, lin.M_dev, eps, x[t:t + 1], y, g, r,
                                    stream)
            stream.synchronize()
            yn = y.cpu().numpy()[0]
            assert int(g.item()) == int(g_ref[t]), (call, t)
            dr = abs(float(r.item()) - float(r_ref[t]))
            dr2 = abs(float(r.item()) ** 2 - float(r_ref[t]) ** 2)
            assert dr <= RHO_TOL or dr2 <= RHO2_TOL, (call, t)
            scale = np.abs(y_ref[t]).max()
            assert np.abs(yn - y_ref[t]).max() <= Y_REL_TOL * scale, (call, t)
    assert set(g_ref.tolist()) == {0, 1}      # both branches exercised
    lin.close()


def test_noalloc_rejects_bad_arguments():
    """Argument checks answer before any CUDA call (fake pointer values)."""
    import ctypes
    from gated_rank_subspace_gsi_gb300 import lib
    cl = lib.library()
    A, B, C = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x20000), ctypes.c_void_p(0x30000)
    X, Y = ctypes.c_void_p(0x40000), ctypes.c_void_p(0x50000)
    f = ctypes.c_float
    assert cl.gsi_forward_noalloc(None, B, C, 64, 64, 16, f(0.1), X, Y, None, None, None) == 1
    assert cl.gsi_forward_noalloc(A, B, C, 64, 64, 16, f(0.1), ctypes.c_void_p(0x40008), Y,
                                  None, None, None) == 1
    assert cl.gsi_forward_noalloc(A, B, C, 64, 64, 16, f(float("nan")), X, Y, None, None,
                                  None) == 1
    assert cl.gsi_forward_noalloc(A, B, C, 64, 60, 16, f(0.1), X, Y, None, None, None) == 2
    assert cl.gsi_forward_noalloc(A, B, C, 64, 2048, 1024, f(0.1), X, Y, None, None, None) == 2
    # a misaligned rho is refused on the host (the kernel stores it as fp32)
    assert cl.gsi_forward_noalloc(A, B, C, 64, 64, 16, f(0.1), X, Y, None,
                                  ctypes.c_void_p(0x60001), None) == 1
