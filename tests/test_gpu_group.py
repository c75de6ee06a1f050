"""gsi_group_*: several independent one-token calls in one launch, through
the C ABI, against the fp64 oracle (same tolerances as the other parity
tests: gates exact outside |rho - eps| <= 1e-4, y within 2e-3 of max|y_ref|
per token, rho within 1e-4).

Covers groups of 2 and 3 members with different shapes, a handle used both
alone and inside groups (each launch of a handle may run on a different
number of CTAs), groups inside a CUDA graph with prefetch links into and out
of the group, and the creation errors.
"""
import ctypes

import numpy as np
import pytest

import gsi_inputs as gi
from gsi_testlib import GpuLinear, check_against_oracle, to_dev

pytestmark = pytest.mark.gpu


def _case(d_out, d, k, T, seed, eps=0.1):
    W = gi.gaussian_weights(d_out, d, seed)
    basis = gi.random_basis(d, k, seed, n_sub=min(200, k))
    rng = np.random.default_rng(seed)
    rho = rng.choice(np.array([0.02, 0.05, 0.3, 0.5]) * 1.0, size=T)
    X = gi.tokens(basis, rho, seed)
    return W, basis, X


def _bufs(lin, T):
    import torch
    return (torch.full((T, lin.d_out), float("nan"), dtype=torch.float32, device="cuda"),
            torch.full((T,), 7, dtype=torch.uint8, device="cuda"),
            torch.full((T,), -1.0, dtype=torch.float32, device="cuda"))


def _run_group(gsi, g, lins, xs, T, stream=None):
    outs = [_bufs(lin, T) for lin in lins]
    for t in range(T):
        gsi.gsi_group_forward(g, [x[t:t + 1] for x in xs], [o[0][t:t + 1] for o in outs],
                              [o[1][t:t + 1] for o in outs], [o[2][t:t + 1] for o in outs],
                              stream)
    return outs


def _check(gsi, orc, lins, Xs, outs, what):
    for i, (lin, X, (y, g, r)) in enumerate(zip(lins, Xs, outs)):
        assert gsi.gsi_device_status(lin.h) == 0
        check_against_oracle(orc, lin, X, y.cpu().numpy(), g.cpu().numpy(), r.cpu().numpy(),
                             what=f"{what} member {i}")


@pytest.mark.parametrize("shapes", [
    [(4096, 4096, 256), (4096, 16384, 256)],                       # GPT-J out_proj | fc_out
    [(2304, 768, 256), (1000, 4104, 256), (520, 1032, 256)],       # ragged, three members
    [(512, 1024, 128), (4096, 2048, 128)],
    [(96, 264, 64), (200, 512, 64)],
])
def test_group_matches_oracle(gsi, orc, shapes):
    T = 8
    cases = [_case(*sh, T, 90 + i) for i, sh in enumerate(shapes)]
    lins = [GpuLinear(gsi, orc, W, b.V_bits, 0.1) for (W, b, X) in cases]
    g = gsi.gsi_group_create([lin.h for lin in lins])
    xs = [to_dev(X) for (_, _, X) in cases]
    outs = _run_group(gsi, g, lins, xs, T)
    _check(gsi, orc, lins, [X for (_, _, X) in cases], outs, f"group {shapes}")
    gsi.gsi_group_destroy(g)
    for lin in lins:
        lin.close()


def test_handle_alone_and_in_groups(gsi, orc):
    """One handle alternates between calls on all SMs and calls inside two
    different groups (different CTA counts per launch)."""
    import torch
    T = 6
    cases = [_case(4096, 4096, 256, T, 101), _case(4096, 16384, 256, T, 102),
             _case(2304, 768, 256, T, 103)]
    lins = [GpuLinear(gsi, orc, W, b.V_bits, 0.1) for (W, b, X) in cases]
    g1 = gsi.gsi_group_create([lins[0].h, lins[1].h])
    g2 = gsi.gsi_group_create([lins[2].h, lins[0].h])
    xs = [to_dev(X) for (_, _, X) in cases]
    outs = [_bufs(lin, T) for lin in lins]
    for t in range(T):
        sl = slice(t, t + 1)
        if t % 3 == 0:
            gsi.gsi_forward(lins[0].h, xs[0][sl], outs[0][0][sl], outs[0][1][sl], outs[0][2][sl])
            gsi.gsi_group_forward(g2, [xs[2][sl], xs[0][sl]], [outs[2][0][sl], outs[0][0][sl]],
                                  [outs[2][1][sl], outs[0][1][sl]], [outs[2][2][sl], outs[0][2][sl]])
            gsi.gsi_forward(lins[1].h, xs[1][sl], outs[1][0][sl], outs[1][1][sl], outs[1][2][sl])
        elif t % 3 == 1:
            gsi.gsi_group_forward(g1, [xs[0][sl], xs[1][sl]], [outs[0][0][sl], outs[1][0][sl]],
                                  [outs[0][1][sl], outs[1][1][sl]], [outs[0][2][sl], outs[1][2][sl]])
            gsi.gsi_forward(lins[2].h, xs[2][sl], outs[2][0][sl], outs[2][1][sl], outs[2][2][sl])
        else:
            gsi.gsi_group_forward(g2, [xs[2][sl], xs[0][sl]], [outs[2][0][sl], outs[0][0][sl]],
                                  [outs[2][1][sl], outs[0][1][sl]], [outs[2][2][sl], outs[0][2][sl]])
            gsi.gsi_group_forward(g1, [xs[0][sl], xs[1][sl]], [outs[0][0][sl], outs[1][0][sl]],
                                  [outs[0][1][sl], outs[1][1][sl]], [outs[0][2][sl], outs[1][2][sl]])
    torch.cuda.synchronize()
    _check(gsi, orc, lins, [X for (_, _, X) in cases], outs, "alone and grouped")
    gsi.gsi_group_destroy(g1)
    gsi.gsi_group_destroy(g2)
    for lin in lins:
        lin.close()


def test_group_in_graph_with_prefetch(gsi, orc):
    """The decode-layer schedule: a call on A, then one launch of (B, C), in a
    CUDA graph; A prefetches the group's operands, the group prefetches A.
    Destroying the group and a handle afterwards removes the links."""
    import torch
    T = 8
    cases = [_case(2304, 768, 256, T, 111), _case(768, 768, 256, T, 112),
             _case(768, 3072, 256, T, 113)]
    lins = [GpuLinear(gsi, orc, W, b.V_bits, 0.1) for (W, b, X) in cases]
    grp = gsi.gsi_group_create([lins[1].h, lins[2].h])
    gsi.gsi_set_prefetch_group(lins[0].h, grp)
    gsi.gsi_group_set_prefetch(grp, lins[0].h)
    xs = [to_dev(X) for (_, _, X) in cases]
    outs = [_bufs(lin, T) for lin in lins]
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            for t in range(T):
                sl = slice(t, t + 1)
                gsi.gsi_forward(lins[0].h, xs[0][sl], outs[0][0][sl], outs[0][1][sl],
                                outs[0][2][sl], s)
                gsi.gsi_group_forward(grp, [xs[1][sl], xs[2][sl]], [outs[1][0][sl], outs[2][0][sl]],
                                      [outs[1][1][sl], outs[2][1][sl]],
                                      [outs[1][2][sl], outs[2][2][sl]], s)
    for rep in range(3):
        for o in outs:
            o[0].fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        _check(gsi, orc, lins, [X for (_, _, X) in cases], outs, f"graph replay {rep}")
    del graph
    gsi.gsi_group_destroy(grp)          # A's link to the group goes with it
    y, g, r = lins[0].forward(cases[0][2], one_by_one=True)
    check_against_oracle(orc, lins[0], cases[0][2], y, g, r, what="after group destroyed")
    for lin in lins:
        lin.close()


def test_group_creation_errors(gsi, orc):
    T = 1
    def lin(d_out, d, k, seed):
        W, basis, _ = _case(d_out, d, k, T, seed)
        return GpuLinear(gsi, orc, W, basis.V_bits, 0.1)
    a, b, c = lin(256, 512, 256, 121), lin(256, 512, 128, 122), lin(136, 1024, 512, 123)
    cl = gsi.library()
    out = ctypes.c_void_p()
    arr = lambda *hs: (ctypes.c_void_p * len(hs))(*[h.value for h in hs])  # noqa: E731
    assert cl.gsi_group_create(2, arr(a.h, a.h), ctypes.byref(out)) == 1      # duplicate
    assert cl.gsi_group_create(2, arr(a.h, b.h), ctypes.byref(out)) == 2      # k differs
    assert cl.gsi_group_create(1, arr(c.h), ctypes.byref(out)) == 2           # k = 512
    assert cl.gsi_group_create(1, arr(a.h), ctypes.byref(out)) == 0
    cl.gsi_group_destroy(out)
    for lin in (a, b, c):
        lin.close()


@pytest.mark.parametrize("pinned", [True, False])
def test_group_forward_host_matches_device(gsi, orc, pinned):
    """gsi_group_forward_host on page-locked buffers (one staging launch, the
    outputs written in place over the host link) and on pageable buffers
    (copies through the handles' staging) gives the device call's bits."""
    import torch
    shapes = [(4096, 4096, 256), (4096, 16384, 256)]
    T = 6
    cases = [_case(do, d, k, T, seed=911 + i) for i, (do, d, k) in enumerate(shapes)]
    lins = [GpuLinear(gsi, orc, W, b.V_bits, 0.1) for (W, b, _) in cases]
    try:
        g = gsi.gsi_group_create([lin.h for lin in lins])
        try:
            xs = [to_dev(X) for (_, _, X) in cases]
            dev = _run_group(gsi, g, lins, xs, T)
            mk = (lambda t: t.pin_memory()) if pinned else (lambda t: t)
            hx = [mk(x.cpu()) for x in xs]
            hy = [mk(torch.full((T, lin.d_out), float("nan"), dtype=torch.float32)) for lin in lins]
            hg = [mk(torch.full((T,), 7, dtype=torch.uint8)) for _ in lins]
            hr = [mk(torch.full((T,), -1.0, dtype=torch.float32)) for _ in lins]
            for t in range(T):
                gsi.gsi_group_forward_host(g, [x[t:t + 1] for x in hx], [y[t] for y in hy],
                                           [q[t:t + 1] for q in hg], [r[t:t + 1] for r in hr])
            torch.cuda.synchronize()
            for i in range(len(lins)):
                assert torch.equal(hy[i], dev[i][0].cpu()), i
                assert torch.equal(hg[i], dev[i][1].cpu()), i
                assert torch.equal(hr[i].view(torch.int32), dev[i][2].cpu().view(torch.int32)), i
            _check(gsi, orc, lins, [X for (_, _, X) in cases], dev, "host group")
        finally:
            gsi.gsi_group_destroy(g)
    finally:
        for lin in lins:
            lin.close()
