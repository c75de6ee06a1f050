"""GPU parity of the gated map against the fp64 oracle, through the C ABI.

Small and ragged shapes spanning several tiles, both paths (T = 1 decode and
T > 1 batched), the degenerate cases of the method (eps = 0, eps = inf,
x = 0, NaN, tokens at the threshold), workspace limits, host buffers and
CUDA-graph replay.  Tolerances: gates exact outside |rho - eps| <= 1e-4, y
within 2e-3 of max|y_ref| per token, rho within 1e-4.
"""
import math

import numpy as np
import pytest

import gsi_inputs as gi
from gsi_testlib import GpuLinear, check_against_oracle, to_bits, to_dev

pytestmark = pytest.mark.gpu

# (d_out, d, k): ragged d_out / d against 128-row MMA tiles, 64-wide K blocks,
# and the decode kernel's per-CTA slices; every supported k.
SHAPES = [(24, 64, 16), (40, 136, 32), (96, 264, 64), (200, 512, 128), (2304, 768, 256),
          (136, 1024, 512), (1000, 4104, 256)]
# One-token shapes besides: 10 row blocks of M per CTA (one warp each), 19
# row blocks staged as two TMA row boxes, and a d of 2 x 1024 with a ragged
# d_out (the slow path's steps run on across groups of 4 rows).
DECODE_SHAPES = SHAPES + [(22800, 1024, 256), (45600, 1024, 128), (1000, 2048, 64)]


def spread_rho(eps: float, T: int, seed: int) -> np.ndarray:
    """Residual targets on both sides of eps, none within bf16 reach of it."""
    rng = np.random.default_rng(seed)
    choices = np.array([0.0, 0.2, 0.5, 0.8, 1.25, 2.0, 4.0]) * eps
    r = rng.choice(choices, size=T)
    r = np.where(r == 0.0, 0.001, r)
    return np.minimum(r, 0.95)


def make_case(d_out, d, k, eps, T, seed):
    W = gi.gaussian_weights(d_out, d, seed)
    basis = gi.random_basis(d, k, seed, n_sub=min(200, k))
    X = gi.tokens(basis, spread_rho(eps, T, seed), seed)
    return W, basis, X


@pytest.mark.parametrize("d_out,d,k", SHAPES)
def test_precompute_M(gsi, orc, d_out, d, k):
    """M = bf16(W V_k) with fp32 accumulation: within one bf16 ulp of the exact
    product plus the worst-case error of a d-term fp32 sum, d 2^-24 sum|W||V|
    (entries that cancel to near zero may move several of their own ulps);
    and bit-identical to the oracle's bf16(W V_k) on >= 99% of entries."""
    W, basis, _ = make_case(d_out, d, k, 0.1, 1, 1)
    lin = GpuLinear(gsi, orc, W, basis.V_bits, 0.1)
    Wd, Vd = orc.bf16_decode(W), orc.bf16_decode(basis.V_bits)
    exact = orc.precompute_M(Wd, Vd)
    absum = orc.precompute_M(np.abs(Wd), np.abs(Vd))
    got_bits = to_bits(lin.M_dev)
    got = orc.bf16_decode(got_bits)
    ulp = np.ldexp(1.0, np.frexp(np.abs(exact))[1] - 8)
    bound = ulp + d * 2.0 ** -24 * absum
    assert (np.abs(got - exact) <= bound).all(), np.abs(got - exact).max()
    ref_bits = orc.bf16_encode(exact)
    assert (got_bits == ref_bits).mean() >= 0.99
    lin.close()


@pytest.mark.parametrize("d_out,d,k", DECODE_SHAPES)
def test_decode_T1(gsi, orc, d_out, d, k):
    eps = 0.10
    W, basis, X = make_case(d_out, d, k, eps, 14, 2)
    lin = GpuLinear(gsi, orc, W, basis.V_bits, eps)
    y, g, r = lin.forward(X, one_by_one=True)
    rep = check_against_oracle(orc, lin, X, y, g, r, what=f"decode {d_out}x{d}x{k}")
    assert 0 < rep["n_slow"] < 14
    lin.close()


@pytest.mark.parametrize("d_out,d,k", SHAPES)
@pytest.mark.parametrize("T", [2, 3, 17, 64, 300])
def test_batched(gsi, orc, d_out, d, k, T):
    eps = 0.10
    W, basis, X = make_case(d_out, d, k, eps, T, 3 + T)
    lin = GpuLinear(gsi, orc, W, basis.V_bits, eps)
    y, g, r = lin.forward(X)
    check_against_oracle(orc, lin, X, y, g, r, what=f"batched T={T} {d_out}x{d}x{k}")
    lin.close()


@pytest.mark.parametrize("rows", ["fewer", "more"])
def test_batched_all_slow_row_blocks(gsi, orc, rows):
    """Every token slow (eps = 0), so the GEMM kernel streams W alone.
    fewer: fewer 128-row blocks of W than the GEMM's CTAs (one per SM), so
    some CTAs take no slow tile; more: more row blocks than CTAs, so CTAs take
    several slow tiles from the queue one after another.  The output must
    repeat bit for bit."""
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    d, k, T = 2048, 128, 72
    d_out = 680 if rows == "fewer" else 128 * (sms + 8) + 40
    W, basis, X = make_case(d_out, d, k, 0.1, T, 41)
    lin = GpuLinear(gsi, orc, W, basis.V_bits, 0.0)
    y, g, r = lin.forward(X)
    assert (g == 1).all() and np.isfinite(y).all()
    sel = None if rows == "fewer" else np.r_[0:200, d_out - 300:d_out]
    check_against_oracle(orc, lin, X, y, g, r, rows=sel, what=f"all slow, {rows} row blocks")
    y2, _, _ = lin.forward(X)
    assert np.array_equal(y2.view(np.int32), y.view(np.int32))
    lin.close()


@pytest.mark.parametrize("k,T", [(64, 8192), (256, 8200)])
def test_batched_long_calls(gsi, orc, k, T):
    """Calls of 8192 and 8200 tokens (a reserved workspace): a gate grid of
    over a thousand CTAs, a partition over 8200 tokens and a GEMM tile queue
    of several token tiles per weight band; both projections (CUDA cores at
    k = 64, tensor cores at k = 256).  Every gate and rho is checked, y on
    sampled tokens."""
    d_out, d = 96, 512
    W, basis, X = make_case(d_out, d, k, 0.1, T, 51 + k)
    lin = GpuLinear(gsi, orc, W, basis.V_bits, 0.1, max_T=T)
    y, g, r = lin.forward(X)
    assert 0 < g.sum() < T and np.isfinite(y).all()
    rng = np.random.default_rng(7)
    sample = np.unique(np.r_[0:40, T - 40:T, rng.choice(T, 200, replace=False)])
    check_against_oracle(orc, lin, X, y, g, r, tokens=sample, what=f"long call k={k} T={T}")
    # every gate and rho, from the oracle's rho alone
    V = gi.bf16_bits_to_f64(basis.V_bits)
    rho_ref = orc.forward(None, V, None, lin.eps, gi.bf16_bits_to_f64(X))["rho"]
    out = np.abs(rho_ref - lin.eps) > 1e-4
    assert np.array_equal(g[out].astype(bool), rho_ref[out] >= lin.eps)
    lin.close()


@pytest.mark.parametrize("k", [128, 256])
def test_batched_fresh_handles_repeat(gsi, orc, k):
    """The batched kernels run with programmatic dependent launch: a kernel's
    CTAs start while the previous kernel runs, and every read of what that
    kernel writes must come after the dependent-launch wait.  Twelve fresh
    handles (first calls, when most SMs are free for the early CTAs), each
    call's gates against the oracle's.  A read moved above the wait showed as
    wrong gates in about three calls of four at k = 128."""
    d_out, d, T = 2048, 4096, 96
    W = gi.gaussian_weights(d_out, d, 302 + k)
    basis = gi.random_basis(d, k, 302 + k)
    X = gi.tokens(basis, np.where(np.arange(T) % 3 == 0, 0.3, 0.05), 302 + k)
    V = gi.bf16_bits_to_f64(basis.V_bits)
    rho_ref = orc.forward(None, V, None, 0.1, gi.bf16_bits_to_f64(X))["rho"]
    want = (rho_ref >= np.float32(0.1)).astype(np.uint8)
    lin = GpuLinear(gsi, orc, W, basis.V_bits, 0.1)
    for _ in range(12):
        gsi.gsi_destroy(lin.h)
        lin.h = gsi.gsi_create(lin.W_dev, lin.V_dev, lin.M_dev, 0.1)
        y, g, r = lin.forward(X)
        assert np.array_equal(g, want)
        assert np.abs(r.astype(np.float64) - rho_ref).max() <= 1e-4
    lin.close()


@pytest.mark.parametrize("T", [1, 40])
def test_eps_zero_and_inf(gsi, orc, T):
    """eps = 0: every token slow, y = W x.  eps = inf: every token fast."""
    d_out, d, k = 384, 1024, 128
    W, basis, X = make_case(d_out, d, k, 0.1, T, 9)
    for eps, want in ((0.0, 1), (math.inf, 0)):
        lin = GpuLinear(gsi, orc, W, basis.V_bits, eps)
        y, g, r = lin.forward(X, one_by_one=(T == 1))
        assert (g == want).all()
        check_against_oracle(orc, lin, X, y, g, r, what=f"eps={eps}")
        lin.close()


@pytest.mark.parametrize("path", ["decode", "batched"])
def test_special_tokens(gsi, orc, path):
    """x = 0 (rho = 0, fast, y = 0), NaN (slow, NaN out), Inf (slow), a pure
    residual token (rho ~ 1), an in-span token (rho ~ 0), and large / small
    token scales inside the supported range."""
    d_out, d, k = 256, 512, 64
    eps = 0.1
    W, basis, X = make_case(d_out, d, k, eps, 8, 11)
    Xf = gi.bf16_bits_to_f64(X)
    Xf[0] = 0.0
    Xf[1, 5] = np.nan
    Xf[2, 7] = np.inf
    Xf[3] = gi.bf16_bits_to_f64(gi.tokens(basis, np.array([1.0]), 12))[0]
    Xf[4] = gi.bf16_bits_to_f64(gi.tokens(basis, np.array([0.0]), 13))[0]
    Xf[5] *= 2.0 ** 40
    Xf[6] *= 2.0 ** -40
    Xb = gi.to_bf16_bits(np.where(np.isnan(Xf), 0, Xf))
    Xb[1, 5] = 0x7FC0
    Xb[2, 7] = 0x7F80
    lin = GpuLinear(gsi, orc, W, basis.V_bits, eps)
    y, g, r = lin.forward(Xb, one_by_one=(path == "decode"))
    assert g[0] == 0 and r[0] == 0 and (y[0] == 0).all()
    assert g[1] == 1 and np.isnan(r[1]) and np.isnan(y[1]).all()
    assert g[2] == 1 and np.isnan(r[2])
    assert g[3] == 1 and abs(r[3] - 1.0) < 1e-2
    assert g[4] == 0 and r[4] < 1e-2
    check_against_oracle(orc, lin, Xb[[0, 1, 3, 4, 5, 6, 7]], y[[0, 1, 3, 4, 5, 6, 7]],
                         g[[0, 1, 3, 4, 5, 6, 7]], r[[0, 1, 3, 4, 5, 6, 7]], what=path)
    lin.close()


@pytest.mark.parametrize("path", ["decode", "batched"])
def test_threshold_band(gsi, orc, path):
    """Tokens placed just either side of eps: outside the 1e-4 band the gate
    must match the oracle exactly; inside it, it must follow the GPU's rho."""
    d_out, d, k = 192, 1024, 128
    W, basis, X0 = make_case(d_out, d, k, 0.1, 1, 21)
    V = gi.bf16_bits_to_f64(basis.V_bits)
    rng = np.random.default_rng(5)
    toks = []
    for t in range(32):
        # tune eps instead of the token: pick a token, compute its oracle rho,
        # and set offsets relative to that rho
        toks.append(gi.tokens(basis, np.array([0.1 * (0.5 + rng.random())]), 100 + t)[0])
    Xb = np.stack(toks)
    rho_ref = orc.forward(None, V, None, 0.1, gi.bf16_bits_to_f64(Xb))["rho"]
    # one eps for all: the median rho, so tokens sit at many small offsets
    eps = float(np.float32(np.median(rho_ref) + 3e-5))
    lin = GpuLinear(gsi, orc, W, basis.V_bits, eps)
    y, g, r = lin.forward(Xb, one_by_one=(path == "decode"))
    rep = check_against_oracle(orc, lin, Xb, y, g, r, what=f"band {path}")
    assert 0 < rep["n_slow"] < 32
    lin.close()


@pytest.mark.parametrize("path", ["decode", "batched"])
@pytest.mark.parametrize("eps", [0.02, 0.05])
def test_threshold_band_small_eps(gsi, orc, path, eps):
    """Small thresholds (the sweep's eps = 0.02 and 0.05) at the GPT-J input
    shape d = 4096, k = 256: tokens whose oracle rho lies 1.5e-4 to 1e-3 on
    either side of eps.  No token is in the 1e-4 band, so every gate must
    equal the oracle's, and rho itself must be within 1e-4 (near a small eps
    an error of 5e-6 in rho^2 alone would be 1.25e-4 in rho)."""
    d_out, d, k = 256, 4096, 256
    seed = 23 + int(eps * 1000)
    W = gi.gaussian_weights(d_out, d, seed)
    basis = gi.random_basis(d, k, seed, n_sub=200)
    V = gi.bf16_bits_to_f64(basis.V_bits)
    rng = np.random.default_rng(seed)
    targets = eps + rng.uniform(-1.2e-3, 1.2e-3, size=160)
    Xc = gi.tokens(basis, targets, seed)
    rho_c = orc.forward(None, V, None, eps, gi.bf16_bits_to_f64(Xc))["rho"]
    off = rho_c - np.float64(np.float32(eps))
    keep = np.nonzero((np.abs(off) >= 1.5e-4) & (np.abs(off) <= 1e-3))[0][:48]
    assert (off[keep] < 0).sum() >= 8 and (off[keep] > 0).sum() >= 8
    Xb = Xc[keep]
    lin = GpuLinear(gsi, orc, W, basis.V_bits, eps)
    y, g, r = lin.forward(Xb, one_by_one=(path == "decode"))
    rep = check_against_oracle(orc, lin, Xb, y, g, r, what=f"eps={eps} {path}")
    assert rep["n_band"] == 0
    assert np.array_equal(g.astype(bool), off[keep] >= 0)
    assert np.abs(r.astype(np.float64) - rho_c[keep]).max() <= 1e-4
    lin.close()


def test_T0_workspace_and_reserve(gsi, orc):
    import torch
    d_out, d, k = 128, 256, 32
    W, basis, X = make_case(d_out, d, k, 0.1, 600, 31)
    lin = GpuLinear(gsi, orc, W, basis.V_bits, 0.1)
    x = to_dev(X)
    y = torch.zeros((600, d_out), dtype=torch.float32, device="cuda")
    gsi.gsi_forward(lin.h, x[:0], y, T=0)                    # no-op
    with pytest.raises(gsi.GsiError) as ei:
        gsi.gsi_forward(lin.h, x, y)                          # 600 > default 512
    assert ei.value.status == gsi.GSI_ERR_WORKSPACE
    gsi.gsi_reserve(lin.h, 600)
    y2, g2, r2 = lin.forward(X)
    check_against_oracle(orc, lin, X, y2, g2, r2, what="after reserve")
    assert gsi.gsi_forward_launch_count(lin.h, 1) == 1
    assert gsi.gsi_forward_launch_count(lin.h, 600) >= 2
    # a misaligned rho is refused on the host, before any launch (fp32 stores)
    rb = torch.zeros(2 * 600 + 4, dtype=torch.float32, device="cuda")
    rho_bad = rb.view(torch.uint8)[1:1 + 4 * 600]
    for T in (1, 600):
        with pytest.raises(gsi.GsiError) as ei:
            gsi.gsi_forward(lin.h, x[:T], y[:T], rho=rho_bad, T=T)
        assert ei.value.status == gsi.GSI_ERR_INVALID_ARG
    assert gsi.gsi_device_status(lin.h) == gsi.GSI_OK
    lin.close()


@pytest.mark.parametrize("T", [1, 33])
def test_forward_host(gsi, orc, T):
    """The host-buffer entry point gives the device path's results: in place on
    page-locked memory for one token, through staging copies otherwise."""
    import torch
    d_out, d, k = 512, 1024, 128
    W, basis, X = make_case(d_out, d, k, 0.1, T, 41)
    lin = GpuLinear(gsi, orc, W, basis.V_bits, 0.1)
    xh = torch.from_numpy(X.view(np.int16)).view(torch.bfloat16).pin_memory()
    yh = torch.empty((T, d_out), dtype=torch.float32).pin_memory()
    gh = torch.empty((T,), dtype=torch.uint8).pin_memory()
    rh = torch.empty((T,), dtype=torch.float32).pin_memory()
    s = torch.cuda.current_stream()
    gsi.gsi_forward_host(lin.h, xh, yh, gh, rh, s)
    s.synchronize()
    check_against_oracle(orc, lin, X, yh.numpy(), gh.numpy(), rh.numpy(), what="host")
    # y, rho and gate consecutive in one pinned allocation: one copy returns them
    nb = T * d_out * 4
    buf = torch.full((nb + T * 5,), 0xEE, dtype=torch.uint8).pin_memory()
    yp = buf[:nb].view(torch.float32).view(T, d_out)
    rp = buf[nb:nb + 4 * T].view(torch.float32)
    gp = buf[nb + 4 * T:]
    gsi.gsi_forward_host(lin.h, xh, yp, gp, rp, s)
    s.synchronize()
    assert np.array_equal(yp.numpy(), yh.numpy()) and np.array_equal(gp.numpy(), gh.numpy())
    assert np.array_equal(rp.numpy().view(np.int32), rh.numpy().view(np.int32))
    # pageable host memory: the staging copies (the device cannot address it)
    xq = torch.from_numpy(X.view(np.int16).copy()).view(torch.bfloat16)
    yq = torch.empty((T, d_out), dtype=torch.float32)
    gq = torch.empty((T,), dtype=torch.uint8)
    rq = torch.empty((T,), dtype=torch.float32)
    gsi.gsi_forward_host(lin.h, xq, yq, gq, rq, s)
    s.synchronize()
    assert np.array_equal(yq.numpy(), yh.numpy()) and np.array_equal(gq.numpy(), gh.numpy())
    assert np.array_equal(rq.numpy().view(np.int32), rh.numpy().view(np.int32))
    # and the device path itself, bit for bit
    y, g, r = lin.forward(X, one_by_one=(T == 1))
    assert np.array_equal(y, yh.numpy()) and np.array_equal(g, gh.numpy())
    lin.close()


def test_graph_replay_decode(gsi, orc):
    """A CUDA graph of many T = 1 calls over two handles replays correctly
    (exercises the device-side launch epoch and grid barrier counters)."""
    import torch
    d_out, d, k = 1024, 2048, 256
    eps = 0.1
    W, basis, X = make_case(d_out, d, k, eps, 24, 51)
    lin = GpuLinear(gsi, orc, W, basis.V_bits, eps)
    W2, basis2, X2 = make_case(512, 1024, 128, eps, 24, 52)
    lin2 = GpuLinear(gsi, orc, W2, basis2.V_bits, eps)
    x = to_dev(X)
    x2 = to_dev(X2)
    y = torch.zeros((24, d_out), dtype=torch.float32, device="cuda")
    y2 = torch.zeros((24, 512), dtype=torch.float32, device="cuda")
    g = torch.zeros((24,), dtype=torch.uint8, device="cuda")
    r = torch.zeros((24,), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        gsi.gsi_forward(lin.h, x[:1], y[:1], g[:1], r[:1], s)   # warm-up outside capture
        s.synchronize()
        with torch.cuda.graph(graph, stream=s):
            for t in range(24):
                gsi.gsi_forward(lin.h, x[t:t + 1], y[t:t + 1], g[t:t + 1], r[t:t + 1], s)
                gsi.gsi_forward(lin2.h, x2[t:t + 1], y2[t:t + 1], None, None, s)
    for rep in range(3):
        y.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert gsi.gsi_device_status(lin.h) == 0 and gsi.gsi_device_status(lin2.h) == 0
        check_against_oracle(orc, lin, X, y.cpu().numpy(), g.cpu().numpy(), r.cpu().numpy(),
                             what=f"graph replay {rep}")
    yy, gg, rr = lin2.forward(X2, one_by_one=True)
    assert np.abs(yy - y2.cpu().numpy()).max() <= 2e-3 * np.abs(yy).max()
    lin.close()
    lin2.close()


def test_handles_of_one_k_with_different_sizes(gsi, orc):
    """Handles of one k but different shapes coexist: creating a small handle
    after a large one must not break the large one's launches."""
    eps = 0.1
    W1, b1, X1 = make_case(4096, 1024, 256, eps, 4, 61)
    big = GpuLinear(gsi, orc, W1, b1.V_bits, eps)
    W2, b2, X2 = make_case(64, 256, 256, eps, 4, 62)
    small = GpuLinear(gsi, orc, W2, b2.V_bits, eps)
    y, g, r = big.forward(X1, one_by_one=True)
    check_against_oracle(orc, big, X1, y, g, r, what="large after small")
    y, g, r = small.forward(X2, one_by_one=True)
    check_against_oracle(orc, small, X2, y, g, r, what="small")
    big.close()
    small.close()


def test_prefetch_links(gsi, orc):
    """gsi_set_prefetch schedules L2 traffic only: linked handles (a chain, a
    self link, a link into a k = 512 handle, inside a CUDA graph) keep
    parity, and destroying a link target leaves its source working."""
    import torch
    eps = 0.1
    cases = [make_case(2304, 768, 256, eps, 6, 71), make_case(512, 1024, 128, eps, 6, 72),
             make_case(136, 1024, 512, eps, 6, 73)]
    lins = [GpuLinear(gsi, orc, W, b.V_bits, eps) for (W, b, X) in cases]
    gsi.gsi_set_prefetch(lins[0].h, lins[1].h)
    gsi.gsi_set_prefetch(lins[1].h, lins[2].h)
    gsi.gsi_set_prefetch(lins[2].h, lins[0].h)
    for lin, (W, b, X) in zip(lins, cases):
        y, g, r = lin.forward(X, one_by_one=True)
        check_against_oracle(orc, lin, X, y, g, r, what="linked")
    # the chain inside a graph, interleaved call by call
    xs = [to_dev(X) for (_, _, X) in cases]
    ys = [torch.zeros((6, lin.d_out), dtype=torch.float32, device="cuda") for lin in lins]
    gs = [torch.zeros((6,), dtype=torch.uint8, device="cuda") for _ in lins]
    rs = [torch.zeros((6,), dtype=torch.float32, device="cuda") for _ in lins]
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            for t in range(6):
                for i, lin in enumerate(lins):
                    gsi.gsi_forward(lin.h, xs[i][t:t + 1], ys[i][t:t + 1], gs[i][t:t + 1],
                                    rs[i][t:t + 1], s)
    for rep in range(2):
        graph.replay()
        torch.cuda.synchronize()
        for i, (lin, (W, b, X)) in enumerate(zip(lins, cases)):
            assert gsi.gsi_device_status(lin.h) == 0
            check_against_oracle(orc, lin, X, ys[i].cpu().numpy(), gs[i].cpu().numpy(),
                                 rs[i].cpu().numpy(), what=f"linked graph {rep}")
    del graph
    # a self link, then removing a link target
    gsi.gsi_set_prefetch(lins[0].h, lins[0].h)
    W, b, X = cases[0]
    y, g, r = lins[0].forward(X, one_by_one=True)
    check_against_oracle(orc, lins[0], X, y, g, r, what="self link")
    gsi.gsi_set_prefetch(lins[0].h, lins[1].h)
    lins[1].close()
    y, g, r = lins[0].forward(X, one_by_one=True)
    check_against_oracle(orc, lins[0], X, y, g, r, what="target destroyed")
    gsi.gsi_set_prefetch(lins[2].h, None)
    lins[0].close()
    lins[2].close()
