"""The five workload configurations at full size against the oracle (GPU).

GPT-2 QKV (T = 64), GPT-J decode layer (512 sequential T = 1 tokens through
three linears), batched T = 512, GPT-J 28-layer stack (depth-coherent
bases) and OPT MLP x 32 with a slow-fraction sweep.  Where the oracle cannot
recompute every output in seconds, every gate and rho is still checked and y
is checked on sampled rows and steps.
"""
import numpy as np
import pytest

import gsi_inputs as gi
from gsi_testlib import GpuLinear, check_against_oracle, to_dev

pytestmark = pytest.mark.gpu


def test_gpt2_qkv_T64(gsi, orc):
    wl = gi.gpt2_qkv()
    spec = wl.linears[0]
    inp = gi.make_linear_inputs(spec, wl.T, wl.extra["n_slow"], wl.seed)
    lin = GpuLinear(gsi, orc, inp.W, inp.V_bits, spec.eps)
    y, g, r = lin.forward(inp.X_bits)
    rep = check_against_oracle(orc, lin, inp.X_bits, y, g, r, what="gpt2 T=64 batched")
    assert rep["n_slow"] == 6 and np.array_equal(g.astype(bool), inp.slow_mask)
    y1, g1, r1 = lin.forward(inp.X_bits, one_by_one=True)
    check_against_oracle(orc, lin, inp.X_bits, y1, g1, r1, what="gpt2 T=1 each")
    lin.close()


def test_batched_T512(gsi, orc):
    wl = gi.batched_prefill()
    spec = wl.linears[0]
    inp = gi.make_linear_inputs(spec, wl.T, wl.extra["n_slow"], wl.seed)
    lin = GpuLinear(gsi, orc, inp.W, inp.V_bits, spec.eps)
    y, g, r = lin.forward(inp.X_bits)
    rep = check_against_oracle(orc, lin, inp.X_bits, y, g, r, what="batched T=512")
    assert rep["n_slow"] == 154
    lin.close()


def test_gptj_layer_decode(gsi, orc):
    """512 sequential T = 1 tokens through the stacked q/k/v/fc_in linear,
    out_proj and fc_out; exactly one slow token in all three."""
    import torch
    wl = gi.gptj_layer()
    n = wl.extra["n_tokens"]
    slow = gi.slow_positions(n, wl.extra["n_slow"], wl.seed)
    rng = np.random.default_rng(wl.seed)
    check_tok = np.unique(np.concatenate([np.nonzero(slow)[0], rng.choice(n, 24, replace=False)]))
    for li, spec in enumerate(wl.linears):
        inp = gi.make_linear_inputs(spec, n, 0, wl.seed, tag=li, slow_mask=slow)
        lin = GpuLinear(gsi, orc, inp.W, inp.V_bits, spec.eps)
        x = to_dev(inp.X_bits)
        y = torch.full((n, spec.d_out), float("nan"), device="cuda")
        gt = torch.zeros((n,), dtype=torch.uint8, device="cuda")
        rt = torch.zeros((n,), dtype=torch.float32, device="cuda")
        for t in range(n):
            gsi.gsi_forward(lin.h, x[t:t + 1], y[t:t + 1], gt[t:t + 1], rt[t:t + 1])
        assert gsi.gsi_device_status(lin.h) == 0
        yn, gn, rn = y.cpu().numpy(), gt.cpu().numpy(), rt.cpu().numpy()
        assert np.array_equal(gn.astype(bool), slow), spec.name
        # all gates and rho; y on a sample of tokens including the slow one
        check_against_oracle(orc, lin, inp.X_bits, yn, gn, rn, rows=np.arange(0), what=spec.name)
        check_against_oracle(orc, lin, inp.X_bits, yn, gn, rn, tokens=check_tok, what=spec.name)
        lin.close()


def _sampled_rows(d_out: int, n: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return np.sort(rng.choice(d_out, size=min(n, d_out), replace=False))


def _run_stack(gsi, orc, specs, n_layers, n_steps, slow, seed, bases, what, y_pairs):
    """Create one handle per (layer, linear), run n_steps sequential T = 1
    steps through every linear in layer order, then check every gate and rho
    against the oracle and y on sampled rows for the (layer, linear) pairs in
    y_pairs (all their slow tokens plus two fast ones)."""
    import torch
    n_lin = len(specs)
    runs = []
    for l in range(n_layers):
        for i, sp in enumerate(specs):
            tag = 100 * l + i
            W = gi.gaussian_weights(sp.d_out, sp.d, seed, tag, device="cuda")
            lin = GpuLinear(gsi, orc, None, bases[l][i].V_bits, sp.eps, W_dev=W)
            rs = gi.rho_targets(n_steps, sp.rho_fast, sp.rho_slow, slow[:, l, i], seed, tag)
            X = gi.tokens(bases[l][i], rs, seed, tag)
            runs.append(dict(lin=lin, X=X, x=to_dev(X),
                             y=torch.full((n_steps, sp.d_out), float("nan"), device="cuda"),
                             g=torch.full((n_steps,), 7, dtype=torch.uint8, device="cuda"),
                             r=torch.zeros((n_steps,), dtype=torch.float32, device="cuda")))
    for s in range(n_steps):
        for R in runs:
            gsi.gsi_forward(R["lin"].h, R["x"][s:s + 1], R["y"][s:s + 1], R["g"][s:s + 1],
                            R["r"][s:s + 1])
    torch.cuda.synchronize()
    rng = np.random.default_rng(seed + 1)
    for j, R in enumerate(runs):
        l, i = divmod(j, n_lin)
        lin = R["lin"]
        assert gsi.gsi_device_status(lin.h) == 0
        gn, rn = R["g"].cpu().numpy(), R["r"].cpu().numpy()
        assert np.array_equal(gn.astype(bool), slow[:, l, i]), f"{what} layer {l} linear {i}"
        yn = R["y"].cpu().numpy()
        check_against_oracle(orc, lin, R["X"], yn, gn, rn, rows=np.arange(0),
                             what=f"{what} l{l} i{i} gates")
        if (l, i) in y_pairs:
            fast = np.nonzero(~slow[:, l, i])[0]
            toks = np.unique(np.concatenate([np.nonzero(slow[:, l, i])[0],
                                             rng.choice(fast, size=min(2, fast.size),
                                                        replace=False)]))
            rows = _sampled_rows(lin.d_out, 384, seed + j)
            check_against_oracle(orc, lin, R["X"], yn, gn, rn, rows=rows, tokens=toks,
                                 what=f"{what} l{l} i{i} y")
    for R in runs:
        R["lin"].close()
    del runs
    torch.cuda.empty_cache()


def test_gptj_stack_decode(gsi, orc):
    """28 GPT-J layers (q/k/v/fc_in stacked, out_proj, fc_out) with
    depth-coherent bases per input chain, 256 sequential decode steps through
    every linear in order, 43 slow draws (0.2%) over (step, layer, linear):
    every gate and rho against the oracle, y on sampled rows of every linear
    that drew a slow token and of a few others."""
    wl = gi.gptj_stack()
    L, S, specs = wl.extra["n_layers"], wl.extra["n_steps"], wl.linears
    slow = gi.slow_positions(S * L * len(specs), wl.extra["n_slow"], wl.seed).reshape(
        S, L, len(specs))
    assert slow.sum() == 43
    bases = [[None] * len(specs) for _ in range(L)]
    for i, sp in enumerate(specs):
        b = gi.random_basis(sp.d, sp.k, wl.seed, tag=i)
        for l in range(L):
            if l > 0:
                b = gi.coherent_next_basis(b, wl.seed, tag=1000 * i + l)
            bases[l][i] = b
    pairs = {(l, i) for l in range(L) for i in range(len(specs)) if slow[:, l, i].any()}
    pairs |= {(0, 0), (13, 1), (27, 2)}
    _run_stack(gsi, orc, specs, L, S, slow, wl.seed, bases, "gptj stack", pairs)


_OPT_BASES = {}


@pytest.mark.parametrize("f", [0.0, 0.02, 0.10, 0.50, 1.00])
def test_opt_mlp_slow_fraction(gsi, orc, f):
    """OPT-6.7B MLP (fc1 4096 -> 16384, fc2 16384 -> 4096) x 32 layers,
    eps = 0.05, 16 sequential decode steps per point of the slow-fraction
    sweep, exact slow counts over (step, layer, linear)."""
    S = 16
    wl = gi.opt_mlp(n_steps=S, slow_fraction=f)
    L, specs = wl.extra["n_layers"], wl.linears
    slow = gi.slow_positions(S * L * len(specs), wl.extra["n_slow"], wl.seed).reshape(
        S, L, len(specs))
    assert slow.sum() == round(f * S * L * len(specs))
    key = (wl.seed, L)
    if key not in _OPT_BASES:  # the same bases serve every point of the sweep
        _OPT_BASES.clear()
        _OPT_BASES[key] = [[gi.random_basis(sp.d, sp.k, wl.seed, tag=100 * l + i)
                            for i, sp in enumerate(specs)] for l in range(L)]
    bases = _OPT_BASES[key]
    pairs = {(0, 0), (0, 1), (L - 1, 0), (L - 1, 1), (L // 2, 1)}
    _run_stack(gsi, orc, specs, L, S, slow, wl.seed, bases, f"opt mlp f={f}", pairs)
