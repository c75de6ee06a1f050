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
