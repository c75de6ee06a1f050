"""The fp64 oracle against what the page and mathematics fix (CPU only)."""
import numpy as np
import pytest

import gsi_inputs as gi
import oracle_pins as pins


@pytest.mark.parametrize("name", pins.ALL_PINS)
def test_pin(orc, name):
    getattr(pins, name)(orc)


@pytest.mark.parametrize("d,d_out,T", [(768, 96, 64), (256, 64, 33)])
def test_decomposition_and_theorem4_on_generated(orc, d, d_out, T):
    """Identity (a) and Theorem 4 (d) on bf16 inputs of the GPT-2 QKV mix."""
    spec = gi.LinearSpec("t", d_out, d, 64 if d < 768 else 256, 0.10, 0.03, 0.3)
    inp = gi.make_linear_inputs(spec, T, n_slow=T // 10, seed=99, tag=d)
    info = pins.pin_decomposition_and_theorem4(orc, inp)
    assert info["w_norm"] > 0


def test_gpt2_qkv_gates_follow_generated_mix(orc):
    """On the GPT-2-shaped QKV workload the oracle's gates equal the intended
    slow/fast mix (rho* is >= 0.02 away from eps, far outside rounding)."""
    wl = gi.gpt2_qkv()
    spec = wl.linears[0]
    inp = gi.make_linear_inputs(spec, wl.T, wl.extra["n_slow"], wl.seed)
    V = orc.bf16_decode(inp.V_bits)
    X = orc.bf16_decode(inp.X_bits)
    out = orc.forward(None, V, None, float(np.float32(spec.eps)), X)
    assert np.array_equal(out["gate"].astype(bool), inp.slow_mask)
    assert int(out["gate"].sum()) == 6
