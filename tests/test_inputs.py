"""The seeded input generator: determinism, structure, exact counts (CPU)."""
import math

import numpy as np

import gsi_inputs as gi


def test_bf16_rounding_matches_torch_on_fp32_values():
    """On values that are exact fp32 numbers, one RNE to bf16 must equal
    torch's fp32 -> bf16 conversion (a library routine)."""
    import torch
    rng = np.random.default_rng(0)
    v = (rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000))).astype(np.float32)
    ours = gi.to_bf16_bits(v.astype(np.float64))
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    assert np.array_equal(gi.bf16_bits_to_f64(ours),
                          torch.from_numpy(v).to(torch.bfloat16).double().numpy())


def test_deterministic():
    a = gi.make_linear_inputs(gi.LinearSpec("t", 32, 128, 16, 0.1, 0.05, 0.4), 9, 2, 1)
    b = gi.make_linear_inputs(gi.LinearSpec("t", 32, 128, 16, 0.1, 0.05, 0.4), 9, 2, 1)
    assert np.array_equal(a.W, b.W) and np.array_equal(a.V_bits, b.V_bits)
    assert np.array_equal(a.X_bits, b.X_bits) and np.array_equal(a.slow_mask, b.slow_mask)
    c = gi.make_linear_inputs(gi.LinearSpec("t", 32, 128, 16, 0.1, 0.05, 0.4), 9, 2, 2)
    assert not np.array_equal(a.X_bits, c.X_bits)


def test_basis_orthonormal_and_perp():
    b = gi.random_basis(512, 64, seed=4)
    assert np.abs(b.Q.T @ b.Q - np.eye(64)).max() < 1e-12
    assert np.abs(b.Q.T @ b.perp).max() < 1e-12
    V = gi.bf16_bits_to_f64(b.V_bits)
    E = V.T @ V - np.eye(64)
    assert np.linalg.norm(E, 2) < 1e-2


def test_target_rho_reached():
    """rho of the stored bf16 token against the stored bf16 basis is within
    5e-3 of the fp64 target (computed here with numpy least squares)."""
    b = gi.random_basis(768, 256, seed=5)
    rs = np.linspace(0.02, 0.4, 25)
    X = gi.bf16_bits_to_f64(gi.tokens(b, rs, seed=5))
    V = gi.bf16_bits_to_f64(b.V_bits)
    z, *_ = np.linalg.lstsq(V, X.T, rcond=None)
    rho = np.linalg.norm(X.T - V @ z, axis=0) / np.linalg.norm(X, axis=1)
    assert np.abs(rho - rs).max() < 5e-3


def test_exact_slow_counts():
    m = gi.slow_positions(512, 154, seed=1)
    assert m.sum() == 154
    wl = gi.batched_prefill()
    assert wl.extra["n_slow"] == 154
    assert gi.gptj_layer().extra["n_slow"] == 1
    assert gi.gptj_stack().extra["n_slow"] == 43
    assert gi.opt_mlp(slow_fraction=0.02).extra["n_slow"] == round(0.02 * 256 * 32 * 2)


def test_depth_coherence():
    """Adjacent-layer subspaces from V + 0.3 E: mean principal-angle cosine
    ~ 1/sqrt(1 + 0.09) ~ 0.96, above the 0.90 the page reports (section 2.3)."""
    b0 = gi.random_basis(1024, 64, seed=8)
    b1 = gi.coherent_next_basis(b0, seed=8, tag=1)
    cos = np.linalg.svd(b0.Q.T @ b1.Q, compute_uv=False)
    assert 0.93 < cos.mean() < 0.99
    assert cos.mean() > 0.90


def test_weights_scale():
    W = gi.bf16_bits_to_f64(gi.gaussian_weights(256, 1024, seed=3))
    assert abs(W.std() * math.sqrt(1024) - 1.0) < 0.01


def test_calibration_activations_planted_spectrum():
    """The calibration stand-in has its planted top-k directions as the
    dominant subspace of its second moment (checked through the oracle's
    eigensolver) and the step of gap^2 in the planted scales."""
    from oracle import calibration as cal
    s = gi.planted_scales(40, 16, decay=0.5, gap=0.5)
    assert np.all(np.diff(s) < 0)
    assert abs((s[16] / s[15]) ** 2 - 0.25 * (16 / 17)) < 1e-12
    cs = gi.calibration_activations(4000, 128, 16, seed=5)
    assert cs.X_bits.shape == (4000, 128) and cs.X_bits.dtype == np.uint16
    X = gi.bf16_bits_to_f64(cs.X_bits)
    V, lam = cal.top_k_subspace(X, 16)
    assert np.max(cal.principal_sines(V, cs.U[:, :16])) < 0.25
    assert lam[15] > 2.5 * cal.top_k_subspace(X, 17)[1][16]
    again = gi.calibration_activations(4000, 128, 16, seed=5)
    assert np.array_equal(again.X_bits, cs.X_bits)
    Q0 = gi.calibration_start(128, 16, seed=5)
    assert Q0.shape == (128, 16) and np.array_equal(Q0, gi.calibration_start(128, 16, seed=5))
