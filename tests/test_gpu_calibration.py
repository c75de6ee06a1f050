"""gsi_calibrate (block power iteration for V_k, tcgen05 GEMMs + CholeskyQR2)
against the fp64 oracle, through the C ABI.

Tolerances, from the arithmetic:
* SIN_TOL: the largest principal-angle sine between span(V_k) from the GPU
  and the oracle's subspace_iteration(X, Q0, iters) on the same bf16 X and
  Q0.  The GPU rounds Q and X Q to bf16 in every iteration and V_k at the
  end; each rounding moves a span by about 2^-9 relative, and the iteration
  damps earlier roundings by the eigenvalue gap ratio lambda_{k+1}/lambda_k
  per step.  With the planted gap of these inputs (ratio <= 0.4) that is a
  few times 2^-9 / (1 - 0.4) ~ 1e-2; the bound is 2e-2.
* ORTH_TOL: max |V^T V - I| for V_k rounded to bf16 from an fp32 basis that
  is orthonormal to ~1e-6: each entry of V^T V moves by at most ~2 * 2^-9.
* ENERGY_RTOL: the fraction of the calibration tokens' energy inside the
  span, GPU vs oracle: first-order insensitive to the span's error (the
  oracle's span is near-stationary for it), so 1e-4 relative.
"""
import math

import numpy as np
import pytest

import gsi_inputs as gi
from gsi_testlib import GpuLinear, to_bits, to_dev

pytestmark = pytest.mark.gpu

SIN_TOL = 2e-2
ORTH_TOL = 1e-2
ENERGY_RTOL = 1e-4


@pytest.fixture(scope="module")
def cal():
    from oracle import calibration
    return calibration


def _run(gsi, X_bits, Q0_bits, iters, stream=None):
    import torch
    n, d = X_bits.shape
    k = Q0_bits.shape[1]
    X = to_dev(X_bits)
    Q0 = to_dev(Q0_bits)
    V = torch.full((d, k), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(gsi.gsi_calibrate_workspace_size(n, d, k), dtype=torch.uint8, device="cuda")
    gsi.gsi_calibrate(X, Q0, iters, V, ws, stream)
    st = gsi.gsi_calibrate_status(ws, stream)
    return V, ws, st


def _check(cal, X_bits, Q0_bits, iters, V_bits, what):
    X = gi.bf16_bits_to_f64(X_bits)
    Q0 = gi.bf16_bits_to_f64(Q0_bits)
    V = gi.bf16_bits_to_f64(V_bits)
    k = V.shape[1]
    assert np.all(np.isfinite(V)), what
    ref = cal.subspace_iteration(X, Q0, iters)
    sines = cal.principal_sines(V, ref)
    orth = np.max(np.abs(V.T @ V - np.eye(k)))
    e_gpu, e_ref = cal.captured_energy(X, V), cal.captured_energy(X, ref)
    assert sines[0] <= SIN_TOL, f"{what}: max sine {sines[0]:.3e}"
    assert orth <= ORTH_TOL, f"{what}: |V^T V - I| = {orth:.3e}"
    assert abs(e_gpu - e_ref) <= ENERGY_RTOL * e_ref, f"{what}: energy {e_gpu} vs {e_ref}"
    return sines[0]


@pytest.mark.parametrize("n,d,k,iters", [
    (256, 128, 16, 10),
    (512, 256, 32, 10),
    (392, 264, 64, 10),      # ragged n (not a multiple of 64) and d (a partial 32-column slice)
    (1024, 1024, 128, 8),
    (1040, 1032, 256, 8),    # k = 256 with a ragged d
])
def test_calibrate_matches_oracle(gsi, cal, n, d, k, iters):
    cs = gi.calibration_activations(n, d, k, seed=300 + k)
    Q0 = gi.calibration_start(d, k, seed=300 + k)
    V, _, st = _run(gsi, cs.X_bits, Q0, iters)
    assert st == 0, gsi.gsi_status_string(st)
    _check(cal, cs.X_bits, Q0, iters, to_bits(V), f"n={n} d={d} k={k}")


def test_calibrate_gptj_size(gsi, cal):
    """The GPT-J-shaped calibration (one 2048-token sequence, d = 4096,
    k = 256, 8 iterations) that the benchmark times."""
    c = gi.calibration_gptj()
    cs = gi.calibration_activations(c["n"], c["d"], c["k"], seed=c["seed"])
    Q0 = gi.calibration_start(c["d"], c["k"], seed=c["seed"])
    V, _, st = _run(gsi, cs.X_bits, Q0, c["iters"])
    assert st == 0, gsi.gsi_status_string(st)
    _check(cal, cs.X_bits, Q0, c["iters"], to_bits(V), "gptj d=4096 k=256")


def test_calibrate_zero_iterations_orthonormalises_start(gsi, cal):
    """iters = 0: V_k is an orthonormal basis of span(Q0), up to the final
    bf16 rounding."""
    d, k = 520, 128
    Q0 = gi.calibration_start(d, k, seed=311)
    X = gi.calibration_activations(128, d, k, seed=311).X_bits
    V, _, st = _run(gsi, X, Q0, 0)
    assert st == 0
    Vf = gi.bf16_bits_to_f64(to_bits(V))
    assert np.max(cal.principal_sines(Vf, gi.bf16_bits_to_f64(Q0))) <= 4e-3
    assert np.max(np.abs(Vf.T @ Vf - np.eye(k))) <= ORTH_TOL


def test_calibrate_converges_to_the_top_k_eigenspace(gsi, cal):
    """With a strong planted gap and enough iterations both the GPU and the
    oracle's iteration reach the top-k eigenspace of X^T X (the definition,
    by the oracle's eigensolver)."""
    n, d, k = 2048, 512, 64
    cs = gi.calibration_activations(n, d, k, seed=321, gap=0.3)
    Q0 = gi.calibration_start(d, k, seed=321)
    V, _, st = _run(gsi, cs.X_bits, Q0, 30)
    assert st == 0
    X = gi.bf16_bits_to_f64(cs.X_bits)
    top, lam = cal.top_k_subspace(X, k + 1)
    assert lam[k] / lam[k - 1] < 0.2
    assert np.max(cal.principal_sines(gi.bf16_bits_to_f64(to_bits(V)), top[:, :k])) <= 1e-2


def test_calibrate_deterministic_and_graph_capturable(gsi):
    """Two eager calls and a CUDA-graph replay give bit-identical V_k (fixed
    summation orders everywhere, no atomics in any sum)."""
    import torch
    n, d, k, iters = 512, 384, 64, 6
    cs = gi.calibration_activations(n, d, k, seed=331)
    Q0b = gi.calibration_start(d, k, seed=331)
    X, Q0 = to_dev(cs.X_bits), to_dev(Q0b)
    ws = torch.empty(gsi.gsi_calibrate_workspace_size(n, d, k), dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(2):
        V = torch.empty((d, k), dtype=torch.bfloat16, device="cuda")
        gsi.gsi_calibrate(X, Q0, iters, V, ws)
        assert gsi.gsi_calibrate_status(ws) == 0
        outs.append(to_bits(V))
    assert np.array_equal(outs[0], outs[1])
    Vg = torch.zeros((d, k), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            gsi.gsi_calibrate(X, Q0, iters, Vg, ws, s)
    for _ in range(2):
        Vg.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert np.array_equal(to_bits(Vg), outs[0])
    assert gsi.gsi_calibrate_status(ws) == 0


def test_calibrate_zero_tokens_report_rank(gsi):
    """X = 0: every column of the block vanishes; the status says so and the
    output stays finite."""
    n, d, k = 128, 256, 32
    X = np.zeros((n, d), dtype=np.uint16)
    Q0 = gi.calibration_start(d, k, seed=341)
    V, ws, st = _run(gsi, X, Q0, 3)
    assert st == gsi.GSI_ERR_RANK
    assert np.all(np.isfinite(gi.bf16_bits_to_f64(to_bits(V))))
    # the next call on the same workspace starts clean
    cs = gi.calibration_activations(n, d, k, seed=341)
    gsi.gsi_calibrate(to_dev(cs.X_bits), to_dev(Q0), 3, V, ws)
    assert gsi.gsi_calibrate_status(ws) == 0


def test_calibrated_basis_drives_the_gated_map(gsi, orc, cal):
    """The step the calibration serves: V_k from gsi_calibrate, M from
    gsi_precompute_M, a handle, and gated calls on held-out tokens of the same
    distribution, against the oracle's own pipeline (its subspace iteration,
    its bf16 rounding of V_k, its M, its rho) on the same tokens.  eps is the
    median of the oracle's rho, so the gate splits the tokens in half.  The
    two bases differ by principal angles of ~1e-2 at most, mostly in the
    weakest directions, which moves a token's rho by ~1e-4 against a spread
    of ~1e-2 across tokens: the fast fractions agree within 2 points and the
    mean rho within 1%."""
    n, d, k, d_out, iters = 2048, 1024, 128, 512, 8
    cs = gi.calibration_activations(n, d, k, seed=351)
    Q0 = gi.calibration_start(d, k, seed=351)
    V, _, st = _run(gsi, cs.X_bits, Q0, iters)
    assert st == 0
    held = gi.calibration_activations(512, d, k, seed=352, U=cs.U).X_bits
    W = gi.gaussian_weights(d_out, d, seed=353)
    ref_V = gi.to_bf16_bits(cal.subspace_iteration(gi.bf16_bits_to_f64(cs.X_bits),
                                                   gi.bf16_bits_to_f64(Q0), iters))
    ref_M = orc.precompute_M_bf16(W, ref_V)
    rho_ref = orc.forward_bf16(W, ref_V, ref_M, np.float32(1.0), held)["rho"]
    eps = float(np.float32(np.median(rho_ref)))
    gate_ref = orc.forward_bf16(W, ref_V, ref_M, np.float32(eps), held)["gate"]
    lin = GpuLinear(gsi, orc, W, to_bits(V), eps, max_T=512)
    try:
        _, gate, rho = lin.forward(held)
    finally:
        lin.close()
    f_gpu, f_ref = 1.0 - np.mean(gate), 1.0 - np.mean(gate_ref)
    assert 0.4 < f_ref < 0.6, f_ref
    assert abs(f_gpu - f_ref) <= 0.02, (f_gpu, f_ref)
    assert abs(np.mean(rho) - np.mean(rho_ref)) <= 1e-2 * np.mean(rho_ref)


def test_cascade_matches_oracle(gsi, cal):
    """Depth cascade over 4 depth-coherent layers (8 iterations for layer 0,
    2 for each later layer from the previous basis) against the oracle's
    cascade; the result equals gsi_calibrate called layer by layer."""
    import torch
    L, n, d, k = 4, 512, 256, 32
    sets = gi.calibration_cascade(L, n, d, k, seed=361)
    Q0b = gi.calibration_start(d, k, seed=361)
    Xs = [to_dev(s.X_bits) for s in sets]
    Q0 = to_dev(Q0b)
    Vs = [torch.full((d, k), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(L)]
    ws = torch.empty(gsi.gsi_calibrate_workspace_size(n, d, k), dtype=torch.uint8, device="cuda")
    gsi.gsi_calibrate_cascade(Xs, Q0, 8, 2, Vs, ws)
    assert gsi.gsi_calibrate_status(ws) == 0
    ref = cal.cascade([gi.bf16_bits_to_f64(s.X_bits) for s in sets],
                      gi.bf16_bits_to_f64(Q0b), 8, 2)
    for layer, (V, R, s) in enumerate(zip(Vs, ref, sets)):
        Vf = gi.bf16_bits_to_f64(to_bits(V))
        X = gi.bf16_bits_to_f64(s.X_bits)
        assert np.max(cal.principal_sines(Vf, R)) <= SIN_TOL, layer
        e_gpu, e_ref = cal.captured_energy(X, Vf), cal.captured_energy(X, R)
        assert abs(e_gpu - e_ref) <= ENERGY_RTOL * e_ref, layer
    # layer by layer through gsi_calibrate: the same bits
    prev = Q0
    for layer in range(L):
        V = torch.empty((d, k), dtype=torch.bfloat16, device="cuda")
        gsi.gsi_calibrate(Xs[layer], prev, 8 if layer == 0 else 2, V, ws)
        assert np.array_equal(to_bits(V), to_bits(Vs[layer])), layer
        prev = V


@pytest.mark.parametrize("k", [64, 128])
@pytest.mark.parametrize("T", [1, 96])
def test_theorem4_holds_on_gpu_outputs(gsi, orc, k, T):
    """Operating points (N4): on power-law tokens with the population top-k
    basis, every token the GPU sends down the fast path has
    ||y - W x|| <= ||W||_2 eps ||x|| (Theorem 4, section 2.2), with W x and
    ||W||_2 from the oracle in fp64; eps = inf (static projection) sends every
    token fast.  The GPU's extra error (bf16 M, fp32 sums) is a few 1e-3 of
    ||y|| and leaves the bound with room at these shapes."""
    d_out, d, n_tok = 2048, 1024, 96
    cs = gi.sweep_activations(n_tok, d, seed=371, r=512)
    W = gi.gaussian_weights(d_out, d, seed=372)
    Vb = gi.to_bf16_bits(cs.U[:, :k])
    w2 = orc.spectral_norm(gi.bf16_bits_to_f64(W)) * (1 + 1e-6)
    Xf = gi.bf16_bits_to_f64(cs.X_bits)
    y_exact = Xf @ gi.bf16_bits_to_f64(W).T
    xn = np.linalg.norm(Xf, axis=1)
    for eps in (0.05, 0.1, float("inf")):
        lin = GpuLinear(gsi, orc, W, Vb, eps, max_T=n_tok)
        try:
            y, gate, rho = lin.forward(cs.X_bits, one_by_one=(T == 1))
        finally:
            lin.close()
        fast = gate == 0
        if math.isinf(eps):
            assert fast.all()
            continue
        assert 0 < fast.sum() < n_tok, (k, eps, fast.sum())
        err = np.linalg.norm(y - y_exact, axis=1)
        ratio = err[fast] / (w2 * eps * xn[fast])
        assert ratio.max() <= 1.0, (k, eps, ratio.max())
