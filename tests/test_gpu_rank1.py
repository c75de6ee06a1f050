"""gsi_refine_rank1 and gsi_calibrate_cascade_rank1 (the depth cascade's
rank-1 DGKS corrections) against the fp64 oracle, through the C ABI.

The result depends on which column each correction picks (an argmax over
residual norms), and the GPU takes that decision on its own fp32 residuals of
a bf16 product C V.  So every comparison replays the GPU's choices in the
oracle (rank1_refine(..., order=gpu_order)) and checks, step by step, that
each choice was a largest residual up to the GPU's rounding.

Tolerances, from the arithmetic:
* NEAR_TOL: C V is formed once from bf16 roundings of V and X V, which moves
  every column of C V by about 2^-8 of the largest column norm; the GPU's
  residual norms carry that error, so a chosen column's oracle residual may
  sit below the oracle's maximum by up to 1e-2 of the largest ||C v_i||.
* SIN_TOL: the same 2^-8 relative error enters each correction's residual
  direction, and the output is rounded to bf16 (2^-9); the corrected columns'
  directions agree to a few times 2^-8: the largest principal sine between
  the GPU's span and the replayed oracle's is at most 2e-2.
* ORTH_TOL: bf16 rounding of an fp32 basis that rotations keep orthonormal to
  ~1e-6: 1e-2.
* ENERGY: the refined basis is not a stationary point of the captured energy
  (a few corrections leave residuals), so a span error of sine delta moves
  the energy at first order; the GPU's captured energy must not fall below
  the oracle's by more than 2 * SIN_TOL * (relative residual) ~ 2e-3.
"""
import math

import numpy as np
import pytest

import gsi_inputs as gi
from gsi_testlib import to_bits, to_dev

pytestmark = pytest.mark.gpu

NEAR_TOL = 1e-2
SIN_TOL = 2e-2
ORTH_TOL = 1e-2
ENERGY_DROP = 2e-3


@pytest.fixture(scope="module")
def cal():
    from oracle import calibration
    return calibration


def _ws(gsi, n, d, k):
    import torch
    return torch.empty(gsi.gsi_refine_rank1_workspace_size(n, d, k), dtype=torch.uint8,
                       device="cuda")


def _refine(gsi, X_bits, V_bits, c, ws=None):
    import torch
    n, d = X_bits.shape
    k = V_bits.shape[1]
    ws = _ws(gsi, n, d, k) if ws is None else ws
    V = torch.full((d, k), float("nan"), dtype=torch.bfloat16, device="cuda")
    order = torch.full((max(1, c),), -1, dtype=torch.int32, device="cuda")
    gsi.gsi_refine_rank1(to_dev(X_bits), to_dev(V_bits), c, V, ws, order=order)
    st = gsi.gsi_calibrate_status(ws)
    return to_bits(V), order.cpu().numpy()[:c].astype(int), st


def _check_replay(cal, X, V_in, c, V_bits, order, what):
    """The GPU's V against the oracle replaying its column choices."""
    Vg = gi.bf16_bits_to_f64(V_bits)
    k = Vg.shape[1]
    assert np.all(np.isfinite(Vg)), what
    assert np.all((order >= 0) & (order < k)), (what, order)
    Q, chosen, norms = cal.rank1_refine(X, V_in, c, order=order)
    assert list(chosen) == list(order)
    Q0 = cal.positive_qr_basis(V_in)
    pmax = np.max(np.linalg.norm(X.T @ (X @ Q0), axis=0))
    for s in range(c):
        gap = np.max(norms[s]) - norms[s][order[s]]
        assert gap <= NEAR_TOL * pmax, f"{what}: step {s} chose {order[s]}, {gap / pmax:.2e} below max"
    sn = np.max(cal.principal_sines(Vg, Q))
    orth = np.max(np.abs(Vg.T @ Vg - np.eye(k)))
    assert sn <= SIN_TOL, f"{what}: max sine {sn:.3e}"
    assert orth <= ORTH_TOL, f"{what}: |V^T V - I| = {orth:.3e}"
    e_g, e_r, e_0 = (cal.captured_energy(X, Vg), cal.captured_energy(X, Q),
                     cal.captured_energy(X, V_in))
    assert e_g >= e_r - ENERGY_DROP * e_r, f"{what}: energy {e_g} vs oracle {e_r}"
    return sn, e_g, e_r, e_0


def _start_pair(n, d, k, seed, mix=0.3):
    """Tokens of a layer and the basis calibrated on the layer before it
    (the oracle's subspace iteration, rounded to bf16): the cascade's input."""
    from oracle import calibration as cal
    sets = gi.calibration_cascade(2, n, d, k, seed=seed, mix=mix)
    Q0 = gi.calibration_start(d, k, seed=seed)
    V0 = cal.subspace_iteration(gi.bf16_bits_to_f64(sets[0].X_bits), gi.bf16_bits_to_f64(Q0), 8)
    return sets[1].X_bits, gi.to_bf16_bits(V0)


@pytest.mark.parametrize("n,d,k,c", [
    (256, 128, 16, 8),
    (512, 256, 32, 16),
    (392, 264, 64, 24),      # ragged n, and d not a multiple of the 32-column slices
    (1024, 1024, 128, 32),
    (1040, 1032, 256, 40),   # k = 256 with a ragged d
])
def test_refine_matches_oracle(gsi, cal, n, d, k, c):
    X_bits, V_bits = _start_pair(n, d, k, seed=400 + k)
    Vg, order, st = _refine(gsi, X_bits, V_bits, c)
    assert st == 0, gsi.gsi_status_string(st)
    X, V_in = gi.bf16_bits_to_f64(X_bits), gi.bf16_bits_to_f64(V_bits)
    _, e_g, _, e_0 = _check_replay(cal, X, V_in, c, Vg, order, f"n={n} d={d} k={k} c={c}")
    assert e_g > e_0, "the corrections did not raise the captured energy"


def test_refine_more_slices_than_ctas(gsi, cal):
    """d = 8200: 257 slices of 32 columns (the last one ragged), more than the
    resident grid (at most one 512-thread CTA per SM), so CTAs own several
    slices and reload each one from memory in every phase."""
    n, d, k, c = 512, 8200, 32, 12
    X_bits, V_bits = _start_pair(n, d, k, seed=461)
    Vg, order, st = _refine(gsi, X_bits, V_bits, c)
    assert st == 0, gsi.gsi_status_string(st)
    X, V_in = gi.bf16_bits_to_f64(X_bits), gi.bf16_bits_to_f64(V_bits)
    _, e_g, _, e_0 = _check_replay(cal, X, V_in, c, Vg, order, f"n={n} d={d} k={k} c={c}")
    assert e_g > e_0


def test_refine_gptj_size(gsi, cal):
    """The GPT-J-shaped refinement the cascade benchmark runs per layer
    (n = 2048 tokens, d = 4096, k = 256), 32 corrections."""
    c = gi.calibration_gptj()
    X_bits, V_bits = _start_pair(c["n"], c["d"], c["k"], seed=c["seed"] + 7)
    Vg, order, st = _refine(gsi, X_bits, V_bits, 32)
    assert st == 0
    _check_replay(cal, gi.bf16_bits_to_f64(X_bits), gi.bf16_bits_to_f64(V_bits), 32, Vg, order,
                  "gptj")


def test_refine_recovers_a_rotated_eigenvector(gsi, cal):
    """C = U diag(lam) U^T whose top-32 eigenvectors are the start basis
    except column 5, rotated by 0.5 rad out of it: one correction picks column
    5 and recovers the rotated eigenvector (up to bf16 roundings)."""
    d, k, j, phi = 256, 32, 5, 0.5
    rng = np.random.default_rng(411)
    G, R = np.linalg.qr(rng.standard_normal((d, d)))
    G = G * np.sign(np.diag(R))
    lam = np.concatenate([np.linspace(10.0, 4.0, k), np.linspace(1.5, 0.05, d - k)])
    U = G.copy()
    U[:, j] = math.cos(phi) * G[:, j] + math.sin(phi) * G[:, k]
    U[:, k] = -math.sin(phi) * G[:, j] + math.cos(phi) * G[:, k]
    X_bits = gi.to_bf16_bits(np.diag(np.sqrt(lam)) @ U.T)
    V_bits = gi.to_bf16_bits(G[:, :k])
    Vg0, _, st = _refine(gsi, X_bits, V_bits, 0)
    assert st == 0
    s0 = np.max(cal.principal_sines(gi.bf16_bits_to_f64(Vg0), U[:, :k]))
    assert abs(s0 - math.sin(phi)) < 1e-2
    Vg, order, st = _refine(gsi, X_bits, V_bits, 1)
    assert st == 0
    assert list(order) == [j]
    Vf = gi.bf16_bits_to_f64(Vg)
    assert np.max(cal.principal_sines(Vf, U[:, :k])) < 1.5e-2
    assert abs(abs(Vf[:, j] @ U[:, j]) - 1.0) < 1e-3


def test_refine_zero_corrections_is_the_positive_qr_factor(gsi, cal):
    """corrections = 0 returns the positive-diagonal QR factor of V_in,
    column by column (the basis, not only the span), rounded to bf16."""
    n, d, k = 256, 520, 64
    X_bits = gi.calibration_activations(n, d, k, seed=421).X_bits
    V_bits = gi.calibration_start(d, k, seed=421)
    Vg, _, st = _refine(gsi, X_bits, V_bits, 0)
    assert st == 0
    Q = cal.positive_qr_basis(gi.bf16_bits_to_f64(V_bits))
    assert np.max(np.abs(gi.bf16_bits_to_f64(Vg) - Q)) <= 4e-3 * np.max(np.abs(Q))


def test_refine_invariant_span_leaves_the_basis(gsi, cal):
    """Tokens that live in span(e_1..e_k) and the start basis e_1..e_k (both
    exact in bf16): span(V) is invariant under C, every residual is rounding
    inside span(V) and vanishes under the re-orthogonalisation, no
    correction rotates, V comes back as it went in, and nothing turns
    non-finite."""
    n, d, k = 256, 256, 32
    rng = np.random.default_rng(431)
    X = np.zeros((n, d))
    X[:, :k] = rng.standard_normal((n, k)) @ np.diag(np.linspace(3.0, 1.0, k))
    V = np.eye(d)[:, :k]
    Vg, order, st = _refine(gsi, gi.to_bf16_bits(X), gi.to_bf16_bits(V), 4)
    assert st == 0
    assert np.array_equal(Vg, gi.to_bf16_bits(V))
    assert np.all((order >= 0) & (order < k))


def test_refine_deterministic_and_graph_capturable(gsi):
    """Two eager calls and a CUDA-graph replay give bit-identical bases and
    the same column choices (fixed summation orders, no atomics in any
    sum)."""
    import torch
    n, d, k, c = 512, 384, 64, 20
    X_bits, V_bits = _start_pair(n, d, k, seed=441)
    X, V0 = to_dev(X_bits), to_dev(V_bits)
    ws = _ws(gsi, n, d, k)
    outs = []
    for _ in range(2):
        V = torch.empty((d, k), dtype=torch.bfloat16, device="cuda")
        od = torch.empty((c,), dtype=torch.int32, device="cuda")
        gsi.gsi_refine_rank1(X, V0, c, V, ws, order=od)
        assert gsi.gsi_calibrate_status(ws) == 0
        outs.append((to_bits(V), od.cpu().numpy()))
    assert np.array_equal(outs[0][0], outs[1][0])
    assert np.array_equal(outs[0][1], outs[1][1])
    Vg = torch.zeros((d, k), dtype=torch.bfloat16, device="cuda")
    og = torch.zeros((c,), dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            gsi.gsi_refine_rank1(X, V0, c, Vg, ws, order=og, stream=s)
    for _ in range(2):
        Vg.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert np.array_equal(to_bits(Vg), outs[0][0])
        assert np.array_equal(og.cpu().numpy(), outs[0][1])
    # in place: V_out may be V_in
    Vi = V0.clone()
    gsi.gsi_refine_rank1(X, Vi, c, Vi, ws)
    assert np.array_equal(to_bits(Vi), outs[0][0])


def test_cascade_rank1_matches_oracle(gsi, cal):
    """The rank-1 cascade over 4 depth-coherent layers (8 iterations for
    layer 0, 16 corrections per later layer) against the oracle, replaying
    the GPU's column choices layer by layer; the cascade equals gsi_calibrate
    followed by gsi_refine_rank1 layer by layer, bit for bit."""
    import torch
    L, n, d, k, c = 4, 512, 256, 32, 16
    sets = gi.calibration_cascade(L, n, d, k, seed=451)
    Q0b = gi.calibration_start(d, k, seed=451)
    Xs = [to_dev(s.X_bits) for s in sets]
    Q0 = to_dev(Q0b)
    Vs = [torch.full((d, k), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(L)]
    order = torch.full(((L - 1) * c,), -1, dtype=torch.int32, device="cuda")
    ws = _ws(gsi, n, d, k)
    gsi.gsi_calibrate_cascade_rank1(Xs, Q0, 8, c, Vs, ws, order=order)
    assert gsi.gsi_calibrate_status(ws) == 0
    od = order.cpu().numpy().reshape(L - 1, c).astype(int)
    Vb = [to_bits(V) for V in Vs]
    # layer 0: the block iteration
    from test_gpu_calibration import _check
    _check(cal, sets[0].X_bits, Q0b, 8, Vb[0], "layer 0")
    for layer in range(1, L):
        _check_replay(cal, gi.bf16_bits_to_f64(sets[layer].X_bits),
                      gi.bf16_bits_to_f64(Vb[layer - 1]), c, Vb[layer], od[layer - 1],
                      f"layer {layer}")
    prev = torch.empty((d, k), dtype=torch.bfloat16, device="cuda")
    ws2 = torch.empty(gsi.gsi_calibrate_workspace_size(n, d, k), dtype=torch.uint8, device="cuda")
    gsi.gsi_calibrate(Xs[0], Q0, 8, prev, ws2)
    assert np.array_equal(to_bits(prev), Vb[0])
    for layer in range(1, L):
        V = torch.empty((d, k), dtype=torch.bfloat16, device="cuda")
        o = torch.empty((c,), dtype=torch.int32, device="cuda")
        gsi.gsi_refine_rank1(Xs[layer], prev, c, V, ws, order=o)
        assert np.array_equal(to_bits(V), Vb[layer]), layer
        assert np.array_equal(o.cpu().numpy(), od[layer - 1]), layer
        prev = V


def test_refine_launch_count(gsi):
    """All corrections run in one persistent launch: the count does not grow
    with the number of corrections."""
    n, d, k = 512, 256, 32
    base = gsi.gsi_refine_rank1_launch_count(n, d, k, 0)
    one = gsi.gsi_refine_rank1_launch_count(n, d, k, 1)
    assert 0 < base < one
    assert gsi.gsi_refine_rank1_launch_count(n, d, k, 500) == one
