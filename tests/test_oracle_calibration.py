"""Pins of the calibration oracle (oracle/calibration.py), CPU only.

Each pin checks one function against a fact that the mathematics fixes
independently of the function's own formula:

* top_k_subspace on a planted spectrum X = A diag(s) B^T (A, B orthonormal,
  s distinct): the eigenvectors are the columns of B up to sign, in the
  order of s, and the eigenvalues are s^2;
* subspace_iteration in two dimensions, where t iterations from the angle a
  give the exact angle atan((s2/s1)^(2t) tan a), and on a diagonal second
  moment with n != d, where the iterate is the normalised s^(2t) * q0;
* the span of the iterate does not depend on the basis of the start block;
* on a gapped planted spectrum, the principal-angle tangents obey the
  textbook bound tan(theta_t) <= (lambda_{k+1}/lambda_k)^t tan(theta_0) and
  reach the planted subspace to rounding;
* principal_sines on hand-built subspaces with known angles, including an
  angle of 1e-9 (full relative accuracy for small angles);
* orthonormal_basis: orthonormal columns spanning the input;
* captured_energy on the planted spectrum: sum of the k largest s^2 over the
  sum of all;
* cascade: with no refinement every layer keeps layer 0's subspace; with
  enough refinement each planted layer reaches its own top-k eigenspace; one
  refinement step is one product with the next layer's second moment applied
  to the previous layer's basis;
* positive_qr_basis: Q^T V is upper triangular with a positive diagonal and
  Q R reproduces V;
* dgks_orthogonalize: a vector within 1e-10 of span(B) comes out orthogonal
  to B to rounding (one classical Gram-Schmidt pass leaves ~1e-6), and the
  second pass runs exactly when the first kept less than 1/sqrt(2) of the
  norm;
* rank1_refine: on a planted spectrum whose top-k eigenvectors are the start
  basis except one, rotated by phi out of it, one correction picks that
  column and recovers the rotated eigenvector exactly (the plane of the
  column and its residual holds it); in two dimensions one correction gives
  the top eigenvector (numpy's eigh); the columns stay orthonormal, the
  captured trace never falls, and on a gapped spectrum the corrections reach
  the top-k eigenspace;
* cascade_rank1: with no corrections every layer keeps layer 0's span; with
  enough corrections each planted layer reaches its own top-k eigenspace.

test_calibration_pins_catch_mutant plants plausible mistakes in a copy of the
oracle's source and requires that at least one pin rejects each copy.
"""
import importlib.util
import math
import os

import numpy as np
import pytest

import oracle.calibration as cal_mod

ORACLE_SRC = cal_mod.__file__


def _orthonormal(rows, cols, seed):
    rng = np.random.default_rng(seed)
    Q, R = np.linalg.qr(rng.standard_normal((rows, cols)))
    return Q * np.sign(np.diag(R))


def _planted(n, d, r, s, seed):
    A = _orthonormal(n, r, seed)
    B = _orthonormal(d, r, seed + 1)
    return A @ np.diag(s) @ B.T, A, B


def pin_top_k_planted(cal):
    s = np.array([9.0, 7.0, 5.5, 4.0, 3.0, 2.0, 1.5, 1.0])
    X, _, B = _planted(30, 20, 8, s, 11)
    k = 5
    V, lam = cal.top_k_subspace(X, k)
    assert V.shape == (20, k)
    M = np.abs(B[:, :k].T @ V)
    assert np.max(np.abs(M - np.eye(k))) < 1e-10, "eigenvectors are not the planted columns"
    assert np.allclose(lam, s[:k] ** 2, rtol=1e-12, atol=0)


def pin_iteration_two_dims(cal):
    s1, s2, a = 2.0, 1.5, 1.0
    X = np.diag([s1, s2])
    Q0 = np.array([[math.cos(a)], [math.sin(a)]])
    for t in range(0, 7):
        Q = cal.subspace_iteration(X, Q0, t)
        assert Q.shape == (2, 1)
        assert abs(np.linalg.norm(Q) - 1.0) < 1e-14
        want = (s2 / s1) ** (2 * t) * math.tan(a)
        got = abs(Q[1, 0] / Q[0, 0])
        assert abs(got - want) <= 1e-12 * want, (t, got, want)


def pin_iteration_diagonal_moment(cal):
    # X = A diag(s) with A (n x d) orthonormal columns: X^T X = diag(s^2),
    # so t iterations from q0 give +-(s^(2t) * q0) / ||s^(2t) * q0||.
    n, d = 7, 4
    s = np.array([1.7, 1.3, 1.1, 0.6])
    X = _orthonormal(n, d, 21) @ np.diag(s)
    q0 = np.array([[0.3], [-0.5], [0.7], [0.4]])
    for t in range(0, 5):
        Q = cal.subspace_iteration(X, q0, t)
        v = (s ** (2 * t))[:, None] * q0
        v /= np.linalg.norm(v)
        assert min(np.max(np.abs(Q - v)), np.max(np.abs(Q + v))) < 1e-13, t


def pin_iteration_span_invariance(cal):
    rng = np.random.default_rng(31)
    X = rng.standard_normal((40, 24))
    Q0 = rng.standard_normal((24, 5))
    R = rng.standard_normal((5, 5)) + 3 * np.eye(5)
    for t in (0, 1, 3):
        Qa = cal.subspace_iteration(X, Q0, t)
        Qb = cal.subspace_iteration(X, Q0 @ R, t)
        assert np.max(cal.principal_sines(Qa, Qb)) < 1e-10, t


def pin_iteration_rate(cal):
    k = 4
    s = np.array([3.0, 2.6, 2.3, 2.0, 1.0, 0.9, 0.7, 0.5, 0.3, 0.2])
    X, _, B = _planted(50, 16, 10, s, 41)
    ratio = (s[k] / s[k - 1]) ** 2          # lambda_{k+1} / lambda_k
    Q0 = np.random.default_rng(42).standard_normal((16, k))

    def tan_max(Q):
        sn = np.max(cal.principal_sines(Q, B[:, :k]))
        return sn / math.sqrt(1.0 - sn * sn)

    t0 = tan_max(cal.subspace_iteration(X, Q0, 0))
    for t in range(1, 8):
        tt = tan_max(cal.subspace_iteration(X, Q0, t))
        assert tt <= ratio ** t * t0 * (1 + 1e-9) + 1e-14, (t, tt, ratio ** t * t0)
    assert tan_max(cal.subspace_iteration(X, Q0, 60)) < 1e-12


def pin_principal_sines(cal):
    e = np.eye(4)
    for th in (1e-9, 0.3, 0.7, math.pi / 2):
        A = e[:, :1]
        B = (math.cos(th) * e[:, 0] + math.sin(th) * e[:, 1])[:, None]
        got = cal.principal_sines(A, B)
        assert abs(got[0] - math.sin(th)) <= 1e-15 + 1e-12 * math.sin(th), (th, got)
    a, b = 0.2, 0.9
    A = e[:, :2]
    B = np.stack([math.cos(a) * e[:, 0] + math.sin(a) * e[:, 2],
                  math.cos(b) * e[:, 1] + math.sin(b) * e[:, 3]], axis=1)
    rot = np.array([[math.cos(0.4), -math.sin(0.4)], [math.sin(0.4), math.cos(0.4)]])
    got = cal.principal_sines(A @ rot, B @ rot.T)
    assert np.allclose(got, [math.sin(b), math.sin(a)], rtol=0, atol=1e-14), got
    Y = np.random.default_rng(51).standard_normal((9, 3))
    same = cal.principal_sines(Y, Y @ np.array([[1.0, 2.0, 0.0], [0.0, 1.0, 3.0], [1.0, 0.0, 1.0]]))
    assert np.max(same) < 1e-14, same


def pin_orthonormal_basis(cal):
    Y = np.random.default_rng(61).standard_normal((12, 4)) @ np.diag([1.0, 1e3, 1e-3, 5.0])
    Q = cal.orthonormal_basis(Y)
    assert Q.shape == (12, 4)
    assert np.max(np.abs(Q.T @ Q - np.eye(4))) < 1e-14
    assert np.max(np.abs(Q @ (Q.T @ Y) - Y)) < 1e-12 * np.max(np.abs(Y))


def pin_captured_energy(cal):
    s = np.array([4.0, 3.0, 2.0, 1.0, 0.5])
    X, _, B = _planted(20, 10, 5, s, 71)
    for k in (1, 2, 5):
        want = float(np.sum(s[:k] ** 2) / np.sum(s ** 2))
        assert abs(cal.captured_energy(X, B[:, :k]) - want) < 1e-13, k


def pin_cascade(cal):
    # (i) no refinement past layer 0: every layer keeps layer 0's subspace,
    # which is the plain iteration on layer 0 (not the start block)
    rng = np.random.default_rng(81)
    Xs = [rng.standard_normal((30, 12)) @ np.diag(np.linspace(3.0, 0.5, 12)) for _ in range(3)]
    Q0 = rng.standard_normal((12, 4))
    Vs = cal.cascade(Xs, Q0, 5, 0)
    assert len(Vs) == 3
    assert np.max(cal.principal_sines(Vs[0], Q0)) > 1e-3
    for V in Vs[1:]:
        assert np.max(cal.principal_sines(V, Vs[0])) < 1e-12
    # (ii) planted layers whose top-4 subspaces differ: enough refinement
    # reaches each layer's own top-4 eigenspace
    s = np.array([3.0, 2.6, 2.3, 2.0, 0.9, 0.7, 0.5, 0.3])
    Xp, Bs = [], []
    for i in range(3):
        X, _, B = _planted(40, 16, 8, s, 90 + 3 * i)
        Xp.append(X)
        Bs.append(B)
    Vs = cal.cascade(Xp, Q0=np.random.default_rng(91).standard_normal((16, 4)),
                     iters_first=40, iters_next=40)
    for V, B in zip(Vs, Bs):
        assert np.max(cal.principal_sines(V, B[:, :4])) < 1e-10
    # (iii) one refinement step from the previous basis: exactly one product
    # with layer 1's second moment applied to layer 0's result
    Vs = cal.cascade(Xp[:2], np.random.default_rng(92).standard_normal((16, 4)), 3, 1)
    want = Xp[1].T @ (Xp[1] @ Vs[0])
    assert np.max(cal.principal_sines(Vs[1], want)) < 1e-10


def pin_positive_qr(cal):
    V = np.random.default_rng(101).standard_normal((14, 5)) @ np.diag([1.0, -2.0, 0.5, 3.0, -1.0])
    Q = cal.positive_qr_basis(V)
    R = Q.T @ V
    assert np.max(np.abs(Q.T @ Q - np.eye(5))) < 1e-14
    assert np.max(np.abs(np.tril(R, -1))) < 1e-13, "R is not upper triangular"
    assert np.all(np.diag(R) > 0), np.diag(R)
    assert np.max(np.abs(Q @ R - V)) < 1e-13


def pin_dgks(cal):
    B = _orthonormal(20, 5, 111)
    rng = np.random.default_rng(112)
    z = rng.standard_normal(20)
    zp = z - B @ (B.T @ z)
    zp /= np.linalg.norm(zp)
    a = rng.standard_normal(5)
    a /= np.linalg.norm(a)
    # a vector within 1e-10 of span(B): one projection leaves ~1e-16 / 1e-10
    r = B @ a + 1e-10 * zp
    q, passes = cal.dgks_orthogonalize(B, r)
    assert passes == 2
    assert np.max(np.abs(B.T @ q)) / np.linalg.norm(q) < 1e-13
    assert abs(np.linalg.norm(q) - 1e-10) < 1e-15
    one = r - B @ (B.T @ r)   # a single classical pass, for scale: the test is sensitive
    assert np.max(np.abs(B.T @ one)) / np.linalg.norm(one) > 1e-9
    # the test keeps 0.8 of the norm: one pass; 0.6: two passes
    for inside, outside, want in ((0.6, 0.8, 1), (0.8, 0.6, 2)):
        r = inside * (B @ a) + outside * zp
        q, passes = cal.dgks_orthogonalize(B, r)
        assert passes == want, (inside, outside, passes)
        assert np.max(np.abs(q - outside * zp)) < 1e-14


def _rotated_planted(phi, seed):
    # C = U diag(lam) U^T; U = G except columns 2 and 4 (G orthogonal 12 x
    # 12): u = cos(phi) g2 + sin(phi) g4 keeps lambda = 5, w = -sin(phi) g2 +
    # cos(phi) g4 gets 1.5, so the top-4 eigenvectors are g0, g1, u, g3
    lam = np.array([9.0, 7.0, 5.0, 4.0, 1.5, 1.0, 0.7, 0.5, 0.3, 0.2, 0.1, 0.05])
    G = _orthonormal(12, 12, seed)
    U = G.copy()
    U[:, 2] = math.cos(phi) * G[:, 2] + math.sin(phi) * G[:, 4]
    U[:, 4] = -math.sin(phi) * G[:, 2] + math.cos(phi) * G[:, 4]
    X = np.diag(np.sqrt(lam)) @ U.T       # X^T X = U diag(lam) U^T
    return X, G, U


def pin_rank1_rotated_eigenvector(cal):
    phi = 0.4
    X, G, U = _rotated_planted(phi, 121)
    M = np.triu(np.random.default_rng(122).uniform(0.2, 1.0, (4, 4))) + np.eye(4)
    V = G[:, :4] @ M                       # positive-diagonal QR factor: G[:, :4]
    Q0, ch0, _ = cal.rank1_refine(X, V, 0)
    assert ch0 == []
    assert np.max(np.abs(Q0 - G[:, :4])) < 1e-13
    assert abs(np.max(cal.principal_sines(Q0, U[:, :4])) - math.sin(phi)) < 1e-13
    Q, chosen, norms = cal.rank1_refine(X, V, 1)
    assert chosen == [2], chosen
    # only column 2 has a residual: (lambda_u - lambda_w) sin(phi) cos(phi)
    want = np.zeros(4)
    want[2] = (5.0 - 1.5) * math.sin(phi) * math.cos(phi)
    assert np.max(np.abs(norms[0] - want)) < 1e-12, norms
    assert np.max(np.abs(Q[:, 2] - U[:, 2])) < 1e-12, "column 2 is not the rotated eigenvector"
    assert np.max(np.abs(Q[:, [0, 1, 3]] - G[:, [0, 1, 3]])) < 1e-13
    assert np.max(cal.principal_sines(Q, U[:, :4])) < 1e-12


def pin_rank1_two_dims(cal):
    X = np.random.default_rng(131).standard_normal((6, 2)) @ np.diag([1.4, 0.8])
    w, E = np.linalg.eigh(X.T @ X)
    top = E[:, np.argmax(w)]
    for start in (np.array([[1.0], [0.0]]), np.array([[0.3], [-0.9]])):
        Q, chosen, _ = cal.rank1_refine(X, start, 1)
        assert chosen == [0]
        assert min(np.max(np.abs(Q[:, 0] - top)), np.max(np.abs(Q[:, 0] + top))) < 1e-13


def pin_rank1_monotone_orthonormal(cal):
    rng = np.random.default_rng(141)
    X = rng.standard_normal((40, 16)) @ np.diag(np.linspace(3.0, 0.3, 16))
    V = rng.standard_normal((16, 5))
    C = X.T @ X
    prev = -1.0
    for c in range(0, 25):
        Q, chosen, norms = cal.rank1_refine(X, V, c)
        assert np.max(np.abs(Q.T @ Q - np.eye(5))) < 1e-12, c
        tr = float(np.trace(Q.T @ C @ Q))
        assert tr >= prev * (1.0 - 1e-13), (c, tr, prev)
        prev = tr
        for st in range(c):
            assert norms[st][chosen[st]] == np.max(norms[st])
    # every correction changed exactly one column of the previous result
    Qa = cal.rank1_refine(X, V, 7)[0]
    Qb, ch, _ = cal.rank1_refine(X, V, 8)
    diff = np.max(np.abs(Qb - Qa), axis=0)
    assert np.count_nonzero(diff > 0) == 1 and diff[ch[7]] > 0


def pin_rank1_converges(cal):
    s = np.array([3.0, 2.6, 2.3, 2.0, 1.0, 0.9, 0.7, 0.5, 0.3, 0.2])
    X, _, B = _planted(50, 16, 10, s, 151)
    V = np.random.default_rng(152).standard_normal((16, 4))
    Q = cal.rank1_refine(X, V, 300)[0]
    assert np.max(cal.principal_sines(Q, B[:, :4])) < 1e-9


def pin_cascade_rank1(cal):
    rng = np.random.default_rng(161)
    Xs = [rng.standard_normal((30, 12)) @ np.diag(np.linspace(3.0, 0.5, 12)) for _ in range(3)]
    Q0 = rng.standard_normal((12, 4))
    Vs = cal.cascade_rank1(Xs, Q0, 5, 0)
    assert len(Vs) == 3
    assert np.max(cal.principal_sines(Vs[0], cal.subspace_iteration(Xs[0], Q0, 5))) < 1e-12
    for V in Vs[1:]:
        assert np.max(cal.principal_sines(V, Vs[0])) < 1e-12
    s = np.array([3.0, 2.6, 2.3, 2.0, 0.9, 0.7, 0.5, 0.3])
    Xp, Bs = [], []
    for i in range(3):
        X, _, B = _planted(40, 16, 8, s, 170 + 3 * i)
        Xp.append(X)
        Bs.append(B)
    Vs = cal.cascade_rank1(Xp, np.random.default_rng(171).standard_normal((16, 4)), 40, 300)
    for V, B in zip(Vs, Bs):
        assert np.max(cal.principal_sines(V, B[:, :4])) < 1e-9


ALL_PINS = [
    pin_top_k_planted, pin_iteration_two_dims, pin_iteration_diagonal_moment,
    pin_iteration_span_invariance, pin_iteration_rate, pin_principal_sines,
    pin_orthonormal_basis, pin_captured_energy, pin_cascade, pin_positive_qr, pin_dgks,
    pin_rank1_rotated_eigenvector, pin_rank1_two_dims, pin_rank1_monotone_orthonormal,
    pin_rank1_converges, pin_cascade_rank1,
]


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_calibration_oracle_pin(pin):
    pin(cal_mod)


MUTANTS = [
    ("smallest eigenvectors", "idx = np.argsort(w)[::-1][:k]", "idx = np.argsort(w)[:k]"),
    ("eigenvectors as rows", "return U[:, idx], w[idx]", "return U[idx, :].T[:, :k], w[idx]"),
    ("token-side moment", "return X.T @ X", "return X @ X.T"),
    ("one product per iteration", "Q = orthonormal_basis(X.T @ Z)", "Q = orthonormal_basis(Z)"),
    ("one iteration short", "for _ in range(int(iters)):", "for _ in range(max(0, int(iters) - 1)):"),
    ("start block not orthonormalised", "Q = orthonormal_basis(Q0)", "Q = _f64(Q0)"),
    ("projector transposed", "R = Qb - Qa @ (Qa.T @ Qb)", "R = Qb - Qa @ (Qb.T @ Qa)"),
    ("sines from cosines",
     "R = Qb - Qa @ (Qa.T @ Qb)\n    s = np.linalg.svd(R, compute_uv=False)",
     "c = np.linalg.svd(Qa.T @ Qb, compute_uv=False)\n    s = np.sqrt(np.maximum(0.0, 1.0 - c ** 2))"),
    ("basis not normalised", "Q, _ = np.linalg.qr(_f64(Y))\n    return Q",
     "Q, Rf = np.linalg.qr(_f64(Y))\n    return Q * np.abs(np.diag(Rf))"),
    ("energy of the sum", "np.sum((X @ Qv) ** 2)", "np.sum(X @ Qv) ** 2"),
    ("cascade restarts from Q0", "        start, t = V, iters_next", "        start, t = Q0, iters_next"),
    ("cascade keeps the first count", "        start, t = V, iters_next", "        start, t = V, iters_first"),
    ("QR signs left as they come", "return Q * np.where(np.diag(R) < 0.0, -1.0, 1.0)", "return Q"),
    ("one Gram-Schmidt pass", "if np.linalg.norm(q) < DGKS_ETA * np.linalg.norm(r):", "if False:"),
    ("DGKS test inverted", "if np.linalg.norm(q) < DGKS_ETA * np.linalg.norm(r):",
     "if np.linalg.norm(q) > DGKS_ETA * np.linalg.norm(r):"),
    ("smallest residual corrected", "j = int(np.argmax(nr)) if order", "j = int(np.argmin(nr)) if order"),
    ("smaller Rayleigh quotient", "t = 0.5 * math.atan2(2.0 * s, a - b)", "t = 0.5 * math.atan2(2.0 * s, b - a)"),
    ("full angle", "t = 0.5 * math.atan2(2.0 * s, a - b)", "t = math.atan2(2.0 * s, a - b)"),
    ("cos and sin swapped", "Q[:, j] = math.cos(t) * Q[:, j] + math.sin(t) * q",
     "Q[:, j] = math.sin(t) * Q[:, j] + math.cos(t) * q"),
    ("C Q not updated", "        P[:, j] = math.cos(t) * P[:, j] + math.sin(t) * Cq\n", ""),
    ("start basis not orthonormalised", "    Q = positive_qr_basis(V)\n    P = X.T @ (X @ Q)",
     "    Q = _f64(V).copy()\n    P = X.T @ (X @ Q)"),
    ("residual without the projection", "        R = P - Q @ (Q.T @ P)\n", "        R = P.copy()\n"),
    ("rank-1 cascade restarts from Q0", "out.append(rank1_refine(X, out[-1], corrections, od)[0])",
     "out.append(rank1_refine(X, Q0, corrections, od)[0])"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_calibration_pins_catch_mutant(tmp_path, name, old, new):
    with open(ORACLE_SRC) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation site for '{name}' not unique"
    path = os.path.join(tmp_path, "calibration_mutant.py")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    spec = importlib.util.spec_from_file_location("calibration_mutant", path)
    mut = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mut)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(mut)
        except (AssertionError, ValueError, np.linalg.LinAlgError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake '{name}'"
