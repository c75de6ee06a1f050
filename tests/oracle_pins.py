"""Pins of the fp64 oracle to facts fixed by the page and by mathematics.

Each ``pin_*`` function takes an ``oracle.OracleLib`` and raises
AssertionError when that oracle disagrees with something other than itself:
hand-derived closed forms (tests/golden), exact rational arithmetic, library
routines in the special cases where the method reduces to them, and
Theorem 4's bound.  ``tests/test_oracle_pins.py`` runs them on the oracle;
``tests/test_oracle_mutants.py`` runs them on copies of the oracle with
planted mistakes and requires that each mistake is caught.

Page cited: "Technical summary: Gated Subspace Inference for transformer
acceleration" [GSI], sections 2.1 (eqs. 1-2) and 2.2 (gate, Theorem 4).
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# --------------------------------------------------------------------------
# fixtures
# --------------------------------------------------------------------------

def load_closed_form():
    """Parse tests/golden/closed_form_d8.txt."""
    W, U, cases = [], [], []
    with open(os.path.join(GOLDEN, "closed_form_d8.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            tag, rest = line.split(None, 1)
            if tag == "W":
                W.append([int(v) for v in rest.split()])
            elif tag in ("U1", "U2"):
                U.append([int(v) for v in rest.split()])
            elif tag == "CASE":
                name, xs, eps, rho2, gate, ys = [p.strip() for p in rest.split("|")]
                p, q = rho2.split("/")
                cases.append(dict(
                    name=name, x=[int(v) for v in xs.split()],
                    eps=math.inf if eps == "inf" else float(Fraction(eps)),
                    eps_exact=None if eps == "inf" else Fraction(eps),
                    rho2=Fraction(int(p), int(q)), gate=int(gate),
                    y=[int(v) for v in ys.split()]))
    return np.array(W, dtype=np.float64), [np.array(u, dtype=np.float64) for u in U], cases


def householder(u: np.ndarray) -> np.ndarray:
    return np.eye(len(u)) - 2.0 * np.outer(u, u) / float(u @ u)


def _frac_householder(u):
    n = len(u)
    uu = sum(Fraction(v) ** 2 for v in u)
    return [[Fraction(int(i == j)) - 2 * Fraction(u[i]) * Fraction(u[j]) / uu
             for j in range(n)] for i in range(n)]


def _frac_matmul(A, B):
    return [[sum(A[i][t] * B[t][j] for t in range(len(B))) for j in range(len(B[0]))]
            for i in range(len(A))]


# --------------------------------------------------------------------------
# bf16 storage
# --------------------------------------------------------------------------

def pin_bf16(orc):
    """bf16 decode is exact, encode is one round-to-nearest-even."""
    # hand-picked patterns: 1.0, -2.0, smallest subnormal, largest finite, +inf
    bits = np.array([0x3F80, 0xC000, 0x0001, 0x7F7F, 0x7F80, 0x0000, 0x8000], np.uint16)
    want = [1.0, -2.0, 2.0 ** -133, 255.0 * 2.0 ** 120, math.inf, 0.0, -0.0]
    got = orc.bf16_decode(bits)
    for g, w in zip(got, want):
        assert g == w, (g, w)
    # ties to even and just-above-half cases around 1.0 (quantum 2^-7)
    vals = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -8 + 2 ** -40,
                     -(1 + 2 ** -8), 2 ** -134, 3 * 2 ** -134, 255.5 * 2.0 ** 120])
    want_bits = [0x3F80, 0x3F82, 0x3F81, 0xBF80, 0x0000, 0x0002, 0x7F80]
    got_bits = orc.bf16_encode(vals)
    assert list(got_bits) == want_bits, [hex(b) for b in got_bits]
    # round trip of every finite pattern
    allb = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    dec = orc.bf16_decode(allb)
    fin = np.isfinite(dec)
    assert np.array_equal(orc.bf16_encode(dec[fin]), allb[fin])
    # brute force: nearest finite bf16 to random doubles, ties to even
    rng = np.random.default_rng(7)
    pos = np.unique(dec[fin & (dec >= 0)])
    v = rng.standard_normal(4000) * np.exp(rng.uniform(-30, 30, 4000))
    enc = orc.bf16_decode(orc.bf16_encode(v))
    for val, e in zip(v, enc):
        a = abs(val)
        i = np.searchsorted(pos, a)
        lo, hi = pos[max(i - 1, 0)], pos[min(i, len(pos) - 1)]
        best = lo if (a - lo) < (hi - a) else hi
        assert abs(e) == best and (e == 0 or np.sign(e) == np.sign(val)), (val, e, best)


# --------------------------------------------------------------------------
# closed forms (tests/golden/closed_form_d8.txt)
# --------------------------------------------------------------------------

def pin_closed_form(orc):
    """Hand-derived d = 8, k = 2 cases, plain and rotated [GSI 2.1-2.2]."""
    W, (u1, u2), cases = load_closed_form()
    V = np.zeros((8, 2))
    V[0, 0] = V[1, 1] = 1.0
    M = W[:, :2].copy()
    Q = householder(u1) @ householder(u2)
    assert np.array_equal(Q @ Q.T, np.eye(8))        # exact: entries k/4
    for rotated in (False, True):
        Vr = Q @ V if rotated else V
        Wr = W @ Q.T if rotated else W
        for c in cases:
            x = np.array(c["x"], dtype=np.float64)
            xr = Q @ x if rotated else x
            out = orc.forward(Wr, Vr, M, c["eps"], xr[None, :], want_g=True)
            tag = (c["name"], rotated)
            assert int(out["gate"][0]) == c["gate"], tag
            assert abs(out["rho"][0] ** 2 - float(c["rho2"])) <= 1e-14, tag
            assert np.array_equal(out["y"][0], np.array(c["y"], dtype=np.float64)), tag
            assert np.array_equal(out["g"][0], x[:2]), tag


def pin_special_values(orc):
    """NaN input takes the slow path and propagates; x = 0 gives rho = 0."""
    W, _, _ = load_closed_form()
    V = np.zeros((8, 2))
    V[0, 0] = V[1, 1] = 1.0
    M = W[:, :2].copy()
    x = np.zeros((2, 8))
    x[0, 3] = np.nan
    out = orc.forward(W, V, M, 0.5, x)
    assert out["gate"][0] == 1 and np.isnan(out["rho"][0]) and np.isnan(out["y"][0]).all()
    assert out["gate"][1] == 0 and out["rho"][1] == 0.0 and (out["y"][1] == 0).all()


# --------------------------------------------------------------------------
# exact rational brute force
# --------------------------------------------------------------------------

def pin_rational(orc, n_cases: int = 40):
    """Exact rationals on d = 8, k = 2 with a dyadic rotated basis.

    V = the first two columns of Q = H(u1) H(u2) (entries multiples of 1/4,
    exactly orthonormal); the gate is decided exactly by comparing
    rho^2 = r.r / x.x with eps^2, no square root needed.
    """
    rng = np.random.default_rng(2024)
    _, (u1, u2), _ = load_closed_form()
    Qf = _frac_matmul(_frac_householder([int(v) for v in u1]),
                      _frac_householder([int(v) for v in u2]))
    Vf = [[Qf[i][0], Qf[i][1]] for i in range(8)]
    V = np.array([[float(v) for v in row] for row in Vf])
    for case in range(n_cases):
        W = rng.integers(-4, 5, size=(3, 8))
        Mf = [[sum(Fraction(int(W[o][i])) * Vf[i][j] for i in range(8)) for j in range(2)]
              for o in range(3)]
        M = np.array([[float(v) for v in row] for row in Mf])
        x = rng.integers(-6, 7, size=8)
        if case % 3 == 0:                 # mostly in span(V): fast tokens
            x = (V @ rng.integers(-6, 7, size=2) * 4).round() + (rng.random(8) < 0.2)
        xf = [Fraction(int(v)) for v in x]
        gf = [sum(Vf[i][j] * xf[i] for i in range(8)) for j in range(2)]
        rf = [xf[i] - sum(Vf[i][j] * gf[j] for j in range(2)) for i in range(8)]
        xx = sum(v * v for v in xf)
        rr = sum(v * v for v in rf)
        rho2 = rr / xx if xx else Fraction(0)
        for eps in (0.125, 0.25, 0.5, 0.75):
            ef = Fraction(eps)
            slow = not (rho2 < ef * ef)
            if xx and abs(float(rho2 - ef * ef)) < 1e-12:
                continue
            out = orc.forward(W.astype(np.float64), V, M, eps,
                              x.astype(np.float64)[None, :], want_g=True)
            assert int(out["gate"][0]) == int(slow), (case, eps)
            yf = ([sum(Fraction(int(W[o][i])) * xf[i] for i in range(8)) for o in range(3)]
                  if slow else
                  [sum(Mf[o][j] * gf[j] for j in range(2)) for o in range(3)])
            for o in range(3):
                assert abs(out["y"][0][o] - float(yf[o])) <= 1e-12 * (1 + abs(float(yf[o])))
            for j in range(2):
                assert abs(out["g"][0][j] - float(gf[j])) <= 1e-13
            assert abs(out["rho"][0] - math.sqrt(float(rho2))) <= 1e-14


# --------------------------------------------------------------------------
# special cases reducing to library routines
# --------------------------------------------------------------------------

def _random_problem(seed, d=48, k=8, d_out=20, T=12):
    rng = np.random.default_rng(seed)
    Q, R = np.linalg.qr(rng.standard_normal((d, k)))
    W = rng.standard_normal((d_out, d)) / math.sqrt(d)
    M = W @ Q
    # tokens with a spread of residual ratios
    a = rng.standard_normal((T, k)) @ Q.T
    b = rng.standard_normal((T, d))
    s = np.linspace(0.0, 0.6, T)
    X = a + s[:, None] * b
    return W, Q, M, X


def pin_library_cases(orc):
    """eps = 0 -> all slow, y = W x; eps = inf -> all fast, y = M V^T x;
    with an exactly orthonormal basis rho is the least-squares residual ratio;
    M = W V matches a library matmul; V = I (k = d) gives rho = 0, y = W x."""
    for seed in range(3):
        W, Q, M, X = _random_problem(seed)
        tol = 1e-12
        out0 = orc.forward(W, Q, M, 0.0, X)
        assert (out0["gate"] == 1).all()
        ref0 = X @ W.T
        assert np.abs(out0["y"] - ref0).max() <= tol * np.abs(ref0).max()
        outi = orc.forward(W, Q, M, math.inf, X, want_g=True, want_r=True)
        assert (outi["gate"] == 0).all()
        G = X @ Q
        assert np.abs(outi["g"] - G).max() <= tol * np.abs(G).max()
        refi = G @ M.T
        assert np.abs(outi["y"] - refi).max() <= tol * np.abs(refi).max()
        # least squares: min_z ||x - Q z|| / ||x||
        z, *_ = np.linalg.lstsq(Q, X.T, rcond=None)
        rho_ls = np.linalg.norm(X.T - Q @ z, axis=0) / np.linalg.norm(X, axis=1)
        assert np.abs(outi["rho"] - rho_ls).max() <= 1e-12
        # the gate follows rho against eps, strictly below = fast
        eps = float(np.median(rho_ls))
        outm = orc.forward(W, Q, M, eps, X)
        assert np.array_equal(outm["gate"], (~(outm["rho"] < eps)).astype(np.uint8))
        assert 0 < outm["gate"].sum() < len(outm["gate"])
        # precompute_M against a library matmul
        Mo = orc.precompute_M(W, Q)
        assert np.abs(Mo - W @ Q).max() <= 1e-13 * np.abs(M).max()
    # V = I, k = d: every token is in the subspace
    rng = np.random.default_rng(11)
    d = 16
    W = rng.standard_normal((5, d))
    X = rng.standard_normal((6, d))
    out = orc.forward(W, np.eye(d), W, 1e-9, X)
    assert (out["gate"] == 0).all() and np.abs(out["rho"]).max() <= 1e-15
    assert np.abs(out["y"] - X @ W.T).max() <= 1e-12 * np.abs(X @ W.T).max()


def pin_scaling(orc):
    """x -> 2^s x leaves rho and the gate unchanged and scales y exactly."""
    W, Q, M, X = _random_problem(5)
    eps = 0.3
    base = orc.forward(W, Q, M, eps, X)
    for s in (-3, 5):
        out = orc.forward(W, Q, M, eps, X * 2.0 ** s)
        assert np.array_equal(out["gate"], base["gate"])
        assert np.abs(out["rho"] - base["rho"]).max() <= 1e-15
        assert np.array_equal(out["y"], base["y"] * 2.0 ** s)


# --------------------------------------------------------------------------
# eq. 1, the basis, and Theorem 4
# --------------------------------------------------------------------------

def pin_spectral_norm(orc):
    """Power iteration against the SVD's largest singular value."""
    rng = np.random.default_rng(3)
    for shape in ((30, 17), (17, 30), (64, 64)):
        A = rng.standard_normal(shape)
        s = orc.spectral_norm(A)
        ref = np.linalg.norm(A, 2)
        assert abs(s - ref) <= 1e-9 * ref, (shape, s, ref)
    # a symmetric matrix with a negative dominant eigenvalue
    D = np.diag([-5.0, 2.0, 1.0])
    Qr, _ = np.linalg.qr(rng.standard_normal((3, 3)))
    assert abs(orc.spectral_norm(Qr @ D @ Qr.T) - 5.0) <= 1e-9


def pin_decomposition_and_theorem4(orc, inputs):
    """On generated bf16 inputs (gsi_inputs.LinearInputs):
    (a) x = V g + r to round-off, V^T r = -(V^T V - I) g, and
        ||V^T V - I||_2 small for the stored bf16 basis;
    (d) every fast token obeys ||M_exact g - W x|| <= ||W||_2 rho ||x||
        < ||W||_2 eps ||x|| (Theorem 4, section 2.2), and with the stored
        bf16 M within the extra ||M - M_exact||_F ||g||."""
    W = orc.bf16_decode(np.asarray(inputs.W))
    V = orc.bf16_decode(inputs.V_bits)
    X = orc.bf16_decode(inputs.X_bits)
    eps = float(np.float32(inputs.spec.eps))
    M_exact = orc.precompute_M(W, V)
    M = orc.bf16_decode(orc.bf16_encode(M_exact))
    out = orc.forward(W, V, M, eps, X, want_g=True, want_r=True)
    G, R = out["g"], out["r"]
    # (a)
    assert np.abs(X - (G @ V.T + R)).max() <= 1e-12 * np.abs(X).max()
    Gm = V.T @ V
    E = Gm - np.eye(V.shape[1])
    assert np.abs(R @ V + G @ E).max() <= 1e-10 * np.abs(G).max()
    e_norm = orc.spectral_norm(E)
    assert 1e-6 < e_norm <= 1e-2, e_norm
    # (d)
    w_norm = orc.spectral_norm(W) * (1 + 1e-6)
    nx = np.linalg.norm(X, axis=1)
    fast = out["gate"] == 0
    assert fast.any()
    err_exact = np.linalg.norm(G @ M_exact.T - X @ W.T, axis=1)
    assert (err_exact[fast] <= w_norm * out["rho"][fast] * nx[fast] * (1 + 1e-9)).all()
    assert (err_exact[fast] < w_norm * eps * nx[fast]).all()
    err_m = np.linalg.norm(M - M_exact)
    err_bf = np.linalg.norm(G @ M.T - X @ W.T, axis=1)
    bound = w_norm * out["rho"] * nx + err_m * np.linalg.norm(G, axis=1)
    assert (err_bf[fast] <= bound[fast] * (1 + 1e-9)).all()
    # the stored y is the bf16-M fast path
    assert np.abs(out["y"][fast] - (G @ M.T)[fast]).max() <= 1e-12 * np.abs(out["y"]).max()
    return dict(e_norm=e_norm, w_norm=w_norm)


def pin_theorem4_tight(orc):
    """The bound is attained when r lies along W's top right singular vector,
    so an oracle ||W||_2 that is too small or too large shows up."""
    rng = np.random.default_rng(9)
    d, k, d_out = 40, 6, 24
    W = rng.standard_normal((d_out, d))
    Q, _ = np.linalg.qr(rng.standard_normal((d, k)))
    _, svals, vt = np.linalg.svd(W)
    v1 = vt[0] - Q @ (Q.T @ vt[0])                       # top direction, made orthogonal to V
    v1 /= np.linalg.norm(v1)
    x = Q @ rng.standard_normal(k) + 0.05 * v1 * 3.0
    M = W @ Q
    out = orc.forward(W, Q, M, math.inf, x[None, :], want_g=True)
    err = np.linalg.norm(out["g"][0] @ M.T - W @ x)
    bound = orc.spectral_norm(W) * out["rho"][0] * np.linalg.norm(x)
    assert err <= bound * (1 + 1e-9)
    # W r with r = c v1: ||W r|| >= (component of v1 on the top singular
    # vector) * sigma_1 ||r||, close to the bound
    assert err >= 0.5 * bound


ALL_PINS = ("pin_bf16", "pin_closed_form", "pin_special_values", "pin_rational",
            "pin_library_cases", "pin_scaling", "pin_spectral_norm",
            "pin_theorem4_tight")
