"""fp64 reference for calibrating the rank-k basis V_k.

TEST INFRASTRUCTURE ONLY, under the same rules as the rest of ``oracle/``:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU legs of ``bench.py``
use it; the CUDA library never imports or calls it and shares no code with
it.  Plain numpy in fp64; library primitives (matmul, Householder QR, a
symmetric eigensolver, an SVD) serve as single steps.

What it follows.  The page "Technical summary: Gated Subspace Inference for
transformer acceleration", section 2.3 ("calibration"), says the basis is
computed once from a single forward pass over a representative calibration
sequence, and gives no algorithm.  The reading taken here: V_k spans the
top-k eigenvectors of the uncentred second moment C = X^T X of the
calibration activations X (n tokens x d).  That subspace minimises
sum_t ||x_t - V V^T x_t||^2 over rank-k orthonormal V, i.e. the residual
r of section 2.1 (eq. 1) summed over the calibration tokens, which is what
the gate of section 2.2 measures.  Uncentred, because the gate projects x
itself, not x minus a mean.

  top_k_subspace(X, k)            the definition, by a symmetric eigensolver
  subspace_iteration(X, Q0, t)    the algorithm the GPU runs: block power
                                  iteration Q <- orth(X^T (X Q)), t times,
                                  from the given start block Q0
  cascade(Xs, Q0, t0, t1)         the depth cascade of section 2.3: layer 0
                                  from Q0 with t0 iterations, layer l + 1
                                  started from layer l's basis with t1
  rank1_refine(X, V, c)           the cascade's refinement in the pages' form:
                                  c rank-1 corrections of the start basis,
                                  each new direction re-orthogonalised by DGKS
  cascade_rank1(Xs, Q0, t0, c)    the depth cascade with that refinement
  principal_sines(A, B)           the comparison between two subspaces

Only span(V_k) matters to the gated map: replacing V_k by V_k R for an
orthogonal k x k R leaves r and rho unchanged and M g = W V_k R R^T V_k^T x
unchanged.  So the functions return orthonormal bases of subspaces, and
results are compared through principal angles, never entry by entry.

rank1_refine is the one function here whose result depends on the basis
inside the span, not on the span alone: it corrects one basis vector at a
time.  Its start basis is therefore fixed exactly (the positive-diagonal QR
factor of the given block, which is unique).

Every function is pinned in tests/test_oracle_calibration.py (closed forms
for planted spectra, the exact two-dimensional iteration, invariance of the
span under a change of start basis, convergence at the rate set by the
eigenvalue gap, exact recovery of a planted rotated eigenvector by one
rank-1 correction, orthogonality restored by the second Gram-Schmidt pass),
and the same file plants mistakes in a copy of this source to check that the
pins catch them.
"""
from __future__ import annotations

import math

import numpy as np


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


def orthonormal_basis(Y) -> np.ndarray:
    """Orthonormal basis (d x k) of span(Y) for a full-column-rank d x k Y:
    the Q factor of a Householder QR."""
    Q, _ = np.linalg.qr(_f64(Y))
    return Q


def second_moment(X) -> np.ndarray:
    """C = X^T X for n tokens x d (the calibration activations' uncentred
    second moment, unnormalised: the 1/n factor changes no eigenvector)."""
    X = _f64(X)
    return X.T @ X


def top_k_subspace(X, k: int):
    """(V, lam): the k eigenvectors of C = X^T X with the largest eigenvalues
    (d x k, orthonormal columns) and those eigenvalues, descending."""
    w, U = np.linalg.eigh(second_moment(X))
    idx = np.argsort(w)[::-1][:k]
    return U[:, idx], w[idx]


def subspace_iteration(X, Q0, iters: int) -> np.ndarray:
    """Block power iteration on C = X^T X from the start block Q0 (d x k):
    Q_0 = orth(Q0); Q_{t+1} = orth(X^T (X Q_t)); returns Q_iters.

    C is applied as two products with X (n x k, then d x k) and never formed.
    span(Q_t) = span(C^t Q0).  When lambda_k > lambda_{k+1} and V_k^T Q0 is
    nonsingular (true for a generic Q0), the tangents of the principal angles
    to the top-k eigenspace shrink by lambda_{k+1} / lambda_k per iteration.
    """
    X = _f64(X)
    Q = orthonormal_basis(Q0)
    for _ in range(int(iters)):
        Z = X @ Q
        Q = orthonormal_basis(X.T @ Z)
    return Q


def cascade(Xs, Q0, iters_first: int, iters_next: int):
    """Depth cascade (section 2.3: a layer's basis starts from the previous
    layer's).  Xs: the calibration tokens of consecutive layers.  Layer 0 is
    subspace_iteration(Xs[0], Q0, iters_first); layer l + 1 is
    subspace_iteration(Xs[l + 1], V_l, iters_next) with V_l the basis just
    computed for layer l.  Returns the list of bases."""
    out = []
    start, t = Q0, iters_first
    for X in Xs:
        V = subspace_iteration(X, start, t)
        out.append(V)
        start, t = V, iters_next
    return out


def positive_qr_basis(V) -> np.ndarray:
    """The Q factor of V = Q R with R upper triangular and a positive
    diagonal (unique for a full-column-rank V): Householder QR, then every
    column whose diagonal entry of R came out negative flips sign."""
    Q, R = np.linalg.qr(_f64(V))
    return Q * np.where(np.diag(R) < 0.0, -1.0, 1.0)


DGKS_ETA = 1.0 / math.sqrt(2.0)


def dgks_orthogonalize(B, r):
    """(q, passes): r minus its component in span(B), B with orthonormal
    columns, by classical Gram-Schmidt with the reorthogonalisation test of
    Daniel, Gragg, Kaufman and Stewart: one projection q = r - B (B^T r); if
    that left less than 1/sqrt(2) of the norm of r, the projection is applied
    once more to q.  q is not normalised; passes is 1 or 2."""
    B = _f64(B)
    r = _f64(r)
    q = r - B @ (B.T @ r)
    if np.linalg.norm(q) < DGKS_ETA * np.linalg.norm(r):
        q = q - B @ (B.T @ q)
        return q, 2
    return q, 1


def rank1_refine(X, V, corrections: int, order=None):
    """(Q, chosen, norms): the start basis V (d x k) refined by `corrections`
    rank-1 corrections for the second moment C = X^T X of the tokens X.

    Section 2.3 of the page starts layer l + 1's basis from layer l's and
    refines it with a few rank-1 corrections, DGKS updates, instead of a full
    decomposition per layer; it gives no further steps.  Reading taken:

      Q = the positive-diagonal QR factor of V;  P = C Q
      for each correction:
        residuals R = P - Q (Q^T P): column i is (I - Q Q^T) C q_i
        j = the column with the largest residual norm (the first such)
        q = R[:, j] re-orthogonalised against Q by DGKS, normalised
        the plane spanned by q_j and q: C restricted to it is
          [[a, s], [s, b]],  a = q_j^T C q_j,  b = q^T C q,  s = q_j^T C q
        q_j <- cos(t) q_j + sin(t) q with t = atan2(2 s, a - b) / 2, the
        unit vector of the plane with the largest Rayleigh quotient
        P[:, j] <- cos(t) P[:, j] + sin(t) C q

    Each correction changes one column, Q <- Q + (q_j' - q_j) e_j^T, a rank-1
    update that keeps the columns orthonormal, and never lowers
    trace(Q^T C Q).  A residual that vanishes after re-orthogonalisation
    (q = 0: span(Q) is invariant under C) leaves the basis as it is.

    order: optional column indices, one per correction, used instead of the
    largest-residual choice (to replay another implementation's choices).
    chosen: the column corrected at each step; norms: (corrections x k) the
    residual norms each choice was made from."""
    X = _f64(X)
    Q = positive_qr_basis(V)
    P = X.T @ (X @ Q)
    chosen, norms = [], []
    for step in range(int(corrections)):
        R = P - Q @ (Q.T @ P)
        nr = np.linalg.norm(R, axis=0)
        j = int(np.argmax(nr)) if order is None else int(order[step])
        chosen.append(j)
        norms.append(nr)
        q, _ = dgks_orthogonalize(Q, R[:, j])
        nq = np.linalg.norm(q)
        if not nq > 0.0:
            continue
        q = q / nq
        Cq = X.T @ (X @ q)
        a = Q[:, j] @ P[:, j]
        b = q @ Cq
        s = Q[:, j] @ Cq
        t = 0.5 * math.atan2(2.0 * s, a - b)
        Q[:, j] = math.cos(t) * Q[:, j] + math.sin(t) * q
        P[:, j] = math.cos(t) * P[:, j] + math.sin(t) * Cq
    return Q, chosen, np.array(norms).reshape(len(norms), Q.shape[1])


def cascade_rank1(Xs, Q0, iters_first: int, corrections: int, orders=None):
    """The depth cascade in the page's form: layer 0 is
    subspace_iteration(Xs[0], Q0, iters_first); layer l + 1 is
    rank1_refine(Xs[l + 1], V_l, corrections) with V_l the basis just
    computed for layer l.  orders: optional per-layer column orders for
    rank1_refine (entry 0 unused).  Returns the list of bases."""
    out = [subspace_iteration(Xs[0], Q0, iters_first)]
    for li, X in enumerate(Xs[1:], start=1):
        od = None if orders is None else orders[li]
        out.append(rank1_refine(X, out[-1], corrections, od)[0])
    return out


def principal_sines(A, B) -> np.ndarray:
    """Sines of the principal angles between span(A) and span(B) (both d x k,
    full column rank), descending.  Taken as the singular values of
    (I - Qa Qa^T) Qb, which keeps full relative accuracy for small angles."""
    Qa = orthonormal_basis(A)
    Qb = orthonormal_basis(B)
    R = Qb - Qa @ (Qa.T @ Qb)
    s = np.linalg.svd(R, compute_uv=False)
    return np.sort(np.clip(s, 0.0, 1.0))[::-1]


def captured_energy(X, V) -> float:
    """Fraction of the calibration tokens' total energy inside span(V):
    ||X Qv||_F^2 / ||X||_F^2 with Qv an orthonormal basis of span(V)."""
    X = _f64(X)
    Qv = orthonormal_basis(V)
    return float(np.sum((X @ Qv) ** 2) / np.sum(X ** 2))
