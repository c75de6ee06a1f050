"""Helpers shared by the GPU parity tests: device transfer of bf16 bit
patterns, the oracle comparison with the gate band rule, and the setup of one
gated linear on both sides (each side computes its own cached image M).
"""
from __future__ import annotations

import math

import numpy as np

RHO_BAND = 1e-4        # |rho_ref - eps| <= band: the GPU's rho decides the branch
Y_REL_TOL = 2e-3       # max|y_gpu - y_ref| <= 2e-3 * max|y_ref| (per token row)
RHO_TOL = 1e-4         # |rho_gpu - rho_ref| for finite rho, or else ...
RHO2_TOL = 5e-6        # ... |rho_gpu^2 - rho_ref^2|: the GPU forms rho^2 as
                       # (||x||^2 - g.g + g^T E g) / ||x||^2 from fp32 sums over d
                       # and k terms (g accumulated on the tensor cores for T > 1),
                       # whose worst-case error is a few 1e-6 of ||x||^2; near
                       # rho = 0 that bounds the error of rho^2, not rho; near any
                       # eps >= 0.05 it moves rho by <= 5e-5 (inside the 1e-4
                       # band); gates are checked exactly regardless


def to_dev(bits: np.ndarray):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).cuda()


def to_bits(t) -> np.ndarray:
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


class GpuLinear:
    """W, V_k on the device, M from gsi_precompute_M, and a libgsi handle;
    the oracle side keeps W, V_k bits and its own M = bf16(W V_k)."""

    def __init__(self, lib, orc, W_bits, V_bits, eps: float, max_T: int = 0, W_dev=None,
                 M_rows=None):
        import torch
        self.lib, self.orc = lib, orc
        self.eps = float(np.float32(eps))
        self.W_dev = W_dev if W_dev is not None else to_dev(W_bits)
        self.V_bits = V_bits
        self.V_dev = to_dev(V_bits)
        d_out, d = self.W_dev.shape
        k = V_bits.shape[1]
        self.d_out, self.d, self.k = d_out, d, k
        self.M_dev = torch.empty((d_out, k), dtype=torch.bfloat16, device="cuda")
        lib.gsi_precompute_M(self.W_dev, self.V_dev, self.M_dev)
        torch.cuda.synchronize()
        self.h = lib.gsi_create(self.W_dev, self.V_dev, self.M_dev, eps)
        if max_T:
            lib.gsi_reserve(self.h, max_T)
        self._W_bits = W_bits
        self._M_ref = None
        self.M_rows = M_rows

    def W_bits(self) -> np.ndarray:
        if self._W_bits is None:
            self._W_bits = to_bits(self.W_dev)
        return self._W_bits

    def W_rows(self, rows) -> np.ndarray:
        if self._W_bits is not None:
            return self._W_bits[rows]
        import torch
        idx = torch.as_tensor(np.asarray(rows), device=self.W_dev.device)
        return to_bits(self.W_dev.index_select(0, idx))

    def M_ref_rows(self, rows) -> np.ndarray:
        """The oracle's own cached image bf16(W V_k) on the given rows."""
        return self.orc.precompute_M_bf16(self.W_rows(rows), self.V_bits)

    def forward(self, X_bits: np.ndarray, stream=None, one_by_one: bool = False):
        """Run the GPU map; returns numpy y, gate, rho."""
        import torch
        T = X_bits.shape[0]
        x = to_dev(X_bits)
        y = torch.full((T, self.d_out), float("nan"), dtype=torch.float32, device="cuda")
        gate = torch.full((T,), 7, dtype=torch.uint8, device="cuda")
        rho = torch.full((T,), -1.0, dtype=torch.float32, device="cuda")
        if one_by_one:
            for t in range(T):
                self.lib.gsi_forward(self.h, x[t:t + 1], y[t:t + 1], gate[t:t + 1],
                                     rho[t:t + 1], stream)
        else:
            self.lib.gsi_forward(self.h, x, y, gate, rho, stream)
        st = self.lib.gsi_device_status(self.h, stream)
        assert st == 0, self.lib.gsi_status_string(st)
        return y.cpu().numpy(), gate.cpu().numpy(), rho.cpu().numpy()

    def close(self):
        self.lib.gsi_destroy(self.h)
        self.h = None


def check_against_oracle(orc, lin: GpuLinear, X_bits, y_gpu, gate_gpu, rho_gpu, rows=None,
                         tokens=None, what=""):
    """Compare GPU outputs with the oracle on the same bf16 inputs.

    Gates must agree exactly for every token with |rho_ref - eps| > 1e-4; in
    the band the GPU's rho picks the branch and the oracle recomputes y on
    that branch.  y is compared per token row on `rows` (all if None):
    max|y_gpu - y_ref| <= 2e-3 max|y_ref|.  Returns a small report dict.
    """
    T = X_bits.shape[0]
    tokens = np.arange(T) if tokens is None else np.asarray(tokens)
    rows = np.arange(lin.d_out) if rows is None else np.asarray(rows)
    Wr = lin.W_rows(rows)
    Mr = lin.M_ref_rows(rows)
    Xs = X_bits[tokens]
    ref = orc.forward_bf16(Wr, lin.V_bits, Mr, lin.eps, Xs)
    y_ref, rho_ref, gate_ref = ref["y"], ref["rho"], ref["gate"].astype(np.int64)
    g_gpu = gate_gpu[tokens].astype(np.int64)
    r_gpu = rho_gpu[tokens]
    band = np.abs(rho_ref - lin.eps) <= RHO_BAND
    # gates: exact outside the band, GPU rho decides inside
    nan_ref = np.isnan(rho_ref)
    assert np.array_equal(np.isnan(r_gpu), nan_ref), f"{what}: NaN rho positions differ"
    out = ~band
    bad = np.nonzero((g_gpu != gate_ref) & out)[0]
    assert bad.size == 0, (f"{what}: gate mismatch at tokens {tokens[bad][:10]} "
                           f"rho_ref={rho_ref[bad][:5]} rho_gpu={r_gpu[bad][:5]} eps={lin.eps}")
    fin = ~nan_ref
    if fin.any():
        drho = np.abs(r_gpu[fin] - rho_ref[fin])
        drho2 = np.abs(r_gpu[fin].astype(np.float64) ** 2 - rho_ref[fin] ** 2)
        bad = (drho > RHO_TOL) & (drho2 > RHO2_TOL)
        assert not bad.any(), (f"{what}: rho differs by {drho[bad].max()} "
                               f"(rho^2 by {drho2[bad].max()})")
    # band tokens: re-decide with the GPU rho and recompute the reference
    for i in np.nonzero(band)[0]:
        want = 0 if r_gpu[i] < lin.eps else 1
        assert g_gpu[i] == want, f"{what}: band token {tokens[i]} gate does not follow its rho"
        if want != gate_ref[i]:
            e = 0.0 if want == 1 else math.inf
            y_ref[i] = orc.forward_bf16(Wr, lin.V_bits, Mr, e, Xs[i:i + 1])["y"][0]
    if len(rows) == 0:
        return dict(worst_rel=0.0, n_band=int(band.sum()), n_slow=int(g_gpu.sum()))
    yg = y_gpu[tokens][:, rows]
    worst = 0.0
    for i in range(len(tokens)):
        yr = y_ref[i]
        if np.isnan(yr).any() or np.isinf(yr).any():
            assert np.array_equal(np.isnan(yg[i]), np.isnan(yr)), f"{what}: NaN pattern differs"
            continue
        scale = np.abs(yr).max()
        err = np.abs(yg[i] - yr).max()
        if scale == 0:
            assert err == 0, f"{what}: token {tokens[i]} expected exact zero"
            continue
        rel = err / scale
        worst = max(worst, rel)
        assert rel <= Y_REL_TOL, f"{what}: token {tokens[i]} y rel err {rel:.3e}"
    # whole-tensor form of the bound too
    finite = np.isfinite(y_ref).all(axis=1)
    if finite.any():
        tot = np.abs(yg[finite] - y_ref[finite]).max() / max(np.abs(y_ref[finite]).max(), 1e-300)
        assert tot <= Y_REL_TOL
    return dict(worst_rel=worst, n_band=int(band.sum()), n_slow=int(g_gpu.sum()))
