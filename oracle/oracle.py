"""ctypes marshalling for the fp64 GSI oracle (``gsi_oracle.c``).

Test infrastructure only; see the package docstring.  No arithmetic of the
method lives here: each method converts numpy arrays to contiguous fp64 (or
uint16 bf16 bit patterns) and calls the C routine that follows the page.

``OracleLib(path)`` wraps one compiled copy of the oracle.  The module-level
functions use the default copy built from ``gsi_oracle.c``; the mutation
tests load deliberately broken copies through the same class.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC_PATH = os.path.join(_HERE, "gsi_oracle.c")
LIB_PATH = os.path.join(_HERE, "libgsi_oracle.so")

_lock = threading.Lock()
_default = None


def build(src: str = SRC_PATH, out: str = LIB_PATH, force: bool = False) -> str:
    """Compile the oracle C source into a shared library (gcc, OpenMP)."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fopenmp",
           "-shared", "-fPIC", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _u16(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"expected bf16 bit patterns as uint16, got {a.dtype}")
    return np.ascontiguousarray(a)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class OracleLib:
    """One loaded copy of the compiled oracle."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        lib.gsi_oracle_bf16_decode.argtypes = [P, P, I64]
        lib.gsi_oracle_bf16_decode.restype = None
        lib.gsi_oracle_bf16_encode.argtypes = [P, P, I64]
        lib.gsi_oracle_bf16_encode.restype = None
        lib.gsi_oracle_precompute_M.argtypes = [P, P, I64, I64, I64, P]
        lib.gsi_oracle_precompute_M.restype = None
        lib.gsi_oracle_forward.argtypes = [P, P, P, I64, I64, I64,
                                           ctypes.c_double, P, I64, P, P, P,
                                           P, P]
        lib.gsi_oracle_forward.restype = ctypes.c_int
        lib.gsi_oracle_spectral_norm.argtypes = [P, I64, I64, ctypes.c_uint64,
                                                 ctypes.c_int, ctypes.c_double]
        lib.gsi_oracle_spectral_norm.restype = ctypes.c_double
        lib.gsi_oracle_num_threads.argtypes = []
        lib.gsi_oracle_num_threads.restype = ctypes.c_int
        self.lib = lib
        self.path = path

    # -- bf16 storage -------------------------------------------------------
    def bf16_decode(self, bits) -> np.ndarray:
        """Exact fp64 values of bf16 bit patterns (uint16 array, any shape)."""
        bits = _u16(bits)
        out = np.empty(bits.shape, dtype=np.float64)
        self.lib.gsi_oracle_bf16_decode(_ptr(bits), _ptr(out), bits.size)
        return out

    def bf16_encode(self, values) -> np.ndarray:
        """fp64 -> bf16 bit patterns, one round-to-nearest-even."""
        v = _f64(values)
        out = np.empty(v.shape, dtype=np.uint16)
        self.lib.gsi_oracle_bf16_encode(_ptr(v), _ptr(out), v.size)
        return out

    # -- the cached image [GSI 2.1, eq. 2] ---------------------------------
    def precompute_M(self, W, V) -> np.ndarray:
        """M = W V_k in exact fp64 sums. W: d_out x d, V: d x k."""
        W = _f64(W)
        V = _f64(V)
        d_out, d = W.shape
        d2, k = V.shape
        if d2 != d:
            raise ValueError("W and V_k disagree on d")
        M = np.empty((d_out, k), dtype=np.float64)
        self.lib.gsi_oracle_precompute_M(_ptr(W), _ptr(V), d_out, d, k, _ptr(M))
        return M

    def precompute_M_bf16(self, W_bits, V_bits) -> np.ndarray:
        """The cached image as stored: bf16(W V_k), from bf16 W and V_k."""
        return self.bf16_encode(self.precompute_M(self.bf16_decode(W_bits),
                                                  self.bf16_decode(V_bits)))

    # -- the gated map [GSI 2.1 - 2.2] --------------------------------------
    def forward(self, W, V, M, eps: float, X, want_g: bool = False,
                want_r: bool = False) -> dict:
        """The gated map on T tokens (rows of X) in fp64.

        W: d_out x d, V: d x k, M: d_out x k, X: T x d (real values).  ``eps``
        is compared as given.  Returns dict(y=T x d_out, rho=T, gate=T uint8
        with 1 = slow path, and optionally g=T x k, r=T x d).  W and M may
        hold any subset of output rows; y then holds the same columns.
        """
        V = _f64(V)
        X = _f64(X)
        if X.ndim == 1:
            X = X[None, :]
        T, d = X.shape
        d2, k = V.shape
        if d2 != d:
            raise ValueError("V_k and x disagree on d")
        W = _f64(W) if W is not None else np.zeros((0, d))
        M = _f64(M) if M is not None else np.zeros((0, k))
        d_out = W.shape[0]
        if W.shape != (d_out, d) or M.shape != (d_out, k):
            raise ValueError("W / M shapes do not match")
        Y = np.empty((T, d_out), dtype=np.float64)
        rho = np.empty(T, dtype=np.float64)
        gate = np.empty(T, dtype=np.uint8)
        G = np.empty((T, k), dtype=np.float64) if want_g else None
        R = np.empty((T, d), dtype=np.float64) if want_r else None
        rc = self.lib.gsi_oracle_forward(
            _ptr(W), _ptr(V), _ptr(M), d_out, d, k, float(eps), _ptr(X), T,
            _ptr(Y), _ptr(rho), _ptr(gate), _ptr(G), _ptr(R))
        if rc != 0:
            raise ValueError("gsi_oracle_forward rejected its arguments")
        out = dict(y=Y, rho=rho, gate=gate)
        if G is not None:
            out["g"] = G
        if R is not None:
            out["r"] = R
        return out

    def forward_bf16(self, W_bits, V_bits, M_bits, eps32: float, X_bits,
                     **kw) -> dict:
        """``forward`` on stored bf16 operands, decoded exactly to fp64.

        ``eps32`` is the fp32 threshold the GPU receives; it is compared as
        the fp64 value of that fp32 number.
        """
        eps = float(np.float32(eps32))
        dec = self.bf16_decode
        return self.forward(dec(W_bits) if W_bits is not None else None,
                            dec(V_bits),
                            dec(M_bits) if M_bits is not None else None,
                            eps, dec(X_bits), **kw)

    # -- Theorem 4's ||W||_2 ------------------------------------------------
    def spectral_norm(self, A, seed: int = 12345, max_iter: int = 5000,
                      tol: float = 1e-13) -> float:
        """Largest singular value of A by power iteration on A^T A.

        The estimate never exceeds the true value (a Rayleigh quotient);
        callers that need an upper bound add a margin.
        """
        A = _f64(A)
        if A.ndim != 2:
            raise ValueError("expected a matrix")
        m, n = A.shape
        s = self.lib.gsi_oracle_spectral_norm(_ptr(A), m, n, seed, max_iter, tol)
        if s < 0:
            raise ValueError("spectral_norm failed")
        return float(s)

    def num_threads(self) -> int:
        """OpenMP threads the oracle uses."""
        return int(self.lib.gsi_oracle_num_threads())


def default() -> OracleLib:
    """The oracle built from gsi_oracle.c (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = OracleLib(build())
        return _default


def bf16_decode(bits):
    return default().bf16_decode(bits)


def bf16_encode(values):
    return default().bf16_encode(values)


def precompute_M(W, V):
    return default().precompute_M(W, V)


def precompute_M_bf16(W_bits, V_bits):
    return default().precompute_M_bf16(W_bits, V_bits)


def forward(W, V, M, eps, X, **kw):
    return default().forward(W, V, M, eps, X, **kw)


def forward_bf16(W_bits, V_bits, M_bits, eps32, X_bits, **kw):
    return default().forward_bf16(W_bits, V_bits, M_bits, eps32, X_bits, **kw)


def spectral_norm(A, **kw):
    return default().spectral_norm(A, **kw)


def num_threads():
    return default().num_threads()
