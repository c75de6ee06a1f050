"""GB300 (sm_103a) implementation of the Gated Subspace Inference linear map.

For each token x: g = V_k^T x, rho = ||x - V_k g|| / ||x||, and y = M g
(M = W V_k, cached) when rho < eps, else y = W x -- as defined on the page
"Technical summary: Gated Subspace Inference for transformer acceleration",
sections 2.1-2.2.  The work runs in hand-written CUDA kernels behind the C
ABI of include/gsi.h (libgsi.so); ``lib`` is its thin ctypes binding.

Importing the package does not load the library; ``lib.library()`` (or any
call) does, building it with nvcc if needed, and raises if it cannot.
"""
from . import build  # noqa: F401

__all__ = ["build", "lib"]


def __getattr__(name):
    if name == "lib":
        import importlib
        return importlib.import_module(__name__ + ".lib")
    raise AttributeError(name)
