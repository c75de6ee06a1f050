"""ctypes binding of libgsi.so, the C ABI in include/gsi.h.

Argument marshalling only: every step of the gated map runs in the library's
CUDA kernels.  Functions keep the C names.  Tensors are torch tensors (device
memory for everything except the *_host variant); PyTorch supplies memory and
streams and nothing else.  If libgsi.so is missing it is built with nvcc; if
that is impossible the import fails loudly: there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

GSI_OK = 0
GSI_ERR_INVALID_ARG = 1
GSI_ERR_UNSUPPORTED_SHAPE = 2
GSI_ERR_NOMEM = 3
GSI_ERR_CUDA = 4
GSI_ERR_WORKSPACE = 5
GSI_ERR_TIMEOUT = 6
GSI_ERR_LAUNCH = 7
GSI_ERR_RANK = 8

# every function declared in include/gsi.h
EXPORTS = ("gsi_create", "gsi_forward", "gsi_forward_host", "gsi_precompute_M",
           "gsi_reserve", "gsi_device_status", "gsi_destroy", "gsi_status_string",
           "gsi_forward_launch_count", "gsi_forward_noalloc", "gsi_set_prefetch",
           "gsi_set_prefetch_group", "gsi_group_create", "gsi_group_forward",
           "gsi_group_forward_host",
           "gsi_group_set_prefetch", "gsi_group_destroy", "gsi_calibrate_workspace_size",
           "gsi_calibrate", "gsi_calibrate_status", "gsi_calibrate_launch_count",
           "gsi_calibrate_timed", "gsi_calibrate_cascade", "gsi_refine_rank1_workspace_size",
           "gsi_refine_rank1", "gsi_calibrate_cascade_rank1", "gsi_refine_rank1_launch_count")

_lock = threading.Lock()
_lib = None


class GsiError(RuntimeError):
    """A call into libgsi returned a status other than GSI_OK."""

    def __init__(self, status: int, what: str):
        self.status = int(status)
        msg = _load().gsi_status_string(self.status).decode()
        super().__init__(f"{what}: {msg}")


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB_PATH
        if not os.path.exists(path):
            _build.build()
        lib = ctypes.CDLL(path)
        P, I64 = ctypes.c_void_p, ctypes.c_int64
        lib.gsi_create.argtypes = [P, P, P, I64, I64, I64, ctypes.c_float, ctypes.POINTER(P)]
        lib.gsi_create.restype = ctypes.c_int
        lib.gsi_forward.argtypes = [P, P, I64, P, P, P, P]
        lib.gsi_forward.restype = ctypes.c_int
        lib.gsi_forward_host.argtypes = [P, P, I64, P, P, P, P]
        lib.gsi_forward_host.restype = ctypes.c_int
        lib.gsi_precompute_M.argtypes = [P, P, P, I64, I64, I64, P]
        lib.gsi_precompute_M.restype = ctypes.c_int
        lib.gsi_reserve.argtypes = [P, I64]
        lib.gsi_reserve.restype = ctypes.c_int
        lib.gsi_device_status.argtypes = [P, P]
        lib.gsi_device_status.restype = ctypes.c_int
        lib.gsi_destroy.argtypes = [P]
        lib.gsi_destroy.restype = None
        lib.gsi_status_string.argtypes = [ctypes.c_int]
        lib.gsi_status_string.restype = ctypes.c_char_p
        lib.gsi_forward_launch_count.argtypes = [P, I64]
        lib.gsi_forward_launch_count.restype = ctypes.c_int
        lib.gsi_forward_noalloc.argtypes = [P, P, P, I64, I64, I64, ctypes.c_float, P, P, P, P, P]
        lib.gsi_forward_noalloc.restype = ctypes.c_int
        lib.gsi_set_prefetch.argtypes = [P, P]
        lib.gsi_set_prefetch.restype = ctypes.c_int
        lib.gsi_set_prefetch_group.argtypes = [P, P]
        lib.gsi_set_prefetch_group.restype = ctypes.c_int
        lib.gsi_group_create.argtypes = [ctypes.c_int, P, ctypes.POINTER(P)]
        lib.gsi_group_create.restype = ctypes.c_int
        lib.gsi_group_forward.argtypes = [P, P, P, P, P, P]
        lib.gsi_group_forward.restype = ctypes.c_int
        lib.gsi_group_forward_host.argtypes = [P, P, P, P, P, P]
        lib.gsi_group_forward_host.restype = ctypes.c_int
        lib.gsi_group_set_prefetch.argtypes = [P, P]
        lib.gsi_group_set_prefetch.restype = ctypes.c_int
        lib.gsi_group_destroy.argtypes = [P]
        lib.gsi_group_destroy.restype = None
        lib.gsi_calibrate_workspace_size.argtypes = [I64, I64, I64, ctypes.POINTER(ctypes.c_size_t)]
        lib.gsi_calibrate_workspace_size.restype = ctypes.c_int
        lib.gsi_calibrate.argtypes = [P, I64, I64, I64, P, ctypes.c_int, P, P, ctypes.c_size_t, P]
        lib.gsi_calibrate.restype = ctypes.c_int
        lib.gsi_calibrate_timed.argtypes = [P, I64, I64, I64, P, ctypes.c_int, P, P, ctypes.c_size_t,
                                            P, P, P, ctypes.c_int, ctypes.POINTER(ctypes.c_int)]
        lib.gsi_calibrate_timed.restype = ctypes.c_int
        lib.gsi_calibrate_cascade.argtypes = [P, ctypes.c_int, I64, I64, I64, P, ctypes.c_int,
                                              ctypes.c_int, P, P, ctypes.c_size_t, P]
        lib.gsi_calibrate_cascade.restype = ctypes.c_int
        lib.gsi_calibrate_status.argtypes = [P, P]
        lib.gsi_calibrate_status.restype = ctypes.c_int
        lib.gsi_calibrate_launch_count.argtypes = [I64, I64, I64, ctypes.c_int]
        lib.gsi_calibrate_launch_count.restype = ctypes.c_int
        lib.gsi_refine_rank1_workspace_size.argtypes = [I64, I64, I64,
                                                        ctypes.POINTER(ctypes.c_size_t)]
        lib.gsi_refine_rank1_workspace_size.restype = ctypes.c_int
        lib.gsi_refine_rank1.argtypes = [P, I64, I64, I64, P, ctypes.c_int, P, P, P,
                                         ctypes.c_size_t, P]
        lib.gsi_refine_rank1.restype = ctypes.c_int
        lib.gsi_calibrate_cascade_rank1.argtypes = [P, ctypes.c_int, I64, I64, I64, P,
                                                    ctypes.c_int, ctypes.c_int, P, P, P,
                                                    ctypes.c_size_t, P]
        lib.gsi_calibrate_cascade_rank1.restype = ctypes.c_int
        lib.gsi_refine_rank1_launch_count.argtypes = [I64, I64, I64, ctypes.c_int]
        lib.gsi_refine_rank1_launch_count.restype = ctypes.c_int
        _lib = lib
        return lib


def library():
    """The loaded ctypes library (built on first use if missing)."""
    return _load()


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _check(st: int, what: str):
    if st != GSI_OK:
        raise GsiError(st, what)


def gsi_status_string(status: int) -> str:
    return _load().gsi_status_string(int(status)).decode()


def gsi_create(W, V_k, M, eps: float) -> ctypes.c_void_p:
    """Handle for one gated linear.  W (d_out x d), V_k (d x k), M (d_out x k):
    bf16 CUDA tensors, borrowed (keep them alive and unchanged)."""
    d_out, d = W.shape
    d2, k = V_k.shape
    if d2 != d or tuple(M.shape) != (d_out, k):
        raise ValueError("W, V_k and M shapes disagree")
    h = ctypes.c_void_p()
    _check(_load().gsi_create(_ptr(W), _ptr(V_k), _ptr(M), d_out, d, k, float(eps),
                              ctypes.byref(h)), "gsi_create")
    return h


def gsi_forward(h, x, y, gate=None, rho=None, stream=None, T=None):
    """y (T x d_out fp32), gate (T uint8) and rho (T fp32) of the gated map on
    x (T x d bf16), all CUDA tensors; asynchronous on `stream`."""
    T = x.shape[0] if T is None else T
    _check(_load().gsi_forward(h, _ptr(x), T, _ptr(y), _ptr(gate), _ptr(rho), _stream(stream)),
           "gsi_forward")


def gsi_forward_host(h, x_host, y_host, gate_host=None, rho_host=None, stream=None, T=None):
    """gsi_forward on host (CPU, ideally pinned) tensors; copies are queued on
    `stream`, which the caller synchronises before reading the outputs."""
    T = x_host.shape[0] if T is None else T
    _check(_load().gsi_forward_host(h, _ptr(x_host), T, _ptr(y_host), _ptr(gate_host),
                                    _ptr(rho_host), _stream(stream)), "gsi_forward_host")


def gsi_precompute_M(W, V_k, M, stream=None):
    """M = bf16(W V_k) on the GPU (fp32 accumulation)."""
    d_out, d = W.shape
    _, k = V_k.shape
    _check(_load().gsi_precompute_M(_ptr(W), _ptr(V_k), _ptr(M), d_out, d, k, _stream(stream)),
           "gsi_precompute_M")


def gsi_reserve(h, max_T: int):
    _check(_load().gsi_reserve(h, int(max_T)), "gsi_reserve")


def gsi_device_status(h, stream=None) -> int:
    """Synchronise the stream, return (and clear) the handle's device status."""
    return int(_load().gsi_device_status(h, _stream(stream)))


def gsi_destroy(h):
    if h is not None:
        _load().gsi_destroy(h)


def gsi_set_prefetch(h, next_h):
    """Make each one-token call on h prefetch next_h's operands into L2
    (next_h None removes the link)."""
    _check(_load().gsi_set_prefetch(h, next_h), "gsi_set_prefetch")


def gsi_set_prefetch_group(h, group):
    """Make each one-token call on h prefetch every member of `group` into L2
    (None removes the link)."""
    _check(_load().gsi_set_prefetch_group(h, group), "gsi_set_prefetch_group")


def _ptr_array(items):
    arr = (ctypes.c_void_p * len(items))()
    for i, t in enumerate(items):
        arr[i] = _ptr(t)
    return arr


def gsi_group_create(handles) -> ctypes.c_void_p:
    """One launch for several independent one-token calls (a group of handles)."""
    arr = (ctypes.c_void_p * len(handles))(*[h.value if isinstance(h, ctypes.c_void_p) else h
                                             for h in handles])
    g = ctypes.c_void_p()
    _check(_load().gsi_group_create(len(handles), arr, ctypes.byref(g)), "gsi_group_create")
    return g


def gsi_group_forward(g, xs, ys, gates=None, rhos=None, stream=None):
    """One token through every member of group g (lists of device tensors)."""
    _check(_load().gsi_group_forward(g, _ptr_array(xs), _ptr_array(ys),
                                     _ptr_array(gates) if gates is not None else None,
                                     _ptr_array(rhos) if rhos is not None else None,
                                     _stream(stream)), "gsi_group_forward")


def gsi_group_forward_host(g, xs, ys, gates=None, rhos=None, stream=None):
    """gsi_group_forward on host buffers (lists of CPU tensors, page-locked
    for the copy-free path)."""
    _check(_load().gsi_group_forward_host(g, _ptr_array(xs), _ptr_array(ys),
                                          _ptr_array(gates) if gates is not None else None,
                                          _ptr_array(rhos) if rhos is not None else None,
                                          _stream(stream)), "gsi_group_forward_host")


def gsi_group_set_prefetch(g, next_h):
    _check(_load().gsi_group_set_prefetch(g, next_h), "gsi_group_set_prefetch")


def gsi_group_destroy(g):
    if g is not None:
        _load().gsi_group_destroy(g)


def gsi_forward_launch_count(h, T: int) -> int:
    return int(_load().gsi_forward_launch_count(h, int(T)))


def gsi_forward_noalloc(W, V_k, M, eps: float, x, y, gate=None, rho=None, stream=None):
    """One token of the gated map with no handle and no allocation (for
    callers whose device memory is owned by another allocator); its scratch is
    a fixed array inside the library, shared by all calls on a device."""
    d_out, d = W.shape
    _, k = V_k.shape
    _check(_load().gsi_forward_noalloc(_ptr(W), _ptr(V_k), _ptr(M), d_out, d, k, float(eps),
                                       _ptr(x), _ptr(y), _ptr(gate), _ptr(rho), _stream(stream)),
           "gsi_forward_noalloc")


class GatedLinear:
    """One gated linear (W, V_k, M, eps) bound to a libgsi handle.

    Holds references to the borrowed tensors so they outlive the handle.
    """

    def __init__(self, W, V_k, M, eps: float, max_T: int = 0):
        import torch
        for name, t in (("W", W), ("V_k", V_k), ("M", M)):
            if not (t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous()):
                raise TypeError(f"{name} must be a contiguous bf16 CUDA tensor")
        self.W, self.V_k, self.M, self.eps = W, V_k, M, float(eps)
        self.d_out, self.d = W.shape
        self.k = V_k.shape[1]
        self.h = gsi_create(W, V_k, M, eps)
        if max_T > 0:
            gsi_reserve(self.h, max_T)

    def forward(self, x, y=None, gate=None, rho=None, stream=None):
        import torch
        T = x.shape[0]
        if y is None:
            y = torch.empty((T, self.d_out), dtype=torch.float32, device=x.device)
        gsi_forward(self.h, x, y, gate, rho, stream)
        return y

    __call__ = forward

    def status(self, stream=None) -> int:
        return gsi_device_status(self.h, stream)

    def close(self):
        if self.h is not None:
            gsi_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ---- calibration of V_k ---------------------------------------------------


def gsi_calibrate_workspace_size(n: int, d: int, k: int) -> int:
    """Device scratch bytes gsi_calibrate needs for n tokens of width d, rank k."""
    out = ctypes.c_size_t()
    _check(_load().gsi_calibrate_workspace_size(int(n), int(d), int(k), ctypes.byref(out)),
           "gsi_calibrate_workspace_size")
    return int(out.value)


def gsi_calibrate(X, Q0, iters: int, V_k, workspace, stream=None):
    """V_k (d x k bf16) = orthonormal basis of span((X^T X)^iters Q0), by block
    power iteration on the GPU.  X (n x d), Q0 (d x k): bf16 CUDA tensors;
    workspace: a CUDA tensor of at least gsi_calibrate_workspace_size bytes."""
    n, d = X.shape
    d2, k = Q0.shape
    if d2 != d or tuple(V_k.shape) != (d, k):
        raise ValueError("X, Q0 and V_k shapes disagree")
    nbytes = workspace.numel() * workspace.element_size()
    _check(_load().gsi_calibrate(_ptr(X), n, d, k, _ptr(Q0), int(iters), _ptr(V_k),
                                 _ptr(workspace), nbytes, _stream(stream)), "gsi_calibrate")


def gsi_calibrate_status(workspace, stream=None) -> int:
    """Synchronise the stream; the device-side status of the last gsi_calibrate."""
    return int(_load().gsi_calibrate_status(_ptr(workspace), _stream(stream)))


def gsi_calibrate_launch_count(n: int, d: int, k: int, iters: int) -> int:
    return int(_load().gsi_calibrate_launch_count(int(n), int(d), int(k), int(iters)))


CAL_KINDS = ("transpose", "tensor-core GEMM", "split-K sum", "Gram matrix", "Cholesky",
             "forward substitution")


def gsi_calibrate_timed(X, Q0, iters: int, V_k, workspace, stream=None, max_launches: int = 4096):
    """gsi_calibrate with an event pair around every launch; returns a list of
    (kind name, ms) in launch order (synchronises the stream)."""
    n, d = X.shape
    _, k = Q0.shape
    ms = (ctypes.c_float * max_launches)()
    kinds = (ctypes.c_int * max_launches)()
    cnt = ctypes.c_int()
    nbytes = workspace.numel() * workspace.element_size()
    _check(_load().gsi_calibrate_timed(_ptr(X), n, d, k, _ptr(Q0), int(iters), _ptr(V_k),
                                       _ptr(workspace), nbytes, _stream(stream), ms, kinds,
                                       max_launches, ctypes.byref(cnt)), "gsi_calibrate_timed")
    return [(CAL_KINDS[kinds[i]], float(ms[i])) for i in range(cnt.value)]


def gsi_calibrate_cascade(Xs, Q0, iters_first: int, iters_next: int, Vs, workspace, stream=None):
    """Depth cascade: V_0 from Q0 with iters_first iterations on Xs[0]; V_l
    from V_{l-1} with iters_next iterations on Xs[l].  Xs: list of n x d bf16
    CUDA tensors; Vs: list of d x k bf16 CUDA tensors (outputs)."""
    if len(Xs) != len(Vs) or not Xs:
        raise ValueError("one output basis per layer")
    n, d = Xs[0].shape
    _, k = Q0.shape
    xa = _ptr_array(Xs)
    va = _ptr_array(Vs)
    nbytes = workspace.numel() * workspace.element_size()
    _check(_load().gsi_calibrate_cascade(xa, len(Xs), n, d, k, _ptr(Q0), int(iters_first),
                                         int(iters_next), va, _ptr(workspace), nbytes,
                                         _stream(stream)), "gsi_calibrate_cascade")


def gsi_refine_rank1_workspace_size(n: int, d: int, k: int) -> int:
    """Device scratch bytes gsi_refine_rank1 (and the rank-1 cascade) need."""
    out = ctypes.c_size_t()
    _check(_load().gsi_refine_rank1_workspace_size(int(n), int(d), int(k), ctypes.byref(out)),
           "gsi_refine_rank1_workspace_size")
    return int(out.value)


def gsi_refine_rank1(X, V_in, corrections: int, V_out, workspace, order=None, stream=None):
    """`corrections` rank-1 DGKS corrections of the start basis V_in (d x k
    bf16) for the tokens X (n x d bf16), into V_out; order (int32 CUDA tensor
    of `corrections` entries, optional) receives the corrected columns."""
    n, d = X.shape
    _, k = V_in.shape
    nbytes = workspace.numel() * workspace.element_size()
    _check(_load().gsi_refine_rank1(_ptr(X), n, d, k, _ptr(V_in), int(corrections), _ptr(V_out),
                                    _ptr(order), _ptr(workspace), nbytes, _stream(stream)),
           "gsi_refine_rank1")


def gsi_calibrate_cascade_rank1(Xs, Q0, iters_first: int, corrections: int, Vs, workspace,
                                order=None, stream=None):
    """Depth cascade in rank-1 form: V_0 = gsi_calibrate(Xs[0], Q0,
    iters_first); V_l = gsi_refine_rank1(Xs[l], V_{l-1}, corrections).  order:
    optional int32 CUDA tensor of (layers - 1) * corrections entries."""
    if len(Xs) != len(Vs) or not Xs:
        raise ValueError("one output basis per layer")
    n, d = Xs[0].shape
    _, k = Q0.shape
    xa = _ptr_array(Xs)
    va = _ptr_array(Vs)
    nbytes = workspace.numel() * workspace.element_size()
    _check(_load().gsi_calibrate_cascade_rank1(xa, len(Xs), n, d, k, _ptr(Q0), int(iters_first),
                                               int(corrections), va, _ptr(order),
                                               _ptr(workspace), nbytes, _stream(stream)),
           "gsi_calibrate_cascade_rank1")


def gsi_refine_rank1_launch_count(n: int, d: int, k: int, corrections: int) -> int:
    return int(_load().gsi_refine_rank1_launch_count(int(n), int(d), int(k), int(corrections)))
