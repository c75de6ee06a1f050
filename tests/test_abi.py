"""The C-ABI library loads and exports every symbol include/gsi.h declares,
and its host-side argument checks answer without touching a GPU (CPU only)."""
import ctypes
import math
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    with open(os.path.join(ROOT, "include", "gsi.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gsi_[a-zA-Z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def cl():
    from gated_rank_subspace_gsi_gb300 import build, lib
    build.build()
    return lib.library()


def test_header_declares_the_boundary():
    fns = header_functions()
    for name in ("gsi_create", "gsi_forward", "gsi_precompute_M", "gsi_destroy",
                 "gsi_reserve", "gsi_device_status", "gsi_status_string",
                 "gsi_forward_host"):
        assert name in fns


def test_library_exports_every_declared_symbol(cl):
    from gated_rank_subspace_gsi_gb300 import lib
    fns = header_functions()
    for name in fns:
        assert hasattr(cl, name), f"{name} declared in gsi.h but not exported"
    assert set(lib.EXPORTS) == set(fns)


def test_status_strings(cl):
    for s in range(9):
        assert cl.gsi_status_string(s)
    assert b"RANK" in cl.gsi_status_string(8)
    assert b"UNSUPPORTED" in cl.gsi_status_string(2)


def _create(cl, W, V, M, d_out, d, k, eps):
    h = ctypes.c_void_p()
    return cl.gsi_create(W, V, M, d_out, d, k, ctypes.c_float(eps), ctypes.byref(h))


def test_host_argument_checks(cl):
    """Checks that reject before any CUDA call (fake, never dereferenced
    pointer values)."""
    A = ctypes.c_void_p(0x10000)       # 16-byte aligned fake addresses
    B = ctypes.c_void_p(0x20000)
    C = ctypes.c_void_p(0x30000)
    MIS = ctypes.c_void_p(0x10008)     # misaligned
    assert _create(cl, None, B, C, 64, 64, 16, 0.1) == 1
    assert _create(cl, MIS, B, C, 64, 64, 16, 0.1) == 1
    assert _create(cl, A, B, C, 64, 64, 16, math.nan) == 1
    assert _create(cl, A, B, C, 64, 60, 16, 0.1) == 2     # d % 8
    assert _create(cl, A, B, C, 60, 64, 16, 0.1) == 2     # d_out % 8
    assert _create(cl, A, B, C, 64, 64, 24, 0.1) == 2     # k not a supported size
    assert _create(cl, A, B, C, 64, 64, 128, 0.1) == 2    # k > d
    assert _create(cl, A, B, C, 0, 64, 16, 0.1) == 2
    h = ctypes.c_void_p()
    assert cl.gsi_create(A, B, C, 64, 64, 16, ctypes.c_float(0.1), None) == 1
    assert cl.gsi_forward(None, A, 1, B, None, None, None) == 1
    assert cl.gsi_forward_host(None, A, 1, B, None, None, None) == 1
    assert cl.gsi_precompute_M(MIS, B, C, 64, 64, 16, None) == 1
    assert cl.gsi_precompute_M(A, B, C, 64, 64, 17, None) == 2
    assert cl.gsi_reserve(None, 8) == 1
    assert cl.gsi_device_status(None, None) == 1
    assert cl.gsi_forward_launch_count(None, 1) == 0
    assert cl.gsi_set_prefetch(None, None) == 1
    assert cl.gsi_set_prefetch_group(None, None) == 1
    g = ctypes.c_void_p()
    assert cl.gsi_group_create(0, None, ctypes.byref(g)) == 1
    assert cl.gsi_group_create(5, (ctypes.c_void_p * 5)(A, B, C, A, B), ctypes.byref(g)) == 1
    assert cl.gsi_group_create(1, (ctypes.c_void_p * 1)(None), ctypes.byref(g)) == 1
    assert cl.gsi_group_create(1, (ctypes.c_void_p * 1)(A), None) == 1
    assert cl.gsi_group_forward(None, None, None, None, None, None) == 1
    assert cl.gsi_group_set_prefetch(None, None) == 1
    cl.gsi_group_destroy(None)
    cl.gsi_destroy(None)
    del h


def test_calibrate_argument_checks(cl):
    """gsi_calibrate's shape, pointer and workspace checks (fake pointers,
    never dereferenced: each case is rejected before any CUDA call)."""
    A = ctypes.c_void_p(0x10000)
    B = ctypes.c_void_p(0x20000)
    C = ctypes.c_void_p(0x30000)
    WS = ctypes.c_void_p(0x100000)     # 256-byte aligned
    size = ctypes.c_size_t()
    assert cl.gsi_calibrate_workspace_size(2048, 4096, 256, None) == 1
    assert cl.gsi_calibrate_workspace_size(2048, 4096, 256, ctypes.byref(size)) == 0
    need = size.value
    assert need > 2048 * 4096 * 2            # holds X^T at least
    assert cl.gsi_calibrate_workspace_size(2048, 4096, 512, ctypes.byref(size)) == 2   # k > 256
    assert cl.gsi_calibrate_workspace_size(2048, 4096, 48, ctypes.byref(size)) == 2    # k not allowed
    assert cl.gsi_calibrate_workspace_size(200, 4096, 256, ctypes.byref(size)) == 2    # n < k
    assert cl.gsi_calibrate_workspace_size(2048, 4100, 256, ctypes.byref(size)) == 2   # d % 8
    assert cl.gsi_calibrate_workspace_size(2044, 4096, 256, ctypes.byref(size)) == 2   # n % 8
    assert cl.gsi_calibrate_workspace_size(64, 64, 16, ctypes.byref(size)) == 0
    assert cl.gsi_calibrate(None, 2048, 4096, 256, B, 8, C, WS, need, None) == 1
    assert cl.gsi_calibrate(A, 2048, 4096, 256, B, -1, C, WS, need, None) == 1
    assert cl.gsi_calibrate(A, 2048, 4096, 256, B, 8, C, ctypes.c_void_p(0x100010), need, None) == 1
    assert cl.gsi_calibrate(ctypes.c_void_p(0x10008), 2048, 4096, 256, B, 8, C, WS, need, None) == 1
    assert cl.gsi_calibrate(A, 2048, 4096, 24, B, 8, C, WS, need, None) == 2
    assert cl.gsi_calibrate(A, 2048, 4096, 256, B, 8, C, WS, need - 1, None) == 5
    assert cl.gsi_calibrate_status(None, None) == 1
    assert cl.gsi_calibrate_launch_count(2048, 4096, 48, 8) == 0


def test_calibrate_cascade_argument_checks(cl):
    A = ctypes.c_void_p(0x10000)
    WS = ctypes.c_void_p(0x100000)
    xs = (ctypes.c_void_p * 2)(0x20000, 0x30000)
    vs_same = (ctypes.c_void_p * 2)(0x40000, 0x40000)
    vs_null = (ctypes.c_void_p * 2)(0x40000, None)
    assert cl.gsi_calibrate_cascade(None, 2, 64, 64, 16, A, 4, 2, vs_same, WS, 1 << 30, None) == 1
    assert cl.gsi_calibrate_cascade(xs, 0, 64, 64, 16, A, 4, 2, vs_same, WS, 1 << 30, None) == 1
    assert cl.gsi_calibrate_cascade(xs, 2, 64, 64, 16, A, 4, 2, vs_same, WS, 1 << 30, None) == 1
    assert cl.gsi_calibrate_cascade(xs, 2, 64, 64, 16, A, 4, 2, vs_null, WS, 1 << 30, None) == 1
    assert cl.gsi_calibrate_cascade(xs, 2, 64, 64, 16, A, 4, -1, vs_same, WS, 1 << 30, None) == 1


def test_refine_rank1_argument_checks(cl):
    """gsi_refine_rank1 and the rank-1 cascade reject bad arguments before any
    CUDA call (fake pointer values, never dereferenced)."""
    A = ctypes.c_void_p(0x10000)
    B = ctypes.c_void_p(0x20000)
    C = ctypes.c_void_p(0x30000)
    WS = ctypes.c_void_p(0x100000)
    size = ctypes.c_size_t()
    cal = ctypes.c_size_t()
    assert cl.gsi_refine_rank1_workspace_size(2048, 4096, 256, None) == 1
    assert cl.gsi_refine_rank1_workspace_size(2048, 4096, 256, ctypes.byref(size)) == 0
    assert cl.gsi_calibrate_workspace_size(2048, 4096, 256, ctypes.byref(cal)) == 0
    need = size.value
    assert need > cal.value + 2 * 256 * 4096 * 4   # V and C V in fp32 beyond the calibration's
    assert cl.gsi_refine_rank1_workspace_size(2048, 4096, 48, ctypes.byref(size)) == 2
    assert cl.gsi_refine_rank1(None, 2048, 4096, 256, B, 4, C, None, WS, need, None) == 1
    assert cl.gsi_refine_rank1(A, 2048, 4096, 256, None, 4, C, None, WS, need, None) == 1
    assert cl.gsi_refine_rank1(A, 2048, 4096, 256, B, -1, C, None, WS, need, None) == 1
    assert cl.gsi_refine_rank1(A, 2048, 4096, 256, B, 4, C, ctypes.c_void_p(0x50002), WS, need,
                               None) == 1                                   # misaligned order
    assert cl.gsi_refine_rank1(A, 2048, 4096, 256, B, 4, C, None, ctypes.c_void_p(0x100040),
                               need, None) == 1                             # workspace alignment
    assert cl.gsi_refine_rank1(A, 2048, 4096, 24, B, 4, C, None, WS, need, None) == 2
    assert cl.gsi_refine_rank1(A, 2048, 4096, 256, B, 4, C, None, WS, cal.value, None) == 5
    xs = (ctypes.c_void_p * 2)(0x20000, 0x30000)
    vs = (ctypes.c_void_p * 2)(0x40000, 0x60000)
    vs_same = (ctypes.c_void_p * 2)(0x40000, 0x40000)
    assert cl.gsi_calibrate_cascade_rank1(None, 2, 2048, 4096, 256, A, 8, 4, vs, None, WS, need,
                                          None) == 1
    assert cl.gsi_calibrate_cascade_rank1(xs, 0, 2048, 4096, 256, A, 8, 4, vs, None, WS, need,
                                          None) == 1
    assert cl.gsi_calibrate_cascade_rank1(xs, 2, 2048, 4096, 256, A, 8, 4, vs_same, None, WS,
                                          need, None) == 1
    assert cl.gsi_calibrate_cascade_rank1(xs, 2, 2048, 4096, 256, A, 8, -1, vs, None, WS, need,
                                          None) == 1
    assert cl.gsi_calibrate_cascade_rank1(xs, 2, 2048, 4096, 256, A, 8, 4, vs, None, WS,
                                          cal.value, None) == 5             # needs the rank-1 size
    assert cl.gsi_refine_rank1_launch_count(2048, 4096, 48, 4) == 0
