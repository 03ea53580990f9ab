"""gs_bin_and_sort_static against gs_bin_and_sort.

The static variant serves callers that cannot allocate device memory (an
application allocator that owns the GPU, a frame loop that must not stall on
an allocation, a plug-in that only gets its inputs and outputs): its scratch
is an array inside the library.  Its results must be the existing entry
point's, bit for bit (integer work), on consecutive calls that share that
array.  This file is collected last so that a failure here comes after every
other test has run."""
import ctypes as C

import numpy as np
import pytest
import torch

import scenes
from parity_util import f32_cams

pytestmark = pytest.mark.gpu


def _gs():
    import __graft_entry__
    __graft_entry__.build()
    import gaussian_splatting_differentiable_gs_gb300 as gs
    return gs


def _projected(gs, params, cams):
    n = params.shape[1]
    splats = torch.empty((n * len(cams), 12), dtype=torch.float32, device="cuda")
    gs.gs_project(torch.from_numpy(params).cuda(), cams, splats)
    return splats


def _reference(gs, n, V, splats, W, H, cap):
    T = gs.tiles_per_view(W, H)
    ws = torch.zeros(gs.gs_bin_workspace_bytes(n * V, cap), dtype=torch.uint8, device="cuda")
    keys = torch.empty(cap, dtype=torch.int64, device="cuda")
    vals = torch.empty(cap, dtype=torch.int32, device="cuda")
    ranges = torch.empty((V * T, 2), dtype=torch.int64, device="cuda")
    st, I = gs.gs_bin_and_sort(n, V, splats, W, H, ws, cap, keys, vals, ranges)
    assert st == gs.GS_OK
    return I, keys[:I].cpu(), vals[:I].cpu(), ranges.cpu()


def _static(gs, n, V, splats, W, H, cap):
    """Calls the C entry point directly (ctypes)."""
    L = gs.lib()
    f = L.gs_bin_and_sort_static
    f.argtypes = [C.c_int64, C.c_int32, C.c_void_p, C.c_void_p, C.c_int32, C.c_int32, C.c_int64,
                  C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p]
    f.restype = C.c_int
    T = gs.tiles_per_view(W, H)
    keys = torch.full((cap,), -1, dtype=torch.int64, device="cuda")
    vals = torch.full((cap,), -1, dtype=torch.int32, device="cuda")
    ranges = torch.full((V * T, 2), -3, dtype=torch.int64, device="cuda")
    out = C.c_int64(0)
    st = f(n, V, splats.data_ptr(), None, W, H, cap, keys.data_ptr(), vals.data_ptr(),
           ranges.data_ptr(), C.byref(out), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    I = int(out.value)
    return st, I, keys[:I].cpu(), vals[:I].cpu(), ranges.cpu()


def _cases():
    cfg = scenes.make("tiny_2k_256")
    a = (cfg["params"], f32_cams(cfg["cams"]))
    params = scenes.uniform_scene(3000, 1.5, (2.0, 8.0), 77)
    cams = f32_cams([scenes.camera(np.eye(3), np.zeros(3), 150, 150, 100, 60, 200, 120),
                     scenes.look_at((0.6, -0.3, -0.4), (0, 0, 5), (0, -1, 0), 160, 150, 200, 120)])
    return [a, (params, cams)]


def test_static_workspace_variant_matches_existing_entry_point():
    gs = _gs()
    cap = 200_000
    for params, cams in _cases() + _cases()[:1]:  # three calls in a row, shared scratch
        n, V = params.shape[1], len(cams)
        W, H = cams[0]["width"], cams[0]["height"]
        splats = _projected(gs, params, cams)
        I, keys, vals, ranges = _reference(gs, n, V, splats, W, H, cap)
        st, I2, keys2, vals2, ranges2 = _static(gs, n, V, splats, W, H, cap)
        assert st == gs.GS_OK
        assert I2 == I > 0
        assert torch.equal(keys2, keys)
        assert torch.equal(vals2, vals)
        assert torch.equal(ranges2, ranges)


def test_static_workspace_variant_rejects_oversize():
    gs = _gs()
    L = gs.lib()
    f = L.gs_bin_and_sort_static
    f.restype = C.c_int
    out = C.c_int64(0)
    # too many rows (65537 x 1 view) and too much capacity: rejected before any work
    assert f(C.c_int64(65537), C.c_int32(1), None, None, C.c_int32(16), C.c_int32(16),
             C.c_int64(16), None, None, None, C.byref(out), None) == gs.GS_ERR_INVALID_ARG
    assert f(C.c_int64(10), C.c_int32(1), None, None, C.c_int32(16), C.c_int32(16),
             C.c_int64(1048577), None, None, None, C.byref(out), None) == gs.GS_ERR_INVALID_ARG
