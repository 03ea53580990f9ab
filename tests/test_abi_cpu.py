"""CPU checks of the C-ABI library: it loads, exports every function that
include/gs.h declares, and its host-side helpers and argument validation
behave as documented.  No call here reaches the GPU."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def gslib():
    import __graft_entry__
    __graft_entry__.build()
    import gaussian_splatting_differentiable_gs_gb300 as gs
    return gs


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"^[a-z_0-9 \*]*?\b(gs_[a-z0-9_]+)\s*\(", src, re.M))
    return names


def test_every_declared_symbol_is_exported(gslib):
    names = _declared()
    assert {"gs_project", "gs_bin_and_sort", "gs_rasterize_fwd", "gs_rasterize_bwd",
            "gs_project_bwd", "gs_adam_step"} <= names
    lib = C.CDLL(gslib.LIB_PATH)
    for name in sorted(names):
        assert hasattr(lib, name), name


def test_status_strings_and_version(gslib):
    assert gslib.version() >= 100
    assert gslib.status_string(0) == "ok"
    assert "capacity" in gslib.status_string(2)
    assert gslib.status_string(99) == "unknown status"
    lib = C.CDLL(gslib.LIB_PATH)
    lib.gs_status_str.restype = C.c_char_p
    lib.gs_status_str.argtypes = [C.c_int]
    for code in (0, 1, 2, 3, 4, 5, 99):
        assert lib.gs_status_str(code).decode() == gslib.status_string(code)


def test_rasterize_workspace_bytes(gslib):
    """768 B per batch slot (32 quarters x 192 bits): one slot per 192 list
    entries of capacity, plus one per (view, tile), plus one."""
    f = gslib.gs_rasterize_workspace_bytes
    assert f(1, 256, 256, 0) == 768 * (0 + 256 + 1)
    assert f(1, 256, 256, 1) == 768 * (1 + 256 + 1)
    assert f(4, 1920, 1080, 22_768_982) == 768 * (-(-22_768_982 // 192) + 4 * 120 * 68 + 1)
    assert f(0, 256, 256, 10) == 0 and f(1, 256, 256, -1) == 0


def test_key_bits_and_workspace(gslib):
    # 256x256, 1 view: 256 tiles -> 8 bits of tile index + 32 depth bits
    assert gslib.gs_key_bits(1, 256, 256) == 40
    assert gslib.gs_key_bits(1, 1024, 768) == 44
    assert gslib.gs_key_bits(4, 1920, 1080) == 47
    assert gslib.gs_key_bits(8, 1920, 1080) == 48
    assert gslib.gs_key_bits(1, 3840, 2160) == 47
    assert gslib.gs_key_bits(1, 16, 16) == 33
    # one capacity-sized key buffer (8 B) and two per-row words (16 B)
    a = gslib.gs_bin_workspace_bytes(1024, 10_240)
    b = gslib.gs_bin_workspace_bytes(1024, 20_480)
    c = gslib.gs_bin_workspace_bytes(2048, 20_480)
    assert a > 8 * 10_240 + 16 * 1024 and b - a >= 8 * 10_240 and c - b >= 16 * 1024
    assert gslib.gs_bin_workspace_bytes(-1, 0) == 0


def test_invalid_arguments_return_before_any_launch(gslib):
    L = gslib.lib()
    cams = gslib.cameras_struct([dict(R=[1, 0, 0, 0, 1, 0, 0, 0, 1], t=[0, 0, 0], fx=1, fy=1, cx=0,
                                      cy=0, width=16, height=16, near_z=0.01, far_z=1e9)])
    cp = C.cast(cams, C.c_void_p)
    assert L.gs_project(10, None, cp, 0, None, None, None) == gslib.GS_ERR_INVALID_ARG  # 0 views
    assert L.gs_project(10, None, cp, 1, None, None, None) == gslib.GS_ERR_INVALID_ARG  # NULL
    assert L.gs_project(-1, None, cp, 1, None, None, None) == gslib.GS_ERR_INVALID_ARG
    assert L.gs_project(0, None, cp, 1, None, None, None) == gslib.GS_OK                # empty
    # a tile-count array not 4-byte aligned is rejected before anything runs
    cbuf = C.create_string_buffer(256)
    a16 = C.c_void_p((C.addressof(cbuf) + 15) & ~15)
    odd = C.c_void_p(a16.value + 2)
    assert L.gs_project(10, a16, cp, 1, a16, odd, None) == gslib.GS_ERR_INVALID_ARG
    bad = gslib.cameras_struct([dict(R=[1, 0, 0, 0, 1, 0, 0, 0, 1], t=[0, 0, 0], fx=1, fy=1, cx=0,
                                     cy=0, width=0, height=16, near_z=0.01, far_z=1e9)])
    assert L.gs_project(0, None, C.cast(bad, C.c_void_p), 1, None, None,
                        None) == gslib.GS_ERR_INVALID_ARG
    assert L.gs_adam_step(5, None, None, None, None, 0, 1e-3, 0.9, 0.999, 1e-8, None,
                          None) == gslib.GS_ERR_INVALID_ARG                        # step 0
    assert L.gs_adam_step(5, None, None, None, None, 1, 1e-3, 0.9, 0.999, 1e-8, None,
                          None) == gslib.GS_ERR_INVALID_ARG                        # NULL
    out = C.c_int64(0)
    assert L.gs_bin_and_sort(10, 1, None, None, 16, 16, None, 0, 0, None, None, None,
                             C.byref(out), None) == gslib.GS_ERR_INVALID_ARG       # no workspace
    ws = C.create_string_buffer(64)
    assert L.gs_bin_and_sort(1 << 29, 8, None, None, 16, 16, ws, 64, 0, None, None, None,
                             C.byref(out), None) == gslib.GS_ERR_INVALID_ARG       # 2^32 rows
    assert L.gs_bin_and_sort(1, 1, None, None, 16 * 65536, 16, ws, 64, 0, None, None, None,
                             C.byref(out), None) == gslib.GS_ERR_INVALID_ARG       # 65536 tiles wide
    assert L.gs_rasterize_fwd(10, 1, None, 16, 16, None, None, None, None, None, None, None,
                              None) == gslib.GS_ERR_INVALID_ARG
    assert L.gs_rasterize_bwd(10, 17, None, None, 16, 16, None, None, None, None, None, None,
                              None, None, None) == gslib.GS_ERR_INVALID_ARG
    assert L.gs_rasterize_fused(10, 1, None, None, 16, 16, None, None, None, None, None, None,
                                None, None, None, None, None, C.c_size_t(0),
                                None) == gslib.GS_ERR_INVALID_ARG
    # a workspace not 16-byte aligned is rejected before anything runs
    buf = C.create_string_buffer(64)
    dummy = C.c_float * 3
    mis = C.c_void_p(((C.addressof(buf) + 15) & ~15) + 4)  # 4 mod 16, inside the buffer
    assert L.gs_rasterize_fused(0, 1, None, None, 16, 16, None, buf, None, dummy(0, 0, 0), buf,
                                buf, buf, buf, buf, None, mis, C.c_size_t(32),
                                None) == gslib.GS_ERR_INVALID_ARG
    assert L.gs_rasterize_fused(0, 1, None, odd, 16, 16, None, buf, None, dummy(0, 0, 0), buf,
                                buf, buf, buf, buf, None, None, C.c_size_t(0),
                                None) == gslib.GS_ERR_INVALID_ARG                  # counts at 2 mod 4
    # the accumulate-only fused call checks the same arguments
    assert L.gs_rasterize_fused_acc(10, 1, None, None, 16, 16, None, None, None, None, None, None,
                                    None, None, None, None, None, C.c_size_t(0),
                                    None) == gslib.GS_ERR_INVALID_ARG
    assert L.gs_rasterize_fused_acc(0, 1, None, None, 16, 16, None, buf, None, dummy(0, 0, 0), buf,
                                    buf, buf, buf, buf, None, mis, C.c_size_t(32),
                                    None) == gslib.GS_ERR_INVALID_ARG
    # the separate zeroing: bad sizes, missing or misaligned buffers; nothing to do for n = 0
    assert L.gs_zero_grads(-1, 1, None, None, 1, None) == gslib.GS_ERR_INVALID_ARG
    assert L.gs_zero_grads(10, 0, None, buf, 1, None) == gslib.GS_ERR_INVALID_ARG
    assert L.gs_zero_grads(10, 17, None, buf, 1, None) == gslib.GS_ERR_INVALID_ARG
    assert L.gs_zero_grads(1 << 32, 1, None, buf, 1, None) == gslib.GS_ERR_INVALID_ARG
    assert L.gs_zero_grads(10, 1, None, None, 1, None) == gslib.GS_ERR_INVALID_ARG      # no grads
    assert L.gs_zero_grads(10, 1, None, mis, 1, None) == gslib.GS_ERR_INVALID_ARG       # 4 mod 16
    assert L.gs_zero_grads(10, 1, odd, buf, 1, None) == gslib.GS_ERR_INVALID_ARG        # counts 2 mod 4
    assert L.gs_zero_grads(0, 1, None, None, 1, None) == gslib.GS_OK
    assert L.gs_tile_order(-1, None, None, None) == gslib.GS_ERR_INVALID_ARG
    assert L.gs_tile_order(5, None, None, None) == gslib.GS_ERR_INVALID_ARG          # NULL
    assert L.gs_tile_order(0, None, None, None) == gslib.GS_OK                       # empty
    assert L.gs_project_bwd(10, None, cp, 1, None, None, None, None, None,
                            None) == gslib.GS_ERR_INVALID_ARG
    assert L.gs_loss_l1(None, None, -1, None, None, None) == gslib.GS_ERR_INVALID_ARG
    # the graph-capturable calls
    assert L.gs_bin_and_sort_async(10, 1, None, None, 16, 16, None, 0, 100, None, None, None,
                                   C.byref(out), None) == gslib.GS_ERR_INVALID_ARG  # no workspace
    assert L.gs_bin_and_sort_async(10, 1, None, None, 16, 16, None, 0, 0, None, None, None, None,
                                   None) == gslib.GS_ERR_INVALID_ARG               # capacity 0
    assert L.gs_adam_step_dev(5, None, None, None, None, None, 1e-3, 0.9, 0.999, 1e-8, None,
                              None, None) == gslib.GS_ERR_INVALID_ARG              # no step
    assert L.gs_adam_step_dev(5, None, None, None, None, C.byref(out), 1e-3, 0.9, 0.999, 1e-8,
                              None, None, None) == gslib.GS_ERR_INVALID_ARG        # NULL arrays
    assert L.gs_adam_step_dev(5, None, None, None, None, C.byref(out), 1e-3, 1.0, 0.999, 1e-8,
                              None, None, None) == gslib.GS_ERR_INVALID_ARG        # beta1 = 1
    assert L.gs_step_advance(None, None, None) == gslib.GS_ERR_INVALID_ARG


def test_no_fallback_when_library_missing(gslib, monkeypatch):
    monkeypatch.setattr(gslib, "_lib", None)
    monkeypatch.setattr(gslib, "LIB_PATH", "/nonexistent/libgs103.so")
    with pytest.raises(RuntimeError, match="not built"):
        gslib.lib()
