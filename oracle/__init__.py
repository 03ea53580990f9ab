"""CPU oracle of the 3DGS training step -- TEST INFRASTRUCTURE.

Only tests/, the smoke check in __graft_entry__ and the CPU-baseline leg of
bench.py may import this package.  The product path (the CUDA library and its
Python binding) never imports it, and it never imports the product.  It is a
thin numpy/ctypes wrapper over gs_oracle.c, which holds the arithmetic and
cites the pages each step follows.

Parity status: every function here is pinned by the CPU tests
(tests/test_oracle_*.py) against closed forms, library routines (scipy's
spherical harmonics and rotations, torch's Adam/SparseAdam and L1 loss),
brute force and central finite differences.  No function is unpinned.
"""
import ctypes as C
import os

import numpy as np

from . import build as _build

NPARAM = 59
TILE = 16


class _Camera(C.Structure):
    _fields_ = [("R", C.c_double * 9), ("t", C.c_double * 3), ("fx", C.c_double),
                ("fy", C.c_double), ("cx", C.c_double), ("cy", C.c_double),
                ("width", C.c_int32), ("height", C.c_int32), ("near_z", C.c_double),
                ("far_z", C.c_double)]


_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = C.CDLL(path)
        vp = C.c_void_p
        i64, i32, dbl = C.c_int64, C.c_int32, C.c_double
        L.or_sh_basis.argtypes = [vp, vp]
        L.or_quat_to_rot.argtypes = [vp, vp]
        L.or_project.argtypes = [i64, vp, i32, vp, i32, vp, vp, vp, vp, vp, vp, vp, vp]
        L.or_project_mt.argtypes = [i64, vp, i32, vp, i32, vp, vp, vp, vp, vp, vp, vp, vp, i32]
        L.or_bin_select.argtypes = [i64, i32, vp, vp, vp, i32, i32, i32, vp, i64, vp, vp]
        L.or_bin_select.restype = i64
        L.or_morton_codes.argtypes = [i64, vp, vp]
        L.or_morton_order.argtypes = [i64, vp, vp]
        L.or_tile_rect.argtypes = [C.c_float, C.c_float, i32, i32, i32, i32, vp]
        L.or_count_isect.argtypes = [i64, vp, vp, i32, i32, i32]
        L.or_count_isect.restype = i64
        L.or_bin.argtypes = [i64, i32, vp, vp, vp, i32, i32, i32, vp, vp, vp]
        L.or_raster_fwd.argtypes = [i64, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, i64,
                                    vp, vp, vp, vp, vp, vp, vp]
        L.or_raster_fwd_mt.argtypes = [i64, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp,
                                       i64, vp, vp, vp, vp, vp, vp, i32]
        L.or_raster_bwd_mt.argtypes = [i64, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp,
                                       vp, i64, vp, vp, vp, vp, i32]
        L.or_project_bwd_mt.argtypes = [i64, vp, i32, vp, i32, vp, vp, vp, vp, vp, vp, i32]
        L.or_adam_mt.argtypes = [i64, i64, vp, vp, vp, vp, i64, dbl, dbl, dbl, dbl, vp, i32]
        L.or_bin_mt.argtypes = [i64, i32, vp, vp, vp, i32, i32, i32, vp, vp, vp, i32]
        L.or_prune_mask.argtypes = [i64, i32, i32, i32, i32, vp, vp, vp, vp, i64, C.c_float, vp]
        L.or_raster_fwd_brute.argtypes = [i64, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp,
                                          vp, vp]
        L.or_loss_l1.argtypes = [i64, vp, vp, vp]
        L.or_loss_l1.restype = dbl
        L.or_raster_bwd.argtypes = [i64, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                    i64, vp, vp, vp, vp]
        L.or_project_bwd.argtypes = [i64, vp, i32, vp, i32, vp, vp, vp, vp, vp, vp]
        L.or_adam.argtypes = [i64, i64, vp, vp, vp, vp, i64, dbl, dbl, dbl, dbl, vp]
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def cameras_struct(cams):
    arr = (_Camera * len(cams))()
    for i, c in enumerate(cams):
        arr[i].R[:] = [float(v) for v in np.asarray(c["R"], dtype=np.float64).reshape(9)]
        arr[i].t[:] = [float(v) for v in np.asarray(c["t"], dtype=np.float64).reshape(3)]
        arr[i].fx, arr[i].fy = float(c["fx"]), float(c["fy"])
        arr[i].cx, arr[i].cy = float(c["cx"]), float(c["cy"])
        arr[i].width, arr[i].height = int(c["width"]), int(c["height"])
        arr[i].near_z, arr[i].far_z = float(c["near_z"]), float(c["far_z"])
    return arr


def sh_basis(d):
    d = _f64(d)
    out = np.zeros(16)
    lib().or_sh_basis(_p(d), _p(out))
    return out


def quat_to_rot(q):
    q = _f64(q)
    out = np.zeros(9)
    lib().or_quat_to_rot(_p(q), _p(out))
    return out.reshape(3, 3)


def project(params, cams, tile=TILE, threads=1):
    """params: [59][n] -> dict of per-row arrays (rows = view*n + g).
    threads > 1 splits the Gaussians over POSIX threads (same result)."""
    params = _f64(params)
    n = params.shape[1]
    V = len(cams)
    rows = n * V
    out = dict(mean2d=np.zeros((rows, 2)), conic=np.zeros((rows, 3)), depth=np.zeros(rows),
               color=np.zeros((rows, 3)), opacity=np.zeros(rows),
               radius=np.zeros(rows, np.int32), tiles=np.zeros(rows, np.int32),
               flags=np.zeros(rows, np.uint8))
    cs = cameras_struct(cams)
    lib().or_project_mt(n, _p(params), V, C.cast(cs, C.c_void_p), tile, _p(out["mean2d"]),
                        _p(out["conic"]), _p(out["depth"]), _p(out["color"]),
                        _p(out["opacity"]), _p(out["radius"]), _p(out["tiles"]),
                        _p(out["flags"]), int(threads))
    return out


def morton_codes(params_f32):
    """Morton codes (uint64) of the means of a [59][n] (or [3+][n]) fp32 array."""
    p = np.ascontiguousarray(params_f32, np.float32)
    n = p.shape[1]
    out = np.zeros(n, np.uint64)
    lib().or_morton_codes(n, _p(p), _p(out))
    return out


def morton_order(params_f32):
    p = np.ascontiguousarray(params_f32, np.float32)
    n = p.shape[1]
    out = np.zeros(n, np.uint32)
    lib().or_morton_order(n, _p(p), _p(out))
    return out


def tile_rect(mx, my, radius, tile, tiles_x, tiles_y):
    out = np.zeros(4, np.int32)
    lib().or_tile_rect(float(np.float32(mx)), float(np.float32(my)), int(radius), tile, tiles_x,
                       tiles_y, _p(out))
    return out


def count_isect(mean2d_f32, radius, width, height, tile=TILE):
    m = np.ascontiguousarray(mean2d_f32, np.float32)
    r = np.ascontiguousarray(radius, np.int32)
    return int(lib().or_count_isect(r.shape[0], _p(m), _p(r), tile, width, height))


def bin_and_sort(n, n_views, mean2d_f32, radius, depth_f32, width, height, tile=TILE,
                 threads=1):
    """-> keys u64[I], vals u32[I], ranges i64[n_views*T][2].  threads > 1
    splits the emission and the per-tile sorts over POSIX threads (same
    result)."""
    m = np.ascontiguousarray(mean2d_f32, np.float32)
    r = np.ascontiguousarray(radius, np.int32)
    d = np.ascontiguousarray(depth_f32, np.float32)
    total = count_isect(m, r, width, height, tile)
    T = ((width + tile - 1) // tile) * ((height + tile - 1) // tile)
    keys = np.zeros(max(total, 1), np.uint64)
    vals = np.zeros(max(total, 1), np.uint32)
    ranges = np.zeros((n_views * T, 2), np.int64)
    if threads > 1:
        lib().or_bin_mt(n, n_views, _p(m), _p(r), _p(d), tile, width, height, _p(keys),
                        _p(vals), _p(ranges), int(threads))
    else:
        lib().or_bin(n, n_views, _p(m), _p(r), _p(d), tile, width, height, _p(keys), _p(vals),
                     _p(ranges))
    return keys[:total], vals[:total], ranges


def bin_select(n, n_views, mean2d_f32, radius, depth_f32, width, height, tile_sel, tile=TILE):
    """Brute-force sorted lists of the selected flattened tiles.
    -> vals u32[total], ranges i64[len(tile_sel)][2] into vals."""
    m = np.ascontiguousarray(mean2d_f32, np.float32)
    r = np.ascontiguousarray(radius, np.int32)
    d = np.ascontiguousarray(depth_f32, np.float32)
    sel = np.ascontiguousarray(tile_sel, np.int64)
    total = lib().or_bin_select(n, n_views, _p(m), _p(r), _p(d), tile, width, height, _p(sel),
                                sel.size, None, None)
    vals = np.zeros(max(total, 1), np.uint32)
    ranges = np.zeros((sel.size, 2), np.int64)
    lib().or_bin_select(n, n_views, _p(m), _p(r), _p(d), tile, width, height, _p(sel), sel.size,
                        _p(vals), _p(ranges))
    return vals[:total], ranges


def raster_fwd(n, n_views, width, height, feats, vals, ranges, bg=(0.0, 0.0, 0.0), tile=TILE,
               tile_sel=None, importance=False, threads=1):
    """feats: dict with mean2d, conic, opacity, color (any float dtype).
    Outputs per pixel: image, T_final, n_contrib, pairs (list entries tested
    before the pixel stopped, the stopping one included), included (pairs
    composited), margin (relative distance of the closest threshold decision).
    importance=True adds each row's largest blending weight alpha T (single
    thread only); threads > 1 splits the tiles over POSIX threads."""
    HW = width * height
    m, co = _f64(feats["mean2d"]), _f64(feats["conic"])
    op, col = _f64(feats["opacity"]), _f64(feats["color"])
    vals = np.ascontiguousarray(vals, np.uint32)
    ranges = np.ascontiguousarray(ranges, np.int64)
    bgv = _f64(bg)
    image = np.zeros((n_views, 3, height, width))
    T_final = np.zeros((n_views, height, width))
    n_contrib = np.zeros((n_views, height, width), np.int32)
    pairs = np.zeros((n_views, height, width), np.int64)
    included = np.zeros((n_views, height, width), np.int64)
    margin = np.full((n_views, height, width), np.inf)
    sel = None if tile_sel is None else np.ascontiguousarray(tile_sel, np.int64)
    imp = np.zeros(m.shape[0]) if importance else None
    if threads > 1 and not importance:
        lib().or_raster_fwd_mt(n, n_views, width, height, tile, _p(m), _p(co), _p(op), _p(col),
                               _p(vals), _p(ranges), _p(bgv), _p(sel),
                               0 if sel is None else sel.size, _p(image), _p(T_final),
                               _p(n_contrib), _p(pairs), _p(included), _p(margin), int(threads))
    else:
        lib().or_raster_fwd(n, n_views, width, height, tile, _p(m), _p(co), _p(op), _p(col),
                            _p(vals), _p(ranges), _p(bgv), _p(sel),
                            0 if sel is None else sel.size, _p(image), _p(T_final),
                            _p(n_contrib), _p(pairs), _p(included), _p(margin), _p(imp))
    del HW
    out = dict(image=image, T_final=T_final, n_contrib=n_contrib, pairs=pairs,
               included=included, margin=margin)
    if importance:
        out["importance"] = imp
    return out


def prune_mask(n, n_views, width, height, vals, ranges, n_contrib, importance_f32, capacity,
               tau, tile=TILE):
    """Per-Gaussian uint8 mask (1 = prune) of the working-set-bounded rule."""
    vals = np.ascontiguousarray(vals, np.uint32)
    ranges = np.ascontiguousarray(ranges, np.int64)
    nc = np.ascontiguousarray(n_contrib, np.int32)
    imp = np.ascontiguousarray(importance_f32, np.float32)
    mask = np.zeros(n, np.uint8)
    lib().or_prune_mask(n, n_views, width, height, tile, _p(vals), _p(ranges), _p(nc), _p(imp),
                        int(capacity), float(np.float32(tau)), _p(mask))
    return mask


def compact_index(mask):
    """Indices of the entries kept (mask == 0), in order."""
    return np.nonzero(np.asarray(mask) == 0)[0].astype(np.uint32)


def raster_fwd_brute(n, n_views, width, height, feats, bg=(0.0, 0.0, 0.0), tile=TILE):
    m, co = _f64(feats["mean2d"]), _f64(feats["conic"])
    op, col = _f64(feats["opacity"]), _f64(feats["color"])
    dep = _f64(feats["depth"])
    rad = np.ascontiguousarray(feats["radius"], np.int32)
    bgv = _f64(bg)
    image = np.zeros((n_views, 3, height, width))
    T_final = np.zeros((n_views, height, width))
    lib().or_raster_fwd_brute(n, n_views, width, height, tile, _p(m), _p(co), _p(op), _p(col),
                              _p(dep), _p(rad), _p(bgv), _p(image), _p(T_final))
    return dict(image=image, T_final=T_final)


def loss_l1(image, target):
    a, b = _f64(image), _f64(target)
    g = np.zeros_like(a)
    loss = lib().or_loss_l1(a.size, _p(a), _p(b), _p(g))
    return loss, g


def raster_bwd(n, n_views, width, height, feats, vals, ranges, dL_dimage, bg=(0.0, 0.0, 0.0),
               tile=TILE, tile_sel=None, threads=1):
    rows = n * n_views
    m, co = _f64(feats["mean2d"]), _f64(feats["conic"])
    op, col = _f64(feats["opacity"]), _f64(feats["color"])
    vals = np.ascontiguousarray(vals, np.uint32)
    ranges = np.ascontiguousarray(ranges, np.int64)
    g_img = _f64(dL_dimage)
    bgv = _f64(bg)
    out = dict(mean2d=np.zeros((rows, 2)), conic=np.zeros((rows, 3)), opacity=np.zeros(rows),
               color=np.zeros((rows, 3)))
    sel = None if tile_sel is None else np.ascontiguousarray(tile_sel, np.int64)
    args = (n, n_views, width, height, tile, _p(m), _p(co), _p(op), _p(col), _p(vals),
            _p(ranges), _p(bgv), _p(g_img), _p(sel), 0 if sel is None else sel.size,
            _p(out["mean2d"]), _p(out["conic"]), _p(out["opacity"]), _p(out["color"]))
    if threads > 1:
        lib().or_raster_bwd_mt(*args, int(threads))
    else:
        lib().or_raster_bwd(*args)
    return out


def project_bwd(params, cams, grads2d, tile=TILE, threads=1):
    """grads2d: dict mean2d/conic/opacity/color per row -> (grad[59][n], visible[n]).
    threads > 1 splits the Gaussians over POSIX threads (same result)."""
    params = _f64(params)
    n = params.shape[1]
    grad = np.zeros((NPARAM, n))
    visible = np.zeros(n, np.uint8)
    cs = cameras_struct(cams)
    gm, gc = _f64(grads2d["mean2d"]), _f64(grads2d["conic"])
    go, gcol = _f64(grads2d["opacity"]), _f64(grads2d["color"])
    args = (n, _p(params), len(cams), C.cast(cs, C.c_void_p), tile, _p(gm), _p(gc), _p(go),
            _p(gcol), _p(grad), _p(visible))
    if threads > 1:
        lib().or_project_bwd_mt(*args, int(threads))
    else:
        lib().or_project_bwd(*args)
    return grad, visible


def adam(p, g, m, v, t, lr, beta1=0.9, beta2=0.999, eps=1e-8, visible=None, threads=1):
    """In place on float64 [rows][n_cols] arrays p, m, v.  threads > 1
    splits the columns over POSIX threads (same result)."""
    assert p.dtype == np.float64 and p.flags.c_contiguous
    g = _f64(g)
    vis = None if visible is None else np.ascontiguousarray(visible, np.uint8)
    rows, cols = p.shape
    if threads > 1:
        lib().or_adam_mt(rows, cols, _p(p), _p(g), _p(m), _p(v), int(t), lr, beta1, beta2, eps,
                         _p(vis), int(threads))
    else:
        lib().or_adam(rows, cols, _p(p), _p(g), _p(m), _p(v), int(t), lr, beta1, beta2, eps,
                      _p(vis))


def tiles_grid(width, height, tile=TILE):
    return (width + tile - 1) // tile, (height + tile - 1) // tile


def render(params, cams, bg=(0.0, 0.0, 0.0), tile=TILE, threads=1):
    """Forward chain: project -> bin -> composite, all in the oracle."""
    n = np.asarray(params).shape[1]
    V = len(cams)
    W, H = int(cams[0]["width"]), int(cams[0]["height"])
    pr = project(params, cams, tile, threads=threads)
    keys, vals, ranges = bin_and_sort(n, V, pr["mean2d"].astype(np.float32), pr["radius"],
                                      pr["depth"].astype(np.float32), W, H, tile,
                                      threads=threads)
    fw = raster_fwd(n, V, W, H, pr, vals, ranges, bg, tile, threads=threads)
    return pr, (keys, vals, ranges), fw


def train_step_grads(params, cams, target, bg=(0.0, 0.0, 0.0), tile=TILE, threads=1):
    """Forward + L1 loss + backward; returns (loss, grad[59][n], visible, parts).
    threads > 1 runs every stage split over POSIX threads."""
    n = np.asarray(params).shape[1]
    V = len(cams)
    W, H = int(cams[0]["width"]), int(cams[0]["height"])
    pr, (keys, vals, ranges), fw = render(params, cams, bg, tile, threads=threads)
    loss, g_img = loss_l1(fw["image"], target)
    g2 = raster_bwd(n, V, W, H, pr, vals, ranges, g_img, bg, tile, threads=threads)
    grad, visible = project_bwd(params, cams, g2, tile, threads=threads)
    return loss, grad, visible, dict(proj=pr, keys=keys, vals=vals, ranges=ranges, fwd=fw,
                                     g_img=g_img, g2d=g2)


def lib_path():
    return os.path.join(os.path.dirname(os.path.abspath(__file__)), "liboracle.so")
