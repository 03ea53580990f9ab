"""GB300 (sm_103a) 3D Gaussian Splatting training step.

Python binding of libgs103.so (include/gs.h).  Each gs_* function here only
marshals arguments -- torch tensors to device pointers, camera dicts to the
C struct, the current CUDA stream -- and calls the C ABI function of the same
name; every step of the computation runs in the library's CUDA kernels.
PyTorch provides device memory and streams only.

There is no fallback: if libgs103.so is missing or cannot be loaded, every
call raises GSError (run `python -c "import __graft_entry__ as g; g.build()"`
or `python gaussian_splatting_differentiable_gs_gb300/build.py`).
"""
import ctypes as C
import math
import os

import torch

NPARAM = 59
TILE = 16
MAX_VIEWS = 16
SPLAT_FLOATS = 12  # 48-byte gs_splat / gs_splat_grad records

GS_OK, GS_ERR_INVALID_ARG, GS_ERR_CAPACITY, GS_ERR_TIMEOUT, GS_ERR_CUDA, GS_ERR_DEVICE_CHECK = range(6)

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libgs103.so")


class GSError(RuntimeError):
    def __init__(self, what, status):
        super().__init__("%s failed: %s (status %d)" % (what, status_string(status), status))
        self.status = status


class Camera(C.Structure):
    _fields_ = [("R", C.c_float * 9), ("t", C.c_float * 3), ("fx", C.c_float), ("fy", C.c_float),
                ("cx", C.c_float), ("cy", C.c_float), ("width", C.c_int32),
                ("height", C.c_int32), ("near_z", C.c_float), ("far_z", C.c_float)]


_lib = None


def lib():
    """Loads libgs103.so once; raises GSError-like RuntimeError if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("libgs103.so not built: %s is missing (run build())" % LIB_PATH)
    L = C.CDLL(LIB_PATH)
    vp, i64, i32, f32, sz = C.c_void_p, C.c_int64, C.c_int32, C.c_float, C.c_size_t
    L.gs_project.argtypes = [i64, vp, vp, i32, vp, vp, vp]
    L.gs_bin_workspace_bytes.argtypes = [i64, i64]
    L.gs_bin_workspace_bytes.restype = sz
    L.gs_key_bits.argtypes = [i32, i32, i32]
    L.gs_key_bits.restype = i32
    L.gs_bin_and_sort.argtypes = [i64, i32, vp, vp, i32, i32, vp, sz, i64, vp, vp, vp, vp, vp]
    L.gs_workspace_status.argtypes = [vp, vp]
    L.gs_bin_and_sort_async.argtypes = [i64, i32, vp, vp, i32, i32, vp, sz, i64, vp, vp, vp, vp,
                                        vp]
    L.gs_adam_step_dev.argtypes = [i64, vp, vp, vp, vp, vp, f32, f32, f32, f32, vp, vp, vp]
    L.gs_step_advance.argtypes = [vp, vp, vp]
    L.gs_tile_order.argtypes = [i64, vp, vp, vp]
    L.gs_rasterize_fwd.argtypes = [i64, i32, vp, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp]
    L.gs_rasterize_fwd_counted.argtypes = [i64, i32, vp, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp,
                                           vp, vp]
    L.gs_loss_l1.argtypes = [vp, vp, i64, vp, vp, vp]
    L.gs_rasterize_bwd.argtypes = [i64, i32, vp, vp, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    L.gs_morton_workspace_bytes.argtypes = [i64]
    L.gs_morton_workspace_bytes.restype = sz
    L.gs_morton_order.argtypes = [i64, vp, vp, sz, vp, vp]
    L.gs_gather_columns.argtypes = [i64, i64, i64, vp, vp, vp, vp]
    L.gs_rasterize_fwd_importance.argtypes = [i64, i32, vp, i32, i32, vp, vp, vp, vp, vp, vp, vp,
                                              vp, vp]
    L.gs_prune_mask.argtypes = [i64, i32, i32, i32, vp, vp, vp, vp, i64, f32, vp, vp]
    L.gs_compact_workspace_bytes.argtypes = [i64]
    L.gs_compact_workspace_bytes.restype = sz
    L.gs_compact_index.argtypes = [i64, vp, vp, sz, vp, vp, vp]
    L.gs_rasterize_fused.argtypes = [i64, i32, vp, vp, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp,
                                     vp, vp, vp, sz, vp]
    L.gs_rasterize_fused_acc.argtypes = L.gs_rasterize_fused.argtypes
    L.gs_zero_grads.argtypes = [i64, i32, vp, vp, i32, vp]
    L.gs_rasterize_workspace_bytes.argtypes = [i32, i32, i32, i64]
    L.gs_rasterize_workspace_bytes.restype = sz
    L.gs_project_bwd.argtypes = [i64, vp, vp, i32, vp, vp, vp, vp, vp, vp]
    L.gs_adam_step.argtypes = [i64, vp, vp, vp, vp, i64, f32, f32, f32, f32, vp, vp]
    L.gs_status_string.argtypes = [C.c_int]
    L.gs_status_string.restype = C.c_char_p
    L.gs_version.restype = i32
    for name in ("gs_project", "gs_bin_and_sort", "gs_workspace_status", "gs_rasterize_fwd",
                 "gs_rasterize_fwd_counted", "gs_loss_l1", "gs_rasterize_bwd", "gs_project_bwd", "gs_adam_step"):
        getattr(L, name).restype = C.c_int
    _lib = L
    return L


def status_string(status):
    return lib().gs_status_string(int(status)).decode()


def version():
    return int(lib().gs_version())


# --------------------------------------------------------------------------
# marshalling helpers


def cameras_struct(cams):
    if not 1 <= len(cams) <= MAX_VIEWS:
        raise ValueError("1..%d cameras" % MAX_VIEWS)
    arr = (Camera * len(cams))()
    for i, c in enumerate(cams):
        R = [float(v) for v in torch.as_tensor(c["R"], dtype=torch.float64).reshape(9)]
        t = [float(v) for v in torch.as_tensor(c["t"], dtype=torch.float64).reshape(3)]
        arr[i].R[:] = R
        arr[i].t[:] = t
        arr[i].fx, arr[i].fy = float(c["fx"]), float(c["fy"])
        arr[i].cx, arr[i].cy = float(c["cx"]), float(c["cy"])
        arr[i].width, arr[i].height = int(c["width"]), int(c["height"])
        arr[i].near_z = float(c["near_z"])
        arr[i].far_z = float(c["far_z"]) if math.isfinite(float(c["far_z"])) else float("inf")
    return arr


def _dev(t, dtype, name):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError("%s must be a contiguous CUDA %s tensor" % (name, dtype))
    return C.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return C.c_void_p(s.cuda_stream)


def _check(what, status):
    if status != GS_OK:
        raise GSError(what, status)


def tiles_per_view(width, height):
    return ((width + TILE - 1) // TILE) * ((height + TILE - 1) // TILE)


# --------------------------------------------------------------------------
# the C ABI, one wrapper per function


def gs_project(params, cams, splats, stream=None, tile_counts=None):
    """tile_counts: None, or a CUDA int32 tensor of V*n entries (then culled
    rows get a count of 0 and no record)."""
    n = params.shape[1]
    cs = cameras_struct(cams)
    _check("gs_project", lib().gs_project(n, _dev(params, torch.float32, "params"), C.cast(cs, C.c_void_p),
                                          len(cams), _dev(splats, torch.float32, "splats"),
                                          _dev(tile_counts, torch.int32, "tile_counts"),
                                          _stream(stream)))


def gs_bin_workspace_bytes(n_rows, capacity):
    return int(lib().gs_bin_workspace_bytes(n_rows, capacity))


def gs_key_bits(n_views, width, height):
    return int(lib().gs_key_bits(n_views, width, height))


def gs_bin_and_sort(n, n_views, splats, width, height, workspace, capacity, keys, vals, ranges,
                    stream=None, tile_counts=None):
    """Returns (status, n_isect); status is GS_OK or GS_ERR_CAPACITY, other
    statuses raise GSError."""
    out = C.c_int64(0)
    st = lib().gs_bin_and_sort(n, n_views, _dev(splats, torch.float32, "splats"),
                               _dev(tile_counts, torch.int32, "tile_counts"), width, height,
                               _dev(workspace, torch.uint8, "workspace"), workspace.numel(), capacity,
                               _dev(keys, torch.int64, "keys"), _dev(vals, torch.int32, "vals"),
                               _dev(ranges, torch.int64, "ranges"), C.byref(out), _stream(stream))
    if st not in (GS_OK, GS_ERR_CAPACITY):
        raise GSError("gs_bin_and_sort", st)
    return st, int(out.value)


def gs_workspace_status(workspace, stream=None):
    return int(lib().gs_workspace_status(_dev(workspace, torch.uint8, "workspace"), _stream(stream)))


def gs_bin_and_sort_async(n, n_views, splats, width, height, workspace, capacity, keys, vals,
                          ranges, n_isect, stream=None, tile_counts=None):
    """gs_bin_and_sort without a host synchronisation; n_isect: CUDA int64 [1]."""
    _check("gs_bin_and_sort_async", lib().gs_bin_and_sort_async(
        n, n_views, _dev(splats, torch.float32, "splats"),
        _dev(tile_counts, torch.int32, "tile_counts"), width, height,
        _dev(workspace, torch.uint8, "workspace"), workspace.numel(), capacity,
        _dev(keys, torch.int64, "keys"), _dev(vals, torch.int32, "vals"),
        _dev(ranges, torch.int64, "ranges"), _dev(n_isect, torch.int64, "n_isect"),
        _stream(stream)))


def gs_adam_step_dev(params, grad, m, v, step, lr, beta1=0.9, beta2=0.999, eps=1e-8,
                     visible=None, bin_workspace=None, stream=None):
    """gs_adam_step with the step number in a CUDA int64 [1] tensor."""
    n = params.shape[1]
    _check("gs_adam_step_dev", lib().gs_adam_step_dev(
        n, _dev(params, torch.float32, "params"), _dev(grad, torch.float32, "grad"),
        _dev(m, torch.float32, "m"), _dev(v, torch.float32, "v"), _dev(step, torch.int64, "step"),
        float(lr), float(beta1), float(beta2), float(eps), _dev(visible, torch.uint8, "visible"),
        _dev(bin_workspace, torch.uint8, "bin_workspace"), _stream(stream)))


def gs_step_advance(step, bin_workspace=None, stream=None):
    _check("gs_step_advance", lib().gs_step_advance(
        _dev(step, torch.int64, "step"), _dev(bin_workspace, torch.uint8, "bin_workspace"),
        _stream(stream)))


def gs_tile_order(ranges, order, stream=None):
    """order[b] = the tile the b-th compositing CTA takes: longest lists first."""
    n_flat = ranges.shape[0]
    if order.numel() < n_flat:
        raise ValueError("gs_tile_order: order shorter than ranges")
    _check("gs_tile_order", lib().gs_tile_order(n_flat, _dev(ranges, torch.int64, "ranges"),
                                                _dev(order, torch.int32, "order"), _stream(stream)))


def gs_rasterize_fwd(n, n_views, splats, width, height, vals, ranges, bg, image, T_final, n_contrib,
                     stream=None, tile_order=None):
    bgv = (C.c_float * 3)(*[float(b) for b in bg])
    _check("gs_rasterize_fwd", lib().gs_rasterize_fwd(
        n, n_views, _dev(splats, torch.float32, "splats"), width, height,
        _dev(vals, torch.int32, "vals"), _dev(ranges, torch.int64, "ranges"),
        _dev(tile_order, torch.int32, "tile_order"), C.cast(bgv, C.c_void_p),
        _dev(image, torch.float32, "image"), _dev(T_final, torch.float32, "T_final"),
        _dev(n_contrib, torch.int32, "n_contrib"), _stream(stream)))


def gs_rasterize_fwd_counted(n, n_views, splats, width, height, vals, ranges, bg, image, T_final,
                             n_contrib, counts, stream=None, tile_order=None, pixel_counts=None):
    bgv = (C.c_float * 3)(*[float(b) for b in bg])
    _check("gs_rasterize_fwd_counted", lib().gs_rasterize_fwd_counted(
        n, n_views, _dev(splats, torch.float32, "splats"), width, height,
        _dev(vals, torch.int32, "vals"), _dev(ranges, torch.int64, "ranges"),
        _dev(tile_order, torch.int32, "tile_order"), C.cast(bgv, C.c_void_p),
        _dev(image, torch.float32, "image"), _dev(T_final, torch.float32, "T_final"),
        _dev(n_contrib, torch.int32, "n_contrib"), _dev(counts, torch.int64, "counts"),
        _dev(pixel_counts, torch.int32, "pixel_counts"), _stream(stream)))


def gs_loss_l1(image, target, loss, dL_dimage, stream=None):
    _check("gs_loss_l1", lib().gs_loss_l1(_dev(image, torch.float32, "image"),
                                          _dev(target, torch.float32, "target"), image.numel(),
                                          _dev(loss, torch.float32, "loss"),
                                          _dev(dL_dimage, torch.float32, "dL_dimage"),
                                          _stream(stream)))


def gs_rasterize_bwd(n, n_views, splats, width, height, vals, ranges, bg, T_final, n_contrib,
                     dL_dimage, grads, stream=None, tile_order=None, tile_counts=None):
    bgv = (C.c_float * 3)(*[float(b) for b in bg])
    _check("gs_rasterize_bwd", lib().gs_rasterize_bwd(
        n, n_views, _dev(splats, torch.float32, "splats"),
        _dev(tile_counts, torch.int32, "tile_counts"), width, height,
        _dev(vals, torch.int32, "vals"), _dev(ranges, torch.int64, "ranges"),
        _dev(tile_order, torch.int32, "tile_order"), C.cast(bgv, C.c_void_p),
        _dev(T_final, torch.float32, "T_final"), _dev(n_contrib, torch.int32, "n_contrib"),
        _dev(dL_dimage, torch.float32, "dL_dimage"), _dev(grads, torch.float32, "grads"),
        _stream(stream)))


def gs_rasterize_workspace_bytes(n_views, width, height, capacity):
    return int(lib().gs_rasterize_workspace_bytes(n_views, width, height, capacity))


def gs_rasterize_fused(n, n_views, splats, width, height, vals, ranges, bg, target, image,
                       T_final, n_contrib, loss, grads, stream=None, tile_order=None,
                       workspace=None, tile_counts=None, accumulate=False):
    """workspace: None, or a CUDA uint8 tensor of gs_rasterize_workspace_bytes()
    bytes (the backward then walks the pairs the forward composited).
    accumulate: add to grads as they stand (gs_rasterize_fused_acc; grads
    zeroed before by gs_zero_grads) instead of zeroing them first."""
    bgv = (C.c_float * 3)(*[float(b) for b in bg])
    fn = lib().gs_rasterize_fused_acc if accumulate else lib().gs_rasterize_fused
    _check("gs_rasterize_fused", fn(
        n, n_views, _dev(splats, torch.float32, "splats"),
        _dev(tile_counts, torch.int32, "tile_counts"), width, height,
        _dev(vals, torch.int32, "vals"), _dev(ranges, torch.int64, "ranges"),
        _dev(tile_order, torch.int32, "tile_order"), C.cast(bgv, C.c_void_p),
        _dev(target, torch.float32, "target"), _dev(image, torch.float32, "image"),
        _dev(T_final, torch.float32, "T_final"), _dev(n_contrib, torch.int32, "n_contrib"),
        _dev(loss, torch.float32, "loss"), _dev(grads, torch.float32, "grads"),
        _dev(workspace, torch.uint8, "workspace"),
        0 if workspace is None else workspace.numel(), _stream(stream)))


def gs_zero_grads(n, n_views, grads, stream=None, tile_counts=None, beside=False):
    """Zeroes the gradient records the compositing backward adds to (all
    rows, or with tile_counts the pairs of rows of which one is visible).
    beside: a small striding grid, for a launch that runs beside other
    kernels on another stream."""
    _check("gs_zero_grads", lib().gs_zero_grads(
        n, n_views, _dev(tile_counts, torch.int32, "tile_counts"),
        _dev(grads, torch.float32, "grads"), 1 if beside else 0, _stream(stream)))


def gs_morton_workspace_bytes(n):
    return int(lib().gs_morton_workspace_bytes(n))


def gs_morton_order(params, workspace, perm, stream=None):
    n = params.shape[1]
    _check("gs_morton_order", lib().gs_morton_order(
        n, _dev(params, torch.float32, "params"), _dev(workspace, torch.uint8, "workspace"),
        workspace.numel(), _dev(perm, torch.int32, "perm"), _stream(stream)))


def gs_gather_columns(src, idx, dst, stream=None):
    """dst[:, i] = src[:, idx[i]] (src [rows][n_src], dst [rows][n_dst])."""
    rows, n_src = src.shape
    n_dst = dst.shape[1]
    if dst.shape[0] != rows or idx.numel() < n_dst:
        raise ValueError("gs_gather_columns: shapes")
    _check("gs_gather_columns", lib().gs_gather_columns(
        rows, n_src, n_dst, _dev(src, torch.float32, "src"), _dev(idx, torch.int32, "idx"),
        _dev(dst, torch.float32, "dst"), _stream(stream)))


def gs_rasterize_fwd_importance(n, n_views, splats, width, height, vals, ranges, bg, image,
                                T_final, n_contrib, importance, stream=None, tile_order=None):
    bgv = (C.c_float * 3)(*[float(b) for b in bg])
    _check("gs_rasterize_fwd_importance", lib().gs_rasterize_fwd_importance(
        n, n_views, _dev(splats, torch.float32, "splats"), width, height,
        _dev(vals, torch.int32, "vals"), _dev(ranges, torch.int64, "ranges"),
        _dev(tile_order, torch.int32, "tile_order"), C.cast(bgv, C.c_void_p),
        _dev(image, torch.float32, "image"), _dev(T_final, torch.float32, "T_final"),
        _dev(n_contrib, torch.int32, "n_contrib"), _dev(importance, torch.float32, "importance"),
        _stream(stream)))


def gs_prune_mask(n, n_views, width, height, vals, ranges, n_contrib, importance, capacity, tau,
                  mask, stream=None):
    _check("gs_prune_mask", lib().gs_prune_mask(
        n, n_views, width, height, _dev(vals, torch.int32, "vals"),
        _dev(ranges, torch.int64, "ranges"), _dev(n_contrib, torch.int32, "n_contrib"),
        _dev(importance, torch.float32, "importance"), int(capacity), float(tau),
        _dev(mask, torch.uint8, "mask"), _stream(stream)))


def gs_compact_workspace_bytes(n):
    return int(lib().gs_compact_workspace_bytes(n))


def gs_compact_index(mask, workspace, idx, n_keep, stream=None):
    _check("gs_compact_index", lib().gs_compact_index(
        mask.numel(), _dev(mask, torch.uint8, "mask"), _dev(workspace, torch.uint8, "workspace"),
        workspace.numel(), _dev(idx, torch.int32, "idx"), _dev(n_keep, torch.int64, "n_keep"),
        _stream(stream)))


def gs_project_bwd(params, cams, splats, grads, grad, visible=None, stream=None,
                   tile_counts=None):
    n = params.shape[1]
    cs = cameras_struct(cams)
    _check("gs_project_bwd", lib().gs_project_bwd(
        n, _dev(params, torch.float32, "params"), C.cast(cs, C.c_void_p), len(cams),
        _dev(splats, torch.float32, "splats"), _dev(tile_counts, torch.int32, "tile_counts"),
        _dev(grads, torch.float32, "grads"),
        _dev(grad, torch.float32, "grad"), _dev(visible, torch.uint8, "visible"), _stream(stream)))


def gs_adam_step(params, grad, m, v, step, lr, beta1=0.9, beta2=0.999, eps=1e-8, visible=None,
                 stream=None):
    n = params.shape[1]
    _check("gs_adam_step", lib().gs_adam_step(
        n, _dev(params, torch.float32, "params"), _dev(grad, torch.float32, "grad"),
        _dev(m, torch.float32, "m"), _dev(v, torch.float32, "v"), int(step), float(lr),
        float(beta1), float(beta2), float(eps), _dev(visible, torch.uint8, "visible"),
        _stream(stream)))


# --------------------------------------------------------------------------
# buffers + one training step, in call order


class TrainStep:
    """Owns the device buffers of one training problem (allocated through
    torch) and runs the seven library calls of a step in order.

    params: CUDA float32 [59][n]; target: CUDA float32 [V][3][H][W].
    sparse: use the visibility-masked Adam update.
    fused: step() composites forward, L1 loss and backward in one call
    (gs_rasterize_fused) instead of three.
    sqrt_batch_lr: scale the learning rate by sqrt(V) for a batch of V views
    ("On Scaling Up 3D Gaussian Splatting Training", independent-gradients
    answer: with the gradient averaged over b views Adam's second moment
    falls as 1/b, and lr sqrt(b) approximates b batch-size-1 updates)."""

    def __init__(self, params, cams, target, lr=1e-3, betas=(0.9, 0.999), eps=1e-8,
                 sparse=False, bg=(0.0, 0.0, 0.0), capacity=None, sqrt_batch_lr=False,
                 fused=False):
        lib()
        dev = params.device
        self.params = params
        self.cams = list(cams)
        self.V = len(cams)
        self.n = params.shape[1]
        self.W, self.H = int(cams[0]["width"]), int(cams[0]["height"])
        self.T = tiles_per_view(self.W, self.H)
        self.target = target
        self.lr, self.betas, self.eps, self.sparse, self.bg = lr, betas, eps, sparse, tuple(bg)
        self.lr_step = lr * math.sqrt(self.V) if sqrt_batch_lr else lr
        self.fused = bool(fused)
        rows = self.V * self.n
        f32 = dict(device=dev, dtype=torch.float32)
        self.splats = torch.empty((rows, SPLAT_FLOATS), **f32)
        # per-row tile counts: a culled row costs these 4 bytes, not a record
        self.tile_counts = torch.zeros(rows, device=dev, dtype=torch.int32)
        self.grads2d = torch.empty((rows, SPLAT_FLOATS), **f32)
        self.grad = torch.empty_like(params)
        self.m = torch.zeros_like(params)
        self.v = torch.zeros_like(params)
        self.visible = torch.zeros(self.n, device=dev, dtype=torch.uint8)
        self.image = torch.empty((self.V, 3, self.H, self.W), **f32)
        self.dL_dimage = torch.empty_like(self.image)
        self.T_final = torch.empty((self.V, self.H, self.W), **f32)
        self.n_contrib = torch.empty((self.V, self.H, self.W), device=dev, dtype=torch.int32)
        self.loss = torch.zeros(1, **f32)
        self.ranges = torch.empty((self.V * self.T, 2), device=dev, dtype=torch.int64)
        self.tile_order = torch.empty(self.V * self.T, device=dev, dtype=torch.int32)
        self.t = 0
        self.n_isect = 0
        # a first guess, bounded so that very large scenes do not reserve sort
        # buffers for 4 intersections per row; grown on GS_ERR_CAPACITY
        self._alloc_isect(capacity if capacity is not None else max(1024, min(4 * rows, 1 << 24)))

    def _alloc_isect(self, capacity):
        dev = self.params.device
        self.capacity = int(capacity)
        self.keys = torch.empty(max(self.capacity, 1), device=dev, dtype=torch.int64)
        self.vals = torch.empty(max(self.capacity, 1), device=dev, dtype=torch.int32)
        ws = gs_bin_workspace_bytes(self.V * self.n, self.capacity)
        self.workspace = torch.zeros(ws, device=dev, dtype=torch.uint8)  # zeroed header
        # the fused compositing's per-batch records of the composited pairs
        self.raster_ws = torch.empty(gs_rasterize_workspace_bytes(self.V, self.W, self.H,
                                                                  self.capacity),
                                     device=dev, dtype=torch.uint8)

    # the seven library calls of a step, in order
    def project(self, stream=None):
        gs_project(self.params, self.cams, self.splats, stream, tile_counts=self.tile_counts)

    def bin_and_sort(self, stream=None):
        st, I = gs_bin_and_sort(self.n, self.V, self.splats, self.W, self.H, self.workspace,
                                self.capacity, self.keys, self.vals, self.ranges, stream,
                                tile_counts=self.tile_counts)
        if st == GS_ERR_CAPACITY:
            self._alloc_isect(int(I * 1.25) + 1024)
            st, I = gs_bin_and_sort(self.n, self.V, self.splats, self.W, self.H, self.workspace,
                                    self.capacity, self.keys, self.vals, self.ranges, stream,
                                    tile_counts=self.tile_counts)
            _check("gs_bin_and_sort", st)
        self.n_isect = I
        gs_tile_order(self.ranges, self.tile_order, stream)

    def rasterize_fwd(self, stream=None, counts=None):
        if counts is None:
            gs_rasterize_fwd(self.n, self.V, self.splats, self.W, self.H, self.vals, self.ranges,
                             self.bg, self.image, self.T_final, self.n_contrib, stream,
                             tile_order=self.tile_order)
        else:
            gs_rasterize_fwd_counted(self.n, self.V, self.splats, self.W, self.H, self.vals,
                                     self.ranges, self.bg, self.image, self.T_final, self.n_contrib,
                                     counts, stream, tile_order=self.tile_order)

    def loss_l1(self, stream=None):
        gs_loss_l1(self.image, self.target, self.loss, self.dL_dimage, stream)

    def rasterize_bwd(self, stream=None):
        gs_rasterize_bwd(self.n, self.V, self.splats, self.W, self.H, self.vals, self.ranges, self.bg,
                         self.T_final, self.n_contrib, self.dL_dimage, self.grads2d, stream,
                         tile_order=self.tile_order, tile_counts=self.tile_counts)

    def rasterize_fused(self, stream=None, accumulate=False):
        gs_rasterize_fused(self.n, self.V, self.splats, self.W, self.H, self.vals, self.ranges,
                           self.bg, self.target, self.image, self.T_final, self.n_contrib,
                           self.loss, self.grads2d, stream, tile_order=self.tile_order,
                           workspace=self.raster_ws, tile_counts=self.tile_counts,
                           accumulate=accumulate)

    def zero_grads(self, stream=None, beside=False):
        gs_zero_grads(self.n, self.V, self.grads2d, stream, tile_counts=self.tile_counts,
                      beside=beside)

    def project_bwd(self, stream=None):
        gs_project_bwd(self.params, self.cams, self.splats, self.grads2d, self.grad, self.visible,
                       stream, tile_counts=self.tile_counts)

    def adam(self, stream=None):
        self.t += 1
        gs_adam_step(self.params, self.grad, self.m, self.v, self.t, self.lr_step, self.betas[0],
                     self.betas[1], self.eps, self.visible if self.sparse else None, stream)

    def forward(self, stream=None):
        self.project(stream)
        self.bin_and_sort(stream)
        self.rasterize_fwd(stream)
        return self.image

    def backward(self, stream=None):
        self.loss_l1(stream)
        self.rasterize_bwd(stream)
        self.project_bwd(stream)

    def update(self, stream=None):
        self.adam(stream)

    def reorder_morton(self, stream=None):
        """Renames the Gaussians in Morton order of their means: permutes the
        parameters and the Adam moments consistently (one gs_morton_order and
        three gs_gather_columns).  Returns perm (new index k holds old
        Gaussian perm[k])."""
        dev = self.params.device
        ws = torch.zeros(gs_morton_workspace_bytes(self.n), dtype=torch.uint8, device=dev)
        perm = torch.empty(self.n, dtype=torch.int32, device=dev)
        gs_morton_order(self.params, ws, perm, stream)
        tmp = torch.empty_like(self.params)
        for buf in (self.params, self.m, self.v):
            gs_gather_columns(buf, perm, tmp, stream)
            buf.copy_(tmp)
        return perm

    def prune_to_capacity(self, capacity, tau=2.0, stream=None):
        """Pruning bounded by the per-tile working set (gs_prune_mask) on the
        current parameters: a forward that records importances, the mask,
        and the compaction of the parameters and Adam moments.  Returns
        (params, m, v, kept index, mask); a new TrainStep takes them over."""
        dev = self.params.device
        self.project(stream)
        self.bin_and_sort(stream)
        imp = torch.empty(self.V * self.n, device=dev, dtype=torch.float32)
        gs_rasterize_fwd_importance(self.n, self.V, self.splats, self.W, self.H, self.vals,
                                    self.ranges, self.bg, self.image, self.T_final,
                                    self.n_contrib, imp, stream, tile_order=self.tile_order)
        mask = torch.empty(self.n, device=dev, dtype=torch.uint8)
        gs_prune_mask(self.n, self.V, self.W, self.H, self.vals, self.ranges, self.n_contrib, imp,
                      capacity, tau, mask, stream)
        ws = torch.empty(gs_compact_workspace_bytes(self.n), device=dev, dtype=torch.uint8)
        idx = torch.empty(self.n, device=dev, dtype=torch.int32)
        n_keep = torch.empty(1, device=dev, dtype=torch.int64)
        gs_compact_index(mask, ws, idx, n_keep, stream)
        k = int(n_keep.item())
        out = []
        for buf in (self.params, self.m, self.v):
            dst = torch.empty((buf.shape[0], k), device=dev, dtype=torch.float32)
            gs_gather_columns(buf, idx, dst, stream)
            out.append(dst)
        return out[0], out[1], out[2], idx[:k], mask

    # ---- one step captured into a CUDA graph and replayed ------------------
    def capture(self, margin=1.25):
        """Captures one training step into a CUDA graph; step() then replays it
        (one launch for the whole step, no host synchronisation).  Needs one
        eager step first (it sizes the intersection buffers, kept with
        `margin` to spare).  The step number lives on the device; a step whose
        intersections outgrow the buffers updates nothing and is reported by
        check()."""
        if self.t == 0:
            raise RuntimeError("capture() needs one eager step first")
        dev = self.params.device
        need = int(self.n_isect * margin) + 1024
        if need > self.capacity:
            self._alloc_isect(need)
        self.step_dev = torch.full((1,), self.t, dtype=torch.int64, device=dev)
        self.n_isect_dev = torch.zeros(1, dtype=torch.int64, device=dev)
        self._side = torch.cuda.Stream(device=dev)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self._graph_body()
        self.graph = g

    def _graph_body(self):
        self.project()
        main = torch.cuda.current_stream()
        if self.fused:
            # the gradient records are zeroed on a second stream while the lists
            # are built: the zeroing needs only the tile counts
            self._side.wait_stream(main)
            self.zero_grads(self._side, beside=True)
        gs_bin_and_sort_async(self.n, self.V, self.splats, self.W, self.H, self.workspace,
                              self.capacity, self.keys, self.vals, self.ranges, self.n_isect_dev,
                              tile_counts=self.tile_counts)
        gs_tile_order(self.ranges, self.tile_order)
        if self.fused:
            main.wait_stream(self._side)
            self.rasterize_fused(accumulate=True)
        else:
            self.rasterize_fwd()
            self.loss_l1()
            self.rasterize_bwd()
        self.project_bwd()
        gs_step_advance(self.step_dev, self.workspace)
        gs_adam_step_dev(self.params, self.grad, self.m, self.v, self.step_dev, self.lr_step,
                         self.betas[0], self.betas[1], self.eps,
                         self.visible if self.sparse else None, self.workspace)

    def check(self):
        """After graph replays: GS_OK, or GS_ERR_CAPACITY when the latest step's
        intersections outgrew the buffers (that step updated nothing; the
        buffers are grown, the graph captured again, and the step should be
        repeated).  Synchronises."""
        st = gs_workspace_status(self.workspace)
        if st == GS_ERR_CAPACITY:
            self.t = int(self.step_dev.item())
            self.n_isect = int(self.n_isect_dev.item())
            self.graph = None
            self.capture()
        elif st != GS_OK:
            raise GSError("training step", st)
        else:
            self.t = int(self.step_dev.item())
        return st

    def step(self, stream=None):
        if getattr(self, "graph", None) is not None:
            self.graph.replay()
            self.t += 1
            return self.loss
        if self.fused:
            self.project(stream)
            self.bin_and_sort(stream)
            self.rasterize_fused(stream)
            self.project_bwd(stream)
        else:
            self.forward(stream)
            self.backward(stream)
        self.update(stream)
        return self.loss
