"""CPU pins of the oracle: forward pieces against closed forms, library
routines (scipy SH / rotations) and brute force.  None of these re-types the
oracle's own formula; each checks it against something independent."""
import math
import os

import numpy as np
import pytest

import scenes

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split()
            vals[k] = float(v)
    return vals


def test_memory_figures_of_the_pages():
    g = _golden("memory_figures.txt")
    assert g["xyz"] + g["scale"] + g["rotation"] + g["opacity"] + g["sh_coeffs"] == g[
        "params_per_gaussian"] == scenes.NPARAM
    # SH degree 3: (3+1)^2 coefficients per colour channel, 3 channels
    assert (3 + 1) ** 2 * 3 == g["sh_coeffs"]
    # params + two Adam moments, fp32
    assert g["params_per_gaussian"] * g["bytes_per_param"] * 3 == g["bytes_per_gaussian_with_adam"]
    assert abs(g["mi300x_hbm_gb"] * 1e9 / g["bytes_per_gaussian_with_adam"] / 1e6
               - g["mi300x_max_gaussians_millions"]) < 1.0
    assert abs(g["params_per_gaussian"] * g["bytes_per_param"] * 1e6 / 1e9
               - g["gb_per_million_gaussians"]) < 1e-12
    assert abs(g["params_per_gaussian"] * g["bytes_per_param"] * g["largest_run_gaussians"] / 1e9
               - g["largest_run_gb"]) < 1e-3


# --------------------------------------------------------------------------
# spherical harmonics


def _real_sh_scipy(l, m, d):
    """Real SH from scipy's complex Y_l^m (Condon-Shortley phase included):
    m>0: sqrt2 Re Y_l^m, m<0: sqrt2 Im Y_l^|m|, m=0: Y_l^0."""
    from scipy.special import sph_harm_y
    x, y, z = d
    theta = math.acos(max(-1.0, min(1.0, z)))
    phi = math.atan2(y, x)
    Y = sph_harm_y(l, abs(m), theta, phi)
    if m > 0:
        return math.sqrt(2.0) * Y.real
    if m < 0:
        return math.sqrt(2.0) * Y.imag
    return Y.real


def test_sh_basis_matches_scipy(oracle_mod):
    rng = np.random.default_rng(0)
    for _ in range(50):
        d = rng.standard_normal(3)
        d /= np.linalg.norm(d)
        got = oracle_mod.sh_basis(d)
        k = 0
        for l in range(4):
            for m in range(-l, l + 1):
                assert got[k] == pytest.approx(_real_sh_scipy(l, m, d), abs=1e-12), (l, m)
                k += 1


def test_sh_basis_orthonormal_by_exact_quadrature(oracle_mod):
    # Gauss-Legendre in cos(theta) x uniform phi integrates polynomials of
    # degree <= 6 on the sphere exactly.
    xs, ws = np.polynomial.legendre.leggauss(8)
    nphi = 16
    G = np.zeros((16, 16))
    for ct, w in zip(xs, ws):
        st = math.sqrt(1 - ct * ct)
        for j in range(nphi):
            ph = 2 * math.pi * j / nphi
            Y = oracle_mod.sh_basis([st * math.cos(ph), st * math.sin(ph), ct])
            G += w * (2 * math.pi / nphi) * np.outer(Y, Y)
    assert np.abs(G - np.eye(16)).max() < 1e-12


def test_quat_to_rot_matches_scipy(oracle_mod):
    from scipy.spatial.transform import Rotation
    rng = np.random.default_rng(1)
    for _ in range(20):
        q = rng.standard_normal(4)
        q /= np.linalg.norm(q)
        ref = Rotation.from_quat([q[1], q[2], q[3], q[0]]).as_matrix()  # scipy: (x,y,z,w)
        assert np.abs(oracle_mod.quat_to_rot(q) - ref).max() < 1e-14


# --------------------------------------------------------------------------
# projection


def _one_gaussian(mu, log_scale, q, logit, sh=None):
    p = np.zeros((59, 1))
    p[0:3, 0] = mu
    p[3:6, 0] = log_scale
    p[6:10, 0] = q
    p[10, 0] = logit
    if sh is not None:
        p[11:59, 0] = np.asarray(sh).reshape(48)
    return p


def _cam(fx=256.0, fy=256.0, cx=128.0, cy=128.0, W=256, H=256, R=None, t=None):
    return scenes.camera(np.eye(3) if R is None else R, np.zeros(3) if t is None else t, fx, fy, cx,
                         cy, W, H)


@pytest.mark.parametrize("z,s,q", [(4.0, 0.05, (1, 0, 0, 0)), (2.5, 0.01, (0.3, -0.5, 0.7, 0.1)),
                                   (10.0, 0.2, (0.5, 0.5, 0.5, 0.5))])
def test_isotropic_gaussian_on_axis_closed_form(oracle_mod, z, s, q):
    f = 300.0
    q = np.asarray(q, float) / np.linalg.norm(q)
    p = _one_gaussian([0, 0, z], [math.log(s)] * 3, q, 0.0)
    pr = oracle_mod.project(p, [_cam(fx=f, fy=f)])
    var = f * f * s * s / (z * z) + 0.3
    assert pr["mean2d"][0] == pytest.approx([128.0, 128.0], abs=1e-12)
    assert pr["conic"][0] == pytest.approx([1 / var, 0.0, 1 / var], rel=1e-12, abs=1e-15)
    assert pr["radius"][0] == math.ceil(3 * math.sqrt(var))
    assert pr["depth"][0] == pytest.approx(z)


def test_sh_degree0_colour_closed_form(oracle_mod):
    sh = np.zeros((16, 3))
    sh[0] = [0.4, -0.2, 1.3]
    rng = np.random.default_rng(5)
    for _ in range(5):
        mu = [rng.uniform(-1, 1), rng.uniform(-1, 1), rng.uniform(2, 6)]
        p = _one_gaussian(mu, [-3] * 3, [1, 0, 0, 0], 0.3, sh)
        pr = oracle_mod.project(p, [_cam()])
        expect = np.maximum(0.5 + sh[0] / (2 * math.sqrt(math.pi)), 0.0)
        assert pr["color"][0] == pytest.approx(expect, abs=1e-14)
        assert pr["opacity"][0] == pytest.approx(1 / (1 + math.exp(-0.3)))


def test_view_dependent_colour_uses_camera_centre(oracle_mod):
    """colour = 0.5 + sum_k Y_k(d) sh_k with d the unit vector from the
    camera centre to the mean; Y_k from scipy."""
    rng = np.random.default_rng(6)
    for _ in range(5):
        pos = rng.uniform(-3, 3, 3) + np.array([0, 0, -8.0])
        cam = scenes.look_at(pos, (0, 0, 0), (0, 1, 0.2), 200, 200, 128, 96)
        mu = rng.uniform(-0.5, 0.5, 3)
        sh = rng.normal(0, 0.3, (16, 3))
        sh[0] += 1.5
        p = _one_gaussian(mu, [-2.5] * 3, [1, 0, 0, 0], 0.0, sh)
        pr = oracle_mod.project(p, [cam])
        assert pr["radius"][0] > 0
        d = mu - pos
        d /= np.linalg.norm(d)
        Y = [_real_sh_scipy(l, m, d) for l in range(4) for m in range(-l, l + 1)]
        expect = np.maximum(0.5 + np.asarray(Y) @ sh, 0.0)
        assert pr["color"][0] == pytest.approx(expect, abs=1e-12)


def _pinhole(p, cam):
    return np.array([cam["fx"] * p[0] / p[2] + cam["cx"], cam["fy"] * p[1] / p[2] + cam["cy"]])


def _fd_jacobian(fn, p, h=1e-6):
    J = np.zeros((2, 3))
    for i in range(3):
        e = np.zeros(3)
        e[i] = h
        J[:, i] = (fn(p + e) - fn(p - e)) / (2 * h)
    return J


@pytest.mark.parametrize("clamp", [False, True])
def test_ewa_covariance_is_linearised_pinhole(oracle_mod, clamp):
    """cov2 = J W Sigma W^T J^T + 0.3 I with J the Jacobian of the pinhole
    map (finite differences), evaluated at the point clamped to 1.3x the half
    field of view; Sigma from scipy's rotation."""
    from scipy.spatial.transform import Rotation
    rng = np.random.default_rng(7 + clamp)
    for _ in range(5):
        Rw = Rotation.random(random_state=rng).as_matrix()
        cam = _cam(fx=220.0, fy=180.0, cx=128.0, cy=100.0, W=256, H=200, R=Rw,
                   t=rng.uniform(-1, 1, 3) + [0, 0, 6])
        pc = np.array([rng.uniform(-0.3, 0.3), rng.uniform(-0.3, 0.3), 1.0]) * rng.uniform(3, 8)
        if clamp:
            pc[0] = 2.0 * 1.3 * (0.5 * 256 / 220.0) * pc[2]  # x/z twice the clamp limit
        mu = Rw.T @ (pc - cam["t"])
        q = rng.standard_normal(4)
        q /= np.linalg.norm(q)
        ls = rng.uniform(-1.5, -0.5, 3)
        p = _one_gaussian(mu, ls, q, 0.0)
        pr = oracle_mod.project(p, [cam])
        Rq = Rotation.from_quat([q[1], q[2], q[3], q[0]]).as_matrix()
        Sig = Rq @ np.diag(np.exp(2 * ls)) @ Rq.T
        pj = pc.copy()
        if clamp:
            pj[0] = 1.3 * (0.5 * 256 / 220.0) * pc[2]
        J = _fd_jacobian(lambda x: _pinhole(x, cam), pj)
        cov2 = J @ Rw @ Sig @ Rw.T @ J.T + 0.3 * np.eye(2)
        if not clamp:
            inv = np.linalg.inv(cov2)
            assert pr["conic"][0] == pytest.approx([inv[0, 0], inv[0, 1], inv[1, 1]], rel=1e-7)
            assert pr["mean2d"][0] == pytest.approx(_pinhole(pc, cam), rel=1e-12)
        else:
            # clamped rows may be culled (footprint off-screen); project the
            # covariance through the oracle's conic when visible
            if pr["radius"][0] > 0:
                inv = np.linalg.inv(cov2)
                assert pr["conic"][0] == pytest.approx([inv[0, 0], inv[0, 1], inv[1, 1]], rel=1e-7)
        lam = np.linalg.eigvalsh(cov2).max()
        if pr["radius"][0] > 0:
            assert pr["radius"][0] == math.ceil(3 * math.sqrt(lam))


def test_culling_near_plane_and_offscreen(oracle_mod):
    cam = _cam()
    p = np.concatenate([_one_gaussian([0, 0, 0.005], [-3] * 3, [1, 0, 0, 0], 0.0),
                        _one_gaussian([0, 0, -2.0], [-3] * 3, [1, 0, 0, 0], 0.0),
                        _one_gaussian([50.0, 0, 2.0], [-3] * 3, [1, 0, 0, 0], 0.0),
                        _one_gaussian([0, 0, 3.0], [-3] * 3, [1, 0, 0, 0], 0.0)], axis=1)
    pr = oracle_mod.project(p, [cam])
    assert list(pr["radius"][:3]) == [0, 0, 0] and list(pr["tiles"][:3]) == [0, 0, 0]
    assert pr["radius"][3] > 0 and pr["tiles"][3] > 0


def test_footprint_rect_covers_radius_disc(oracle_mod):
    """Every in-image pixel centre within `radius` of the mean lies in a tile
    of the rectangle."""
    rng = np.random.default_rng(11)
    W, H, tile = 200, 120, 16
    tx, ty = (W + tile - 1) // tile, (H + tile - 1) // tile
    ys, xs = np.mgrid[0:H, 0:W]
    for _ in range(200):
        mx, my = rng.uniform(-40, W + 40), rng.uniform(-40, H + 40)
        r = int(rng.integers(1, 60))
        x0, x1, y0, y1 = oracle_mod.tile_rect(mx, my, r, tile, tx, ty)
        inside = (xs + 0.5 - np.float32(mx)) ** 2 + (ys + 0.5 - np.float32(my)) ** 2 <= r * r
        ptx, pty = xs // tile, ys // tile
        in_rect = (ptx >= x0) & (ptx < x1) & (pty >= y0) & (pty < y1)
        assert not np.any(inside & ~in_rect)


def test_binning_brute_force(oracle_mod):
    """Enumerate every (row, tile) pair by a direct containment test, sort the
    (key, id) tuples with Python's sort and compare bit for bit."""
    cfg = scenes.make("tiny_2k_256", n_override=300)
    cams = [cfg["cams"][0], scenes.camera(np.eye(3), [0.3, -0.2, 0.5], 256, 256, 128, 128, 256, 256)]
    n = 300
    pr = oracle_mod.project(cfg["params"], cams)
    m32 = pr["mean2d"].astype(np.float32)
    d32 = pr["depth"].astype(np.float32)
    keys, vals, ranges = oracle_mod.bin_and_sort(n, 2, m32, pr["radius"], d32, 256, 256)
    tile = np.float32(16)
    T = 16 * 16
    items = []
    for r in range(2 * n):
        if pr["radius"][r] <= 0:
            continue
        fr = np.float32(pr["radius"][r])
        mx, my = m32[r]
        x0 = min(max(math.floor(np.float32(mx - fr) / tile), 0), 16)
        x1 = min(max(math.ceil(np.float32(mx + fr) / tile), 0), 16)
        y0 = min(max(math.floor(np.float32(my - fr) / tile), 0), 16)
        y1 = min(max(math.ceil(np.float32(my + fr) / tile), 0), 16)
        view, g = divmod(r, n)
        for t in range(T):
            tx_, ty_ = t % 16, t // 16
            if x0 <= tx_ < x1 and y0 <= ty_ < y1:
                dbits = int(np.array([d32[r]], np.float32).view(np.uint32)[0])
                items.append((((view * T + t) << 32) | dbits, g))
    items.sort()
    assert keys.size == len(items) == int(pr["tiles"].sum())
    assert [int(k) for k in keys] == [k for k, _ in items]
    assert [int(v) for v in vals] == [v for _, v in items]
    for f in range(2 * T):
        sel = [i for i, (k, _) in enumerate(items) if (k >> 32) == f]
        if sel:
            assert list(ranges[f]) == [sel[0], sel[-1] + 1]
        else:
            assert list(ranges[f]) == [0, 0]
    # per-tile brute-force lists (used on scenes too large to bin on the CPU)
    tsel = np.array([0, 17, 100, 255, T + 3, T + 136, 2 * T - 1], np.int64)
    svals, sranges = oracle_mod.bin_select(n, 2, m32, pr["radius"], d32, 256, 256, tsel)
    for i, f in enumerate(tsel):
        want = [v for k, v in items if (k >> 32) == f]
        a, b = sranges[i]
        assert [int(v) for v in svals[a:b]] == want


def test_threaded_projection_is_identical(oracle_mod):
    cfg = scenes.make("tiny_2k_256", n_override=1001)
    cams = [cfg["cams"][0], scenes.camera(np.eye(3), [0.3, -0.2, 0.5], 256, 256, 128, 128, 256, 256)]
    one = oracle_mod.project(cfg["params"], cams)
    many = oracle_mod.project(cfg["params"], cams, threads=5)
    for k in one:
        assert np.array_equal(one[k], many[k]), k


# --------------------------------------------------------------------------
# compositing


def _centre_scene(logits, depths, colors_dc, W=64, H=64, px=(20, 33)):
    """Gaussians on the optical axis of a camera whose principal point sits on
    the centre of pixel px; degree-0 colour only."""
    k = len(logits)
    p = np.concatenate([
        _one_gaussian([0, 0, depths[i]], [-2.5] * 3, [1, 0, 0, 0], logits[i],
                      np.concatenate([colors_dc[i], np.zeros(45)])) for i in range(k)], axis=1)
    cam = _cam(fx=60.0, fy=60.0, cx=px[0] + 0.5, cy=px[1] + 0.5, W=W, H=H)
    return p, cam


def test_single_gaussian_at_pixel_centre(oracle_mod):
    for logit in (-2.0, 0.0, 1.5, 6.0):
        dc = np.array([0.7, -0.1, 0.25])
        p, cam = _centre_scene([logit], [3.0], [dc])
        pr, _, fw = oracle_mod.render(p, [cam])
        a = min(0.99, 1 / (1 + math.exp(-logit)))
        col = np.maximum(0.5 + dc / (2 * math.sqrt(math.pi)), 0)
        assert fw["image"][0, :, 33, 20] == pytest.approx(a * col, abs=1e-14)
        assert fw["T_final"][0, 33, 20] == pytest.approx(1 - a, abs=1e-14)
        assert fw["n_contrib"][0, 33, 20] == 1


def test_stack_transmittance_is_product(oracle_mod):
    rng = np.random.default_rng(3)
    k = 6
    logits = rng.uniform(-1.0, 1.0, k)
    depths = np.sort(rng.uniform(2, 8, k))[::-1]  # given back to front
    dcs = rng.uniform(-0.5, 1.0, (k, 3))
    p, cam = _centre_scene(list(logits), list(depths), list(dcs))
    pr, _, fw = oracle_mod.render(p, [cam])
    order = np.argsort(depths)  # front to back
    a = 1 / (1 + np.exp(-logits[order]))
    cols = np.maximum(0.5 + dcs[order] / (2 * math.sqrt(math.pi)), 0)
    T = np.concatenate([[1.0], np.cumprod(1 - a)])
    assert fw["T_final"][0, 33, 20] == pytest.approx(T[-1], rel=1e-13)
    expect = (cols * (a * T[:-1])[:, None]).sum(0)
    assert fw["image"][0, :, 33, 20] == pytest.approx(expect, rel=1e-13)


def test_two_gaussians_closed_form(oracle_mod):
    dcs = [np.array([1.0, 0.2, -0.3]), np.array([-0.4, 0.9, 0.5])]
    p, cam = _centre_scene([0.4, -0.7], [2.0, 5.0], dcs)
    _, _, fw = oracle_mod.render(p, [cam])
    a1, a2 = 1 / (1 + math.exp(-0.4)), 1 / (1 + math.exp(0.7))
    c1, c2 = [np.maximum(0.5 + d / (2 * math.sqrt(math.pi)), 0) for d in dcs]
    assert fw["image"][0, :, 33, 20] == pytest.approx(a1 * c1 + (1 - a1) * a2 * c2, rel=1e-13)


def test_early_termination_excludes_stopping_gaussian(oracle_mod):
    """alpha 0.85 each: T = 0.15^k; the 5th would take T below 1e-4, so it
    and everything behind it is excluded."""
    logit = math.log(0.85 / 0.15)
    k = 8
    dcs = [np.array([0.3 * i, 0.1, 0.2]) for i in range(k)]
    p, cam = _centre_scene([logit] * k, [2.0 + i for i in range(k)], dcs)
    _, _, fw = oracle_mod.render(p, [cam])
    a = 0.85
    cols = [np.maximum(0.5 + d / (2 * math.sqrt(math.pi)), 0) for d in dcs]
    expect = sum(cols[i] * a * 0.15 ** i for i in range(4))
    assert fw["n_contrib"][0, 33, 20] == 4
    assert fw["T_final"][0, 33, 20] == pytest.approx(0.15 ** 4, rel=1e-12)
    assert fw["image"][0, :, 33, 20] == pytest.approx(expect, rel=1e-12)


def test_brute_mode_equals_tiled_mode(oracle_mod):
    """Block size alters no pixel: per-pixel global (depth, id) order with the
    footprint test gives exactly the tiled result ("On Scaling Up 3D Gaussian
    Splatting Training", answer (1) on the pixel block size)."""
    cfg = scenes.make("tiny_2k_256", n_override=500)
    cams = cfg["cams"]
    pr, (keys, vals, ranges), fw = oracle_mod.render(cfg["params"], cams)
    feats = dict(pr)
    feats["depth"] = pr["depth"].astype(np.float32).astype(np.float64)
    bf = oracle_mod.raster_fwd_brute(500, 1, 256, 256, feats)
    assert np.array_equal(bf["image"], fw["image"])
    assert np.array_equal(bf["T_final"], fw["T_final"])


def test_rigid_motion_invariance(oracle_mod):
    """Moving the world and the camera by the same rigid motion leaves the
    image unchanged (degree-0 colour, so SH need no rotation).  Catches a
    transposed camera rotation or a wrong quaternion convention."""
    from scipy.spatial.transform import Rotation
    cfg = scenes.make("tiny_2k_256", n_override=400)
    p = cfg["params"].astype(np.float64)
    p[14:] = 0.0
    cam = cfg["cams"][0]
    _, _, fw0 = oracle_mod.render(p, [cam])
    rng = np.random.default_rng(9)
    Q = Rotation.random(random_state=rng)
    Qm = Q.as_matrix()
    tau = rng.uniform(-2, 2, 3)
    p2 = p.copy()
    p2[0:3] = Qm @ p[0:3] + tau[:, None]
    qx, qy, qz, qw = Q.as_quat()
    w, x, y, z = p[6], p[7], p[8], p[9]
    p2[6] = qw * w - qx * x - qy * y - qz * z
    p2[7] = qw * x + qx * w + qy * z - qz * y
    p2[8] = qw * y - qx * z + qy * w + qz * x
    p2[9] = qw * z + qx * y - qy * x + qz * w
    R2 = cam["R"] @ Qm.T
    cam2 = scenes.camera(R2, cam["t"] - R2 @ tau, cam["fx"], cam["fy"], cam["cx"], cam["cy"],
                         cam["width"], cam["height"])
    pr1, _, fw1 = oracle_mod.render(p2, [cam2])
    ok = pr1["flags"] == 0
    assert ok.mean() > 0.9
    assert np.abs(fw1["image"] - fw0["image"]).max() < 1e-9


# --------------------------------------------------------------------------
# Morton order


def test_morton_order_is_the_z_curve_on_a_grid(oracle_mod):
    """Points on an 8x8x8 grid (bounding box [0,7]^3, shuffled): the sorted
    order must list the eight octants as consecutive blocks of 64, in the
    order x-bit | y-bit << 1 | z-bit << 2, and recursively the 2x2x2 cells
    of each octant as blocks of 8 -- the Z-order curve, which pins the bit
    interleave and the monotone quantisation without re-deriving the code."""
    g = np.stack(np.meshgrid(np.arange(8), np.arange(8), np.arange(8), indexing="ij"), 0)
    pts = g.reshape(3, -1).astype(np.float32)
    rng = np.random.default_rng(3)
    sh = rng.permutation(pts.shape[1])
    pts = pts[:, sh]
    order = oracle_mod.morton_order(pts)
    assert sorted(order.tolist()) == list(range(512))
    p = pts[:, order].astype(int)
    for level, size in ((4, 64), (2, 8), (1, 1)):
        cell = (p // level) % 2  # the bit chosen at this level
        idx = cell[0] + 2 * cell[1] + 4 * cell[2]
        blocks = idx.reshape(-1, size)
        assert np.all(blocks == blocks[:, :1])  # one cell per block
        assert np.array_equal(blocks[:8, 0] if size > 1 else idx[:8], np.arange(8))
    # consecutive points never jump more than the curve allows inside a cell
    assert np.all(np.abs(np.diff(p[:, :8], axis=1)).max(axis=0) <= 1)


def test_morton_codes_closed_forms(oracle_mod):
    p = np.array([[0, 1, 0, 0, 1, 0.5],
                  [0, 0, 1, 0, 1, 0.5],
                  [0, 0, 0, 1, 1, 0.5]], np.float32)
    c = oracle_mod.morton_codes(p)
    xs = sum(1 << (3 * b) for b in range(21))
    assert [int(v) for v in c[:5]] == [0, xs, xs << 1, xs << 2, (1 << 63) - 1]
    # the centre quantises to 2^20 on every axis: only code bits 60, 61, 62
    assert int(c[5]) == 7 << 60
    # a flat axis (all z equal) contributes no bits; duplicates keep index order
    q = np.array([[3, 1, 3, 1], [2, 2, 2, 2], [5, 5, 5, 5]], np.float32)
    cq = oracle_mod.morton_codes(q)
    assert int(cq[0]) == int(cq[2]) == xs and int(cq[1]) == 0
    assert oracle_mod.morton_order(q).tolist() == [1, 3, 0, 2]


# --------------------------------------------------------------------------
# importance and pruning bounded by the per-tile working set


def test_importance_is_largest_blending_weight(oracle_mod):
    """Two Gaussians on the axis through a pixel centre, both peaking there
    (the back one is narrower than the front one's hole): importances are
    their weights at that pixel, alpha1 and (1 - alpha1) alpha2."""
    p, cam = _centre_scene([0.4, -0.7], [2.0, 5.0], [np.zeros(3), np.zeros(3)])
    pr = oracle_mod.project(p, [cam])
    m32, d32 = pr["mean2d"].astype(np.float32), pr["depth"].astype(np.float32)
    _, vals, ranges = oracle_mod.bin_and_sort(2, 1, m32, pr["radius"], d32, 64, 64)
    fw = oracle_mod.raster_fwd(2, 1, 64, 64, pr, vals, ranges, importance=True)
    a1, a2 = 1 / (1 + math.exp(-0.4)), 1 / (1 + math.exp(0.7))
    assert fw["importance"][0] == pytest.approx(a1, rel=1e-12)
    assert fw["importance"][1] == pytest.approx((1 - a1) * a2, rel=1e-12)


def test_prune_mask_hand_cases(oracle_mod):
    """Two tiles of one 32x16 view.  Tile 0 lists Gaussians 0..9 with
    importances .5 .1 .3 .3 .05 .9 .2 .01 | .4 .3 and its pixels composite at
    most 8 entries (working set = the first 8); tile 1 lists 10, 11."""
    W, H, n = 32, 16, 12
    vals = np.arange(12, dtype=np.uint32)
    ranges = np.array([[0, 10], [10, 12]], np.int64)
    imp = np.array([.5, .1, .3, .3, .05, .9, .2, .01, .4, .3, .02, .03], np.float32)
    nc = np.zeros((1, H, W), np.int32)
    nc[0, 3, 5], nc[0, 0, 0], nc[0, 9, 20] = 8, 2, 2

    def pruned(K, tau):
        return np.nonzero(oracle_mod.prune_mask(n, 1, W, H, vals, ranges, nc, imp, K, tau))[0].tolist()

    assert pruned(8, 2.0) == []                    # within capacity
    assert pruned(5, 2.0) == [1, 4, 7]             # 5th largest of the working set is .2
    assert pruned(5, 0.08) == [4, 7]               # quality floor keeps .1
    assert pruned(3, 2.0) == [1, 4, 6, 7]          # 3rd largest .3 is tied: both kept
    assert pruned(1, 2.0) == [0, 1, 2, 3, 4, 6, 7, 10]  # tile 1 over capacity too
    # a second view where Gaussian 5 is unimportant marks it as well
    vals2 = np.concatenate([vals, vals])
    ranges2 = np.array([[0, 10], [10, 12], [12, 22], [22, 24]], np.int64)
    imp2 = np.concatenate([imp, imp])
    imp2[12 + 5] = 0.001
    nc2 = np.concatenate([nc, nc])
    m = oracle_mod.prune_mask(n, 2, W, H, vals2, ranges2, nc2, imp2, 5, 2.0)
    assert np.nonzero(m)[0].tolist() == [1, 4, 5, 7]


def _list_at_pixel(opacities, offsets, W=16, H=16, px=(3, 5)):
    """Hand-made projected rows, all in one tile's list in the given order:
    entry i has its mean at the centre of pixel px shifted by offsets[i]
    (pixels) and the unit conic, so its raw alpha at px is
    opacities[i] * exp(-|offset|^2 / 2) exactly."""
    k = len(opacities)
    c = np.array([px[0] + 0.5, px[1] + 0.5])
    feats = dict(mean2d=c + np.asarray(offsets, np.float64).reshape(k, 2),
                 conic=np.tile([1.0, 0.0, 1.0], (k, 1)), opacity=np.asarray(opacities, np.float64),
                 color=np.full((k, 3), 0.5))
    vals = np.arange(k, dtype=np.uint32)
    ranges = np.array([[0, k]], np.int64)
    return feats, vals, ranges


def _margin_closed_form(raw):
    """Smallest relative distance of the pixel's decisions from their cut-offs:
    each tested alpha against 1/255 and 0.99, and each next transmittance that
    is formed (alpha passed the 1/255 test) against 1e-4; stops at the pair
    that would take T below 1e-4."""
    m, T = math.inf, 1.0
    for a_raw in raw:
        m = min(m, abs(a_raw - 1 / 255) * 255, abs(a_raw - 0.99) / 0.99)
        a = min(a_raw, 0.99)
        if a < 1 / 255:
            continue
        Tn = T * (1 - a)
        m = min(m, abs(Tn - 1e-4) / 1e-4)
        if Tn < 1e-4:
            break
        T = Tn
    return m


@pytest.mark.parametrize("opac,stop,incl,last,binding", [
    # entry 1 lies 10 px away (skipped); T = 0.4, 0.02, 4e-4, then entry 4
    # would take it to 4e-5 < 1e-4: it stops the pixel; 0.98 is 1 % from 0.99
    ([0.6, 0.5, 0.95, 0.98, 0.9, 0.7], 5, 3, 4, "alpha 0.99"),
    # T = 0.1, 0.01, 1e-3, then 1e-3 * (1 - 0.902) = 0.98e-4: stop, 2 % from 1e-4
    ([0.9, 0.5, 0.9, 0.9, 0.902, 0.3], 5, 3, 4, "T 1e-4"),
    # alpha 0.004 is 2 % above 1/255 and composited; no stop: every entry tested
    ([0.3, 0.5, 0.004, 0.2], 4, 3, 4, "alpha 1/255"),
])
def test_pairs_included_margin_closed_forms(oracle_mod, opac, stop, incl, last, binding):
    """The per-pixel work counts and the threshold margin of the forward:
    pairs = list entries tested up to and including the one that stops the
    pixel (all of them when none stops), included = pairs composited,
    margin = the decision closest to its cut-off (each cut-off made binding
    by one case)."""
    k = len(opac)
    off = np.zeros((k, 2))
    off[1] = [10.0, 0.0]  # exp(-50): skipped by the 1/255 test
    feats, vals, ranges = _list_at_pixel(opac, off)
    fw = oracle_mod.raster_fwd(k, 1, 16, 16, feats, vals, ranges)
    raw = [opac[i] * math.exp(-0.5 * float(off[i] @ off[i])) for i in range(k)]
    assert fw["pairs"][0, 5, 3] == stop
    assert fw["included"][0, 5, 3] == incl
    m = _margin_closed_form(raw)
    assert fw["margin"][0, 5, 3] == pytest.approx(m, rel=1e-9)
    # which cut-off binds, by construction
    a_min = min(abs(r - 1 / 255) * 255 for r in raw[:stop])
    a_max = min(abs(r - 0.99) / 0.99 for r in raw[:stop])
    if binding == "alpha 0.99":
        assert m == pytest.approx(a_max)
    elif binding == "alpha 1/255":
        assert m == pytest.approx(a_min)
    else:
        assert m < min(a_min, a_max)
    # a pixel that no entry reaches: every entry tested, none composited
    assert fw["pairs"][0, 15, 15] == k and fw["included"][0, 15, 15] == 0
    assert fw["margin"][0, 15, 15] > 0.9
    assert fw["n_contrib"][0, 5, 3] == last


def test_pairs_and_included_sum_to_the_lists(oracle_mod):
    """Without any stop, every pixel tests its whole tile list; included
    counts exactly the pairs at or above alpha 1/255 (brute count)."""
    cfg = scenes.make("tiny_2k_256", n_override=300)
    pr, (keys, vals, ranges), fw = oracle_mod.render(cfg["params"], cfg["cams"])
    lens = (ranges[:, 1] - ranges[:, 0]).reshape(16, 16)
    # T never falls by more than the factor 1 - 0.99, so a pixel that ends at
    # T >= 0.01 never formed a next transmittance below 1e-4: it did not stop
    nostop = fw["T_final"][0] >= 0.01
    assert nostop.mean() > 0.5
    full = np.kron(lens, np.ones((16, 16), np.int64))
    assert np.array_equal(fw["pairs"][0][nostop], full[nostop])
    # brute count of alpha >= 1/255 over each non-stopping pixel's list
    ys, xs = np.nonzero(nostop)
    for y, x in list(zip(ys, xs))[::97]:
        t = (y // 16) * 16 + x // 16
        ids = vals[ranges[t, 0]:ranges[t, 1]]
        d = np.array([x + 0.5, y + 0.5]) - pr["mean2d"][ids]
        co = pr["conic"][ids]
        power = -0.5 * (co[:, 0] * d[:, 0] ** 2 + co[:, 2] * d[:, 1] ** 2) - co[:, 1] * d[:, 0] * d[:, 1]
        alpha = np.minimum(0.99, pr["opacity"][ids] * np.exp(power))
        assert fw["included"][0, y, x] == int((alpha >= 1 / 255).sum())


def test_threaded_oracle_equals_single_thread(oracle_mod):
    """The _mt variants only split loops over threads: binning, compositing
    forward, projection backward and Adam give identical results; compositing
    backward equal up to the order of fp64 sums."""
    cfg = scenes.make("tiny_2k_256", n_override=1500)
    cams = [cfg["cams"][0], scenes.camera(np.eye(3), [0.3, -0.2, 0.5], 256, 256, 128, 128, 256, 256)]
    p64 = cfg["params"].astype(np.float64)
    n, V = p64.shape[1], 2
    pr = oracle_mod.project(p64, cams)
    m32, d32 = pr["mean2d"].astype(np.float32), pr["depth"].astype(np.float32)
    one = oracle_mod.bin_and_sort(n, V, m32, pr["radius"], d32, 256, 256)
    many = oracle_mod.bin_and_sort(n, V, m32, pr["radius"], d32, 256, 256, threads=7)
    for a, b in zip(one, many):
        assert np.array_equal(a, b)
    keys, vals, ranges = one
    f1 = oracle_mod.raster_fwd(n, V, 256, 256, pr, vals, ranges)
    f7 = oracle_mod.raster_fwd(n, V, 256, 256, pr, vals, ranges, threads=7)
    for k in f1:
        assert np.array_equal(f1[k], f7[k]), k
    target = scenes.target_images(V, 256, 256, 5)
    _, g_img = oracle_mod.loss_l1(f1["image"], target)
    b1 = oracle_mod.raster_bwd(n, V, 256, 256, pr, vals, ranges, g_img)
    b7 = oracle_mod.raster_bwd(n, V, 256, 256, pr, vals, ranges, g_img, threads=7)
    for k in b1:
        assert np.abs(b7[k] - b1[k]).max() <= 1e-12 * max(1e-300, np.abs(b1[k]).max()), k
    g1, v1 = oracle_mod.project_bwd(p64, cams, b1)
    g7, v7 = oracle_mod.project_bwd(p64, cams, b1, threads=7)
    assert np.array_equal(g1, g7) and np.array_equal(v1, v7)
    rng = np.random.default_rng(2)
    pa, ma, va = p64.copy(), np.zeros_like(p64), np.zeros_like(p64)
    pb, mb, vb = p64.copy(), np.zeros_like(p64), np.zeros_like(p64)
    vis = (rng.random(n) < 0.5).astype(np.uint8)
    for t in (1, 2, 3):
        oracle_mod.adam(pa, g1, ma, va, t, 1e-3, visible=vis)
        oracle_mod.adam(pb, g1, mb, vb, t, 1e-3, visible=vis, threads=7)
    assert np.array_equal(pa, pb) and np.array_equal(ma, mb) and np.array_equal(va, vb)
