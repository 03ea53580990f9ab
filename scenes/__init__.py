"""Seeded synthetic scenes, cameras and target images.

This module is the only code shared by the CPU oracle side (tests) and the
GPU side (tests, smoke check, benchmark).  It only draws inputs: it holds none
of the method's arithmetic (no projection, colour, compositing or update).

No dataset is available, so the pages' real-scene workloads (Rubble, Building,
MatrixCity, Mip-NeRF 360, Tanks & Temples, DeepBlending in "On Scaling Up 3D
Gaussian Splatting Training") are replaced by these seeded synthetic scenes of
the stated sizes.  Random numbers come from numpy's PCG64 generator, which
produces the same stream on every platform; seed = 1000 + config index.

Parameter layout: float32 [59][n]: rows 0-2 mean, 3-5 log-scale, 6-9
quaternion (w, x, y, z), 10 opacity logit, 11 + 3*k + c SH coefficient k of
colour channel c.  A camera is a dict: R (world->camera rotation, 3x3, OpenCV
axes: +x right, +y down, +z forward), t (p_cam = R p + t), fx, fy, cx, cy,
width, height, near_z, far_z.
"""
import math

import numpy as np

NPARAM = 59
NEAR_Z = 0.01

# name -> (index, description); index sets the seed.
CONFIGS = {
    "tiny_2k_256": 1,
    "small_200k_1024x768": 2,
    "ring_3m_4x1080p": 3,
    "dense_20m_4k": 4,
    "city_100m_8x1080p": 5,
}


def camera(R, t, fx, fy, cx, cy, width, height, near_z=NEAR_Z, far_z=math.inf):
    return dict(R=np.asarray(R, np.float64).reshape(3, 3), t=np.asarray(t, np.float64).reshape(3),
                fx=float(fx), fy=float(fy), cx=float(cx), cy=float(cy), width=int(width),
                height=int(height), near_z=float(near_z), far_z=float(far_z))


def look_at(position, target, up, fx, fy, width, height, near_z=NEAR_Z, far_z=math.inf):
    """OpenCV-axes camera at `position` looking at `target`, `up` = world up."""
    pos = np.asarray(position, np.float64)
    f = np.asarray(target, np.float64) - pos
    f /= np.linalg.norm(f)
    r = np.cross(f, np.asarray(up, np.float64))
    r /= np.linalg.norm(r)
    d = np.cross(f, r)
    R = np.stack([r, d, f])
    t = -R @ pos
    return camera(R, t, fx, fy, width / 2.0, height / 2.0, width, height, near_z, far_z)


def _common_params(rng, means, logscale_mu, logscale_sd):
    n = means.shape[0]
    p = np.empty((NPARAM, n), np.float32)
    p[0:3] = means.T
    p[3:6] = rng.normal(logscale_mu, logscale_sd, size=(3, n))
    q = rng.standard_normal(size=(4, n))
    q /= np.linalg.norm(q, axis=0, keepdims=True)
    p[6:10] = q
    p[10] = rng.standard_normal(n)
    sh = rng.normal(0.0, 0.05, size=(16, 3, n))
    sh[0] = rng.normal(0.5, 0.2, size=(3, n))
    p[11:59] = sh.reshape(48, n)
    return p


CHUNK = 4_000_000


def _chunked_params(n, seed, draw_means, logscale_mu, logscale_sd):
    """Large scenes: Gaussians are drawn in chunks of CHUNK, chunk c from its
    own PCG64 stream seeded by (seed, c), in parallel threads, straight into
    one float32 [59][n] array (bounded temporaries, same result for any thread
    count).  draw_means(rng, m) -> (m, 3) means of one chunk."""
    import concurrent.futures as cf
    import os
    p = np.empty((NPARAM, n), np.float32)

    def fill(c):
        a, b = c * CHUNK, min(n, (c + 1) * CHUNK)
        rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, c])))
        p[:, a:b] = _common_params(rng, draw_means(rng, b - a), logscale_mu, logscale_sd)

    chunks = range((n + CHUNK - 1) // CHUNK)
    with cf.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
        list(ex.map(fill, chunks))
    return p


def uniform_scene(n, xy, z, seed, logscale=(-3.0, 0.5)):
    """Means x, y ~ U[-xy, xy], z ~ U[z0, z1]; the rest as the tiny config."""
    rng = np.random.Generator(np.random.PCG64(seed))
    means = np.stack([rng.uniform(-xy, xy, n), rng.uniform(-xy, xy, n),
                      rng.uniform(z[0], z[1], n)], axis=1)
    return _common_params(rng, means, *logscale)


def target_images(n_views, width, height, seed):
    rng = np.random.Generator(np.random.PCG64(seed + 7919))
    return rng.random((n_views, 3, height, width), dtype=np.float32)


def make(name, n_override=None):
    """Returns dict(params [59][n] f32, cams [list], target [V][3][H][W] f32,
    lr, steps, sparse_adam, name)."""
    idx = CONFIGS[name]
    seed = 1000 + idx
    if idx == 1:
        n = n_override or 2000
        params = uniform_scene(n, 1.0, (2.0, 6.0), seed)
        cams = [camera(np.eye(3), np.zeros(3), 256, 256, 128, 128, 256, 256)]
        steps, sparse = 1, False
    elif idx == 2:
        n = n_override or 200_000
        params = uniform_scene(n, 4.0, (2.0, 20.0), seed)
        cams = [camera(np.eye(3), np.zeros(3), 900, 900, 512, 384, 1024, 768)]
        steps, sparse = 10, False
    elif idx == 3:
        n = n_override or 3_000_000
        rng = np.random.Generator(np.random.PCG64(seed))
        centres = rng.uniform(-20.0, 20.0, size=(256, 3))
        which = rng.integers(0, 256, size=n)
        means = centres[which] + rng.normal(0.0, 0.3, size=(n, 3))
        params = _common_params(rng, means, -4.0, 0.7)
        cams = []
        for k in range(4):
            th = k * math.pi / 2
            cams.append(look_at((30 * math.cos(th), 30 * math.sin(th), 0.0), (0, 0, 0), (0, 0, 1),
                                1000, 1000, 1920, 1080))
        steps, sparse = 1, False
    elif idx == 4:
        n = n_override or 20_000_000
        rng = np.random.Generator(np.random.PCG64(seed))
        W, H, f = 3840, 2160, 3000.0
        u = rng.uniform(0, W, 64)
        v = rng.uniform(0, H, 64)
        zc = rng.uniform(4.0, 12.0, 64)
        centres = np.stack([(u - W / 2) * zc / f, (v - H / 2) * zc / f, zc], axis=1)

        def dense_means(r, m):
            return centres[r.integers(0, 64, size=m)] + r.normal(0.0, 0.1, size=(m, 3))

        params = _chunked_params(n, seed, dense_means, -3.0, 0.5)
        cams = [camera(np.eye(3), np.zeros(3), f, f, W / 2, H / 2, W, H)]
        steps, sparse = 1, False
    elif idx == 5:
        n = n_override or 100_000_000
        rng = np.random.Generator(np.random.PCG64(seed))
        heights = rng.uniform(0.0, 40.0, size=(20, 20))
        cams = city_cameras(rng)

        def city_means(r, m):
            x = r.uniform(0.0, 1000.0, m)
            y = r.uniform(0.0, 1000.0, m)
            cx_ = np.minimum((x // 50).astype(np.int64), 19)
            cy_ = np.minimum((y // 50).astype(np.int64), 19)
            return np.stack([x, y, heights[cx_, cy_]], axis=1)

        params = _chunked_params(n, seed, city_means, -2.0, 0.8)
        steps, sparse = 1, True
    else:
        raise KeyError(name)
    V = len(cams)
    W, H = cams[0]["width"], cams[0]["height"]
    return dict(name=name, params=params, cams=cams, target=target_images(V, W, H, seed),
                lr=1e-3, steps=steps, sparse_adam=sparse)


CITY_FAR_Z = 250.0


def city_cameras(rng):
    """8 street-level cameras (1.7 m) on cell borders, looking along the street."""
    cams = []
    for k in range(8):
        street = 50.0 * rng.integers(2, 19)
        along = rng.uniform(100.0, 900.0)
        sign = 1.0 if k % 2 == 0 else -1.0
        if k < 4:   # street along x at y = street
            pos = (along, street, 1.7)
            tgt = (along + sign * 100.0, street, 1.7)
        else:       # street along y at x = street
            pos = (street, along, 1.7)
            tgt = (street, along + sign * 100.0, 1.7)
        cams.append(look_at(pos, tgt, (0, 0, 1), 1000, 1000, 1920, 1080, far_z=CITY_FAR_Z))
    return cams
