"""Helpers shared by the GPU parity tests: packing oracle outputs into the
library's 48-byte records, fp32-rounded cameras so both sides see identical
inputs, and the comparison metrics with their tolerances."""
import numpy as np

import scenes

# Tolerances.  The pages fix three of them (images max-abs 1e-5 on [0,1]
# colour, gradients and Adam results relative L2 1e-4, intersection lists
# bit-exact).  The rest are derived from fp32 arithmetic.
IMAGE_MAX_ABS = 1e-5
GRAD_REL_L2 = 1e-4
ADAM_REL_L2 = 1e-4
# a pixel whose threshold decisions lie within this relative distance of a
# cut-off may legitimately be decided differently in fp32 (exp error of the
# fast exponential ~2 ulp + argument rounding ~ |power| ulp, << 1e-5; the
# transmittance is carried to ~2 ulp whatever the number of contributors)
MARGIN = 1e-5

# The library's own chain (its fp32 projection) against the oracle's (fp64
# projection): the projected mean is stored in fp32, one ulp ~6e-5 px at
# 512..1024 px, and the exponent moves by |Q d| times that: ~1e-4 relative in
# alpha for the steepest (dilation-limited) splats.  So the chain comparisons
# flag decisions within CHAIN_MARGIN of a cut-off and hold the image to
# CHAIN_IMAGE_MAX_ABS (the sum of alpha c T over a pixel is <= 1, times the
# ~1e-4 relative move), the gradients to CHAIN_GRAD_REL_L2; on identical stage
# inputs the per-call bars above apply.
CHAIN_MARGIN = 1e-4
CHAIN_IMAGE_MAX_ABS = 1e-4
CHAIN_GRAD_REL_L2 = 1e-3


def flagged_allowance(n_pixels, n_pairs, margin=MARGIN):
    """Upper bound on the pixels flagged by `margin`, from the geometry of the
    cut-offs (a Poisson count: mean bound E, allowance E + 4 sqrt(E) + 1).

    Alpha cut-offs (1/255 and 0.99): for one Gaussian the pixels whose alpha
    lies within relative m of a level form an elliptic ring of area
    4 pi m sqrt(det Sigma) (the region where the power exceeds -p has area
    2 pi p sqrt(det Sigma)), while the tile rectangle of the pixels that test
    it holds at least (2r)^2 >= 36 lambda_max >= 36 sqrt(det Sigma) pixels.  A
    tested pair is thus in one band with probability <= pi m / 9, in either
    of the two <= 2 pi m / 9.

    Transmittance cut-off (1e-4): the transmittance of a pixel falls by a
    factor (1 - alpha) <= 1 - 1/255 per contributor, so the values it takes
    hit a band of relative width 2m about 1e-4 with probability <= 2m / (1/255)
    = 510 m per pixel."""
    e = 2.0 * np.pi / 9.0 * margin * n_pairs + 510.0 * margin * n_pixels
    return e + 4.0 * np.sqrt(e) + 1.0


def f32_cams(cams):
    """Cameras with every value rounded to fp32, as the library receives them."""
    out = []
    for c in cams:
        out.append(scenes.camera(np.float32(c["R"]).astype(np.float64),
                                 np.float32(c["t"]).astype(np.float64),
                                 np.float32(c["fx"]), np.float32(c["fy"]), np.float32(c["cx"]),
                                 np.float32(c["cy"]), c["width"], c["height"],
                                 np.float32(c["near_z"]), np.float32(c["far_z"])))
    return out


def pack_records(pr):
    """Oracle projection (dict of fp64 arrays) -> float32 [rows][12] records."""
    rows = pr["radius"].shape[0]
    rec = np.zeros((rows, 12), np.float32)
    rec[:, 0:2] = pr["mean2d"]
    rec[:, 2:5] = pr["conic"]
    rec[:, 5] = pr["opacity"]
    rec[:, 6:9] = pr["color"]
    rec[:, 9] = pr["depth"]
    ints = rec.view(np.int32)
    ints[:, 10] = pr["radius"]
    ints[:, 11] = pr["tiles"]
    return rec


def unpack_records(rec):
    rec = np.asarray(rec, np.float32)
    ints = rec.view(np.int32)
    return dict(mean2d=rec[:, 0:2].astype(np.float64), conic=rec[:, 2:5].astype(np.float64),
                opacity=rec[:, 5].astype(np.float64), color=rec[:, 6:9].astype(np.float64),
                depth=rec[:, 9].astype(np.float64), radius=ints[:, 10].copy(),
                tiles=ints[:, 11].copy())


def feats32(pr):
    """The fp32 values of the projected features, as fp64 arrays."""
    return unpack_records(pack_records(pr))


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / den) if den > 0 else float(np.linalg.norm(a - b))


def grads_to_rows(g):
    """[rows][12] gradient records -> dict of fp64 arrays."""
    g = np.asarray(g, np.float64)
    return dict(mean2d=g[:, 0:2], conic=g[:, 2:5], opacity=g[:, 5], color=g[:, 6:9])


def rows_to_grads(d):
    rows = d["opacity"].shape[0]
    g = np.zeros((rows, 12), np.float32)
    g[:, 0:2] = d["mean2d"]
    g[:, 2:5] = d["conic"]
    g[:, 5] = d["opacity"]
    g[:, 6:9] = d["color"]
    return g


PARAM_GROUPS = {"mean": (0, 3), "log_scale": (3, 6), "quat": (6, 10), "opacity": (10, 11),
                "sh_dc": (11, 14), "sh_rest": (14, 59)}
