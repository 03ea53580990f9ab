"""GPU parity: every library call against the CPU oracle on identical seeded
inputs.  Stage inputs come from the oracle (its projection rounded to fp32,
its sorted lists), so each call is checked on exactly what the oracle saw;
the end-to-end tests then run the library's own chain.

Cases: the tiny (2k, 256x256) and small (200k, 1024x768) configurations at
full size, and a ragged two-view case (200x120: partial tiles on the right
and bottom edges)."""
import numpy as np
import pytest
import torch

import scenes
from parity_util import (ADAM_REL_L2, CHAIN_GRAD_REL_L2, CHAIN_IMAGE_MAX_ABS, CHAIN_MARGIN,
                         GRAD_REL_L2, IMAGE_MAX_ABS, MARGIN, flagged_allowance,
                         PARAM_GROUPS, f32_cams, feats32, grads_to_rows, pack_records, rel_l2,
                         rows_to_grads, unpack_records)

pytestmark = pytest.mark.gpu

CASES = ["tiny", "ragged2", "small"]


def _case(name):
    if name == "tiny":
        cfg = scenes.make("tiny_2k_256")
        return cfg["params"], f32_cams(cfg["cams"]), cfg["target"]
    if name == "small":
        cfg = scenes.make("small_200k_1024x768")
        return cfg["params"], f32_cams(cfg["cams"]), cfg["target"]
    if name == "ragged2":
        params = scenes.uniform_scene(3000, 1.5, (2.0, 8.0), 77)
        cams = [scenes.camera(np.eye(3), np.zeros(3), 150, 150, 100, 60, 200, 120),
                scenes.look_at((0.6, -0.3, -0.4), (0, 0, 5), (0, -1, 0), 160, 150, 200, 120)]
        return params, f32_cams(cams), scenes.target_images(2, 200, 120, 77)
    raise KeyError(name)


_cache = {}


def oracle_side(name):
    """Oracle chain on a case, fp32 rounding applied where the library stores
    fp32 values (projected features, image gradient)."""
    if name in _cache:
        return _cache[name]
    import oracle
    params, cams, target = _case(name)
    n, V = params.shape[1], len(cams)
    W, H = cams[0]["width"], cams[0]["height"]
    p64 = params.astype(np.float64)
    pr = oracle.project(p64, cams)
    f32 = feats32(pr)
    keys, vals, ranges = oracle.bin_and_sort(n, V, f32["mean2d"].astype(np.float32), f32["radius"],
                                             f32["depth"].astype(np.float32), W, H)
    fw = oracle.raster_fwd(n, V, W, H, f32, vals, ranges)
    loss, g_img = oracle.loss_l1(fw["image"], target)
    g_img32 = g_img.astype(np.float32)
    g2 = oracle.raster_bwd(n, V, W, H, f32, vals, ranges, g_img32)
    g2_32 = grads_to_rows(rows_to_grads(g2))
    grad, visible = oracle.project_bwd(p64, cams, g2_32)
    out = dict(params=params, cams=cams, target=target, n=n, V=V, W=W, H=H, pr=pr, f32=f32,
               keys=keys, vals=vals, ranges=ranges, fw=fw, loss=loss, g_img32=g_img32, g2=g2,
               g2_32=g2_32, grad=grad, visible=visible)
    _cache[name] = out
    return out


def _gs():
    import __graft_entry__
    __graft_entry__.build()
    import gaussian_splatting_differentiable_gs_gb300 as gs
    return gs


def _cuda(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def _gpu_bin(gs, n, V, rec32, W, H, capacity=None):
    rows = n * V
    T = gs.tiles_per_view(W, H)
    cap = capacity if capacity is not None else max(1, int(rec32.view(np.int32)[:, 11].astype(np.int64).sum()))
    ws = torch.zeros(gs.gs_bin_workspace_bytes(rows, cap), dtype=torch.uint8, device="cuda")
    keys = torch.empty(max(cap, 1), dtype=torch.int64, device="cuda")
    vals = torch.empty(max(cap, 1), dtype=torch.int32, device="cuda")
    ranges = torch.full((V * T, 2), -7, dtype=torch.int64, device="cuda")
    st, I = gs.gs_bin_and_sort(n, V, _cuda(rec32), W, H, ws, cap, keys, vals, ranges)
    return st, I, keys, vals, ranges, ws


@pytest.mark.parametrize("case", CASES)
def test_project_matches_oracle(case):
    gs = _gs()
    o = oracle_side(case)
    n, V = o["n"], o["V"]
    splats = torch.empty((n * V, 12), dtype=torch.float32, device="cuda")
    gs.gs_project(_cuda(o["params"]), o["cams"], splats)
    g = unpack_records(splats.cpu().numpy())
    pr = o["pr"]
    flagged = pr["flags"] != 0
    both = (g["radius"] > 0) & (pr["radius"] > 0)
    vis_mismatch = ((g["radius"] > 0) != (pr["radius"] > 0)) & ~flagged
    print("rows %d visible %d flagged %d" % (n * V, int((pr["radius"] > 0).sum()), int(flagged.sum())))
    assert not vis_mismatch.any()
    ok = both & ~flagged
    assert np.array_equal(g["radius"][ok], pr["radius"][ok])
    assert np.array_equal(g["tiles"][ok], pr["tiles"][ok])
    assert np.abs(g["mean2d"][ok] - pr["mean2d"][ok]).max() < 1e-3
    for f in ("conic", "color", "opacity", "depth", "mean2d"):
        e = rel_l2(g[f][ok], pr[f][ok])
        print("%s rel-L2 %.2e" % (f, e))
        assert e < 1e-5, f
    rel_conic = np.abs(g["conic"][ok] - pr["conic"][ok]).max(axis=1) / np.abs(pr["conic"][ok]).max(axis=1)
    assert rel_conic.max() < 1e-3
    assert np.abs(g["color"][ok] - pr["color"][ok]).max() < 1e-5
    # culled rows: radius and tiles zero
    culled = g["radius"] == 0
    assert np.all(g["tiles"][culled] == 0)


@pytest.mark.parametrize("case", CASES)
def test_bin_and_sort_bit_exact(case):
    gs = _gs()
    o = oracle_side(case)
    rec = pack_records(o["pr"])
    st, I, keys, vals, ranges, ws = _gpu_bin(gs, o["n"], o["V"], rec, o["W"], o["H"])
    assert st == gs.GS_OK
    assert I == o["keys"].size == int(o["f32"]["tiles"].astype(np.int64).sum())
    assert np.array_equal(keys[:I].cpu().numpy().view(np.uint64), o["keys"])
    assert np.array_equal(vals[:I].cpu().numpy().view(np.uint32), o["vals"])
    assert np.array_equal(ranges.cpu().numpy(), o["ranges"])
    assert gs.gs_workspace_status(ws) == gs.GS_OK


def test_bin_and_sort_equal_depth_ties_break_by_id():
    """Many Gaussians at one depth in the same tiles: the sorted lists fall
    back to Gaussian id."""
    import oracle
    gs = _gs()
    n = 5000
    rng = np.random.default_rng(5)
    pr = dict(mean2d=rng.uniform(0, 64, (n, 2)), conic=np.ones((n, 3)), opacity=np.full(n, 0.5),
              color=np.full((n, 3), 0.5), depth=np.where(rng.random(n) < 0.5, 3.0, 4.0),
              radius=rng.integers(0, 20, n).astype(np.int32), tiles=np.zeros(n, np.int32))
    for r in range(n):
        if pr["radius"][r] > 0:
            x0, x1, y0, y1 = oracle.tile_rect(pr["mean2d"][r, 0], pr["mean2d"][r, 1],
                                              pr["radius"][r], 16, 4, 4)
            pr["tiles"][r] = (x1 - x0) * (y1 - y0)
    pr["radius"][pr["tiles"] == 0] = 0
    rec = pack_records(pr)
    keys_o, vals_o, ranges_o = oracle.bin_and_sort(n, 1, rec[:, 0:2], pr["radius"], rec[:, 9], 64, 64)
    st, I, keys, vals, ranges, _ = _gpu_bin(gs, n, 1, rec, 64, 64)
    assert st == gs.GS_OK and I == keys_o.size
    assert np.array_equal(vals[:I].cpu().numpy().view(np.uint32), vals_o)
    assert np.array_equal(ranges.cpu().numpy(), ranges_o)


@pytest.mark.parametrize("rmax", [6, 120])
@pytest.mark.parametrize("V,W,H,passes", [(16, 1040, 1024, 3), (16, 16400, 16400, 4)])
def test_bin_and_sort_three_and_four_tile_passes(V, W, H, passes, rmax):
    """Views x tiles beyond 2^16 and 2^24: three and four radix passes on the
    tile bits (the buffer chain ends from the other side than with two), with
    equal depths across views and Gaussians; bit for bit against the oracle.
    Radii below 6 px keep rows at one to four tiles (emission by partitions of
    rows); up to 120 px they average more than eight (emission in balanced
    chunks of intersections, with the tile digits counted from the rows'
    rectangles)."""
    import oracle
    gs = _gs()
    n = 2500
    tx, ty = (W + 15) // 16, (H + 15) // 16
    assert (gs.gs_key_bits(V, W, H) - 32 + 7) // 8 == passes
    rng = np.random.default_rng(11 + passes + rmax)
    rows = V * n
    pr = dict(mean2d=np.stack([rng.uniform(-40, W + 40, rows), rng.uniform(-40, H + 40, rows)], 1),
              conic=np.ones((rows, 3)), opacity=np.full(rows, 0.5), color=np.full((rows, 3), 0.5),
              depth=rng.choice([0.5, 2.0, 2.0000002, 7.0], rows),
              radius=rng.integers(0, rmax, rows).astype(np.int32), tiles=np.zeros(rows, np.int32))
    for r in range(rows):
        if pr["radius"][r] > 0:
            x0, x1, y0, y1 = oracle.tile_rect(pr["mean2d"][r, 0], pr["mean2d"][r, 1],
                                              pr["radius"][r], 16, tx, ty)
            pr["tiles"][r] = (x1 - x0) * (y1 - y0)
    pr["radius"][pr["tiles"] == 0] = 0
    rec = pack_records(pr)
    mean_tiles = pr["tiles"].sum() / max(1, int((pr["tiles"] > 0).sum()))
    assert (mean_tiles >= 8) == (rmax > 60), mean_tiles  # the emission form this case exercises
    keys_o, vals_o, ranges_o = oracle.bin_and_sort(n, V, rec[:, 0:2], pr["radius"], rec[:, 9], W, H)
    st, I, keys, vals, ranges, ws = _gpu_bin(gs, n, V, rec, W, H)
    assert st == gs.GS_OK and I == keys_o.size > 0
    assert np.array_equal(keys[:I].cpu().numpy().view(np.uint64), keys_o)
    assert np.array_equal(vals[:I].cpu().numpy().view(np.uint32), vals_o)
    assert np.array_equal(ranges.cpu().numpy(), ranges_o)
    assert gs.gs_workspace_status(ws) == gs.GS_OK


def test_bin_and_sort_capacity_and_empty():
    gs = _gs()
    o = oracle_side("tiny")
    rec = pack_records(o["pr"])
    I_true = o["keys"].size
    st, I, *_ = _gpu_bin(gs, o["n"], o["V"], rec, o["W"], o["H"], capacity=I_true - 1)
    assert st == gs.GS_ERR_CAPACITY and I == I_true
    empty = rec.copy()
    empty.view(np.int32)[:, 10:12] = 0
    st, I, keys, vals, ranges, _ = _gpu_bin(gs, o["n"], o["V"], empty, o["W"], o["H"], capacity=16)
    assert st == gs.GS_OK and I == 0
    assert np.all(ranges.cpu().numpy() == 0)


def _gpu_fwd(gs, o, rec=None):
    n, V, W, H = o["n"], o["V"], o["W"], o["H"]
    rec = pack_records(o["pr"]) if rec is None else rec
    splats = _cuda(rec)
    vals = _cuda(o["vals"].view(np.int32))
    ranges = _cuda(o["ranges"])
    image = torch.empty((V, 3, H, W), device="cuda")
    T_final = torch.empty((V, H, W), device="cuda")
    n_contrib = torch.empty((V, H, W), dtype=torch.int32, device="cuda")
    gs.gs_rasterize_fwd(n, V, splats, W, H, vals, ranges, (0, 0, 0), image, T_final, n_contrib)
    return splats, vals, ranges, image, T_final, n_contrib


@pytest.mark.parametrize("case", ["ragged2", "small"])
def test_tile_order_longest_first_same_results(case):
    """gs_tile_order: tiles by descending floor(log2(list length)), empty
    last, ties in tile order; compositing in that order gives the same image,
    T_final and n_contrib bit for bit, and the same gradients up to the order
    of float atomics."""
    gs = _gs()
    o = oracle_side(case)
    n, V, W, H = o["n"], o["V"], o["W"], o["H"]
    lens = o["ranges"][:, 1] - o["ranges"][:, 0]
    bucket = np.array([int(x).bit_length() for x in lens])
    expect = np.lexsort((np.arange(lens.size), -bucket))
    ranges = _cuda(o["ranges"])
    order = torch.full((lens.size,), -1, dtype=torch.int32, device="cuda")
    gs.gs_tile_order(ranges, order)
    assert np.array_equal(order.cpu().numpy(), expect)
    splats, vals, ranges, image, T_final, n_contrib = _gpu_fwd(gs, o)
    image2, T2, nc2 = torch.empty_like(image), torch.empty_like(T_final), torch.empty_like(n_contrib)
    gs.gs_rasterize_fwd(n, V, splats, W, H, vals, ranges, (0, 0, 0), image2, T2, nc2,
                        tile_order=order)
    assert torch.equal(image2, image) and torch.equal(T2, T_final) and torch.equal(nc2, n_contrib)
    target = torch.from_numpy(np.ascontiguousarray(o["target"], np.float32)).cuda() \
        if "target" in o else torch.rand_like(image)
    outs = []
    for tile_order in (None, order):
        img, Tf, nc = torch.empty_like(image), torch.empty_like(T_final), torch.empty_like(n_contrib)
        loss = torch.empty(1, device="cuda")
        grads = torch.empty((V * n, 12), device="cuda")
        gs.gs_rasterize_fused(n, V, splats, W, H, vals, ranges, (0, 0, 0), target, img, Tf, nc,
                              loss, grads, tile_order=tile_order)
        outs.append((img, loss, grads))
    assert torch.equal(outs[0][0], outs[1][0])
    assert outs[1][1].item() == pytest.approx(outs[0][1].item(), rel=1e-5)  # float atomics
    g0, g1 = outs[0][2].cpu().numpy(), outs[1][2].cpu().numpy()
    assert rel_l2(g1, g0) <= 1e-5


def test_tile_order_buckets_of_huge_lists():
    """gs_tile_order on fabricated ranges (no lists behind them) whose lengths
    reach 2^31 and beyond: buckets 32 and 33 (the last one also takes every
    length >= 2^33) order exactly like the short ones."""
    gs = _gs()
    rng = np.random.default_rng(8)
    choices = np.array([0, 1, 3, 5, 4096, 2 ** 31 - 1, 2 ** 31, 2 ** 31 + 5, 2 ** 32 + 7,
                        2 ** 33 - 1, 2 ** 33, 2 ** 34 + 3], np.int64)
    lens = rng.choice(choices, 1000)
    starts = rng.integers(0, 2 ** 20, lens.size)
    ranges = np.stack([starts, starts + lens], 1).astype(np.int64)
    bucket = np.minimum([int(x).bit_length() for x in lens], 33)
    expect = np.lexsort((np.arange(lens.size), -bucket))
    order = torch.full((lens.size,), -1, dtype=torch.int32, device="cuda")
    gs.gs_tile_order(_cuda(ranges), order)
    assert np.array_equal(order.cpu().numpy(), expect)


@pytest.mark.parametrize("case", CASES)
def test_rasterize_fwd_matches_oracle(case):
    gs = _gs()
    o = oracle_side(case)
    _, _, _, image, T_final, n_contrib = _gpu_fwd(gs, o)
    fw = o["fw"]
    ok = fw["margin"] > MARGIN
    frac = 1.0 - ok.mean()
    img = image.cpu().numpy()
    err = np.abs(img - fw["image"]).max(axis=1)
    allow = flagged_allowance(ok.size, int(fw["pairs"].sum()))
    print("flagged pixels %d (fraction %.2e; 1e-4 of the pixels is %.1f, the allowance from the "
          "cut-offs' geometry %.1f), max err unflagged %.2e, flagged %.2e" %
          ((~ok).sum(), frac, 1e-4 * ok.size, allow, err[ok].max(),
           err[~ok].max() if (~ok).any() else 0.0))
    assert (~ok).sum() <= allow
    assert err[ok].max() <= IMAGE_MAX_ABS
    assert np.abs(T_final.cpu().numpy() - fw["T_final"])[ok].max() <= IMAGE_MAX_ABS
    assert np.array_equal(n_contrib.cpu().numpy()[ok], fw["n_contrib"][ok])


@pytest.mark.parametrize("case", CASES)
def test_counted_pairs_match_oracle(case):
    """The work counts behind the compositing roofline: per pixel, the list
    entries tested before the pixel stopped (the stopping one included) and
    the pairs composited equal the oracle's counts exactly on every unflagged
    pixel; the totals in counts[0..1] are the per-pixel sums; on a flagged
    pixel the tested count stays within the tile's list."""
    gs = _gs()
    o = oracle_side(case)
    n, V, W, H = o["n"], o["V"], o["W"], o["H"]
    splats = _cuda(pack_records(o["pr"]))
    vals = _cuda(o["vals"].view(np.int32))
    ranges = _cuda(o["ranges"])
    image = torch.empty((V, 3, H, W), device="cuda")
    T_final = torch.empty((V, H, W), device="cuda")
    n_contrib = torch.empty((V, H, W), dtype=torch.int32, device="cuda")
    counts = torch.zeros(2, dtype=torch.int64, device="cuda")
    pix = torch.full((2, V, H, W), -1, dtype=torch.int32, device="cuda")
    gs.gs_rasterize_fwd_counted(n, V, splats, W, H, vals, ranges, (0, 0, 0), image, T_final,
                                n_contrib, counts, pixel_counts=pix)
    fw = o["fw"]
    ok = fw["margin"] > MARGIN
    pc = pix.cpu().numpy().astype(np.int64)
    c = counts.cpu().numpy()
    print("tested %d (oracle %d), composited %d (oracle %d), flagged pixels %d" %
          (c[0], fw["pairs"].sum(), c[1], fw["included"].sum(), (~ok).sum()))
    assert np.array_equal(pc[0][ok], fw["pairs"][ok])
    assert np.array_equal(pc[1][ok], fw["included"][ok])
    assert c[0] == pc[0].sum() and c[1] == pc[1].sum()
    T = gs.tiles_per_view(W, H)
    tx = (W + 15) // 16
    lens = (o["ranges"][:, 1] - o["ranges"][:, 0]).reshape(V, -1)
    yy, xx = np.meshgrid(np.arange(H), np.arange(W), indexing="ij")
    tile_len = lens[:, (yy // 16) * tx + xx // 16]
    assert T == lens.shape[1]
    assert np.all(pc[0] <= tile_len) and np.all(pc[1] <= pc[0]) and np.all(pc >= 0)
    # the backward's evaluated pairs (sum of n_contrib) on unflagged pixels
    assert np.array_equal(n_contrib.cpu().numpy()[ok], fw["n_contrib"][ok])


def test_loss_l1_matches_oracle():
    import oracle
    gs = _gs()
    rng = np.random.default_rng(3)
    for count in (1, 7, 4096 + 3, 3 * 768 * 1024):
        a = rng.random(count).astype(np.float32)
        b = rng.random(count).astype(np.float32)
        b[::97] = a[::97]
        loss_o, g_o = oracle.loss_l1(a.astype(np.float64), b.astype(np.float64))
        loss = torch.empty(1, device="cuda")
        g = torch.empty(count, device="cuda")
        gs.gs_loss_l1(_cuda(a), _cuda(b), loss, g)
        assert loss.item() == pytest.approx(loss_o, rel=1e-5)
        assert np.array_equal(np.sign(g.cpu().numpy()), np.sign(g_o))
        assert np.abs(g.cpu().numpy() - g_o).max() <= 1e-7 / count


@pytest.mark.parametrize("case", CASES)
def test_rasterize_bwd_matches_oracle(case):
    gs = _gs()
    o = oracle_side(case)
    n, V, W, H = o["n"], o["V"], o["W"], o["H"]
    splats, vals, ranges, image, T_final, n_contrib = _gpu_fwd(gs, o)
    grads = torch.empty((n * V, 12), device="cuda")
    gs.gs_rasterize_bwd(n, V, splats, W, H, vals, ranges, (0, 0, 0), T_final, n_contrib,
                        _cuda(o["g_img32"]), grads)
    g = grads_to_rows(grads.cpu().numpy())
    for f in ("mean2d", "conic", "opacity", "color"):
        e = rel_l2(g[f], o["g2"][f])
        print("%s rel-L2 %.2e" % (f, e))
        assert e <= GRAD_REL_L2, f
    assert np.all(grads.cpu().numpy()[:, 9:12] == 0)


@pytest.mark.parametrize("case", CASES)
def test_project_bwd_matches_oracle(case):
    gs = _gs()
    o = oracle_side(case)
    n, V = o["n"], o["V"]
    grad = torch.empty((59, n), device="cuda")
    visible = torch.empty(n, dtype=torch.uint8, device="cuda")
    gs.gs_project_bwd(_cuda(o["params"]), o["cams"], _cuda(pack_records(o["pr"])),
                      _cuda(rows_to_grads(o["g2_32"])), grad, visible)
    gg = grad.cpu().numpy()
    for name, (a, b) in PARAM_GROUPS.items():
        e = rel_l2(gg[a:b], o["grad"][a:b])
        print("%s rel-L2 %.2e" % (name, e))
        assert e <= GRAD_REL_L2, name
    assert np.array_equal(visible.cpu().numpy(), o["visible"])


@pytest.mark.parametrize("n", [10_001, 10_000])
@pytest.mark.parametrize("sparse", [False, True])
def test_adam_matches_oracle(sparse, n):
    """Five Adam steps against the oracle; sparse mode with n % 4 == 0 takes
    the 16-byte path, otherwise the per-column one.  Columns not visible keep
    p, m and v bit for bit."""
    import oracle
    gs = _gs()
    rng = np.random.default_rng(11)
    p = rng.standard_normal((59, n)).astype(np.float32)
    m = np.zeros((59, n), np.float32)
    v = np.zeros((59, n), np.float32)
    P, M, Vv = _cuda(p), _cuda(m), _cuda(v)
    po, mo, vo = p.astype(np.float64), m.astype(np.float64), v.astype(np.float64)
    ever_visible = np.zeros(n, bool)
    for t in range(1, 6):
        g = (rng.standard_normal((59, n)) * 10.0 ** rng.uniform(-6, -2, (59, n))).astype(np.float32)
        vis = (rng.random(n) < 0.4).astype(np.uint8) if sparse else None
        if sparse:
            vis[: n // 3 // 4 * 4] = 0  # whole groups of four columns never visible
            ever_visible |= vis.astype(bool)
        gs.gs_adam_step(P, _cuda(g), M, Vv, t, 1e-3, visible=None if vis is None else _cuda(vis))
        oracle.adam(po, g.astype(np.float64), mo, vo, t, 1e-3, visible=vis)
    assert rel_l2(P.cpu().numpy(), po) <= ADAM_REL_L2
    assert rel_l2(P.cpu().numpy() - p, po - p) <= 1e-3
    assert rel_l2(M.cpu().numpy(), mo) <= ADAM_REL_L2
    assert rel_l2(Vv.cpu().numpy(), vo) <= ADAM_REL_L2
    if sparse:
        never = ~ever_visible
        assert np.array_equal(P.cpu().numpy()[:, never], p[:, never])
        assert np.all(M.cpu().numpy()[:, never] == 0) and np.all(Vv.cpu().numpy()[:, never] == 0)


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("case", ["tiny", "ragged2"])
def test_train_step_end_to_end(case, fused):
    """The library's own chain from the fp32 parameters against the oracle's
    chain: loss, image, gradients and the Adam result, at the chain bars (the
    library's fp32 projection against the oracle's fp64 one)."""
    import oracle
    gs = _gs()
    o = oracle_side(case)
    params = o["params"]
    step = gs.TrainStep(_cuda(params), o["cams"], _cuda(o["target"]), lr=1e-3, fused=fused)
    if fused:
        step.project()
        step.bin_and_sort()
        step.rasterize_fused()
        step.project_bwd()
    else:
        step.forward()
        step.backward()
    loss_o, grad_o, vis_o, parts = oracle.train_step_grads(params.astype(np.float64), o["cams"],
                                                           o["target"])
    img = step.image.cpu().numpy()
    ok = parts["fwd"]["margin"] > CHAIN_MARGIN
    err = np.abs(img - parts["fwd"]["image"]).max(axis=1)[ok].max()
    print("e2e image max err %.2e, loss %.6f vs %.6f" % (err, step.loss.item(), loss_o))
    assert step.loss.item() == pytest.approx(loss_o, rel=1e-5)
    assert err <= CHAIN_IMAGE_MAX_ABS
    gg = step.grad.cpu().numpy()
    for name, (a, b) in PARAM_GROUPS.items():
        e = rel_l2(gg[a:b], grad_o[a:b])
        print("e2e %s grad rel-L2 %.2e" % (name, e))
        assert e <= CHAIN_GRAD_REL_L2, name
    step.update()
    po = params.astype(np.float64)
    mo, vo = np.zeros_like(po), np.zeros_like(po)
    oracle.adam(po, grad_o, mo, vo, 1, 1e-3)
    assert rel_l2(step.params.cpu().numpy(), po) <= ADAM_REL_L2


def _far_footprints(seed=91, W=256, H=192):
    """Projected records (fp32) of a street-level situation: elongated
    footprints whose means lie 50..4000 px off screen with the long axis
    pointing across the image, mixed with ordinary small splats inside it."""
    import oracle
    rng = np.random.default_rng(seed)
    n_far, n_small = 240, 360
    n = n_far + n_small
    mean = np.empty((n, 2))
    dist = 10.0 ** rng.uniform(np.log10(50.0), np.log10(4000.0), n_far)
    ang = rng.uniform(0, 2 * np.pi, n_far)
    centre = np.array([W / 2, H / 2])
    mean[:n_far] = centre + dist[:, None] * np.stack([np.cos(ang), np.sin(ang)], 1)
    axis = ang + np.pi + rng.normal(0, 0.02, n_far)  # towards the image, with jitter
    s_long = dist / rng.uniform(1.5, 3.0, n_far)
    s_short = rng.uniform(0.2, 2.0, n_far)
    mean[n_far:] = rng.uniform(-8, [W + 8, H + 8], (n_small, 2))
    th = rng.uniform(0, np.pi, n_small)
    s1, s2 = np.exp(rng.normal(0.5, 0.6, (2, n_small)))
    axis = np.concatenate([axis, th])
    sl = np.concatenate([s_long, s1])
    ss = np.concatenate([s_short, s2])
    c, s = np.cos(axis), np.sin(axis)
    R = np.stack([np.stack([c, -s], -1), np.stack([s, c], -1)], -2)
    D = np.zeros((n, 2, 2))
    D[:, 0, 0], D[:, 1, 1] = sl ** 2, ss ** 2
    cov = R @ D @ np.swapaxes(R, 1, 2) + 0.3 * np.eye(2)
    inv = np.linalg.inv(cov)
    lam = np.linalg.eigvalsh(cov)[:, 1]
    radius = np.ceil(3.0 * np.sqrt(lam)).astype(np.int32)
    rec = np.zeros((n, 12), np.float32)
    rec[:, 0:2] = mean
    rec[:, 2:5] = np.stack([inv[:, 0, 0], inv[:, 0, 1], inv[:, 1, 1]], 1)
    rec[:, 5] = rng.uniform(0.02, 1.0, n)
    rec[:, 6:9] = rng.random((n, 3))
    rec[:, 9] = rng.uniform(1.0, 50.0, n)
    ints = rec.view(np.int32)
    ints[:, 10] = radius
    tx, ty = (W + 15) // 16, (H + 15) // 16
    for i in range(n):
        x0, x1, y0, y1 = oracle.tile_rect(rec[i, 0], rec[i, 1], int(radius[i]), 16, tx, ty)
        ints[i, 11] = max(0, x1 - x0) * max(0, y1 - y0)
    ints[ints[:, 11] == 0, 10] = 0
    return n, W, H, rec


def test_far_elongated_footprints():
    """Binning and compositing (forward and backward) where the means lie far
    off screen: pixel offsets of thousands of px and near-singular conics,
    which the literal fp32 exponent gets wrong by order one."""
    import oracle
    gs = _gs()
    n, W, H, rec = _far_footprints()
    f32 = unpack_records(rec)
    print("rows %d, on-screen footprints %d, max |mean| %.0f px" %
          (n, int((f32["radius"] > 0).sum()), np.abs(f32["mean2d"]).max()))
    _, vals, ranges = oracle.bin_and_sort(n, 1, rec[:, 0:2], f32["radius"], rec[:, 9], W, H)
    st, I, _, vals_d, ranges_d, _ = _gpu_bin(gs, n, 1, rec, W, H)
    assert st == gs.GS_OK and I == vals.size
    assert np.array_equal(vals_d[:I].cpu().numpy().view(np.uint32), vals)
    assert np.array_equal(ranges_d.cpu().numpy(), ranges)
    fw = oracle.raster_fwd(n, 1, W, H, f32, vals, ranges)
    image = torch.empty((1, 3, H, W), device="cuda")
    T_final = torch.empty((1, H, W), device="cuda")
    n_contrib = torch.empty((1, H, W), dtype=torch.int32, device="cuda")
    splats = _cuda(rec)
    gs.gs_rasterize_fwd(n, 1, splats, W, H, vals_d, ranges_d, (0, 0, 0), image, T_final, n_contrib)
    ok = fw["margin"] > MARGIN
    err = np.abs(image.cpu().numpy() - fw["image"]).max(axis=1)
    print("pairs %d, flagged %d, max err %.2e, max T err %.2e" %
          (int(fw["pairs"].sum()), int((~ok).sum()), err[ok].max(),
           np.abs(T_final.cpu().numpy() - fw["T_final"])[ok].max()))
    assert (~ok).sum() <= flagged_allowance(ok.size, int(fw["pairs"].sum()))
    assert err[ok].max() <= IMAGE_MAX_ABS
    assert np.array_equal(n_contrib.cpu().numpy()[ok], fw["n_contrib"][ok])
    target = scenes.target_images(1, W, H, 91)
    _, g_img = oracle.loss_l1(fw["image"], target)
    g_img = g_img.astype(np.float32)
    g2 = oracle.raster_bwd(n, 1, W, H, f32, vals, ranges, g_img)
    grads = torch.empty((n, 12), device="cuda")
    gs.gs_rasterize_bwd(n, 1, splats, W, H, vals_d, ranges_d, (0, 0, 0), T_final, n_contrib,
                        _cuda(g_img), grads)
    g = grads_to_rows(grads.cpu().numpy())
    for f in ("mean2d", "conic", "opacity", "color"):
        e = rel_l2(g[f], g2[f])
        print("%s rel-L2 %.2e" % (f, e))
        assert e <= GRAD_REL_L2, f


def test_sqrt_batch_lr_step_matches_oracle():
    """A two-view step with the sqrt(b) learning-rate rule: the library's
    update equals the oracle's Adam at lr sqrt(2) on the oracle's gradient."""
    import oracle
    gs = _gs()
    o = oracle_side("ragged2")
    params = o["params"]
    step = gs.TrainStep(_cuda(params), o["cams"], _cuda(o["target"]), lr=1e-3, sqrt_batch_lr=True)
    step.step()
    _, grad_o, _, _ = oracle.train_step_grads(params.astype(np.float64), o["cams"], o["target"])
    po = params.astype(np.float64)
    mo, vo = np.zeros_like(po), np.zeros_like(po)
    oracle.adam(po, grad_o, mo, vo, 1, 1e-3 * np.sqrt(2.0))
    moved = step.params.cpu().numpy().astype(np.float64) - params
    moved_o = po - params
    # at t = 1 the update is lr g / (|g| + eps): lr sqrt(2) wherever |g| >> eps
    big = np.abs(grad_o) > 1e-3 * np.abs(grad_o).max()
    print("max |update| / lr %.5f, big-gradient entries %d" % (np.abs(moved).max() / 1e-3, big.sum()))
    assert rel_l2(step.params.cpu().numpy(), po) <= ADAM_REL_L2
    # (fp32 parameters of magnitude <= 8 round the update by <= 5e-7)
    assert np.abs(moved).max() == pytest.approx(1e-3 * np.sqrt(2.0), rel=2e-3)
    assert np.abs(moved[big] - moved_o[big]).max() <= 2e-6


@pytest.mark.parametrize("with_ws", [False, True])
@pytest.mark.parametrize("case", CASES)
def test_rasterize_fused_matches_oracle_and_separate_calls(case, with_ws):
    """gs_rasterize_fused (forward + L1 + backward in one launch) against the
    oracle's chain and against the three separate library calls; with the
    workspace the backward walks the pairs the forward recorded, without it
    every entry whose box meets the block."""
    gs = _gs()
    o = oracle_side(case)
    n, V, W, H = o["n"], o["V"], o["W"], o["H"]
    splats, vals, ranges, image_s, T_s, nc_s = _gpu_fwd(gs, o)
    target = _cuda(o["target"])
    loss_s = torch.empty(1, device="cuda")
    g_img = torch.empty_like(image_s)
    gs.gs_loss_l1(image_s, target, loss_s, g_img)
    grads_s = torch.empty((n * V, 12), device="cuda")
    gs.gs_rasterize_bwd(n, V, splats, W, H, vals, ranges, (0, 0, 0), T_s, nc_s, g_img, grads_s)
    image = torch.empty_like(image_s)
    T_final = torch.empty_like(T_s)
    n_contrib = torch.empty_like(nc_s)
    loss = torch.full((1,), 7.0, device="cuda")
    grads = torch.full((n * V, 12), 3.0, device="cuda")
    ws = None
    if with_ws:
        ws = torch.full((gs.gs_rasterize_workspace_bytes(V, W, H, int(o["vals"].size)),), 0xA5,
                        dtype=torch.uint8, device="cuda")  # no initialisation needed
    gs.gs_rasterize_fused(n, V, splats, W, H, vals, ranges, (0, 0, 0), target, image, T_final,
                          n_contrib, loss, grads, workspace=ws)
    # the forward is the same code: identical results
    assert torch.equal(image, image_s) and torch.equal(T_final, T_s) and torch.equal(n_contrib, nc_s)
    assert loss.item() == pytest.approx(loss_s.item(), rel=1e-5)  # fp32 sums in another order
    e_sep = rel_l2(grads.cpu().numpy(), grads_s.cpu().numpy())
    # against the oracle (its own image, L1 gradient and backward)
    assert loss.item() == pytest.approx(o["loss"], rel=1e-5)
    g = grads_to_rows(grads.cpu().numpy())
    errs = {f: rel_l2(g[f], o["g2"][f]) for f in ("mean2d", "conic", "opacity", "color")}
    print("fused vs separate grads rel-L2 %.2e; vs oracle %s" %
          (e_sep, ", ".join("%s %.2e" % kv for kv in errs.items())))
    assert e_sep <= 1e-5
    for f, e in errs.items():
        assert e <= GRAD_REL_L2, f
    assert np.all(grads.cpu().numpy()[:, 9:12] == 0)


def test_fused_far_footprints_and_empty_tiles():
    """The fused call on the far-footprint records (long lists, many batches
    left staged by the forward) against the separate calls."""
    gs = _gs()
    n, W, H, rec = _far_footprints()
    f32 = unpack_records(rec)
    st, I, _, vals, ranges, _ = _gpu_bin(gs, n, 1, rec, W, H)
    assert st == gs.GS_OK
    splats = _cuda(rec)
    target = _cuda(scenes.target_images(1, W, H, 91))
    image_s = torch.empty((1, 3, H, W), device="cuda")
    T_s = torch.empty((1, H, W), device="cuda")
    nc_s = torch.empty((1, H, W), dtype=torch.int32, device="cuda")
    gs.gs_rasterize_fwd(n, 1, splats, W, H, vals, ranges, (0.2, 0.1, 0.3), image_s, T_s, nc_s)
    loss_s = torch.empty(1, device="cuda")
    g_img = torch.empty_like(image_s)
    gs.gs_loss_l1(image_s, target, loss_s, g_img)
    grads_s = torch.empty((n, 12), device="cuda")
    gs.gs_rasterize_bwd(n, 1, splats, W, H, vals, ranges, (0.2, 0.1, 0.3), T_s, nc_s, g_img,
                        grads_s)
    for ws_bytes in (None, "full", "short"):
        image, T_final = torch.empty_like(image_s), torch.empty_like(T_s)
        n_contrib, loss = torch.empty_like(nc_s), torch.empty(1, device="cuda")
        grads = torch.empty((n, 12), device="cuda")
        ws = None
        if ws_bytes is not None:
            full = gs.gs_rasterize_workspace_bytes(1, W, H, I)
            # "short": room for only some tiles' records; the others walk the boxes
            ws = torch.empty(full if ws_bytes == "full" else full // 3 // 16 * 16,
                             dtype=torch.uint8, device="cuda")
        gs.gs_rasterize_fused(n, 1, splats, W, H, vals, ranges, (0.2, 0.1, 0.3), target, image,
                              T_final, n_contrib, loss, grads, workspace=ws)
        assert torch.equal(image, image_s) and torch.equal(n_contrib, nc_s)
        assert loss.item() == pytest.approx(loss_s.item(), rel=1e-5)  # fp32 sums in another order
        e = rel_l2(grads.cpu().numpy(), grads_s.cpu().numpy())
        print("workspace %s: fused vs separate grads rel-L2 %.2e, longest list %d" %
              (ws_bytes, e, int((ranges[:, 1] - ranges[:, 0]).max().item())))
        assert e <= 1e-5


@pytest.mark.parametrize("case", CASES)
def test_tile_counts_path_matches_records_path(case):
    """With a tile-count array the projection writes no record for a culled
    row, and binning, compositing and the projection backward never read
    one (nor a culled row's gradient record): culled records and gradient
    records are pre-filled with a sentinel whose tile field is positive, and
    every result must equal the path without the array."""
    gs = _gs()
    o = oracle_side(case)
    n, V, W, H = o["n"], o["V"], o["W"], o["H"]
    params = _cuda(o["params"])
    rows = n * V
    sa = torch.empty((rows, 12), dtype=torch.float32, device="cuda")
    gs.gs_project(params, o["cams"], sa)
    sentinel = torch.full((rows, 12), 0x7F7F7F7F, dtype=torch.int32, device="cuda")
    sb = sentinel.clone().view(torch.float32)
    counts = torch.full((rows,), -5, dtype=torch.int32, device="cuda")
    gs.gs_project(params, o["cams"], sb, tile_counts=counts)
    rec_tiles = sa.view(torch.int32)[:, 11]
    assert torch.equal(counts, rec_tiles)
    vis = counts > 0
    assert int(vis.sum()) > 0
    assert case == "tiny" or int(vis.sum()) < rows  # the tiny scene culls nothing
    assert torch.equal(sb.view(torch.int32)[vis], sa.view(torch.int32)[vis])
    assert torch.equal(sb.view(torch.int32)[~vis], sentinel[~vis])
    # binning: identical lists
    cap = max(1, int(rec_tiles.to(torch.int64).sum().item()))
    T = gs.tiles_per_view(W, H)
    out = []
    for s, c in ((sa, None), (sb, counts)):
        ws = torch.zeros(gs.gs_bin_workspace_bytes(rows, cap), dtype=torch.uint8, device="cuda")
        keys = torch.empty(cap, dtype=torch.int64, device="cuda")
        vals = torch.empty(cap, dtype=torch.int32, device="cuda")
        ranges = torch.empty((V * T, 2), dtype=torch.int64, device="cuda")
        st, I = gs.gs_bin_and_sort(n, V, s, W, H, ws, cap, keys, vals, ranges, tile_counts=c)
        assert st == gs.GS_OK and I == cap
        out.append((keys, vals, ranges))
    assert all(torch.equal(a, b) for a, b in zip(out[0], out[1]))
    keys, vals, ranges = out[0]
    # fused compositing: same image, same gradients on visible rows, culled
    # gradient records untouched
    target = _cuda(o["target"])
    res = []
    for s, c in ((sa, None), (sb, counts)):
        image = torch.empty((V, 3, H, W), device="cuda")
        T_final = torch.empty((V, H, W), device="cuda")
        n_contrib = torch.empty((V, H, W), dtype=torch.int32, device="cuda")
        loss = torch.empty(1, device="cuda")
        grads = torch.full((rows, 12), 3.0, device="cuda")
        ws = torch.empty(gs.gs_rasterize_workspace_bytes(V, W, H, cap), dtype=torch.uint8,
                         device="cuda")
        gs.gs_rasterize_fused(n, V, s, W, H, vals, ranges, (0, 0, 0), target, image, T_final,
                              n_contrib, loss, grads, workspace=ws, tile_counts=c)
        res.append((image, T_final, n_contrib, loss, grads))
    (ia, ta, na, la, ga), (ib, tb, nb, lb, gb) = res
    assert torch.equal(ia, ib) and torch.equal(ta, tb) and torch.equal(na, nb)
    assert lb.item() == pytest.approx(la.item(), rel=1e-5)
    assert rel_l2(gb[vis].cpu().numpy(), ga[vis].cpu().numpy()) <= 1e-5
    assert torch.all(ga[~vis] == 0.0)
    # culled rows: zeroed only as the pair partner of a visible row (rows 2k, 2k+1)
    partner = torch.arange(rows, device="cuda") ^ 1
    pair_vis = vis | vis[partner.clamp(max=rows - 1)]
    assert torch.all(gb[~pair_vis] == 3.0) and torch.all(gb[~vis & pair_vis] == 0.0)
    # separate backward: the same
    g_img = torch.empty_like(ia)
    gs.gs_loss_l1(ia, target, torch.empty(1, device="cuda"), g_img)
    gsep = torch.full((rows, 12), 3.0, device="cuda")
    gs.gs_rasterize_bwd(n, V, sb, W, H, vals, ranges, (0, 0, 0), ta, na, g_img, gsep,
                        tile_counts=counts)
    assert rel_l2(gsep[vis].cpu().numpy(), ga[vis].cpu().numpy()) <= 1e-5
    assert torch.all(gsep[~pair_vis] == 3.0) and torch.all(gsep[~vis & pair_vis] == 0.0)
    # projection backward on identical visible inputs: bit for bit
    gc = ga.clone()
    gc[~vis] = float("nan")
    grad_a = torch.empty((59, n), device="cuda")
    grad_b = torch.full((59, n), 5.0, device="cuda")
    vis_a = torch.empty(n, dtype=torch.uint8, device="cuda")
    vis_b = torch.full((n,), 9, dtype=torch.uint8, device="cuda")
    gs.gs_project_bwd(params, o["cams"], sa, ga, grad_a, vis_a)
    gs.gs_project_bwd(params, o["cams"], sb, gc, grad_b, vis_b, tile_counts=counts)
    assert torch.equal(grad_a, grad_b)
    assert torch.equal(vis_a, vis_b)


def test_bin_and_sort_device_check_on_inconsistent_record():
    """A record whose tile count disagrees with its rectangle (records not
    made by gs_project) is reported, not trusted: the synchronous call
    returns GS_ERR_DEVICE_CHECK; the asynchronous one finishes with the row
    emitting nothing (its lists equal the oracle's without that row) and
    reports the check through the workspace status, which the next call
    clears."""
    import oracle
    gs = _gs()
    o = oracle_side("ragged2")
    n, V, W, H = o["n"], o["V"], o["W"], o["H"]
    rec = pack_records(o["pr"]).copy()
    tiles = rec.view(np.int32)[:, 11]
    bad = int(np.nonzero(tiles > 0)[0][5])
    rec.view(np.int32)[bad, 11] += 1
    cap = int(tiles.astype(np.int64).sum()) + 64
    with pytest.raises(gs.GSError) as e:
        _gpu_bin(gs, n, V, rec, W, H, capacity=cap)
    assert e.value.status == gs.GS_ERR_DEVICE_CHECK
    # the asynchronous call: same workspace shape, the row left out of the lists
    rows = n * V
    T = gs.tiles_per_view(W, H)
    ws = torch.zeros(gs.gs_bin_workspace_bytes(rows, cap), dtype=torch.uint8, device="cuda")
    keys = torch.empty(cap, dtype=torch.int64, device="cuda")
    vals = torch.empty(cap, dtype=torch.int32, device="cuda")
    ranges = torch.empty((V * T, 2), dtype=torch.int64, device="cuda")
    nd = torch.zeros(1, dtype=torch.int64, device="cuda")
    gs.gs_bin_and_sort_async(n, V, _cuda(rec), W, H, ws, cap, keys, vals, ranges, nd)
    assert gs.gs_workspace_status(ws) == gs.GS_ERR_DEVICE_CHECK
    radius = o["f32"]["radius"].copy()
    radius[bad] = 0
    keys_o, vals_o, ranges_o = oracle.bin_and_sort(n, V, o["f32"]["mean2d"].astype(np.float32),
                                                   radius, o["f32"]["depth"].astype(np.float32),
                                                   W, H)
    I = int(nd.item())
    assert I == keys_o.size
    assert np.array_equal(keys[:I].cpu().numpy().view(np.uint64), keys_o)
    assert np.array_equal(vals[:I].cpu().numpy().view(np.uint32), vals_o)
    assert np.array_equal(ranges.cpu().numpy(), ranges_o)
    # a consistent call on the same workspace is clean again
    good = pack_records(o["pr"])
    gs.gs_bin_and_sort_async(n, V, _cuda(good), W, H, ws, cap, keys, vals, ranges, nd)
    assert gs.gs_workspace_status(ws) == gs.GS_OK
    assert int(nd.item()) == o["keys"].size


@pytest.mark.parametrize("case", ["ragged2", "small"])
@pytest.mark.parametrize("with_ws", [True, False])
def test_zero_grads_then_fused_acc_equals_fused(case, with_ws):
    """gs_zero_grads on a second stream (ordered by events) followed by
    gs_rasterize_fused_acc gives what gs_rasterize_fused gives, with and
    without tile counts, with either grid of the zeroing; the
    accumulate-only call adds to what it finds."""
    gs = _gs()
    o = oracle_side(case)
    n, V, W, H = o["n"], o["V"], o["W"], o["H"]
    splats, vals, ranges, _, _, _ = _gpu_fwd(gs, o)
    target = _cuda(o["target"])
    counts = torch.from_numpy(pack_records(o["pr"]).view(np.int32)[:, 11].copy()).cuda()
    ws = None
    if with_ws:  # the backward walks the recorded pairs; without it, the boxes
        ws = torch.empty(gs.gs_rasterize_workspace_bytes(V, W, H, int(o["vals"].size)),
                         dtype=torch.uint8, device="cuda")
    for tc, beside in ((None, False), (None, True), (counts, False), (counts, True)):
        outs = []
        for split in (False, True):
            image = torch.empty((V, 3, H, W), device="cuda")
            T_final = torch.empty((V, H, W), device="cuda")
            n_contrib = torch.empty((V, H, W), dtype=torch.int32, device="cuda")
            loss = torch.empty(1, device="cuda")
            grads = torch.full((n * V, 12), 5.0, device="cuda")
            if split:
                main = torch.cuda.current_stream()
                side = torch.cuda.Stream()
                side.wait_stream(main)
                gs.gs_zero_grads(n, V, grads, side, tile_counts=tc, beside=beside)
                main.wait_stream(side)
                gs.gs_rasterize_fused(n, V, splats, W, H, vals, ranges, (0, 0, 0), target, image,
                                      T_final, n_contrib, loss, grads, workspace=ws,
                                      tile_counts=tc, accumulate=True)
            else:
                gs.gs_rasterize_fused(n, V, splats, W, H, vals, ranges, (0, 0, 0), target, image,
                                      T_final, n_contrib, loss, grads, workspace=ws,
                                      tile_counts=tc)
            torch.cuda.synchronize()
            outs.append((image, T_final, n_contrib, loss, grads))
        (i0, t0, c0, l0, g0), (i1, t1, c1, l1, g1) = outs
        assert torch.equal(i0, i1) and torch.equal(t0, t1) and torch.equal(c0, c1)
        assert l1.item() == pytest.approx(l0.item(), rel=1e-6)
        vis = torch.ones(n * V, dtype=torch.bool, device="cuda") if tc is None else tc > 0
        assert rel_l2(g1[vis].cpu().numpy(), g0[vis].cpu().numpy()) <= 1e-6
    # without a zeroing first the call adds to the records as they stand
    grads = torch.zeros((n * V, 12), device="cuda")
    gs.gs_rasterize_fused(n, V, splats, W, H, vals, ranges, (0, 0, 0), target, image, T_final,
                          n_contrib, loss, grads, workspace=ws)
    twice = grads.clone()
    gs.gs_rasterize_fused(n, V, splats, W, H, vals, ranges, (0, 0, 0), target, image, T_final,
                          n_contrib, loss, twice, workspace=ws, accumulate=True)
    assert rel_l2(twice.cpu().numpy(), 2 * grads.cpu().numpy()) <= 1e-6
