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
from parity_util import (ADAM_REL_L2, GRAD_REL_L2, IMAGE_MAX_ABS, MARGIN, MAX_FLAGGED_FRACTION,
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
    print("flagged pixel fraction %.2e, max err unflagged %.2e, flagged %.2e" %
          (frac, err[ok].max(), err[~ok].max() if (~ok).any() else 0.0))
    assert frac <= MAX_FLAGGED_FRACTION
    assert err[ok].max() <= IMAGE_MAX_ABS
    assert np.abs(T_final.cpu().numpy() - fw["T_final"])[ok].max() <= IMAGE_MAX_ABS
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


@pytest.mark.parametrize("sparse", [False, True])
def test_adam_matches_oracle(sparse):
    import oracle
    gs = _gs()
    rng = np.random.default_rng(11)
    n = 10_001
    p = rng.standard_normal((59, n)).astype(np.float32)
    m = np.zeros((59, n), np.float32)
    v = np.zeros((59, n), np.float32)
    P, M, Vv = _cuda(p), _cuda(m), _cuda(v)
    po, mo, vo = p.astype(np.float64), m.astype(np.float64), v.astype(np.float64)
    for t in range(1, 6):
        g = (rng.standard_normal((59, n)) * 10.0 ** rng.uniform(-6, -2, (59, n))).astype(np.float32)
        vis = (rng.random(n) < 0.4).astype(np.uint8) if sparse else None
        gs.gs_adam_step(P, _cuda(g), M, Vv, t, 1e-3, visible=None if vis is None else _cuda(vis))
        oracle.adam(po, g.astype(np.float64), mo, vo, t, 1e-3, visible=vis)
    assert rel_l2(P.cpu().numpy(), po) <= ADAM_REL_L2
    assert rel_l2(P.cpu().numpy() - p, po - p) <= 1e-3
    assert rel_l2(M.cpu().numpy(), mo) <= ADAM_REL_L2
    assert rel_l2(Vv.cpu().numpy(), vo) <= ADAM_REL_L2


@pytest.mark.parametrize("case", ["tiny", "ragged2"])
def test_train_step_end_to_end(case):
    """The library's own chain from the fp32 parameters against the oracle's
    chain: loss, image, gradients and the Adam result."""
    import oracle
    gs = _gs()
    o = oracle_side(case)
    params = o["params"]
    step = gs.TrainStep(_cuda(params), o["cams"], _cuda(o["target"]), lr=1e-3)
    step.forward()
    step.backward()
    loss_o, grad_o, vis_o, parts = oracle.train_step_grads(params.astype(np.float64), o["cams"],
                                                           o["target"])
    img = step.image.cpu().numpy()
    ok = parts["fwd"]["margin"] > 1e-4
    err = np.abs(img - parts["fwd"]["image"]).max(axis=1)[ok].max()
    print("e2e image max err %.2e, loss %.6f vs %.6f" % (err, step.loss.item(), loss_o))
    assert step.loss.item() == pytest.approx(loss_o, rel=1e-4)
    assert err <= 1e-4
    gg = step.grad.cpu().numpy()
    for name, (a, b) in PARAM_GROUPS.items():
        e = rel_l2(gg[a:b], grad_o[a:b])
        print("e2e %s grad rel-L2 %.2e" % (name, e))
        assert e <= 1e-3, name
    step.update()
    po = params.astype(np.float64)
    mo, vo = np.zeros_like(po), np.zeros_like(po)
    oracle.adam(po, grad_o, mo, vo, 1, 1e-3)
    assert rel_l2(step.params.cpu().numpy(), po) <= ADAM_REL_L2
