"""GPU parity on the two largest configurations, at full size, on sampled
outputs the oracle can compute one by one.

dense_20m_4k: 20,000,000 Gaussians in 64 tight clusters, one 3840x2160 view;
3.4e9 intersections (80 GB of sort buffers).  The oracle projects every row;
the library bins the oracle's fp32 records and the sampled tiles' lists must
equal the oracle's brute-force lists bit for bit.

city_100m_8x1080p: 100,000,000 Gaussians, 8 street cameras, sparse Adam.  The
library runs its own whole step.  The oracle projects a sample of Gaussians
(compared row by row) and, chunk by chunk over all Gaussians, the rows that
touch the sampled tiles; the library's lists on those tiles must equal the
oracle's up to rows the oracle flags as within 1e-4 of a rounding boundary,
with the common rows in the same order.  Sparse Adam is checked on sampled
columns, untouched columns bit for bit.

Compositing (forward and backward) is compared on identical inputs: the rows
of the sampled tiles are renumbered compactly and both sides composite those
tiles from the same fp32 records and lists."""
import os

import numpy as np
import pytest
import torch

import scenes
from parity_util import (ADAM_REL_L2, GRAD_REL_L2, IMAGE_MAX_ABS, MARGIN, PARAM_GROUPS,
                         f32_cams, feats32, flagged_allowance, grads_to_rows, pack_records, rel_l2,
                         rows_to_grads, unpack_records)

pytestmark = pytest.mark.gpu
THREADS = min(16, os.cpu_count() or 1)


def _gs():
    import __graft_entry__
    __graft_entry__.build()
    import gaussian_splatting_differentiable_gs_gb300 as gs
    return gs


def _grid(W, H):
    tx, ty = (W + 15) // 16, (H + 15) // 16
    return tx, ty, tx * ty


def _tile_mask(sel, V, W, H):
    tx, _, T = _grid(W, H)
    mask = np.zeros((V, H, W), bool)
    for f in sel:
        v, t = divmod(int(f), T)
        y, x = divmod(t, tx)
        mask[v, y * 16:(y + 1) * 16, x * 16:(x + 1) * 16] = True
    return mask


def _compact(sel, lists, V, T, rows_of):
    """Renumber the Gaussians of the sampled tiles' lists per view.
    lists: flat tile -> ordered Gaussian ids; rows_of(view, ids) -> (records
    [k][12] f32, features dict of k rows).  Returns n_c, records [V*n_c][12],
    features over V*n_c rows, vals, ranges (library layout over all tiles)."""
    per_view = {v: np.unique(np.concatenate([lists[f] for f in sel if f // T == v] or
                                            [np.zeros(0, np.int64)])) for v in range(V)}
    n_c = max(1, max(ids.size for ids in per_view.values()))
    rec = np.zeros((V * n_c, 12), np.float32)
    feats = {k: np.zeros((V * n_c,) + s) for k, s in (("mean2d", (2,)), ("conic", (3,)),
                                                     ("opacity", ()), ("color", (3,)))}
    for v, ids in per_view.items():
        if ids.size == 0:
            continue
        r, f = rows_of(v, ids)
        rec[v * n_c:v * n_c + ids.size] = r
        for k in feats:
            feats[k][v * n_c:v * n_c + ids.size] = f[k]
    vals, ranges, off = [], np.zeros((V * T, 2), np.int64), 0
    for f in sel:
        ids = lists[f]
        loc = np.searchsorted(per_view[f // T], ids)
        vals.append(loc.astype(np.uint32))
        ranges[f] = (off, off + ids.size)
        off += ids.size
    return n_c, rec, feats, np.concatenate(vals), ranges


def _raster_parity(gs, oracle, n_c, V, W, H, rec, feats, vals, ranges, sel, target):
    """Compositing forward and backward of the sampled tiles on identical inputs."""
    rec_d = torch.from_numpy(rec).cuda()
    vals_d = torch.from_numpy(vals.view(np.int32).copy()).cuda()
    ranges_d = torch.from_numpy(ranges).cuda()
    fw = oracle.raster_fwd(n_c, V, W, H, feats, vals, ranges, tile_sel=sel)
    image = torch.zeros((V, 3, H, W), device="cuda")
    T_final = torch.ones((V, H, W), device="cuda")
    n_contrib = torch.zeros((V, H, W), dtype=torch.int32, device="cuda")
    gs.gs_rasterize_fwd(n_c, V, rec_d, W, H, vals_d, ranges_d, (0, 0, 0), image, T_final, n_contrib)
    mask = _tile_mask(sel, V, W, H)
    ok = mask & (fw["margin"] > MARGIN)
    err = np.abs(image.cpu().numpy() - fw["image"]).max(axis=1)
    lens = ranges[sel, 1] - ranges[sel, 0]
    pairs = int(fw["pairs"][mask].sum())
    allow = flagged_allowance(mask.sum(), pairs)
    nc = n_contrib.cpu().numpy()
    worst = np.unravel_index(np.argmax(np.where(ok, err, -1.0)), err.shape)
    print("tiles %d (list lengths %d..%d) pixels %d pairs %d flagged %d (bound %.1f) max err %.2e" %
          (sel.size, lens.min(), lens.max(), mask.sum(), pairs, (mask & ~ok).sum(), allow,
           err[ok].max()))
    print("worst pixel %s: n_contrib %d / %d, T_final %.6e / %.6e, margin %.2e, pairs %d" %
          (tuple(int(i) for i in worst), nc[worst], fw["n_contrib"][worst],
           T_final.cpu().numpy()[worst], fw["T_final"][worst], fw["margin"][worst],
           fw["pairs"][worst]))
    assert (mask & ~ok).sum() <= allow
    assert err[ok].max() <= IMAGE_MAX_ABS
    assert np.array_equal(nc[ok], fw["n_contrib"][ok])
    _, g_img = oracle.loss_l1(fw["image"], target)
    g_img = (g_img * mask[:, None]).astype(np.float32)
    g2 = oracle.raster_bwd(n_c, V, W, H, feats, vals, ranges, g_img, tile_sel=sel)
    grads = torch.empty((n_c * V, 12), device="cuda")
    gs.gs_rasterize_bwd(n_c, V, rec_d, W, H, vals_d, ranges_d, (0, 0, 0), T_final, n_contrib,
                        torch.from_numpy(g_img).cuda(), grads)
    gg = grads_to_rows(grads.cpu().numpy())
    for f in ("mean2d", "conic", "opacity", "color"):
        e = rel_l2(gg[f], g2[f])
        print("raster bwd %s rel-L2 %.2e" % (f, e))
        assert e <= GRAD_REL_L2, f


def test_dense_20m_4k():
    import oracle
    gs = _gs()
    cfg = scenes.make("dense_20m_4k")
    params, cams, target = cfg["params"], f32_cams(cfg["cams"]), cfg["target"]
    n, V = params.shape[1], 1
    W, H = cams[0]["width"], cams[0]["height"]
    tx, ty, T = _grid(W, H)
    pr = oracle.project(params.astype(np.float64), cams, threads=THREADS)
    f32 = feats32(pr)
    rec = pack_records(pr)
    m32, d32 = rec[:, 0:2].copy(), rec[:, 9].copy()
    I = oracle.count_isect(m32, f32["radius"], W, H)
    print("intersections", I)
    # tiles under random visible means (dense), plus the ragged corner and random ones
    rng = np.random.default_rng(44)
    vis = np.nonzero(f32["radius"] > 0)[0]
    sel = {int(min(max(int(m32[r, 1] // 16), 0), ty - 1) * tx + min(max(int(m32[r, 0] // 16), 0), tx - 1))
           for r in rng.choice(vis, 12, replace=False)}
    sel |= {T - 1, int(rng.integers(0, T)), int(rng.integers(0, T))}
    sel = np.array(sorted(sel), np.int64)
    svals, sranges = oracle.bin_select(n, V, m32, f32["radius"], d32, W, H, sel)

    # binning of every intersection by the library; sampled tiles bit for bit
    rec_d = torch.from_numpy(rec).cuda()
    ws = torch.zeros(gs.gs_bin_workspace_bytes(n * V, I), dtype=torch.uint8, device="cuda")
    keys = torch.empty(I, dtype=torch.int64, device="cuda")
    vals = torch.empty(I, dtype=torch.int32, device="cuda")
    ranges = torch.empty((V * T, 2), dtype=torch.int64, device="cuda")
    st, I_gpu = gs.gs_bin_and_sort(n, V, rec_d, W, H, ws, I, keys, vals, ranges)
    assert st == gs.GS_OK and I_gpu == I
    del ws
    rg = ranges.cpu().numpy()
    assert rg[:, 1].max() == I and np.all(rg[:, 1] >= rg[:, 0])
    lists = {}
    for i, f in enumerate(sel):
        a, b = rg[f]
        sa, sb = sranges[i]
        assert b - a == sb - sa, f
        assert np.array_equal(vals[a:b].cpu().numpy().view(np.uint32), svals[sa:sb])
        k = keys[a:b].cpu().numpy().view(np.uint64)
        assert np.all(k >> np.uint64(32) == np.uint64(f)) and np.all(k[1:] >= k[:-1])
        lists[int(f)] = svals[sa:sb].astype(np.int64)
    idx = torch.arange(0, I - 1, max(1, I // 100_000), device="cuda")
    assert np.all(keys[idx + 1].cpu().numpy().view(np.uint64) >= keys[idx].cpu().numpy().view(np.uint64))
    del keys, vals, rec_d

    def rows_of(v, ids):
        r = v * n + ids
        return rec[r], {k: f32[k][r] for k in ("mean2d", "conic", "opacity", "color")}

    n_c, rec_c, feats_c, vals_c, ranges_c = _compact(sel, lists, V, T, rows_of)
    _raster_parity(gs, oracle, n_c, V, W, H, rec_c, feats_c, vals_c, ranges_c, sel, target)

    # projection backward and Adam on a slice of 1M Gaussians (row gradients
    # drawn at random: the chain rule is exercised for every visible row)
    a0, m = 7_000_000, 1_000_000
    g_rows = (rng.standard_normal((n * V, 12)) * 1e-6).astype(np.float32)
    g_rows[:, 9:] = 0
    dev_params = torch.from_numpy(params).cuda()
    grad = torch.empty((59, n), device="cuda")
    visible = torch.empty(n, dtype=torch.uint8, device="cuda")
    gs.gs_project_bwd(dev_params, cams, torch.from_numpy(rec).cuda(), torch.from_numpy(g_rows).cuda(),
                      grad, visible)
    sub = np.ascontiguousarray(params[:, a0:a0 + m].astype(np.float64))
    grows = grads_to_rows(g_rows)
    sg2 = {k: np.ascontiguousarray(v.reshape(V, n, -1)[:, a0:a0 + m].reshape(V * m, -1).squeeze())
           for k, v in grows.items()}
    grad_o, vis_o = oracle.project_bwd(sub, cams, sg2)
    gnp = grad[:, a0:a0 + m].cpu().numpy()
    for name, (a, b) in PARAM_GROUPS.items():
        e = rel_l2(gnp[a:b], grad_o[a:b])
        print("project bwd %s rel-L2 %.2e" % (name, e))
        assert e <= GRAD_REL_L2, name
    assert np.array_equal(visible[a0:a0 + m].cpu().numpy(), vis_o)
    mm, vv = torch.zeros_like(dev_params), torch.zeros_like(dev_params)
    gs.gs_adam_step(dev_params, grad, mm, vv, 1, cfg["lr"])
    po = sub.copy()
    mo, vo = np.zeros_like(po), np.zeros_like(po)
    oracle.adam(po, gnp.astype(np.float64), mo, vo, 1, cfg["lr"])
    assert rel_l2(dev_params[:, a0:a0 + m].cpu().numpy(), po) <= ADAM_REL_L2


def test_city_100m_sparse():
    import oracle
    gs = _gs()
    cfg = scenes.make("city_100m_8x1080p")
    params, cams, target = cfg["params"], f32_cams(cfg["cams"]), cfg["target"]
    n, V = params.shape[1], len(cams)
    W, H = cams[0]["width"], cams[0]["height"]
    tx, ty, T = _grid(W, H)
    dev_params = torch.from_numpy(params).cuda()
    step = gs.TrainStep(dev_params, cams, torch.from_numpy(target).cuda(), lr=cfg["lr"], sparse=True)
    step.forward()
    torch.cuda.synchronize()
    vis_rows = int((step.tile_counts > 0).sum().item())
    print("visible rows %d of %d (%.2f%% per view), intersections %d" %
          (vis_rows, n * V, 100.0 * vis_rows / (n * V), step.n_isect))

    # projection of a sample of Gaussians, row by row
    rng = np.random.default_rng(55)
    gsel = np.sort(rng.choice(n, 200_000, replace=False))
    pr_s = oracle.project(params[:, gsel].astype(np.float64), cams, threads=THREADS)
    rows_d = torch.from_numpy((np.arange(V)[:, None] * n + gsel[None, :]).reshape(-1)).cuda()
    g = unpack_records(step.splats[rows_d].cpu().numpy())
    seen = step.tile_counts[rows_d].cpu().numpy() > 0  # culled rows have no record
    clean = pr_s["flags"] == 0
    assert not ((seen != (pr_s["radius"] > 0)) & clean).any()
    assert np.array_equal(g["tiles"][seen], step.tile_counts[rows_d].cpu().numpy()[seen])
    ok = seen & (pr_s["radius"] > 0) & clean
    assert ok.sum() > 1000
    assert np.array_equal(g["radius"][ok], pr_s["radius"][ok])
    for f in ("mean2d", "conic", "color", "opacity", "depth"):
        assert rel_l2(g[f][ok], pr_s[f][ok]) < 1e-5, f

    # the library's own lists on sampled tiles against the oracle's
    rg = step.ranges.cpu().numpy()
    nonempty = np.nonzero(rg[:, 1] > rg[:, 0])[0]
    sel = np.sort(rng.choice(nonempty, 16, replace=False))
    sel_t = [(int(f) // T, (int(f) % T) % tx, (int(f) % T) // tx) for f in sel]
    kept = {k: [] for k in ("id", "view", "flags")}
    kept_rec = []
    chunk = 4_000_000
    for a in range(0, n, chunk):
        b = min(n, a + chunk)
        pr = oracle.project(params[:, a:b].astype(np.float64), cams, threads=THREADS)
        rec = pack_records(pr)
        rad = rec.view(np.int32)[:, 10]
        keep = np.zeros(rec.shape[0], bool)
        view = np.repeat(np.arange(V), b - a)
        fr = rad.astype(np.float32)
        x0 = np.floor((rec[:, 0] - fr) / np.float32(16))
        x1 = np.ceil((rec[:, 0] + fr) / np.float32(16))
        y0 = np.floor((rec[:, 1] - fr) / np.float32(16))
        y1 = np.ceil((rec[:, 1] + fr) / np.float32(16))
        for v, sx, sy in sel_t:
            keep |= (rad > 0) & (view == v) & (x0 <= sx) & (sx < x1) & (y0 <= sy) & (sy < y1)
        idx = np.nonzero(keep)[0]
        kept["id"].append(idx % (b - a) + a)
        kept["view"].append(idx // (b - a))
        kept["flags"].append(pr["flags"][idx])
        kept_rec.append(rec[idx])
    kept = {k: np.concatenate(v) for k, v in kept.items()}
    kept_rec = np.concatenate(kept_rec)
    lists = {}
    for (v, sx, sy), f in zip(sel_t, sel):
        r = kept_rec
        rad = r.view(np.int32)[:, 10].astype(np.float32)
        inside = np.nonzero((kept["view"] == v) & (np.floor((r[:, 0] - rad) / np.float32(16)) <= sx) &
                            (sx < np.ceil((r[:, 0] + rad) / np.float32(16))) &
                            (np.floor((r[:, 1] - rad) / np.float32(16)) <= sy) &
                            (sy < np.ceil((r[:, 1] + rad) / np.float32(16))))[0]
        dbits = r[inside, 9].view(np.uint32)
        order = np.lexsort((kept["id"][inside], dbits))
        ora = kept["id"][inside][order]
        flagged = set(kept["id"][inside][kept["flags"][inside] != 0].tolist())
        a, b = rg[f]
        lib = step.vals[a:b].cpu().numpy().view(np.uint32).astype(np.int64)
        only_o = set(ora.tolist()) - set(lib.tolist())
        only_l = set(lib.tolist()) - set(ora.tolist())
        assert only_o <= flagged and len(only_l) <= len(flagged), (f, len(only_o), len(only_l))
        common = [i for i in ora.tolist() if i not in only_o]
        libc = [i for i in lib.tolist() if i not in only_l]
        assert len(common) == len(libc)
        if common != libc:  # only rows of (nearly) equal fp32 depth may swap
            dmap = dict(zip(kept["id"][inside].tolist(), dbits.tolist()))
            bad = [k for k in range(len(common)) if common[k] != libc[k]]
            assert all(abs(int(dmap[common[k]]) - int(dmap[libc[k]])) <= 4 for k in bad), f
        lists[int(f)] = ora

    # compositing on identical inputs (the oracle's rows of the sampled tiles)
    pos = {(int(v), int(i)): j for j, (v, i) in enumerate(zip(kept["view"], kept["id"]))}
    f32k = unpack_records(kept_rec)

    def rows_of(v, ids):
        j = np.array([pos[(v, int(i))] for i in ids], np.int64)
        return kept_rec[j], {k: f32k[k][j] for k in ("mean2d", "conic", "opacity", "color")}

    n_c, rec_c, feats_c, vals_c, ranges_c = _compact(sel, lists, V, T, rows_of)
    _raster_parity(gs, oracle, n_c, V, W, H, rec_c, feats_c, vals_c, ranges_c, sel, target)

    # the library's own backward and sparse Adam
    step.backward()
    step.update()
    torch.cuda.synchronize()
    visible = step.visible.cpu().numpy()
    vis_o = (pr_s["radius"].reshape(V, -1) > 0).any(axis=0).astype(np.uint8)
    amb = (pr_s["flags"].reshape(V, -1) != 0).any(axis=0)
    assert np.array_equal(visible[gsel][~amb], vis_o[~amb])
    print("visible Gaussians %.2f%%" % (100.0 * visible.mean()))
    cols_u = np.nonzero(visible == 0)[0]
    cu = np.sort(cols_u[rng.choice(cols_u.size, min(200_000, cols_u.size), replace=False)])
    assert np.array_equal(dev_params[:, torch.from_numpy(cu).cuda()].cpu().numpy(), params[:, cu])
    cols = np.nonzero(visible)[0]
    cs = np.sort(cols[rng.choice(cols.size, min(200_000, cols.size), replace=False)])
    csd = torch.from_numpy(cs).cuda()
    g_sel = step.grad[:, csd].cpu().numpy().astype(np.float64)
    po = np.ascontiguousarray(params[:, cs], dtype=np.float64)
    mo, vo = np.zeros_like(po), np.zeros_like(po)
    oracle.adam(po, g_sel, mo, vo, 1, cfg["lr"])
    assert rel_l2(dev_params[:, csd].cpu().numpy(), po) <= ADAM_REL_L2
