"""GPU parity at full size on the benchmark workload: 3,000,000 Gaussians in
256 clusters, 4 cameras at 1920x1080 (the configuration bench.py times, with
the same library calls and launch shapes).

The oracle projects all 12M (view, Gaussian) rows and bins all intersections;
compositing (forward and backward) is compared on sampled tiles the oracle
computes one by one: 64 random non-empty tiles, the tile with the longest
list, and tiles on the ragged bottom row and right column.  For the backward,
the image gradient is zero outside the sampled tiles, so the library's
full-image backward accumulates exactly the sampled tiles' contributions."""
import numpy as np
import pytest
import torch

import scenes
from parity_util import (ADAM_REL_L2, GRAD_REL_L2, IMAGE_MAX_ABS, MARGIN, flagged_allowance,
                         PARAM_GROUPS, f32_cams, feats32, grads_to_rows, pack_records, rel_l2,
                         rows_to_grads, unpack_records)

pytestmark = pytest.mark.gpu


def _gs():
    import __graft_entry__
    __graft_entry__.build()
    import gaussian_splatting_differentiable_gs_gb300 as gs
    return gs


def _pick_tiles(ranges, V, tiles_x, tiles_y, rng):
    lens = ranges[:, 1] - ranges[:, 0]
    nonempty = np.nonzero(lens > 0)[0]
    sel = set(rng.choice(nonempty, 64, replace=False).tolist())
    sel.add(int(np.argmax(lens)))
    T = tiles_x * tiles_y
    for v in range(V):
        bottom = [v * T + (tiles_y - 1) * tiles_x + x for x in range(tiles_x)]
        right = [v * T + y * tiles_x + tiles_x - 1 for y in range(tiles_y)]
        for group in (bottom, right):
            cand = [t for t in group if lens[t] > 0]
            if cand:
                sel.add(int(cand[len(cand) // 2]))
    return np.array(sorted(sel), np.int64)


def _tile_pixels(sel, V, W, H, tiles_x):
    T = tiles_x * ((H + 15) // 16)
    mask = np.zeros((V, H, W), bool)
    for f in sel:
        v, t = divmod(int(f), T)
        ty, tx = divmod(t, tiles_x)
        mask[v, ty * 16:(ty + 1) * 16, tx * 16:(tx + 1) * 16] = True
    return mask


def test_ring_3m_full_size():
    import oracle
    gs = _gs()
    cfg = scenes.make("ring_3m_4x1080p")
    params, cams, target = cfg["params"], f32_cams(cfg["cams"]), cfg["target"]
    n, V = params.shape[1], len(cams)
    W, H = cams[0]["width"], cams[0]["height"]
    tiles_x, tiles_y = (W + 15) // 16, (H + 15) // 16
    p64 = params.astype(np.float64)
    pr = oracle.project(p64, cams)
    f32 = feats32(pr)
    rec = pack_records(pr)

    # projection, every row
    dev_params = torch.from_numpy(params).cuda()
    splats = torch.empty((n * V, 12), dtype=torch.float32, device="cuda")
    gs.gs_project(dev_params, cams, splats)
    g = unpack_records(splats.cpu().numpy())
    flagged = pr["flags"] != 0
    assert not (((g["radius"] > 0) != (pr["radius"] > 0)) & ~flagged).any()
    ok = (g["radius"] > 0) & (pr["radius"] > 0) & ~flagged
    assert np.array_equal(g["radius"][ok], pr["radius"][ok])
    assert np.array_equal(g["tiles"][ok], pr["tiles"][ok])
    for f in ("mean2d", "conic", "color", "opacity", "depth"):
        assert rel_l2(g[f][ok], pr[f][ok]) < 1e-5, f
    del g, splats

    # binning: every intersection, bit for bit, from the oracle's projection
    keys_o, vals_o, ranges_o = oracle.bin_and_sort(n, V, rec[:, 0:2], f32["radius"], rec[:, 9], W, H)
    I = keys_o.size
    ws = torch.zeros(gs.gs_bin_workspace_bytes(n * V, I), dtype=torch.uint8, device="cuda")
    keys = torch.empty(I, dtype=torch.int64, device="cuda")
    vals = torch.empty(I, dtype=torch.int32, device="cuda")
    ranges = torch.empty((V * tiles_x * tiles_y, 2), dtype=torch.int64, device="cuda")
    rec_d = torch.from_numpy(rec).cuda()
    st, I_gpu = gs.gs_bin_and_sort(n, V, rec_d, W, H, ws, I, keys, vals, ranges)
    assert st == gs.GS_OK and I_gpu == I
    assert np.array_equal(keys.cpu().numpy().view(np.uint64), keys_o)
    assert np.array_equal(vals.cpu().numpy().view(np.uint32), vals_o)
    assert np.array_equal(ranges.cpu().numpy(), ranges_o)
    del keys, ws

    # compositing forward on sampled tiles
    rng = np.random.default_rng(2024)
    sel = _pick_tiles(ranges_o, V, tiles_x, tiles_y, rng)
    fw = oracle.raster_fwd(n, V, W, H, f32, vals_o, ranges_o, tile_sel=sel)
    image = torch.empty((V, 3, H, W), device="cuda")
    T_final = torch.empty((V, H, W), device="cuda")
    n_contrib = torch.empty((V, H, W), dtype=torch.int32, device="cuda")
    gs.gs_rasterize_fwd(n, V, rec_d, W, H, vals, ranges, (0, 0, 0), image, T_final, n_contrib)
    mask = _tile_pixels(sel, V, W, H, tiles_x)
    okp = mask & (fw["margin"] > MARGIN)
    err = np.abs(image.cpu().numpy() - fw["image"]).max(axis=1)
    pairs = int(fw["pairs"][mask].sum())
    allow = flagged_allowance(mask.sum(), pairs)
    print("sampled tiles %d, pixels %d, pairs %d, flagged %d (bound %.1f), max err %.2e" %
          (sel.size, mask.sum(), pairs, (mask & ~okp).sum(), allow, err[okp].max()))
    assert (mask & ~okp).sum() <= allow
    assert err[okp].max() <= IMAGE_MAX_ABS
    assert np.array_equal(n_contrib.cpu().numpy()[okp], fw["n_contrib"][okp])
    # the roofline's work counts on the sampled tiles, pixel by pixel
    counts = torch.zeros(2, dtype=torch.int64, device="cuda")
    pix = torch.empty((2, V, H, W), dtype=torch.int32, device="cuda")
    gs.gs_rasterize_fwd_counted(n, V, rec_d, W, H, vals, ranges, (0, 0, 0), image, T_final,
                                n_contrib, counts, pixel_counts=pix)
    pc = pix.cpu().numpy().astype(np.int64)
    assert np.array_equal(pc[0][okp], fw["pairs"][okp])
    assert np.array_equal(pc[1][okp], fw["included"][okp])
    c = counts.cpu().numpy()
    assert c[0] == pc[0].sum() and c[1] == pc[1].sum()
    print("counted: tested %d composited %d over the image; sampled tiles equal the oracle's "
          "%d / %d" % (c[0], c[1], fw["pairs"][okp].sum(), fw["included"][okp].sum()))
    del pix

    # compositing backward restricted to the sampled tiles
    _, g_img = oracle.loss_l1(fw["image"], target)
    g_img = (g_img * mask[:, None]).astype(np.float32)
    g2 = oracle.raster_bwd(n, V, W, H, f32, vals_o, ranges_o, g_img, tile_sel=sel)
    grads = torch.empty((n * V, 12), device="cuda")
    gs.gs_rasterize_bwd(n, V, rec_d, W, H, vals, ranges, (0, 0, 0), T_final, n_contrib,
                        torch.from_numpy(g_img).cuda(), grads)
    gg = grads_to_rows(grads.cpu().numpy())
    for f in ("mean2d", "conic", "opacity", "color"):
        e = rel_l2(gg[f], g2[f])
        print("raster bwd %s rel-L2 %.2e" % (f, e))
        assert e <= GRAD_REL_L2, f
    del grads

    # the fused call over every tile against the three separate calls
    target_d = torch.from_numpy(target).cuda()
    image_s = torch.empty((V, 3, H, W), device="cuda")
    T_s = torch.empty((V, H, W), device="cuda")
    nc_s = torch.empty((V, H, W), dtype=torch.int32, device="cuda")
    gs.gs_rasterize_fwd(n, V, rec_d, W, H, vals, ranges, (0, 0, 0), image_s, T_s, nc_s)
    loss_s = torch.empty(1, device="cuda")
    g_img_s = torch.empty_like(image_s)
    gs.gs_loss_l1(image_s, target_d, loss_s, g_img_s)
    grads_s = torch.empty((n * V, 12), device="cuda")
    gs.gs_rasterize_bwd(n, V, rec_d, W, H, vals, ranges, (0, 0, 0), T_s, nc_s, g_img_s, grads_s)
    del g_img_s
    image_f, T_f, nc_f = torch.empty_like(image_s), torch.empty_like(T_s), torch.empty_like(nc_s)
    loss_f = torch.empty(1, device="cuda")
    grads_f = torch.empty((n * V, 12), device="cuda")
    ws = torch.empty(gs.gs_rasterize_workspace_bytes(V, W, H, I), dtype=torch.uint8, device="cuda")
    gs.gs_rasterize_fused(n, V, rec_d, W, H, vals, ranges, (0, 0, 0), target_d, image_f, T_f, nc_f,
                          loss_f, grads_f, workspace=ws)
    del ws
    assert torch.equal(image_f, image_s) and torch.equal(T_f, T_s) and torch.equal(nc_f, nc_s)
    assert loss_f.item() == pytest.approx(loss_s.item(), rel=1e-5)  # fp32 sums in another order
    e = ((grads_f - grads_s).norm() / grads_s.norm()).item()
    print("fused vs separate: loss %.6f / %.6f, grads rel-L2 %.2e" % (loss_f.item(), loss_s.item(), e))
    assert e <= 1e-5
    del image_s, T_s, nc_s, grads_s, image_f, T_f, nc_f, grads_f, target_d

    # projection backward, every Gaussian, from the oracle's row gradients
    g2_32 = grads_to_rows(rows_to_grads(g2))
    grad_o, visible_o = oracle.project_bwd(p64, cams, g2_32)
    grad = torch.empty((59, n), device="cuda")
    visible = torch.empty(n, dtype=torch.uint8, device="cuda")
    gs.gs_project_bwd(dev_params, cams, rec_d, torch.from_numpy(rows_to_grads(g2_32)).cuda(), grad,
                      visible)
    gnp = grad.cpu().numpy()
    for name, (a, b) in PARAM_GROUPS.items():
        e = rel_l2(gnp[a:b], grad_o[a:b])
        print("project bwd %s rel-L2 %.2e" % (name, e))
        assert e <= GRAD_REL_L2, name
    assert np.array_equal(visible.cpu().numpy(), visible_o)

    # Adam over all 59 x 3M parameters
    m = torch.zeros_like(dev_params)
    v = torch.zeros_like(dev_params)
    gs.gs_adam_step(dev_params, torch.from_numpy(grad_o.astype(np.float32)).cuda(), m, v, 1,
                    cfg["lr"])
    po = p64.copy()
    mo, vo = np.zeros_like(po), np.zeros_like(po)
    oracle.adam(po, grad_o.astype(np.float32).astype(np.float64), mo, vo, 1, cfg["lr"])
    assert rel_l2(dev_params.cpu().numpy(), po) <= ADAM_REL_L2
