"""Ten training steps of the 200k-Gaussian, 1024x768 configuration against
the oracle ("On Scaling Up 3D Gaussian Splatting Training", comparison to
the original implementation: loss and gradients match at every step).

The oracle runs its chain once from the fp32 start: fp64 parameters and Adam
moments, steps t = 1..10.  Two comparisons per step.

Lockstep, on identical stage inputs: the library gets the oracle's state
after step t - 1 -- its parameters and moments rounded to fp32, the projected
rows of those fp32 parameters rounded to the fp32 records, the step number --
and runs the rest of its step: binning, fused compositing with the L1 loss,
projection backward, and Adam with the carried moments and the bias
correction of step t.  The oracle evaluates its step at the same fp32
parameters and composites the same fp32 records; its Adam update applies to
its fp64 parameters.  Image, gradients and
the updated parameters and moments must meet the stated bars: image max-abs
1e-5 and loss relative 1e-5 from the fused call, relative L2 1e-4 per
parameter group and for the Adam results.  As in the per-call comparisons,
a pixel whose threshold decisions lie within 1e-5 of a cut-off may be decided
either way, and so may the sign of the L1 gradient of a channel whose colour
lies within 1e-5 of its target (about three channels per step here); their
image gradient is set to zero on both sides (the library's through its
separate backward call, whose gradients equal the fused call's), so that
they move no gradient; and a Gaussian whose projection the
oracle flags in some view (a radius, rectangle, clamp or depth within 1e-4 of
a discontinuity) is left out of the gradient comparison, as in the per-call
projection comparison.

Free-running: the library's own chain of ten steps, its projection included,
against the oracle's own chain (its fp64 projection and unmasked image
gradient, its own parameters and moments).
Two effects keep this chain from matching the oracle pixel by pixel: the fp32
projection moves a steep splat's alpha at its rim by ~1e-5 relative, enough
to take a decision across the 1/255 cut-off; and Adam's first update,
-lr g / (|g| + eps), steps by lr against the sign of g, so where a gradient
lies within rounding of zero the two chains step in opposite directions.  It
is held to the loss (relative 1e-5) and the parameters (relative L2 1e-4) at
every step, and its update p_t - p_0 to relative L2 1e-3."""
import os

import numpy as np
import pytest
import torch

import scenes
from parity_util import (ADAM_REL_L2, GRAD_REL_L2, IMAGE_MAX_ABS, MARGIN, PARAM_GROUPS, f32_cams,
                         feats32, grads_to_rows, pack_records, rel_l2, rows_to_grads)

pytestmark = pytest.mark.gpu

FREE_LOSS_REL = 1e-5
FREE_PARAM_REL_L2 = 1e-4
FREE_UPDATE_REL_L2 = 1e-3


def _decided(fw, target):
    """Channels whose image gradient both sides decide alike: the pixel's
    threshold decisions clear of the cut-offs, the colour clear of the target
    (the L1 gradient's sign)."""
    return (fw["margin"] > MARGIN)[:, None] & (np.abs(fw["image"] - target) > IMAGE_MAX_ABS)


def _oracle_step(oracle, p64, cams, target, threads):
    """The oracle's step with the compositing on the fp32-rounded projected
    rows (the library's record format), as in the per-call comparisons; the
    image gradient is zeroed at flagged pixels.  Returns the projection, the
    forward, the loss, the masked image gradient (fp32) and the gradient."""
    n, V = p64.shape[1], len(cams)
    W, H = cams[0]["width"], cams[0]["height"]
    pr = oracle.project(p64, cams, threads=threads)
    f32 = feats32(pr)
    _, vals, ranges = oracle.bin_and_sort(n, V, f32["mean2d"].astype(np.float32), f32["radius"],
                                          f32["depth"].astype(np.float32), W, H, threads=threads)
    fw = oracle.raster_fwd(n, V, W, H, f32, vals, ranges, threads=threads)
    loss, g_img = oracle.loss_l1(fw["image"], target)
    keep = _decided(fw, target)
    g_img = (g_img * keep).astype(np.float32)
    g2 = oracle.raster_bwd(n, V, W, H, f32, vals, ranges, g_img, threads=threads)
    grad, _ = oracle.project_bwd(p64, cams, grads_to_rows(rows_to_grads(g2)), threads=threads)
    return pr, fw, loss, g_img, grad


def test_small_200k_ten_steps_against_oracle():
    import __graft_entry__
    __graft_entry__.build()
    import gaussian_splatting_differentiable_gs_gb300 as gs
    import oracle
    cfg = scenes.make("small_200k_1024x768")
    assert cfg["steps"] == 10
    params, cams, target = cfg["params"], f32_cams(cfg["cams"]), cfg["target"]
    lr = cfg["lr"]
    threads = min(32, os.cpu_count() or 1)
    tgt = torch.from_numpy(target).cuda()
    lock = gs.TrainStep(torch.from_numpy(params).cuda(), cams, tgt, lr=lr, fused=True)
    free = gs.TrainStep(torch.from_numpy(params).cuda(), cams, tgt, lr=lr, fused=True)
    po = params.astype(np.float64)
    mo, vo = np.zeros_like(po), np.zeros_like(po)
    pf = params.astype(np.float64)  # the oracle's own chain, for the free-running comparison
    mf, vf = np.zeros_like(pf), np.zeros_like(pf)
    n, V = params.shape[1], len(cams)
    for t in range(1, cfg["steps"] + 1):
        p32 = po.astype(np.float32)
        pr, fw, loss_o, g_img_o, grad_o = _oracle_step(oracle, p32.astype(np.float64), cams,
                                                       target, threads)
        clean = (pr["flags"].reshape(V, n) == 0).all(axis=0)
        # lockstep: the oracle's state after step t - 1 into the library
        lock.params.copy_(torch.from_numpy(p32))
        lock.m.copy_(torch.from_numpy(mo.astype(np.float32)))
        lock.v.copy_(torch.from_numpy(vo.astype(np.float32)))
        lock.t = t - 1
        rec = pack_records(pr)
        lock.splats.copy_(torch.from_numpy(rec))
        lock.tile_counts.copy_(torch.from_numpy(np.ascontiguousarray(rec.view(np.int32)[:, 11])))
        lock.bin_and_sort()
        lock.rasterize_fused()
        # the gradient with the flagged pixels' image gradient zeroed
        loss_fused = lock.loss.item()
        lock.loss_l1()
        keep = _decided(fw, target)
        lock.dL_dimage.mul_(torch.from_numpy(np.ascontiguousarray(keep, np.float32)).cuda())
        lock.rasterize_bwd()
        lock.project_bwd()
        free.project()
        free.bin_and_sort()
        free.rasterize_fused()
        free.project_bwd()
        ok = fw["margin"] > MARGIN
        err = np.abs(lock.image.cpu().numpy() - fw["image"]).max(axis=1)[ok].max()
        gg = lock.grad.cpu().numpy()
        gerr = {name: rel_l2(gg[a:b, clean], grad_o[a:b, clean])
                for name, (a, b) in PARAM_GROUPS.items()}
        lock.adam()
        free.adam()
        oracle.adam(po, grad_o, mo, vo, t, lr, threads=threads)
        loss_f, grad_f, _, _ = oracle.train_step_grads(pf, cams, target, threads=threads)
        oracle.adam(pf, grad_f, mf, vf, t, lr, threads=threads)
        perr = rel_l2(lock.params.cpu().numpy(), po)
        merr = rel_l2(lock.m.cpu().numpy(), mo)
        verr = rel_l2(lock.v.cpu().numpy(), vo)
        p_free = free.params.cpu().numpy()
        f_perr = rel_l2(p_free, pf)
        f_uerr = rel_l2(p_free.astype(np.float64) - params, pf - params)
        print("step %2d lockstep: loss %.7f / %.7f image %.2e (%d flagged) grad %.2e (%d flagged "
              "Gaussians left out) params %.2e m %.2e v %.2e | free: loss %.7f params %.2e "
              "updates %.2e"
              % (t, loss_fused, loss_o, err, int((~ok).sum()), max(gerr.values()),
                 int((~clean).sum()), perr, merr, verr, free.loss.item(), f_perr, f_uerr))
        assert loss_fused == pytest.approx(loss_o, rel=1e-5)
        assert err <= IMAGE_MAX_ABS
        for name, e in gerr.items():
            assert e <= GRAD_REL_L2, (t, name)
        assert perr <= ADAM_REL_L2 and merr <= ADAM_REL_L2 and verr <= ADAM_REL_L2
        assert free.loss.item() == pytest.approx(loss_f, rel=FREE_LOSS_REL)
        assert f_perr <= FREE_PARAM_REL_L2 and f_uerr <= FREE_UPDATE_REL_L2
    assert lock.t == 10 and free.t == 10
