"""Morton reordering of the Gaussians on the GPU against the oracle: the
permutation bit for bit (its codes are integer decisions taken in fp32 on
both sides), the column gather bit for bit, and a training step on the
reordered scene against the oracle's step on the same renamed scene."""
import numpy as np
import pytest
import torch

import scenes
from parity_util import ADAM_REL_L2, PARAM_GROUPS, f32_cams, rel_l2

pytestmark = pytest.mark.gpu


def _gs():
    import __graft_entry__
    __graft_entry__.build()
    import gaussian_splatting_differentiable_gs_gb300 as gs
    return gs


def _gpu_perm(gs, params):
    p = torch.from_numpy(np.ascontiguousarray(params)).cuda()
    ws = torch.zeros(gs.gs_morton_workspace_bytes(p.shape[1]), dtype=torch.uint8, device="cuda")
    perm = torch.empty(p.shape[1], dtype=torch.int32, device="cuda")
    gs.gs_morton_order(p, ws, perm)
    assert gs.gs_workspace_status(ws) == gs.GS_OK
    return perm


@pytest.mark.parametrize("name", ["tiny_2k_256", "small_200k_1024x768", "ring_3m_4x1080p"])
def test_morton_order_matches_oracle(name):
    import oracle
    gs = _gs()
    params = scenes.make(name)["params"]
    perm = _gpu_perm(gs, params).cpu().numpy().view(np.uint32)
    perm_o = oracle.morton_order(params)
    assert np.array_equal(perm, perm_o)
    codes = oracle.morton_codes(params)[perm_o]
    assert np.all(codes[1:] >= codes[:-1])
    print("%s: %d Gaussians, %d distinct codes" % (name, params.shape[1], np.unique(codes).size))


def test_morton_order_stable_on_duplicates_and_ragged_sizes():
    """Means snapped to a coarse grid (many equal codes: ties keep index
    order), at sizes that leave ragged sort partitions."""
    import oracle
    gs = _gs()
    rng = np.random.default_rng(8)
    for n in (1, 2, 4095, 4097, 70_001):
        p = np.zeros((59, n), np.float32)
        p[0:3] = np.round(rng.uniform(-2, 2, (3, n)) * 2) / 2
        perm = _gpu_perm(gs, p).cpu().numpy().view(np.uint32)
        assert np.array_equal(perm, oracle.morton_order(p)), n


def test_gather_columns_exact():
    gs = _gs()
    rng = np.random.default_rng(4)
    src = rng.standard_normal((59, 10_007)).astype(np.float32)
    perm = rng.permutation(10_007).astype(np.uint32)
    dst = torch.empty((59, 10_007), device="cuda")
    gs.gs_gather_columns(torch.from_numpy(src).cuda(), torch.from_numpy(perm.view(np.int32)).cuda(),
                          dst)
    assert np.array_equal(dst.cpu().numpy(), src[:, perm])


def test_step_after_morton_reorder_matches_oracle():
    """A step on the reordered scene equals the oracle's step on the scene
    renamed the same way, and its gradient is the original one permuted."""
    import oracle
    gs = _gs()
    cfg = scenes.make("tiny_2k_256")
    params, cams, target = cfg["params"], f32_cams(cfg["cams"]), cfg["target"]
    base = gs.TrainStep(torch.from_numpy(params).cuda(), cams, torch.from_numpy(target).cuda(),
                        lr=1e-3, fused=True)
    base.step()
    step = gs.TrainStep(torch.from_numpy(params).cuda(), cams, torch.from_numpy(target).cuda(),
                        lr=1e-3, fused=True)
    perm = step.reorder_morton().cpu().numpy().view(np.uint32)
    assert np.array_equal(perm, oracle.morton_order(params))
    renamed = np.ascontiguousarray(params[:, perm])
    assert np.array_equal(step.params.cpu().numpy(), renamed)
    step.step()
    loss_o, grad_o, _, parts = oracle.train_step_grads(renamed.astype(np.float64), cams, target)
    assert step.loss.item() == pytest.approx(loss_o, rel=1e-4)
    g = step.grad.cpu().numpy()
    for name, (a, b) in PARAM_GROUPS.items():
        assert rel_l2(g[a:b], grad_o[a:b]) <= 1e-3, name
    # the same step as before the reorder, with the Gaussians renamed
    assert step.loss.item() == pytest.approx(base.loss.item(), rel=1e-5)  # atomic order
    e = rel_l2(g, base.grad.cpu().numpy()[:, perm])
    print("reordered vs original gradient rel-L2 %.2e" % e)
    assert e <= 1e-5
    po = renamed.astype(np.float64)
    mo, vo = np.zeros_like(po), np.zeros_like(po)
    oracle.adam(po, grad_o, mo, vo, 1, 1e-3)
    assert rel_l2(step.params.cpu().numpy(), po) <= ADAM_REL_L2
