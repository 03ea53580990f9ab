"""Pruning bounded by the per-tile working set, on the GPU against the oracle.

The importance pass (largest blending weight per row) is compared with the
oracle's within fp32 rounding; the mask, an integer decision, is compared
bit for bit on identical inputs (the oracle's fp32 importances, lists and
n_contrib go to both sides); the compaction bit for bit."""
import numpy as np
import pytest
import torch

import scenes
from parity_util import f32_cams, feats32, pack_records

pytestmark = pytest.mark.gpu

_cache = {}


def _gs():
    import __graft_entry__
    __graft_entry__.build()
    import gaussian_splatting_differentiable_gs_gb300 as gs
    return gs


def _oracle_case(name):
    if name in _cache:
        return _cache[name]
    import oracle
    cfg = scenes.make(name)
    params, cams = cfg["params"], f32_cams(cfg["cams"])
    n, V = params.shape[1], len(cams)
    W, H = cams[0]["width"], cams[0]["height"]
    pr = oracle.project(params.astype(np.float64), cams)
    f32 = feats32(pr)
    _, vals, ranges = oracle.bin_and_sort(n, V, f32["mean2d"].astype(np.float32), f32["radius"],
                                          f32["depth"].astype(np.float32), W, H)
    fw = oracle.raster_fwd(n, V, W, H, f32, vals, ranges, importance=True)
    out = dict(n=n, V=V, W=W, H=H, rec=pack_records(pr), vals=vals, ranges=ranges, fw=fw,
               params=params)
    _cache[name] = out
    return out


def _cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("name", ["tiny_2k_256", "small_200k_1024x768"])
def test_importance_matches_oracle(name):
    gs = _gs()
    o = _oracle_case(name)
    n, V, W, H = o["n"], o["V"], o["W"], o["H"]
    image = torch.empty((V, 3, H, W), device="cuda")
    T_final = torch.empty((V, H, W), device="cuda")
    n_contrib = torch.empty((V, H, W), dtype=torch.int32, device="cuda")
    imp = torch.full((n * V,), 5.0, device="cuda")
    gs.gs_rasterize_fwd_importance(n, V, _cuda(o["rec"]), W, H, _cuda(o["vals"].view(np.int32)),
                                   _cuda(o["ranges"]), (0, 0, 0), image, T_final, n_contrib, imp)
    g = imp.cpu().numpy().astype(np.float64)
    ref = o["fw"]["importance"]
    err = np.abs(g - ref)
    bad = err > 1e-5 + 1e-4 * ref
    print("rows %d, composited %d, rel-L2 %.2e, rows off by more than 1e-4 rel: %d" %
          (g.size, int((ref > 0).sum()), np.linalg.norm(g - ref) / np.linalg.norm(ref), bad.sum()))
    assert np.linalg.norm(g - ref) / np.linalg.norm(ref) <= 1e-5
    # a row's maximum moves only through a pixel whose decisions lie at a cut-off
    assert bad.sum() <= max(2, 1e-4 * g.size)


@pytest.mark.parametrize("name,K,tau", [("tiny_2k_256", 16, 2.0), ("tiny_2k_256", 16, 0.05),
                                        ("small_200k_1024x768", 64, 2.0),
                                        ("small_200k_1024x768", 256, 0.02),
                                        ("small_200k_1024x768", 100000, 2.0)])
def test_prune_mask_bit_exact(name, K, tau):
    import oracle
    gs = _gs()
    o = _oracle_case(name)
    n, V, W, H = o["n"], o["V"], o["W"], o["H"]
    imp32 = o["fw"]["importance"].astype(np.float32)
    nc = o["fw"]["n_contrib"]
    mask = torch.full((n,), 7, dtype=torch.uint8, device="cuda")
    gs.gs_prune_mask(n, V, W, H, _cuda(o["vals"].view(np.int32)), _cuda(o["ranges"]), _cuda(nc),
                     _cuda(imp32), K, tau, mask)
    ref = oracle.prune_mask(n, V, W, H, o["vals"], o["ranges"], nc, imp32, K, tau)
    print("K %d tau %.2f: pruned %d of %d" % (K, tau, int(ref.sum()), n))
    assert np.array_equal(mask.cpu().numpy(), ref)


def test_compact_index_bit_exact():
    import oracle
    gs = _gs()
    rng = np.random.default_rng(9)
    for n, p in ((0, 0.5), (1, 0.0), (1, 1.0), (4095, 0.3), (4096, 0.9), (4097, 0.01),
                 (1_000_003, 0.37)):
        m = (rng.random(n) < p).astype(np.uint8)
        ws = torch.empty(max(1, gs.gs_compact_workspace_bytes(n)), dtype=torch.uint8, device="cuda")
        idx = torch.full((max(n, 1),), -1, dtype=torch.int32, device="cuda")
        k = torch.full((1,), -1, dtype=torch.int64, device="cuda")
        gs.gs_compact_index(_cuda(m) if n else torch.empty(0, dtype=torch.uint8, device="cuda"),
                            ws, idx, k)
        ref = oracle.compact_index(m)
        assert int(k.item()) == ref.size, n
        assert np.array_equal(idx[:ref.size].cpu().numpy().view(np.uint32), ref), n


def test_prune_to_capacity_compacts_consistently():
    """The step's pruning call: kept columns are exactly the unmasked ones,
    in order, for the parameters and both Adam moments."""
    gs = _gs()
    cfg = scenes.make("small_200k_1024x768")
    params = torch.from_numpy(cfg["params"]).cuda()
    step = gs.TrainStep(params.clone(), f32_cams(cfg["cams"]), torch.from_numpy(cfg["target"]).cuda())
    step.step()
    p, m, v, idx, mask = step.prune_to_capacity(64, tau=2.0)
    keep = np.nonzero(mask.cpu().numpy() == 0)[0]
    assert np.array_equal(idx.cpu().numpy(), keep)
    ii = torch.from_numpy(keep).cuda()
    assert torch.equal(p, step.params[:, ii]) and torch.equal(m, step.m[:, ii])
    assert torch.equal(v, step.v[:, ii])
    print("kept %d of %d" % (keep.size, step.n))
    assert 0 < keep.size < step.n
