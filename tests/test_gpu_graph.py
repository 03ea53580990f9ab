"""A training step captured once into a CUDA graph and replayed: the
asynchronous binning against the synchronous one (bit for bit), its overflow
report, Adam with the step number on the device, and replayed steps against
eager ones."""
import numpy as np
import pytest
import torch

import scenes
from parity_util import f32_cams, pack_records, rel_l2

pytestmark = pytest.mark.gpu


def _gs():
    import __graft_entry__
    __graft_entry__.build()
    import gaussian_splatting_differentiable_gs_gb300 as gs
    return gs


def _records(name):
    import oracle
    cfg = scenes.make(name)
    cams = f32_cams(cfg["cams"])
    pr = oracle.project(cfg["params"].astype(np.float64), cams)
    return cfg["params"].shape[1], len(cams), cams[0]["width"], cams[0]["height"], pack_records(pr)


def _bufs(gs, n, V, W, H, cap):
    ws = torch.zeros(gs.gs_bin_workspace_bytes(n * V, cap), dtype=torch.uint8, device="cuda")
    keys = torch.empty(cap, dtype=torch.int64, device="cuda")
    vals = torch.empty(cap, dtype=torch.int32, device="cuda")
    ranges = torch.full((V * gs.tiles_per_view(W, H), 2), -3, dtype=torch.int64, device="cuda")
    return ws, keys, vals, ranges


@pytest.mark.parametrize("name", ["tiny_2k_256", "small_200k_1024x768"])
def test_async_binning_equals_sync(name):
    gs = _gs()
    n, V, W, H, rec = _records(name)
    splats = torch.from_numpy(rec).cuda()
    cap = int(rec.view(np.int32)[:, 11].astype(np.int64).sum()) + 777
    ws, keys, vals, ranges = _bufs(gs, n, V, W, H, cap)
    st, I = gs.gs_bin_and_sort(n, V, splats, W, H, ws, cap, keys, vals, ranges)
    assert st == gs.GS_OK
    ws2, keys2, vals2, ranges2 = _bufs(gs, n, V, W, H, cap)
    nd = torch.full((1,), -1, dtype=torch.int64, device="cuda")
    gs.gs_bin_and_sort_async(n, V, splats, W, H, ws2, cap, keys2, vals2, ranges2, nd)
    assert gs.gs_workspace_status(ws2) == gs.GS_OK
    assert int(nd.item()) == I
    assert torch.equal(keys2[:I], keys[:I]) and torch.equal(vals2[:I], vals[:I])
    assert torch.equal(ranges2, ranges)


def test_async_binning_equals_sync_large_footprints():
    """Rows of 40 tiles on average: both calls emit in balanced chunks of
    intersections (the asynchronous one sized by its capacity, the
    synchronous one by the counts); lists bit for bit equal, and equal to the
    oracle's."""
    import oracle
    gs = _gs()
    V, W, H, n = 2, 1024, 768, 3000
    tx, ty = (W + 15) // 16, (H + 15) // 16
    rng = np.random.default_rng(5)
    rows = V * n
    pr = dict(mean2d=np.stack([rng.uniform(-40, W + 40, rows), rng.uniform(-40, H + 40, rows)], 1),
              conic=np.ones((rows, 3)), opacity=np.full(rows, 0.5), color=np.full((rows, 3), 0.5),
              depth=rng.choice([1.0, 3.0, 3.0000002, 9.0], rows),
              radius=rng.integers(40, 80, rows).astype(np.int32), tiles=np.zeros(rows, np.int32))
    for r in range(rows):
        x0, x1, y0, y1 = oracle.tile_rect(pr["mean2d"][r, 0], pr["mean2d"][r, 1], pr["radius"][r],
                                          16, tx, ty)
        pr["tiles"][r] = (x1 - x0) * (y1 - y0)
    pr["radius"][pr["tiles"] == 0] = 0
    rec = pack_records(pr)
    I_o = int(pr["tiles"].astype(np.int64).sum())
    assert I_o >= 8 * rows
    keys_o, vals_o, ranges_o = oracle.bin_and_sort(n, V, rec[:, 0:2], pr["radius"], rec[:, 9], W, H)
    splats = torch.from_numpy(rec).cuda()
    cap = I_o + 777
    ws, keys, vals, ranges = _bufs(gs, n, V, W, H, cap)
    st, I = gs.gs_bin_and_sort(n, V, splats, W, H, ws, cap, keys, vals, ranges)
    assert st == gs.GS_OK and I == I_o
    ws2, keys2, vals2, ranges2 = _bufs(gs, n, V, W, H, cap)
    nd = torch.full((1,), -1, dtype=torch.int64, device="cuda")
    gs.gs_bin_and_sort_async(n, V, splats, W, H, ws2, cap, keys2, vals2, ranges2, nd)
    assert gs.gs_workspace_status(ws2) == gs.GS_OK
    assert int(nd.item()) == I
    assert np.array_equal(keys[:I].cpu().numpy().view(np.uint64), keys_o)
    assert np.array_equal(vals[:I].cpu().numpy().view(np.uint32), vals_o)
    assert np.array_equal(ranges.cpu().numpy(), ranges_o)
    assert torch.equal(keys2[:I], keys[:I]) and torch.equal(vals2[:I], vals[:I])
    assert torch.equal(ranges2, ranges)


def test_async_binning_overflow_and_recovery():
    gs = _gs()
    n, V, W, H, rec = _records("tiny_2k_256")
    splats = torch.from_numpy(rec).cuda()
    I = int(rec.view(np.int32)[:, 11].astype(np.int64).sum())
    ws, keys, vals, ranges = _bufs(gs, n, V, W, H, I + 10)
    nd = torch.zeros(1, dtype=torch.int64, device="cuda")
    gs.gs_bin_and_sort_async(n, V, splats, W, H, ws, I - 1, keys, vals, ranges, nd)
    torch.cuda.synchronize()
    assert int(nd.item()) == I
    assert torch.all(ranges == 0)
    # Adam and the step counter skip while the binning reports an overflow
    p = torch.randn((59, 64), device="cuda")
    p0 = p.clone()
    m, v = torch.zeros_like(p), torch.zeros_like(p)
    step = torch.ones(1, dtype=torch.int64, device="cuda")
    gs.gs_step_advance(step, ws)
    gs.gs_adam_step_dev(p, torch.randn_like(p), m, v, step, 1e-3, bin_workspace=ws)
    assert torch.equal(p, p0) and int(step.item()) == 1
    assert gs.gs_workspace_status(ws) == gs.GS_ERR_CAPACITY
    # the next call with enough capacity builds the lists and clears the report
    gs.gs_bin_and_sort_async(n, V, splats, W, H, ws, I + 10, keys, vals, ranges, nd)
    assert gs.gs_workspace_status(ws) == gs.GS_OK
    ws3, k3, v3, r3 = _bufs(gs, n, V, W, H, I + 10)
    st, I2 = gs.gs_bin_and_sort(n, V, splats, W, H, ws3, I + 10, k3, v3, r3)
    assert st == gs.GS_OK and I2 == I and torch.equal(r3, ranges)
    assert torch.equal(k3[:I], keys[:I]) and torch.equal(v3[:I], vals[:I])


def test_adam_step_dev_matches_host_step():
    gs = _gs()
    rng = np.random.default_rng(2)
    p = torch.from_numpy(rng.standard_normal((59, 5003)).astype(np.float32)).cuda()
    pa, pb = p.clone(), p.clone()
    ma, va, mb, vb = (torch.zeros_like(p) for _ in range(4))
    step = torch.zeros(1, dtype=torch.int64, device="cuda")
    for t in range(1, 4):
        g = torch.from_numpy((rng.standard_normal((59, 5003)) * 1e-3).astype(np.float32)).cuda()
        gs.gs_adam_step(pa, g, ma, va, t, 1e-3)
        gs.gs_step_advance(step)
        gs.gs_adam_step_dev(pb, g, mb, vb, step, 1e-3)
    assert int(step.item()) == 3
    for a, b in ((pa, pb), (ma, mb), (va, vb)):
        assert rel_l2(b.cpu().numpy(), a.cpu().numpy()) <= 1e-7


@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("name", ["tiny_2k_256", "small_200k_1024x768"])
def test_replayed_steps_match_eager_steps(name, fused):
    gs = _gs()
    cfg = scenes.make(name)
    cams = f32_cams(cfg["cams"])
    target = torch.from_numpy(cfg["target"]).cuda()
    eager = gs.TrainStep(torch.from_numpy(cfg["params"]).cuda(), cams, target, lr=1e-3, fused=fused)
    graph = gs.TrainStep(torch.from_numpy(cfg["params"]).cuda(), cams, target, lr=1e-3, fused=fused)
    losses_e, losses_g = [], []
    for _ in range(4):
        losses_e.append(eager.step().item())
    losses_g.append(graph.step().item())  # eager, sizes the buffers
    graph.capture()
    for _ in range(3):
        losses_g.append(graph.step().item())
    assert graph.check() == gs.GS_OK and graph.t == 4
    print("losses eager %s graph %s" % (losses_e, losses_g))
    # fp32 atomics make two eager runs differ too (a gradient near zero can
    # change sign, and Adam's first steps move by lr sign(g)): the Adam bar
    assert np.allclose(losses_g, losses_e, rtol=1e-5)
    for a, b in ((eager.params, graph.params), (eager.m, graph.m), (eager.v, graph.v)):
        assert rel_l2(b.cpu().numpy(), a.cpu().numpy()) <= 1e-4


def test_replay_recovers_from_capacity_overflow():
    gs = _gs()
    cfg = scenes.make("tiny_2k_256")
    step = gs.TrainStep(torch.from_numpy(cfg["params"]).cuda(), f32_cams(cfg["cams"]),
                        torch.from_numpy(cfg["target"]).cuda(), lr=1e-3, fused=True)
    step.step()
    step.capture(margin=1.0)
    cap = step.capacity
    with torch.no_grad():
        step.params[3:6] += 0.7  # larger footprints: more intersections than the graph holds
    p_before = step.params.clone()
    step.step()
    assert torch.equal(step.params, p_before)  # the overflowing step updated nothing
    assert step.check() == gs.GS_ERR_CAPACITY
    assert step.capacity > cap and step.graph is not None
    step.step()
    assert step.check() == gs.GS_OK
    assert not torch.equal(step.params, p_before)
