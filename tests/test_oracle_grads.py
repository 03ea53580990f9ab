"""CPU pins of the oracle's backward pass and optimizer: central finite
differences in fp64 (every one of the 59 parameter rows), the batch-averaging
statement of the pages, torch's L1 loss and Adam as library references."""
import math

import numpy as np
import pytest

import scenes

W = H = 32


def _fd_scene(seed, n_views=1):
    """8 Gaussians in front of a 32x32 camera, plus special members: one with
    opacity above the 0.99 cap, one outside the J clamp region with a footprint
    reaching the image, one with a colour channel clamped at 0, and an opaque
    stack that drives transmittance below 1e-4."""
    rng = np.random.default_rng(seed)
    n = 12
    p = np.zeros((59, n))
    p[0] = rng.uniform(-0.5, 0.5, n)
    p[1] = rng.uniform(-0.5, 0.5, n)
    p[2] = rng.uniform(2.5, 5.0, n)
    p[3:6] = rng.uniform(-2.6, -1.6, (3, n))
    q = rng.standard_normal((4, n))
    p[6:10] = q / np.linalg.norm(q, axis=0)
    p[10] = rng.uniform(-1.0, 1.5, n)
    p[11:59] = rng.normal(0, 0.15, (48, n))
    p[11:14] += 0.6
    p[10, 0] = 6.0                      # capped alpha near its centre
    p[0, 1], p[2, 1] = 3.3, 4.0         # x/z = 0.83 > 1.3 * 0.5 clamp limit
    p[3:6, 1] = -0.9                    # large enough to reach the image
    p[11, 2] = -3.0                     # red channel clamped at zero
    for i in (3, 4, 5, 6):              # opaque stack near the centre
        p[0, i], p[1, i] = 0.05 * (i - 4), 0.03 * (i - 4)
        p[10, i] = 3.5
        p[3:6, i] = -1.7
    cams = [scenes.camera(np.eye(3), np.zeros(3), 32, 32, 16, 16, W, H)]
    if n_views == 2:
        cams.append(scenes.look_at((0.8, -0.4, -0.5), (0, 0, 3.5), (0, -1, 0), 30, 34, W, H))
    target = rng.random((n_views, 3, H, W))
    return p, cams, target


def _loss(oracle, p, cams, target):
    _, _, fw = oracle.render(p, cams)
    return oracle.loss_l1(fw["image"], target)[0]


def _clean_scene(oracle, n_views=1):
    """First seed whose decisions all sit far from every threshold, so the
    loss is smooth around it."""
    for seed in range(200):
        p, cams, target = _fd_scene(seed, n_views)
        pr, (keys, vals, ranges), fw = oracle.render(p, cams)
        if np.any(pr["flags"]):
            continue
        if np.min(fw["margin"]) < 2e-3:
            continue
        if np.min(np.abs(fw["image"] - target)) < 1e-5:
            continue
        if pr["radius"][0] == 0 or pr["radius"][1] == 0:
            continue
        # the special members must actually be exercised
        if not np.any(fw["T_final"] < 1e-3):
            continue
        return p, cams, target
    raise AssertionError("no clean scene")


def _grads(oracle, p, cams, target):
    loss, grad, visible, parts = oracle.train_step_grads(p, cams, target)
    return loss, grad, visible, parts


def _stencil(f, h):
    """Fourth-order central difference."""
    return (-f(2) + 8 * f(1) - 8 * f(-1) + f(-2)) / (12 * h)


def _check(a, f, what):
    scale = np.abs(f).max()
    err = np.abs(a - f)
    tol = 1e-6 * np.maximum(np.abs(f), 1e-2 * scale) + 1e-12
    bad = np.argwhere(err > tol)
    assert bad.size == 0, (what, bad[:5], a[tuple(bad[0])], f[tuple(bad[0])])


@pytest.mark.parametrize("n_views", [1, 2])
def test_full_chain_gradient_matches_finite_differences(oracle_mod, n_views):
    p, cams, target = _clean_scene(oracle_mod, n_views)
    loss, grad, visible, parts = _grads(oracle_mod, p, cams, target)
    n = p.shape[1]
    fd = np.zeros_like(grad)
    base_keys = parts["keys"]
    for row in range(59):
        for g in range(n):
            h = 3e-5 * max(1.0, abs(p[row, g]))

            def f(k):
                pk = p.copy()
                pk[row, g] += k * h
                return _loss(oracle_mod, pk, cams, target)

            fd[row, g] = _stencil(f, h)
    assert base_keys.size > 0
    _check(grad, fd, "grad[59][n]")
    # every parameter group gets a non-trivial gradient
    for a, b in [(0, 3), (3, 6), (6, 10), (10, 11), (11, 14), (14, 59)]:
        assert np.abs(grad[a:b]).max() > 1e-7
    # the colour-clamped channel passes no gradient to its SH coefficients
    pr = parts["proj"]
    assert pr["color"][2, 0] == 0.0
    assert np.all(grad[11::3, 2] == 0.0)


def test_raster_gradient_matches_finite_differences(oracle_mod):
    """Compositing backward alone: perturb the 2D features directly."""
    p, cams, target = _clean_scene(oracle_mod)
    n = p.shape[1]
    pr, (keys, vals, ranges), fw = oracle_mod.render(p, cams)
    _, g_img = oracle_mod.loss_l1(fw["image"], target)
    g2 = oracle_mod.raster_bwd(n, 1, W, H, pr, vals, ranges, g_img)

    def L(feats):
        out = oracle_mod.raster_fwd(n, 1, W, H, feats, vals, ranges)
        return oracle_mod.loss_l1(out["image"], target)[0]

    for name, width in (("mean2d", 2), ("conic", 3), ("opacity", 1), ("color", 3)):
        fd = np.zeros((n, width))
        for r in range(n):
            if pr["radius"][r] == 0:
                continue
            for c in range(width):
                base = pr[name].reshape(n, width)
                h = 1e-5 * max(1.0, abs(base[r, c]))

                def f(k):
                    fk = {key: v.copy() for key, v in pr.items()}
                    fk[name].reshape(n, width)[r, c] += k * h
                    return L(fk)

                fd[r, c] = _stencil(f, h)
        _check(g2[name].reshape(n, width), fd, name)


def test_batch_gradient_is_mean_of_view_gradients(oracle_mod):
    """Gradients of a batch of views are the average of the per-view
    gradients ("On Scaling Up 3D Gaussian Splatting Training", independent
    gradients answer: gradients averaged over the views)."""
    p, cams, target = _fd_scene(3, n_views=2)
    _, g_batch, _, _ = _grads(oracle_mod, p, cams, target)
    _, g0, _, _ = _grads(oracle_mod, p, cams[:1], target[:1])
    _, g1, _, _ = _grads(oracle_mod, p, cams[1:], target[1:])
    assert np.abs(g_batch - 0.5 * (g0 + g1)).max() <= 1e-15 + 1e-12 * np.abs(g_batch).max()


def test_l1_loss_matches_torch(oracle_mod):
    import torch
    rng = np.random.default_rng(2)
    a = rng.random((2, 3, 7, 9))
    b = rng.random((2, 3, 7, 9))
    b.flat[5] = a.flat[5]  # sign(0) = 0
    loss, g = oracle_mod.loss_l1(a, b)
    ta = torch.tensor(a, requires_grad=True)
    tl = torch.nn.functional.l1_loss(ta, torch.tensor(b), reduction="mean")
    tl.backward()
    assert loss == pytest.approx(tl.item(), rel=1e-14)
    assert np.abs(g - ta.grad.numpy()).max() < 1e-18


def _torch_adam_steps(p0, grads, lr, betas, eps, visibles=None):
    import torch
    p = torch.tensor(p0.copy())
    m = torch.zeros_like(p)
    v = torch.zeros_like(p)
    for t, g in enumerate(grads, start=1):
        cols = np.arange(p.shape[1]) if visibles is None else np.nonzero(visibles[t - 1])[0]
        idx = torch.tensor(cols, dtype=torch.long)
        sub = torch.nn.Parameter(p[:, idx].clone())
        opt = torch.optim.Adam([sub], lr=lr, betas=betas, eps=eps, foreach=False)
        opt.state[sub] = {"step": torch.tensor(float(t - 1)), "exp_avg": m[:, idx].clone(),
                          "exp_avg_sq": v[:, idx].clone()}
        sub.grad = torch.tensor(g)[:, idx].clone()
        opt.step()
        p[:, idx] = sub.detach()
        m[:, idx] = opt.state[sub]["exp_avg"]
        v[:, idx] = opt.state[sub]["exp_avg_sq"]
    return p.numpy(), m.numpy(), v.numpy()


@pytest.mark.parametrize("sparse", [False, True])
def test_adam_matches_torch(oracle_mod, sparse):
    rng = np.random.default_rng(4)
    rows, cols, steps = 59, 37, 6
    p0 = rng.standard_normal((rows, cols))
    grads = [rng.standard_normal((rows, cols)) * 10.0 ** rng.uniform(-7, -1, (rows, cols))
             for _ in range(steps)]
    vis = [(rng.random(cols) < 0.6).astype(np.uint8) for _ in range(steps)] if sparse else None
    lr, b1, b2, eps = 1e-3, 0.9, 0.999, 1e-8
    p, m, v = p0.copy(), np.zeros_like(p0), np.zeros_like(p0)
    for t in range(1, steps + 1):
        oracle_mod.adam(p, grads[t - 1], m, v, t, lr, b1, b2, eps,
                        None if vis is None else vis[t - 1])
    tp, tm, tv = _torch_adam_steps(p0, grads, lr, (b1, b2), eps, vis)
    # torch updates the moments with lerp, so rounding differs in the last bit
    assert np.abs(p - tp).max() <= 1e-14 * np.abs(tp).max()
    assert np.abs(m - tm).max() <= 1e-14 * np.abs(tm).max()
    assert np.abs(v - tv).max() <= 1e-14 * np.abs(tv).max()
    if sparse:
        never = np.all(np.stack(vis) == 0, axis=0)
        assert np.array_equal(p[:, never], p0[:, never])


def test_adam_first_step_closed_form(oracle_mod):
    """At t = 1 the bias-corrected update is -lr g / (|g| + eps)."""
    rng = np.random.default_rng(8)
    g = rng.standard_normal((59, 10)) * 1e-3
    p = rng.standard_normal((59, 10))
    p0 = p.copy()
    m, v = np.zeros_like(p), np.zeros_like(p)
    oracle_mod.adam(p, g, m, v, 1, 1e-3)
    expect = p0 - 1e-3 * g / (np.abs(g) + 1e-8)
    assert np.abs(p - expect).max() < 1e-15


def test_sqrt_batch_learning_rate_rule(oracle_mod):
    """The premise and the consequence of the sqrt(b) learning-rate rule
    ("On Scaling Up 3D Gaussian Splatting Training", independent-gradients
    answer), on the oracle's Adam.  Per-view gradients are i.i.d. with mean mu
    and deviation sigma; their mean over a batch of b views is then exactly
    N(mu, sigma^2 / b), drawn directly.  (1) Adam's second moment settles at
    sigma^2 / b (plus mu^2).  (2) With lr sqrt(b), one batch-b step moves the
    parameters as far, on average, as b batch-size-1 steps."""
    rng = np.random.default_rng(5)
    rows, cols, steps, burn = 59, 400, 1500, 300
    mu, sigma, lr = 0.05, 1.0, 1e-3
    drift = {}
    for b in (1, 4, 16):
        p = np.zeros((rows, cols))
        m, v = np.zeros_like(p), np.zeros_like(p)
        moved = 0.0
        for t in range(1, steps + 1):
            g = rng.normal(mu, sigma / math.sqrt(b), (rows, cols))
            before = p.copy()
            oracle_mod.adam(p, g, m, v, t, lr * math.sqrt(b))
            if t > burn:
                moved += float((before - p).mean())
        v_hat = v.mean() / (1.0 - 0.999 ** steps)
        assert v_hat == pytest.approx(sigma ** 2 / b + mu ** 2, rel=0.05)
        drift[b] = moved / (steps - burn)
    for b in (4, 16):
        assert drift[b] / drift[1] == pytest.approx(b, rel=0.08)
