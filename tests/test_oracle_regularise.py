"""Pins for the oracle's Sobolev regulariser and Adam step.

Paper: "A Scalable Distributed Framework for Multimodal GigaVoxel Image
Registration", "Background": L(phi) = C(F, M o phi) + R(phi) with R a Sobolev
norm; the method's overview updates the warp by gradient descent with
optimiser state [m1], [m2] kept per voxel beside u.

Each check ties the oracle to something other than itself: closed forms
(constant and linear fields), the quadratic form u^T L u of the grid graph's
Laplacian built by scipy.sparse.csgraph, central differences, and
torch.optim.Adam (float64) over several steps.
"""
import numpy as np
import pytest
import torch

import oracle


def _grid_laplacian(shape):
    import scipy.sparse as sp
    from scipy.sparse.csgraph import laplacian
    D, H, W = shape
    n = D * H * W
    idx = np.arange(n).reshape(shape)
    rows, cols = [], []
    for a, (dz, dy, dx) in enumerate([(0, 0, 1), (0, 1, 0), (1, 0, 0)]):
        src = idx[:D - dz, :H - dy, :W - dx].ravel()
        dst = idx[dz:, dy:, dx:].ravel()
        rows += [src, dst]
        cols += [dst, src]
    A = sp.coo_matrix((np.ones(sum(r.size for r in rows)), (np.concatenate(rows), np.concatenate(cols))),
                      shape=(n, n)).tocsr()
    return laplacian(A)


def test_constant_field_has_zero_energy_and_gradient():
    u = np.broadcast_to(np.array([0.25, -0.5, 0.125], np.float32), (4, 5, 6, 3)).copy()
    r = oracle.sobolev(u, 2.0)
    assert r["R"] == 0.0 and np.all(r["dR"] == 0.0)


def test_linear_field_closed_form():
    # u_c(i) = alpha_c * i_x + beta_c * i_z: every x edge contributes alpha_c^2,
    # every z edge beta_c^2, every y edge 0
    D, H, W = 5, 6, 7
    alpha = np.array([0.5, -0.25, 0.125])
    beta = np.array([0.0, 0.375, -0.5])
    zz, yy, xx = np.meshgrid(np.arange(D), np.arange(H), np.arange(W), indexing="ij")
    u = (xx[..., None] * alpha + zz[..., None] * beta).astype(np.float32)
    lam = 0.7
    N = D * H * W
    nx, nz = D * H * (W - 1), (D - 1) * H * W
    ref = lam / N * (nx * np.sum(alpha ** 2) + nz * np.sum(beta ** 2))
    r = oracle.sobolev(u, lam)
    assert abs(r["R"] - ref) <= 1e-12 * ref
    # interior gradient of a linear field is zero (the discrete Laplacian vanishes)
    assert np.max(np.abs(r["dR"][1:-1, 1:-1, 1:-1])) <= 1e-12


@pytest.mark.parametrize("shape", [(3, 4, 5), (6, 2, 7)])
def test_matches_the_grid_graph_laplacian(shape):
    rng = np.random.default_rng(sum(shape))
    u = rng.normal(size=shape + (3,)).astype(np.float32)
    lam = 1.3
    N = int(np.prod(shape))
    L = _grid_laplacian(shape)
    U = u.reshape(-1, 3).astype(np.float64)
    R_ref = lam / N * float(np.sum(U * (L @ U)))
    G_ref = 2.0 * lam / N * (L @ U)
    r = oracle.sobolev(u, lam)
    assert abs(r["R"] - R_ref) <= 1e-12 * abs(R_ref)
    assert np.max(np.abs(r["dR"].reshape(-1, 3) - G_ref)) <= 1e-12 * np.max(np.abs(G_ref))


def test_gradient_central_differences():
    rng = np.random.default_rng(3)
    u = rng.normal(size=(3, 4, 5, 3)).astype(np.float32).astype(np.float64)
    lam = 0.9
    r = oracle.sobolev(u, lam)
    h = 2.0 ** -10
    for (z, y, x, c) in [(0, 0, 0, 0), (1, 2, 3, 1), (2, 3, 4, 2), (1, 0, 4, 0)]:
        up = u.copy(); up[z, y, x, c] += h
        um = u.copy(); um[z, y, x, c] -= h
        fd = (oracle.sobolev(up, lam, False)["R"] - oracle.sobolev(um, lam, False)["R"]) / (2 * h)
        assert abs(fd - r["dR"][z, y, x, c]) <= 1e-9


def test_adam_matches_torch_optim_adam():
    rng = np.random.default_rng(4)
    n = 257
    x0 = rng.normal(size=n)
    grads = [rng.normal(size=n) * s for s in (1.0, 0.1, 3.0, 1e-4)]
    lr, b1, b2, eps = 0.05, 0.9, 0.999, 1e-8
    p = torch.nn.Parameter(torch.tensor(x0, dtype=torch.float64))
    opt = torch.optim.Adam([p], lr=lr, betas=(b1, b2), eps=eps)
    x, m1, m2 = x0.copy(), np.zeros(n), np.zeros(n)
    for t, g in enumerate(grads, start=1):
        p.grad = torch.tensor(g, dtype=torch.float64)
        opt.step()
        x, m1, m2 = oracle.adam(x, g, m1, m2, lr, b1, b2, eps, t)
        st = opt.state[p]
        assert np.max(np.abs(x - p.detach().numpy())) <= 1e-13
        assert np.max(np.abs(m1 - st["exp_avg"].numpy())) <= 1e-15
        assert np.max(np.abs(m2 - st["exp_avg_sq"].numpy())) <= 1e-15


def test_first_adam_step_moves_by_lr_times_sign():
    # t = 1: m1 / (1 - b1) = g and m2 / (1 - b2) = g^2, so the step is lr g / (|g| + eps)
    g = np.array([2.0, -0.5, 1e-3, -7.0])
    x, _, _ = oracle.adam(np.zeros(4), g, np.zeros(4), np.zeros(4), 0.1, 0.9, 0.99, 0.0, 1)
    assert np.allclose(x, -0.1 * np.sign(g), atol=1e-15)


def test_regularised_step_adds_the_regulariser_gradient():
    rng = np.random.default_rng(5)
    u = rng.normal(size=(3, 4, 5, 3)).astype(np.float32)
    g = rng.normal(size=u.shape)
    m1 = rng.normal(size=u.shape) * 0.1
    m2 = np.abs(rng.normal(size=u.shape)) * 0.01
    r = oracle.sobolev_adam_step(u, g, m1, m2, 0.5, 0.01, 0.9, 0.999, 1e-8, 3)
    dR = oracle.sobolev(u, 0.5)["dR"]
    x, n1, n2 = oracle.adam(u.astype(np.float64), g + dR, m1, m2, 0.01, 0.9, 0.999, 1e-8, 3)
    assert np.array_equal(r["u"], x) and np.array_equal(r["m1"], n1) and np.array_equal(r["m2"], n2)


def test_golden_sobolev_ramp():
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.txt")
    row = [l for l in open(path) if l.startswith("sobolev_ramp2")][0]
    _, inp, exp = [s.strip() for s in row.split("|")]
    kv = dict(tok.split("=") for tok in (inp + " " + exp).split())
    u = np.zeros((2, 2, 2, 3), np.float32)
    u[..., 0] = np.arange(2)[None, None, :]
    r = oracle.sobolev(u, float(kv["lambda"]))
    assert abs(r["R"] - float(kv["R"])) <= 1e-15
    lo, hi = (float(v) for v in kv["dRx"].split(","))
    assert np.allclose(r["dR"][..., 0, 0], lo, atol=1e-15) and np.allclose(r["dR"][..., 1, 0], hi, atol=1e-15)
    assert np.all(r["dR"][..., 1:] == 0.0)
