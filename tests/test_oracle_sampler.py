"""Pins for the oracle's composite implicit grid sampler and its backward.

Each check ties the oracle to something other than itself: exact special
cases (identity, integer shifts), the closed form of trilinear interpolation
on a linear image, the library routine torch.nn.functional.grid_sample
(float64, align_corners=True, zero padding) with autograd, and central finite
differences.  Paper: "A Scalable Distributed Framework for Multimodal
GigaVoxel Image Registration", Key designs item 1 (fused_grid_sampler
I(Ax+t+Su(x)) with implicit x_bounds, backward including the affine gradient).
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as Fnn

import oracle
from oracle import Transform


def _rand_vol(shape, seed):
    return np.random.default_rng(seed).uniform(-1, 1, shape).astype(np.float32)


def test_identity_returns_M_exactly():
    M = _rand_vol((7, 9, 11), 1)
    J = oracle.grid_sample(M, M.shape, None, Transform.identity())
    assert np.max(np.abs(J - M.astype(np.float64))) <= 1e-12


@pytest.mark.parametrize("k", [(1, -2, 3), (0, 0, -1), (-3, 1, 0)])
def test_integer_translation_shifts_exactly(k):
    D, H, W = 6, 8, 10
    M = _rand_vol((D, H, W), 2)
    n = np.array([W, H, D], np.float64)
    T = Transform.identity()
    T.t = 2.0 * np.asarray(k, np.float64) / (n - 1)
    J = oracle.grid_sample(M, M.shape, None, T)
    ref = np.zeros_like(J)
    kx, ky, kz = k
    for z in range(D):
        for y in range(H):
            for x in range(W):
                xs, ys, zs = x + kx, y + ky, z + kz
                if 0 <= xs < W and 0 <= ys < H and 0 <= zs < D:
                    ref[z, y, x] = M[zs, ys, xs]
    assert np.max(np.abs(J - ref)) <= 1e-12


def test_linear_image_is_reproduced_with_closed_form_gradients():
    # M[z,y,x] = ax*x + ay*y + az*z + b0 is reproduced exactly by trilinear
    # interpolation at interior points, with dJ/dq = (ax, ay, az).
    D, H, W = 9, 10, 12
    ax, ay, az, b0 = 0.5, -1.25, 2.0, 0.375
    zz, yy, xx = np.meshgrid(np.arange(D), np.arange(H), np.arange(W), indexing="ij")
    M = (ax * xx + ay * yy + az * zz + b0).astype(np.float64)
    assert np.all(M.astype(np.float32).astype(np.float64) == M)  # exactly representable
    # fixed grid 5x6x7, mapped strictly inside M by a shrinking affine + offset
    fs = (5, 6, 7)
    rng = np.random.default_rng(3)
    A = np.diag([0.6, 0.55, 0.5]) + rng.uniform(-0.05, 0.05, (3, 3))
    t = rng.uniform(-0.1, 0.1, 3)
    T = Transform(A, t, np.eye(3), -np.ones(3), np.ones(3))
    J, G = oracle.grid_sample(M.astype(np.float32), fs, None, T, want_grad=True)
    nM = np.array([W, H, D], np.float64)
    # independent recomputation of q in closed form
    Df, Hf, Wf = fs
    for z in range(Df):
        for y in range(Hf):
            for x in range(Wf):
                xc = np.array([-1 + 2 * x / (Wf - 1), -1 + 2 * y / (Hf - 1), -1 + 2 * z / (Df - 1)])
                p = A @ xc + t
                q = (p + 1) / 2 * (nM - 1)
                assert np.all(q > 0) and np.all(q < nM - 1)
                assert abs(J[z, y, x] - (ax * q[0] + ay * q[1] + az * q[2] + b0)) < 1e-12
                assert np.allclose(G[z, y, x], np.array([ax, ay, az]) * (nM - 1) / 2, atol=1e-12)
    # closed-form backward for L = sum g*J on this linear image
    g = rng.normal(size=fs)
    du, dA, dt = oracle.grid_sample_bwd(M.astype(np.float32), fs, None, T, g)
    grad_p = np.array([ax, ay, az]) * (nM - 1) / 2
    xs = np.linspace(-1, 1, Wf)
    ys = np.linspace(-1, 1, Hf)
    zs = np.linspace(-1, 1, Df)
    Z, Y, X = np.meshgrid(zs, ys, xs, indexing="ij")
    coords = np.stack([X, Y, Z], -1)
    dA_ref = np.outer(grad_p, (g[..., None] * coords).reshape(-1, 3).sum(0))
    dt_ref = grad_p * g.sum()
    assert np.allclose(dA.reshape(3, 3), dA_ref, atol=1e-10)
    assert np.allclose(dt, dt_ref, atol=1e-10)
    assert np.allclose(du, g[..., None] * grad_p, atol=1e-12)


def _torch_objective(M, fs, u, T, g):
    """L = sum g * grid_sample(M, A x + t + S u) in float64 with autograd."""
    Mt = torch.tensor(M, dtype=torch.float64)[None, None]
    A = torch.tensor(T.A, dtype=torch.float64, requires_grad=True)
    t = torch.tensor(T.t, dtype=torch.float64, requires_grad=True)
    S = torch.tensor(T.S, dtype=torch.float64)
    ut = torch.tensor(u, dtype=torch.float64, requires_grad=True)
    D, H, W = fs
    xs = torch.linspace(float(T.xmin[0]), float(T.xmax[0]), W, dtype=torch.float64)
    ys = torch.linspace(float(T.xmin[1]), float(T.xmax[1]), H, dtype=torch.float64)
    zs = torch.linspace(float(T.xmin[2]), float(T.xmax[2]), D, dtype=torch.float64)
    Z, Y, X = torch.meshgrid(zs, ys, xs, indexing="ij")
    x = torch.stack([X, Y, Z], -1)
    grid = x @ A.T + t + ut @ S.T
    J = Fnn.grid_sample(Mt, grid[None], mode="bilinear", padding_mode="zeros", align_corners=True)[0, 0]
    L = (J * torch.tensor(g, dtype=torch.float64)).sum()
    L.backward()
    return J.detach().numpy(), ut.grad.numpy(), A.grad.numpy(), t.grad.numpy()


@pytest.mark.parametrize("seed", [0, 1])
def test_matches_torch_grid_sample_with_autograd(seed):
    rng = np.random.default_rng(10 + seed)
    fs = (5, 6, 7)
    M = _rand_vol((6, 8, 9), 20 + seed)  # moving grid differs from the fixed grid
    u = (rng.normal(size=fs + (3,)) * 0.15).astype(np.float32)
    A = (np.eye(3) + rng.uniform(-0.15, 0.15, (3, 3))).astype(np.float32)
    t = rng.uniform(-0.1, 0.1, 3).astype(np.float32)
    S = (np.eye(3) * 0.8 + rng.uniform(-0.1, 0.1, (3, 3))).astype(np.float32)
    xmin = np.array([-0.9, -1.0, -0.8], np.float32)
    xmax = np.array([0.95, 0.9, 1.0], np.float32)
    T = Transform(A.astype(np.float64), t.astype(np.float64), S.astype(np.float64),
                  xmin.astype(np.float64), xmax.astype(np.float64))
    g = rng.normal(size=fs)
    J_t, du_t, dA_t, dt_t = _torch_objective(M, fs, u.astype(np.float64), T, g)
    J = oracle.grid_sample(M, fs, u, T)
    du, dA, dt = oracle.grid_sample_bwd(M, fs, u, T, g)
    # torch computes coordinates in a different association order: agree to
    # double rounding, except for the rare voxel whose coordinate sits within
    # rounding of an integer (where the one-sided slope may differ).
    assert np.max(np.abs(J - J_t)) < 1e-12
    close = np.abs(du - du_t) < 1e-9
    assert close.mean() > 0.999
    assert np.allclose(dt, dt_t, rtol=1e-9, atol=1e-9)
    assert np.allclose(dA.reshape(3, 3), dA_t, rtol=1e-9, atol=1e-9)


def test_backward_matches_central_differences():
    rng = np.random.default_rng(5)
    fs = (4, 5, 6)
    M = _rand_vol((5, 6, 7), 6)
    u = (rng.normal(size=fs + (3,)) * 0.1)
    T = Transform(np.eye(3) + rng.uniform(-0.1, 0.1, (3, 3)), rng.uniform(-0.05, 0.05, 3),
                  np.eye(3) + rng.uniform(-0.1, 0.1, (3, 3)), -np.ones(3), np.ones(3))
    g = rng.normal(size=fs)
    # u is passed as float32 to the oracle: evaluate L at float32-exact points
    u32 = u.astype(np.float32)
    du, dA, dt = oracle.grid_sample_bwd(M, fs, u32, T, g)
    _, G = oracle.grid_sample(M, fs, u32, T, want_grad=True)

    def L_of(Tx, uu):
        return float((oracle.grid_sample(M, fs, uu, Tx) * g).sum())

    h = 1e-5
    # A and t: perturb in double (the transform is passed in double)
    for r in range(3):
        for c in range(3):
            Tp = Transform(T.A.copy(), T.t, T.S, T.xmin, T.xmax)
            Tm = Transform(T.A.copy(), T.t, T.S, T.xmin, T.xmax)
            Tp.A[r, c] += h
            Tm.A[r, c] -= h
            fd = (L_of(Tp, u32) - L_of(Tm, u32)) / (2 * h)
            assert abs(fd - dA[r * 3 + c]) < 1e-5 * max(1.0, abs(fd))
        Tp = Transform(T.A, T.t.copy(), T.S, T.xmin, T.xmax)
        Tm = Transform(T.A, T.t.copy(), T.S, T.xmin, T.xmax)
        Tp.t[r] += h
        Tm.t[r] -= h
        fd = (L_of(Tp, u32) - L_of(Tm, u32)) / (2 * h)
        assert abs(fd - dt[r]) < 1e-5 * max(1.0, abs(fd))
    # du: central differences in u itself.  J is linear along each axis inside
    # a trilinear cell (the S-mixed step is cubic in h, so central differences
    # leave an O(h^2) error of ~1e-7 here); u is
    # float32, so divide by the step actually representable.
    nM = np.array([7, 6, 5], np.float64)
    hu = 1e-3
    checked = 0
    for idx in [(0, 0, 0), (1, 2, 3), (3, 4, 5), (2, 1, 4), (1, 3, 1)]:
        z, y, x = idx
        xc = np.array([-1 + 2 * x / 5, -1 + 2 * y / 4, -1 + 2 * z / 3])
        p0 = T.A @ xc + T.t + T.S @ u32[idx].astype(np.float64)
        q = (p0 + 1) / 2 * (nM - 1)
        if np.min(np.abs(q - np.round(q))) < 0.05:
            continue
        for c in range(3):
            up = u32.copy()
            um = u32.copy()
            up[idx + (c,)] = np.float32(u32[idx + (c,)] + hu)
            um[idx + (c,)] = np.float32(u32[idx + (c,)] - hu)
            step = float(up[idx + (c,)]) - float(um[idx + (c,)])
            fd = (L_of(T, up) - L_of(T, um)) / step
            assert abs(fd - du[idx + (c,)]) < 1e-6 * max(1.0, abs(fd))
        checked += 1
    assert checked >= 2
