"""Pins for the oracle's C-channel sampler (warp composition, image gradient)
and its MSE similarity.

Paper: "A Scalable Distributed Framework for Multimodal GigaVoxel Image
Registration".  "Background": L = C(F, M o phi) + R(phi) with C one of MSE,
LNCC or MI, and deformation interpolation / warp composition named as a
memory bottleneck; Key designs item 1: the sampler I(Ax+t+Su(x)) with its
backward (as PyTorch's, plus the affine gradient); item 5: MSE is a
per-voxel loss.

Each check ties the oracle to something other than itself: exact special
cases (identity, integer shifts, constant and linear fields), the adjoint
identity of the sampling operator (the image gradient dV is the transpose of
sampling, so <dV, W> = <g, sample(W)> for any W), the library routine
torch.nn.functional.grid_sample in float64 with autograd (channels, the
image gradient, u, A, t), central finite differences, and the closed form of
the mean squared error.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as Fnn

import oracle
from oracle import Transform


def _rand(shape, seed, lo=-1.0, hi=1.0):
    return np.random.default_rng(seed).uniform(lo, hi, shape).astype(np.float32)


def _transform(seed, scale=0.15):
    rng = np.random.default_rng(seed)
    A = (np.eye(3) + rng.uniform(-scale, scale, (3, 3))).astype(np.float32)
    t = rng.uniform(-0.1, 0.1, 3).astype(np.float32)
    S = (np.eye(3) * 0.8 + rng.uniform(-0.1, 0.1, (3, 3))).astype(np.float32)
    xmin = np.array([-0.95, -1.0, -0.9], np.float32)
    xmax = np.array([1.0, 0.92, 0.97], np.float32)
    f64 = lambda v: np.asarray(v, np.float64)
    return Transform(f64(A), f64(t), f64(S), f64(xmin), f64(xmax))


@pytest.mark.parametrize("C", [1, 3, 4])
def test_identity_returns_V_exactly(C):
    V = _rand((6, 7, 9, C), 1)
    out = oracle.sample_channels(V, V.shape[:3], None, Transform.identity())
    assert np.max(np.abs(out - V.astype(np.float64))) <= 1e-12


def test_integer_translation_shifts_every_channel():
    D, H, W, C = 6, 8, 10, 3
    V = _rand((D, H, W, C), 2)
    k = (2, -1, 1)
    n = np.array([W, H, D], np.float64)
    T = Transform.identity()
    T.t = 2.0 * np.asarray(k, np.float64) / (n - 1)
    out = oracle.sample_channels(V, (D, H, W), None, T)
    ref = np.zeros((D, H, W, C))
    for z in range(D):
        for y in range(H):
            for x in range(W):
                xs, ys, zs = x + k[0], y + k[1], z + k[2]
                if 0 <= xs < W and 0 <= ys < H and 0 <= zs < D:
                    ref[z, y, x] = V[zs, ys, xs]
    assert np.max(np.abs(out - ref)) <= 1e-12


def test_composition_with_constant_and_linear_fields():
    # A displacement field that is linear in the voxel index of its own grid,
    # V_c[z,y,x] = a_c . (x, y, z) + b_c, is reproduced exactly at interior
    # points, so the composed displacement is d = S u + a q(p) + b in closed
    # form (q = voxel coordinates of p); a constant field adds a constant.
    Dv, Hv, Wv = 9, 10, 12
    zz, yy, xx = np.meshgrid(np.arange(Dv), np.arange(Hv), np.arange(Wv), indexing="ij")
    a = np.array([[0.25, -0.5, 0.125], [0.0, 0.375, -0.25], [-0.125, 0.0, 0.5]])
    b = np.array([0.0625, -0.125, 0.25])
    V = np.stack([a[c, 0] * xx + a[c, 1] * yy + a[c, 2] * zz + b[c] for c in range(3)], -1)
    assert np.all(V.astype(np.float32) == V)
    fs = (4, 5, 6)
    rng = np.random.default_rng(4)
    A = np.diag([0.6, 0.55, 0.5]) + rng.uniform(-0.05, 0.05, (3, 3))
    t = rng.uniform(-0.05, 0.05, 3)
    S = np.eye(3) * 0.9 + rng.uniform(-0.05, 0.05, (3, 3))
    u = (rng.normal(size=fs + (3,)) * 0.02).astype(np.float32)
    T = Transform(A, t, S, -np.ones(3), np.ones(3))
    out = oracle.sample_channels(V.astype(np.float32), fs, u, T, compose=True)
    nV = np.array([Wv, Hv, Dv], np.float64)
    for z in range(fs[0]):
        for y in range(fs[1]):
            for x in range(fs[2]):
                xc = np.array([-1 + 2 * x / (fs[2] - 1), -1 + 2 * y / (fs[1] - 1), -1 + 2 * z / (fs[0] - 1)])
                su = S @ u[z, y, x].astype(np.float64)
                p = A @ xc + t + su
                q = (p + 1) / 2 * (nV - 1)
                assert np.all(q > 0) and np.all(q < nV - 1)
                assert np.allclose(out[z, y, x], su + a @ q + b, atol=1e-12)
    Vc = np.broadcast_to(np.array([0.5, -0.25, 0.125], np.float32), (Dv, Hv, Wv, 3)).copy()
    out = oracle.sample_channels(Vc, fs, u, T, compose=True)
    su = np.einsum("rc,zyxc->zyxr", S, u.astype(np.float64))
    assert np.allclose(out, su + Vc[0, 0, 0], atol=1e-12)


@pytest.mark.parametrize("C", [1, 3])
def test_image_gradient_is_the_adjoint_of_sampling(C):
    # out = S_phi V is linear in V, so dV = S_phi^T g: <dV, W> = <g, S_phi W>
    # for any W.  Points leave the image on purpose (zero padding).
    fs = (5, 6, 7)
    V = _rand((6, 8, 9, C), 5)
    W = _rand((6, 8, 9, C), 6)
    rng = np.random.default_rng(7)
    u = (rng.normal(size=fs + (3,)) * 0.3).astype(np.float32)
    T = _transform(8)
    g = rng.normal(size=fs + (C,))
    _, _, _, dV = oracle.sample_channels_bwd(V, fs, u, T, g)
    lhs = float(np.sum(dV * W.astype(np.float64)))
    rhs = float(np.sum(g * oracle.sample_channels(W, fs, u, T)))
    assert abs(lhs - rhs) <= 1e-12 * max(1.0, abs(rhs))
    # partition of unity: sum over corners of the weights is 1 where all taps are inside
    Ti = Transform(np.eye(3) * 0.5, np.zeros(3), np.eye(3), -np.ones(3), np.ones(3))
    _, _, _, dV1 = oracle.sample_channels_bwd(V, fs, None, Ti, g)
    assert np.allclose(dV1.sum(axis=(0, 1, 2)), g.sum(axis=(0, 1, 2)), atol=1e-12)


def _torch_channels(V, fs, u, T, g, compose):
    """L = sum g * out with out = grid_sample(V, A x + t + S u) (+ S u), float64 autograd."""
    Vt = torch.tensor(np.moveaxis(V, -1, 0), dtype=torch.float64, requires_grad=True)
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
    su = ut @ S.T
    grid = x @ A.T + t + su
    out = Fnn.grid_sample(Vt[None], grid[None], mode="bilinear", padding_mode="zeros", align_corners=True)[0]
    out = out.permute(1, 2, 3, 0)
    if compose:
        out = out + su
    L = (out * torch.tensor(g, dtype=torch.float64)).sum()
    L.backward()
    return (out.detach().numpy(), ut.grad.numpy(), A.grad.numpy(), t.grad.numpy(),
            np.moveaxis(Vt.grad.numpy(), 0, -1))


@pytest.mark.parametrize("C,compose", [(1, False), (2, False), (3, True), (4, False)])
def test_matches_torch_grid_sample_with_autograd(C, compose):
    rng = np.random.default_rng(30 + C)
    fs = (5, 6, 7)
    V = _rand((6, 8, 9, C), 40 + C)
    u = (rng.normal(size=fs + (3,)) * 0.15).astype(np.float32)
    T = _transform(50 + C)
    g = rng.normal(size=fs + (C,))
    out_t, du_t, dA_t, dt_t, dV_t = _torch_channels(V, fs, u, T, g, compose)
    out = oracle.sample_channels(V, fs, u, T, compose=compose)
    du, dA, dt, dV = oracle.sample_channels_bwd(V, fs, u, T, g, compose=compose)
    assert np.max(np.abs(out - out_t)) <= 1e-12
    assert np.max(np.abs(du - du_t)) <= 1e-10
    assert np.max(np.abs(dA - dA_t)) <= 1e-10
    assert np.max(np.abs(dt - dt_t)) <= 1e-10
    assert np.max(np.abs(dV - dV_t)) <= 1e-12


def test_central_differences_of_u_A_t():
    rng = np.random.default_rng(60)
    fs = (4, 5, 6)
    C = 3
    V = _rand((5, 6, 7, C), 61)
    u = (rng.normal(size=fs + (3,)) * 0.1).astype(np.float64)
    T = _transform(62)
    g = rng.normal(size=fs + (C,))
    du, dA, dt, _ = oracle.sample_channels_bwd(V, fs, u.astype(np.float32), T, g, compose=True,
                                               want_dV=False)

    def L(uu=None, A=None, t=None):
        Tx = Transform(T.A if A is None else A, T.t if t is None else t, T.S, T.xmin, T.xmax)
        # float64 u: pass through float32 would round, so perturb only exactly-representable steps
        return float(np.sum(g * oracle.sample_channels(V, fs, (u if uu is None else uu).astype(np.float32),
                                                       Tx, compose=True)))

    h = 2.0 ** -12  # exact in float32 for |u| < 2^11 ulp budget
    u = u.astype(np.float32).astype(np.float64)
    for (z, y, x, c) in [(0, 1, 2, 0), (3, 4, 5, 2), (2, 0, 3, 1)]:
        up = u.copy(); up[z, y, x, c] += h
        um = u.copy(); um[z, y, x, c] -= h
        fd = (L(uu=up) - L(uu=um)) / (2 * h)
        assert abs(fd - du[z, y, x, c]) <= 2e-3 * max(1.0, abs(fd))
    e = 1e-6
    for r in range(3):
        for c in range(3):
            Ap = T.A.copy(); Ap[r, c] += e
            Am = T.A.copy(); Am[r, c] -= e
            fd = (L(A=Ap) - L(A=Am)) / (2 * e)
            assert abs(fd - dA[r, c]) <= 1e-5 * max(1.0, abs(fd))
        tp = T.t.copy(); tp[r] += e
        tm = T.t.copy(); tm[r] -= e
        fd = (L(t=tp) - L(t=tm)) / (2 * e)
        assert abs(fd - dt[r]) <= 1e-5 * max(1.0, abs(fd))


def test_mse_closed_form_and_gradient():
    rng = np.random.default_rng(70)
    F = rng.uniform(0, 1, (3, 4, 5)).astype(np.float32)
    J = rng.uniform(0, 1, (3, 4, 5))
    r = oracle.mse(F, J)
    d = J - F.astype(np.float64)
    assert abs(r["mse"] - float(np.mean(d * d))) <= 1e-15
    # same image: zero loss and zero gradient
    r0 = oracle.mse(F, F.astype(np.float64))
    assert r0["mse"] == 0.0 and np.all(r0["dJ"] == 0.0)
    # central differences (the loss is quadratic: exact up to rounding)
    h = 1e-4
    for k in [0, 17, 59]:
        Jp = J.copy().reshape(-1); Jp[k] += h
        Jm = J.copy().reshape(-1); Jm[k] -= h
        fd = (oracle.mse(F, Jp, False)["mse"] - oracle.mse(F, Jm, False)["mse"]) / (2 * h)
        assert abs(fd - r["dJ"].reshape(-1)[k]) <= 1e-9
    # a constant offset c gives MSE = c^2
    assert abs(oracle.mse(F, F.astype(np.float64) + 0.25)["mse"] - 0.0625) <= 1e-15


def test_mse_objective_finite_differences_through_the_sampler():
    rng = np.random.default_rng(80)
    fs = (4, 5, 6)
    F = rng.uniform(0, 1, fs).astype(np.float32)
    M = rng.uniform(0, 1, (5, 6, 7)).astype(np.float32)
    u = (rng.normal(size=fs + (3,)) * 0.05).astype(np.float32)
    T = _transform(81, 0.1)
    w = 0.75
    r = oracle.objective_mse(F, M, u, T, w)
    J = oracle.grid_sample(M, fs, u, T)
    assert abs(r["loss"][1] - float(np.mean((J - F) ** 2))) <= 1e-15
    assert abs(r["loss"][0] - w * r["loss"][1]) <= 1e-15
    e = 1e-6

    def L(A=None, t=None):
        Tx = Transform(T.A if A is None else A, T.t if t is None else t, T.S, T.xmin, T.xmax)
        return oracle.objective_mse(F, M, u, Tx, w, want_du=False)["loss"][0]

    for rr in range(3):
        tp = T.t.copy(); tp[rr] += e
        tm = T.t.copy(); tm[rr] -= e
        fd = (L(t=tp) - L(t=tm)) / (2 * e)
        assert abs(fd - r["dt"][rr]) <= 1e-5 * max(1.0, abs(fd))
        Ap = T.A.copy(); Ap[rr, 1] += e
        Am = T.A.copy(); Am[rr, 1] -= e
        fd = (L(A=Ap) - L(A=Am)) / (2 * e)
        assert abs(fd - r["dA"][rr, 1]) <= 1e-5 * max(1.0, abs(fd))


def _golden(name):
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.txt")
    for line in open(path):
        line = line.strip()
        if line and not line.startswith("#") and line.split("|")[0].strip() == name:
            _, inp, exp = [s.strip() for s in line.split("|")]
            kv = lambda s: dict(tok.split("=") for tok in s.split())
            num = lambda s: np.array([float(v) for v in s.split(",")])
            return {k: num(v) for k, v in kv(inp).items()}, {k: num(v) for k, v in kv(exp).items()}
    raise KeyError(name)


def test_golden_composition_and_image_gradient():
    inp, exp = _golden("compose_linear2")
    V = np.zeros((2, 2, 2, 3), np.float32)
    for z in range(2):
        for y in range(2):
            for x in range(2):
                for c in range(3):
                    V[z, y, x, c] = (c + 1) * (x + 2 * y + 4 * z)
    u = np.zeros((2, 2, 2, 3), np.float32)
    u[0, 0, 0] = inp["u"]
    # A = 0: the first fixed voxel lands on t + u = p
    T = Transform(np.zeros((3, 3)), inp["p"] - u[0, 0, 0].astype(np.float64), np.eye(3), -np.ones(3), np.ones(3))
    out = oracle.sample_channels(V, (2, 2, 2), u, T, compose=True)
    assert np.allclose(out[0, 0, 0], exp["d"], atol=1e-6)  # u enters as float32
    g = np.zeros((2, 2, 2, 3))
    g[0, 0, 0, 0] = 1.0
    _, _, _, dV = oracle.sample_channels_bwd(V, (2, 2, 2), u, T, g, compose=True)
    assert np.allclose(dV[..., 0].ravel(), exp["dV0"], atol=1e-6)
    assert np.all(dV[..., 1:] == 0.0)


def test_golden_mse():
    inp, exp = _golden("mse_four")
    r = oracle.mse(inp["F"].astype(np.float32), inp["J"])
    assert abs(r["mse"] - exp["MSE"][0]) <= 1e-15
    assert np.allclose(r["dJ"], exp["dJ"], atol=1e-15)
