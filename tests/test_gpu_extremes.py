"""GPU parity at the extreme grid shapes the library accepts: one axis at the
2^20 maximum with the other two at the minimum of 2 voxels (rows of a million
voxels for the lane walk and the LNCC tiles; a million planes for the z
segments; two-voxel axes everywhere else), against the CPU oracle.

Tolerances: |delta| <= 1e-5 on sampled values, relative 1e-4 on losses,
relative 1e-3 (L2) on gradients.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import TOL_GRAD, TOL_J, TOL_LOSS, host, oracle_T, rel_err, rel_l2

pytestmark = pytest.mark.gpu

LONG = 1 << 20
SHAPES = [(2, 2, LONG), (2, LONG, 2), (LONG, 2, 2)]


@pytest.fixture(scope="module")
def ffdp():
    from voxel_grid_sampler_gb300 import build, ffdp as f
    build.build()
    return f


def _cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _smooth_along(shape, seed, long_axis):
    # smooth along the long axis (so the warp moves within a coherent signal), noisy across
    rng = np.random.default_rng(seed)
    n = shape[long_axis]
    x = np.arange(n) / n
    base = 0.5 + 0.3 * np.sin(2 * np.pi * 37 * x) + 0.1 * np.sin(2 * np.pi * 411 * x)
    v = np.broadcast_to(base.reshape([-1 if a == long_axis else 1 for a in range(3)]), shape).copy()
    return (v + rng.normal(size=shape) * 0.01).astype(np.float32)


def _transform(long_axis):
    # a small shift and stretch along the long axis (a few voxels over the million)
    A = np.eye(3, dtype=np.float32)
    t = np.zeros(3, np.float32)
    c = 2 - long_axis  # (x, y, z) component of the long axis
    A[c, c] = 1.0 - 3e-6
    t[c] = 4.0 / LONG
    return A, t


@pytest.mark.parametrize("shape", SHAPES)
def test_objective_on_extreme_grids(ffdp, shape):
    la = shape.index(LONG)
    F = _smooth_along(shape, 1 + la, la)
    M = (1.0 - F ** 2).astype(np.float32)
    u = (np.random.default_rng(5 + la).normal(size=shape + (3,)) * 1e-7).astype(np.float32)
    A, t = _transform(la)
    T = ffdp.transform(A, t)
    fr = (float(F.min()), float(F.max()))
    mr = (float(M.min()), float(M.max()))
    To = oracle_T(A, t)
    for wmi, wln, store in ((1.0, 1.0, False), (1.0, 0.0, True), (1.0, 0.0, False)):
        P = ffdp.objective_params(wmi, wln, 32, fr, mr, 5, 1e-5)
        loss, du, dA, dt = ffdp.ffdp_objective(_cuda(F), _cuda(M), _cuda(u), T, P, store_slope=store)
        ref = oracle.objective(F, M, u, To, oracle.ObjectiveParams(wmi, wln, 32, fr, mr, 5, 1e-5))
        l = host(loss)
        for k in range(3):
            if ref["loss"][k] != 0.0:
                assert rel_err(l[k], ref["loss"][k]) <= TOL_LOSS, (shape, k, l, ref["loss"])
        assert rel_l2(host(du), ref["du"]) <= TOL_GRAD, shape
        assert rel_l2(np.r_[host(dA), host(dt)], np.r_[ref["dA"].ravel(), ref["dt"]]) <= TOL_GRAD, shape


@pytest.mark.parametrize("shape", SHAPES)
def test_sampler_composition_and_step_on_extreme_grids(ffdp, shape):
    la = shape.index(LONG)
    rng = np.random.default_rng(11 + la)
    M = _smooth_along(shape, 21 + la, la)
    u = (rng.normal(size=shape + (3,)) * 1e-7).astype(np.float32)
    A, t = _transform(la)
    T = ffdp.transform(A, t)
    To = oracle_T(A, t)
    J = host(ffdp.ffdp_grid_sample_fwd(_cuda(M), shape, _cuda(u), T))
    assert np.max(np.abs(J - oracle.grid_sample(M, shape, u, To))) <= TOL_J
    V = np.stack([_smooth_along(shape, 31 + la + c, la) * 1e-3 for c in range(3)], -1)
    out = host(ffdp.ffdp_sample_channels_fwd(_cuda(V), shape, _cuda(u), T, True))
    assert np.max(np.abs(out - oracle.sample_channels(V, shape, u, To, True))) <= TOL_J
    g = (rng.normal(size=shape + (3,)) * 1e-4).astype(np.float32)
    P = ffdp.sobolev_adam_params(*(float(np.float32(v)) for v in (0.5, 1e-3, 0.9, 0.999, 1e-8)), 1)
    m1 = torch.zeros(shape + (3,), device="cuda")
    m2 = torch.zeros(shape + (3,), device="cuda")
    uo, loss = ffdp.ffdp_sobolev_adam_step(_cuda(V), _cuda(g), m1, m2, P)
    ref = oracle.sobolev_adam_step(V, g, np.zeros(V.shape), np.zeros(V.shape), P.lambda_, P.lr, P.beta1, P.beta2,
                                   P.eps, 1)
    assert rel_err(host(loss)[0], ref["R"]) <= TOL_LOSS
    assert rel_l2(host(uo) - V, ref["u"] - V) <= 1e-4
