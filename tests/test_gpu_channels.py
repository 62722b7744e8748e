"""GPU parity of the C-channel sampler (warp composition and the image
gradient dV) and of the MSE similarity and fused MSE objective: the CUDA
library through its C ABI against the CPU oracle, element by element, on
seeded inputs spanning several CTA iterations and ragged tails, with samples
leaving the sampled volume, every channel count, and fixed / sampled grids of
different shapes.

Tolerances: |delta| <= 1e-5 on sampled values, relative 1e-4 on losses,
relative 1e-3 (L2) on gradients (du; (dA, dt) as one 12-vector; dV).
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import TOL_GRAD, TOL_J, TOL_LOSS, host, oracle_T, random_transform, rel_err, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ffdp():
    from voxel_grid_sampler_gb300 import build, ffdp as f
    build.build()
    return f


def _cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _field(shape, C, seed, sigma=1.5):
    from voxel_grid_sampler_gb300 import synth
    g = torch.Generator().manual_seed(seed)
    v = torch.stack([synth.gaussian_smooth(torch.rand(shape, generator=g), sigma) for _ in range(C)], -1)
    return ((v - 0.5) * 2.0).numpy().astype(np.float32)


CHAN_CASES = [
    # fixed shape, V shape, channels, compose, displacement scale, transform scale
    ((7, 9, 11), (8, 10, 12), 1, False, 0.05, 0.1),
    ((9, 13, 37), (10, 12, 30), 2, False, 0.05, 0.1),
    ((9, 13, 37), (10, 12, 30), 3, False, 0.05, 0.1),
    ((9, 13, 37), (10, 12, 30), 3, True, 0.05, 0.1),
    ((9, 13, 37), (10, 12, 30), 4, False, 0.05, 0.1),
    ((33, 41, 71), (30, 44, 64), 3, True, 0.03, 0.1),
    ((16, 16, 16), (16, 16, 16), 3, True, 0.4, 0.3),   # many samples leave V
    ((16, 16, 16), (16, 16, 16), 1, False, 0.4, 0.3),
    ((2, 2, 2), (2, 2, 2), 3, True, 0.1, 0.1),            # smallest grids
    ((3, 2, 257), (2, 5, 300), 1, False, 0.05, 0.1),      # elongated, two-voxel axes
    ((2, 3, 130), (4, 2, 129), 4, False, 0.05, 0.1),
]


@pytest.mark.parametrize("fs,vs,C,compose,us,ts", CHAN_CASES)
def test_sample_channels_fwd_bwd(ffdp, fs, vs, C, compose, us, ts):
    rng = np.random.default_rng(sum(fs) + 7 * C + int(compose))
    V = _field(vs, C, 5 + C)
    u = (rng.normal(size=fs + (3,)) * us).astype(np.float32)
    A, t, S, xmin, xmax = random_transform(rng, ts)
    T = ffdp.transform(A, t, S, xmin, xmax)
    To = oracle_T(A, t, S, xmin, xmax)
    out = host(ffdp.ffdp_sample_channels_fwd(_cuda(V), fs, _cuda(u), T, compose))
    outo = oracle.sample_channels(V, fs, u, To, compose)
    assert np.max(np.abs(out - outo)) <= TOL_J
    g = rng.normal(size=fs + (C,)).astype(np.float32)
    du, dA, dt, dV = ffdp.ffdp_sample_channels_bwd(_cuda(V), _cuda(u), T, _cuda(g), compose)
    duo, dAo, dto, dVo = oracle.sample_channels_bwd(V, fs, u, To, g, compose)
    assert rel_l2(host(du), duo) <= TOL_GRAD
    assert rel_l2(np.r_[host(dA), host(dt)], np.r_[dAo.ravel(), dto]) <= TOL_GRAD
    assert rel_l2(host(dV), dVo) <= TOL_GRAD


def test_sample_channels_without_u_and_partial_outputs(ffdp):
    rng = np.random.default_rng(11)
    fs, vs = (10, 12, 14), (9, 11, 15)
    V = _field(vs, 3, 12)
    A, t, S, xmin, xmax = random_transform(rng, 0.1)
    T = ffdp.transform(A, t, S, xmin, xmax)
    To = oracle_T(A, t, S, xmin, xmax)
    out = host(ffdp.ffdp_sample_channels_fwd(_cuda(V), fs, None, T, True))
    assert np.max(np.abs(out - oracle.sample_channels(V, fs, None, To, True))) <= TOL_J
    g = rng.normal(size=fs + (3,)).astype(np.float32)
    # dV only (du, dA, dt skipped) and du only (dV skipped)
    _, _, _, dVo = oracle.sample_channels_bwd(V, fs, None, To, g, True)
    Vd, gd = _cuda(V), _cuda(g)
    dV = torch.empty_like(Vd)
    du, _, _, dV = ffdp.ffdp_sample_channels_bwd(Vd, None, T, gd, True, dV=dV, want_du=False)
    assert du is None and rel_l2(host(dV), dVo) <= TOL_GRAD
    duo, _, _, _ = oracle.sample_channels_bwd(V, fs, None, To, g, True, want_dV=False)
    du, _, _, dV = ffdp.ffdp_sample_channels_bwd(Vd, None, T, gd, True, want_dV=False)
    assert dV is None and rel_l2(host(du), duo) <= TOL_GRAD


def test_identity_and_shift_exact_every_channel(ffdp):
    V = _field((9, 10, 11), 4, 13)
    fs = V.shape[:3]
    out = host(ffdp.ffdp_sample_channels_fwd(_cuda(V), fs, None, ffdp.transform()))
    assert np.max(np.abs(out - V)) == 0.0
    k = np.array([2, -1, 3])
    n = np.array([11, 10, 9])
    out = host(ffdp.ffdp_sample_channels_fwd(_cuda(V), fs, None, ffdp.transform(t=2.0 * k / (n - 1))))
    ref = np.zeros_like(V)
    ref[0:9 - 3, 1:10, 0:11 - 2] = V[3:9, 0:9, 2:11]
    assert np.max(np.abs(out - ref)) <= 1e-6


def test_image_gradient_of_the_moving_image(ffdp):
    # C = 1 on M itself: du, dA, dt equal the scalar sampler backward's, and dV = dM
    rng = np.random.default_rng(14)
    fs, ms = (12, 17, 29), (14, 15, 31)
    M = _field(ms, 1, 15)
    u = (rng.normal(size=fs + (3,)) * 0.05).astype(np.float32)
    A, t, S, xmin, xmax = random_transform(rng, 0.1)
    T = ffdp.transform(A, t, S, xmin, xmax)
    g = rng.normal(size=fs).astype(np.float32)
    du, dA, dt, dM = ffdp.ffdp_sample_channels_bwd(_cuda(M), _cuda(u), T, _cuda(g[..., None]))
    du2, dA2, dt2 = ffdp.ffdp_grid_sample_bwd(_cuda(M[..., 0]), _cuda(u), T, _cuda(g))
    assert rel_l2(host(du), host(du2)) <= 1e-5
    assert rel_l2(np.r_[host(dA), host(dt)], np.r_[host(dA2), host(dt2)]) <= 1e-5
    _, _, _, dMo = oracle.sample_channels_bwd(M, fs, u, oracle_T(A, t, S, xmin, xmax), g[..., None])
    assert rel_l2(host(dM), dMo) <= TOL_GRAD


def test_compose_large_grid(ffdp):
    # several CTA rounds of the persistent grid, rows not a multiple of 32
    rng = np.random.default_rng(16)
    fs = (41, 199, 257)
    V = _field(fs, 3, 17, sigma=3.0) * 0.01
    u = (rng.normal(size=fs + (3,)) * 0.004).astype(np.float32)
    A, t, S, xmin, xmax = random_transform(rng, 0.01)
    T = ffdp.transform(A, t, S, xmin, xmax)
    To = oracle_T(A, t, S, xmin, xmax)
    out = host(ffdp.ffdp_sample_channels_fwd(_cuda(V), fs, _cuda(u), T, True))
    outo = oracle.sample_channels(V, fs, u, To, True)
    assert np.max(np.abs(out - outo)) <= TOL_J
    g = rng.normal(size=fs + (3,)).astype(np.float32)
    du, dA, dt, dV = ffdp.ffdp_sample_channels_bwd(_cuda(V), _cuda(u), T, _cuda(g), True)
    duo, dAo, dto, dVo = oracle.sample_channels_bwd(V, fs, u, To, g, True)
    assert rel_l2(host(du), duo) <= TOL_GRAD
    assert rel_l2(np.r_[host(dA), host(dt)], np.r_[dAo.ravel(), dto]) <= TOL_GRAD
    assert rel_l2(host(dV), dVo) <= TOL_GRAD


# ----------------------------------------------------------------------- MSE
@pytest.mark.parametrize("shape,dt_", [((7, 9, 11), np.float32), ((7, 9, 11), np.float16),
                                       ((16, 16, 16), np.float32), ((33, 41, 77), np.float16)])
def test_mse_on_materialised_J(ffdp, shape, dt_):
    rng = np.random.default_rng(sum(shape))
    F = rng.uniform(0, 1, shape).astype(dt_)
    J = (F.astype(np.float32) + rng.normal(size=shape) * 0.1).astype(np.float32)
    loss, dJ = ffdp.ffdp_mse_fwd_bwd(_cuda(F), _cuda(J))
    r = oracle.mse(F, J)
    assert rel_err(host(loss)[0], r["mse"]) <= TOL_LOSS
    assert rel_l2(host(dJ), r["dJ"]) <= TOL_GRAD
    # J = F: zero loss and gradient
    Ff = F.astype(np.float32)
    loss, dJ = ffdp.ffdp_mse_fwd_bwd(_cuda(F), _cuda(Ff))
    assert host(loss)[0] == 0.0 and not np.any(host(dJ))


MSE_OBJ_CASES = [
    # fixed shape, moving shape, F dtype, M dtype, w_mse
    ((7, 9, 11), (8, 10, 12), np.float32, np.float32, 1.0),
    ((13, 17, 35), (12, 18, 33), np.float16, np.float16, 0.5),
    ((13, 17, 35), (13, 17, 35), np.float32, np.float16, 2.0),
    ((41, 199, 257), (41, 199, 257), np.float32, np.float32, 1.0),
    ((41, 199, 257), (41, 199, 257), np.float16, np.float16, 1.0),
]


@pytest.mark.parametrize("fs,ms,fdt,mdt,w", MSE_OBJ_CASES)
def test_objective_mse(ffdp, fs, ms, fdt, mdt, w):
    from voxel_grid_sampler_gb300 import synth
    rng = np.random.default_rng(sum(fs) + sum(ms))
    g = torch.Generator().manual_seed(sum(fs))
    F = synth.gaussian_smooth(torch.rand(fs, generator=g), 1.5).numpy()
    M = synth.gaussian_smooth(torch.rand(ms, generator=g), 1.5).numpy()
    F, M = F.astype(fdt), M.astype(mdt)
    u = (rng.normal(size=fs + (3,)) * 0.01).astype(np.float32)
    A, t, S, xmin, xmax = random_transform(rng, 0.05)
    T = ffdp.transform(A, t, S, xmin, xmax)
    loss, du, dA, dt = ffdp.ffdp_objective_mse(_cuda(F), _cuda(M), _cuda(u), T, w)
    ref = oracle.objective_mse(F, M, u, oracle_T(A, t, S, xmin, xmax), w)
    l = host(loss)
    assert rel_err(l[0], ref["loss"][0]) <= TOL_LOSS and rel_err(l[1], ref["loss"][1]) <= TOL_LOSS
    assert rel_l2(host(du), ref["du"]) <= TOL_GRAD
    assert rel_l2(np.r_[host(dA), host(dt)], np.r_[ref["dA"].ravel(), ref["dt"]]) <= TOL_GRAD


def test_objective_mse_matches_the_unfused_pipeline(ffdp):
    # fused one-pass objective == sampler -> MSE on J -> sampler backward (all on the GPU)
    rng = np.random.default_rng(21)
    fs = (20, 24, 36)
    F = rng.uniform(0, 1, fs).astype(np.float32)
    M = rng.uniform(0, 1, fs).astype(np.float32)
    u = (rng.normal(size=fs + (3,)) * 0.02).astype(np.float32)
    A, t, S, xmin, xmax = random_transform(rng, 0.05)
    T = ffdp.transform(A, t, S, xmin, xmax)
    Fd, Md, ud = _cuda(F), _cuda(M), _cuda(u)
    loss, du, dA, dt = ffdp.ffdp_objective_mse(Fd, Md, ud, T, 0.75)
    J = ffdp.ffdp_grid_sample_fwd(Md, fs, ud, T)
    l2, gJ = ffdp.ffdp_mse_fwd_bwd(Fd, J)
    du2, dA2, dt2 = ffdp.ffdp_grid_sample_bwd(Md, ud, T, gJ * 0.75)
    assert rel_err(host(loss)[1], host(l2)[0]) <= 1e-5
    assert rel_l2(host(du), host(du2)) <= 1e-5
    assert rel_l2(np.r_[host(dA), host(dt)], np.r_[host(dA2), host(dt2)]) <= 1e-5


def test_no_device_error_after_channel_runs(ffdp):
    assert not ffdp.device_error()
