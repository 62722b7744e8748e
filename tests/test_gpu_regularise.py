"""GPU parity of the Sobolev regulariser and the fused regularised Adam step
of the displacement field against the CPU oracle, on ragged grids (rows and
volumes not a multiple of the 32-voxel warp groups) and over several steps.

Tolerances: relative 1e-4 on the regulariser value, relative 1e-3 (L2) on its
gradient, relative 1e-4 (L2) on the update u_out - u and 1e-5 on the moments.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import TOL_GRAD, TOL_LOSS, host, rel_err, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ffdp():
    from voxel_grid_sampler_gb300 import build, ffdp as f
    build.build()
    return f


def _cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _field(shape, seed, scale=0.01):
    from voxel_grid_sampler_gb300 import synth
    g = torch.Generator().manual_seed(seed)
    v = torch.stack([synth.gaussian_smooth(torch.randn(shape, generator=g), 2.0) for _ in range(3)], -1)
    return (v * scale / v.abs().max()).numpy().astype(np.float32)


# W and N multiples of 4 take the 16-byte vector form, the others the per-voxel form
SHAPES = [(2, 2, 2), (5, 7, 33), (9, 31, 17), (17, 19, 45), (16, 32, 64), (5, 7, 32), (3, 3, 4), (7, 9, 20)]


@pytest.mark.parametrize("shape", SHAPES)
def test_sobolev_fwd_bwd(ffdp, shape):
    u = _field(shape, sum(shape))
    loss, dR = ffdp.ffdp_sobolev_fwd_bwd(_cuda(u), 0.8)
    r = oracle.sobolev(u, 0.8)
    assert rel_err(host(loss)[0], r["R"]) <= TOL_LOSS
    assert rel_l2(host(dR), r["dR"]) <= TOL_GRAD


@pytest.mark.parametrize("shape", SHAPES[1:])
def test_sobolev_adam_steps(ffdp, shape):
    rng = np.random.default_rng(sum(shape))
    u = _field(shape, 2 * sum(shape))
    # the parameters the library receives are float32: hand the oracle the same values
    lam, lr, b1, b2, eps = (float(np.float32(v)) for v in (0.5, 1e-3, 0.9, 0.999, 1e-8))
    m1 = np.zeros(u.shape)
    m2 = np.zeros(u.shape)
    ud, m1d, m2d = _cuda(u), _cuda(m1.astype(np.float32)), _cuda(m2.astype(np.float32))
    uo = torch.empty_like(ud)
    for t in range(1, 4):
        g = (rng.normal(size=u.shape) * 1e-4).astype(np.float32)
        P = ffdp.sobolev_adam_params(lam, lr, b1, b2, eps, t)
        uo, loss = ffdp.ffdp_sobolev_adam_step(ud, _cuda(g), m1d, m2d, P, u_out=uo)
        ref = oracle.sobolev_adam_step(host(ud), g, m1, m2, lam, lr, b1, b2, eps, t)
        assert rel_err(host(loss)[0], ref["R"]) <= TOL_LOSS
        assert rel_l2(host(uo) - host(ud), ref["u"] - host(ud)) <= 1e-4
        assert rel_l2(host(m1d), ref["m1"]) <= 1e-5
        assert rel_l2(host(m2d), ref["m2"]) <= 1e-5
        m1, m2 = ref["m1"], ref["m2"]          # continue both sides from their own state
        ud, uo = uo, ud                        # ping-pong


def test_step_and_mse_objective_are_bitwise_reproducible(ffdp):
    # fixed-order reductions, no float atomics on these paths
    rng = np.random.default_rng(9)
    shape = (12, 20, 36)
    u = _cuda(_field(shape, 31))
    g = _cuda((rng.normal(size=shape + (3,)) * 1e-4).astype(np.float32))
    P = ffdp.sobolev_adam_params(0.3, 1e-3, 0.9, 0.999, 1e-8, 2)
    outs = []
    for _ in range(2):
        m1 = torch.full_like(u, 1e-5)
        m2 = torch.full_like(u, 1e-9)
        uo, loss = ffdp.ffdp_sobolev_adam_step(u, g, m1, m2, P)
        outs.append([host(x) for x in (uo, loss, m1, m2)])
    for a, b in zip(*outs):
        assert np.array_equal(a, b)
    F = _cuda(rng.uniform(0, 1, shape).astype(np.float32))
    M = _cuda(rng.uniform(0, 1, shape).astype(np.float32))
    T = ffdp.transform()
    r1 = [host(x) for x in ffdp.ffdp_objective_mse(F, M, u, T, 1.0)]
    r2 = [host(x) for x in ffdp.ffdp_objective_mse(F, M, u, T, 1.0)]
    for a, b in zip(r1, r2):
        assert np.array_equal(a, b)
