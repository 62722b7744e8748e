"""Failure reporting of the sweeps' bounded waits, without a GPU fault.

The library's test hook arms the first ring slot of the next objective call
with 16 bytes that never arrive, so every wait on it runs out (about one
second each).  The call must report through ffdp_device_error and NaN losses,
leave no copy in flight, and the next normal call must be correct again.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import TOL_GRAD, TOL_LOSS, host, oracle_T, random_transform, rel_err, rel_l2

pytestmark = pytest.mark.gpu


def _case():
    from voxel_grid_sampler_gb300 import synth
    g = torch.Generator().manual_seed(71)
    base = synth.gaussian_smooth(torch.rand((32, 48, 64), generator=g), 2.0)
    base = ((base - base.min()) / (base.max() - base.min())).numpy().astype(np.float32)
    M = (1.0 - base ** 2).astype(np.float32)
    rng = np.random.default_rng(72)
    u = (rng.normal(size=base.shape + (3,)) * 0.002).astype(np.float32)
    return base, M, u, random_transform(rng, 0.01)


def test_ring_wait_runs_out_and_reports():
    from voxel_grid_sampler_gb300 import build, ffdp
    build.build()
    # generic sample positions (not on grid points, where the slope is one-sided)
    F, M, u, (A, t, S, xmin, xmax) = _case()
    fr, mr = (float(F.min()), float(F.max())), (float(M.min()), float(M.max()))
    T = ffdp.transform(A, t, S, xmin, xmax)
    P = ffdp.objective_params(1.0, 0.0, 32, fr, mr, 5)
    Fd, Md, ud = (torch.from_numpy(x).cuda() for x in (F, M, u))
    ffdp.device_error()  # start from a clear word
    ffdp.test_ring_stall(True)
    loss, du, dA, dt = ffdp.ffdp_objective(Fd, Md, ud, T, P)
    torch.cuda.synchronize()
    assert ffdp.device_error()
    assert np.all(np.isnan(host(loss)))
    # the context stays usable and the next call is correct
    loss, du, dA, dt = ffdp.ffdp_objective(Fd, Md, ud, T, P)
    torch.cuda.synchronize()
    assert not ffdp.device_error()
    ref = oracle.objective(F, M, u, oracle_T(A, t, S, xmin, xmax),
                           oracle.ObjectiveParams(1.0, 0.0, 32, fr, mr, 5, 1e-5))
    assert rel_err(host(loss)[0], ref["loss"][0]) <= TOL_LOSS
    assert rel_l2(host(du), ref["du"]) <= TOL_GRAD
