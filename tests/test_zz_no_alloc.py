"""The workspace-free MI objective (for callers that cannot allocate device
memory: it runs on scratch reserved inside the library image).

Called through the C ABI and checked, on two calls in a row, against
ffdp_objective (caller-provided workspace) and against the double-precision
oracle, within the parity tolerances of the other GPU tests, at a small odd
shape and at a larger one (41 x 199 x 257, several CTA iterations per SM and
a ragged last chunk).  This file is collected last so that a failure here
cannot hide the rest of the suite.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from helpers import TOL_GRAD, TOL_LOSS, oracle_T_of, rel_err, rel_l2

pytestmark = pytest.mark.gpu


def _case(seed, shape=(19, 23, 37), dtype=torch.float32):
    from voxel_grid_sampler_gb300 import synth
    pair = synth.random_pair(shape, seed=seed, device="cpu", dtype=dtype)
    dev = torch.device("cuda")
    return pair, pair.F.to(dev), pair.M.to(dev), pair.u.to(dev)


def _check(got, ref, what):
    assert rel_err(got[0][0], ref[0][0]) <= TOL_LOSS, (what, got[0], ref[0])
    assert rel_err(got[0][1], ref[0][1]) <= TOL_LOSS, (what, got[0], ref[0])
    assert got[0][2] == 0.0
    assert rel_l2(got[1], ref[1]) <= TOL_GRAD, what
    assert rel_l2(np.r_[np.ravel(got[2]), got[3]], np.r_[np.ravel(ref[2]), ref[3]]) <= TOL_GRAD, what


@pytest.mark.parametrize("shape", [(19, 23, 37), (41, 199, 257)])
def test_static_scratch_objective_matches_workspace_objective_and_oracle(shape):
    from voxel_grid_sampler_gb300 import build, ffdp
    build.build()
    for call, (seed, B, dt_) in enumerate([(1, 32, torch.float32), (2, 64, torch.float16)]):
        pair, F, M, u = _case(seed, shape=shape, dtype=dt_)
        T = ffdp.transform(pair.A, pair.t, pair.S, pair.xmin, pair.xmax)
        P = ffdp.objective_params(0.8, 0.0, B, pair.f_range, pair.m_range, 5)
        ref = [x.cpu().numpy() for x in ffdp.ffdp_objective(F, M, u, T, P)]
        o = oracle.objective(pair.F.float().numpy(), pair.M.float().numpy(), pair.u.numpy(), oracle_T_of(pair),
                             oracle.ObjectiveParams(0.8, 0.0, B, pair.f_range, pair.m_range, 5, 1e-5))
        ora = [o["loss"], o["du"], o["dA"], o["dt"]]
        loss = torch.empty(3, device="cuda")
        du = torch.empty(tuple(F.shape) + (3,), device="cuda")
        dA = torch.empty(9, device="cuda")
        dt = torch.empty(3, device="cuda")
        torch.cuda.synchronize()
        before = torch.cuda.memory_allocated()
        ffdp.ffdp_objective_mi_static(F, M, u, T, P, loss, du, dA, dt)
        torch.cuda.synchronize()
        assert torch.cuda.memory_allocated() == before
        got = [x.cpu().numpy() for x in (loss, du, dA, dt)]
        _check(got, ref, ("vs workspace objective", shape, call))
        _check(got, ora, ("vs oracle", shape, call))


def test_static_scratch_objective_rejects_lncc_and_reports_its_size():
    from voxel_grid_sampler_gb300 import build, ffdp
    build.build()
    L = ffdp.lib()
    L.ffdp_static_scratch_bytes.restype = ctypes.c_size_t
    assert L.ffdp_static_scratch_bytes() == 512 * 1024
    pair, F, M, u = _case(3)
    T = ffdp.transform()
    P = ffdp.objective_params(1.0, 1.0, 32, pair.f_range, pair.m_range, 5)
    out = [torch.empty(3, device="cuda"), torch.empty(tuple(F.shape) + (3,), device="cuda"),
           torch.empty(9, device="cuda"), torch.empty(3, device="cuda")]
    with pytest.raises(ffdp.FfdpError) as ei:
        ffdp.ffdp_objective_mi_static(F, M, u, T, P, *out)
    assert ei.value.status == 2 and "MI only" in str(ei.value)
