"""Full-size parity on the five benchmark workloads, in the launch
configuration bench.py times (one ffdp_objective call on the whole volume).

Workloads 1-4 are compared element by element against the oracle on whole
arrays (du in full, dA, dt, all three loss values, and the sampled image J);
workload 5 (1024^3, ~1.07e9 voxels) streams the oracle slab by slab and
compares the losses, dA and dt, du (relative L2 over the whole array, and on
four whole z-planes: the first, two inner and the last) and J (every voxel)
in full -- in both MI modes: stored J and slope (the mode bench.py times) and
implicit.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import TOL_GRAD, TOL_J, TOL_LOSS, oracle_T_of, rel_err, rel_l2, report

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module")
def ffdp():
    from voxel_grid_sampler_gb300 import build, ffdp as f
    build.build()
    return f


def _run_gpu(ffdp, pair, store_slope=False):
    wl = pair.workload
    T = ffdp.transform(pair.A, pair.t, pair.S, pair.xmin, pair.xmax)
    P = ffdp.objective_params(wl.w_mi, wl.w_lncc, wl.bins, pair.f_range, pair.m_range, wl.window, wl.eps)
    loss, du, dA, dt = ffdp.ffdp_objective(pair.F, pair.M, pair.u, T, P, store_slope=store_slope)
    J = ffdp.ffdp_grid_sample_fwd(pair.M, pair.F.shape, pair.u, T)
    torch.cuda.synchronize()
    return loss.cpu().numpy(), du, dA.cpu().numpy(), dt.cpu().numpy(), J


def _oparams(pair):
    wl = pair.workload
    return oracle.ObjectiveParams(wl.w_mi, wl.w_lncc, wl.bins, pair.f_range, pair.m_range, wl.window,
                                  wl.eps)


def _check_losses(l, ref):
    for k in range(3):
        if ref[k] != 0.0:
            assert rel_err(l[k], ref[k]) <= TOL_LOSS, (k, l, ref)
        else:
            assert l[k] == 0.0


@pytest.mark.parametrize("k", [1, 2, 3, 4])
def test_workload_full_arrays(ffdp, k):
    from voxel_grid_sampler_gb300 import synth
    pair = synth.make_pair(k, device="cuda")
    l, du, dA, dt, J = _run_gpu(ffdp, pair)
    F = pair.F.cpu().float().numpy()
    M = pair.M.cpu().float().numpy()
    u = pair.u.cpu().numpy()
    du = du.cpu().numpy()
    J = J.cpu().numpy()
    del pair.F, pair.M, pair.u
    torch.cuda.empty_cache()
    ref = oracle.objective(F, M, u, oracle_T_of(pair), _oparams(pair))
    report("workload %d" % k, J=np.max(np.abs(J - ref["J"])),
           loss=max(rel_err(l[i], ref["loss"][i]) for i in range(3) if ref["loss"][i] != 0),
           du=rel_l2(du, ref["du"]), dAdt=rel_l2(np.r_[dA, dt], np.r_[ref["dA"].ravel(), ref["dt"]]))
    assert np.max(np.abs(J - ref["J"])) <= TOL_J
    _check_losses(l, ref["loss"])
    assert rel_l2(du, ref["du"]) <= TOL_GRAD
    assert rel_l2(np.r_[dA, dt], np.r_[ref["dA"].ravel(), ref["dt"]]) <= TOL_GRAD


@pytest.mark.parametrize("store_slope", [True, False], ids=["stored", "implicit"])
def test_workload5_gigavoxel_streamed(ffdp, store_slope):
    from voxel_grid_sampler_gb300 import synth
    pair = synth.make_pair(5, device="cuda")
    l, du, dA, dt, J = _run_gpu(ffdp, pair, store_slope=store_slope)
    D, H, W = pair.F.shape
    N = pair.F.numel()
    plane = H * W
    planes = [0, 417, 730, D - 1]
    idx = np.unique(np.concatenate([np.random.default_rng(5).choice(N, 4096, replace=False)] +
                                   [np.arange(z * plane, (z + 1) * plane) for z in planes]))
    F = pair.F.cpu().float().numpy()
    M = pair.M.cpu().float().numpy()
    u = pair.u.cpu().numpy()
    del pair.F, pair.M, pair.u
    torch.cuda.empty_cache()
    # du and J compared in full, slab by slab as the streamed oracle produces
    # them (the GPU arrays stay on the device; one slab at a time comes back)
    acc = dict(num=0.0, den=0.0, jmax=0.0, per_plane={})

    def on_slab(z0, z1, du_ref, J_ref):
        g = du[z0:z1].double().cpu().numpy()
        d = g - du_ref
        acc["num"] += float(np.sum(d * d))
        acc["den"] += float(np.sum(du_ref * du_ref))
        jd = J[z0:z1].double().cpu().numpy() - J_ref
        acc["jmax"] = max(acc["jmax"], float(np.max(np.abs(jd))))
        for z in planes:
            if z0 <= z < z1:
                acc["per_plane"][z] = rel_l2(g[z - z0], du_ref[z - z0])

    ref = oracle.objective_mi_slabs(F, M, u, oracle_T_of(pair), _oparams(pair), slab=16, du_index=idx,
                                    on_slab=on_slab)
    du_full = float(np.sqrt(acc["num"] / acc["den"]))
    per_plane = [acc["per_plane"][z] for z in planes]
    report("workload 5 (%s)" % ("stored" if store_slope else "implicit"), J=acc["jmax"],
           loss=rel_err(l[0], ref["loss"][0]), du=du_full, du_planes=max(per_plane),
           dAdt=rel_l2(np.r_[dA, dt], np.r_[ref["dA"].ravel(), ref["dt"]]))
    assert acc["jmax"] <= TOL_J
    _check_losses(l, ref["loss"])
    assert rel_l2(np.r_[dA, dt], np.r_[ref["dA"].ravel(), ref["dt"]]) <= TOL_GRAD
    assert du_full <= TOL_GRAD
    assert max(per_plane) <= TOL_GRAD, per_plane


# ------------------------------------------- next rows at the bench's full size
def _pair_T(ffdp, pair):
    return ffdp.transform(pair.A, pair.t, pair.S, pair.xmin, pair.xmax)


def test_mse_objective_512_full_arrays(ffdp):
    # bench.py --path mse: the one-pass MSE objective on the 512^3 pair
    from voxel_grid_sampler_gb300 import synth
    pair = synth.make_pair(4, device="cuda")
    loss, du, dA, dt = ffdp.ffdp_objective_mse(pair.F, pair.M, pair.u, _pair_T(ffdp, pair), 1.0)
    torch.cuda.synchronize()
    l, du, dA, dt = loss.cpu().numpy(), du.cpu().numpy(), dA.cpu().numpy(), dt.cpu().numpy()
    F = pair.F.cpu().float().numpy()
    M = pair.M.cpu().float().numpy()
    u = pair.u.cpu().numpy()
    del pair.F, pair.M, pair.u
    torch.cuda.empty_cache()
    ref = oracle.objective_mse(F, M, u, oracle_T_of(pair), 1.0)
    report("mse 512^3", loss=rel_err(l[1], ref["loss"][1]), du=rel_l2(du, ref["du"]),
           dAdt=rel_l2(np.r_[dA, dt], np.r_[ref["dA"].ravel(), ref["dt"]]))
    assert rel_err(l[0], ref["loss"][0]) <= TOL_LOSS and rel_err(l[1], ref["loss"][1]) <= TOL_LOSS
    assert rel_l2(du, ref["du"]) <= TOL_GRAD
    assert rel_l2(np.r_[dA, dt], np.r_[ref["dA"].ravel(), ref["dt"]]) <= TOL_GRAD


def test_compose_512_sampled_planes_and_adjoint(ffdp):
    # bench.py --path compose: the pair's field composed with itself on 512^3.
    # out and du on sampled planes and dA, dt in full against the oracle; dV
    # (the whole 512^3 x 3 volume) through the adjoint identity
    # <dV, W> = <gout, sample(W)> for a random W, both sides on the GPU.
    from voxel_grid_sampler_gb300 import synth
    pair = synth.make_pair(4, device="cuda")
    T = _pair_T(ffdp, pair)
    V, u = pair.u, pair.u
    shape = tuple(pair.F.shape)
    g = torch.Generator(device="cuda").manual_seed(7)
    gout = torch.randn(shape + (3,), device="cuda", generator=g)
    out = ffdp.ffdp_sample_channels_fwd(V, shape, u, T, True)
    du, dA, dt, dV = ffdp.ffdp_sample_channels_bwd(V, u, T, gout, True)
    W = torch.randn(V.shape, device="cuda", generator=g)
    outW = ffdp.ffdp_sample_channels_fwd(W, shape, u, T, False)
    lhs = float((dV.double() * W.double()).sum())
    rhs = float((gout.double() * outW.double()).sum())
    del W, outW
    To = oracle_T_of(pair)
    Vh, uh = V.cpu().numpy(), u.cpu().numpy()
    planes = [0, 1, 255, 511]
    for z in planes:
        o = oracle.sample_channels(Vh, shape, uh, To, True, z, z + 1)
        assert np.max(np.abs(out[z].cpu().numpy() - o[0])) <= TOL_J
    gh = gout.cpu().numpy()
    dA_o = np.zeros(9)
    dt_o = np.zeros(3)
    du_o, _, _, _ = oracle.sample_channels_bwd(Vh, shape, uh, To, gh, True, want_dV=False, dA=dA_o, dt=dt_o)
    du = du.cpu().numpy()
    report("compose 512^3", adjoint=abs(lhs - rhs) / abs(rhs), du=rel_l2(du, du_o),
           dAdt=rel_l2(np.r_[dA.cpu().numpy(), dt.cpu().numpy()], np.r_[dA_o, dt_o]))
    assert abs(lhs - rhs) <= 1e-4 * abs(rhs)
    assert rel_l2(du, du_o) <= TOL_GRAD
    assert rel_l2(np.r_[dA.cpu().numpy(), dt.cpu().numpy()], np.r_[dA_o, dt_o]) <= TOL_GRAD


def test_adam_step_512_full_arrays(ffdp):
    # bench.py --path adam: the regularised Adam step on the 512^3 pair's field (vector form)
    from voxel_grid_sampler_gb300 import synth
    pair = synth.make_pair(4, device="cuda")
    u = pair.u
    del pair.F, pair.M
    torch.cuda.empty_cache()
    g = torch.Generator(device="cuda").manual_seed(2025)
    gr = torch.randn(u.shape, device="cuda", generator=g) * 1e-6
    m1 = torch.randn(u.shape, device="cuda", generator=g) * 1e-7
    m2 = torch.rand(u.shape, device="cuda", generator=g) * 1e-12
    lam, lr, b1, b2, eps = (float(np.float32(v)) for v in (0.1, 1e-3, 0.9, 0.999, 1e-8))
    uh, gh, m1h, m2h = (x.cpu().numpy() for x in (u, gr, m1, m2))
    uo, loss = ffdp.ffdp_sobolev_adam_step(u, gr, m1, m2, ffdp.sobolev_adam_params(lam, lr, b1, b2, eps, 7))
    torch.cuda.synchronize()
    ref = oracle.sobolev_adam_step(uh, gh, m1h, m2h, lam, lr, b1, b2, eps, 7)
    upd = uo.cpu().numpy().astype(np.float64) - uh
    report("adam 512^3", R=rel_err(loss.item(), ref["R"]), update=rel_l2(upd, ref["u"] - uh),
           m1=rel_l2(m1.cpu().numpy(), ref["m1"]), m2=rel_l2(m2.cpu().numpy(), ref["m2"]))
    assert rel_err(loss.item(), ref["R"]) <= TOL_LOSS
    assert rel_l2(upd, ref["u"] - uh) <= 1e-4
    assert rel_l2(m1.cpu().numpy(), ref["m1"]) <= 1e-5
    assert rel_l2(m2.cpu().numpy(), ref["m2"]) <= 1e-5
