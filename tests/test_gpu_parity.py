"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle,
element by element, on seeded inputs that span several CTA iterations / tiles
and ragged tails, plus the degenerate cases (identity, integer shifts, samples
outside the moving image, clamped intensities).

Tolerances: |dJ| <= 1e-5 on sampled intensities, relative 1e-4 on losses,
relative 1e-3 (L2) on gradients.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import (TOL_GRAD, TOL_J, TOL_LOSS, host, oracle_T, random_transform, rel_err, rel_l2)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ffdp():
    from voxel_grid_sampler_gb300 import build, ffdp as f
    build.build()
    return f


def _vol(shape, seed, lo=0.0, hi=1.0, dtype=np.float32, sigma=1.0):
    from voxel_grid_sampler_gb300 import synth
    g = torch.Generator().manual_seed(seed)
    v = synth.gaussian_smooth(torch.rand(shape, generator=g), sigma)
    v = (v - v.min()) / (v.max() - v.min()) * (hi - lo) + lo
    return v.numpy().astype(dtype)


def _cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


# ------------------------------------------------------------------ sampler
SAMPLER_CASES = [
    # fixed shape, moving shape, M dtype, displacement scale, transform scale
    ((7, 9, 11), (8, 10, 12), np.float32, 0.05, 0.1),
    ((5, 5, 17), (5, 5, 17), np.float16, 0.05, 0.05),
    ((33, 41, 71), (30, 44, 64), np.float32, 0.03, 0.1),
    ((16, 16, 16), (16, 16, 16), np.float32, 0.4, 0.3),  # many samples fall outside M
]


@pytest.mark.parametrize("fs,ms,mdt,us,ts", SAMPLER_CASES)
def test_grid_sample_fwd_bwd(ffdp, fs, ms, mdt, us, ts):
    rng = np.random.default_rng(hash((fs, ms)) % 2**31)
    M = _vol(ms, 1, -0.5, 1.5, mdt)
    u = (rng.normal(size=fs + (3,)) * us).astype(np.float32)
    A, t, S, xmin, xmax = random_transform(rng, ts)
    T = ffdp.transform(A, t, S, xmin, xmax)
    To = oracle_T(A, t, S, xmin, xmax)
    J = host(ffdp.ffdp_grid_sample_fwd(_cuda(M), fs, _cuda(u), T))
    Jo = oracle.grid_sample(M, fs, u, To)
    assert np.max(np.abs(J - Jo)) <= TOL_J
    g = rng.normal(size=fs).astype(np.float32)
    du, dA, dt = ffdp.ffdp_grid_sample_bwd(_cuda(M), _cuda(u), T, _cuda(g))
    duo, dAo, dto = oracle.grid_sample_bwd(M, fs, u, To, g)
    assert rel_l2(host(du), duo) <= TOL_GRAD
    assert rel_l2(np.r_[host(dA), host(dt)], np.r_[dAo, dto]) <= TOL_GRAD


def test_identity_and_integer_shift_exact(ffdp):
    M = _vol((9, 10, 11), 3)
    fs = M.shape
    J = host(ffdp.ffdp_grid_sample_fwd(_cuda(M), fs, None, ffdp.transform()))
    assert np.max(np.abs(J - M)) == 0.0
    k = np.array([2, -1, 3])
    n = np.array([11, 10, 9])
    J = host(ffdp.ffdp_grid_sample_fwd(_cuda(M), fs, None, ffdp.transform(t=2.0 * k / (n - 1))))
    ref = np.zeros_like(M)
    ref[0:9 - 3, 1:10, 0:11 - 2] = M[3:9, 0:9, 2:11]
    assert np.max(np.abs(J - ref)) <= 1e-6


# ----------------------------------------------------------------------- MI
@pytest.mark.parametrize("B", [8, 16, 32, 40, 64])
@pytest.mark.parametrize("fdt", [np.float32, np.float16])
def test_mi_fwd_bwd(ffdp, B, fdt):
    shape = (19, 23, 37)  # 16169 voxels: several CTA iterations and a ragged tail
    F = _vol(shape, 5, 0.0, 1.0, fdt)
    J = (0.6 * _vol(shape, 5).astype(np.float64) + 0.4 * _vol(shape, 6)).astype(np.float32)
    f_range = (float(F.min()), float(F.max()))
    j_range = (0.1, 0.85)  # part of J is clamped
    p = ffdp.mi_params(B, f_range, j_range)
    loss, dJ = ffdp.ffdp_mi_fwd_bwd(_cuda(F), _cuda(J), p)
    r = oracle.mi(F, J.astype(np.float64), B, f_range, j_range)
    assert rel_err(host(loss)[0], -r["mi"]) <= TOL_LOSS
    assert rel_l2(host(dJ), r["dJ"]) <= TOL_GRAD


def test_mi_is_deterministic_and_order_free(ffdp):
    # The histogram is integer fixed point: the result does not depend on the
    # order in which CTAs and lanes add their voxels (partial aggregation).
    shape = (24, 32, 40)
    F = _vol(shape, 7)
    J = _vol(shape, 8)
    p = ffdp.mi_params(32, (0.0, 1.0), (0.0, 1.0))
    l1, _ = ffdp.ffdp_mi_fwd_bwd(_cuda(F), _cuda(J), p, want_grad=False)
    l2, _ = ffdp.ffdp_mi_fwd_bwd(_cuda(F), _cuda(J), p, want_grad=False)
    perm = np.random.default_rng(0).permutation(F.size)
    Fp = F.reshape(-1)[perm].reshape(shape)
    Jp = J.reshape(-1)[perm].reshape(shape)
    l3, _ = ffdp.ffdp_mi_fwd_bwd(_cuda(Fp), _cuda(Jp), p, want_grad=False)
    a, b, c = host(l1)[0], host(l2)[0], host(l3)[0]
    assert a == b == c


# --------------------------------------------------------------------- LNCC
LNCC_CASES = [((20, 37, 70), 5), ((9, 16, 32), 3), ((13, 17, 45), 7), ((11, 12, 40), 9), ((70, 17, 6), 5),
              # windows above 7: the separable wide-window passes; 13 and 21
              # are wider than some axes (clipped sums, divisor still w^3)
              ((20, 37, 70), 11), ((9, 16, 32), 13), ((13, 17, 45), 21),
              # wider than every axis: every window holds the whole grid (the
              # radius is capped at the largest extent, the divisor stays w^3)
              ((9, 16, 32), 101)]


@pytest.mark.parametrize("shape,w", LNCC_CASES)
@pytest.mark.parametrize("fdt", [np.float32, np.float16])
def test_lncc_fwd_bwd(ffdp, shape, w, fdt):
    F = _vol(shape, 11, 0.0, 1.0, fdt)
    J = (0.5 * F.astype(np.float64) + 0.5 * _vol(shape, 12)).astype(np.float32)
    p = ffdp.lncc_params(w, 1e-5)
    loss, dJ = ffdp.ffdp_lncc_fwd_bwd(_cuda(F), _cuda(J), p)
    r = oracle.lncc(F, J.astype(np.float64), w, 1e-5)
    assert rel_err(host(loss)[0], -r["lncc"]) <= TOL_LOSS
    assert rel_l2(host(dJ), r["dJ"]) <= TOL_GRAD


def test_wide_window_loss_only_matches_full_call(ffdp):
    # the wide-window passes without a dL/dJ output give the same loss
    F = _vol((14, 19, 45), 15, 0.0, 1.0)
    J = (0.6 * F.astype(np.float64) + 0.4 * _vol((14, 19, 45), 16)).astype(np.float32)
    p = ffdp.lncc_params(15, 1e-5)
    l1, dJ = ffdp.ffdp_lncc_fwd_bwd(_cuda(F), _cuda(J), p)
    l2, none = ffdp.ffdp_lncc_fwd_bwd(_cuda(F), _cuda(J), p, want_grad=False)
    assert none is None and host(l1)[0] == host(l2)[0]
    r = oracle.lncc(F, J.astype(np.float64), 15, 1e-5)
    assert rel_err(host(l2)[0], -r["lncc"]) <= TOL_LOSS


def test_lncc_of_scaled_image_is_one(ffdp):
    F = _vol((12, 20, 36), 13, 0.2, 1.0)
    J = (3.0 * F).astype(np.float32)
    loss, _ = ffdp.ffdp_lncc_fwd_bwd(_cuda(F), _cuda(J), ffdp.lncc_params(5, 0.0), want_grad=False)
    assert abs(host(loss)[0] + 1.0) <= 1e-4


# ---------------------------------------------------------------- objective
OBJ_CASES = [
    # fixed, moving, dtype, w_mi, w_lncc, bins, window
    ((18, 21, 35), (20, 22, 33), np.float32, 1.0, 1.0, 32, 5),
    ((18, 21, 35), (18, 21, 35), np.float32, 0.7, 0.0, 64, 5),
    ((18, 21, 35), (18, 21, 35), np.float32, 0.0, 1.3, 32, 7),
    ((17, 19, 37), (17, 19, 37), np.float16, 1.0, 0.5, 48, 3),
    # window 9 (the separable wide-window passes) with the MI term fused, both table sizes
    ((16, 18, 40), (16, 18, 40), np.float32, 1.0, 1.0, 64, 9),
    ((15, 17, 33), (15, 17, 33), np.float16, 1.0, 0.5, 32, 9),
    # rows a multiple of 4 voxels: full tiles stage the stored slope by 16-byte
    # copies, the ragged last tile in x and y by 4-byte copies
    ((19, 37, 100), (19, 37, 100), np.float32, 1.0, 1.0, 64, 5),
    ((12, 16, 64), (12, 16, 64), np.float32, 0.5, 1.0, 32, 9),
    ((10, 48, 96), (10, 48, 96), np.float16, 0.0, 1.0, 32, 3),
    # windows above 7 (wide-window passes), with and without the MI term
    ((16, 18, 40), (16, 18, 40), np.float32, 1.0, 1.0, 64, 11),
    ((15, 17, 33), (15, 17, 33), np.float16, 1.0, 0.5, 32, 13),
    ((12, 16, 64), (12, 16, 64), np.float32, 0.0, 1.0, 32, 11),
]


@pytest.mark.parametrize("store", [False, True])
@pytest.mark.parametrize("fs,ms,dt_,wmi,wln,B,w", OBJ_CASES)
def test_objective(ffdp, fs, ms, dt_, wmi, wln, B, w, store):
    rng = np.random.default_rng(sum(fs) + B + w)
    F = _vol(fs, 21, 0.0, 1.0, dt_)
    M = _vol(ms, 22, 0.0, 1.0, dt_)
    u = (rng.normal(size=fs + (3,)) * 0.04).astype(np.float32)
    A, t, S, xmin, xmax = random_transform(rng, 0.08)
    fr = (float(F.min()), float(F.max()))
    mr = (float(M.min()), float(M.max()))
    T = ffdp.transform(A, t, S, xmin, xmax)
    P = ffdp.objective_params(wmi, wln, B, fr, mr, w, 1e-5)
    loss, du, dA, dt = ffdp.ffdp_objective(_cuda(F), _cuda(M), _cuda(u), T, P, store_slope=store)
    ref = oracle.objective(F, M, u, oracle_T(A, t, S, xmin, xmax),
                           oracle.ObjectiveParams(wmi, wln, B, fr, mr, w, 1e-5))
    l = host(loss)
    for k in range(3):
        if ref["loss"][k] != 0.0:
            assert rel_err(l[k], ref["loss"][k]) <= TOL_LOSS, (k, l, ref["loss"])
        else:
            assert l[k] == 0.0
    assert rel_l2(host(du), ref["du"]) <= TOL_GRAD
    assert rel_l2(np.r_[host(dA), host(dt)], np.r_[ref["dA"].ravel(), ref["dt"]]) <= TOL_GRAD


# Larger grids: several CTA iterations per persistent CTA (the streamed-input
# ring wraps), rows that are not a multiple of 32 voxels and a ragged last
# chunk.  M is an intensity remap of F (as in the registration workloads), so
# MI is of order 1 instead of the near-zero MI of two independent volumes,
# whose relative error is ill-conditioned.
LARGE_CASES = [
    # shape, dtype, w_mi, w_lncc, bins, window, store_slope
    ((41, 199, 257), np.float32, 1.0, 1.0, 64, 5, False),
    ((41, 199, 257), np.float16, 1.0, 0.0, 32, 5, False),
    ((41, 199, 257), np.float16, 1.0, 0.0, 32, 5, True),
    ((41, 199, 257), np.float32, 1.0, 0.0, 64, 5, True),
]


@pytest.mark.parametrize("fs,dt_,wmi,wln,B,w,store", LARGE_CASES)
def test_objective_large(ffdp, fs, dt_, wmi, wln, B, w, store):
    rng = np.random.default_rng(sum(fs) + B)
    base = _vol(fs, 23, sigma=2.0)
    F = base.astype(dt_)
    M = (1.0 - base ** 2 + rng.normal(size=fs) * 0.01).astype(dt_)
    u = (rng.normal(size=fs + (3,)) * 0.002).astype(np.float32)
    A, t, S, _, _ = random_transform(rng, 0.003)
    xmin, xmax = np.full(3, -1.0, np.float32), np.full(3, 1.0, np.float32)  # grids aligned
    fr = (float(F.min()), float(F.max()))
    mr = (float(M.min()), float(M.max()))
    T = ffdp.transform(A, t, S, xmin, xmax)
    P = ffdp.objective_params(wmi, wln, B, fr, mr, w, 1e-5)
    loss, du, dA, dt = ffdp.ffdp_objective(_cuda(F), _cuda(M), _cuda(u), T, P, store_slope=store)
    ref = oracle.objective(F, M, u, oracle_T(A, t, S, xmin, xmax),
                           oracle.ObjectiveParams(wmi, wln, B, fr, mr, w, 1e-5))
    l = host(loss)
    assert abs(ref["loss"][1]) > 0.05  # MI of order 1
    for k in range(3):
        if ref["loss"][k] != 0.0:
            assert rel_err(l[k], ref["loss"][k]) <= TOL_LOSS, (k, l, ref["loss"])
    assert rel_l2(host(du), ref["du"]) <= TOL_GRAD
    assert rel_l2(np.r_[host(dA), host(dt)], np.r_[ref["dA"].ravel(), ref["dt"]]) <= TOL_GRAD


def test_objective_is_deterministic(ffdp):
    rng = np.random.default_rng(3)
    fs = (16, 20, 24)
    F = _vol(fs, 31)
    M = _vol(fs, 32)
    u = (rng.normal(size=fs + (3,)) * 0.03).astype(np.float32)
    T = ffdp.transform()
    P = ffdp.objective_params(1.0, 1.0, 32, (0.0, 1.0), (0.0, 1.0), 5)
    r1 = [host(x) for x in ffdp.ffdp_objective(_cuda(F), _cuda(M), _cuda(u), T, P)]
    r2 = [host(x) for x in ffdp.ffdp_objective(_cuda(F), _cuda(M), _cuda(u), T, P)]
    for a, b in zip(r1, r2):
        assert np.array_equal(a, b)


def test_workspace_is_independent_of_volume_size_for_mi(ffdp):
    p = ffdp.objective_params(1.0, 0.0, 64, (0, 1), (0, 1), 5)
    a = ffdp.ffdp_workspace_bytes(ffdp.FFDP_OP_OBJECTIVE, (64, 64, 64), p)
    b = ffdp.ffdp_workspace_bytes(ffdp.FFDP_OP_OBJECTIVE, (512, 512, 512), p)
    assert a == b and a < (1 << 20)
    # stored J and slope (ffdp_objective_stored): 16 bytes per voxel on top
    c = ffdp.ffdp_workspace_bytes(ffdp.FFDP_OP_OBJECTIVE_STORED, (512, 512, 512), p)
    assert 16 * 512 ** 3 <= c - a <= 16 * 512 ** 3 + 4096
    # LNCC on: the same two per-voxel buffers (the sampler backward runs in the
    # backward window kernel), the three g-terms the forward window kernel
    # hands it (12 bytes per voxel), plus the 64-bin polynomial cells
    r = ffdp.objective_params(0.5, 0.5, 64, (0, 1), (0, 1), 5)
    d = ffdp.ffdp_workspace_bytes(ffdp.FFDP_OP_OBJECTIVE, (512, 512, 512), r)
    assert 28 * 512 ** 3 <= d - a <= 28 * 512 ** 3 + 64 * 64 * 12 * 4 + 4096


def test_no_device_error_after_runs(ffdp):
    # every bounded wait of the sweeps above completed
    assert not ffdp.device_error()
