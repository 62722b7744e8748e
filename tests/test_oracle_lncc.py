"""Pins for the oracle's local normalised cross correlation and its gradient.

Paper: "A Scalable Distributed Framework for Multimodal GigaVoxel Image
Registration", Key designs item 2 (LNCC from the window-w sums of I, J, I^2,
J^2 and IJ).  Reading: squared local correlation cross^2/(varI varJ + eps)
from zero-padded w^3 box sums with divisor w^3, averaged over all voxels.

Independent anchors: closed forms (J = aF gives LNCC = 1 everywhere with
eps = 0; J = aF + b gives cc = 1 wherever the window lies inside the grid),
the Cauchy-Schwarz bound 0 <= cc <= 1, the library routine conv3d with
autograd in float64, and central finite differences.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as Fnn

import oracle


def _vol(shape, seed):
    rng = np.random.default_rng(seed)
    return rng.uniform(0.1, 1.0, shape).astype(np.float32)


@pytest.mark.parametrize("a", [2.0, -0.5])
def test_scaled_image_has_unit_lncc(a):
    F = _vol((7, 8, 9), 1)
    r = oracle.lncc(F, a * F.astype(np.float64), 3, eps=0.0, want_cc=True)
    assert abs(r["lncc"] - 1.0) < 1e-12
    assert np.max(np.abs(r["cc"] - 1.0)) < 1e-12


@pytest.mark.parametrize("w", [3, 5])
def test_affine_image_has_unit_cc_in_the_interior(w):
    F = _vol((9, 10, 11), 2)
    J = 1.7 * F.astype(np.float64) + 0.4
    cc = oracle.lncc(F, J, w, eps=0.0, want_cc=True, want_grad=False)["cc"]
    r = (w - 1) // 2
    inner = cc[r:-r, r:-r, r:-r]
    assert np.max(np.abs(inner - 1.0)) < 1e-10
    border = cc.copy()
    border[r:-r, r:-r, r:-r] = 1.0
    assert np.max(np.abs(border - 1.0)) > 1e-3  # zero padding breaks it at the faces


def test_cc_bounded_by_cauchy_schwarz():
    F = _vol((8, 8, 8), 3)
    J = _vol((8, 8, 8), 4).astype(np.float64)
    cc = oracle.lncc(F, J, 5, eps=1e-5, want_cc=True, want_grad=False)["cc"]
    assert cc.min() >= 0.0 and cc.max() <= 1.0


def _torch_lncc(F, J, w, eps):
    r = (w - 1) // 2
    n = float(w ** 3)
    Ft = torch.tensor(F, dtype=torch.float64)[None, None]
    Jt = torch.tensor(J, dtype=torch.float64, requires_grad=True)
    J5 = Jt[None, None]
    k = torch.ones((1, 1, w, w, w), dtype=torch.float64)

    def box(x):
        return Fnn.conv3d(x, k, padding=r)

    sF, sJ, sFF, sJJ, sFJ = box(Ft), box(J5), box(Ft * Ft), box(J5 * J5), box(Ft * J5)
    cross = sFJ - sF * sJ / n
    vF = sFF - sF * sF / n
    vJ = sJJ - sJ * sJ / n
    cc = cross * cross / (vF * vJ + eps)
    L = cc.mean()
    (-L).backward()
    return float(L), cc[0, 0].detach().numpy(), Jt.grad.numpy()


@pytest.mark.parametrize("shape,w", [((6, 7, 8), 3), ((9, 10, 12), 5), ((12, 12, 12), 7)])
def test_matches_conv3d_with_autograd(shape, w):
    F = _vol(shape, 5)
    J = (0.5 * F + 0.5 * _vol(shape, 6)).astype(np.float64)
    L_t, cc_t, dJ_t = _torch_lncc(F, J, w, 1e-5)
    r = oracle.lncc(F, J, w, eps=1e-5, want_cc=True)
    assert abs(r["lncc"] - L_t) < 1e-12
    assert np.max(np.abs(r["cc"] - cc_t)) < 1e-10
    assert np.max(np.abs(r["dJ"] - dJ_t)) < 1e-10 * max(1.0, np.max(np.abs(dJ_t)))


def test_gradient_matches_central_differences():
    F = _vol((6, 7, 8), 7)
    J = (0.3 * F + 0.7 * _vol((6, 7, 8), 8)).astype(np.float64)
    r = oracle.lncc(F, J, 3, eps=1e-5)
    rng = np.random.default_rng(0)
    h = 1e-6
    for _ in range(20):
        idx = tuple(int(rng.integers(0, s)) for s in J.shape)
        Jp = J.copy()
        Jm = J.copy()
        Jp[idx] += h
        Jm[idx] -= h
        fd = -(oracle.lncc(F, Jp, 3, 1e-5, want_grad=False)["lncc"]
               - oracle.lncc(F, Jm, 3, 1e-5, want_grad=False)["lncc"]) / (2 * h)
        assert abs(fd - r["dJ"][idx]) < 1e-6 * max(abs(fd), 1e-4)
