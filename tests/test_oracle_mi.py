"""Pins for the oracle's Mattes mutual information and its gradient.

Paper: "A Scalable Distributed Framework for Multimodal GigaVoxel Image
Registration", Key designs item 2 (MI as the KL divergence of P(X,Y) from
P(X)P(Y), Parzen estimate P_I(v) = (1/N) sum_k kappa(v - I_k) on B bins; the
naive form materialises Psi_I(j,k) = kappa(b_j - I_k)) and item 5 (local
histograms merged with weights N_h/N).

Independent anchors: scipy's B-spline basis element, the 4-fold convolution
of the unit box, the dense Psi construction of the naive method, closed-form
MI values (ln K for K well-separated voxels; the entropy of F for the box
kernel), MI invariances, slab aggregation and central differences.
"""
import math

import numpy as np
import pytest
from scipy.interpolate import BSpline

import oracle

_CUBIC = BSpline.basis_element([-2.0, -1.0, 0.0, 1.0, 2.0], extrapolate=False)


def _beta_scipy(s):
    v = _CUBIC(np.asarray(s, np.float64))
    return np.nan_to_num(v, nan=0.0)


def test_bspline_values_and_partition_of_unity():
    assert oracle.bspline(0.0) == pytest.approx(2.0 / 3.0, abs=1e-15)
    assert oracle.bspline(1.0) == pytest.approx(1.0 / 6.0, abs=1e-15)
    assert oracle.bspline(-1.0) == pytest.approx(1.0 / 6.0, abs=1e-15)
    assert oracle.bspline(2.0) == 0.0 and oracle.bspline(-2.0) == 0.0
    rng = np.random.default_rng(0)
    for c in rng.uniform(2, 20, 50):
        js = np.arange(int(c) - 3, int(c) + 4)
        assert abs(sum(oracle.bspline(j - c) for j in js) - 1.0) < 1e-14
        assert abs(sum(oracle.bspline_deriv(j - c) for j in js)) < 1e-14


def test_bspline_matches_scipy_and_box_convolution():
    s = np.linspace(-2.5, 2.5, 1001)
    ours = np.array([oracle.bspline(v) for v in s])
    assert np.max(np.abs(ours - _beta_scipy(s))) < 1e-14
    # the cubic B-spline is the unit box convolved with itself four times
    h = 1e-3
    x = np.arange(-0.5, 0.5, h) + h / 2
    box = np.ones_like(x)
    k = box
    for _ in range(3):
        k = np.convolve(k, box) * h
    grid = (np.arange(k.size) - (k.size - 1) / 2) * h
    ours_g = np.array([oracle.bspline(v) for v in grid])
    assert np.max(np.abs(ours_g - k)) < 2e-6
    # derivative against central differences of scipy's spline
    for v in np.linspace(-1.95, 1.95, 37):
        fd = (_beta_scipy(v + 1e-6) - _beta_scipy(v - 1e-6)) / 2e-6
        assert abs(oracle.bspline_deriv(v) - fd) < 1e-7


def test_bin_coordinate_map():
    B, lo, hi = 32, -0.5, 1.5
    assert oracle.bin_coord(lo, lo, hi, B)[0] == pytest.approx(2.0)
    assert oracle.bin_coord(hi, lo, hi, B)[0] == pytest.approx(B - 3.0)
    c, d = oracle.bin_coord(0.5, lo, hi, B)
    assert c == pytest.approx(2.0 + 0.5 * (B - 5)) and d == pytest.approx((B - 5) / 2.0)
    c, d = oracle.bin_coord(-3.0, lo, hi, B)
    assert c == pytest.approx(2.0) and d == 0.0
    c, d = oracle.bin_coord(7.0, lo, hi, B)
    assert c == pytest.approx(B - 3.0) and d == 0.0


def _brute_force_psi(F, J, B, f_range, j_range):
    """Naive method: dense Psi_F, Psi_J in R^{B x N}, P = Psi_F Psi_J^T / N."""
    def coords(v, lo, hi):
        v = np.clip(np.asarray(v, np.float64).reshape(-1), lo, hi)
        return 2.0 + (v - lo) / (hi - lo) * (B - 5)
    cf = coords(F, *f_range)
    cj = coords(J, *j_range)
    bins = np.arange(B, dtype=np.float64)[:, None]
    PsiF = _beta_scipy(bins - cf[None, :])
    PsiJ = _beta_scipy(bins - cj[None, :])
    N = cf.size
    P = PsiF @ PsiJ.T / N
    PF = PsiF.sum(1) / N
    PJ = PsiJ.sum(1) / N
    nz = P > 0
    mi = float(np.sum(P[nz] * (np.log(P[nz]) - np.log(np.outer(PF, PJ)[nz]))))
    return mi, P, PF, PJ


@pytest.mark.parametrize("B", [8, 32, 64])
def test_histogram_equals_dense_psi_product(B):
    rng = np.random.default_rng(B)
    N = 3000
    F = rng.uniform(0, 1, N).astype(np.float32)
    J = 0.6 * F + 0.4 * rng.uniform(0, 1, N)
    fr = (float(F.min()), float(F.max()))
    jr = (0.1, 0.9)  # some J values clamp
    r = oracle.mi(F, J, B, fr, jr, want_grad=False)
    mi_b, P, PF, PJ = _brute_force_psi(F, J, B, fr, jr)
    assert np.max(np.abs(r["P"] - P)) < 1e-14
    assert np.max(np.abs(r["PF"] - PF)) < 1e-14
    assert np.max(np.abs(r["PJ"] - PJ)) < 1e-14
    assert abs(r["mi"] - mi_b) < 1e-12
    # separately accumulated marginals equal the joint's row / column sums
    assert np.max(np.abs(r["P"].sum(1) - r["PF"])) < 1e-14
    assert np.max(np.abs(r["P"].sum(0) - r["PJ"])) < 1e-14
    assert abs(r["P"].sum() - 1.0) < 1e-12


@pytest.mark.parametrize("K", [2, 3, 5])
def test_mi_of_well_separated_values_is_ln_K(K):
    # K voxels whose bin coordinates are >= 4 apart: the joint splits into K
    # disjoint blocks w_a w_b / K with marginals w_a / K, so MI = ln K exactly.
    B = 8 + 4 * K
    lo, hi = 0.0, float(B - 5)
    vals = np.array([4.0 * i for i in range(K)], np.float32)  # bins 2, 6, 10, ...
    r = oracle.mi(vals, vals.astype(np.float64), B, (lo, hi), (lo, hi), want_grad=False)
    assert abs(r["mi"] - math.log(K)) < 1e-14


def test_box_kernel_mi_of_image_with_itself_is_its_entropy():
    rng = np.random.default_rng(4)
    F = rng.uniform(0, 1, 5000).astype(np.float32)
    r = oracle.mi(F, F.astype(np.float64), 32, (0.0, 1.0), (0.0, 1.0), degree=0, want_grad=False)
    PF = r["PF"]
    H = -float(np.sum(PF[PF > 0] * np.log(PF[PF > 0])))
    assert abs(r["mi"] - H) < 1e-12
    assert np.count_nonzero(r["P"] - np.diag(np.diag(r["P"]))) == 0


def test_mi_invariances():
    rng = np.random.default_rng(7)
    F = rng.uniform(0, 1, 4000).astype(np.float32)
    G = (np.sin(3 * F) + 0.3 * rng.normal(size=F.size)).astype(np.float32)
    rF = (float(F.min()), float(F.max()))
    rG = (float(G.min()), float(G.max()))
    m_fg = oracle.mi(F, G.astype(np.float64), 32, rF, rG, want_grad=False)["mi"]
    m_gf = oracle.mi(G, F.astype(np.float64), 32, rG, rF, want_grad=False)["mi"]
    m_ff = oracle.mi(F, F.astype(np.float64), 32, rF, rF, want_grad=False)["mi"]
    assert m_fg >= 0 and abs(m_fg - m_gf) < 1e-12
    assert m_ff >= m_fg
    # affine intensity change with the image's own range: identical bin coordinates
    J = 2.5 * F.astype(np.float64) + 0.75
    m_aff = oracle.mi(F, J, 32, rF, (float(J.min()), float(J.max())), want_grad=False)["mi"]
    assert abs(m_aff - m_ff) < 1e-10


def test_slab_histograms_merge_to_global():
    rng = np.random.default_rng(8)
    F = rng.uniform(0, 1, 6000).astype(np.float32)
    J = (F + 0.2 * rng.normal(size=F.size))
    B = 32
    fr, jr = (0.0, 1.0), (float(J.min()), float(J.max()))
    full = oracle.mi(F, J, B, fr, jr, want_grad=False)
    # per-shard normalised histograms P^(h), merged with weights N_h / N
    cuts = [0, 1000, 1700, 4200, 6000]
    P = np.zeros((B, B))
    PF = np.zeros(B)
    PJ = np.zeros(B)
    for a, b in zip(cuts[:-1], cuts[1:]):
        r = oracle.mi(F[a:b], J[a:b], B, fr, jr, want_grad=False)
        w = (b - a) / F.size
        P += w * r["P"]
        PF += w * r["PF"]
        PJ += w * r["PJ"]
    assert np.max(np.abs(P - full["P"])) < 1e-15
    assert np.max(np.abs(PF - full["PF"])) < 1e-15
    nz = P > 0
    mi = float(np.sum(P[nz] * (np.log(P[nz]) - np.log(np.outer(PF, PJ)[nz]))))
    assert abs(mi - full["mi"]) < 1e-12


def test_gradient_matches_finite_differences_of_dense_psi_mi():
    rng = np.random.default_rng(9)
    N, B = 400, 16
    F = rng.uniform(0, 1, N).astype(np.float32)
    J = 0.5 * F + 0.5 * rng.uniform(0, 1, N)
    fr, jr = (0.0, 1.0), (0.05, 0.95)
    r = oracle.mi(F, J, B, fr, jr)
    dJ = r["dJ"]
    h = 1e-6
    for k in rng.choice(N, 25, replace=False):
        Jp = J.copy()
        Jm = J.copy()
        Jp[k] += h
        Jm[k] -= h
        fd = -(_brute_force_psi(F, Jp, B, fr, jr)[0] - _brute_force_psi(F, Jm, B, fr, jr)[0]) / (2 * h)
        assert abs(fd - dJ[k]) < 1e-6 * max(abs(fd), 1e-3), (k, fd, dJ[k])


def test_dropped_terms_cancel():
    # The +1 term and the marginal term of the full chain rule sum to zero by
    # partition of unity, so d(-MI)/dJ_k = (c'/N) sum T(a,b) beta(a-cF) beta'(b-cJ)
    # with T = ln P - ln P_F - ln P_J.
    rng = np.random.default_rng(10)
    N, B = 2000, 32
    F = rng.uniform(0, 1, N).astype(np.float32)
    J = np.cos(2 * F) + 0.1 * rng.normal(size=N)
    fr, jr = (0.0, 1.0), (float(J.min()), float(J.max()))
    r = oracle.mi(F, J, B, fr, jr)
    P, PF, PJ = r["P"], r["PF"], r["PJ"]
    with np.errstate(divide="ignore", invalid="ignore"):
        T = np.where(P > 0, np.log(P) - np.log(PF)[:, None] - np.log(PJ)[None, :], 0.0)
    short = np.empty(N)
    for k in range(N):
        cf, _ = oracle.bin_coord(F[k], *fr, B)
        cj, dc = oracle.bin_coord(J[k], *jr, B)
        a0, b0 = int(math.floor(cf)) - 1, int(math.floor(cj)) - 1
        s = 0.0
        for ia in range(4):
            for ib in range(4):
                s += T[a0 + ia, b0 + ib] * oracle.bspline(a0 + ia - cf) * oracle.bspline_deriv(b0 + ib - cj)
        short[k] = dc / N * s
    assert np.max(np.abs(short - r["dJ"])) < 1e-12 * max(1.0, np.max(np.abs(short)))
