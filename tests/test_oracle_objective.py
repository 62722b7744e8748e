"""End-to-end pins for the oracle's objective L = w_mi(-MI) + w_lncc(-LNCC)
composed with the sampler, and its gradient with respect to u, A and t.

Paper: "A Scalable Distributed Framework for Multimodal GigaVoxel Image
Registration": Background (L = C(F, M o phi) + R(phi), phi = Ax + t + u(x)),
Key designs items 1, 2 and 5.  The worked examples in
tests/golden/worked_examples.txt are derived by hand from the definitions.
"""
import os

import numpy as np
import pytest

import oracle
from oracle import ObjectiveParams, Transform

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.txt")


def _golden():
    rows = {}
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        name, inp, exp = [s.strip() for s in line.split("|")]
        kv = lambda s: dict(tok.split("=") for tok in s.split())
        rows[name] = (kv(inp), kv(exp))
    return rows


def _nums(s):
    return np.array([float(v) for v in s.split(",")])


def test_golden_trilinear_examples():
    M = np.zeros((2, 2, 2), np.float32)
    for z in range(2):
        for y in range(2):
            for x in range(2):
                M[z, y, x] = x + 2 * y + 4 * z
    rows = _golden()
    for name in ("trilinear_linear2", "trilinear_pad"):
        inp, exp = rows[name]
        p = _nums(inp["p"])
        # a 2x2x2 fixed grid whose first voxel maps to p via t (A = 0)
        T = Transform(np.zeros((3, 3)), p, np.eye(3), -np.ones(3), np.ones(3))
        J, G = oracle.grid_sample(M, (2, 2, 2), None, T, want_grad=True)
        assert abs(J[0, 0, 0] - float(exp["J"])) < 1e-14
        assert np.allclose(G[0, 0, 0], _nums(exp["dJdp"]), atol=1e-14)


def test_golden_mi_examples():
    rows = _golden()
    for name, degree in (("mi_two_voxels", 3), ("mi_box_entropy", 0)):
        inp, exp = rows[name]
        rng_ = tuple(_nums(inp["range"]))
        F = _nums(inp["F"]).astype(np.float32)
        J = _nums(inp["J"])
        r = oracle.mi(F, J, int(inp["B"]), rng_, rng_, degree=degree, want_grad=False)
        assert abs(r["mi"] - float(exp["MI"])) < 1e-14


def _small_problem(seed=0, shape=(6, 7, 8), mshape=(7, 8, 9)):
    rng = np.random.default_rng(seed)
    F = rng.uniform(0, 1, shape).astype(np.float32)
    M = rng.uniform(0, 1, mshape).astype(np.float32)
    u = (rng.normal(size=shape + (3,)) * 0.05).astype(np.float32)
    T = Transform(np.eye(3) + rng.uniform(-0.05, 0.05, (3, 3)), rng.uniform(-0.05, 0.05, 3),
                  np.eye(3) + rng.uniform(-0.05, 0.05, (3, 3)), np.array([-0.95, -1.0, -0.9]),
                  np.array([1.0, 0.9, 0.95]))
    p = ObjectiveParams(w_mi=0.7, w_lncc=1.3, bins=16, f_range=(0.0, 1.0), m_range=(0.0, 1.0),
                        window=3, eps=1e-5)
    return F, M, u, T, p


def test_objective_gradient_matches_finite_differences():
    F, M, u, T, p = _small_problem()
    r = oracle.objective(F, M, u, T, p)

    def L(Tx, uu):
        return float(oracle.objective(F, M, uu, Tx, p, want_du=False)["loss"][0])

    h = 1e-6
    for k in range(9):
        Tp = Transform(T.A.copy(), T.t, T.S, T.xmin, T.xmax)
        Tm = Transform(T.A.copy(), T.t, T.S, T.xmin, T.xmax)
        Tp.A.flat[k] += h
        Tm.A.flat[k] -= h
        fd = (L(Tp, u) - L(Tm, u)) / (2 * h)
        assert abs(fd - r["dA"].flat[k]) < 2e-5 * max(1.0, abs(fd)), (k, fd, r["dA"].flat[k])
    for k in range(3):
        Tp = Transform(T.A, T.t.copy(), T.S, T.xmin, T.xmax)
        Tm = Transform(T.A, T.t.copy(), T.S, T.xmin, T.xmax)
        Tp.t[k] += h
        Tm.t[k] -= h
        fd = (L(Tp, u) - L(Tm, u)) / (2 * h)
        assert abs(fd - r["dt"][k]) < 2e-5 * max(1.0, abs(fd)), (k, fd, r["dt"][k])
    rng = np.random.default_rng(1)
    hu = 2e-4
    for _ in range(6):
        idx = tuple(int(rng.integers(0, s)) for s in F.shape) + (int(rng.integers(0, 3)),)
        up = u.copy()
        um = u.copy()
        up[idx] = np.float32(u[idx] + hu)
        um[idx] = np.float32(u[idx] - hu)
        step = float(up[idx]) - float(um[idx])
        fd = (L(T, up) - L(T, um)) / step
        assert abs(fd - r["du"][idx]) < 1e-4 * max(1e-3, abs(fd)), (idx, fd, r["du"][idx])


def test_slab_streamed_mi_objective_equals_whole_array():
    F, M, u, T, p = _small_problem(seed=3, shape=(9, 7, 8))
    p.w_lncc = 0.0
    whole = oracle.objective(F, M, u, T, p)
    idx = np.array([0, 5, 77, 200, F.size - 1])
    slabs = oracle.objective_mi_slabs(F, M, u, T, p, slab=2, du_index=idx)
    assert np.allclose(slabs["loss"], whole["loss"], rtol=1e-13, atol=1e-15)
    assert np.allclose(slabs["dA"], whole["dA"], rtol=1e-11, atol=1e-14)
    assert np.allclose(slabs["dt"], whole["dt"], rtol=1e-11, atol=1e-14)
    assert np.allclose(slabs["du_samples"], whole["du"].reshape(-1, 3)[idx], rtol=1e-12, atol=1e-16)
