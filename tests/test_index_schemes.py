"""Host checks of the index schemes the CUDA kernels rely on, restated in
Python from their descriptions (no code shared with the kernels):

* the image-gradient scatter sends the 2C adjacent floats of a cell row's two
  x taps as zero-padded 16-byte chunks aligned to the array, with scalar
  fallbacks where a chunk would leave the array -- every float lands once,
  nothing outside [0, nV) is touched;
* the vector form of the regularised step treats [N][3] arrays as flat float4
  vectors: element f is channel f mod 3 of voxel f / 3, its x neighbours are
  elements f -/+ 3 and its y / z neighbours the same lane 3W/4 and 3HW/4
  vectors away -- the resulting energy and gradient equal the oracle's.
"""
import numpy as np
import pytest

import oracle


def _scatter_pair(out, f0, vals, chunk=4):
    nV = out.size
    N = len(vals)
    a = f0 & ~(chunk - 1)
    off = f0 - a
    nch = (off + N + chunk - 1) // chunk
    for k in range(nch):
        base = a + chunk * k
        v = [vals[chunk * k + j - off] if 0 <= chunk * k + j - off < N else 0.0 for j in range(chunk)]
        if base >= 0 and base + chunk <= nV:
            out[base:base + chunk] += v
        else:
            for j in range(chunk):
                src = chunk * k + j - off
                if 0 <= src < N and 0 <= base + j < nV:
                    out[base + j] += v[j]


@pytest.mark.parametrize("C", [1, 2, 3, 4])
def test_scatter_chunks_place_every_float_once(C):
    for nV in (4 * C, 4 * C + 1, 4 * C + 3, 37 * C):
        for f0 in range(-2 * C, nV):
            vals = np.arange(1, 2 * C + 1, dtype=float)
            out = np.zeros(nV)
            _scatter_pair(out, f0, vals)
            ref = np.zeros(nV)
            for i in range(2 * C):
                if 0 <= f0 + i < nV:
                    ref[f0 + i] += vals[i]
            assert np.array_equal(out, ref), (C, nV, f0)


def _step_vector_form(u, lam):
    D, H, W = u.shape[:3]
    N = D * H * W
    V = u.reshape(-1).astype(np.float64).reshape(-1, 4)
    NQ = V.shape[0]
    QY, QZ = 3 * W // 4, 3 * W * H // 4
    dR = np.zeros(3 * N)
    s = 0.0
    for q in range(NQ):
        f0 = 4 * q
        v0, c0 = f0 // 3, f0 % 3
        xyz = lambda v: (v % W, (v // W) % H, v // (W * H))
        p0, p1 = xyz(v0), xyz(min(v0 + 1, N - 1))
        flat = lambda e: V.reshape(-1)[e] if 0 <= e < 3 * N else 0.0
        for j in range(4):
            x, y, z = p1 if c0 + j >= 3 else p0
            f = f0 + j
            d = 0.0
            for cond, e, fwd in ((x > 0, f - 3, False), (x + 1 < W, f + 3, True), (y > 0, f - 4 * QY, False),
                                 (y + 1 < H, f + 4 * QY, True), (z > 0, f - 4 * QZ, False), (z + 1 < D, f + 4 * QZ, True)):
                if cond:
                    diff = flat(e) - flat(f)
                    d += diff
                    if fwd:
                        s += diff * diff
            dR[f] = -2.0 * lam / N * d
    return lam * s / N, dR.reshape(u.shape)


@pytest.mark.parametrize("shape", [(2, 2, 4), (3, 5, 8), (4, 3, 12), (5, 7, 4)])
def test_vector_form_of_the_step_stencil(shape):
    u = np.random.default_rng(sum(shape)).normal(size=shape + (3,)).astype(np.float32)
    R, dR = _step_vector_form(u, 0.7)
    r = oracle.sobolev(u, 0.7)
    assert abs(R - r["R"]) <= 1e-12 * abs(r["R"])
    assert np.max(np.abs(dR - r["dR"])) <= 1e-12 * np.max(np.abs(r["dR"]))
