"""Double-precision CPU oracle for the FFDP registration objective.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The product path (the CUDA
library and its binding) never imports this package.

The arithmetic lives in ``ffdp_oracle.c`` (plain C, double precision, one
definition per quantity; see its header for the page sections it follows and
the readings taken where the page is silent).  This module only compiles that
file with gcc, loads it with ctypes and composes its functions into the
objective:

    J      = M(A x + t + S u(x))                  (sampler, design 1)
    L      = w_mi * (-MI(F, J)) + w_lncc * (-LNCC(F, J))   (design 2)
    dL/dJ  = w_mi * d(-MI)/dJ + w_lncc * d(-LNCC)/dJ
    du, dA, dt = sampler backward of dL/dJ         (design 1)

and, for the next rows of the path, the sampler on a C-channel volume (warp
composition, the gradient dV of the sampled volume) and the MSE objective.

Inputs are numpy arrays holding exactly the values the GPU path receives:
fp16 volumes are widened to float32 (exact), transforms are the float32 values
widened to float64 (exact).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ffdp_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libffdp_oracle.so")
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_fp = ctypes.POINTER(ctypes.c_float)
_ip = ctypes.POINTER(ctypes.c_int64)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP if available).  Returns the .so path."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + ".tmp%d" % os.getpid()
    base = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        L.oracle_max_threads.restype = ctypes.c_int
        L.oracle_set_threads.argtypes = [ctypes.c_int]
        L.oracle_grid_sample.argtypes = [_fp, _ip, _ip, _fp, _dp, ctypes.c_int64, ctypes.c_int64, _dp, _dp]
        L.oracle_grid_sample_bwd.argtypes = [_fp, _ip, _ip, _fp, _dp, ctypes.c_int64, ctypes.c_int64,
                                             _dp, _dp, _dp, _dp]
        L.oracle_bspline.argtypes = [ctypes.c_int, ctypes.c_double]
        L.oracle_bspline.restype = ctypes.c_double
        L.oracle_bspline_deriv.argtypes = [ctypes.c_int, ctypes.c_double]
        L.oracle_bspline_deriv.restype = ctypes.c_double
        L.oracle_bin_coord.argtypes = [ctypes.c_double, ctypes.c_double, ctypes.c_double, ctypes.c_int, _dp]
        L.oracle_bin_coord.restype = ctypes.c_double
        L.oracle_mi_accumulate.argtypes = [_fp, _dp, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_double, ctypes.c_double, ctypes.c_double,
                                           ctypes.c_double, _dp, _dp, _dp]
        L.oracle_mi_finish.argtypes = [_dp, _dp, _dp, ctypes.c_int, ctypes.c_double, _dp, _dp, _dp]
        L.oracle_mi_finish.restype = ctypes.c_double
        L.oracle_mi_grad.argtypes = [_fp, _dp, ctypes.c_int64, ctypes.c_int, ctypes.c_double,
                                     ctypes.c_double, ctypes.c_double, ctypes.c_double, _dp, _dp, _dp,
                                     ctypes.c_double, _dp]
        L.oracle_mi.argtypes = [_fp, _dp, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                ctypes.c_double, ctypes.c_double, ctypes.c_double, _dp, _dp, _dp, _dp]
        L.oracle_mi.restype = ctypes.c_double
        L.oracle_lncc.argtypes = [_fp, _dp, _ip, ctypes.c_int, ctypes.c_double, _dp, _dp]
        L.oracle_lncc.restype = ctypes.c_double
        L.oracle_sample_channels.argtypes = [_fp, ctypes.c_int, _ip, _ip, _fp, _dp, ctypes.c_int,
                                             ctypes.c_int64, ctypes.c_int64, _dp]
        L.oracle_sample_channels_bwd.argtypes = [_fp, ctypes.c_int, _ip, _ip, _fp, _dp, ctypes.c_int,
                                                 ctypes.c_int64, ctypes.c_int64, _dp, _dp, _dp, _dp, _dp]
        L.oracle_mse.argtypes = [_fp, _dp, ctypes.c_int64, _dp]
        L.oracle_mse.restype = ctypes.c_double
        L.oracle_sobolev.argtypes = [_fp, _ip, ctypes.c_double, _dp]
        L.oracle_sobolev.restype = ctypes.c_double
        L.oracle_adam.argtypes = [_dp, _dp, _dp, _dp, ctypes.c_int64, ctypes.c_double, ctypes.c_double,
                                  ctypes.c_double, ctypes.c_double, ctypes.c_int]
        _lib = L
    return _lib


def set_threads(n: int) -> None:
    lib().oracle_set_threads(int(n))


def max_threads() -> int:
    return int(lib().oracle_max_threads())


# ----------------------------------------------------------------- marshalling
def _f32(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype == np.float16:
        a = a.astype(np.float32)  # exact widening
    return np.ascontiguousarray(a, dtype=np.float32)


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _pf(a):
    return None if a is None else a.ctypes.data_as(_fp)


def _pd(a):
    return None if a is None else a.ctypes.data_as(_dp)


def _dims(shape) -> np.ndarray:
    return np.asarray(list(shape), dtype=np.int64)


@dataclass
class Transform:
    """A (3x3), t (3), S (3x3), x_min (3), x_max (3); rows/cols in (x, y, z) order."""
    A: np.ndarray
    t: np.ndarray
    S: np.ndarray
    xmin: np.ndarray
    xmax: np.ndarray

    def packed(self) -> np.ndarray:
        return _f64(np.concatenate([np.asarray(self.A, np.float64).reshape(9),
                                    np.asarray(self.t, np.float64).reshape(3),
                                    np.asarray(self.S, np.float64).reshape(9),
                                    np.asarray(self.xmin, np.float64).reshape(3),
                                    np.asarray(self.xmax, np.float64).reshape(3)]))

    @staticmethod
    def identity() -> "Transform":
        return Transform(np.eye(3), np.zeros(3), np.eye(3), -np.ones(3), np.ones(3))


# --------------------------------------------------------------------- sampler
def grid_sample(M, fixed_shape, u, T: Transform, z0: int = 0, z1: int | None = None,
                want_grad: bool = False):
    """J[z0:z1] (and dJ/dp, [..., 3]) for the fixed grid ``fixed_shape`` (D, H, W)."""
    M = _f32(M)
    D, H, W = fixed_shape
    z1 = D if z1 is None else z1
    u32 = None if u is None else _f32(u)
    J = np.empty((z1 - z0, H, W), np.float64)
    G = np.empty((z1 - z0, H, W, 3), np.float64) if want_grad else None
    lib().oracle_grid_sample(_pf(M), _dims(M.shape).ctypes.data_as(_ip),
                             _dims(fixed_shape).ctypes.data_as(_ip), _pf(u32),
                             _pd(T.packed()), z0, z1, _pd(J), _pd(G))
    return (J, G) if want_grad else J


def grid_sample_bwd(M, fixed_shape, u, T: Transform, gJ, z0: int = 0, z1: int | None = None,
                    want_du: bool = True, dA=None, dt=None):
    """Sampler backward for planes [z0, z1): returns (du, dA, dt).

    dA / dt are accumulated into the given arrays (fresh zeros if None)."""
    M = _f32(M)
    D, H, W = fixed_shape
    z1 = D if z1 is None else z1
    u32 = None if u is None else _f32(u)
    g = _f64(gJ)
    du = np.empty((z1 - z0, H, W, 3), np.float64) if want_du else None
    dA = np.zeros(9, np.float64) if dA is None else dA
    dt = np.zeros(3, np.float64) if dt is None else dt
    lib().oracle_grid_sample_bwd(_pf(M), _dims(M.shape).ctypes.data_as(_ip),
                                 _dims(fixed_shape).ctypes.data_as(_ip), _pf(u32),
                                 _pd(T.packed()), z0, z1, _pd(g), _pd(du), _pd(dA), _pd(dt))
    return du, dA, dt


# ------------------------------------------------- C-channel sampler / compose
def sample_channels(V, fixed_shape, u, T: Transform, compose: bool = False, z0: int = 0,
                    z1: int | None = None):
    """out[z0:z1] = V(A x + t + S u(x)) (+ S u(x) when compose) for a channel-last
    volume V of shape (Dv, Hv, Wv, C); returns (z1-z0, H, W, C) float64."""
    V = _f32(V)
    C = V.shape[3]
    D, H, W = fixed_shape
    z1 = D if z1 is None else z1
    u32 = None if u is None else _f32(u)
    out = np.empty((z1 - z0, H, W, C), np.float64)
    lib().oracle_sample_channels(_pf(V), C, _dims(V.shape[:3]).ctypes.data_as(_ip),
                                 _dims(fixed_shape).ctypes.data_as(_ip), _pf(u32), _pd(T.packed()),
                                 int(bool(compose)), z0, z1, _pd(out))
    return out


def sample_channels_bwd(V, fixed_shape, u, T: Transform, gout, compose: bool = False,
                        want_du: bool = True, want_dV: bool = True, z0: int = 0, z1: int | None = None,
                        dA=None, dt=None):
    """Backward of sample_channels for planes [z0, z1) (gout indexed from z0):
    (du, dA, dt, dV).  dA / dt are accumulated into the given arrays (fresh
    zeros if None); dV covers the whole volume V."""
    V = _f32(V)
    C = V.shape[3]
    D, H, W = fixed_shape
    z1 = D if z1 is None else z1
    u32 = None if u is None else _f32(u)
    g = _f64(gout)
    du = np.empty((z1 - z0, H, W, 3), np.float64) if want_du else None
    dA = np.zeros(9, np.float64) if dA is None else dA
    dt = np.zeros(3, np.float64) if dt is None else dt
    dV = np.zeros(V.shape, np.float64) if want_dV else None
    lib().oracle_sample_channels_bwd(_pf(V), C, _dims(V.shape[:3]).ctypes.data_as(_ip),
                                     _dims(fixed_shape).ctypes.data_as(_ip), _pf(u32), _pd(T.packed()),
                                     int(bool(compose)), z0, z1, _pd(g), _pd(du), _pd(dA), _pd(dt), _pd(dV))
    return du, dA.reshape(3, 3), dt, dV


# ------------------------------------------------------------------------ MSE
def mse(F, J, want_grad: bool = True):
    """Returns dict(mse, dJ) for same-size F and J."""
    F32 = _f32(F).reshape(-1)
    J64 = _f64(J).reshape(-1)
    dJ = np.empty(F32.size, np.float64) if want_grad else None
    v = lib().oracle_mse(_pf(F32), _pd(J64), F32.size, _pd(dJ))
    return dict(mse=float(v), dJ=None if dJ is None else dJ.reshape(np.shape(J)))


def objective_mse(F, M, u, T: Transform, w_mse: float = 1.0, want_du: bool = True):
    """MSE objective L = w_mse * MSE(F, M o phi) and its sampler backward.

    Returns dict(loss=[w_mse * MSE, MSE], J, gJ, du, dA, dt)."""
    F32 = _f32(F)
    shape = F32.shape
    J = grid_sample(M, shape, u, T)
    r = mse(F32, J)
    gJ = w_mse * r["dJ"]
    du, dA, dt = grid_sample_bwd(M, shape, u, T, gJ, want_du=want_du)
    return dict(loss=np.array([w_mse * r["mse"], r["mse"]]), J=J, gJ=gJ, du=du, dA=dA.reshape(3, 3), dt=dt)


# ------------------------------------------------- Sobolev regulariser, Adam
def sobolev(u, lam: float, want_grad: bool = True):
    """Returns dict(R, dR) for a displacement field u of shape (D, H, W, 3)."""
    u32 = _f32(u)
    dR = np.empty(u32.shape, np.float64) if want_grad else None
    v = lib().oracle_sobolev(_pf(u32), _dims(u32.shape[:3]).ctypes.data_as(_ip), float(lam), _pd(dR))
    return dict(R=float(v), dR=dR)


def adam(x, g, m1, m2, lr, b1, b2, eps, t):
    """One Adam step: returns updated float64 copies (x, m1, m2)."""
    x = _f64(x).copy()
    m1 = _f64(m1).copy()
    m2 = _f64(m2).copy()
    gg = _f64(g)
    lib().oracle_adam(_pd(x), _pd(gg), _pd(m1), _pd(m2), x.size, float(lr), float(b1), float(b2), float(eps),
                      int(t))
    return x, m1, m2


def sobolev_adam_step(u, g, m1, m2, lam, lr, b1, b2, eps, t):
    """One regularised iteration on u: G = g + dR/du, Adam step on u.

    Returns dict(R, u, m1, m2, G)."""
    r = sobolev(u, lam)
    G = _f64(g) + r["dR"]
    x, n1, n2 = adam(_f32(u).astype(np.float64), G, m1, m2, lr, b1, b2, eps, t)
    return dict(R=r["R"], u=x, m1=n1, m2=n2, G=G)


# ------------------------------------------------------------------------- MI
def bspline(s: float, degree: int = 3) -> float:
    return float(lib().oracle_bspline(degree, float(s)))


def bspline_deriv(s: float, degree: int = 3) -> float:
    return float(lib().oracle_bspline_deriv(degree, float(s)))


def bin_coord(v: float, lo: float, hi: float, bins: int):
    d = ctypes.c_double(0.0)
    c = lib().oracle_bin_coord(float(v), float(lo), float(hi), int(bins), ctypes.byref(d))
    return float(c), float(d.value)


def mi(F, J, bins: int, f_range, j_range, degree: int = 3, want_grad: bool = True):
    """Returns dict(mi, P, PF, PJ, dJ) for images F (any shape) and J (same size)."""
    F32 = _f32(F).reshape(-1)
    J64 = _f64(J).reshape(-1)
    n = F32.size
    P = np.zeros(bins * bins, np.float64)
    PF = np.zeros(bins, np.float64)
    PJ = np.zeros(bins, np.float64)
    dJ = np.empty(n, np.float64) if want_grad else None
    v = lib().oracle_mi(_pf(F32), _pd(J64), n, bins, degree, float(f_range[0]), float(f_range[1]),
                        float(j_range[0]), float(j_range[1]), _pd(P), _pd(PF), _pd(PJ), _pd(dJ))
    return dict(mi=float(v), P=P.reshape(bins, bins), PF=PF, PJ=PJ,
                dJ=None if dJ is None else dJ.reshape(np.shape(J)))


def mi_accumulate(F, J, bins, f_range, j_range, H, HF, HJ, degree: int = 3):
    F32 = _f32(F).reshape(-1)
    J64 = _f64(J).reshape(-1)
    lib().oracle_mi_accumulate(_pf(F32), _pd(J64), F32.size, bins, degree, float(f_range[0]),
                               float(f_range[1]), float(j_range[0]), float(j_range[1]),
                               _pd(H), _pd(HF), _pd(HJ))


def mi_finish(H, HF, HJ, bins, N):
    P = np.empty(bins * bins, np.float64)
    PF = np.empty(bins, np.float64)
    PJ = np.empty(bins, np.float64)
    v = lib().oracle_mi_finish(_pd(_f64(H)), _pd(_f64(HF)), _pd(_f64(HJ)), bins, float(N),
                               _pd(P), _pd(PF), _pd(PJ))
    return float(v), P, PF, PJ


def mi_grad(F, J, bins, f_range, j_range, P, PF, PJ, N):
    F32 = _f32(F).reshape(-1)
    J64 = _f64(J).reshape(-1)
    dJ = np.empty(F32.size, np.float64)
    lib().oracle_mi_grad(_pf(F32), _pd(J64), F32.size, bins, float(f_range[0]), float(f_range[1]),
                         float(j_range[0]), float(j_range[1]), _pd(_f64(P)), _pd(_f64(PF)),
                         _pd(_f64(PJ)), float(N), _pd(dJ))
    return dJ


# ----------------------------------------------------------------------- LNCC
def lncc(F, J, window: int, eps: float = 1e-5, want_cc: bool = False, want_grad: bool = True):
    """Returns dict(lncc, cc, dJ) for same-shape 3-D volumes F and J."""
    F32 = _f32(F)
    J64 = _f64(J)
    cc = np.empty(F32.shape, np.float64) if want_cc else None
    dJ = np.empty(F32.shape, np.float64) if want_grad else None
    v = lib().oracle_lncc(_pf(F32), _pd(J64), _dims(F32.shape).ctypes.data_as(_ip), int(window),
                          float(eps), _pd(cc), _pd(dJ))
    return dict(lncc=float(v), cc=cc, dJ=dJ)


# ------------------------------------------------------------------ objective
@dataclass
class ObjectiveParams:
    w_mi: float = 1.0
    w_lncc: float = 1.0
    bins: int = 32
    f_range: tuple = (0.0, 1.0)
    m_range: tuple = (0.0, 1.0)
    window: int = 5
    eps: float = 1e-5


def objective(F, M, u, T: Transform, p: ObjectiveParams, want_du: bool = True):
    """Full objective on whole arrays.

    Returns dict(loss=[total, -MI, -LNCC], J, gJ, du, dA, dt, mi, lncc).
    A term whose weight is 0 is not evaluated and reports 0."""
    F32 = _f32(F)
    shape = F32.shape
    N = F32.size
    J = grid_sample(M, shape, u, T)
    gJ = np.zeros(shape, np.float64)
    mi_loss = 0.0
    lncc_loss = 0.0
    mi_v = None
    lncc_v = None
    if p.w_mi != 0.0:
        r = mi(F32, J, p.bins, p.f_range, p.m_range)
        mi_v = r["mi"]
        mi_loss = -mi_v
        gJ += p.w_mi * r["dJ"].reshape(shape)
    if p.w_lncc != 0.0:
        r = lncc(F32, J, p.window, p.eps)
        lncc_v = r["lncc"]
        lncc_loss = -lncc_v
        gJ += p.w_lncc * r["dJ"]
    du, dA, dt = grid_sample_bwd(M, shape, u, T, gJ, want_du=want_du)
    total = p.w_mi * mi_loss + p.w_lncc * lncc_loss
    return dict(loss=np.array([total, mi_loss, lncc_loss]), J=J, gJ=gJ, du=du,
                dA=dA.reshape(3, 3), dt=dt, mi=mi_v, lncc=lncc_v, N=N)


def objective_mi_slabs(F, M, u, T: Transform, p: ObjectiveParams, slab: int = 16,
                       du_index=None, on_slab=None):
    """MI-only objective evaluated slab by slab, so no N-sized double array is held.

    The histogram is accumulated over z-slabs and merged with the slab weights
    N_h/N implied by plain accumulation (design 5's partial-aggregation
    identity).  Returns dict(loss, dA, dt, du_samples) where du_samples holds
    du at the flat voxel indices ``du_index`` (sorted or not).  on_slab, if
    given, is called as on_slab(z0, z1, du, J) with each slab's du
    [z1-z0, H, W, 3] and J [z1-z0, H, W] (float64) as they are computed."""
    F32 = _f32(F)
    shape = F32.shape
    D, H, W = shape
    N = F32.size
    B = p.bins
    Hh = np.zeros(B * B, np.float64)
    HF = np.zeros(B, np.float64)
    HJ = np.zeros(B, np.float64)
    u32 = None if u is None else _f32(u)
    M32 = _f32(M)
    for z0 in range(0, D, slab):
        z1 = min(D, z0 + slab)
        J = grid_sample(M32, shape, u32, T, z0, z1)
        mi_accumulate(F32[z0:z1], J, B, p.f_range, p.m_range, Hh, HF, HJ)
    mi_v, P, PF, PJ = mi_finish(Hh, HF, HJ, B, N)
    dA = np.zeros(9, np.float64)
    dt = np.zeros(3, np.float64)
    idx = None if du_index is None else np.asarray(du_index, np.int64)
    du_s = None if idx is None else np.zeros((idx.size, 3), np.float64)
    J_s = None if idx is None else np.zeros(idx.size, np.float64)
    plane = H * W
    for z0 in range(0, D, slab):
        z1 = min(D, z0 + slab)
        J = grid_sample(M32, shape, u32, T, z0, z1)
        gJ = p.w_mi * mi_grad(F32[z0:z1], J, B, p.f_range, p.m_range, P, PF, PJ, N)
        du, dA, dt = grid_sample_bwd(M32, shape, u32, T, gJ, z0, z1,
                                     want_du=idx is not None or on_slab is not None, dA=dA, dt=dt)
        if on_slab is not None:
            on_slab(z0, z1, du, J)
        if idx is not None:
            sel = (idx >= z0 * plane) & (idx < z1 * plane)
            du_s[sel] = du.reshape(-1, 3)[idx[sel] - z0 * plane]
            J_s[sel] = J.reshape(-1)[idx[sel] - z0 * plane]
    loss = np.array([p.w_mi * -mi_v, -mi_v, 0.0])
    return dict(loss=loss, dA=dA.reshape(3, 3), dt=dt, du_samples=du_s, J_samples=J_s, mi=mi_v, P=P,
                PF=PF, PJ=PJ)
