"""Shared helpers for the GPU parity tests: marshal one synthetic pair to both
the CUDA library (through its C ABI binding) and the CPU oracle."""
import numpy as np

import oracle

TOL_J = 1e-5        # |delta| on sampled intensities
TOL_LOSS = 1e-4     # relative, loss values
TOL_GRAD = 1e-3     # relative L2, gradients


def rel_l2(a, b):
    a = np.asarray(a, np.float64).ravel()
    b = np.asarray(b, np.float64).ravel()
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (nb if nb > 0 else 1.0))


def rel_err(a, b, floor=1e-12):
    return float(abs(float(a) - float(b)) / max(abs(float(b)), floor))


def oracle_T(A, t, S=None, xmin=None, xmax=None):
    S = np.eye(3, dtype=np.float32) if S is None else S
    xmin = -np.ones(3, np.float32) if xmin is None else xmin
    xmax = np.ones(3, np.float32) if xmax is None else xmax
    f64 = lambda v: np.asarray(v, np.float32).astype(np.float64)
    return oracle.Transform(f64(A).reshape(3, 3), f64(t).reshape(3), f64(S).reshape(3, 3), f64(xmin),
                            f64(xmax))


def oracle_T_of(pair):
    return oracle_T(pair.A, pair.t, pair.S, pair.xmin, pair.xmax)


def gpu_T_of(pair):
    from voxel_grid_sampler_gb300 import ffdp
    return ffdp.transform(pair.A, pair.t, pair.S, pair.xmin, pair.xmax)


def host(t):
    return t.detach().cpu().numpy()


def random_transform(rng, scale=0.1, s_offdiag=True):
    A = (np.eye(3) + rng.uniform(-scale, scale, (3, 3))).astype(np.float32)
    t = rng.uniform(-scale, scale, 3).astype(np.float32)
    S = (np.eye(3) * 0.9 + (rng.uniform(-0.1, 0.1, (3, 3)) if s_offdiag else 0)).astype(np.float32)
    xmin = np.array([-0.95, -1.0, -0.9], np.float32)
    xmax = np.array([1.0, 0.92, 0.97], np.float32)
    return A, t, S, xmin, xmax


def report(name, **errs):
    """Print measured errors next to their tolerances (visible with pytest -s)."""
    parts = ["%s=%.3g" % (k, float(v)) for k, v in errs.items()]
    print("[parity] %s: %s" % (name, " ".join(parts)))
