"""ctypes binding of libffdp (include/ffdp.h): argument marshalling only.

Every function here has the name of the C entry point it calls and does no
arithmetic of its own: it checks that tensors are CUDA, contiguous and of the
expected dtype, allocates outputs (and the workspace) with torch when the
caller did not pass them, and hands raw pointers plus the current torch
stream to the library.  If the shared library is missing, calls raise
``FfdpError``; there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libffdp.so")

FFDP_F32, FFDP_F16 = 0, 1
FFDP_OP_GRID_SAMPLE_BWD, FFDP_OP_MI, FFDP_OP_LNCC, FFDP_OP_OBJECTIVE = 1, 2, 3, 4
FFDP_OP_SAMPLE_CHANNELS_BWD, FFDP_OP_MSE, FFDP_OP_OBJECTIVE_MSE, FFDP_OP_SOBOLEV = 5, 6, 7, 8
FFDP_OP_OBJECTIVE_STORED = 9
STATUS = {0: "FFDP_OK", 1: "FFDP_ERR_INVALID_ARGUMENT", 2: "FFDP_ERR_UNSUPPORTED",
          3: "FFDP_ERR_WORKSPACE", 4: "FFDP_ERR_CUDA", 5: "FFDP_ERR_INTERNAL"}


class FfdpError(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__("%s: %s" % (STATUS.get(status, status), detail))
        self.status = status


class ffdp_dims(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int64), ("h", ctypes.c_int64), ("w", ctypes.c_int64)]


class ffdp_transform(ctypes.Structure):
    _fields_ = [("A", ctypes.c_float * 9), ("t", ctypes.c_float * 3), ("S", ctypes.c_float * 9),
                ("xmin", ctypes.c_float * 3), ("xmax", ctypes.c_float * 3)]


class ffdp_mi_params(ctypes.Structure):
    _fields_ = [("bins", ctypes.c_int), ("f_lo", ctypes.c_float), ("f_hi", ctypes.c_float),
                ("m_lo", ctypes.c_float), ("m_hi", ctypes.c_float)]


class ffdp_lncc_params(ctypes.Structure):
    _fields_ = [("window", ctypes.c_int), ("eps", ctypes.c_float)]


class ffdp_sobolev_adam_params(ctypes.Structure):
    _fields_ = [("lambda_", ctypes.c_float), ("lr", ctypes.c_float), ("beta1", ctypes.c_float),
                ("beta2", ctypes.c_float), ("eps", ctypes.c_float), ("step", ctypes.c_int)]


class ffdp_objective_params(ctypes.Structure):
    _fields_ = [("w_mi", ctypes.c_float), ("w_lncc", ctypes.c_float), ("mi", ffdp_mi_params),
                ("lncc", ffdp_lncc_params)]


_lib = None
_vp = ctypes.c_void_p


def lib() -> ctypes.CDLL:
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise FfdpError(5, "libffdp.so not built at %s (run voxel_grid_sampler_gb300.build.build())"
                            % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        L.ffdp_workspace_bytes.restype = ctypes.c_size_t
        L.ffdp_workspace_bytes.argtypes = [ctypes.c_int, ffdp_dims, _vp]
        L.ffdp_grid_sample_fwd.argtypes = [_vp, ctypes.c_int, ffdp_dims, ffdp_dims, _vp,
                                           ctypes.POINTER(ffdp_transform), _vp, _vp]
        L.ffdp_grid_sample_bwd.argtypes = [_vp, ctypes.c_int, ffdp_dims, ffdp_dims, _vp,
                                           ctypes.POINTER(ffdp_transform), _vp, _vp, _vp, _vp, _vp,
                                           ctypes.c_size_t, _vp]
        L.ffdp_mi_fwd_bwd.argtypes = [_vp, ctypes.c_int, _vp, ffdp_dims, ctypes.POINTER(ffdp_mi_params),
                                      _vp, _vp, _vp, ctypes.c_size_t, _vp]
        L.ffdp_lncc_fwd_bwd.argtypes = [_vp, ctypes.c_int, _vp, ffdp_dims,
                                        ctypes.POINTER(ffdp_lncc_params), _vp, _vp, _vp, ctypes.c_size_t,
                                        _vp]
        for f in ("ffdp_objective", "ffdp_objective_stored"):
            getattr(L, f).argtypes = [_vp, ctypes.c_int, ffdp_dims, _vp, ctypes.c_int, ffdp_dims, _vp,
                                      ctypes.POINTER(ffdp_transform),
                                      ctypes.POINTER(ffdp_objective_params), _vp, _vp, _vp, _vp, _vp,
                                      ctypes.c_size_t, _vp]
        L.ffdp_sample_channels_fwd.argtypes = [_vp, ctypes.c_int, ffdp_dims, ffdp_dims, _vp,
                                               ctypes.POINTER(ffdp_transform), ctypes.c_int, _vp, _vp]
        L.ffdp_sample_channels_bwd.argtypes = [_vp, ctypes.c_int, ffdp_dims, ffdp_dims, _vp,
                                               ctypes.POINTER(ffdp_transform), ctypes.c_int, _vp, _vp, _vp,
                                               _vp, _vp, _vp, ctypes.c_size_t, _vp]
        L.ffdp_mse_fwd_bwd.argtypes = [_vp, ctypes.c_int, _vp, ffdp_dims, _vp, _vp, _vp, ctypes.c_size_t, _vp]
        L.ffdp_objective_mse.argtypes = [_vp, ctypes.c_int, ffdp_dims, _vp, ctypes.c_int, ffdp_dims, _vp,
                                         ctypes.POINTER(ffdp_transform), ctypes.c_float, _vp, _vp, _vp, _vp,
                                         _vp, ctypes.c_size_t, _vp]
        L.ffdp_sobolev_fwd_bwd.argtypes = [_vp, ffdp_dims, ctypes.c_float, _vp, _vp, _vp, ctypes.c_size_t, _vp]
        L.ffdp_sobolev_adam_step.argtypes = [_vp, _vp, _vp, _vp, _vp, ffdp_dims,
                                             ctypes.POINTER(ffdp_sobolev_adam_params), _vp, _vp, ctypes.c_size_t,
                                             _vp]
        for f in ("ffdp_grid_sample_fwd", "ffdp_grid_sample_bwd", "ffdp_mi_fwd_bwd",
                  "ffdp_lncc_fwd_bwd", "ffdp_objective", "ffdp_objective_stored", "ffdp_sample_channels_fwd",
                  "ffdp_sample_channels_bwd", "ffdp_mse_fwd_bwd", "ffdp_objective_mse",
                  "ffdp_sobolev_fwd_bwd", "ffdp_sobolev_adam_step"):
            getattr(L, f).restype = ctypes.c_int
        L.ffdp_status_string.restype = ctypes.c_char_p
        L.ffdp_status_string.argtypes = [ctypes.c_int]
        L.ffdp_last_error.restype = ctypes.c_char_p
        L.ffdp_launch_count.restype = ctypes.c_uint64
        L.ffdp_timing_enable.argtypes = [ctypes.c_int]
        L.ffdp_timing_enable.restype = ctypes.c_int
        L.ffdp_timing_read.argtypes = [ctypes.c_char_p, ctypes.POINTER(ctypes.c_int),
                                       ctypes.POINTER(ctypes.c_double), ctypes.c_int]
        L.ffdp_timing_read.restype = ctypes.c_int
        L.ffdp_device_error.argtypes = [ctypes.POINTER(ctypes.c_int)]
        L.ffdp_device_error.restype = ctypes.c_int
        L.ffdp_test_ring_stall.argtypes = [ctypes.c_int]
        L.ffdp_test_ring_stall.restype = ctypes.c_int
        _lib = L
    return _lib


# ---------------------------------------------------------------- marshalling
def dims_of(shape) -> ffdp_dims:
    d, h, w = (int(s) for s in shape)
    return ffdp_dims(d, h, w)


def transform(A=None, t=None, S=None, xmin=None, xmax=None) -> ffdp_transform:
    """Host transform struct; defaults: A = S = I, t = 0, x_bounds = (-1, 1)."""
    T = ffdp_transform()
    A = np.eye(3) if A is None else np.asarray(A, np.float64).reshape(3, 3)
    S = np.eye(3) if S is None else np.asarray(S, np.float64).reshape(3, 3)
    t = np.zeros(3) if t is None else np.asarray(t, np.float64).reshape(3)
    xmin = -np.ones(3) if xmin is None else np.asarray(xmin, np.float64).reshape(3)
    xmax = np.ones(3) if xmax is None else np.asarray(xmax, np.float64).reshape(3)
    T.A[:] = [float(v) for v in A.reshape(9)]
    T.S[:] = [float(v) for v in S.reshape(9)]
    T.t[:] = [float(v) for v in t]
    T.xmin[:] = [float(v) for v in xmin]
    T.xmax[:] = [float(v) for v in xmax]
    return T


def mi_params(bins, f_range, m_range) -> ffdp_mi_params:
    return ffdp_mi_params(int(bins), float(f_range[0]), float(f_range[1]), float(m_range[0]),
                          float(m_range[1]))


def lncc_params(window, eps=1e-5) -> ffdp_lncc_params:
    return ffdp_lncc_params(int(window), float(eps))


def objective_params(w_mi, w_lncc, bins, f_range, m_range, window, eps=1e-5) -> ffdp_objective_params:
    return ffdp_objective_params(float(w_mi), float(w_lncc), mi_params(bins, f_range, m_range),
                                 lncc_params(window, eps))


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return FFDP_F32
    if t.dtype == torch.float16:
        return FFDP_F16
    raise FfdpError(1, "volumes must be float32 or float16, got %s" % t.dtype)


def _dev(t, name, dtype=None, ndim=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise FfdpError(1, "%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise FfdpError(1, "%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise FfdpError(1, "%s must be %s" % (name, dtype))
    if ndim is not None and t.dim() != ndim:
        raise FfdpError(1, "%s must have %d dims" % (name, ndim))
    return t


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(status: int):
    if status != 0:
        raise FfdpError(status, (lib().ffdp_last_error() or b"").decode())


def ffdp_workspace_bytes(op: int, fixed_shape, params=None) -> int:
    p = None if params is None else ctypes.byref(params)
    return int(lib().ffdp_workspace_bytes(op, dims_of(fixed_shape), p))


def workspace(op: int, fixed_shape, params=None, device="cuda") -> torch.Tensor:
    n = ffdp_workspace_bytes(op, fixed_shape, params)
    if n == 0:
        raise FfdpError(1, (lib().ffdp_last_error() or b"invalid workspace request").decode())
    return torch.empty(n, dtype=torch.uint8, device=device)


# ------------------------------------------------------------------ entries
def ffdp_grid_sample_fwd(M, out_shape, u, T: ffdp_transform, J_out=None, stream=None):
    _dev(M, "M", ndim=3)
    _dev(u, "u", torch.float32, 4)
    if J_out is None:
        J_out = torch.empty(tuple(out_shape), dtype=torch.float32, device=M.device)
    _dev(J_out, "J_out", torch.float32, 3)
    _check(lib().ffdp_grid_sample_fwd(_ptr(M), _dtype_code(M), dims_of(M.shape), dims_of(out_shape),
                                      _ptr(u), ctypes.byref(T), _ptr(J_out), _stream(stream)))
    return J_out


def ffdp_grid_sample_bwd(M, u, T: ffdp_transform, gJ, du=None, dA=None, dt=None, ws=None,
                         stream=None, want_du=True):
    _dev(M, "M", ndim=3)
    _dev(gJ, "gJ", torch.float32, 3)
    _dev(u, "u", torch.float32, 4)
    shape = tuple(gJ.shape)
    if du is None and want_du:
        du = torch.empty(shape + (3,), dtype=torch.float32, device=M.device)
    if dA is None:
        dA = torch.empty(9, dtype=torch.float32, device=M.device)
    if dt is None:
        dt = torch.empty(3, dtype=torch.float32, device=M.device)
    if ws is None:
        ws = workspace(FFDP_OP_GRID_SAMPLE_BWD, shape, None, M.device)
    _check(lib().ffdp_grid_sample_bwd(_ptr(M), _dtype_code(M), dims_of(M.shape), dims_of(shape), _ptr(u),
                                      ctypes.byref(T), _ptr(gJ), _ptr(du), _ptr(dA), _ptr(dt), _ptr(ws),
                                      ws.numel(), _stream(stream)))
    return du, dA, dt


def ffdp_mi_fwd_bwd(F, J, params: ffdp_mi_params, loss=None, dJ=None, ws=None, stream=None,
                    want_grad=True):
    _dev(F, "F", ndim=3)
    _dev(J, "J", torch.float32, 3)
    if loss is None:
        loss = torch.empty(1, dtype=torch.float32, device=F.device)
    if dJ is None and want_grad:
        dJ = torch.empty_like(J)
    if ws is None:
        ws = workspace(FFDP_OP_MI, F.shape, params, F.device)
    _check(lib().ffdp_mi_fwd_bwd(_ptr(F), _dtype_code(F), _ptr(J), dims_of(F.shape), ctypes.byref(params),
                                 _ptr(loss), _ptr(dJ), _ptr(ws), ws.numel(), _stream(stream)))
    return loss, dJ


def ffdp_lncc_fwd_bwd(F, J, params: ffdp_lncc_params, loss=None, dJ=None, ws=None, stream=None,
                      want_grad=True):
    _dev(F, "F", ndim=3)
    _dev(J, "J", torch.float32, 3)
    if loss is None:
        loss = torch.empty(1, dtype=torch.float32, device=F.device)
    if dJ is None and want_grad:
        dJ = torch.empty_like(J)
    if ws is None:
        ws = workspace(FFDP_OP_LNCC, F.shape, params, F.device)
    _check(lib().ffdp_lncc_fwd_bwd(_ptr(F), _dtype_code(F), _ptr(J), dims_of(F.shape),
                                   ctypes.byref(params), _ptr(loss), _ptr(dJ), _ptr(ws), ws.numel(),
                                   _stream(stream)))
    return loss, dJ


def ffdp_objective(F, M, u, T: ffdp_transform, params: ffdp_objective_params, loss=None, du=None,
                   dA=None, dt=None, ws=None, stream=None, want_du=True, store_slope=False):
    """The fused objective; store_slope selects ffdp_objective_stored (an MI-only
    objective keeps J and its slope in the workspace for a streaming gradient pass)."""
    _dev(F, "F", ndim=3)
    _dev(M, "M", ndim=3)
    _dev(u, "u", torch.float32, 4)
    dev = F.device
    if loss is None:
        loss = torch.empty(3, dtype=torch.float32, device=dev)
    if du is None and want_du:
        du = torch.empty(tuple(F.shape) + (3,), dtype=torch.float32, device=dev)
    if dA is None:
        dA = torch.empty(9, dtype=torch.float32, device=dev)
    if dt is None:
        dt = torch.empty(3, dtype=torch.float32, device=dev)
    if ws is None:
        ws = workspace(FFDP_OP_OBJECTIVE_STORED if store_slope else FFDP_OP_OBJECTIVE, F.shape, params, dev)
    fn = lib().ffdp_objective_stored if store_slope else lib().ffdp_objective
    _check(fn(_ptr(F), _dtype_code(F), dims_of(F.shape), _ptr(M), _dtype_code(M),
              dims_of(M.shape), _ptr(u), ctypes.byref(T), ctypes.byref(params),
              _ptr(loss), _ptr(du), _ptr(dA), _ptr(dt), _ptr(ws), ws.numel(),
              _stream(stream)))
    return loss, du, dA, dt


# ------------------------------------------------------------ instrumentation
def ffdp_sample_channels_fwd(V, out_shape, u, T: ffdp_transform, compose=False, out=None, stream=None):
    """out = V(A x + t + S u) (+ S u when compose) for a channel-last float32 volume V
    of shape (Dv, Hv, Wv, C); returns (D, H, W, C)."""
    _dev(V, "V", torch.float32, 4)
    _dev(u, "u", torch.float32, 4)
    C = int(V.shape[3])
    if out is None:
        out = torch.empty(tuple(out_shape) + (C,), dtype=torch.float32, device=V.device)
    _dev(out, "out", torch.float32, 4)
    _check(lib().ffdp_sample_channels_fwd(_ptr(V), C, dims_of(V.shape[:3]), dims_of(out_shape), _ptr(u),
                                          ctypes.byref(T), int(bool(compose)), _ptr(out), _stream(stream)))
    return out


def ffdp_sample_channels_bwd(V, u, T: ffdp_transform, gout, compose=False, du=None, dA=None, dt=None,
                             dV=None, ws=None, stream=None, want_du=True, want_dV=True):
    """Backward of ffdp_sample_channels_fwd: returns (du, dA, dt, dV)."""
    _dev(V, "V", torch.float32, 4)
    _dev(u, "u", torch.float32, 4)
    _dev(gout, "gout", torch.float32, 4)
    C = int(V.shape[3])
    shape = tuple(gout.shape[:3])
    dev = V.device
    if du is None and want_du:
        du = torch.empty(shape + (3,), dtype=torch.float32, device=dev)
    if dV is None and want_dV:
        dV = torch.empty_like(V)
    if dA is None:
        dA = torch.empty(9, dtype=torch.float32, device=dev)
    if dt is None:
        dt = torch.empty(3, dtype=torch.float32, device=dev)
    if ws is None:
        ws = workspace(FFDP_OP_SAMPLE_CHANNELS_BWD, shape, None, dev)
    _check(lib().ffdp_sample_channels_bwd(_ptr(V), C, dims_of(V.shape[:3]), dims_of(shape), _ptr(u),
                                          ctypes.byref(T), int(bool(compose)), _ptr(gout), _ptr(du), _ptr(dA),
                                          _ptr(dt), _ptr(dV), _ptr(ws), ws.numel(), _stream(stream)))
    return du, dA, dt, dV


def ffdp_mse_fwd_bwd(F, J, loss=None, dJ=None, ws=None, stream=None, want_grad=True):
    _dev(F, "F", ndim=3)
    _dev(J, "J", torch.float32, 3)
    if loss is None:
        loss = torch.empty(1, dtype=torch.float32, device=F.device)
    if dJ is None and want_grad:
        dJ = torch.empty_like(J)
    if ws is None:
        ws = workspace(FFDP_OP_MSE, F.shape, None, F.device)
    _check(lib().ffdp_mse_fwd_bwd(_ptr(F), _dtype_code(F), _ptr(J), dims_of(F.shape), _ptr(loss), _ptr(dJ),
                                  _ptr(ws), ws.numel(), _stream(stream)))
    return loss, dJ


def ffdp_objective_mse(F, M, u, T: ffdp_transform, w_mse=1.0, loss=None, du=None, dA=None, dt=None,
                       ws=None, stream=None, want_du=True):
    """Fused L = w_mse * MSE(F, M o phi): returns (loss[2] = {w_mse MSE, MSE}, du, dA, dt)."""
    _dev(F, "F", ndim=3)
    _dev(M, "M", ndim=3)
    _dev(u, "u", torch.float32, 4)
    dev = F.device
    if loss is None:
        loss = torch.empty(2, dtype=torch.float32, device=dev)
    if du is None and want_du:
        du = torch.empty(tuple(F.shape) + (3,), dtype=torch.float32, device=dev)
    if dA is None:
        dA = torch.empty(9, dtype=torch.float32, device=dev)
    if dt is None:
        dt = torch.empty(3, dtype=torch.float32, device=dev)
    if ws is None:
        ws = workspace(FFDP_OP_OBJECTIVE_MSE, F.shape, None, dev)
    _check(lib().ffdp_objective_mse(_ptr(F), _dtype_code(F), dims_of(F.shape), _ptr(M), _dtype_code(M),
                                    dims_of(M.shape), _ptr(u), ctypes.byref(T), float(w_mse), _ptr(loss),
                                    _ptr(du), _ptr(dA), _ptr(dt), _ptr(ws), ws.numel(), _stream(stream)))
    return loss, du, dA, dt


def sobolev_adam_params(lam, lr, beta1=0.9, beta2=0.999, eps=1e-8, step=1) -> ffdp_sobolev_adam_params:
    return ffdp_sobolev_adam_params(float(lam), float(lr), float(beta1), float(beta2), float(eps), int(step))


def ffdp_sobolev_fwd_bwd(u, lam, loss=None, dR=None, ws=None, stream=None, want_grad=True):
    """R(u) (first-order Sobolev seminorm) and dR/du for u of shape (D, H, W, 3)."""
    _dev(u, "u", torch.float32, 4)
    shape = tuple(u.shape[:3])
    if loss is None:
        loss = torch.empty(1, dtype=torch.float32, device=u.device)
    if dR is None and want_grad:
        dR = torch.empty_like(u)
    if ws is None:
        ws = workspace(FFDP_OP_SOBOLEV, shape, None, u.device)
    _check(lib().ffdp_sobolev_fwd_bwd(_ptr(u), dims_of(shape), float(lam), _ptr(loss), _ptr(dR), _ptr(ws),
                                      ws.numel(), _stream(stream)))
    return loss, dR


def ffdp_sobolev_adam_step(u, g, m1, m2, params: ffdp_sobolev_adam_params, u_out=None, loss=None, ws=None,
                           stream=None):
    """One regularised Adam step: returns (u_out, loss[1] = R(u)); m1, m2 are updated in place."""
    for t, n in ((u, "u"), (g, "g"), (m1, "m1"), (m2, "m2")):
        _dev(t, n, torch.float32, 4)
    shape = tuple(u.shape[:3])
    if u_out is None:
        u_out = torch.empty_like(u)
    if loss is None:
        loss = torch.empty(1, dtype=torch.float32, device=u.device)
    if ws is None:
        ws = workspace(FFDP_OP_SOBOLEV, shape, None, u.device)
    _check(lib().ffdp_sobolev_adam_step(_ptr(u), _ptr(u_out), _ptr(g), _ptr(m1), _ptr(m2), dims_of(shape),
                                        ctypes.byref(params), _ptr(loss), _ptr(ws), ws.numel(), _stream(stream)))
    return u_out, loss


def launch_count() -> int:
    return int(lib().ffdp_launch_count())


def device_error() -> bool:
    """True if a sweep kernel gave up a bounded wait since the last call
    (synchronises the current device and clears the flag)."""
    flag = ctypes.c_int(0)
    _check(lib().ffdp_device_error(ctypes.byref(flag)))
    return bool(flag.value)


def test_ring_stall(on: bool = True) -> None:
    """Arm (or disarm) the one-shot ring stall of the next objective call (tests)."""
    _check(lib().ffdp_test_ring_stall(1 if on else 0))


def timing_enable(capacity: int) -> None:
    _check(lib().ffdp_timing_enable(int(capacity)))


def timing_read(max_kernels: int = 32) -> dict:
    names = ctypes.create_string_buffer(64 * max_kernels)
    counts = (ctypes.c_int * max_kernels)()
    ms = (ctypes.c_double * max_kernels)()
    n = lib().ffdp_timing_read(names, counts, ms, max_kernels)
    out = {}
    for k in range(min(n, max_kernels)):
        nm = names.raw[64 * k:64 * k + 64].split(b"\0", 1)[0].decode()
        out[nm] = (int(counts[k]), float(ms[k]))
    return out


def ffdp_objective_mi_static(F, M, u, T: ffdp_transform, params: ffdp_objective_params, loss, du, dA, dt,
                             stream=None):
    """Workspace-free MI objective (see include/ffdp.h): for callers that cannot
    allocate device memory.  All outputs must be passed in; nothing is allocated."""
    L = lib()
    fn = L.ffdp_objective_mi_static
    fn.restype = ctypes.c_int
    fn.argtypes = [_vp, ctypes.c_int, ffdp_dims, _vp, ctypes.c_int, ffdp_dims, _vp,
                   ctypes.POINTER(ffdp_transform), ctypes.POINTER(ffdp_objective_params), _vp, _vp, _vp,
                   _vp, _vp]
    _dev(F, "F", ndim=3)
    _dev(M, "M", ndim=3)
    _dev(u, "u", torch.float32, 4)
    _check(fn(_ptr(F), _dtype_code(F), dims_of(F.shape), _ptr(M), _dtype_code(M), dims_of(M.shape), _ptr(u),
              ctypes.byref(T), ctypes.byref(params), _ptr(loss), _ptr(du), _ptr(dA), _ptr(dt),
              _stream(stream)))
    return loss, du, dA, dt
