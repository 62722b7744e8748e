"""Host-side checks of the C ABI (no GPU needed): the library builds for
sm_103a, loads, exports every entry point include/ffdp.h declares, and
rejects invalid arguments with a status before anything is enqueued."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ffdp.h")


@pytest.fixture(scope="module")
def lib():
    from voxel_grid_sampler_gb300 import build, ffdp
    build.build()
    return ffdp.lib()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ffdp_[a-z_0-9]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert "ffdp_objective" in names and "ffdp_grid_sample_fwd" in names
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    from voxel_grid_sampler_gb300 import ffdp
    for code, name in ffdp.STATUS.items():
        assert lib.ffdp_status_string(code).decode() == name


# The calls below only ever pass arguments that validation rejects; they are
# skipped where a GPU is present (the GPU suite exercises real calls there).
nogpu = pytest.mark.skipif(torch.cuda.is_available(), reason="host-only validation checks")


@nogpu
def test_invalid_arguments_are_rejected_before_launch(lib):
    from voxel_grid_sampler_gb300 import ffdp
    n0 = lib.ffdp_launch_count()
    T = ffdp.transform()
    good = ffdp.dims_of((8, 8, 8))
    fake = ctypes.c_void_p(0x1000)       # never dereferenced: every call below is invalid
    odd = ctypes.c_void_p(0x1004)        # misaligned
    P = ffdp.objective_params(1.0, 1.0, 32, (0, 1), (0, 1), 5)
    ws = ctypes.c_void_p(0x2000)
    st = lib.ffdp_objective(None, 0, good, fake, 0, good, fake, ctypes.byref(T), ctypes.byref(P), fake,
                            fake, fake, fake, ws, 1 << 30, None)
    assert st == 1
    st = lib.ffdp_objective(odd, 0, good, fake, 0, good, fake, ctypes.byref(T), ctypes.byref(P), fake,
                            fake, fake, fake, ws, 1 << 30, None)
    assert st == 1
    st = lib.ffdp_grid_sample_fwd(fake, 0, good, ffdp.dims_of((1, 8, 8)), None, ctypes.byref(T), fake, None)
    assert st == 1
    st = lib.ffdp_grid_sample_fwd(fake, 7, good, good, None, ctypes.byref(T), fake, None)
    assert st == 1
    bad = ffdp.objective_params(1.0, 0.0, 65, (0, 1), (0, 1), 5)
    st = lib.ffdp_objective(fake, 0, good, fake, 0, good, fake, ctypes.byref(T), ctypes.byref(bad), fake,
                            fake, fake, fake, ws, 1 << 30, None)
    assert st == 1
    bad = ffdp.objective_params(0.0, 1.0, 32, (0, 1), (0, 1), 4)
    st = lib.ffdp_objective(fake, 0, good, fake, 0, good, fake, ctypes.byref(T), ctypes.byref(bad), fake,
                            fake, fake, fake, ws, 1 << 30, None)
    assert st == 1
    bad = ffdp.objective_params(1.0, 0.0, 32, (1, 1), (0, 1), 5)
    st = lib.ffdp_objective(fake, 0, good, fake, 0, good, fake, ctypes.byref(T), ctypes.byref(bad), fake,
                            fake, fake, fake, ws, 1 << 30, None)
    assert st == 1
    zero = ffdp.objective_params(0.0, 0.0, 32, (0, 1), (0, 1), 5)
    st = lib.ffdp_objective(fake, 0, good, fake, 0, good, fake, ctypes.byref(T), ctypes.byref(zero), fake,
                            fake, fake, fake, ws, 1 << 30, None)
    assert st == 1
    # workspace too small / missing
    st = lib.ffdp_objective(fake, 0, good, fake, 0, good, fake, ctypes.byref(T), ctypes.byref(P), fake,
                            fake, fake, fake, ws, 16, None)
    assert st == 3
    st = lib.ffdp_objective(fake, 0, good, fake, 0, good, fake, ctypes.byref(T), ctypes.byref(P), fake,
                            fake, fake, fake, None, 0, None)
    assert st == 3
    mp = ffdp.mi_params(32, (0, 1), (2, 1))
    st = lib.ffdp_mi_fwd_bwd(fake, 0, fake, good, ctypes.byref(mp), fake, fake, ws, 1 << 30, None)
    assert st == 1
    for w in (10, 1, -3):  # even, below 3
        lp = ffdp.lncc_params(w)
        st = lib.ffdp_lncc_fwd_bwd(fake, 0, fake, good, ctypes.byref(lp), fake, fake, ws, 1 << 30, None)
        assert st == 1
    assert lib.ffdp_launch_count() == n0
    assert len(lib.ffdp_last_error()) > 0


def test_workspace_is_o1_for_mi_and_sampler(lib):
    from voxel_grid_sampler_gb300 import ffdp
    p = ffdp.mi_params(64, (0, 1), (0, 1))
    small = ffdp.ffdp_workspace_bytes(ffdp.FFDP_OP_MI, (16, 16, 16), p)
    large = ffdp.ffdp_workspace_bytes(ffdp.FFDP_OP_MI, (1024, 1024, 1024), p)
    assert small == large > 0
    a = ffdp.ffdp_workspace_bytes(ffdp.FFDP_OP_GRID_SAMPLE_BWD, (16, 16, 16))
    b = ffdp.ffdp_workspace_bytes(ffdp.FFDP_OP_GRID_SAMPLE_BWD, (1024, 1024, 1024))
    assert a == b > 0
    # with LNCC the objective keeps J (4 bytes per voxel)
    q = ffdp.objective_params(1.0, 1.0, 64, (0, 1), (0, 1), 5)
    c = ffdp.ffdp_workspace_bytes(ffdp.FFDP_OP_OBJECTIVE, (64, 64, 64), q)
    assert c >= 4 * 64 ** 3
    assert ffdp.ffdp_workspace_bytes(ffdp.FFDP_OP_OBJECTIVE, (1, 64, 64), q) == 0


def test_objective_params_are_the_contract_struct(lib):
    # {w_mi, w_lncc, mi {bins, f_lo, f_hi, m_lo, m_hi}, lncc {window, eps}}: no
    # trailing field, so a caller laying the struct out as the boundary
    # specifies passes exactly what the library reads
    from voxel_grid_sampler_gb300 import ffdp
    names = [f[0] for f in ffdp.ffdp_objective_params._fields_]
    assert names == ["w_mi", "w_lncc", "mi", "lncc"]
    assert ctypes.sizeof(ffdp.ffdp_objective_params) == 4 + 4 + 20 + 8


def test_stored_objective_workspace(lib):
    # ffdp_objective_stored: an MI-only objective keeps J and its slope (16
    # bytes per voxel); with LNCC both entry points hold the same buffers
    from voxel_grid_sampler_gb300 import ffdp
    dims = (40, 50, 60)
    N = 40 * 50 * 60
    p = ffdp.objective_params(1.0, 0.0, 32, (0, 1), (0, 1), 5)
    a = ffdp.ffdp_workspace_bytes(ffdp.FFDP_OP_OBJECTIVE, dims, p)
    b = ffdp.ffdp_workspace_bytes(ffdp.FFDP_OP_OBJECTIVE_STORED, dims, p)
    assert 16 * N <= b - a <= 16 * N + 1024
    q = ffdp.objective_params(1.0, 1.0, 32, (0, 1), (0, 1), 5)
    assert (ffdp.ffdp_workspace_bytes(ffdp.FFDP_OP_OBJECTIVE, dims, q) ==
            ffdp.ffdp_workspace_bytes(ffdp.FFDP_OP_OBJECTIVE_STORED, dims, q))


def test_wide_lncc_windows_take_two_five_channel_buffers(lib):
    # windows up to 7 run as the forward / backward window-kernel pair, which
    # hands the three g-terms over in the workspace (12 bytes per voxel);
    # wider ones as separable box-sum passes through two [5][N] float buffers
    # (40 bytes per voxel); any odd window >= 3 is accepted
    from voxel_grid_sampler_gb300 import ffdp
    dims = (20, 30, 40)
    N = 20 * 30 * 40
    tiled = ffdp.ffdp_workspace_bytes(ffdp.FFDP_OP_LNCC, dims, ffdp.lncc_params(7))
    assert 12 * N <= tiled < 12 * N + (1 << 20)
    for w in (9, 11, 13, 61, 1001):
        wide = ffdp.ffdp_workspace_bytes(ffdp.FFDP_OP_LNCC, dims, ffdp.lncc_params(w))
        assert wide - tiled >= 28 * N and wide - tiled < 28 * N + 1024
    q7 = ffdp.objective_params(1.0, 1.0, 64, (0, 1), (0, 1), 7)
    q9 = ffdp.objective_params(1.0, 1.0, 64, (0, 1), (0, 1), 9)
    o7 = ffdp.ffdp_workspace_bytes(ffdp.FFDP_OP_OBJECTIVE, dims, q7)
    o9 = ffdp.ffdp_workspace_bytes(ffdp.FFDP_OP_OBJECTIVE, dims, q9)
    assert o9 - o7 >= 28 * N and o9 - o7 < 28 * N + 1024


@nogpu
def test_channel_sampler_and_mse_reject_invalid_arguments(lib):
    from voxel_grid_sampler_gb300 import ffdp
    n0 = lib.ffdp_launch_count()
    T = ffdp.transform()
    good = ffdp.dims_of((8, 8, 8))
    fake = ctypes.c_void_p(0x1000)
    odd = ctypes.c_void_p(0x1004)
    ws = ctypes.c_void_p(0x2000)
    # channels outside [1, 4]; compose with C != 3; misaligned V; null gout
    for C in (0, 5):
        assert lib.ffdp_sample_channels_fwd(fake, C, good, good, None, ctypes.byref(T), 0, fake, None) == 1
    assert lib.ffdp_sample_channels_fwd(fake, 2, good, good, None, ctypes.byref(T), 1, fake, None) == 1
    assert lib.ffdp_sample_channels_fwd(odd, 3, good, good, None, ctypes.byref(T), 0, fake, None) == 1
    assert lib.ffdp_sample_channels_bwd(fake, 3, good, good, None, ctypes.byref(T), 1, None, fake, fake, fake,
                                        fake, ws, 1 << 30, None) == 1
    assert lib.ffdp_sample_channels_bwd(fake, 3, good, good, None, ctypes.byref(T), 1, fake, fake, fake, fake,
                                        odd, ws, 1 << 30, None) == 1
    assert lib.ffdp_sample_channels_bwd(fake, 3, good, good, None, ctypes.byref(T), 1, fake, fake, fake, fake,
                                        fake, ws, 16, None) == 3
    # MSE: misaligned J, tiny dims, zero or non-finite weight, missing workspace
    assert lib.ffdp_mse_fwd_bwd(fake, 0, odd, good, fake, fake, ws, 1 << 30, None) == 1
    assert lib.ffdp_mse_fwd_bwd(fake, 0, fake, ffdp.dims_of((8, 1, 8)), fake, fake, ws, 1 << 30, None) == 1
    for w in (0.0, float("inf")):
        assert lib.ffdp_objective_mse(fake, 0, good, fake, 0, good, fake, ctypes.byref(T), w, fake, fake, fake,
                                      fake, ws, 1 << 30, None) == 1
    assert lib.ffdp_objective_mse(fake, 0, good, fake, 0, good, fake, ctypes.byref(T), 1.0, fake, fake, fake,
                                  fake, None, 0, None) == 3
    assert lib.ffdp_launch_count() == n0


def test_channel_and_mse_workspaces_are_o1(lib):
    from voxel_grid_sampler_gb300 import ffdp
    for op in (ffdp.FFDP_OP_SAMPLE_CHANNELS_BWD, ffdp.FFDP_OP_MSE, ffdp.FFDP_OP_OBJECTIVE_MSE):
        a = ffdp.ffdp_workspace_bytes(op, (16, 16, 16))
        b = ffdp.ffdp_workspace_bytes(op, (1024, 1024, 1024))
        assert a == b > 0


@nogpu
def test_regulariser_and_step_reject_invalid_arguments(lib):
    from voxel_grid_sampler_gb300 import ffdp
    n0 = lib.ffdp_launch_count()
    good = ffdp.dims_of((8, 8, 8))
    a, b, c, d, e = (ctypes.c_void_p(0x100000 * k) for k in range(1, 6))
    ws = ctypes.c_void_p(0x2000)
    p = ffdp.sobolev_adam_params(0.1, 0.01)
    assert lib.ffdp_sobolev_fwd_bwd(a, good, -1.0, b, c, ws, 1 << 30, None) == 1
    assert lib.ffdp_sobolev_fwd_bwd(a, good, 1.0, b, a, ws, 1 << 30, None) == 1       # dR overlaps u
    assert lib.ffdp_sobolev_fwd_bwd(a, good, 1.0, b, c, None, 0, None) == 3
    assert lib.ffdp_sobolev_adam_step(a, a, b, c, d, good, ctypes.byref(p), e, ws, 1 << 30, None) == 1  # u_out = u
    assert lib.ffdp_sobolev_adam_step(a, b, c, d, d, good, ctypes.byref(p), e, ws, 1 << 30, None) == 1  # m1 = m2
    for bad in (ffdp.sobolev_adam_params(0.1, 0.01, beta1=1.0), ffdp.sobolev_adam_params(0.1, 0.01, step=0),
                ffdp.sobolev_adam_params(0.1, 0.01, eps=-1.0), ffdp.sobolev_adam_params(float("nan"), 0.01)):
        assert lib.ffdp_sobolev_adam_step(a, b, c, d, e, good, ctypes.byref(bad), ctypes.c_void_p(0x600000), ws,
                                          1 << 30, None) == 1
    assert lib.ffdp_launch_count() == n0
