"""Seeded synthetic volume pairs for the five registration workloads.

This module only makes inputs.  It holds none of the objective's arithmetic:
it draws noise, rasterises ellipsoid phantoms analytically, smooths with a
separable Gaussian and, to make a moving image from a noise image, calls the
library routine ``torch.nn.functional.grid_sample``.  The CUDA library and the
CPU oracle both consume the bytes produced here.

The datasets the paper evaluates on (OASIS, Faux-OASIS, the 100 um ex-vivo
brain) are not available; these volumes stand in for them with the shapes,
value ranges and structure of each workload:

  1  64^3 fp32        smoothed uniform noise; M = affine+elastic warp of F,
                      remapped 1 - x^2 plus N(0, 0.01); MI(32) and LNCC(5)
  2  160x192x224 fp32 3-tissue phantom (sigma 1.5); M = sin remap of the
                      warped phantom + Rician noise 0.03; MI(32)
  3  256^3 fp32       smoothed noise + ellipsoid blobs; M = elastic warp
                      (max 6 vox) + N(0, 0.02); LNCC(7)
  4  512^3 fp32       as 2 at 512^3; MI(64) + LNCC(5)
  5  1024^3 fp16 F/M  as 2 at 1024^3, field max 8 vox; MI(32)

Conventions: volumes are [D][H][W]; "N(0, s)" is standard deviation s;
Gaussian smoothing is separable, truncated at 4 sigma, replicate borders;
"smoothed noise in [0,1]" is smoothed then min-max rescaled; a smooth
displacement field of max m voxels is 3 channels of N(0,1) smoothed with
sigma, scaled so the largest Euclidean norm is m voxels, then converted to
the normalised units of the moving image (2/(n-1) per axis).  The evaluation
point (A, t, u) is an independent draw from the workload's own warp
distribution (affine only for workload 1; A = I, t = 0 otherwise), S = I and
x_bounds = (-1, 1).  MI intensity ranges are each image's own min and max.
"""
from __future__ import annotations

import hashlib
import math
from dataclasses import dataclass, field

import numpy as np
import torch
import torch.nn.functional as Fnn


@dataclass
class Workload:
    index: int
    name: str
    shape: tuple          # fixed and moving grid (D, H, W)
    dtype: str            # "f32" or "f16" for F and M; u is always f32
    w_mi: float
    w_lncc: float
    bins: int
    window: int
    eps: float = 1e-5
    kind: str = "noise"   # "noise" | "phantom" | "blobs"
    gen_disp_vox: float = 2.0
    gen_disp_sigma: float = 4.0
    eval_disp_vox: float = 2.0
    affine: bool = False


WORKLOADS = {
    1: Workload(1, "64^3 fp32 noise pair, MI32 + LNCC5", (64, 64, 64), "f32", 1.0, 1.0, 32, 5,
                kind="noise", gen_disp_vox=2.0, eval_disp_vox=2.0, affine=True),
    2: Workload(2, "160x192x224 fp32 phantom pair, MI32", (160, 192, 224), "f32", 1.0, 0.0, 32, 5,
                kind="phantom", gen_disp_vox=4.0, eval_disp_vox=4.0),
    3: Workload(3, "256^3 fp32 blob pair, LNCC7", (256, 256, 256), "f32", 0.0, 1.0, 32, 7,
                kind="blobs", gen_disp_vox=6.0, gen_disp_sigma=8.0, eval_disp_vox=6.0),
    4: Workload(4, "512^3 fp32 phantom pair, MI64 + LNCC5", (512, 512, 512), "f32", 1.0, 1.0, 64, 5,
                kind="phantom", gen_disp_vox=4.0, eval_disp_vox=4.0),
    5: Workload(5, "1024^3 fp16 phantom pair, MI32", (1024, 1024, 1024), "f16", 1.0, 0.0, 32, 5,
                kind="phantom", gen_disp_vox=8.0, eval_disp_vox=8.0),
}


@dataclass
class Pair:
    """One generated problem: images, displacement and evaluation transform."""
    F: torch.Tensor                 # [D,H,W] f32 or f16
    M: torch.Tensor                 # [D,H,W] f32 or f16
    u: torch.Tensor                 # [D,H,W,3] f32, normalised units of M
    A: np.ndarray                   # 3x3 float32
    t: np.ndarray                   # 3 float32
    S: np.ndarray = field(default_factory=lambda: np.eye(3, dtype=np.float32))
    xmin: np.ndarray = field(default_factory=lambda: -np.ones(3, dtype=np.float32))
    xmax: np.ndarray = field(default_factory=lambda: np.ones(3, dtype=np.float32))
    f_range: tuple = (0.0, 1.0)
    m_range: tuple = (0.0, 1.0)
    workload: Workload | None = None

    def checksums(self) -> dict:
        out = {}
        for k in ("F", "M", "u"):
            t = getattr(self, k).detach().contiguous().cpu()
            out[k] = hashlib.sha256(t.view(torch.uint8).numpy().tobytes()).hexdigest()[:16] \
                if t.numel() * t.element_size() < (1 << 28) else "skipped(large)"
        return out


# ----------------------------------------------------------------- primitives
def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def gaussian_smooth(vol: torch.Tensor, sigma: float, chunk_elems: int = 1 << 27) -> torch.Tensor:
    """Separable Gaussian (truncated at 4 sigma, replicate borders) of a [D,H,W] float32 volume."""
    if sigma <= 0:
        return vol
    rad = int(math.ceil(4.0 * sigma))
    xs = torch.arange(-rad, rad + 1, dtype=torch.float64)
    k = torch.exp(-0.5 * (xs / sigma) ** 2)
    k = (k / k.sum()).to(device=vol.device, dtype=torch.float32).view(1, 1, -1)
    out = vol
    for axis in range(3):
        v = out.movedim(axis, -1).contiguous()
        shp = v.shape
        v = v.view(-1, 1, shp[-1])
        res = torch.empty_like(v)
        rows = max(1, chunk_elems // shp[-1])
        for s in range(0, v.shape[0], rows):
            part = Fnn.pad(v[s:s + rows], (rad, rad), mode="replicate")
            res[s:s + rows] = Fnn.conv1d(part, k)
        out = res.view(shp).movedim(-1, axis).contiguous()
        del v, res
    return out


def _rescale01(v: torch.Tensor) -> torch.Tensor:
    lo, hi = v.min(), v.max()
    return (v - lo) / (hi - lo)


def smooth_field_vox(shape, sigma: float, max_vox: float, g: torch.Generator, device) -> torch.Tensor:
    """[D,H,W,3] displacement in voxels (x, y, z components), max Euclidean norm max_vox."""
    comps = []
    for _ in range(3):
        n = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        comps.append(gaussian_smooth(n, sigma))
        del n
    d = torch.stack(comps, dim=-1)
    del comps
    norm = torch.sqrt((d * d).sum(-1)).max()
    return d * (max_vox / norm)


def vox_to_norm(d_vox: torch.Tensor, shape) -> torch.Tensor:
    D, H, W = shape
    scale = torch.tensor([2.0 / (W - 1), 2.0 / (H - 1), 2.0 / (D - 1)], device=d_vox.device,
                         dtype=torch.float32)
    return d_vox * scale


def _norm_axes(shape, device, z0=0, z1=None):
    D, H, W = shape
    z1 = D if z1 is None else z1
    zs = torch.linspace(-1, 1, D, device=device, dtype=torch.float32)[z0:z1]
    ys = torch.linspace(-1, 1, H, device=device, dtype=torch.float32)
    xs = torch.linspace(-1, 1, W, device=device, dtype=torch.float32)
    return zs, ys, xs


def _random_ellipsoids(rng: np.random.Generator, nested: bool, count: int):
    """Ellipsoids in normalised coordinates: (centre[3], semi-axes[3], rotation 3x3)."""
    out = []
    scale = 0.9
    centre = rng.uniform(-0.05, 0.05, 3)
    for i in range(count):
        if nested:
            axes = np.array([scale, scale * rng.uniform(0.8, 1.0), scale * rng.uniform(0.7, 0.95)])
            scale *= rng.uniform(0.7, 0.8)
            c = centre + rng.uniform(-0.05, 0.05, 3) * i
        else:
            axes = rng.uniform(0.08, 0.3, 3)
            c = rng.uniform(-0.6, 0.6, 3)
        q = rng.normal(size=4)
        q /= np.linalg.norm(q)
        w, x, y, z = q
        R = np.array([[1 - 2 * (y * y + z * z), 2 * (x * y - z * w), 2 * (x * z + y * w)],
                      [2 * (x * y + z * w), 1 - 2 * (x * x + z * z), 2 * (y * z - x * w)],
                      [2 * (x * z - y * w), 2 * (y * z + x * w), 1 - 2 * (x * x + y * y)]])
        out.append((c, axes, R))
    return out


def _raster_ellipsoids(shape, ells, values, device, disp_norm=None, nested=True,
                       planes_per_chunk: int = 16) -> torch.Tensor:
    """Rasterise ellipsoids analytically at voxel centres (optionally displaced by
    disp_norm, [D,H,W,3] normalised units).  Nested: value of the innermost
    containing ellipsoid; else the sum of the values of containing blobs."""
    D, H, W = shape
    out = torch.zeros(shape, dtype=torch.float32, device=device)
    for z0 in range(0, D, planes_per_chunk):
        z1 = min(D, z0 + planes_per_chunk)
        zs, ys, xs = _norm_axes(shape, device, z0, z1)
        Z, Y, X = torch.meshgrid(zs, ys, xs, indexing="ij")
        P = torch.stack([X, Y, Z], dim=-1)
        if disp_norm is not None:
            P = P + disp_norm[z0:z1]
        acc = torch.zeros(P.shape[:-1], dtype=torch.float32, device=device)
        for (c, axes, R), val in zip(ells, values):
            Rt = torch.tensor(R.T, dtype=torch.float32, device=device)
            ct = torch.tensor(c, dtype=torch.float32, device=device)
            at = torch.tensor(axes, dtype=torch.float32, device=device)
            L = ((P - ct) @ Rt) / at
            inside = (L * L).sum(-1) <= 1.0
            if nested:
                acc = torch.where(inside, torch.full_like(acc, val), acc)
            else:
                acc = acc + inside.float() * val
        out[z0:z1] = acc
        del P, acc
    return out


def _affine_draw(rng: np.random.Generator, shape, max_deg=5.0, scale=(0.95, 1.05), max_shift_vox=3.0):
    axis = rng.normal(size=3)
    axis /= np.linalg.norm(axis)
    ang = math.radians(rng.uniform(-max_deg, max_deg))
    Kx = np.array([[0, -axis[2], axis[1]], [axis[2], 0, -axis[0]], [-axis[1], axis[0], 0]])
    R = np.eye(3) + math.sin(ang) * Kx + (1 - math.cos(ang)) * (Kx @ Kx)
    A = R @ np.diag(rng.uniform(scale[0], scale[1], 3))
    D, H, W = shape
    shift_vox = rng.uniform(-max_shift_vox, max_shift_vox, 3)
    t = shift_vox * np.array([2.0 / (W - 1), 2.0 / (H - 1), 2.0 / (D - 1)])
    return A.astype(np.float32), t.astype(np.float32)


def _warp_library(vol: torch.Tensor, A, t, disp_norm) -> torch.Tensor:
    """Moving image for the noise workloads: torch.nn.functional.grid_sample of vol
    at A x + t + d(x) (library routine, trilinear, align_corners=True, zeros)."""
    D, H, W = vol.shape
    device = vol.device
    out = torch.empty_like(vol)
    At = torch.tensor(A, dtype=torch.float32, device=device)
    tt = torch.tensor(t, dtype=torch.float32, device=device)
    for z0 in range(0, D, 16):
        z1 = min(D, z0 + 16)
        zs, ys, xs = _norm_axes((D, H, W), device, z0, z1)
        Z, Y, X = torch.meshgrid(zs, ys, xs, indexing="ij")
        P = torch.stack([X, Y, Z], dim=-1) @ At.T + tt + disp_norm[z0:z1]
        s = Fnn.grid_sample(vol[None, None], P[None], mode="bilinear", padding_mode="zeros",
                            align_corners=True)
        out[z0:z1] = s[0, 0]
    return out


# ------------------------------------------------------------------ workloads
def make_pair(index: int, device="cpu", shape=None, seed: int | None = None) -> Pair:
    """Generate workload ``index`` (1..5).  ``shape`` overrides the size (same recipe)."""
    wl = WORKLOADS[index]
    shape = tuple(shape) if shape is not None else wl.shape
    seed = 1000 + index if seed is None else seed
    rng = np.random.default_rng(seed)
    g_img = _gen(seed * 16 + 1, device)
    g_gen = _gen(seed * 16 + 2, device)
    g_eval = _gen(seed * 16 + 3, device)
    g_noise = _gen(seed * 16 + 4, device)
    with torch.no_grad():
        gen_d = vox_to_norm(smooth_field_vox(shape, wl.gen_disp_sigma, wl.gen_disp_vox, g_gen, device),
                            shape)
        if wl.kind == "phantom":
            ells = _random_ellipsoids(rng, nested=True, count=3)
            vals = [0.25, 0.55, 0.85]
            F = gaussian_smooth(_raster_ellipsoids(shape, ells, vals, device), 1.5)
            Mw = gaussian_smooth(_raster_ellipsoids(shape, ells, vals, device, disp_norm=gen_d), 1.5)
            del gen_d
            Mw = 0.5 + 0.4 * torch.sin(3.0 * math.pi * Mw)
            n1 = torch.randn(shape, generator=g_noise, device=device) * 0.03
            n2 = torch.randn(shape, generator=g_noise, device=device) * 0.03
            M = torch.sqrt((Mw + n1) ** 2 + n2 ** 2)
            del Mw, n1, n2
            A_gen = None
        else:
            if wl.kind == "noise":
                F = _rescale01(gaussian_smooth(torch.rand(shape, generator=g_img, device=device), 2.0))
            else:  # blobs
                base = _rescale01(gaussian_smooth(torch.rand(shape, generator=g_img, device=device), 2.0))
                ells = _random_ellipsoids(rng, nested=False, count=8)
                vals = list(rng.uniform(0.2, 0.5, len(ells)))
                blobs = gaussian_smooth(_raster_ellipsoids(shape, ells, vals, device, nested=False), 1.5)
                F = 0.5 * base + blobs
                del base, blobs
            if wl.affine:
                A_gen, t_gen = _affine_draw(rng, shape)
            else:
                A_gen, t_gen = np.eye(3, dtype=np.float32), np.zeros(3, np.float32)
            Mw = _warp_library(F, A_gen, t_gen, gen_d)
            del gen_d
            if wl.kind == "noise":
                M = 1.0 - Mw * Mw + torch.randn(shape, generator=g_noise, device=device) * 0.01
            else:
                M = Mw + torch.randn(shape, generator=g_noise, device=device) * 0.02
            del Mw
        # evaluation point: an independent draw of the workload's warp distribution
        u = vox_to_norm(smooth_field_vox(shape, wl.gen_disp_sigma, wl.eval_disp_vox, g_eval, device),
                        shape).contiguous()
        if wl.affine:
            A, t = _affine_draw(rng, shape)
        else:
            A, t = np.eye(3, dtype=np.float32), np.zeros(3, np.float32)
        if wl.dtype == "f16":
            F = F.to(torch.float16)
            M = M.to(torch.float16)
        F = F.contiguous()
        M = M.contiguous()
        f_range = (float(F.min()), float(F.max()))
        m_range = (float(M.min()), float(M.max()))
    return Pair(F=F, M=M, u=u, A=A, t=t, f_range=f_range, m_range=m_range, workload=wl)


def random_pair(shape, mshape=None, seed: int = 0, device="cpu", disp_vox: float = 1.5,
                dtype=torch.float32, affine: bool = True) -> Pair:
    """Small generic pair for parity tests (odd shapes, M shape may differ)."""
    mshape = tuple(shape) if mshape is None else tuple(mshape)
    rng = np.random.default_rng(seed)
    g = _gen(seed * 16 + 7, device)
    with torch.no_grad():
        F = _rescale01(gaussian_smooth(torch.rand(shape, generator=g, device=device), 1.0))
        M = _rescale01(gaussian_smooth(torch.rand(mshape, generator=g, device=device), 1.0))
        u = vox_to_norm(smooth_field_vox(tuple(shape), 2.0, disp_vox, g, device), mshape).contiguous()
    if affine:
        A, t = _affine_draw(rng, mshape)
    else:
        A, t = np.eye(3, dtype=np.float32), np.zeros(3, np.float32)
    F = F.to(dtype).contiguous()
    M = M.to(dtype).contiguous()
    return Pair(F=F, M=M, u=u, A=A, t=t, f_range=(float(F.min()), float(F.max())),
                m_range=(float(M.min()), float(M.max())))
