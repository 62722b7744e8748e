"""The seeded generators: shapes, dtypes, value ranges and reproducibility."""
import numpy as np
import pytest
import torch

from voxel_grid_sampler_gb300 import synth


@pytest.mark.parametrize("k", [1, 2, 3, 4, 5])
def test_workload_recipe_small(k):
    shape = (12, 14, 16)
    p = synth.make_pair(k, device="cpu", shape=shape)
    wl = synth.WORKLOADS[k]
    assert tuple(p.F.shape) == shape and tuple(p.M.shape) == shape
    assert tuple(p.u.shape) == shape + (3,) and p.u.dtype == torch.float32
    want = torch.float16 if wl.dtype == "f16" else torch.float32
    assert p.F.dtype == want and p.M.dtype == want
    assert p.f_range[1] > p.f_range[0] and p.m_range[1] > p.m_range[0]
    # max displacement in voxels matches the recipe
    n = torch.tensor([shape[2] - 1, shape[1] - 1, shape[0] - 1], dtype=torch.float32) / 2
    vox = (p.u * n).norm(dim=-1).max().item()
    assert abs(vox - wl.eval_disp_vox) < 1e-3 * wl.eval_disp_vox
    q = synth.make_pair(k, device="cpu", shape=shape)
    assert torch.equal(p.F, q.F) and torch.equal(p.M, q.M) and torch.equal(p.u, q.u)
    assert np.array_equal(p.A, q.A)


def test_phantom_has_three_tissues_and_background():
    p = synth.make_pair(2, device="cpu", shape=(40, 48, 56))
    F = p.F.numpy()
    assert F.min() == pytest.approx(0.0, abs=1e-6)
    assert F.max() == pytest.approx(0.85, abs=0.02)
    for v in (0.25, 0.55):
        assert np.mean(np.abs(F - v) < 0.01) > 0.01
