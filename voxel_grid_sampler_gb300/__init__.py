"""GB300-native fused registration objective of FFDP (single GPU, sm_103a).

The compute lives in libffdp (CUDA, C ABI in include/ffdp.h); ``ffdp`` is its
ctypes binding, ``synth`` makes the seeded synthetic volume pairs and
``build`` compiles the library.
"""
from . import ffdp  # noqa: F401
from .ffdp import (FfdpError, ffdp_grid_sample_bwd, ffdp_grid_sample_fwd, ffdp_lncc_fwd_bwd,  # noqa: F401
                   ffdp_mi_fwd_bwd, ffdp_objective, ffdp_workspace_bytes)
