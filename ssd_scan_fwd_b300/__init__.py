"""B300-native SSD selective-scan forward pass.

The compute lives in ``libssd_scan_fwd.so`` (CUDA for sm_103a, C ABI in
``include/ssd.h``); this package is its Python binding.  Importing the package
does not load the library; the first call does, and fails loudly if it has
not been built.
"""
from .api import (chunk_cumsum, chunk_scan, chunk_state, make_args, make_step_args,  # noqa: F401
                  ssd_bwd, ssd_fwd, ssd_fwd_ex, ssd_fwd_host, ssd_fwd_mimo, ssd_fwd_rot, ssd_step,
                  state_passing,
                  workspace_size)
from ._lib import SsdError  # noqa: F401
