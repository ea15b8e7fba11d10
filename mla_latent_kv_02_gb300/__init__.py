"""GB300-native absorbed paged MLA decode.

The compute path is the C-ABI library ``_lib/libmla.so`` (CUDA kernels for
sm_103a); :mod:`.api` is its Python binding.  :mod:`.workloads` draws the
seeded synthetic inputs.
"""
from . import workloads  # noqa: F401

__all__ = ["api", "workloads"]
