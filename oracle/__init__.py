"""CPU oracle for absorbed paged MLA decode (test infrastructure only).

Importable only by the tests, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py``.  Plain NumPy float64; shares no code with the CUDA path.
"""
from .mla_oracle import *  # noqa: F401,F403
from . import mla_oracle  # noqa: F401
from . import fp8_cache  # noqa: F401,E402
from . import nvfp4_cache  # noqa: F401,E402
