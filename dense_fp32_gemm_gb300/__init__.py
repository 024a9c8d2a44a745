"""GB300-native (sm_103a) single-precision GEMM: C = alpha*A*B + beta*C.

The compute path is the CUDA library built from ``csrc/`` (see
``include/sgemm_gb300.h`` for the C ABI); ``binding`` calls it through ctypes
and ``workloads`` draws the seeded synthetic inputs. Nothing here falls back
to the CPU.
"""
from . import binding  # noqa: F401  (loads the library lazily, on first call)
from .binding import SgemmError, gemm  # noqa: F401
