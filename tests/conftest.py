import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def compiled_config_count():
    """Number of tile configurations in the library, read from the config
    list in the sources (so collecting tests never needs the library)."""
    import re
    text = open(os.path.join(ROOT, "dense_fp32_gemm_gb300", "csrc", "configs.inc")).read()
    block = text[text.index("#define SGEMM_GB300_CONFIGS(X)"):]
    return len(re.findall(r"^\s*X\(", block, flags=re.M))


def pytest_sessionstart(session):
    """Build the CUDA library and the oracle if they are missing (nvcc
    cross-compiles without a GPU)."""
    from dense_fp32_gemm_gb300 import build as cuda_build
    if not os.path.exists(cuda_build.LIB_PATH):
        cuda_build.build()
