"""The C-ABI library loads without a GPU and exports every function the
public header declares; pure host entry points work on the CPU."""
import ctypes
import os
import re

from dense_fp32_gemm_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names.update(re.findall(r"\b(sgemm\w*)\s*\(", text))
    return names


def test_header_declares_the_boundary():
    names = declared_functions()
    assert "sgemm" in names and "sgemm_poll_device_status" in names
    assert len(names) >= 10


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(binding.library_path())
    missing = [n for n in sorted(declared_functions()) if not hasattr(lib, n)]
    assert missing == []


def test_status_strings():
    for code in range(0, -12, -1):
        assert binding.sgemm_status_string(code) not in ("", "unknown status")
    assert binding.sgemm_status_string(12345) == "unknown status"


def test_validation_happens_before_any_device_call():
    # runs on a machine without a GPU: the argument checks return first
    assert binding.sgemm(-1, 4, 4, 1.0, 16, 4, 16, 4, 0.0, 16, 4, None) == binding.SGEMM_ERR_INVALID_DIM
    assert binding.sgemm(4, 4, 4, 1.0, 16, 3, 16, 4, 0.0, 16, 4, None) == binding.SGEMM_ERR_INVALID_LD
    assert binding.sgemm(4, 4, 4, 1.0, 16, 4, 16, 4, 0.0, 0, 4, None) == binding.SGEMM_ERR_NULL_PTR
    assert binding.sgemm(4, 4, 4, 1.0, 18, 4, 16, 4, 0.0, 16, 4, None) == binding.SGEMM_ERR_MISALIGNED
    assert binding.sgemm(0, 4, 4, 1.0, 0, 4, 0, 4, 0.0, 0, 4, None) == binding.SGEMM_OK
    T = binding.SGEMM_OP_T
    assert binding.sgemm_ex(T, 0, 8, 4, 4, 1.0, 16, 4, 16, 4, 0.0, 16, 4, None) == binding.SGEMM_ERR_INVALID_LD
    assert binding.sgemm_ex(0, T, 4, 8, 6, 1.0, 16, 6, 16, 5, 0.0, 16, 8, None) == binding.SGEMM_ERR_INVALID_LD
    assert binding.sgemm_ex(3, 0, 4, 4, 4, 1.0, 16, 4, 16, 4, 0.0, 16, 4, None) == binding.SGEMM_ERR_INVALID_VALUE
    assert binding.sgemm_strided_batched(0, 0, 4, 4, 4, 1.0, 16, 4, 16, 16, 4, 16, 0.0, 16, 4, 16, -1,
                                         None) == binding.SGEMM_ERR_INVALID_DIM
    assert binding.sgemm_strided_batched(0, 0, 4, 4, 4, 1.0, 16, 4, 16, 16, 4, 16, 0.0, 16, 4, 16, 0,
                                         None) == binding.SGEMM_OK
    for k in binding.LADDER_KERNELS:
        assert binding.sgemm_ladder(k, 4, -4, 4, 1.0, 16, 4, 16, 4, 0.0, 16, 4, None) == binding.SGEMM_ERR_INVALID_DIM
        assert binding.sgemm_ladder(k, 4, 4, 4, 1.0, 16, 4, 16, 3, 0.0, 16, 4, None) == binding.SGEMM_ERR_INVALID_LD
        assert binding.sgemm_ladder(k, 4, 4, 4, 1.0, 16, 4, 16, 4, 0.0, 17, 4, None) == binding.SGEMM_ERR_MISALIGNED
        assert binding.sgemm_ladder(k, 0, 4, 4, 1.0, 0, 4, 0, 4, 0.0, 0, 4, None) == binding.SGEMM_OK
    for form in (0, 3, 4):
        assert binding.sgemm_3xtf32_set_kernel_form(form) == binding.SGEMM_ERR_INVALID_VALUE
    assert binding.sgemm_3xtf32_set_kernel_form(binding.SGEMM_X3_SINGLE) == binding.SGEMM_X3_PAIR
    assert binding.sgemm_3xtf32_set_kernel_form(binding.SGEMM_X3_PAIR) == binding.SGEMM_X3_SINGLE
    assert binding.sgemm_host_set_pipeline(-1, 0, 0, 0) == binding.SGEMM_ERR_INVALID_VALUE
    assert binding.sgemm_host_set_pipeline(0, 0, 0, 9) == binding.SGEMM_ERR_INVALID_VALUE
    for bad in (-1, 3):
        assert binding.sgemm_set_staged_a(bad) == binding.SGEMM_ERR_INVALID_VALUE
    assert binding.sgemm_set_staged_a(1) == 1
    for k in (0, 1, 6, 9):
        assert binding.sgemm_ladder(k, 4, 4, 4, 1.0, 16, 4, 16, 4, 0.0, 16, 4, None) == binding.SGEMM_ERR_INVALID_VALUE


def test_config_registry():
    n = binding.sgemm_config_count()
    assert n >= 4
    names = set()
    for i in range(n):
        name, params = binding.sgemm_config_info(i)
        names.add(name)
        assert binding.sgemm_cfg_check(params)[0] == 0, name
    assert len(names) == n
    assert binding.sgemm_force_config(n) == binding.SGEMM_ERR_INVALID_VALUE
    assert binding.sgemm_force_config(-1) == 0


def test_tf32_rate_probe_rejects_bad_arguments():
    # checked on the host before any device call
    assert binding.sgemm_diag_tf32_mma_rate(0)[0] == binding.SGEMM_ERR_INVALID_VALUE
    assert binding.sgemm_diag_tf32_pair_mma_rate(0)[0] == binding.SGEMM_ERR_INVALID_VALUE
