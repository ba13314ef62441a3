"""Host-side checks of the C ABI library: it builds, loads, exports every declared
entry point, and rejects bad arguments before touching a GPU."""
import ctypes
import os
import re

import pytest

from ragged_matmul_gb300 import binding
from ragged_matmul_gb300 import build as gbuild


def declared_functions():
    names = set()
    for f in os.listdir(gbuild.INCLUDE_DIR):
        if f.endswith(".h"):
            text = re.sub(r"/\*.*?\*/", "", open(os.path.join(gbuild.INCLUDE_DIR, f)).read(), flags=re.S)
            names |= set(re.findall(r"^\s*(?:const\s+)?\w[\w\s\*]*?\b(gmm_\w+)\s*\(", text, flags=re.M))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    return binding.load_library(gbuild.build())


def test_header_declares_the_boundary():
    assert declared_functions() == sorted(binding.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_error_strings(lib):
    for code in range(-6, 1):
        s = binding.gmm_error_string(code)
        assert s and s != "unknown error code"
    assert binding.gmm_error_string(12345) == "unknown error code"


def test_null_handle_and_bad_arguments_are_rejected_on_the_host(lib):
    P = ctypes.c_void_p
    assert lib.gmm_run(None, P(16), P(16), P(16), P(16), P(16), P(16), 1, 64, 64, None) == binding.GMM_ERR_INVALID_ARG
    assert lib.gmm_run_int4(None, P(16), P(16), P(16), P(16), P(16), P(16), P(16), 1, 64, 128, 128, None) \
        == binding.GMM_ERR_INVALID_ARG
    assert lib.gmm_query_status(None, None) == binding.GMM_ERR_INVALID_ARG
    assert lib.gmm_destroy(None) == binding.GMM_OK
    out = P()
    assert lib.gmm_create(None, 4, 0) == binding.GMM_ERR_INVALID_ARG
    assert lib.gmm_create(ctypes.byref(out), 0, 0) == binding.GMM_ERR_INVALID_ARG


def test_create_without_a_gpu_reports_no_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    out = ctypes.c_void_p()
    assert lib.gmm_create(ctypes.byref(out), 4, 0) == binding.GMM_ERR_NO_DEVICE
    assert not out.value


def test_product_package_does_not_reach_the_oracle():
    """The CUDA path and the oracle share nothing: no import of oracle/ in the package."""
    pkg = gbuild.PKG_DIR
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, flags=re.M), f
                assert "oracle.c" not in text and "liboracle" not in text, f


def test_dense_int4_rejects_operands_of_another_rank():
    """gmm_matmul_int4 raises for non-rank-2 operands (as the dense quantised GEMM's page
    says its function does), before touching the library or a device."""
    import torch
    from ragged_matmul_gb300 import binding
    a = torch.zeros(4, 64, dtype=torch.bfloat16)
    c = torch.zeros(4, 16, dtype=torch.bfloat16)
    q = torch.zeros(16, 8, dtype=torch.int32)
    s = torch.zeros(16, 1, dtype=torch.bfloat16)
    for bad in ("a", "c", "q", "s"):
        args = {"a": a, "c": c, "q": q, "s": s}
        args[bad] = args[bad].unsqueeze(0)
        with pytest.raises(ValueError, match="rank-2"):
            binding.gmm_matmul_int4(None, args["c"], args["a"], args["q"], args["s"], group_size=64)
