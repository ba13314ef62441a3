"""GB300 (sm_103a) ragged grouped GEMM for mixture-of-experts layers.

The compute lives in libgmm.so (hand-written CUDA, C ABI in include/gmm.h);
this package holds its ctypes binding, the in-tree build step and the seeded
workload generators.  Importing the package does not load the library; the
first call does, and raises if the library is missing.
"""
from .binding import (EXPORTED, GMM_ERR_BAD_INPUT, GMM_ERR_CUDA, GMM_ERR_DEVICE_TIMEOUT,  # noqa: F401
                      GMM_ERR_INVALID_ARG, GMM_ERR_NO_DEVICE, GMM_ERR_UNSUPPORTED, GMM_OK, GmmError,
                      GMM_ACT_GELU_TANH, GMM_ACT_NONE, GMM_ACT_RELU, GMM_ACT_SILU,
                      Handle, gmm_create, gmm_destroy, gmm_error_string, gmm_query_status, gmm_run,
                      gmm_matmul_int4, gmm_run_ex, gmm_run_fp8, gmm_run_int4, gmm_run_planes, gmm_run_int4_ex, library_path,
                      load_library)
