"""The allocation-free entry point, gmm_run_noalloc, called through the C ABI.

It exists for callers that cannot call cudaMalloc when they run the GEMM (code
inside an allocator callback, a framework owning all device memory, a runtime
that forbids allocations after start-up), so it takes its scratch from a fixed
array inside the library.  This file is collected last so that a run stopping at
the first failure has already run every other test.  On two calls in a row with
different problems it checks the output against the oracle (and against what
gmm_run produces on the same inputs) within the tolerance the other tests use,
and that the device's free memory does not change across the two calls.
"""
import ctypes

import numpy as np
import pytest

import oracle
from ragged_matmul_gb300 import binding
from ragged_matmul_gb300 import workloads as wl

from gpu_util import ATOL, RTOL, assert_close, bits_of, f32_of_bits, live_row_mask, sentinel_dev, to_dev_i32, \
    to_dev_u16

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _problem(seed, E, N, K, loads, ids):
    r = wl.make_routing("na", E, N, K, loads, ids, a_dist=("normal", 1.0), b_dist=("normal", 1.0))
    v = wl.host_values(r, seed)
    t = {"a": to_dev_u16(v["a"], DEV), "b": to_dev_u16(v["b"], DEV),
         "off": to_dev_i32(r.a_offsets, DEV), "ids": to_dev_i32(r.expert_ids, DEV),
         "c": sentinel_dev(r.rows, r.N, DEV), "stats": to_dev_i32(np.full(4, 0xFFFFFFFF, np.uint32), DEV)}
    return r, v, t


def _noalloc(lib, r, t, stream):
    """One call into the library; every buffer it touches is allocated beforehand."""
    P = ctypes.c_void_p
    return lib.gmm_run_noalloc(P(t["c"].data_ptr()), P(t["a"].data_ptr()), P(t["off"].data_ptr()),
                               P(t["b"].data_ptr()), P(t["ids"].data_ptr()), P(t["stats"].data_ptr()), r.E, r.G,
                               r.N, r.K, P(stream.cuda_stream))


def _with_handle(r, t, stream):
    h = binding.gmm_create(r.E, 0)
    c = sentinel_dev(r.rows, r.N, DEV)
    stats = to_dev_i32(np.full(4, 0xFFFFFFFF, np.uint32), DEV)
    binding.gmm_run(h, c, t["a"], t["off"], t["b"], t["ids"], stats, stream=stream)
    assert binding.gmm_query_status(h, stream) == binding.GMM_OK
    binding.gmm_destroy(h)
    return c, stats


def test_noalloc_matches_oracle_on_two_calls_in_a_row_without_allocating():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from ragged_matmul_gb300 import build
    lib = binding.load_library(build.build())
    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream(0)
    problems = [
        _problem(21, 6, 384, 320, [1, 130, 0, 257, 16, 40, 300], [5, 0, 1, -1, 3, 2, 4]),
        _problem(22, 3, 256, 1096, [513, 7, 64], [2, -1, 0]),
    ]
    # A first call on a small problem of its own does the one-time set-up on this device
    # (and loads the library's module there, if no earlier call did).
    rw, _, warm = _problem(23, 2, 64, 64, [5, 11], [1, 0])
    assert _noalloc(lib, rw, warm, stream) == binding.GMM_OK
    torch.cuda.synchronize()

    free0, _ = torch.cuda.mem_get_info(0)
    rcs = [_noalloc(lib, r, t, stream) for r, _, t in problems]      # two calls in a row
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info(0)
    assert rcs == [binding.GMM_OK, binding.GMM_OK], [binding.gmm_error_string(x) for x in rcs]
    assert free1 == free0, f"device free memory changed by {free0 - free1} bytes across the two calls"

    for r, v, t in problems:
        ref = oracle.gmm_bf16(v["a"], r.a_offsets, v["b"], r.expert_ids, c_init=wl.sentinel_c(r.rows, r.N),
                              stats_init=np.full(4, wl.SENTINEL_STATS, np.uint32))
        got = bits_of(t["c"])
        live = live_row_mask(r.rows, r.a_offsets, r.expert_ids, r.E)
        assert np.array_equal(got[~live], ref.c[~live])               # untouched rows stay untouched
        assert_close(got, ref.ref32, live, where="gmm_run_noalloc against the oracle")
        assert np.array_equal(t["stats"].cpu().numpy().view(np.uint32), ref.stats)
        # and against the handle-based entry point on the same inputs
        c_ref, st_ref = _with_handle(r, t, stream)
        w = f32_of_bits(bits_of(c_ref)[live]).astype(np.float64)
        g = f32_of_bits(got[live]).astype(np.float64)
        assert np.all(np.abs(g - w) <= ATOL + RTOL * np.abs(w))
        assert np.array_equal(t["stats"].cpu().numpy(), st_ref.cpu().numpy())


def test_noalloc_rejects_bad_arguments_before_launch():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = binding.load_library()
    P = ctypes.c_void_p
    a = torch.zeros((16, 64), dtype=torch.bfloat16, device=DEV)
    b = torch.zeros((2, 64, 64), dtype=torch.bfloat16, device=DEV)
    c = torch.zeros((16, 64), dtype=torch.bfloat16, device=DEV)
    off = to_dev_i32([0, 16], DEV)
    ids = to_dev_i32([0], DEV)
    st = to_dev_i32([0, 0], DEV)
    args = [P(c.data_ptr()), P(a.data_ptr()), P(off.data_ptr()), P(b.data_ptr()), P(ids.data_ptr()),
            P(st.data_ptr())]
    assert lib.gmm_run_noalloc(*args, 0, 1, 64, 64, None) == binding.GMM_ERR_INVALID_ARG      # no experts
    assert lib.gmm_run_noalloc(*args, 2, 1, 64, 60, None) == binding.GMM_ERR_INVALID_ARG      # K % 8
    assert lib.gmm_run_noalloc(*args, 2, 4097, 64, 64, None) == binding.GMM_ERR_UNSUPPORTED   # too many groups
