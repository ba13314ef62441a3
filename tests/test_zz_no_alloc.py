"""The allocation-free entry point, gmm_run_noalloc, called through the C ABI.

It exists for callers that cannot call cudaMalloc when they run the GEMM (code
inside an allocator callback, a framework owning all device memory, a runtime
that forbids allocations after start-up), so it takes its scratch from a fixed
array inside the library.  This file is collected last so that a run stopping at
the first failure has already run every other test.  It checks, on two calls in
a row with different problems, that the output equals what gmm_run produces on
the same inputs, within the tolerance the other tests use.
"""
import ctypes

import numpy as np
import pytest

from ragged_matmul_gb300 import binding
from ragged_matmul_gb300 import workloads as wl

from gpu_util import ATOL, RTOL, bits_of, f32_of_bits, live_row_mask, sentinel_dev, to_dev_i32, to_dev_u16

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _problem(seed, E, N, K, loads, ids):
    r = wl.make_routing("na", E, N, K, loads, ids, a_dist=("normal", 1.0), b_dist=("normal", 1.0))
    v = wl.host_values(r, seed)
    return r, {"a": to_dev_u16(v["a"], DEV), "b": to_dev_u16(v["b"], DEV),
               "off": to_dev_i32(r.a_offsets, DEV), "ids": to_dev_i32(r.expert_ids, DEV)}


def _noalloc(lib, r, t, stream):
    import torch
    c = sentinel_dev(r.rows, r.N, DEV)
    stats = to_dev_i32(np.full(4, 0xFFFFFFFF, np.uint32), DEV)
    P = ctypes.c_void_p
    rc = lib.gmm_run_noalloc(P(c.data_ptr()), P(t["a"].data_ptr()), P(t["off"].data_ptr()), P(t["b"].data_ptr()),
                             P(t["ids"].data_ptr()), P(stats.data_ptr()), r.E, r.G, r.N, r.K,
                             P(stream.cuda_stream))
    assert rc == binding.GMM_OK, binding.gmm_error_string(rc)
    return c, stats


def _with_handle(r, t, stream):
    h = binding.gmm_create(r.E, 0)
    c = sentinel_dev(r.rows, r.N, DEV)
    stats = to_dev_i32(np.full(4, 0xFFFFFFFF, np.uint32), DEV)
    binding.gmm_run(h, c, t["a"], t["off"], t["b"], t["ids"], stats, stream=stream)
    assert binding.gmm_query_status(h, stream) == binding.GMM_OK
    binding.gmm_destroy(h)
    return c, stats


def test_noalloc_matches_gmm_run_on_two_calls_in_a_row():
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
    outs = [_noalloc(lib, r, t, stream) for r, t in problems]        # two calls in a row
    for (r, t), (c_na, st_na) in zip(problems, outs):
        c_ref, st_ref = _with_handle(r, t, stream)
        torch.cuda.synchronize()
        got, ref = bits_of(c_na), bits_of(c_ref)
        live = live_row_mask(r.rows, r.a_offsets, r.expert_ids, r.E)
        assert np.array_equal(got[~live], ref[~live])                 # untouched rows stay untouched
        g, w = f32_of_bits(got[live]).astype(np.float64), f32_of_bits(ref[live]).astype(np.float64)
        assert np.all(np.abs(g - w) <= ATOL + RTOL * np.abs(w))
        assert np.array_equal(st_na.cpu().numpy(), st_ref.cpu().numpy())
        assert st_na.cpu().numpy().view(np.uint32)[1] == int(r.active_mask().sum())


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
