"""Helpers for the GPU parity tests: move seeded inputs to the device, run the
CUDA path through the binding, run the oracle on the same inputs, compare.

Tolerance for floating-point outputs (per bf16 element of C):
    |gpu - ref| <= 1e-2 + 1e-2 * |ref|
with ref the oracle's fp32 sum.  Rows no active group covers and
expert_usage_stats are compared bit for bit.
"""
from __future__ import annotations

import numpy as np

import oracle
from ragged_matmul_gb300 import binding
from ragged_matmul_gb300 import workloads as wl

ATOL = 1e-2
RTOL = 1e-2


def _torch():
    import torch
    return torch


def to_dev_u16(x, dev):
    torch = _torch()
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(dev).view(torch.bfloat16)


def to_dev_i32(x, dev):
    torch = _torch()
    arr = np.ascontiguousarray(np.asarray(x).astype(np.int64).astype(np.uint32)).view(np.int32)
    return torch.from_numpy(arr).to(dev)


def bits_of(t):
    """bf16 device tensor -> host uint16 bits."""
    torch = _torch()
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def f32_of_bits(h):
    return (np.asarray(h, np.uint16).astype(np.uint32) << 16).view(np.float32)


def sentinel_dev(rows, N, dev):
    torch = _torch()
    return torch.full((rows, N), wl.SENTINEL_BF16, dtype=torch.int16, device=dev).view(torch.bfloat16)


def run_gpu(h, a_bits, off, ids, *, b_bits=None, packed=None, scales=None, group_size=128, N=None,
            rows_alloc=None, stats_init=None, epilogue=None, dev="cuda:0"):
    """Upload host inputs, run the CUDA path, return (C bits, stats, status code).
    `epilogue`: optional dict(bias_bits=[E, N] bf16 bits, row_scale=[rows] fp32, activation=name)."""
    torch = _torch()
    epi = {}
    if epilogue:
        if epilogue.get("bias_bits") is not None:
            epi["bias"] = to_dev_u16(epilogue["bias_bits"], dev)
        if epilogue.get("row_scale") is not None:
            epi["row_scale"] = torch.from_numpy(np.ascontiguousarray(epilogue["row_scale"], np.float32)).to(dev)
        epi["activation"] = epilogue.get("activation", "none")
    rows = a_bits.shape[0] if rows_alloc is None else rows_alloc
    a = to_dev_u16(a_bits, dev)
    c = sentinel_dev(rows, N, dev)
    stats = to_dev_i32(np.full(4, 0xFFFFFFFF, np.uint32) if stats_init is None else stats_init, dev)
    off_d = to_dev_i32(off, dev)
    ids_d = to_dev_i32(ids, dev)
    if packed is None:
        b = to_dev_u16(b_bits, dev)
        if epi:
            binding.gmm_run_ex(h, c, a, off_d, b, ids_d, stats, **epi)
        else:
            binding.gmm_run(h, c, a, off_d, b, ids_d, stats)
    else:
        q = torch.from_numpy(np.ascontiguousarray(packed).view(np.int32)).to(dev)
        s = to_dev_u16(scales, dev)
        if epi:
            binding.gmm_run_int4_ex(h, c, a, off_d, q, s, ids_d, stats, group_size=group_size, **epi)
        else:
            binding.gmm_run_int4(h, c, a, off_d, q, s, ids_d, stats, group_size=group_size)
    status = binding.gmm_query_status(h)
    return bits_of(c), stats.cpu().numpy().view(np.uint32), status


def assert_close(gpu_bits, ref32, live_rows, where=""):
    got = f32_of_bits(gpu_bits[live_rows]).astype(np.float64)
    ref = ref32[live_rows].astype(np.float64)
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{where}: {int(bad.sum())} of {bad.size} elements out of tolerance, e.g. "
                             + ", ".join(f"{tuple(i)} gpu={got[tuple(i)]} ref={ref[tuple(i)]}" for i in idx))
    return float(err.max()) if err.size else 0.0


def live_row_mask(rows_alloc, off, ids, E):
    live = np.zeros(rows_alloc, bool)
    off = np.asarray(off, np.int64)
    for g, e in enumerate(np.asarray(ids)):
        if 0 <= e < E:
            live[off[g]:off[g + 1]] = True
    return live


def check_against_oracle(h, r: wl.Routing, vals, *, rows_alloc=None, exact=False, epilogue=None, where=""):
    """Full-output comparison of the CUDA path with the oracle on host inputs (with the
    optional epilogue, given as in run_gpu, applied on both sides)."""
    rows_alloc = r.rows if rows_alloc is None else rows_alloc
    c0 = wl.sentinel_c(rows_alloc, r.N)
    st0 = np.full(4, wl.SENTINEL_STATS, np.uint32)
    if r.int4:
        ref = oracle.gmm_int4(vals["a"], r.a_offsets, vals["packed"], vals["scales"], r.expert_ids,
                              group_size=r.group_size, c_init=c0, stats_init=st0)
        got, stats, status = run_gpu(h, vals["a"], r.a_offsets, r.expert_ids, packed=vals["packed"],
                                     scales=vals["scales"], group_size=r.group_size, N=r.N,
                                     rows_alloc=rows_alloc, epilogue=epilogue)
    else:
        ref = oracle.gmm_bf16(vals["a"], r.a_offsets, vals["b"], r.expert_ids, c_init=c0, stats_init=st0)
        got, stats, status = run_gpu(h, vals["a"], r.a_offsets, r.expert_ids, b_bits=vals["b"], N=r.N,
                                     rows_alloc=rows_alloc, epilogue=epilogue)
    if epilogue:
        ref = oracle.apply_epilogue(ref, r.a_offsets, r.expert_ids, r.E, bias_bits=epilogue.get("bias_bits"),
                                    row_scale=epilogue.get("row_scale"),
                                    activation=epilogue.get("activation", "none"))
    live = live_row_mask(rows_alloc, r.a_offsets, r.expert_ids, r.E)
    if ref.flags & oracle.BAD_OFFSETS:
        live[:] = False
    assert np.array_equal(got[~live], ref.c[~live]), f"{where}: rows outside active groups changed"
    assert np.array_equal(stats, ref.stats), f"{where}: stats {stats} != {ref.stats}"
    if exact:
        assert np.array_equal(got[live], ref.c[live]), f"{where}: not bit-exact"
        err = 0.0
    else:
        err = assert_close(got, ref.ref32, live, where)
    return got, ref, status, err


# ---------------------------------------------------------------- block-scaled e4m3 path

def to_dev_u8(x, dev):
    torch = _torch()
    return torch.from_numpy(np.ascontiguousarray(x, np.uint8)).to(dev)


def to_dev_f32(x, dev):
    torch = _torch()
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(dev)


def run_gpu_fp8(h, vals, off, ids, granularity, *, N, rows_alloc=None, stats_init=None, epilogue=None,
                dev="cuda:0"):
    """Upload e4m3 operands and fp32 scales, run gmm_run_fp8, return (C bits, stats, status)."""
    torch = _torch()
    epi = {}
    if epilogue:
        if epilogue.get("bias_bits") is not None:
            epi["bias"] = to_dev_u16(epilogue["bias_bits"], dev)
        if epilogue.get("row_scale") is not None:
            epi["row_scale"] = to_dev_f32(epilogue["row_scale"], dev)
        epi["activation"] = epilogue.get("activation", "none")
    rows = vals["a8"].shape[0] if rows_alloc is None else rows_alloc
    c = sentinel_dev(rows, N, dev)
    stats = to_dev_i32(np.full(4, 0xFFFFFFFF, np.uint32) if stats_init is None else stats_init, dev)
    binding.gmm_run_fp8(h, c, to_dev_u8(vals["a8"], dev), to_dev_i32(off, dev), to_dev_u8(vals["w8"], dev),
                        to_dev_i32(ids, dev), stats, to_dev_f32(vals["input_scale"], dev),
                        to_dev_f32(vals["weight_scale"], dev), granularity, **epi)
    status = binding.gmm_query_status(h)
    torch.cuda.synchronize()
    return bits_of(c), stats.cpu().numpy().view(np.uint32), status


def check_fp8_against_oracle(h, r: wl.Routing, vals, granularity, *, rows_alloc=None, exact=False,
                             epilogue=None, where=""):
    """Full-output comparison of gmm_run_fp8 with the oracle (scales, then the optional
    epilogue, on both sides)."""
    rows_alloc = r.rows if rows_alloc is None else rows_alloc
    gm, gn, gk = granularity
    gran = (gm, gn, r.K if gk is None else gk)
    ref = oracle.gmm_fp8(vals["a8"], r.a_offsets, vals["w8"], r.expert_ids, vals["input_scale"],
                         vals["weight_scale"], gran, c_init=wl.sentinel_c(rows_alloc, r.N),
                         stats_init=np.full(4, wl.SENTINEL_STATS, np.uint32))
    got, stats, status = run_gpu_fp8(h, vals, r.a_offsets, r.expert_ids, granularity, N=r.N,
                                     rows_alloc=rows_alloc, epilogue=epilogue)
    if epilogue:
        ref = oracle.apply_epilogue(ref, r.a_offsets, r.expert_ids, r.E, bias_bits=epilogue.get("bias_bits"),
                                    row_scale=epilogue.get("row_scale"),
                                    activation=epilogue.get("activation", "none"))
    live = live_row_mask(rows_alloc, r.a_offsets, r.expert_ids, r.E)
    if ref.flags & oracle.BAD_OFFSETS:
        live[:] = False
    assert np.array_equal(got[~live], ref.c[~live]), f"{where}: rows outside active groups changed"
    assert np.array_equal(stats, ref.stats), f"{where}: stats {stats} != {ref.stats}"
    if exact:
        assert np.array_equal(got[live], ref.c[live]), f"{where}: not bit-exact"
        err = 0.0
    else:
        err = assert_close(got, ref.ref32, live, where)
    return got, ref, status, err


# ---------------------------------------------------------------- handles

VARIANTS = ("pair", "single")   # CTA-pair kernels (default) and one CTA per tile
_handles = {}


def handle(E, variant="pair"):
    """A handle per (E, kernel variant), shared by the test modules; the variant is fixed
    when the handle is created (GMM_VARIANT)."""
    import os
    key = (E, variant)
    if key not in _handles:
        old = os.environ.get("GMM_VARIANT")
        os.environ["GMM_VARIANT"] = variant
        try:
            _handles[key] = binding.gmm_create(E, 0)
        finally:
            if old is None:
                del os.environ["GMM_VARIANT"]
            else:
                os.environ["GMM_VARIANT"] = old
    return _handles[key]
