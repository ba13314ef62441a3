"""Edge cases that full-size workloads can reach, each against the oracle:

- the 4-bit dequantisation's rounding, bit for bit: one-hot rows of A select single
  weights w = bf16((q - 8) * s) with random bf16 scales, so C holds w itself;
- the fused activations with accumulators of magnitude 100 to 300 of both signs, where
  silu's e^-y overflows (its limit, 0, must come out) and the tanh form of GELU
  saturates, on the bf16 and both e4m3 kernels;
- a guard region after C: nothing is written past C's last row, for the bf16, 4-bit,
  e4m3 (one scale over K) and per-K-block e4m3 kernels;
- the device-timeout path (Modular "multistage_gemm_q", section "Raises": errors are
  reported, here through gmm_query_status): a test hook makes one stage never fill, the
  kernel's waits give up after a shortened limit, the call reports
  GMM_ERR_DEVICE_TIMEOUT promptly, and the next call on the same handle is correct.
"""
import os
import time

import numpy as np
import pytest

import oracle
from ragged_matmul_gb300 import binding
from ragged_matmul_gb300 import workloads as wl

from gpu_util import (VARIANTS, assert_close, bits_of, check_against_oracle, check_fp8_against_oracle, handle,
                      live_row_mask, to_dev_f32, to_dev_i32, to_dev_u16, to_dev_u8)

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _need_gpu():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


# ---------------------------------------------------------------- 4-bit rounding, bit for bit

@pytest.mark.parametrize("variant", VARIANTS)
def test_int4_one_hot_rows_random_scales_bit_exact(variant):
    """Row r of A is e_k(r): C[r, n] = sum_k A[r, k] w[e, n, k] = w[e, n, k(r)] exactly (one
    product, exact in fp32), so C must equal the oracle's bf16((q - 8) * s) bit for bit.
    The k(r) cover every nibble position of a word and several scale groups; the scales
    are random bf16 values of both binades around the workloads' range."""
    _need_gpu()
    E, N, K, gs = 3, 256, 512, 64
    loads, ids = [40, 0, 64, 25], [2, 1, 0, 2]
    r = wl.make_routing("oh", E, N, K, loads, ids, a_dist=("normal", 1.0), b_dist=None, int4=True, group_size=gs,
                        scale_range=(0.003, 0.05))
    v = wl.host_values(r, 41)
    rng = np.random.default_rng(42)
    ks = rng.integers(0, K, r.rows)
    ks[:16] = np.arange(16) * 33 % K          # every position k % 8, and spread over the scale groups
    a = np.zeros((r.rows, K), np.uint16)
    a[np.arange(r.rows), ks] = 0x3F80        # bf16 1.0
    v["a"] = a
    # scales: random bf16 bit patterns in [0.003, 0.05] (full 8-bit mantissas)
    v["scales"] = wl._to_bf16_bits(rng.uniform(0.003, 0.05, v["scales"].shape).astype(np.float32))
    got, ref, status, _ = check_against_oracle(handle(E, variant), r, v, exact=True, where=f"int4 one-hot {variant}")
    assert status == binding.GMM_OK
    # and the oracle's values are the dequantised weights themselves
    w = [oracle.dequant_int4(v["packed"][e], v["scales"][e], gs) for e in range(E)]
    live = live_row_mask(r.rows, r.a_offsets, r.expert_ids, E)
    exp = np.zeros((r.rows, N), np.uint16)
    for g, e in enumerate(ids):
        lo, hi = int(r.a_offsets[g]), int(r.a_offsets[g + 1])
        exp[lo:hi] = w[e][:, ks[lo:hi]].T
    assert np.array_equal(got[live], exp[live])


# ---------------------------------------------------------------- activations at large |acc|

def _large_acc_case(E, N, K, seed):
    """A[r, k] = 1 for k < m_r (m_r in 100 .. 300), else 0; B[e, n, k] = +1 for even n and
    -1 for odd n: acc[r, n] = +-m_r exactly."""
    loads, ids = [7, 33, 0, 24], [1, 0, 2, 1]
    r = wl.make_routing("big", E, N, K, loads, ids)
    rng = np.random.default_rng(seed)
    m = rng.integers(100, 301, r.rows)
    a = (np.arange(K)[None, :] < m[:, None]).astype(np.float32)
    b = np.where(np.arange(N)[None, :, None] % 2 == 0, 1.0, -1.0) * np.ones((E, N, K), np.float32)
    bias = rng.normal(0.0, 0.5, (E, N)).astype(np.float32)
    return r, a, b, bias


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("activation", ["silu", "gelu_tanh", "relu"])
def test_activations_with_large_accumulators_bf16(activation, variant):
    _need_gpu()
    E, N, K = 3, 136, 320
    r, a, b, bias = _large_acc_case(E, N, K, 43)
    v = {"a": wl._to_bf16_bits(a), "b": wl._to_bf16_bits(b)}
    epi = {"bias_bits": wl._to_bf16_bits(bias), "row_scale": None, "activation": activation}
    _, _, status, _ = check_against_oracle(handle(E, variant), r, v, epilogue=epi,
                                           where=f"bf16 {activation} large |acc| {variant}")
    assert status == binding.GMM_OK


@pytest.mark.parametrize("gran", [(1, 128, None), (1, 128, 128)])
@pytest.mark.parametrize("activation", ["silu", "gelu_tanh"])
def test_activations_with_large_accumulators_e4m3(activation, gran):
    _need_gpu()
    E, N, K = 3, 256, 384
    r, a, b, bias = _large_acc_case(E, N, K, 44)
    s_in, s_w = wl.fp8_scale_shapes(r.rows, E, N, K, gran)
    v = {"a8": wl._to_e4m3_bits(a), "w8": wl._to_e4m3_bits(b),
         "input_scale": np.ones(s_in, np.float32), "weight_scale": np.ones(s_w, np.float32)}
    epi = {"bias_bits": wl._to_bf16_bits(bias), "row_scale": None, "activation": activation}
    _, _, status, _ = check_fp8_against_oracle(handle(E), r, v, gran, epilogue=epi,
                                               where=f"e4m3 {gran} {activation} large |acc|")
    assert status == binding.GMM_OK


# ---------------------------------------------------------------- guard region after C

GUARD = 4096   # bf16 elements of sentinel after C's last row


def _guarded_c(rows, N):
    import torch
    big = torch.full((rows * N + GUARD,), wl.SENTINEL_BF16, dtype=torch.int16, device=DEV)
    return big, big[: rows * N].view(torch.bfloat16).view(rows, N)


def _check_guard(big, rows, N, where):
    tail = big[rows * N:].cpu().numpy().view(np.uint16)
    assert np.all(tail == wl.SENTINEL_BF16), f"{where}: {int((tail != wl.SENTINEL_BF16).sum())} guard elements written"


@pytest.mark.parametrize("variant", VARIANTS)
def test_nothing_written_past_c(variant):
    """C is a view at the front of a larger sentinel buffer; the last group ends at C's
    last row and N is a tail width (not a multiple of 128 or 256)."""
    _need_gpu()
    import torch
    E, N, K = 4, 264, 512
    loads, ids = [5, 130, 0, 61], [3, 0, 1, 2]
    r = wl.make_routing("g", E, N, K, loads, ids, a_dist=("normal", 1.0), b_dist=("normal", 1.0))
    h = handle(E, variant)
    off, ids_d = to_dev_i32(r.a_offsets, DEV), to_dev_i32(r.expert_ids, DEV)
    st = to_dev_i32(np.zeros(4, np.uint32), DEV)
    live = live_row_mask(r.rows, r.a_offsets, r.expert_ids, E)

    # bf16
    v = wl.host_values(r, 45)
    big, c = _guarded_c(r.rows, N)
    binding.gmm_run(h, c, to_dev_u16(v["a"], DEV), off, to_dev_u16(v["b"], DEV), ids_d, st)
    assert binding.gmm_query_status(h) == binding.GMM_OK
    ref = oracle.gmm_bf16(v["a"], r.a_offsets, v["b"], r.expert_ids)
    assert_close(bits_of(c), ref.ref32, live, where="guard bf16")
    _check_guard(big, r.rows, N, f"bf16 {variant}")

    # 4-bit
    r4 = wl.make_routing("g4", E, N, K, loads, ids, a_dist=("normal", 1.0), b_dist=None, int4=True, group_size=128)
    v4 = wl.host_values(r4, 46)
    big, c = _guarded_c(r4.rows, N)
    binding.gmm_run_int4(h, c, to_dev_u16(v4["a"], DEV), off,
                         torch.from_numpy(np.ascontiguousarray(v4["packed"]).view(np.int32)).to(DEV),
                         to_dev_u16(v4["scales"], DEV), ids_d, st, group_size=128)
    assert binding.gmm_query_status(h) == binding.GMM_OK
    ref = oracle.gmm_int4(v4["a"], r4.a_offsets, v4["packed"], v4["scales"], r4.expert_ids, group_size=128)
    assert_close(bits_of(c), ref.ref32, live, where="guard 4-bit")
    _check_guard(big, r4.rows, N, f"4-bit {variant}")

    # e4m3, one scale over K and per-K-block scales
    for gran in ((1, 128, None), (1, 32, 128)):
        v8 = wl.fp8_host_values(r, 47, gran)
        big, c = _guarded_c(r.rows, N)
        binding.gmm_run_fp8(h, c, to_dev_u8(v8["a8"], DEV), off, to_dev_u8(v8["w8"], DEV), ids_d, st,
                            to_dev_f32(v8["input_scale"], DEV), to_dev_f32(v8["weight_scale"], DEV), gran)
        assert binding.gmm_query_status(h) == binding.GMM_OK
        gk = K if gran[2] is None else gran[2]
        ref = oracle.gmm_fp8(v8["a8"], r.a_offsets, v8["w8"], r.expert_ids, v8["input_scale"], v8["weight_scale"],
                             (gran[0], gran[1], gk))
        assert_close(bits_of(c), ref.ref32, live, where=f"guard e4m3 {gran}")
        _check_guard(big, r.rows, N, f"e4m3 {gran} {variant}")


# ---------------------------------------------------------------- device timeout

def test_device_timeout_is_reported_promptly_and_the_handle_recovers():
    """GMM_TEST_WAIT_LIMIT_NS shortens every pipeline wait to 5 ms and GMM_TEST_STALL_STAGE
    makes the one-CTA bf16 kernel's producer skip its second stage (no copy, no arrival):
    that stage never fills, the MMA warp's wait gives up, every role stops, copies already
    issued land, and gmm_query_status reports GMM_ERR_DEVICE_TIMEOUT.  The same handle then
    computes the next call correctly."""
    _need_gpu()
    import torch
    E, N, K = 2, 256, 512
    r = wl.make_routing("to", E, N, K, [64, 40], [1, 0], a_dist=("normal", 1.0), b_dist=("normal", 1.0))
    v = wl.host_values(r, 48)
    h = handle(E, "single")
    os.environ["GMM_TEST_WAIT_LIMIT_NS"] = "5000000"
    os.environ["GMM_TEST_STALL_STAGE"] = "1"
    try:
        a, b = to_dev_u16(v["a"], DEV), to_dev_u16(v["b"], DEV)
        off, ids = to_dev_i32(r.a_offsets, DEV), to_dev_i32(r.expert_ids, DEV)
        c = torch.zeros((r.rows, N), dtype=torch.bfloat16, device=DEV)
        st = to_dev_i32(np.zeros(4, np.uint32), DEV)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        binding.gmm_run(h, c, a, off, b, ids, st)
        status = binding.gmm_query_status(h)
        dt = time.perf_counter() - t0
    finally:
        del os.environ["GMM_TEST_WAIT_LIMIT_NS"]
        del os.environ["GMM_TEST_STALL_STAGE"]
    assert status == binding.GMM_ERR_DEVICE_TIMEOUT, binding.gmm_error_string(status)
    assert dt < 1.0, f"the timeout took {dt:.3f} s to surface"
    # the next call on the same handle, without the hooks
    _, _, status, _ = check_against_oracle(h, r, v, where="after a timeout")
    assert status == binding.GMM_OK
