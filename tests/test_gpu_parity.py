"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Small and medium shapes are compared element by element; the full-size
workloads are compared on sampled rows and columns that the oracle computes,
in the same launch configuration the bench times.
"""
import numpy as np
import pytest

import oracle
from ragged_matmul_gb300 import binding
from ragged_matmul_gb300 import workloads as wl

from gpu_util import (VARIANTS, assert_close, bits_of, check_against_oracle, handle, live_row_mask, run_gpu,
                      sentinel_dev, to_dev_i32, to_dev_u16)

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from ragged_matmul_gb300 import build
    build.build()
    torch.cuda.set_device(0)


def routing(E, N, K, loads, ids, dist=("uniform", -1.0, 1.0), base=0, int4=False, gs=128):
    return wl.make_routing("t", E, N, K, loads, ids, a_dist=dist, b_dist=None if int4 else dist,
                           base=base, int4=int4, group_size=gs)


# ---------------------------------------------------------------- named tiny workload

@pytest.mark.parametrize("variant", VARIANTS)
def test_tiny_workload(variant):
    r = wl.routing("tiny")
    v = wl.host_values(r, 0)
    _, _, status, _ = check_against_oracle(handle(r.E, variant), r, v, where="tiny")
    assert status == binding.GMM_OK


# ---------------------------------------------------------------- exact arithmetic

@pytest.mark.parametrize("variant", VARIANTS)
def test_small_integers_bit_exact(variant):
    """Integer operands in [-3, 3], K <= 28: every sum is exact, so C must match bit for bit."""
    r = routing(5, 392, 24, [1, 17, 0, 130, 33, 256, 7, 300], [4, 0, 2, 3, -1, 1, 4, 2], dist=("int", -3, 3))
    v = wl.host_values(r, 1)
    check_against_oracle(handle(5, variant), r, v, exact=True, where="int")


@pytest.mark.parametrize("variant", VARIANTS)
def test_unit_rows_select_weight_columns(variant):
    """A rows that are unit vectors e_k return B[e, n, k] exactly: pins operand orientation."""
    E, N, K = 3, 256, 64
    rng = np.random.default_rng(2)
    b = wl._to_bf16_bits(rng.uniform(-2, 2, (E, N, K)).astype(np.float32))
    A = np.zeros((3 * K, K), np.float32)
    for g in range(3):
        A[g * K + np.arange(K), np.arange(K)] = 1.0
    ids = [2, 0, 1]
    off = wl.offsets_from_loads([K, K, K])
    got, stats, status = run_gpu(handle(E, variant), wl._to_bf16_bits(A), off, ids, b_bits=b, N=N)
    for g in range(3):
        for k in range(K):
            assert np.array_equal(got[g * K + k], b[ids[g], :, k]), (g, k)
    assert stats[1] == 3 and status == binding.GMM_OK


# ---------------------------------------------------------------- ragged shapes and tails

@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("N,K", [(384, 320), (136, 200), (256, 64), (1024, 1096), (648, 512)])
def test_ragged_groups_tails(N, K, variant):
    loads = [1, 15, 16, 17, 31, 32, 33, 127, 128, 129, 255, 256, 257, 300, 513, 0, 2]
    ids = [3, 0, 5, 1, 7, 2, 6, 4, 3, 0, 1, 2, 6, 7, 5, 1, 4]
    r = routing(8, N, K, loads, ids, dist=("normal", 1.0))
    v = wl.host_values(r, 3)
    _, _, status, _ = check_against_oracle(handle(8, variant), r, v, where=f"ragged N={N} K={K} {variant}")
    assert status == binding.GMM_OK


def test_single_group_dense():
    r = routing(2, 512, 512, [700], [1], dist=("normal", 1.0))
    v = wl.host_values(r, 4)
    check_against_oracle(handle(2), r, v, where="single group")


def test_offset_base_and_trailing_rows_untouched():
    """a_offsets[0] > 0 and rows after a_offsets[G]: both stay untouched."""
    r = routing(4, 128, 128, [40, 9, 100], [1, -1, 3], base=37)
    rows_alloc = r.rows + 21
    v = wl.host_values(r, 5, rows=rows_alloc)
    check_against_oracle(handle(4), r, v, rows_alloc=rows_alloc, where="offset base")


def test_skipped_groups_with_rows_and_duplicates():
    r = routing(4, 256, 192, [50, 300, 20, 64, 64], [-1, 2, -5, 2, 0])
    v = wl.host_values(r, 6)
    _, _, status, _ = check_against_oracle(handle(4), r, v, where="skips")
    assert status == binding.GMM_OK


def test_all_groups_skipped_and_empty_problem():
    r = routing(4, 128, 64, [30, 40], [-1, -1])
    v = wl.host_values(r, 7)
    check_against_oracle(handle(4), r, v, where="all skipped")
    r0 = routing(4, 128, 64, [], [])
    got, stats, status = run_gpu(handle(4), np.zeros((16, 64), np.uint16), r0.a_offsets, r0.expert_ids,
                                 b_bits=np.zeros((4, 128, 64), np.uint16), N=128)
    assert stats.tolist() == [0xFFFFFFFF, 0, 0xFFFFFFFF, 0xFFFFFFFF]
    assert np.all(got == wl.SENTINEL_BF16) and status == binding.GMM_OK


def test_bad_offsets_compute_nothing_and_report():
    r = routing(4, 128, 64, [30, 40, 10], [0, 1, 2])
    v = wl.host_values(r, 8)
    off = np.array([0, 30, 20, 80], np.uint32)       # decreasing at g = 1
    got, stats, status = run_gpu(handle(4), v["a"], off, r.expert_ids, b_bits=v["b"], N=128, rows_alloc=80)
    ref = oracle.gmm_bf16(v["a"], off, v["b"], r.expert_ids, c_init=wl.sentinel_c(80, 128),
                          stats_init=np.full(4, 0xFFFFFFFF, np.uint32))
    assert ref.flags & oracle.BAD_OFFSETS
    assert np.array_equal(got, ref.c) and np.array_equal(stats, ref.stats)
    assert status == binding.GMM_ERR_BAD_INPUT
    assert binding.gmm_query_status(handle(4)) == binding.GMM_OK    # the query cleared it


def test_expert_id_out_of_range_is_skipped_and_reported():
    r = routing(4, 128, 64, [30, 40, 10], [0, 9, 2])
    v = wl.host_values(r, 9)
    _, ref, status, _ = check_against_oracle(handle(4), r, v, where="bad id")
    assert ref.flags == oracle.BAD_EXPERT_ID
    assert status == binding.GMM_ERR_BAD_INPUT


# ---------------------------------------------------------------- invariants

@pytest.mark.parametrize("variant", VARIANTS)
def test_group_permutation_and_determinism(variant):
    loads = [300, 7, 129, 0, 64, 511]
    ids = [1, 0, 3, 2, -1, 1]
    r = routing(4, 640, 256, loads, ids, dist=("normal", 1.0))
    v = wl.host_values(r, 10)
    h = handle(4, variant)
    base, _, _ = run_gpu(h, v["a"], r.a_offsets, r.expert_ids, b_bits=v["b"], N=r.N)
    again, _, _ = run_gpu(h, v["a"], r.a_offsets, r.expert_ids, b_bits=v["b"], N=r.N)
    assert np.array_equal(base, again), "repeated runs differ"
    perm = np.random.default_rng(11).permutation(len(loads))
    off = r.a_offsets.astype(np.int64)
    row_perm = np.concatenate([np.arange(off[g], off[g + 1]) for g in perm]).astype(np.int64)
    got, _, _ = run_gpu(h, v["a"][row_perm], wl.offsets_from_loads(np.asarray(loads)[perm]),
                        np.asarray(ids)[perm], b_bits=v["b"], N=r.N)
    assert np.array_equal(got, base[row_perm])


def test_argument_validation_codes():
    import torch
    h = handle(4)
    a = torch.zeros((16, 60), dtype=torch.bfloat16, device=DEV)       # K = 60: not a multiple of 8
    b = torch.zeros((4, 64, 60), dtype=torch.bfloat16, device=DEV)
    c = torch.zeros((16, 64), dtype=torch.bfloat16, device=DEV)
    off = to_dev_i32([0, 16], DEV)
    ids = to_dev_i32([0], DEV)
    st = to_dev_i32([0, 0], DEV)
    assert binding.gmm_run(h, c, a, off, b, ids, st, check=False) == binding.GMM_ERR_INVALID_ARG
    big = torch.zeros(4097, dtype=torch.int32, device=DEV)
    a = torch.zeros((16, 64), dtype=torch.bfloat16, device=DEV)
    b = torch.zeros((4, 64, 64), dtype=torch.bfloat16, device=DEV)
    offs = torch.zeros(4098, dtype=torch.int32, device=DEV)
    assert binding.gmm_run(h, c, a, offs, b, big, st, check=False) == binding.GMM_ERR_UNSUPPORTED
    q = torch.zeros((4, 64, 8), dtype=torch.int32, device=DEV)
    s = torch.zeros((4, 64, 2), dtype=torch.bfloat16, device=DEV)
    assert binding.gmm_run_int4(h, c, a, off, q, s, ids, st, group_size=32, check=False) \
        == binding.GMM_ERR_UNSUPPORTED


# ---------------------------------------------------------------- scaled-down named workloads

def _scaled(name, N, K):
    full = wl.routing(name)
    return wl.make_routing(name + "_small", full.E, N, K, full.loads, full.expert_ids, a_dist=full.a_dist,
                           b_dist=full.b_dist, int4=full.int4, group_size=full.group_size,
                           scale_range=full.scale_range)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("name,N,K", [("decode", 2816, 256), ("prefill", 512, 512),
                                      ("fine_grained", 256, 448), ("int4", 512, 512)])
def test_named_workload_routing_at_reduced_width(name, N, K, variant):
    """The full routing (all rows, all groups, skips) with N and K cut down."""
    r = _scaled(name, N, K)
    v = wl.host_values(r, 12)
    _, _, status, _ = check_against_oracle(handle(r.E, variant), r, v, where=f"{name} {variant}")
    assert status == binding.GMM_OK


# ---------------------------------------------------------------- 4-bit variant

@pytest.mark.parametrize("variant", VARIANTS)
def test_int4_integer_case_bit_exact(variant):
    rng = np.random.default_rng(13)
    E, N, K, gs = 3, 256, 256, 128
    r = routing(E, N, K, [7, 0, 130, 45], [2, 1, 0, 2], int4=True, gs=gs)
    a = wl._to_bf16_bits(rng.integers(-2, 3, (r.rows, K)).astype(np.float32))
    q = rng.integers(0, 16, (E, N, K))
    v = {"a": a, "packed": wl.pack_nibbles(q),
         "scales": wl._to_bf16_bits(np.ones((E, N, K // gs), np.float32))}
    check_against_oracle(handle(E, variant), r, v, exact=True, where="int4 exact")


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("gs", [64, 128, 256])
def test_int4_random(gs, variant):
    r = routing(6, 384, 512, [33, 0, 257, 16, 100, 1], [5, 0, 1, -1, 3, 2], dist=("normal", 1.0),
                int4=True, gs=gs)
    v = wl.host_values(r, 14)
    _, _, status, _ = check_against_oracle(handle(6, variant), r, v, where=f"int4 gs={gs} {variant}")
    assert status == binding.GMM_OK


@pytest.mark.parametrize("N,K,gs", [(136, 192, 64), (200, 320, 64), (128, 64, 64), (72, 1088, 64), (136, 576, 192)])
def test_int4_k_and_n_tails(N, K, gs):
    """K an odd multiple of 64 (the last 128-wide K stage has one half past K), N not a
    multiple of 128 (rows past N in the last weight block), and a group size that is
    not a power-of-two multiple of 64."""
    r = routing(5, N, K, [1, 17, 160, 161, 40], [4, 0, 2, 3, -1], dist=("normal", 1.0), int4=True, gs=gs)
    v = wl.host_values(r, 15)
    _, _, status, _ = check_against_oracle(handle(5), r, v, where=f"int4 tails N={N} K={K}")
    assert status == binding.GMM_OK


# ---------------------------------------------------------------- full-size sampled parity

def sampled_full_size(name, rows_per_group=2, ncols=96, seed=0):
    """Run the full named workload on the GPU; check sampled outputs against the oracle."""
    import torch
    r = wl.routing(name)
    v = wl.device_values(r, seed, device=DEV)
    h = handle(r.E)
    c = sentinel_dev(r.rows, r.N, DEV)
    stats = to_dev_i32(np.full(4, 0xFFFFFFFF, np.uint32), DEV)
    off_d, ids_d = to_dev_i32(r.a_offsets, DEV), to_dev_i32(r.expert_ids, DEV)
    if r.int4:
        binding.gmm_run_int4(h, c, v["a"], off_d, v["packed"], v["scales"], ids_d, stats, group_size=r.group_size)
    else:
        binding.gmm_run(h, c, v["a"], off_d, v["b"], ids_d, stats)
    assert binding.gmm_query_status(h) == binding.GMM_OK
    assert stats.cpu().numpy().view(np.uint32).tolist() == [0xFFFFFFFF, int(r.active_mask().sum()),
                                                            0xFFFFFFFF, 0xFFFFFFFF]
    live = live_row_mask(r.rows, r.a_offsets, r.expert_ids, r.E)
    dead = torch.from_numpy(~live).to(DEV)      # rows outside active groups: still all sentinel
    assert bool((c.view(torch.int16)[dead] == wl.SENTINEL_BF16).all())
    rng = np.random.default_rng(seed + 100)
    rows, loads = [], []
    for g in range(r.G):
        lo, hi = int(r.a_offsets[g]), int(r.a_offsets[g + 1])
        pick = sorted(set([lo, hi - 1] + rng.integers(lo, hi, rows_per_group).tolist())) if hi > lo else []
        rows += pick
        loads.append(len(pick))
    rows = np.asarray(rows, np.int64)
    cols = np.unique(np.concatenate([[0, r.N - 1], rng.choice(r.N, ncols, replace=False)]))
    rows_t = torch.from_numpy(rows).to(DEV)
    cols_t = torch.from_numpy(cols).to(DEV)
    a_s = bits_of(v["a"][rows_t])
    off_s = wl.offsets_from_loads(loads)
    if r.int4:
        q_s = v["packed"][:, cols_t, :].contiguous().cpu().numpy().view(np.uint32)
        s_s = bits_of(v["scales"][:, cols_t, :])
        ref = oracle.gmm_int4(a_s, off_s, q_s, s_s, r.expert_ids, group_size=r.group_size)
    else:
        b_s = bits_of(v["b"][:, cols_t, :])
        ref = oracle.gmm_bf16(a_s, off_s, b_s, r.expert_ids)
    got = bits_of(c[rows_t][:, cols_t])
    live_s = live_row_mask(len(rows), off_s, r.expert_ids, r.E)
    err = assert_close(got, ref.ref32, live_s, where=name)
    assert np.all(got[~live_s] == wl.SENTINEL_BF16)
    return err


@pytest.mark.parametrize("name", ["decode", "prefill", "fine_grained", "int4"])
def test_full_size_sampled(name):
    sampled_full_size(name)


# ---------------------------------------------------------------- optional epilogue

def _epilogue_case(r, seed, activation, bias=True, scale=True, rows_alloc=None):
    rng = np.random.default_rng(seed)
    rows = r.rows if rows_alloc is None else rows_alloc
    epi = {"activation": activation}
    if bias:
        epi["bias_bits"] = wl._to_bf16_bits(rng.normal(0.0, 1.0, (r.E, r.N)).astype(np.float32))
    if scale:
        epi["row_scale"] = rng.uniform(0.1, 2.0, rows).astype(np.float32)
    return epi


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("activation", ["none", "relu", "silu", "gelu_tanh"])
def test_epilogue_bf16(activation, variant):
    """act(acc + bias[e, n]) * row_scale[r] fused before the bf16 store, against the oracle."""
    loads = [1, 17, 0, 130, 33, 257, 7]
    ids = [2, 0, 1, 3, -1, 1, 0]
    r = routing(4, 392, 200, loads, ids, dist=("normal", 0.5))
    v = wl.host_values(r, 30)
    epi = _epilogue_case(r, 31, activation)
    _, _, status, _ = check_against_oracle(handle(4, variant), r, v, epilogue=epi,
                                           where=f"epilogue {activation} {variant}")
    assert status == binding.GMM_OK


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("K", [520, 1096])
def test_epilogue_bf16_long_k(K, variant):
    """The fused epilogue with K above 512, where the kernel runs 4 epilogue warps (8 below)."""
    loads = [1, 17, 0, 130, 33, 257, 7]
    ids = [2, 0, 1, 3, -1, 1, 0]
    r = routing(4, 392, K, loads, ids, dist=("normal", 0.5))
    v = wl.host_values(r, 32)
    epi = _epilogue_case(r, 33, "silu")
    _, _, status, _ = check_against_oracle(handle(4, variant), r, v, epilogue=epi,
                                           where=f"epilogue K={K} {variant}")
    assert status == binding.GMM_OK


@pytest.mark.parametrize("parts", [(True, False), (False, True)])
def test_epilogue_bias_only_and_scale_only(parts):
    r = routing(3, 256, 128, [40, 0, 129], [1, 2, 0], dist=("normal", 1.0))
    v = wl.host_values(r, 32)
    epi = _epilogue_case(r, 33, "silu", bias=parts[0], scale=parts[1])
    check_against_oracle(handle(3), r, v, epilogue=epi, where=f"epilogue parts {parts}")


@pytest.mark.parametrize("activation", ["relu", "gelu_tanh"])
def test_epilogue_int4(activation):
    r = routing(5, 200, 320, [1, 17, 160, 161, 40], [4, 0, 2, 3, -1], dist=("normal", 1.0), int4=True, gs=64)
    v = wl.host_values(r, 34)
    epi = _epilogue_case(r, 35, activation)
    _, _, status, _ = check_against_oracle(handle(5), r, v, epilogue=epi, where=f"int4 epilogue {activation}")
    assert status == binding.GMM_OK


def test_epilogue_exact_integer_case():
    """Integer operands and bias, power-of-two row scales, relu: every value is exact."""
    r = routing(5, 392, 24, [1, 17, 0, 130, 33, 256], [4, 0, 2, 3, -1, 1], dist=("int", -3, 3))
    v = wl.host_values(r, 36)
    rng = np.random.default_rng(37)
    epi = {"bias_bits": wl._to_bf16_bits(rng.integers(-20, 21, (5, 392)).astype(np.float32)),
           "row_scale": rng.choice([0.5, 1.0, 2.0], r.rows).astype(np.float32), "activation": "relu"}
    check_against_oracle(handle(5), r, v, epilogue=epi, exact=True, where="epilogue exact")


def test_epilogue_argument_errors():
    import torch
    h = handle(4)
    r = routing(4, 128, 64, [8], [1])
    v = wl.host_values(r, 38)
    c = sentinel_dev(r.rows, 128, DEV)
    av = torch.from_numpy(v["a"].view(np.int16)).to(DEV).view(torch.bfloat16)
    b = torch.from_numpy(v["b"].view(np.int16)).to(DEV).view(torch.bfloat16)
    off = to_dev_i32(r.a_offsets, DEV)
    ids = to_dev_i32(r.expert_ids, DEV)
    st = to_dev_i32(np.zeros(4), DEV)
    rc = binding.gmm_run_ex(h, c, av, off, b, ids, st, activation=7, check=False)
    assert rc == binding.GMM_ERR_INVALID_ARG      # unknown activation: nothing launched
    assert np.all(bits_of(c) == wl.SENTINEL_BF16)


# ---------------------------------------------------------------- dense rank-2 4-bit GEMM

@pytest.mark.parametrize("M,N,K,gs", [(1, 128, 128, 128), (150, 200, 320, 64), (300, 256, 512, 128),
                                      (33, 72, 1088, 64)])
def test_dense_int4_matches_single_group_oracle(M, N, K, gs):
    """gmm_matmul_int4 (the dense quantised GEMM) = the grouped 4-bit oracle with one group."""
    import torch
    r = routing(1, N, K, [M], [0], dist=("normal", 1.0), int4=True, gs=gs)
    v = wl.host_values(r, 40)
    ref = oracle.gmm_int4(v["a"], r.a_offsets, v["packed"], v["scales"], r.expert_ids, group_size=gs)
    h = handle(3)
    a = torch.from_numpy(v["a"].view(np.int16)).to(DEV).view(torch.bfloat16)
    q = torch.from_numpy(np.ascontiguousarray(v["packed"][0]).view(np.int32)).to(DEV)
    s = torch.from_numpy(np.ascontiguousarray(v["scales"][0]).view(np.int16)).to(DEV).view(torch.bfloat16)
    c = sentinel_dev(M, N, DEV)
    binding.gmm_matmul_int4(h, c, a, q, s, group_size=gs)
    assert binding.gmm_query_status(h) == binding.GMM_OK
    assert_close(bits_of(c), ref.ref32, np.ones(M, bool), f"dense int4 M={M} N={N} K={K}")


def test_dense_int4_zero_rows_and_epilogue():
    import torch
    h = handle(3)
    N, K, gs, M = 128, 256, 128, 70
    r = routing(1, N, K, [M], [0], dist=("normal", 1.0), int4=True, gs=gs)
    v = wl.host_values(r, 41)
    a = torch.from_numpy(v["a"].view(np.int16)).to(DEV).view(torch.bfloat16)
    q = torch.from_numpy(np.ascontiguousarray(v["packed"][0]).view(np.int32)).to(DEV)
    s = torch.from_numpy(np.ascontiguousarray(v["scales"][0]).view(np.int16)).to(DEV).view(torch.bfloat16)
    c0 = sentinel_dev(0, N, DEV)
    assert binding.gmm_matmul_int4(h, c0, a[:0], q, s, group_size=gs) == binding.GMM_OK   # nothing launched
    rng = np.random.default_rng(42)
    bias = wl._to_bf16_bits(rng.normal(0, 1, (1, N)).astype(np.float32))
    scale = rng.uniform(0.5, 1.5, M).astype(np.float32)
    c = sentinel_dev(M, N, DEV)
    binding.gmm_matmul_int4(h, c, a, q, s, group_size=gs, bias=to_dev_u16(bias, DEV),
                            row_scale=torch.from_numpy(scale).to(DEV), activation="silu")
    ref = oracle.apply_epilogue(oracle.gmm_int4(v["a"], r.a_offsets, v["packed"], v["scales"], r.expert_ids,
                                                group_size=gs),
                                r.a_offsets, r.expert_ids, 1, bias_bits=bias, row_scale=scale, activation="silu")
    assert_close(bits_of(c), ref.ref32, np.ones(M, bool), "dense int4 epilogue")


# ---------------------------------------------------------------- A-plane row offsetting

def _planes_case(h, r, splits, seed, rows_alloc=None, epilogue=None, where=""):
    rows_alloc = r.rows if rows_alloc is None else rows_alloc
    rng = np.random.default_rng(seed)
    a = wl._to_bf16_bits(rng.standard_normal((3 * rows_alloc, r.K)).astype(np.float32))
    b = wl._to_bf16_bits((0.1 * rng.standard_normal((r.E, r.N, r.K))).astype(np.float32))
    c0 = wl.sentinel_c(rows_alloc, r.N)
    # The planes are a_offsets[G] rows apart: lay A out with that stride.
    M = r.rows
    a_dev_rows = np.concatenate([a[p * rows_alloc:p * rows_alloc + M] for p in range(3)] +
                                [np.zeros((3 * rows_alloc - 3 * M, r.K), np.uint16)])
    ref = oracle.gmm_bf16_planes(a_dev_rows, r.a_offsets, b, r.expert_ids, splits, c_init=c0,
                                 stats_init=np.full(4, wl.SENTINEL_STATS, np.uint32))
    if epilogue:
        ref = oracle.apply_epilogue(ref, r.a_offsets, r.expert_ids, r.E, bias_bits=epilogue.get("bias_bits"),
                                    row_scale=epilogue.get("row_scale"), activation=epilogue.get("activation", "none"))
    import torch
    c = sentinel_dev(rows_alloc, r.N, DEV)
    st = to_dev_i32(np.full(4, 0xFFFFFFFF, np.uint32), DEV)
    epi = {}
    if epilogue:
        epi = {"bias": to_dev_u16(epilogue["bias_bits"], DEV),
               "row_scale": torch.from_numpy(epilogue["row_scale"]).to(DEV), "activation": epilogue["activation"]}
    binding.gmm_run_planes(h, c, to_dev_u16(a_dev_rows, DEV), to_dev_i32(r.a_offsets, DEV), to_dev_u16(b, DEV),
                           to_dev_i32(r.expert_ids, DEV), st, splits, **epi)
    assert binding.gmm_query_status(h) == binding.GMM_OK
    got = bits_of(c)
    live = live_row_mask(rows_alloc, r.a_offsets, r.expert_ids, r.E)
    assert np.array_equal(got[~live], ref.c[~live]), where
    assert np.array_equal(st.cpu().numpy().view(np.uint32), ref.stats), where
    assert_close(got, ref.ref32, live, where)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("N,splits", [(768, (256, 256)), (1280, (512, 256)), (512, (0, 512)), (512, (512, 0)),
                                      (1024, (0, 0)), (1536, (1024, 256))])
def test_a_plane_splits(N, splits, variant):
    """Each output column reads its plane of A (rows p * a_offsets[G] + r); ragged groups,
    a skipped group, N tails inside the last plane."""
    r = routing(4, N, 192, [1, 17, 0, 130, 33, 257, 7], [2, 0, 1, 3, -1, 1, 0])
    _planes_case(handle(4, variant), r, splits, 50, where=f"planes N={N} {splits} {variant}")


def test_a_plane_splits_with_epilogue_and_trailing_rows():
    r = routing(3, 1040, 128, [40, 300, 9], [2, 0, 1])
    rng = np.random.default_rng(52)
    epi = {"bias_bits": wl._to_bf16_bits(rng.normal(0, 0.5, (3, 1040)).astype(np.float32)),
           "row_scale": rng.uniform(0.5, 2.0, r.rows + 13).astype(np.float32), "activation": "silu"}
    _planes_case(handle(3), r, (512, 256), 51, rows_alloc=r.rows + 13, epilogue=epi, where="planes epilogue")


def test_a_plane_splits_argument_errors():
    import ctypes
    h = handle(2)
    r = routing(2, 512, 64, [8], [1])
    c = sentinel_dev(r.rows, 512, DEV)
    a = to_dev_u16(np.zeros((3 * r.rows, 64), np.uint16), DEV)
    b = to_dev_u16(np.zeros((2, 512, 64), np.uint16), DEV)
    off, ids, st = to_dev_i32(r.a_offsets, DEV), to_dev_i32(r.expert_ids, DEV), to_dev_i32(np.zeros(4), DEV)
    lib = binding.load_library()
    P = ctypes.c_void_p

    def call(splits):
        sp = None if splits is None else (ctypes.c_int * 2)(*splits)
        return lib.gmm_run_planes(h.ptr, P(c.data_ptr()), P(a.data_ptr()), P(off.data_ptr()), P(b.data_ptr()),
                                  P(ids.data_ptr()), P(st.data_ptr()), 1, 512, 64, sp, None, binding.stream_handle(0))
    assert call((128, 256)) == binding.GMM_ERR_UNSUPPORTED      # not a multiple of 256
    assert call((256, 512)) == binding.GMM_ERR_INVALID_ARG      # past N
    assert call((-256, 0)) == binding.GMM_ERR_INVALID_ARG
    assert call(None) == binding.GMM_ERR_INVALID_ARG
    assert np.all(bits_of(c) == wl.SENTINEL_BF16)


def test_lora_qkv_full_size_sampled():
    """The full lora_qkv workload (A-plane row offsetting) on sampled rows and columns."""
    import torch
    r = wl.routing("lora_qkv")
    v = wl.device_values(r, 0, device=DEV)
    h = handle(r.E)
    c = sentinel_dev(r.rows, r.N, DEV)
    st = to_dev_i32(np.full(4, 0xFFFFFFFF, np.uint32), DEV)
    binding.gmm_run_planes(h, c, v["a"], to_dev_i32(r.a_offsets, DEV), v["b"], to_dev_i32(r.expert_ids, DEV), st,
                           r.meta["planes"])
    assert binding.gmm_query_status(h) == binding.GMM_OK
    rng = np.random.default_rng(7)
    rows, loads = [], []
    for g in range(r.G):
        lo, hi = int(r.a_offsets[g]), int(r.a_offsets[g + 1])
        pick = sorted(set([lo, hi - 1] + rng.integers(lo, hi, 3).tolist())) if hi > lo else []
        rows += pick
        loads.append(len(pick))
    rows = np.asarray(rows, np.int64)
    cols = np.unique(np.concatenate([[0, 4095, 4096, 5119, 5120, r.N - 1], rng.choice(r.N, 90, replace=False)]))
    M = r.rows
    a_s = np.concatenate([bits_of(v["a"][torch.from_numpy(rows + p * M).to(DEV)]) for p in range(3)])
    b_s = bits_of(v["b"][:, torch.from_numpy(cols).to(DEV), :])
    off_s = wl.offsets_from_loads(loads)
    # The sampled columns keep their planes: recompute the split sizes in the sample.
    planes = oracle.plane_of_columns(r.N, r.meta["planes"])[cols]
    s0, s1 = int((planes == 0).sum()), int((planes == 1).sum())
    ref = oracle.gmm_bf16_planes(a_s, off_s, b_s, r.expert_ids, (s0, s1) if (s0, s1) != (0, 0) else (0, len(cols)))
    got = bits_of(c[torch.from_numpy(rows).to(DEV)][:, torch.from_numpy(cols).to(DEV)])
    assert_close(got, ref.ref32, np.ones(len(rows), bool), "lora_qkv sampled")


# ---------------------------------------------------------------- maximum sizes

@pytest.mark.parametrize("variant", VARIANTS)
def test_max_groups(variant):
    """The largest supported group count (4096): rows 0..3 per group, ids over 64 experts with
    skipped ones, every group in the scan, the schedule and the tile decode."""
    rng = np.random.default_rng(60)
    G = 4096
    loads = rng.integers(0, 4, G)
    ids = rng.integers(-1, 64, G).astype(np.int32)
    r = routing(64, 264, 128, loads, ids, dist=("normal", 1.0))
    v = wl.host_values(r, 61)
    _, _, status, _ = check_against_oracle(handle(64, variant), r, v, where=f"max groups {variant}")
    assert status == binding.GMM_OK


def test_long_k():
    """K = 16384 (128 pipeline stages per tile) with ragged groups and an N tail."""
    r = routing(3, 264, 16384, [1, 130, 257], [2, 0, 1], dist=("normal", 0.5))
    v = wl.host_values(r, 62)
    check_against_oracle(handle(3), r, v, where="long K")


def test_max_groups_int4():
    rng = np.random.default_rng(63)
    G = 4096
    r = routing(32, 256, 256, rng.integers(0, 3, G), rng.integers(-1, 32, G).astype(np.int32),
                dist=("normal", 1.0), int4=True, gs=128)
    v = wl.host_values(r, 64)
    _, _, status, _ = check_against_oracle(handle(32), r, v, where="max groups int4")
    assert status == binding.GMM_OK


# ---------------------------------------------------------------- CUDA graph capture

def _capture(fn):
    """Capture fn() (one library call on the current stream) in a CUDA graph."""
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()                      # once outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fn()
    torch.cuda.synchronize()
    return g


def test_cuda_graph_replay_bf16_and_dense_int4():
    """gmm_run and gmm_matmul_int4 (whose routing words are written by value nodes) captured
    once and replayed on new inputs written into the same buffers."""
    import torch
    h = handle(4)
    r = routing(4, 384, 512, [5, 130, 0, 77], [2, 0, -1, 3], dist=("normal", 1.0))
    a = torch.empty((r.rows, r.K), dtype=torch.bfloat16, device=DEV)
    b = torch.empty((4, r.N, r.K), dtype=torch.bfloat16, device=DEV)
    c = sentinel_dev(r.rows, r.N, DEV)
    off, ids = to_dev_i32(r.a_offsets, DEV), to_dev_i32(r.expert_ids, DEV)
    st = to_dev_i32(np.full(4, 0xFFFFFFFF, np.uint32), DEV)
    g = _capture(lambda: binding.gmm_run(h, c, a, off, b, ids, st))
    live = live_row_mask(r.rows, r.a_offsets, r.expert_ids, r.E)
    for seed in (80, 81):
        v = wl.host_values(r, seed)
        a.copy_(to_dev_u16(v["a"], DEV))
        b.copy_(to_dev_u16(v["b"], DEV))
        c.copy_(sentinel_dev(r.rows, r.N, DEV))
        g.replay()
        torch.cuda.synchronize()
        assert binding.gmm_query_status(h) == binding.GMM_OK
        ref = oracle.gmm_bf16(v["a"], r.a_offsets, v["b"], r.expert_ids, c_init=wl.sentinel_c(r.rows, r.N))
        got = bits_of(c)
        assert np.array_equal(got[~live], ref.c[~live])
        assert_close(got, ref.ref32, live, f"graph replay bf16 seed {seed}")

    h1 = handle(1)
    M, N, K, gs = 150, 256, 512, 128
    rd = routing(1, N, K, [M], [0], dist=("normal", 1.0), int4=True, gs=gs)
    a4 = torch.empty((M, K), dtype=torch.bfloat16, device=DEV)
    q = torch.empty((N, K // 8), dtype=torch.int32, device=DEV)
    sc = torch.empty((N, K // gs), dtype=torch.bfloat16, device=DEV)
    c4 = sentinel_dev(M, N, DEV)
    g4 = _capture(lambda: binding.gmm_matmul_int4(h1, c4, a4, q, sc, group_size=gs))
    for seed in (82, 83):
        v = wl.host_values(rd, seed)
        a4.copy_(to_dev_u16(v["a"], DEV))
        q.copy_(torch.from_numpy(np.ascontiguousarray(v["packed"][0]).view(np.int32)).to(DEV))
        sc.copy_(to_dev_u16(v["scales"][0], DEV))
        g4.replay()
        torch.cuda.synchronize()
        ref = oracle.gmm_int4(v["a"], rd.a_offsets, v["packed"], v["scales"], rd.expert_ids, group_size=gs)
        assert_close(bits_of(c4), ref.ref32, np.ones(M, bool), f"graph replay dense int4 seed {seed}")


def test_two_handles_on_two_streams_concurrently():
    """Handles share no device state: two handles, each launching on its own stream with
    no ordering between them, both match the oracle."""
    import torch
    ha = binding.gmm_create(4, 0)
    hb = binding.gmm_create(6, 0)
    try:
        ra = routing(4, 512, 1024, [100, 7, 300, 0], [1, 3, 0, 2], dist=("normal", 1.0))
        rb = routing(6, 768, 512, [50, 250, 1, 90, 33], [5, 0, 2, -1, 4], dist=("normal", 1.0))
        va, vb = wl.host_values(ra, 100), wl.host_values(rb, 101)
        sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
        outs = []
        for h, r, v, s in ((ha, ra, va, sa), (hb, rb, vb, sb)):
            c = sentinel_dev(r.rows, r.N, DEV)
            st = to_dev_i32(np.full(4, 0xFFFFFFFF, np.uint32), DEV)
            args = (to_dev_u16(v["a"], DEV), to_dev_i32(r.a_offsets, DEV), to_dev_u16(v["b"], DEV),
                    to_dev_i32(r.expert_ids, DEV))
            outs.append((h, r, v, s, c, st, args))
        torch.cuda.synchronize()
        for _ in range(5):                     # interleave launches on the two streams
            for h, r, v, s, c, st, (a, off, b, ids) in outs:
                binding.gmm_run(h, c, a, off, b, ids, st, stream=s)
        torch.cuda.synchronize()
        for h, r, v, s, c, st, _ in outs:
            assert binding.gmm_query_status(h) == binding.GMM_OK
            ref = oracle.gmm_bf16(v["a"], r.a_offsets, v["b"], r.expert_ids, c_init=wl.sentinel_c(r.rows, r.N),
                                  stats_init=np.full(4, 0xFFFFFFFF, np.uint32))
            got = bits_of(c)
            live = live_row_mask(r.rows, r.a_offsets, r.expert_ids, r.E)
            assert np.array_equal(got[~live], ref.c[~live])
            assert np.array_equal(st.cpu().numpy().view(np.uint32), ref.stats)
            assert_close(got, ref.ref32, live, f"concurrent handle E={r.E}")
    finally:
        binding.gmm_destroy(ha)
        binding.gmm_destroy(hb)


def _nonfinite_compare(got_bits, ref, live, where):
    got = (np.asarray(got_bits, np.uint16).astype(np.uint32) << 16).view(np.float32)[live]
    r32 = ref.ref32[live]
    assert np.array_equal(np.isnan(got), np.isnan(r32)), f"{where}: NaN positions differ"
    inf = np.isinf(r32)
    assert np.array_equal(np.isinf(got), inf) and np.array_equal(np.sign(got[inf]), np.sign(r32[inf])), \
        f"{where}: Inf positions or signs differ"
    fin = np.isfinite(r32)
    err = np.abs(got[fin].astype(np.float64) - r32[fin])
    assert np.all(err <= 1e-2 + 1e-2 * np.abs(r32[fin])), where


@pytest.mark.parametrize("variant", VARIANTS)
def test_nonfinite_inputs_propagate_like_the_oracle(variant):
    """NaN and +-Inf in A reach exactly the outputs the oracle says they reach (its row, all
    columns; with Inf, NaN where products of opposite infinities meet)."""
    r = routing(3, 264, 192, [9, 40, 0, 17], [2, 0, 1, -1], dist=("normal", 1.0))
    v = wl.host_values(r, 110)
    a = v["a"].copy()
    a[3, 5] = 0x7FC0          # NaN
    a[12, 0] = 0x7F80         # +Inf
    a[20, 7] = 0xFF80         # -Inf
    a[20, 9] = 0x7F80         # +Inf in the same row: that row's sums see +Inf and -Inf
    v = dict(v, a=a)
    got, stats, status = run_gpu(handle(3, variant), a, r.a_offsets, r.expert_ids, b_bits=v["b"], N=r.N)
    ref = oracle.gmm_bf16(a, r.a_offsets, v["b"], r.expert_ids, c_init=wl.sentinel_c(r.rows, r.N),
                          stats_init=np.full(4, 0xFFFFFFFF, np.uint32))
    live = live_row_mask(r.rows, r.a_offsets, r.expert_ids, r.E)
    assert np.isnan(ref.ref32[3]).all() and np.isinf(ref.ref32[12]).any()
    assert np.array_equal(got[~live], ref.c[~live]) and np.array_equal(stats, ref.stats)
    _nonfinite_compare(got, ref, live, f"non-finite {variant}")
