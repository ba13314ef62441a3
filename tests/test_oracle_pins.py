"""Pins for the CPU oracle, checked against things other than itself.

Each test ties the oracle to something fixed outside its own code: hand-worked
values (tests/golden), a library routine the special case reduces to (numpy
matmul / einsum in fp64, torch's bf16 cast), closed forms, invariants, and
brute force on tiny inputs.  Together they fail on a dropped term, a wrong
sign, a transposed operand, a wrong expert index, a wrong skip rule, a wrong
stats entry, a wrong nibble order, zero point or scale index.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from ragged_matmul_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_bits(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bits_to_f32(h):
    return (np.asarray(h, np.uint16).astype(np.uint32) << 16).view(np.float32)


# ------------------------------------------------------------------ rounding

def test_round_bf16_matches_torch_cast():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * 10,
        (rng.integers(0, 2**32, 20000, dtype=np.uint64).astype(np.uint32)).view(np.float32),
        np.array([0.0, -0.0, np.inf, -np.inf, 1.0 + 2**-8, 1.0 + 3 * 2**-8, 1e-40, -1e-40,
                  3.3895314e38, 3.40282e38], np.float32),
    ])
    # exact ties: upper 16 bits arbitrary, lower 16 bits = 0x8000
    ties = ((rng.integers(0, 2**16, 5000).astype(np.uint32) << 16) | 0x8000).view(np.float32)
    x = np.concatenate([x, ties])
    mine = oracle.round_bf16(x)
    ref = bf16_bits(x)
    nan = np.isnan(x)
    assert np.array_equal(mine[~nan], ref[~nan])
    assert np.all(np.isnan(bits_to_f32(mine[nan])))


# ------------------------------------------------------------------ hand-worked fixtures

def _parse_golden_bf16():
    lines = [l.split() for l in open(os.path.join(GOLDEN, "hand_worked_bf16.txt")) if l.strip() and not l.startswith("#")]
    d, i = {}, 0
    while i < len(lines):
        key = lines[i][0]
        if key in ("E", "N", "K", "stats1"):
            d[key] = int(lines[i][1]); i += 1
        elif key in ("offsets", "ids"):
            d[key] = [int(v) for v in lines[i][1:]]; i += 1
        elif key in ("A", "B0", "B1", "C"):
            rows = []
            i += 1
            while i < len(lines) and lines[i][0] not in ("A", "B0", "B1", "C", "stats1"):
                rows.append(lines[i]); i += 1
            d[key] = rows
        else:
            raise ValueError(key)
    return d


def test_bf16_bits_to_f32_matches_torch_on_every_pattern():
    """All 65,536 bf16 bit patterns widen to the fp32 torch gives (NaNs compared as NaN)."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle.bf16_bits_to_f32(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))   # signed zeros too


def test_validate_flags_and_active_count_hand_worked():
    """grouped_matmul_sm100_persistent, Args (expert_ids, a_offsets): a negative id skips its
    group and the stats count the active groups.  Where the page is silent the reading taken
    is that an id of E or more is skipped, not counted and flagged, and that decreasing offsets
    are flagged."""
    E = 4
    # ids 3, -1, 0, 2: three active; offsets non-decreasing (an empty group included)
    assert oracle.validate([0, 5, 5, 9, 12], [3, -1, 0, 2], E) == (0, 3)
    # all skipped: no flags, no active group
    assert oracle.validate([0, 1, 2], [-1, -7], E) == (0, 0)
    # id == E is out of range: flagged and not counted
    flags, active = oracle.validate([0, 2, 4], [4, 1], E)
    assert flags == oracle.BAD_EXPERT_ID and active == 1
    # a decreasing offset is flagged whatever the ids
    flags, active = oracle.validate([0, 6, 3], [0, -1], E)
    assert flags == oracle.BAD_OFFSETS and active == 1
    # both problems at once
    flags, _ = oracle.validate([4, 2], [9], E)
    assert flags == oracle.BAD_OFFSETS | oracle.BAD_EXPERT_ID
    # no groups at all
    assert oracle.validate([0], np.zeros(0, np.int32), E) == (0, 0)


def test_hand_worked_bf16_example():
    d = _parse_golden_bf16()
    A = np.array([[float(v) for v in r] for r in d["A"]], np.float32)
    B = np.stack([np.array([[float(v) for v in r] for r in d[f"B{e}"]], np.float32) for e in range(d["E"])])
    assert B.shape == (d["E"], d["N"], d["K"])
    c0 = wl.sentinel_c(A.shape[0], d["N"])
    res = oracle.gmm_bf16(bf16_bits(A), d["offsets"], bf16_bits(B), d["ids"], c_init=c0,
                          stats_init=np.full(4, wl.SENTINEL_STATS, np.uint32))
    assert res.flags == 0
    for r, row in enumerate(d["C"]):
        for n, v in enumerate(row):
            if v == "untouched":
                assert res.c[r, n] == wl.SENTINEL_BF16
            else:
                assert bits_to_f32(res.c[r, n]) == float(v), (r, n)
    assert res.stats[1] == d["stats1"]
    assert res.stats[0] == wl.SENTINEL_STATS and res.stats[2] == wl.SENTINEL_STATS


def test_hand_worked_int4_example():
    d = {}
    for l in open(os.path.join(GOLDEN, "hand_worked_int4.txt")):
        if l.strip() and not l.startswith("#"):
            k, *v = l.split()
            d[k] = v
    K, gs = int(d["K"][0]), int(d["group_size"][0])
    words = np.array([[int(w, 16) for w in d["words"]]], np.uint32)
    scales = bf16_bits(np.array([[float(s) for s in d["scales"]]], np.float32))
    w = oracle.dequant_int4(words, scales, gs)
    assert np.array_equal(bits_to_f32(w[0]), np.array([float(v) for v in d["W"]], np.float32))
    A = np.zeros((3, K), np.float32)
    A[0] = 1.0
    A[1, 3] = 1.0
    A[2, 9] = 1.0
    res = oracle.gmm_int4(bf16_bits(A), [0, 3], words[None], scales[None], [0], group_size=gs)
    got = bits_to_f32(res.c[:, 0])
    assert got.tolist() == [float(d["A_ones"][0]), float(d["A_unit3"][0]), float(d["A_unit9"][0])]


# ------------------------------------------------------------------ library special cases

def _rand_problem(seed, E, N, K, loads, ids, base=0, dist=("uniform", -1.0, 1.0)):
    r = wl.make_routing("t", E, N, K, loads, ids, a_dist=dist, b_dist=dist, base=base)
    v = wl.host_values(r, seed)
    return r, v


def test_single_group_is_dense_matmul():
    """G = 1 reduces to C = A @ B[e]^T; fp32 accumulation stays within its error bound."""
    r, v = _rand_problem(1, E=3, N=40, K=72, loads=[37], ids=[2])
    res = oracle.gmm_bf16(v["a"], r.a_offsets, v["b"], r.expert_ids, want64=True)
    A = bits_to_f32(v["a"]).astype(np.float64)
    B = bits_to_f32(v["b"]).astype(np.float64)
    exact = A @ B[2].T
    bound = r.K * 2.0**-24 * (np.abs(A) @ np.abs(B[2]).T) * 1.01 + 1e-30
    assert np.all(np.abs(res.ref32 - exact) <= bound)
    assert np.allclose(res.ref64, exact, rtol=1e-12, atol=1e-12)
    assert np.array_equal(res.c, bf16_bits(res.ref32))


def test_multi_group_matches_gathered_einsum():
    """Per-row expert gather + einsum (a different route) agrees with the oracle's fp64 sums."""
    loads = [5, 0, 9, 1, 14, 3, 7]
    ids = [3, 0, -1, 1, 3, 2, -1]
    r, v = _rand_problem(2, E=4, N=24, K=40, loads=loads, ids=ids)
    res = oracle.gmm_bf16(v["a"], r.a_offsets, v["b"], r.expert_ids, want64=True,
                          c_init=wl.sentinel_c(r.rows, r.N))
    expert_of_row = np.repeat(np.asarray(ids), loads)
    live = expert_of_row >= 0
    A = bits_to_f32(v["a"]).astype(np.float64)
    B = bits_to_f32(v["b"]).astype(np.float64)
    ref = np.einsum("rk,rnk->rn", A[live], B[expert_of_row[live]])
    assert np.allclose(res.ref64[live], ref, rtol=1e-12, atol=1e-12)
    assert np.all(res.c[~live] == wl.SENTINEL_BF16)
    assert res.stats[1] == 5


def test_unit_rows_select_weight_entries():
    """A row equal to the unit vector e_k yields C[r, n] = B[e, n, k] exactly (pins B's layout)."""
    E, N, K = 3, 5, 7
    rng = np.random.default_rng(3)
    B = bf16_bits(rng.uniform(-2, 2, (E, N, K)).astype(np.float32))
    loads, ids = [K, K, K], [2, 0, 1]
    A = np.zeros((3 * K, K), np.float32)
    for g in range(3):
        for k in range(K):
            A[g * K + k, k] = 1.0
    res = oracle.gmm_bf16(bf16_bits(A), wl.offsets_from_loads(loads), B, ids)
    for g in range(3):
        for k in range(K):
            assert np.array_equal(res.c[g * K + k], B[ids[g], :, k])


def test_small_integers_are_exact():
    """Integer operands in [-3, 3]: every sum is an exact integer; compare with int64 matmul."""
    rng = np.random.default_rng(4)
    E, N, K = 4, 48, 28
    loads, ids = [6, 11, 0, 17, 4], [1, 3, 0, -1, 2]
    off = wl.offsets_from_loads(loads)
    Ai = rng.integers(-3, 4, (off[-1], K))
    Bi = rng.integers(-3, 4, (E, N, K))
    res = oracle.gmm_bf16(bf16_bits(Ai), off, bf16_bits(Bi), ids)
    for g, e in enumerate(ids):
        if e < 0:
            continue
        rows = slice(off[g], off[g + 1])
        want = Ai[rows] @ Bi[e].T
        assert np.array_equal(bits_to_f32(res.c[rows]), want.astype(np.float32))


# ------------------------------------------------------------------ invariants

def test_group_permutation_invariance():
    loads = [13, 2, 0, 21, 8, 5]
    ids = [1, 0, 2, -1, 3, 1]
    r, v = _rand_problem(5, E=4, N=32, K=64, loads=loads, ids=ids)
    base = oracle.gmm_bf16(v["a"], r.a_offsets, v["b"], r.expert_ids, c_init=wl.sentinel_c(r.rows, r.N))
    perm = np.random.default_rng(6).permutation(len(loads))
    off = r.a_offsets.astype(np.int64)
    blocks = [np.arange(off[g], off[g + 1]) for g in range(len(loads))]
    row_perm = np.concatenate([blocks[g] for g in perm]).astype(np.int64)
    loads_p = np.asarray(loads)[perm]
    ids_p = np.asarray(ids)[perm]
    res = oracle.gmm_bf16(v["a"][row_perm], wl.offsets_from_loads(loads_p), v["b"], ids_p,
                          c_init=wl.sentinel_c(r.rows, r.N))
    assert np.array_equal(res.c, base.c[row_perm])
    assert res.stats[1] == base.stats[1]


def test_skipped_groups_with_rows_stay_untouched_and_stats_count():
    loads = [4, 9, 3, 0, 6]
    ids = [-1, 2, -7, 1, -1]
    r, v = _rand_problem(7, E=3, N=16, K=32, loads=loads, ids=ids, base=5)
    rows_alloc = r.rows + 3            # rows before a_offsets[0] and after a_offsets[G] exist too
    a = np.concatenate([v["a"], v["a"][:3]])
    c0 = wl.sentinel_c(rows_alloc, r.N)
    stats0 = np.array([11, 22, 33, 44], np.uint32)
    res = oracle.gmm_bf16(a, r.a_offsets, v["b"], r.expert_ids, c_init=c0, stats_init=stats0)
    live = np.zeros(rows_alloc, bool)
    live[r.a_offsets[1]:r.a_offsets[2]] = True
    assert np.all(res.c[~live] == wl.SENTINEL_BF16)
    assert not np.any(res.c[live] == wl.SENTINEL_BF16)
    assert res.stats.tolist() == [11, 2, 33, 44]      # ids 2 and 1 are active (the empty group counts)


def test_invalid_inputs_are_flagged():
    b = np.zeros((2, 8, 8), np.uint16)
    a = np.zeros((10, 8), np.uint16)
    c0 = wl.sentinel_c(10, 8)
    res = oracle.gmm_bf16(a, [0, 6, 4, 10], b, [0, 1, 0], c_init=c0)
    assert res.flags & oracle.BAD_OFFSETS
    assert np.all(res.c == wl.SENTINEL_BF16)            # nothing computed
    assert res.stats[1] == 3
    res = oracle.gmm_bf16(a, [0, 4, 10], b, [0, 2], c_init=c0)
    assert res.flags == oracle.BAD_EXPERT_ID
    assert np.all(res.c[4:] == wl.SENTINEL_BF16) and not np.any(res.c[:4] == wl.SENTINEL_BF16)
    assert res.stats[1] == 1


def test_empty_problem_writes_only_stats():
    b = np.zeros((2, 8, 8), np.uint16)
    res = oracle.gmm_bf16(np.zeros((0, 8), np.uint16), [0], b, np.zeros(0, np.int32),
                          stats_init=np.full(4, 7, np.uint32))
    assert res.stats.tolist() == [7, 0, 7, 7] and res.flags == 0


def test_fp32_result_within_bound_of_fp64():
    r, v = _rand_problem(8, E=2, N=64, K=1024, loads=[40, 30], ids=[1, 0], dist=("normal", 1.0))
    res = oracle.gmm_bf16(v["a"], r.a_offsets, v["b"], r.expert_ids, want64=True)
    A = np.abs(bits_to_f32(v["a"]).astype(np.float64))
    B = np.abs(bits_to_f32(v["b"]).astype(np.float64))
    expert_of_row = np.repeat(r.expert_ids, r.loads)
    bound = r.K * 2.0**-24 * np.einsum("rk,rnk->rn", A, B[expert_of_row])
    assert np.all(np.abs(res.ref32 - res.ref64) <= bound)


def test_thread_count_does_not_change_bits():
    r, v = _rand_problem(9, E=3, N=40, K=96, loads=[17, 3, 29, 1], ids=[0, 2, 1, 0])
    one = oracle.gmm_bf16(v["a"], r.a_offsets, v["b"], r.expert_ids, nthreads=1)
    many = oracle.gmm_bf16(v["a"], r.a_offsets, v["b"], r.expert_ids, nthreads=7)
    assert np.array_equal(one.c, many.c)
    assert np.array_equal(one.ref32.view(np.uint32), many.ref32.view(np.uint32))


def test_tiny_workload_brute_force():
    """The tiny named workload against plain Python loops in double precision."""
    r = wl.routing("tiny")
    v = wl.host_values(r, 0)
    res = oracle.gmm_bf16(v["a"], r.a_offsets, v["b"], r.expert_ids, want64=True,
                          c_init=wl.sentinel_c(r.rows, r.N))
    A = bits_to_f32(v["a"]).tolist()
    B = bits_to_f32(v["b"])
    rng = np.random.default_rng(10)
    off = r.a_offsets.tolist()
    for g, e in enumerate(r.expert_ids.tolist()):
        for row in range(off[g], off[g + 1]):
            for n in rng.choice(r.N, 24, replace=False):
                if e < 0:
                    assert res.c[row, n] == wl.SENTINEL_BF16
                    continue
                w = B[e, n].tolist()
                s = 0.0
                for k in range(r.K):
                    s += A[row][k] * w[k]
                assert abs(res.ref64[row, n] - s) <= 1e-12 * (1 + abs(s))
                assert abs(res.ref32[row, n] - s) <= 1e-4
    assert res.stats[1] == 3


# ------------------------------------------------------------------ 4-bit variant

def test_int4_dequant_matches_independent_unpack():
    rng = np.random.default_rng(11)
    N, K, gs = 6, 64, 16
    q = rng.integers(0, 16, (N, K))
    words = np.zeros((N, K // 8), np.uint64)
    for k in range(K):                                    # pack by explicit place value
        words[:, k // 8] += q[:, k].astype(np.uint64) * (16 ** (k % 8))
    words = words.astype(np.uint32)
    s = rng.uniform(0.005, 0.02, (N, K // gs)).astype(np.float32)
    sb = bf16_bits(s)
    w = oracle.dequant_int4(words, sb, gs)
    want = bf16_bits((q - 8).astype(np.float32) * np.repeat(bits_to_f32(sb), gs, axis=1))
    assert np.array_equal(w, want)
    # the generator's packer agrees with the place-value packing
    assert np.array_equal(wl.pack_nibbles(q), words)


def test_int4_zero_point_gives_zero():
    N, K = 8, 32
    words = wl.pack_nibbles(np.full((1, N, K), 8))
    scales = bf16_bits(np.full((1, N, K // 16), 0.013, np.float32))
    a = bf16_bits(np.random.default_rng(12).standard_normal((5, K)).astype(np.float32))
    res = oracle.gmm_int4(a, [0, 5], words, scales, [0], group_size=16)
    assert np.all(bits_to_f32(res.c) == 0.0)


def test_int4_integer_case_is_exact():
    rng = np.random.default_rng(13)
    E, N, K, gs = 3, 16, 64, 32
    q = rng.integers(0, 16, (E, N, K))
    scales = bf16_bits(np.ones((E, N, K // gs), np.float32))
    Ai = rng.integers(-2, 3, (20, K))
    loads, ids = [7, 0, 13], [2, 1, 0]
    off = wl.offsets_from_loads(loads)
    res = oracle.gmm_int4(bf16_bits(Ai), off, wl.pack_nibbles(q), scales, ids, group_size=gs)
    for g, e in enumerate(ids):
        rows = slice(off[g], off[g + 1])
        assert np.array_equal(bits_to_f32(res.c[rows]), (Ai[rows] @ (q[e] - 8).T).astype(np.float32))


def test_int4_equals_bf16_path_on_dequantised_weights():
    """The 4-bit oracle is the bf16 oracle applied to the dequantised weights."""
    r = wl.make_routing("q", 4, 32, 256, [9, 0, 23, 4], [3, 1, -1, 0], a_dist=("normal", 1.0),
                        b_dist=None, int4=True, group_size=128)
    v = wl.host_values(r, 14)
    res4 = oracle.gmm_int4(v["a"], r.a_offsets, v["packed"], v["scales"], r.expert_ids, group_size=128)
    w = np.stack([oracle.dequant_int4(v["packed"][e], v["scales"][e], 128) for e in range(r.E)])
    res16 = oracle.gmm_bf16(v["a"], r.a_offsets, w, r.expert_ids)
    assert np.array_equal(res4.c, res16.c)
    assert res4.stats[1] == res16.stats[1] == 3


# ------------------------------------------------------------------ generators

def test_named_routings_have_the_stated_structure():
    t = wl.routing("tiny")
    assert t.loads.tolist() == [3, 17, 0, 40] and t.expert_ids.tolist() == [2, 0, -1, 3]
    d = wl.routing("decode")
    assert d.rows == 2048 and d.G == 64 and (d.N, d.K) == (2816, 2048)
    p = wl.routing("prefill")
    assert p.rows == 32768 and np.all(np.abs(p.loads - 4096) <= 409.6)
    f = wl.routing("fine_grained")
    assert f.rows == 32768 and int((f.expert_ids < 0).sum()) == 13 and (f.N, f.K) == (4096, 7168)
    q = wl.routing("int4")
    assert q.rows == 8192 and q.int4 and (q.N, q.K, q.group_size) == (4096, 4096, 128)


# ------------------------------------------------------------------ optional epilogue

def test_epilogue_activations_against_independent_forms():
    """relu exactly; silu against scipy's logistic function; the tanh form of GELU against
    the exact (erf) GELU within the approximation's error, and both fixed points."""
    sp = pytest.importorskip("scipy.special")
    y = np.concatenate([np.linspace(-12, 12, 2001), [0.0, -0.0, 30.0, -30.0]])
    assert np.array_equal(oracle.activation_ref("relu", y), np.where(y > 0, y, 0.0))
    assert np.allclose(oracle.activation_ref("silu", y), y * sp.expit(y), rtol=1e-12, atol=1e-300)
    gelu_exact = 0.5 * y * (1.0 + sp.erf(y / np.sqrt(2.0)))
    assert np.max(np.abs(oracle.activation_ref("gelu_tanh", y) - gelu_exact)) < 1e-3
    for name in ("relu", "silu", "gelu_tanh"):
        assert oracle.activation_ref(name, np.array([0.0]))[0] == 0.0
        assert abs(oracle.activation_ref(name, np.array([30.0]))[0] - 30.0) < 1e-9   # identity far right
    assert np.array_equal(oracle.activation_ref("none", y), y)


def test_epilogue_small_integer_case_is_exact():
    """Integer A, B and bias, row scales that are powers of two: every value is exact, so
    C must equal bf16(act(A.B^T + bias) * scale) computed with int64 arithmetic."""
    rng = np.random.default_rng(21)
    E, N, K = 3, 40, 24
    loads, ids = [5, 0, 9, 7], [2, 1, -1, 0]
    r = wl.make_routing("t", E, N, K, loads, ids, a_dist=("int", -3, 3), b_dist=("int", -3, 3))
    v = wl.host_values(r, 22)
    bias = rng.integers(-20, 21, (E, N))
    scale = rng.choice([0.5, 1.0, 2.0, 4.0], r.rows).astype(np.float32)
    c0 = wl.sentinel_c(r.rows, N)
    base = oracle.gmm_bf16(v["a"], r.a_offsets, v["b"], r.expert_ids, c_init=c0)
    A = bits_to_f32(v["a"]).astype(np.int64)
    B = bits_to_f32(v["b"]).astype(np.int64)
    for act in ("none", "relu"):
        got = oracle.apply_epilogue(base, r.a_offsets, r.expert_ids, E, bias_bits=bf16_bits(bias),
                                    row_scale=scale, activation=act)
        want = c0.copy()
        off = r.a_offsets
        for g, e in enumerate(ids):
            if e < 0:
                continue
            y = A[off[g]:off[g + 1]] @ B[e].T + bias[e][None, :]
            if act == "relu":
                y = np.maximum(y, 0)
            want[off[g]:off[g + 1]] = bf16_bits(y * scale[off[g]:off[g + 1], None].astype(np.float64))
        assert np.array_equal(got.c, want), act


def test_epilogue_leaves_rows_outside_active_groups():
    r = wl.make_routing("t", 2, 16, 16, [3, 4, 2], [1, -1, 0], a_dist=("normal", 1.0), b_dist=("normal", 1.0))
    v = wl.host_values(r, 23)
    c0 = wl.sentinel_c(r.rows + 5, 16)
    base = oracle.gmm_bf16(np.concatenate([v["a"], np.zeros((5, 16), np.uint16)]), r.a_offsets, v["b"],
                           r.expert_ids, c_init=c0)
    got = oracle.apply_epilogue(base, r.a_offsets, r.expert_ids, 2, activation="silu",
                                row_scale=np.full(r.rows + 5, 3.0, np.float32))
    skipped = np.zeros(r.rows + 5, bool)
    skipped[3:7] = True
    skipped[r.rows:] = True
    assert np.all(got.c[skipped] == wl.SENTINEL_BF16)
    assert not np.any(got.c[~skipped] == wl.SENTINEL_BF16)


# ------------------------------------------------------------------ scaled e4m3 variant

def test_e4m3_decode_matches_torch_and_format_values():
    """All 256 patterns against torch's float8_e4m3fn, plus values the format fixes:
    bias 7, 3 mantissa bits, subnormals at exponent 0, S.1111.111 the only NaN."""
    bits = np.arange(256, dtype=np.uint8)
    got = oracle.e4m3_to_f32(bits)
    ref = torch.from_numpy(bits).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2
    assert np.array_equal(got[~nan], ref[~nan])
    fixed = {0x38: 1.0, 0xB8: -1.0, 0x40: 2.0, 0x30: 0.5, 0x7E: 448.0, 0x08: 2.0**-6,
             0x01: 2.0**-9, 0x07: 7 * 2.0**-9, 0x00: 0.0, 0x3C: 1.5}
    for b, v in fixed.items():
        assert got[b] == v, hex(b)
    assert np.signbit(got[0x80]) and got[0x80] == 0.0


def test_fp8_hand_worked_example():
    """One row, one weight row, K=2: a = (1, 2), w = (0.5, -1.5), input scale 2,
    weight scale 0.25: (1*0.5 + 2*(-1.5)) * 2 * 0.25 = -1.25."""
    a8 = np.array([[0x38, 0x40]], np.uint8)
    w8 = np.array([[[0x30, 0xBC]]], np.uint8)
    res = oracle.gmm_fp8(a8, [0, 1], w8, [0], np.array([[2.0]], np.float32),
                         np.array([[[0.25]]], np.float32), (1, 1, 2))
    assert res.ref64[0, 0] == -1.25 and res.ref32[0, 0] == -1.25
    assert res.c[0, 0] == bf16_bits([-1.25])[0]


def _fp8_problem(seed, E, N, K, loads, ids, gran):
    r = wl.make_routing("t", E, N, K, loads, ids)
    v = wl.fp8_host_values(r, seed, gran)
    return r, v


def test_fp8_per_element_brute_force():
    """Tiny problem, granularities that do not divide the sizes: every output against
    a triple loop that scales each product by its own two block scales."""
    gran = (2, 4, 5)
    r, v = _fp8_problem(3, E=3, N=7, K=13, loads=[2, 1, 3, 0], ids=[2, -1, 0, 1], gran=gran)
    c0 = wl.sentinel_c(r.rows, r.N)
    res = oracle.gmm_fp8(v["a8"], r.a_offsets, v["w8"], r.expert_ids, v["input_scale"],
                         v["weight_scale"], gran, c_init=c0)
    a = oracle.e4m3_to_f32(v["a8"]).astype(np.float64)
    w = oracle.e4m3_to_f32(v["w8"]).astype(np.float64)
    gm, gn, gk = gran
    for g in range(r.G):
        e = int(r.expert_ids[g])
        for row in range(int(r.a_offsets[g]), int(r.a_offsets[g + 1])):
            if e < 0:
                assert np.all(res.c[row] == wl.SENTINEL_BF16)
                continue
            for n in range(r.N):
                acc = 0.0
                for k in range(r.K):
                    acc += (a[row, k] * w[e, n, k] * float(v["input_scale"][row // gm, k // gk])
                            * float(v["weight_scale"][e, n // gn, k // gk]))
                assert abs(res.ref64[row, n] - acc) <= 1e-12 * max(1.0, abs(acc))
    assert res.stats[1] == 3 and res.flags == 0


def test_fp8_unit_granularity_is_matmul_of_prescaled_operands():
    """(1, 1, 1): every element has its own scale, so the result is the plain matmul of
    (a * input_scale) and (w * weight_scale)."""
    gran = (1, 1, 1)
    r, v = _fp8_problem(5, E=2, N=24, K=40, loads=[9, 6], ids=[1, 0], gran=gran)
    res = oracle.gmm_fp8(v["a8"], r.a_offsets, v["w8"], r.expert_ids, v["input_scale"],
                         v["weight_scale"], gran)
    a = oracle.e4m3_to_f32(v["a8"]).astype(np.float64) * v["input_scale"]
    w = oracle.e4m3_to_f32(v["w8"]).astype(np.float64) * v["weight_scale"]
    exact = np.concatenate([a[:9] @ w[1].T, a[9:] @ w[0].T])
    assert np.allclose(res.ref64, exact, rtol=1e-12, atol=1e-300)


def test_fp8_unit_scales_equal_the_bf16_oracle():
    """Unit scales: the grouped GEMM of the decoded values (e4m3 values are bf16 values),
    which the C oracle computes independently; the fp32 sums agree within their bound."""
    gran = (1, 128, None)
    r, v = _fp8_problem(7, E=4, N=40, K=96, loads=[5, 0, 11, 3], ids=[3, 1, 0, -1], gran=gran)
    ones_in = np.ones_like(v["input_scale"])
    ones_w = np.ones_like(v["weight_scale"])
    res = oracle.gmm_fp8(v["a8"], r.a_offsets, v["w8"], r.expert_ids, ones_in, ones_w, (1, 128, 96))
    a_bits = bf16_bits(oracle.e4m3_to_f32(v["a8"]))
    w_bits = bf16_bits(oracle.e4m3_to_f32(v["w8"]))
    ref = oracle.gmm_bf16(a_bits, r.a_offsets, w_bits, r.expert_ids, want64=True)
    act = ~np.isnan(ref.ref64[:, 0])
    assert np.array_equal(act, ~np.isnan(res.ref64[:, 0]))
    assert np.allclose(res.ref64[act], ref.ref64[act], rtol=1e-12, atol=1e-300)
    assert np.array_equal(res.stats, ref.stats) and res.flags == ref.flags


def test_fp8_whole_k_scales_factorise():
    """gk = K: the result is input_scale[r // gm] * weight_scale[e, n // gn] times the
    unscaled sum (the form the CUDA path computes in its epilogue)."""
    gran = (3, 16, None)
    r, v = _fp8_problem(9, E=2, N=48, K=64, loads=[7, 10], ids=[0, 1], gran=gran)
    res = oracle.gmm_fp8(v["a8"], r.a_offsets, v["w8"], r.expert_ids, v["input_scale"],
                         v["weight_scale"], (3, 16, 64))
    unit = oracle.gmm_fp8(v["a8"], r.a_offsets, v["w8"], r.expert_ids, np.ones_like(v["input_scale"]),
                          np.ones_like(v["weight_scale"]), (3, 16, 64))
    rows = np.arange(r.rows)
    e_of_row = np.repeat(r.expert_ids, r.loads)
    isc = v["input_scale"].astype(np.float64)
    wsc = v["weight_scale"].astype(np.float64)
    scale = isc[rows // 3, 0][:, None] * wsc[e_of_row][:, np.arange(48) // 16, 0]
    assert np.allclose(res.ref64, unit.ref64 * scale, rtol=1e-12, atol=1e-300)


def test_fp8_invalid_inputs_follow_the_grouped_rules():
    r, v = _fp8_problem(11, E=2, N=8, K=16, loads=[2, 2], ids=[0, 1], gran=(1, 8, None))
    c0 = wl.sentinel_c(4, 8)
    bad = oracle.gmm_fp8(v["a8"], [0, 3, 2], v["w8"], [0, 1], v["input_scale"], v["weight_scale"],
                         (1, 8, 16), c_init=c0, stats_init=np.full(4, 7, np.uint32))
    assert bad.flags & oracle.BAD_OFFSETS and np.all(bad.c == wl.SENTINEL_BF16)
    assert list(bad.stats) == [7, 2, 7, 7]
    oob = oracle.gmm_fp8(v["a8"], r.a_offsets, v["w8"], [0, 5], v["input_scale"], v["weight_scale"],
                         (1, 8, 16), c_init=c0)
    assert oob.flags & oracle.BAD_EXPERT_ID and oob.stats[1] == 1
    assert np.all(oob.c[2:] == wl.SENTINEL_BF16) and not np.any(oob.c[:2] == wl.SENTINEL_BF16)


# ------------------------------------------------------------------ A-plane row offsetting

def _plane_problem(seed, E, N, K, loads, ids, planes=3):
    r = wl.make_routing("t", E, N, K, loads, ids, a_dist=("normal", 1.0), b_dist=("normal", 1.0))
    rng = np.random.default_rng(seed)
    a = bf16_bits(rng.standard_normal((planes * r.rows, K)).astype(np.float32))
    b = bf16_bits(rng.standard_normal((E, N, K)).astype(np.float32))
    return r, a, b


def test_planes_disabled_is_the_grouped_gemm():
    r, a, b = _plane_problem(1, 3, 40, 24, [5, 0, 9], [2, 1, 0])
    got = oracle.gmm_bf16_planes(a, r.a_offsets, b, r.expert_ids, (0, 0))
    ref = oracle.gmm_bf16(a[:r.rows], r.a_offsets, b, r.expert_ids)
    assert np.array_equal(got.c, ref.c) and np.array_equal(got.stats, ref.stats)


def test_planes_brute_force():
    """Every output against a loop that reads row p(n) * M + r of A."""
    r, a, b = _plane_problem(2, 2, 12, 8, [3, 2, 4], [1, -1, 0])
    splits = (5, 4)
    got = oracle.gmm_bf16_planes(a, r.a_offsets, b, r.expert_ids, splits)
    A, B = bits_to_f32(a).astype(np.float64), bits_to_f32(b).astype(np.float64)
    M = r.rows
    for g in range(r.G):
        e = int(r.expert_ids[g])
        for row in range(int(r.a_offsets[g]), int(r.a_offsets[g + 1])):
            for n in range(12):
                if e < 0:
                    assert np.isnan(got.ref32[row, n])
                    continue
                p = 0 if n < 5 else (1 if n < 9 else 2)
                exact = sum(A[p * M + row, k] * B[e, n, k] for k in range(8))
                assert abs(got.ref32[row, n] - exact) <= 8 * 2.0**-24 * sum(abs(A[p * M + row, k] * B[e, n, k]) for k in range(8)) + 1e-30


def test_planes_identical_planes_and_whole_plane_splits():
    """Three copies of one plane give the grouped GEMM; (0, N) sends every column to plane 1."""
    r, a, b = _plane_problem(3, 2, 32, 16, [7, 6], [0, 1])
    M = r.rows
    same = np.concatenate([a[:M]] * 3)
    got = oracle.gmm_bf16_planes(same, r.a_offsets, b, r.expert_ids, (8, 16))
    ref = oracle.gmm_bf16(a[:M], r.a_offsets, b, r.expert_ids)
    assert np.array_equal(got.c, ref.c)
    got1 = oracle.gmm_bf16_planes(a, r.a_offsets, b, r.expert_ids, (0, 32))
    ref1 = oracle.gmm_bf16(a[M:2 * M], r.a_offsets, b, r.expert_ids)
    assert np.array_equal(got1.c, ref1.c)
    assert list(oracle.plane_of_columns(6, (2, 3))) == [0, 0, 1, 1, 1, 2]


def test_c_init_memory_order_does_not_matter():
    """A non-contiguous c_init (a column slice) gives the same result as a contiguous copy."""
    r, v = _rand_problem(41, E=2, N=24, K=16, loads=[5, 4], ids=[1, 0])
    wide = wl.sentinel_c(r.rows, 48)
    view = wide[:, ::2]
    assert not view.flags["C_CONTIGUOUS"]
    a = oracle.gmm_bf16(v["a"], r.a_offsets, v["b"], r.expert_ids, c_init=view)
    b = oracle.gmm_bf16(v["a"], r.a_offsets, v["b"], r.expert_ids, c_init=np.ascontiguousarray(view))
    assert np.array_equal(a.c, b.c)
