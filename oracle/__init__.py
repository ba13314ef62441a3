"""CPU oracle for the ragged grouped GEMM — TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
leg of ``bench.py`` may import this package.  The product path (the
``ragged_matmul_gb300`` package and its CUDA library) never does, and shares
no code with it.

The bf16 and 4-bit grouped GEMMs live in ``oracle.c`` (plain C, one thread
per slice of output rows); this module compiles it with gcc, loads it with
ctypes and marshals numpy arrays.  See ``oracle.c`` for the definition it
implements and the page sections it follows (Modular
"grouped_matmul_sm100_persistent", section "Args"; Modular "multistage_gemm_q",
section "Parameters").  The optional epilogue and the block-scaled e4m3
variant (Modular "k_matmul_ragged_paged_scale", sections "Args" and the
scales_granularity_mnk parameter) are written here in numpy, in fp64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

BAD_OFFSETS = 1
BAD_EXPERT_ID = 2

_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so beside it (portable flags: x86_64 and aarch64)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
             "-o", tmp, _SRC, "-lm"],
            check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int
        lib.oracle_gmm_bf16.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I]
        lib.oracle_gmm_bf16.restype = I
        lib.oracle_gmm_int4.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I]
        lib.oracle_gmm_int4.restype = I
        lib.oracle_dequant_int4.argtypes = [P, P, P, I, I, I]
        lib.oracle_dequant_int4.restype = None
        lib.oracle_round_bf16_array.argtypes = [P, P, ctypes.c_int64]
        lib.oracle_round_bf16_array.restype = None
        lib.oracle_validate.argtypes = [P, P, I, I, P]
        lib.oracle_validate.restype = I
        _lib = lib
    return _lib


def _ptr(x):
    return None if x is None else x.ctypes.data_as(ctypes.c_void_p)


def _c_u16(x, shape=None):
    x = np.ascontiguousarray(x, dtype=np.uint16)
    if shape is not None:
        assert x.shape == tuple(shape), (x.shape, shape)
    return x


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover - non-Linux
        return os.cpu_count() or 1


@dataclass
class OracleResult:
    c: np.ndarray          # uint16 bf16 bits [rows_alloc, N]; untouched rows keep c_init
    ref32: np.ndarray      # float32 sums (NaN where no active group wrote)
    ref64: np.ndarray | None
    stats: np.ndarray      # uint32 copy of expert_usage_stats after the call
    flags: int             # BAD_OFFSETS | BAD_EXPERT_ID


def round_bf16(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bits, round to nearest even (the oracle's own rounding)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().oracle_round_bf16_array(_ptr(out), _ptr(x), x.size)
    return out


def validate(a_offsets, expert_ids, num_experts: int):
    off = np.ascontiguousarray(a_offsets, dtype=np.uint32)
    ids = np.ascontiguousarray(expert_ids, dtype=np.int32)
    cnt = np.zeros(1, dtype=np.uint32)
    flags = _load().oracle_validate(_ptr(off), _ptr(ids), ids.size, num_experts, _ptr(cnt))
    return flags, int(cnt[0])


def gmm_bf16(a_bits, a_offsets, b_bits, expert_ids, *, c_init=None, stats_init=None,
             want64: bool = False, nthreads: int | None = None) -> OracleResult:
    """Grouped GEMM on bf16 bit arrays: a [rows, K], b [E, N, K]."""
    a = _c_u16(a_bits)
    b = _c_u16(b_bits)
    E, N, K = b.shape
    rows = a.shape[0]
    assert a.shape[1] == K
    off = np.ascontiguousarray(a_offsets, dtype=np.uint32)
    ids = np.ascontiguousarray(expert_ids, dtype=np.int32)
    G = ids.size
    assert off.size == G + 1
    c = (np.zeros((rows, N), np.uint16) if c_init is None
         else np.array(c_init, dtype=np.uint16, copy=True, order="C").reshape(rows, N))
    ref32 = np.full((rows, N), np.nan, np.float32)
    ref64 = np.full((rows, N), np.nan, np.float64) if want64 else None
    stats = (np.zeros(4, np.uint32) if stats_init is None
             else np.array(stats_init, dtype=np.uint32, copy=True))
    flags = _load().oracle_gmm_bf16(
        _ptr(c), _ptr(ref32), _ptr(ref64), _ptr(a), _ptr(off), _ptr(b), _ptr(ids), _ptr(stats),
        G, E, N, K, nthreads or default_threads())
    if flags < 0:
        raise MemoryError("oracle allocation failed")
    return OracleResult(c, ref32, ref64, stats, flags)


def dequant_int4(packed, scales, group_size: int) -> np.ndarray:
    """packed [N, K/8] uint32 + scales [N, K/group_size] bf16 bits -> bf16 bits [N, K]."""
    p = np.ascontiguousarray(packed, dtype=np.uint32)
    s = _c_u16(scales)
    N, kw = p.shape
    K = kw * 8
    assert s.shape == (N, K // group_size)
    w = np.empty((N, K), np.uint16)
    _load().oracle_dequant_int4(_ptr(w), _ptr(p), _ptr(s), N, K, group_size)
    return w


def gmm_int4(a_bits, a_offsets, packed, scales, expert_ids, *, group_size: int = 128,
             c_init=None, stats_init=None, want64: bool = False,
             nthreads: int | None = None) -> OracleResult:
    """4-bit grouped GEMM: packed [E, N, K/8] uint32, scales [E, N, K/group_size] bf16 bits."""
    a = _c_u16(a_bits)
    p = np.ascontiguousarray(packed, dtype=np.uint32)
    s = _c_u16(scales)
    E, N, kw = p.shape
    K = kw * 8
    rows = a.shape[0]
    assert a.shape[1] == K and s.shape == (E, N, K // group_size)
    off = np.ascontiguousarray(a_offsets, dtype=np.uint32)
    ids = np.ascontiguousarray(expert_ids, dtype=np.int32)
    G = ids.size
    assert off.size == G + 1
    c = (np.zeros((rows, N), np.uint16) if c_init is None
         else np.array(c_init, dtype=np.uint16, copy=True, order="C").reshape(rows, N))
    ref32 = np.full((rows, N), np.nan, np.float32)
    ref64 = np.full((rows, N), np.nan, np.float64) if want64 else None
    stats = (np.zeros(4, np.uint32) if stats_init is None
             else np.array(stats_init, dtype=np.uint32, copy=True))
    flags = _load().oracle_gmm_int4(
        _ptr(c), _ptr(ref32), _ptr(ref64), _ptr(a), _ptr(off), _ptr(p), _ptr(s), _ptr(ids),
        _ptr(stats), G, E, N, K, group_size, nthreads or default_threads())
    if flags == -2:
        raise ValueError("K must be a multiple of 8 and of group_size")
    if flags < 0:
        raise MemoryError("oracle allocation failed")
    return OracleResult(c, ref32, ref64, stats, flags)


# ---------------------------------------------------------------- optional epilogue
# The grouped and quantised GEMM pages both take an optional elementwise function of
# the output (Modular "grouped_matmul_sm100_persistent" and "multistage_gemm_q",
# section "Parameters", elementwise_lambda_fn).  The library offers the common MoE
# steps instead of a function:  y = act(ref[r, n] + bias[e, n]) * row_scale[r], with e
# the expert of row r's group; C = bf16(y).  Rows outside active groups are untouched.

def activation_ref(name: str, y: np.ndarray) -> np.ndarray:
    """The activations, written from their definitions (fp64)."""
    y = np.asarray(y, dtype=np.float64)
    if name == "none":
        return y
    if name == "relu":
        return np.maximum(y, 0.0)
    if name == "silu":                      # y * sigmoid(y)
        return y / (1.0 + np.exp(-y))
    if name == "gelu_tanh":                 # the tanh form of GELU (Hendrycks and Gimpel)
        return 0.5 * y * (1.0 + np.tanh(np.sqrt(2.0 / np.pi) * (y + 0.044715 * y ** 3)))
    raise ValueError(f"unknown activation {name!r}")


def apply_epilogue(res: OracleResult, a_offsets, expert_ids, num_experts: int, *, bias_bits=None,
                   row_scale=None, activation: str = "none") -> OracleResult:
    """The optional epilogue on an oracle result: returns C with it applied to the rows
    of active groups, and `ref32` = y (fp32) there, for the comparison."""
    off = np.asarray(a_offsets, dtype=np.int64)
    ids = np.asarray(expert_ids, dtype=np.int64)
    c = res.c.copy()
    ref = res.ref32.copy()
    if res.flags & BAD_OFFSETS:
        return OracleResult(c, ref, res.ref64, res.stats, res.flags)
    bias = None if bias_bits is None else bf16_bits_to_f32(bias_bits).astype(np.float64)
    scale = None if row_scale is None else np.asarray(row_scale, dtype=np.float64)
    for g, e in enumerate(ids):
        if not (0 <= e < num_experts) or off[g + 1] <= off[g]:
            continue
        r0, r1 = off[g], off[g + 1]
        y = res.ref32[r0:r1].astype(np.float64)
        if bias is not None:
            y = y + bias[e][None, :]
        y = activation_ref(activation, y)
        if scale is not None:
            y = y * scale[r0:r1, None]
        ref[r0:r1] = y.astype(np.float32)
        c[r0:r1] = round_bf16(ref[r0:r1])
    return OracleResult(c, ref, res.ref64, res.stats, res.flags)


def bf16_bits_to_f32(bits) -> np.ndarray:
    """bf16 bit patterns -> fp32 (exact: bf16 is the top half of an fp32)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------- FP8 (e4m3) scaled variant
# The scaled ragged matmul page (Modular "k_matmul_ragged_paged_scale", section "Args":
# input_scale and weight_scale are multiplied to the input and to the weight; template
# parameter scales_granularity_mnk) scales both operands in blocks of a given (m, n, k)
# granularity.  The page prints no formula; the reading taken here is the usual one for
# block-scaled low-precision GEMMs: input_scale holds one value per gm rows and gk
# columns of A, weight_scale one per gn rows and gk columns of each expert's weight, and
#     ref[r, n] = sum_kb input_scale[r // gm, kb] * weight_scale[e, n // gn, kb]
#                        * sum_{k in block kb} a8[r, k] * w8[e, n, k]
# with kb = k // gk.  Offsets, expert ids, skipped groups, untouched rows and
# expert_usage_stats follow the bf16 grouped GEMM exactly.

def e4m3_to_f32(bits) -> np.ndarray:
    """e4m3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; no infinities,
    S.1111.111 is NaN) bit patterns -> fp32, from the format's definition."""
    b = np.asarray(bits, dtype=np.uint8).astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    exp = (b >> 3) & 0xF
    man = b & 0x7
    normal = sign * (1.0 + man / 8.0) * np.power(2.0, exp - 7)
    subnormal = sign * (man / 8.0) * 2.0 ** -6
    out = np.where(exp == 0, subnormal, normal)
    out = np.where((exp == 0xF) & (man == 0x7), np.nan, out)
    return out.astype(np.float32)


def gmm_fp8(a8, a_offsets, w8, expert_ids, input_scale, weight_scale, granularity, *,
            c_init=None, stats_init=None) -> OracleResult:
    """Block-scaled FP8 grouped GEMM.

    a8 [rows, K] and w8 [E, N, K]: e4m3 bit patterns (uint8).  granularity = (gm, gn, gk).
    input_scale fp32 [ceil(rows / gm), ceil(K / gk)]; weight_scale fp32
    [E, ceil(N / gn), ceil(K / gk)].  Sums in fp64 (products of e4m3 values are exact)."""
    gm, gn, gk = (int(x) for x in granularity)
    a = e4m3_to_f32(a8).astype(np.float64)
    w = e4m3_to_f32(w8).astype(np.float64)
    E, N, K = w.shape
    rows = a.shape[0]
    assert a.shape[1] == K and min(gm, gn, gk) >= 1
    nkb = -(-K // gk)
    isc = np.asarray(input_scale, np.float64).reshape(-(-rows // gm) if rows else 0, nkb)
    wsc = np.asarray(weight_scale, np.float64).reshape(E, -(-N // gn), nkb)
    off = np.asarray(a_offsets, dtype=np.int64)
    ids = np.asarray(expert_ids, dtype=np.int64)
    flags, active = validate(a_offsets, expert_ids, E)
    c = (np.zeros((rows, N), np.uint16) if c_init is None
         else np.array(c_init, dtype=np.uint16, copy=True, order="C").reshape(rows, N))
    ref32 = np.full((rows, N), np.nan, np.float32)
    ref64 = np.full((rows, N), np.nan, np.float64)
    stats = (np.zeros(4, np.uint32) if stats_init is None
             else np.array(stats_init, dtype=np.uint32, copy=True))
    stats[1] = active
    if flags & BAD_OFFSETS:
        return OracleResult(c, ref32, ref64, stats, flags)
    ncol = np.arange(N) // gn
    for g, e in enumerate(ids):
        r0, r1 = int(off[g]), int(off[g + 1])
        if not (0 <= e < E) or r1 <= r0:
            continue
        mrow = np.arange(r0, r1) // gm
        y = np.zeros((r1 - r0, N), np.float64)
        for kb in range(nkb):
            ks = slice(kb * gk, min(K, (kb + 1) * gk))
            part = a[r0:r1, ks] @ w[e][:, ks].T
            y += part * isc[mrow, kb][:, None] * wsc[e][ncol, kb][None, :]
        ref64[r0:r1] = y
        ref32[r0:r1] = y.astype(np.float32)
        c[r0:r1] = round_bf16(ref32[r0:r1])
    return OracleResult(c, ref32, ref64, stats, flags)


# ---------------------------------------------------------------- A-plane row offsetting
# The grouped GEMM page's a_plane_splits parameter (Modular "grouped_matmul_sm100_persistent",
# section "Parameters": per-plane split sizes for fused LoRA QKV A-plane row offsetting;
# (0, 0) disables it).  The reading taken: A holds three planes of M = a_offsets[G] rows
# stacked along its rows (the q, k and v inputs of a fused QKV projection), the split
# sizes (s0, s1) cut the N columns of C and B into the q, k and v parts, and column n
# reads the plane p(n) its part belongs to:
#     ref[r, n] = sum_k A[p(n) * M + r, k] * B[e, n, k],
#     p(n) = 0 for n < s0, 1 for s0 <= n < s0 + s1, 2 otherwise.

def plane_of_columns(N: int, splits) -> np.ndarray:
    """p(n) for n in [0, N): the plane each output column reads (all 0 when splits = (0, 0))."""
    s0, s1 = (int(x) for x in splits)
    n = np.arange(N)
    if s0 == 0 and s1 == 0:
        return np.zeros(N, np.int64)
    return (n >= s0).astype(np.int64) + (n >= s0 + s1).astype(np.int64)


def gmm_bf16_planes(a_bits, a_offsets, b_bits, expert_ids, splits, *, c_init=None,
                    stats_init=None, nthreads: int | None = None) -> OracleResult:
    """The grouped GEMM with A-plane row offsetting: the bf16 oracle run once per plane on
    that plane's rows of A and its columns of B, the results put in their columns of C."""
    a = np.asarray(a_bits, np.uint16)
    b = np.asarray(b_bits, np.uint16)
    E, N, K = b.shape
    off = np.asarray(a_offsets, np.uint32)
    M = int(off[-1]) if off.size else 0
    planes = plane_of_columns(N, splits)
    first = gmm_bf16(a[:M] if M else a, a_offsets, b[:, :0, :] if N == 0 else b[:, :1, :], expert_ids,
                     stats_init=stats_init, nthreads=nthreads)   # flags and stats only
    rows = M
    c = (np.zeros((rows, N), np.uint16) if c_init is None
         else np.array(c_init, dtype=np.uint16, copy=True)[:rows].reshape(rows, N))
    ref32 = np.full((rows, N), np.nan, np.float32)
    for p in range(3):
        cols = np.flatnonzero(planes == p)
        if cols.size == 0:
            continue
        part = gmm_bf16(a[p * M:(p + 1) * M], a_offsets, b[:, cols, :], expert_ids,
                        c_init=c[:, cols], nthreads=nthreads)
        c[:, cols] = part.c
        ref32[:, cols] = part.ref32
    if c_init is not None:
        full = np.array(c_init, dtype=np.uint16, copy=True)
        full[:rows] = c
        c = full
        r32 = np.full(full.shape, np.nan, np.float32)
        r32[:rows] = ref32
        ref32 = r32
    return OracleResult(c, ref32, None, first.stats, first.flags)
