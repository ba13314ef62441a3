"""Thin ctypes binding over libgmm.so (the C ABI in include/gmm.h).

Argument marshalling only: every step of the grouped GEMM runs in the CUDA
kernels of libgmm.so.  If the library is missing this module raises; there is
no fallback of any kind.  The functions keep the C names:

    h = gmm_create(num_experts, device)
    gmm_run(h, c, a, a_offsets, b, expert_ids, expert_usage_stats)
    gmm_run_int4(h, c, a, a_offsets, b_packed, b_scales, expert_ids, expert_usage_stats, group_size)
    gmm_query_status(h)            # syncs the stream; returns the code
    gmm_error_string(code)
    gmm_destroy(h)

Tensors are torch CUDA tensors: c/a/b bf16, a_offsets uint32 (or int32 holding
the same bits), expert_ids int32, expert_usage_stats uint32/int32 with at least
2 entries, b_packed int32/uint32 words, b_scales bf16.  `stream` defaults to
torch's current stream on the handle's device.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

GMM_OK = 0
GMM_ERR_INVALID_ARG = -1
GMM_ERR_UNSUPPORTED = -2
GMM_ERR_CUDA = -3
GMM_ERR_DEVICE_TIMEOUT = -4
GMM_ERR_BAD_INPUT = -5
GMM_ERR_NO_DEVICE = -6

EXPORTED = ("gmm_create", "gmm_run", "gmm_run_ex", "gmm_run_int4", "gmm_run_int4_ex", "gmm_matmul_int4",
            "gmm_run_fp8", "gmm_run_planes", "gmm_run_noalloc", "gmm_query_status", "gmm_error_string", "gmm_destroy")

# Activations of the optional epilogue (GMM_ACT_* in gmm.h).
GMM_ACT_NONE = 0
GMM_ACT_RELU = 1
GMM_ACT_SILU = 2
GMM_ACT_GELU_TANH = 3
ACTIVATIONS = {"none": GMM_ACT_NONE, "relu": GMM_ACT_RELU, "silu": GMM_ACT_SILU, "gelu_tanh": GMM_ACT_GELU_TANH}


class GmmEpilogue(ctypes.Structure):
    """gmm_epilogue: y = act(acc + bias[e, n]) * row_scale[r] before the bf16 store."""
    _fields_ = [("bias", ctypes.c_void_p), ("row_scale", ctypes.c_void_p), ("activation", ctypes.c_int)]

_lib = None


class GmmError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {gmm_error_string(code)} ({code})")
        self.code = code


def library_path() -> str:
    return _build.LIB_PATH


def load_library(path: str | None = None):
    """Load libgmm.so (raises RuntimeError if it is not built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    path = path or library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library {path} is not built; call ragged_matmul_gb300.build.build()")
    lib = ctypes.CDLL(path)
    P, I = ctypes.c_void_p, ctypes.c_int
    lib.gmm_create.argtypes = [ctypes.POINTER(P), I, I]
    lib.gmm_create.restype = I
    lib.gmm_run.argtypes = [P, P, P, P, P, P, P, I, I, I, P]
    lib.gmm_run.restype = I
    lib.gmm_run_int4.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, P]
    lib.gmm_run_int4.restype = I
    EP = ctypes.POINTER(GmmEpilogue)
    lib.gmm_run_ex.argtypes = [P, P, P, P, P, P, P, I, I, I, EP, P]
    lib.gmm_run_ex.restype = I
    lib.gmm_run_int4_ex.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, EP, P]
    lib.gmm_run_int4_ex.restype = I
    lib.gmm_matmul_int4.argtypes = [P, P, P, P, P, I, I, I, I, EP, P]
    lib.gmm_run_planes.restype = I
    lib.gmm_run_planes.argtypes = [P, P, P, P, P, P, P, I, I, I, P, EP, P]
    lib.gmm_run_fp8.restype = I
    lib.gmm_run_fp8.argtypes = [P, P, P, P, P, P, P, I, I, I, P, P, P, EP, P]
    lib.gmm_matmul_int4.restype = I
    lib.gmm_run_noalloc.argtypes = [P, P, P, P, P, P, I, I, I, I, P]
    lib.gmm_run_noalloc.restype = I
    lib.gmm_query_status.argtypes = [P, P]
    lib.gmm_query_status.restype = I
    lib.gmm_error_string.argtypes = [I]
    lib.gmm_error_string.restype = ctypes.c_char_p
    lib.gmm_destroy.argtypes = [P]
    lib.gmm_destroy.restype = I
    if path == library_path():
        _lib = lib
    return lib


def gmm_error_string(code: int) -> str:
    return load_library().gmm_error_string(int(code)).decode()


class Handle:
    """Owns a gmm_handle_t; released by gmm_destroy or at garbage collection."""

    def __init__(self, ptr: int, device: int, num_experts: int):
        self.ptr = ptr
        self.device = device
        self.num_experts = num_experts

    def __del__(self):
        try:
            gmm_destroy(self)
        except Exception:
            pass


def gmm_create(num_experts: int, device: int | None = None) -> Handle:
    import torch
    if device is None:
        device = torch.cuda.current_device()
    h = ctypes.c_void_p()
    rc = load_library().gmm_create(ctypes.byref(h), int(num_experts), int(device))
    if rc != GMM_OK:
        raise GmmError(rc, "gmm_create")
    return Handle(h.value, int(device), int(num_experts))


def gmm_destroy(h: Handle) -> None:
    if h is not None and h.ptr:
        ptr, h.ptr = h.ptr, None
        rc = load_library().gmm_destroy(ptr)
        if rc != GMM_OK:
            raise GmmError(rc, "gmm_destroy")


def stream_handle(device: int, stream=None) -> ctypes.c_void_p:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream))


def _check(t, name, dtypes, device, min_numel=0):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda" or t.device.index != device:
        raise ValueError(f"{name} must live on cuda:{device}")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.numel() < min_numel:
        raise ValueError(f"{name} needs at least {min_numel} elements")
    return ctypes.c_void_p(t.data_ptr())


def _i32_types():
    import torch
    return (torch.int32,) + ((torch.uint32,) if hasattr(torch, "uint32") else ())


def _routing_args(h, a_offsets, expert_ids, stats):
    import torch
    G = expert_ids.numel()
    return (_check(a_offsets, "a_offsets", _i32_types(), h.device, G + 1),
            _check(expert_ids, "expert_ids", (torch.int32,), h.device),
            _check(stats, "expert_usage_stats", _i32_types(), h.device, 2), G)


def _epilogue(h: Handle, rows: int, N: int, bias, row_scale, activation) -> GmmEpilogue:
    """Marshal the optional epilogue's operands (checked like the others)."""
    import torch
    act = ACTIVATIONS[activation] if isinstance(activation, str) else int(activation)
    pb = None
    if bias is not None:
        if tuple(bias.shape) != (h.num_experts, N):
            raise ValueError(f"bias must be [E, N] = [{h.num_experts}, {N}], got {tuple(bias.shape)}")
        pb = _check(bias, "bias", (torch.bfloat16,), h.device).value
    ps = None
    if row_scale is not None:
        if row_scale.dim() != 1 or row_scale.numel() < rows:
            raise ValueError(f"row_scale must be 1-D with at least {rows} entries")
        ps = _check(row_scale, "row_scale", (torch.float32,), h.device).value
    return GmmEpilogue(pb, ps, act)


def gmm_run(h: Handle, c, a, a_offsets, b, expert_ids, expert_usage_stats, stream=None,
            check: bool = True) -> int:
    """C[r, :] = A[r, :] @ B[expert_ids[g]].T for rows of active groups (asynchronous)."""
    return gmm_run_ex(h, c, a, a_offsets, b, expert_ids, expert_usage_stats, stream=stream, check=check)


def gmm_run_ex(h: Handle, c, a, a_offsets, b, expert_ids, expert_usage_stats, bias=None, row_scale=None,
               activation=GMM_ACT_NONE, stream=None, check: bool = True) -> int:
    """gmm_run with the optional epilogue y = act(acc + bias[e, n]) * row_scale[r] (asynchronous)."""
    import torch
    if a.dim() != 2 or b.dim() != 3 or c.dim() != 2:
        raise ValueError("a must be [rows, K], b [E, N, K], c [rows, N]")
    E, N, K = b.shape
    if a.shape[1] != K or c.shape[1] != N or c.shape[0] != a.shape[0] or E != h.num_experts:
        raise ValueError(f"shape mismatch: a {tuple(a.shape)}, b {tuple(b.shape)}, c {tuple(c.shape)}, "
                         f"handle E={h.num_experts}")
    bf = (torch.bfloat16,)
    pc = _check(c, "c", bf, h.device)
    pa = _check(a, "a", bf, h.device)
    pb = _check(b, "b", bf, h.device)
    po, pi, ps, G = _routing_args(h, a_offsets, expert_ids, expert_usage_stats)
    lib = load_library()
    if bias is None and row_scale is None and not activation:
        rc = lib.gmm_run(h.ptr, pc, pa, po, pb, pi, ps, G, N, K, stream_handle(h.device, stream))
    else:
        epi = _epilogue(h, a.shape[0], N, bias, row_scale, activation)
        rc = lib.gmm_run_ex(h.ptr, pc, pa, po, pb, pi, ps, G, N, K, ctypes.byref(epi),
                            stream_handle(h.device, stream))
    if check and rc != GMM_OK:
        raise GmmError(rc, "gmm_run")
    return rc


def gmm_run_int4(h: Handle, c, a, a_offsets, b_packed, b_scales, expert_ids, expert_usage_stats,
                 group_size: int = 128, stream=None, check: bool = True) -> int:
    """4-bit variant: b_packed [E, N, K/8] 32-bit words, b_scales [E, N, K/group_size] bf16."""
    return gmm_run_int4_ex(h, c, a, a_offsets, b_packed, b_scales, expert_ids, expert_usage_stats,
                           group_size=group_size, stream=stream, check=check)


def gmm_run_int4_ex(h: Handle, c, a, a_offsets, b_packed, b_scales, expert_ids, expert_usage_stats,
                    group_size: int = 128, bias=None, row_scale=None, activation=GMM_ACT_NONE, stream=None,
                    check: bool = True) -> int:
    """gmm_run_int4 with the optional epilogue y = act(acc + bias[e, n]) * row_scale[r]."""
    import torch
    if a.dim() != 2 or b_packed.dim() != 3 or c.dim() != 2 or b_scales.dim() != 3:
        raise ValueError("a must be [rows, K], b_packed [E, N, K/8], b_scales [E, N, K/gs], c [rows, N]")
    E, N, KW = b_packed.shape
    K = KW * 8
    if (a.shape[1] != K or c.shape[1] != N or c.shape[0] != a.shape[0] or E != h.num_experts
            or group_size <= 0 or tuple(b_scales.shape) != (E, N, K // group_size)):
        raise ValueError("shape mismatch between a, b_packed, b_scales, c")
    bf = (torch.bfloat16,)
    pc = _check(c, "c", bf, h.device)
    pa = _check(a, "a", bf, h.device)
    pq = _check(b_packed, "b_packed", _i32_types(), h.device)
    psc = _check(b_scales, "b_scales", bf, h.device)
    po, pi, ps, G = _routing_args(h, a_offsets, expert_ids, expert_usage_stats)
    lib = load_library()
    if bias is None and row_scale is None and not activation:
        rc = lib.gmm_run_int4(h.ptr, pc, pa, po, pq, psc, pi, ps, G, N, K, int(group_size),
                              stream_handle(h.device, stream))
    else:
        epi = _epilogue(h, a.shape[0], N, bias, row_scale, activation)
        rc = lib.gmm_run_int4_ex(h.ptr, pc, pa, po, pq, psc, pi, ps, G, N, K, int(group_size), ctypes.byref(epi),
                                 stream_handle(h.device, stream))
    if check and rc != GMM_OK:
        raise GmmError(rc, "gmm_run_int4")
    return rc


def gmm_run_planes(h: Handle, c, a, a_offsets, b, expert_ids, expert_usage_stats, a_plane_splits=(0, 0),
                   bias=None, row_scale=None, activation=GMM_ACT_NONE, stream=None, check: bool = True) -> int:
    """bf16 grouped GEMM with A-plane row offsetting: a holds three planes of a_offsets[G] rows
    ([3 * rows, K] with rows = c.shape[0]); output columns n < s0 read plane 0, n < s0 + s1
    plane 1, the rest plane 2 (s0, s1 multiples of 256); then the optional epilogue."""
    import torch
    if a.dim() != 2 or b.dim() != 3 or c.dim() != 2:
        raise ValueError("a must be [3 * rows, K], b [E, N, K], c [rows, N]")
    E, N, K = b.shape
    s0, s1 = (int(x) for x in a_plane_splits)
    planes = 1 if (s0, s1) == (0, 0) else 3
    if a.shape[1] != K or c.shape[1] != N or a.shape[0] < planes * c.shape[0] or E != h.num_experts:
        raise ValueError(f"shape mismatch: a {tuple(a.shape)} (needs {planes} planes of {c.shape[0]} rows), "
                         f"b {tuple(b.shape)}, c {tuple(c.shape)}, handle E={h.num_experts}")
    bf = (torch.bfloat16,)
    pc = _check(c, "c", bf, h.device)
    pa = _check(a, "a", bf, h.device)
    pb = _check(b, "b", bf, h.device)
    po, pi, ps, G = _routing_args(h, a_offsets, expert_ids, expert_usage_stats)
    splits = (ctypes.c_int * 2)(s0, s1)
    epi = None
    if bias is not None or row_scale is not None or activation:
        epi = ctypes.byref(_epilogue(h, c.shape[0], N, bias, row_scale, activation))
    rc = load_library().gmm_run_planes(h.ptr, pc, pa, po, pb, pi, ps, G, N, K, splits, epi,
                                       stream_handle(h.device, stream))
    if check and rc != GMM_OK:
        raise GmmError(rc, "gmm_run_planes")
    return rc


def _fp8_types():
    import torch
    return (torch.uint8,) + ((torch.float8_e4m3fn,) if hasattr(torch, "float8_e4m3fn") else ())


def gmm_run_fp8(h: Handle, c, a, a_offsets, b, expert_ids, expert_usage_stats, input_scale, weight_scale,
                scales_granularity_mnk=(1, 128, None), bias=None, row_scale=None, activation=GMM_ACT_NONE,
                stream=None, check: bool = True) -> int:
    """Block-scaled e4m3 grouped GEMM: a [rows, K] and b [E, N, K] e4m3 (uint8 bit patterns or
    float8_e4m3fn), input_scale fp32 [ceil(rows / gm), ...], weight_scale fp32 [E, ceil(N / gn), ...]
    with (gm, gn, gk) = scales_granularity_mnk (gk None: K); then the optional epilogue."""
    import torch
    if a.dim() != 2 or b.dim() != 3 or c.dim() != 2:
        raise ValueError("a must be [rows, K], b [E, N, K], c [rows, N]")
    E, N, K = b.shape
    rows = a.shape[0]
    if a.shape[1] != K or c.shape[1] != N or c.shape[0] != rows or E != h.num_experts:
        raise ValueError(f"shape mismatch: a {tuple(a.shape)}, b {tuple(b.shape)}, c {tuple(c.shape)}, "
                         f"handle E={h.num_experts}")
    gm, gn, gk = scales_granularity_mnk
    gk = K if gk is None else gk
    gran = (ctypes.c_int * 3)(int(gm), int(gn), int(gk))
    nkb = -(-K // gk) if gk > 0 else 0
    if gm > 0 and input_scale.numel() != -(-rows // gm) * nkb:
        raise ValueError(f"input_scale needs ceil(rows / gm) * ceil(K / gk) = {-(-rows // gm) * nkb} entries")
    if gn > 0 and (weight_scale.shape[0] != E or weight_scale.numel() != E * -(-N // gn) * nkb):
        raise ValueError(f"weight_scale must be [E, ceil(N / gn), ceil(K / gk)] = [{E}, {-(-N // gn)}, {nkb}]")
    pc = _check(c, "c", (torch.bfloat16,), h.device)
    pa = _check(a, "a", _fp8_types(), h.device)
    pb = _check(b, "b", _fp8_types(), h.device)
    pis = _check(input_scale, "input_scale", (torch.float32,), h.device)
    pws = _check(weight_scale, "weight_scale", (torch.float32,), h.device)
    po, pi, ps, G = _routing_args(h, a_offsets, expert_ids, expert_usage_stats)
    epi = None
    if bias is not None or row_scale is not None or activation:
        epi = ctypes.byref(_epilogue(h, rows, N, bias, row_scale, activation))
    rc = load_library().gmm_run_fp8(h.ptr, pc, pa, po, pb, pi, ps, G, N, K, pis, pws, gran, epi,
                                    stream_handle(h.device, stream))
    if check and rc != GMM_OK:
        raise GmmError(rc, "gmm_run_fp8")
    return rc


def gmm_matmul_int4(h: Handle, c, a, b_packed, b_scales, group_size: int = 128, bias=None, row_scale=None,
                    activation=GMM_ACT_NONE, stream=None, check: bool = True) -> int:
    """Dense 4-bit GEMM C = A . w^T (Modular "multistage_gemm_q"): a [M, K] bf16,
    b_packed [N, K/8] 32-bit words, b_scales [N, K/group_size] bf16, c [M, N] bf16.
    Raises ValueError when an operand is not rank-2, as the page's function does.
    `bias` (if given) is [1, N] bf16: the single expert's row."""
    import torch
    for name, t_ in (("c", c), ("a", a), ("b_packed", b_packed), ("b_scales", b_scales)):
        if t_.dim() != 2:
            raise ValueError(f"{name} must be rank-2, got rank {t_.dim()}")
    M, K = a.shape
    N, KW = b_packed.shape
    if KW * 8 != K or tuple(c.shape) != (M, N) or group_size <= 0 or tuple(b_scales.shape) != (N, K // group_size):
        raise ValueError(f"shape mismatch: a {tuple(a.shape)}, b_packed {tuple(b_packed.shape)}, "
                         f"b_scales {tuple(b_scales.shape)}, c {tuple(c.shape)}")
    bf = (torch.bfloat16,)
    pc = _check(c, "c", bf, h.device)
    pa = _check(a, "a", bf, h.device)
    pq = _check(b_packed, "b_packed", _i32_types(), h.device)
    psc = _check(b_scales, "b_scales", bf, h.device)
    epi = None
    if bias is not None or row_scale is not None or activation:
        pb = None
        if bias is not None:
            if tuple(bias.shape) != (1, N):
                raise ValueError(f"bias must be [1, {N}]")
            pb = _check(bias, "bias", bf, h.device).value
        ps = None
        if row_scale is not None:
            if row_scale.dim() != 1 or row_scale.numel() < M:
                raise ValueError(f"row_scale must be 1-D with at least {M} entries")
            ps = _check(row_scale, "row_scale", (torch.float32,), h.device).value
        act = ACTIVATIONS[activation] if isinstance(activation, str) else int(activation)
        epi = ctypes.byref(GmmEpilogue(pb, ps, act))
    rc = load_library().gmm_matmul_int4(h.ptr, pc, pa, pq, psc, M, N, K, int(group_size), epi,
                                        stream_handle(h.device, stream))
    if check and rc != GMM_OK:
        raise GmmError(rc, "gmm_matmul_int4")
    return rc


def gmm_query_status(h: Handle, stream=None) -> int:
    return load_library().gmm_query_status(h.ptr, stream_handle(h.device, stream))
