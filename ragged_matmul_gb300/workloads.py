"""Seeded synthetic inputs for the ragged grouped GEMM.

This module builds routing (per-group row counts, expert ids, the a_offsets
prefix array) and operand values.  It holds none of the grouped GEMM's
arithmetic: it is shared by the tests, the smoke check and the bench so that
the CUDA path and the CPU oracle see the same inputs.

Named workloads (sizes and value distributions of the mixture-of-experts
shapes this library targets):

  tiny          E=4, N=K=256, rows per group [3, 17, 0, 40], expert ids
                [2, 0, -1, 3]; A, B ~ U[-1, 1].
  decode        256 tokens routed top-8 over E=64 experts: 2048 rows with
                Multinomial(2048, p_e ~ (e+1)^-1.1) loads, one group per expert
                (empty groups kept), K=2048, N=2816; A, B ~ N(0, 0.02).
  prefill       16384 tokens top-2 over E=8: 32768 rows, each expert within
                +-10% of 4096, K=4096, N=14336; A ~ N(0, 1), B ~ N(0, 0.02).
  fine_grained  4096 tokens top-8 over E=128: 32768 rows with
                Multinomial(32768, p_e ~ (e+1)^-1.0) loads, K=7168, N=4096;
                13 of 128 groups (chosen by a seeded permutation) carry expert
                id -1; A ~ N(0, 1), B ~ N(0, 0.02).
  int4          E=64, 8192 rows with uniform Multinomial routing, K=N=4096;
                B packed 8 unsigned 4-bit values per uint32 along K (low
                nibble first), zero point 8, one bf16 scale per 128 K elements,
                scales ~ U[0.005, 0.02]; A ~ N(0, 1).
  int4_dense    the int4 workload as one dense problem: E=1, one group of 8192
                rows, K=N=4096.
  fp8_prefill,  the prefill / decode routings and shapes with e4m3 operands:
  fp8_decode    A, B ~ e4m3(N(0, 2)) (the fp32 draw cast to e4m3, round to
                nearest even), fp32 scales at granularity (1, 128, K):
                input_scale ~ U[0.25, 1], weight_scale ~ U[0.002, 0.008].
  lora_qkv      a fused LoRA QKV expand with A-plane row offsetting: 8192 tokens
                over E=8 adapters (uniform Multinomial), K=64, N=6144 with splits
                (4096, 1024); A [3 x 8192, 64] ~ N(0, 1), B ~ N(0, 0.02).
  fp8_block_prefill,  the same with per-K-block scales: granularity
  fp8_block_decode    (1, 128, 128), one scale per row (input) or per 128
                weight rows (weight) and 128 of K.

Values are drawn in fp32 and rounded to bf16 (round to nearest even).  Host
generation uses numpy's PCG64 (``default_rng``); device generation, used for
the large shapes, uses torch's CUDA generator with the same seed.  The two
give different (equally distributed) values; each caller sticks to one.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import numpy as np

SENTINEL_BF16 = 0x7FA5          # a NaN payload no kernel produces; marks rows that must stay untouched
SENTINEL_STATS = 0xFFFFFFFF
TILE_ROWS_HINT = 128            # only used to size "several tiles" test shapes


@dataclass(frozen=True)
class Routing:
    name: str
    E: int
    N: int
    K: int
    loads: np.ndarray           # int64 [G] rows per group
    expert_ids: np.ndarray      # int32 [G]
    a_offsets: np.ndarray       # uint32 [G+1]
    a_dist: tuple               # ("normal", std) or ("uniform", lo, hi)
    b_dist: tuple
    int4: bool = False
    group_size: int = 128
    scale_range: tuple = (0.005, 0.02)
    meta: dict = field(default_factory=dict)

    @property
    def G(self) -> int:
        return int(self.expert_ids.size)

    @property
    def rows(self) -> int:
        """Rows of A and C (the allocation): the end of the last group."""
        return int(self.a_offsets[-1]) if self.a_offsets.size else 0

    def active_mask(self) -> np.ndarray:
        return (self.expert_ids >= 0) & (self.expert_ids < self.E)


def offsets_from_loads(loads, base: int = 0) -> np.ndarray:
    loads = np.asarray(loads, dtype=np.int64)
    off = np.empty(loads.size + 1, dtype=np.int64)
    off[0] = base
    off[1:] = base + np.cumsum(loads)
    assert off[-1] < 2**32
    return off.astype(np.uint32)


def make_routing(name, E, N, K, loads, expert_ids, *, a_dist=("uniform", -1.0, 1.0),
                 b_dist=("uniform", -1.0, 1.0), base: int = 0, int4: bool = False,
                 group_size: int = 128, scale_range=(0.005, 0.02), a_offsets=None) -> Routing:
    loads = np.asarray(loads, dtype=np.int64)
    ids = np.asarray(expert_ids, dtype=np.int32)
    assert loads.size == ids.size
    off = offsets_from_loads(loads, base) if a_offsets is None else np.asarray(a_offsets, np.uint32)
    return Routing(name, int(E), int(N), int(K), loads, ids, off, tuple(a_dist),
                   None if b_dist is None else tuple(b_dist), int4, int(group_size), tuple(scale_range))


def _zipf_loads(rng, total, E, s):
    p = (np.arange(1, E + 1, dtype=np.float64)) ** (-s)
    p /= p.sum()
    return rng.multinomial(total, p).astype(np.int64)


def _balanced_loads(rng, total, E, spread):
    base = total // E
    u = rng.uniform(-spread, spread, size=E)
    loads = np.rint(base * (1.0 + u)).astype(np.int64)
    lo, hi = int(np.ceil(base * (1 - spread))), int(np.floor(base * (1 + spread)))
    loads = np.clip(loads, lo, hi)
    diff = total - int(loads.sum())
    e = 0
    while diff != 0:                      # spread the residual +-1 round robin, staying in range
        step = 1 if diff > 0 else -1
        if lo <= loads[e] + step <= hi:
            loads[e] += step
            diff -= step
        e = (e + 1) % E
    return loads


WORKLOAD_NAMES = ("tiny", "decode", "prefill", "fine_grained", "int4", "int4_dense", "fp8_prefill",
                  "fp8_decode", "fp8_block_prefill", "fp8_block_decode", "lora_qkv")
WORKLOAD_SEEDS = {name: i for i, name in enumerate(WORKLOAD_NAMES)}


def routing(name: str, seed: int | None = None) -> Routing:
    """Routing of one named workload; the seed defaults to the workload's index."""
    if seed is None:
        seed = WORKLOAD_SEEDS[name]
    rng = np.random.default_rng([seed, 0])
    if name == "tiny":
        return make_routing("tiny", 4, 256, 256, [3, 17, 0, 40], [2, 0, -1, 3],
                            a_dist=("uniform", -1.0, 1.0), b_dist=("uniform", -1.0, 1.0))
    if name == "decode":
        E = 64
        loads = _zipf_loads(rng, 2048, E, 1.1)
        return make_routing("decode", E, 2816, 2048, loads, np.arange(E),
                            a_dist=("normal", 0.02), b_dist=("normal", 0.02))
    if name == "prefill":
        E = 8
        loads = _balanced_loads(rng, 32768, E, 0.10)
        return make_routing("prefill", E, 14336, 4096, loads, np.arange(E),
                            a_dist=("normal", 1.0), b_dist=("normal", 0.02))
    if name == "fine_grained":
        E = 128
        loads = _zipf_loads(rng, 32768, E, 1.0)
        ids = np.arange(E, dtype=np.int32)
        skipped = rng.permutation(E)[: int(round(0.1 * E))]
        ids[skipped] = -1
        return make_routing("fine_grained", E, 4096, 7168, loads, ids,
                            a_dist=("normal", 1.0), b_dist=("normal", 0.02))
    if name == "int4":
        E = 64
        loads = rng.multinomial(8192, np.full(E, 1.0 / E)).astype(np.int64)
        return make_routing("int4", E, 4096, 4096, loads, np.arange(E),
                            a_dist=("normal", 1.0), b_dist=None, int4=True, group_size=128,
                            scale_range=(0.005, 0.02))
    if name == "int4_dense":
        # The dense quantised GEMM (one expert, one group): the int4 workload's rows,
        # shapes and value distributions as a single 8192 x 4096 x 4096 problem.
        return make_routing("int4_dense", 1, 4096, 4096, [8192], [0],
                            a_dist=("normal", 1.0), b_dist=None, int4=True, group_size=128,
                            scale_range=(0.005, 0.02))
    if name in ("fp8_prefill", "fp8_decode"):
        # The scaled e4m3 variant on the prefill / decode routings and shapes; operand
        # values come from fp8_host_values / fp8_device_values.
        base = routing(name[4:], seed)
        return replace(base, name=name, meta={"fp8": True, "granularity": (1, 128, None)})
    if name in ("fp8_block_prefill", "fp8_block_decode"):
        # The same with per-K-block scales: granularity (1, 128, 128).
        base = routing(name[10:], seed)
        return replace(base, name=name, meta={"fp8": True, "granularity": (1, 128, 128)})
    if name == "lora_qkv":
        # A fused LoRA QKV expand: 8192 tokens over 8 adapters (Multinomial, uniform), rank
        # K = 64, N = 4096 (q) + 1024 (k) + 1024 (v) columns; A holds the three planes of
        # the shrink outputs (A-plane row offsetting with splits (4096, 1024)).
        E = 8
        loads = rng.multinomial(8192, np.full(E, 1.0 / E)).astype(np.int64)
        r = make_routing("lora_qkv", E, 6144, 64, loads, np.arange(E),
                         a_dist=("normal", 1.0), b_dist=("normal", 0.02))
        return replace(r, meta={"planes": (4096, 1024)})
    raise KeyError(name)


def a_rows(r: Routing, rows: int | None = None) -> int:
    """Rows of A to allocate: one plane of `rows` (default the end of the last group), or
    three with A-plane row offsetting."""
    rows = r.rows if rows is None else rows
    return 3 * rows if r.meta.get("planes") else rows


def with_rows(r: Routing, total: int, seed: int = 0) -> Routing:
    """The routing redrawn for `total` rows: Multinomial(total, p) over its groups with p
    proportional to its loads (sizes, ids and value distributions kept)."""
    rng = np.random.default_rng([seed, 3])
    p = np.asarray(r.loads, np.float64)
    p = p / p.sum() if p.sum() > 0 else np.full(p.size, 1.0 / p.size)
    loads = rng.multinomial(int(total), p).astype(np.int64)
    return Routing(f"{r.name}@{total}", r.E, r.N, r.K, loads, r.expert_ids.copy(), offsets_from_loads(loads),
                   r.a_dist, r.b_dist, r.int4, r.group_size, r.scale_range, dict(r.meta))


def group_range(r: Routing, lo: int, hi: int) -> Routing:
    """The sub-workload made of groups lo .. hi-1 of r (rows renumbered from 0, E kept)."""
    loads = r.loads[lo:hi].copy()
    ids = r.expert_ids[lo:hi].copy()
    return Routing(f"{r.name}[{lo}:{hi}]", r.E, r.N, r.K, loads, ids, offsets_from_loads(loads), r.a_dist,
                   r.b_dist, r.int4, r.group_size, r.scale_range, dict(r.meta))


def first_groups(r: Routing, G: int) -> Routing:
    """The sub-workload made of the first G groups of r (rows, ids and distributions kept;
    E shrunk to the largest expert id used + 1)."""
    ids = r.expert_ids[:G]
    valid = ids[(ids >= 0) & (ids < r.E)]
    E = int(valid.max()) + 1 if valid.size else 1
    return Routing(f"{r.name}[:{G}]", E, r.N, r.K, r.loads[:G].copy(), ids.copy(),
                   offsets_from_loads(r.loads[:G]), r.a_dist, r.b_dist, r.int4, r.group_size,
                   r.scale_range, dict(r.meta))


# ---------------------------------------------------------------- host values (numpy)

def _to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even, via torch's CPU cast."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def _draw(rng, dist, size):
    if dist[0] == "normal":
        return rng.standard_normal(size, dtype=np.float32) * np.float32(dist[1])
    if dist[0] == "uniform":
        return rng.uniform(dist[1], dist[2], size).astype(np.float32)
    if dist[0] == "int":                     # small integers, exact in bf16
        return rng.integers(dist[1], dist[2] + 1, size).astype(np.float32)
    raise KeyError(dist)


def host_values(r: Routing, seed: int = 0, rows: int | None = None) -> dict:
    """Operands as numpy bf16 bit arrays (uint16) plus the packed 4-bit form when r.int4.

    rows: rows of A to allocate (defaults to the end of the last group).
    """
    rng = np.random.default_rng([seed, 1])
    rows = a_rows(r, rows)
    out = {"a": _to_bf16_bits(_draw(rng, r.a_dist, (rows, r.K)))}
    if r.int4:
        q = rng.integers(0, 16, size=(r.E, r.N, r.K), dtype=np.uint32)
        out["packed"] = pack_nibbles(q)
        lo, hi = r.scale_range
        out["scales"] = _to_bf16_bits(rng.uniform(lo, hi, (r.E, r.N, r.K // r.group_size)))
    else:
        out["b"] = _to_bf16_bits(_draw(rng, r.b_dist, (r.E, r.N, r.K)))
    return out


def pack_nibbles(q: np.ndarray) -> np.ndarray:
    """[..., K] values in [0, 16) -> [..., K/8] uint32, value k%8 at bits 4*(k%8) (storage format)."""
    q = np.asarray(q, dtype=np.uint32)
    assert q.shape[-1] % 8 == 0
    q = q.reshape(*q.shape[:-1], q.shape[-1] // 8, 8)
    words = np.zeros(q.shape[:-1], dtype=np.uint32)
    for i in range(8):
        words |= (q[..., i] & np.uint32(0xF)) << np.uint32(4 * i)
    return words


def sentinel_c(rows: int, N: int) -> np.ndarray:
    return np.full((rows, N), SENTINEL_BF16, dtype=np.uint16)


# ---------------------------------------------------------------- device values (torch CUDA generator)

def device_values(r: Routing, seed: int = 0, device="cuda", chunk_elems: int = 1 << 27) -> dict:
    """Operands generated on the device with torch's seeded CUDA generator.

    Returns torch tensors: a bf16 [rows, K]; b bf16 [E, N, K] or packed int32 [E, N, K/8]
    (bit pattern of the uint32 words) and scales bf16 [E, N, K/group_size].
    """
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1000003 + 17)

    def fill(shape, dist):
        out = torch.empty(shape, dtype=torch.bfloat16, device=device)
        flat = out.view(-1)
        for s in range(0, flat.numel(), chunk_elems):
            n = min(chunk_elems, flat.numel() - s)
            if dist[0] == "normal":
                x = torch.randn(n, generator=g, device=device, dtype=torch.float32) * dist[1]
            elif dist[0] == "uniform":
                x = torch.rand(n, generator=g, device=device, dtype=torch.float32)
                x = x * (dist[2] - dist[1]) + dist[1]
            else:
                raise KeyError(dist)
            flat[s:s + n] = x.to(torch.bfloat16)
        return out

    out = {"a": fill((a_rows(r), r.K), r.a_dist)}
    if r.int4:
        words = torch.empty((r.E, r.N, r.K // 8), dtype=torch.int32, device=device)
        flat = words.view(-1)
        step = max(1, chunk_elems // 8)
        for s in range(0, flat.numel(), step):
            n = min(step, flat.numel() - s)
            q = torch.randint(0, 16, (n, 8), generator=g, device=device, dtype=torch.int64)
            shifts = torch.arange(0, 32, 4, device=device, dtype=torch.int64)
            w = (q << shifts).sum(dim=1)                       # < 2**32, fits int64
            w = torch.where(w >= 2**31, w - 2**32, w)          # uint32 bit pattern as int32
            flat[s:s + n] = w.to(torch.int32)
        out["packed"] = words
        lo, hi = r.scale_range
        out["scales"] = fill((r.E, r.N, r.K // r.group_size), ("uniform", lo, hi))
    else:
        out["b"] = fill((r.E, r.N, r.K), r.b_dist)
    return out


# ---------------------------------------------------------------- e4m3 operands and block scales

FP8_STD = 2.0                       # e4m3 operands ~ e4m3(N(0, FP8_STD))
FP8_IN_SCALE = (0.25, 1.0)          # input_scale ~ U[lo, hi]
FP8_W_SCALE = (0.002, 0.008)        # weight_scale ~ U[lo, hi]


def fp8_scale_shapes(rows: int, E: int, N: int, K: int, granularity) -> tuple:
    """Shapes of input_scale and weight_scale for granularity (gm, gn, gk); gk None means K."""
    gm, gn, gk = granularity
    gk = K if gk is None else gk
    nkb = -(-K // gk)
    return (-(-rows // gm), nkb), (E, -(-N // gn), nkb)


def _to_e4m3_bits(x) -> np.ndarray:
    """fp32 -> e4m3 bit patterns (uint8), round to nearest even, via torch's CPU cast."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()


def fp8_host_values(r: Routing, seed: int = 0, granularity=(1, 128, None), rows: int | None = None) -> dict:
    """e4m3 operands (uint8 bit patterns) and fp32 scales as numpy arrays:
    a8 [rows, K], w8 [E, N, K], input_scale and weight_scale (fp8_scale_shapes)."""
    rng = np.random.default_rng([seed, 2])
    rows = r.rows if rows is None else rows
    s_in, s_w = fp8_scale_shapes(rows, r.E, r.N, r.K, granularity)
    return {
        "a8": _to_e4m3_bits(rng.standard_normal((rows, r.K), dtype=np.float32) * np.float32(FP8_STD)),
        "w8": _to_e4m3_bits(rng.standard_normal((r.E, r.N, r.K), dtype=np.float32) * np.float32(FP8_STD)),
        "input_scale": rng.uniform(*FP8_IN_SCALE, s_in).astype(np.float32),
        "weight_scale": rng.uniform(*FP8_W_SCALE, s_w).astype(np.float32),
    }


def fp8_device_values(r: Routing, seed: int = 0, granularity=(1, 128, None), device="cuda",
                      chunk_elems: int = 1 << 27) -> dict:
    """The same distributions drawn on the device with torch's seeded CUDA generator
    (values differ from fp8_host_values).  Operands are uint8 tensors of e4m3 bits."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1000003 + 29)

    def fill(shape):
        out = torch.empty(shape, dtype=torch.uint8, device=device)
        flat = out.view(-1)
        for s in range(0, flat.numel(), chunk_elems):
            n = min(chunk_elems, flat.numel() - s)
            x = torch.randn(n, generator=g, device=device, dtype=torch.float32) * FP8_STD
            flat[s:s + n] = x.to(torch.float8_e4m3fn).view(torch.uint8)
        return out

    def uniform(shape, lo, hi):
        return torch.rand(shape, generator=g, device=device, dtype=torch.float32) * (hi - lo) + lo

    s_in, s_w = fp8_scale_shapes(r.rows, r.E, r.N, r.K, granularity)
    return {"a8": fill((r.rows, r.K)), "w8": fill((r.E, r.N, r.K)),
            "input_scale": uniform(s_in, *FP8_IN_SCALE), "weight_scale": uniform(s_w, *FP8_W_SCALE)}
