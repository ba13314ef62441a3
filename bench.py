"""Benchmark of the ragged grouped GEMM on GB300: useful TFLOP/s and fraction of roofline, per config.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload all|decode|prefill|...]
                    [--impl ours|reference]

With no --workload (or --workload all) one run measures the five configurations
of the mixture-of-experts shapes in turn, tiny (E=4, 60 rows, N=K=256), decode
(2048 rows over 64 experts, K=2048, N=2816), prefill (32768 rows over 8 experts,
K=4096, N=14336), fine_grained (32768 rows over 128 experts with 13 skipped,
K=7168, N=4096) and int4 (8192 rows over 64 experts of packed 4-bit weights,
K=N=4096), then fp8_block_prefill (the prefill shape with e4m3 operands and fp32
scales per 128 of K).  Each gets its own timed region, roofline, end-to-end number,
CPU oracle baseline with a parity check of the timed output, and clock record, under
"configs".  The top-level line repeats the entry of prefill, the largest of the five
mixture-of-experts shapes.

One step = one gmm_run (gmm_run_int4 for the 4-bit workload) over the whole
workload: every group, every row, all N columns.  Inputs are seeded synthetic
tensors already resident in HBM.  Between steps, outside the timed events, L2
is flushed: a 512 MiB buffer is written, then a different 512 MiB buffer is
read, so each step starts with a cold L2 that holds no dirty lines (without the
read, the timed kernel would also pay for writing the flush's dirty lines back
to HBM).  Each step is timed with CUDA events on the launching stream; `value`
is useful FLOPs / mean step time.

Under torchrun each rank runs its own replica of the workload (the groups are
independent problems and need no exchange), so scaling is weak and `value` =
FLOPs of all ranks / the slowest rank's time.

--impl reference times the CPU oracle (oracle/, plain C, all host cores of this
process) on a bounded sample of each workload: the first rows of its active
groups in routing order, all N columns, grown until one pass takes about a
second.  It is a baseline for context, not the target.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from ragged_matmul_gb300 import workloads as wl  # noqa: E402

# Roofline denominators.  MEASURED_PEAKS.json (written per GPU pool: a STREAM-style copy and a
# cuBLAS bf16 8192^3 GEMM, burst and sustained) wins when present; RECORDED_PEAKS is the copy of
# that measurement taken on the GB300s, used when the file is absent; FALLBACK_PEAKS is
# an older single GB300 measurement.
RECORDED_PEAKS = {"hbm_gbs": 6782.8, "bf16_tflops": 1921.8, "bf16_tflops_sustained": 1713.6}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FLUSH_BYTES = 512 << 20
METRIC = "grouped GEMM useful TFLOP/s and % of roofline (tensor or HBM) per config, 1xGB300"


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    return dict(RECORDED_PEAKS), "measured (recorded copy)"


def work_counts(r: wl.Routing):
    """Useful FLOPs and algorithmic bytes of one pass (padding and L2 re-reads not counted)."""
    act = r.active_mask()
    rows = int(r.loads[act].sum())
    flops = 2.0 * r.N * r.K * rows
    experts = np.unique(r.expert_ids[act & (r.loads > 0)])   # an empty group reads no weights
    if r.int4:
        wbytes = r.N * r.K // 2 + r.N * (r.K // r.group_size) * 2
    elif is_fp8(r):   # e4m3 weights and their fp32 scales; e4m3 activations and their scales
        gm, gn, gk = fp8_gran(r)
        nkb = -(-r.K // gk)
        wbytes = r.N * r.K + (-(-r.N // gn)) * nkb * 4
    else:
        wbytes = r.N * r.K * 2
    abytes = rows * (r.K + 4 * -(-r.K // fp8_gran(r)[2])) if is_fp8(r) else rows * r.K * 2
    if r.meta.get("planes"):   # each of the three planes of A is read once
        abytes *= 3
    nbytes = len(experts) * wbytes + abytes + rows * r.N * 2 + 4 * (2 * r.G + 2)
    return flops, float(nbytes), rows


def is_fp8(r: wl.Routing) -> bool:
    return bool(r.meta.get("fp8", False))


def fp8_gran(r: wl.Routing):
    """Scale granularity (m, n, k) of an e4m3 workload, k resolved to K when it spans all of K."""
    gm, gn, gk = r.meta.get("granularity", (1, 128, None))
    return gm, gn, (r.K if gk is None else gk)


def kernel_source_hash():
    """Hash of the CUDA sources with comments and whitespace removed: it changes when the
    code the profiles were captured on changes, not when a comment does."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "ragged_matmul_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        text = re.sub(r"\s+", " ", text)
        h.update(f.encode() + text.encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it matches the current kernel."""
    paths = [os.path.join(ROOT, "profiles", f"{k}_{workload}.md") for k in ("gmm_grouped_kernel", "gmm_fp8_block_kernel")]
    paths = [x for x in paths if os.path.exists(x)]
    if not paths:
        return None
    path = paths[0]
    text = open(path).read()
    m = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    hm = re.search(r"kernel_source_hash:\s*([0-9a-f]+)", text)
    if not m or not hm or hm.group(1) != kernel_source_hash():
        return None
    return float(m.group(1))


class ClockSampler:
    """SM clock, power and clock-event reasons, sampled every 10 ms from a thread.

    Reads them through NVML (libnvidia-ml, shipped with the driver) with ctypes:
    read-only queries, no setting of the GPU is touched.  Falls back to no samples
    when NVML cannot be loaded.
    """

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, index: int, period_s: float = 0.01):
        self.index = index
        self.period = period_s
        self.samples = []
        self._stop = threading.Event()
        self.thread = None
        self.nvml = None
        self.handle = None
        self.max_mhz = None

    def _open(self):
        import ctypes
        for name in ("libnvidia-ml.so.1", "libnvidia-ml.so"):
            try:
                lib = ctypes.CDLL(name)
                break
            except OSError:
                lib = None
        if lib is None or lib.nvmlInit_v2() != 0:
            return False
        h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.index), ctypes.byref(h)) != 0:
            return False
        self.nvml, self.handle = lib, h
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:   # 1 = SM clock
            self.max_mhz = mx.value
        return True

    def _poll(self):
        import ctypes
        lib, h = self.nvml, self.handle
        mhz, mw, reasons = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        get_reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._stop.is_set():
            ok = lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz)) == 0
            lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(mw))
            get_reasons(h, ctypes.byref(reasons))
            if ok:
                self.samples.append((time.time(), mhz.value, mw.value / 1000.0, reasons.value))
            self._stop.wait(self.period)

    def start(self):
        try:
            if not self._open():
                return
        except Exception:
            return
        self.thread = threading.Thread(target=self._poll, daemon=True)
        self.thread.start()

    def stop(self):
        self._stop.set()
        if self.thread:
            self.thread.join(timeout=2)

    def summary(self, t0, t1):
        inside = [x for x in self.samples if t0 <= x[0] <= t1]
        reasons = sorted({name for x in inside for bit, name in self.REASONS.items() if x[3] & bit})
        return {"sm_mhz": statistics.median([x[1] for x in inside]) if inside else None,
                "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "power_w_max": max((x[2] for x in inside), default=None),
                "samples": len(inside), "source": "nvml" if self.nvml else "unavailable"}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(x: float, world: int, device="cpu") -> float:
    """Maximum of x over the ranks (the slowest rank's time)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_tflops(world: int, flops_per_rank: float, slowest_ms: float) -> float:
    """Whole-job throughput of `world` replicas: every rank's FLOPs over the slowest rank's time."""
    return world * flops_per_rank / (slowest_ms * 1e-3) / 1e12


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ CPU oracle arm

def host_values_as_tensors(r: wl.Routing, seed: int = 0):
    """Seeded host-generated operands as CPU torch tensors (for hosts without a GPU)."""
    import torch
    if is_fp8(r):
        return {k: torch.from_numpy(x) for k, x in wl.fp8_host_values(r, seed, fp8_gran(r)).items()}
    v = wl.host_values(r, seed)
    out = {"a": torch.from_numpy(v["a"].view(np.int16)).view(torch.bfloat16)}
    if r.int4:
        out["packed"] = torch.from_numpy(v["packed"].view(np.int32))
        out["scales"] = torch.from_numpy(v["scales"].view(np.int16)).view(torch.bfloat16)
    else:
        out["b"] = torch.from_numpy(v["b"].view(np.int16)).view(torch.bfloat16)
    return out


def oracle_sample(r: wl.Routing, vals_dev, n_rows: int):
    """The first n_rows rows of the active groups in routing order (the last group
    touched may be cut short), all N columns, as host arrays."""
    import torch
    rows, loads, ids = [], [], []
    for g in np.flatnonzero(r.active_mask()):
        if len(rows) >= n_rows:
            break
        lo, hi = int(r.a_offsets[g]), int(r.a_offsets[g + 1])
        hi = min(hi, lo + n_rows - len(rows))
        if hi <= lo:
            continue
        rows += range(lo, hi)
        loads.append(hi - lo)
        ids.append(int(r.expert_ids[g]))
    akey = "a8" if is_fp8(r) else "a"
    idx = torch.tensor(rows, dtype=torch.int64, device=vals_dev[akey].device)
    sample = {"off": wl.offsets_from_loads(loads), "groups": len(loads), "rows": len(rows), "row_idx": list(rows)}
    if is_fp8(r):
        sample["a8"] = vals_dev["a8"][idx].cpu().numpy()
        sample["input_scale"] = vals_dev["input_scale"][idx].cpu().numpy()   # one per row (m granularity 1)
    elif r.meta.get("planes"):   # the sampled rows of each plane, the planes len(rows) apart
        M = r.rows
        sample["a"] = np.concatenate([vals_dev["a"][idx + p * M].contiguous().view(torch.int16).cpu().numpy()
                                      .view(np.uint16) for p in range(3)])
    else:
        sample["a"] = vals_dev["a"][idx].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    used = sorted(set(ids))
    remap = {e: i for i, e in enumerate(used)}           # keep only the experts the sample uses
    sample["ids"] = np.asarray([remap[e] for e in ids], np.int32)
    sel = torch.tensor(used, dtype=torch.int64, device=vals_dev[akey].device)
    if is_fp8(r):
        sample["w8"] = vals_dev["w8"][sel].cpu().numpy()
        sample["weight_scale"] = vals_dev["weight_scale"][sel].cpu().numpy()
    elif r.int4:
        sample["packed"] = vals_dev["packed"][sel].cpu().numpy().view(np.uint32)
        sample["scales"] = vals_dev["scales"][sel].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    else:
        sample["b"] = vals_dev["b"][sel].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    sample["flops"] = 2.0 * r.N * r.K * len(rows)
    return sample


def run_oracle(r: wl.Routing, s, nthreads):
    """One oracle pass over the sample; returns its wall time and keeps its fp32 sums in s["ref32"]."""
    import oracle
    t0 = time.perf_counter()
    if is_fp8(r):
        res = oracle.gmm_fp8(s["a8"], s["off"], s["w8"], s["ids"], s["input_scale"], s["weight_scale"],
                             fp8_gran(r))
    elif r.meta.get("planes"):
        res = oracle.gmm_bf16_planes(s["a"], s["off"], s["b"], s["ids"], r.meta["planes"], nthreads=nthreads)
    elif r.int4:
        res = oracle.gmm_int4(s["a"], s["off"], s["packed"], s["scales"], s["ids"], group_size=r.group_size,
                              nthreads=nthreads)
    else:
        res = oracle.gmm_bf16(s["a"], s["off"], s["b"], s["ids"], nthreads=nthreads)
    dt = time.perf_counter() - t0
    s["ref32"] = res.ref32
    return dt


def sample_parity(s, c_dev):
    """The timed run's output rows of the oracle sample against the oracle (per element
    |gpu - ref| <= 1e-2 + 1e-2 |ref|): the largest error as a fraction of its bound."""
    import torch
    idx = torch.tensor(s["row_idx"], dtype=torch.int64, device=c_dev.device)
    got = c_dev[idx].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    got32 = (got.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ref = s["ref32"].astype(np.float64)
    ratio = np.abs(got32 - ref) / (1e-2 + 1e-2 * np.abs(ref))
    worst = float(np.nanmax(ratio)) if ratio.size else 0.0
    return {"rows": int(len(s["row_idx"])), "elements": int(ratio.size), "max_err_over_bound": worst,
            "ok": bool(worst <= 1.0 and not np.isnan(ratio).any())}


def pick_oracle_sample(r, vals_dev, nthreads, target_s):
    """Grow the sample's row count until one oracle pass takes about target_s (or the
    whole workload is taken)."""
    total_rows = int(r.loads[r.active_mask()].sum())
    n = min(total_rows, 16)
    while True:
        s = oracle_sample(r, vals_dev, n)
        dt = run_oracle(r, s, nthreads)
        if dt >= 0.5 * target_s or n >= total_rows:
            return s, dt
        grow = 4.0 if dt <= 0 else min(8.0, max(1.25, target_s / dt))
        n = min(total_rows, max(n + 1, int(n * grow)))


def sample_desc(r, s):
    return (f"first {s['rows']} rows of the active groups in routing order ({s['groups']} group(s), "
            f"the last possibly cut short), all N={r.N} columns, K={r.K}")


# ------------------------------------------------------------------ main

# The configurations of the default run, in order: the five mixture-of-experts shapes,
# then the prefill shape with e4m3 operands and per-K-block scales (the block-scaled
# kernel).  The headline of the JSON line is prefill, the largest of the five.
DEFAULT_CONFIGS = ("tiny", "decode", "prefill", "fine_grained", "int4", "fp8_block_prefill")
HEADLINE = "prefill"


def describe(r: wl.Routing, args):
    """Work counts, roofline terms and the `config` object of one workload."""
    flops, nbytes, rows = work_counts(r)
    peaks, peaks_kind = load_peaks()
    # e4m3 MMAs run at twice the bf16 rate (the nominal dense ratio 4.5 : 2.25 PFLOP/s):
    # their tensor peak is the measured bf16 peak times 2.
    tensor_peak = peaks["bf16_tflops"] * (2.0 if is_fp8(r) else 1.0)
    t_tensor = flops / (tensor_peak * 1e12)
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    config = {"workload": r.name, "E": r.E, "N": r.N, "K": r.K, "groups": r.G,
              "active_groups": int(r.active_mask().sum()), "rows": rows,
              "useful_flops": flops, "algorithmic_bytes": nbytes,
              "l2": "flushed between steps (512 MiB written, then another 512 MiB read: cold, clean L2)",
              "weights": "int4" if r.int4 else ("e4m3" if is_fp8(r) else "bf16")}
    if is_fp8(r):
        gm, gn, gk = fp8_gran(r)
        config["scales"] = (f"fp32 input_scale per {gm} row(s) and weight_scale per {gn} weight rows of each "
                            f"expert, " + ("over all of K" if gk >= r.K else f"per {gk} of K") +
                            f" (granularity ({gm}, {gn}, {gk}))")
    if args.epilogue != "none":
        config["epilogue"] = f"{args.epilogue}(acc + bias[e, n]) * row_scale[r], fused before the bf16 store"
    return {"flops": flops, "nbytes": nbytes, "rows": rows, "peaks": peaks, "peaks_kind": peaks_kind,
            "tensor_peak": tensor_peak, "t_tensor": t_tensor, "t_hbm": t_hbm,
            "bound": "tensor" if t_tensor >= t_hbm else "hbm", "config": config}


def dtype_name(r):
    return "int4 weights, bf16 MMA" if r.int4 else ("e4m3" if is_fp8(r) else "bf16")


def kernel_name(r, variant):
    if is_fp8(r) and fp8_gran(r)[2] < r.K:
        return "gmm_fp8_block_kernel"
    pair = variant != "single"   # the library runs CTA pairs unless told otherwise
    return "gmm_grouped_kernel<%s, %s, %s>" % ("true" if r.int4 else "false", "true" if pair else "false",
                                               "true" if is_fp8(r) else "false")


def select_routing(name, args):
    r = wl.routing(name)
    if args.groups:
        r = wl.first_groups(r, args.groups)
    if args.group_range:
        lo, hi = (int(x) for x in args.group_range.split(":"))
        r = wl.group_range(r, lo, hi)
    if args.rows:
        r = wl.with_rows(r, args.rows)
    return r


def reference_config(r, args, n_configs):
    """The reference arm on one workload: the CPU oracle, timed as it stands."""
    import torch
    d = describe(r, args)
    local = dist_env()[2]
    if torch.cuda.is_available():
        vals = (wl.fp8_device_values(r, 0, fp8_gran(r), device=torch.device(f"cuda:{local}")) if is_fp8(r)
                else wl.device_values(r, 0, device=torch.device(f"cuda:{local}")))
    else:
        vals = host_values_as_tensors(r, 0)
    nthreads = len(os.sched_getaffinity(0))
    # The whole run (every config, warm-up and timed passes) takes a couple of minutes.
    per_step = max(0.1, min(args.oracle_seconds, 100.0 / ((args.steps + 1) * n_configs)))
    s, _ = pick_oracle_sample(r, vals, nthreads, per_step)
    del vals
    if torch.cuda.is_available():
        torch.cuda.empty_cache()
    for _ in range(min(args.warmup, 1)):
        run_oracle(r, s, nthreads)
    times = [run_oracle(r, s, nthreads) for _ in range(args.steps)]
    t = statistics.mean(times)
    value = s["flops"] / t / 1e12
    return {"value": value, "unit": "TFLOP/s", "ms_per_step": t * 1e3, "config": d["config"],
            "dtype": ("e4m3 inputs, fp64 sums (numpy, CPU)" if is_fp8(r)
                      else "bf16 inputs, fp32 accumulation (C, CPU)"),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": nthreads, "kind": "oracle",
                             "sample": sample_desc(r, s)},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def measure_config(r, args, world, rank, local, dev):
    """Our arm on one workload: the timed region, the end-to-end run through host buffers,
    the yardstick, the CPU oracle baseline and the parity of the timed output."""
    import torch
    from ragged_matmul_gb300 import binding
    d = describe(r, args)
    flops, nbytes = d["flops"], d["nbytes"]
    vals = wl.fp8_device_values(r, rank, fp8_gran(r), device=dev) if is_fp8(r) else wl.device_values(r, rank, device=dev)
    akey = "a8" if is_fp8(r) else "a"
    h = binding.gmm_create(r.E, local)
    c = torch.full((r.rows, r.N), wl.SENTINEL_BF16, dtype=torch.int16, device=dev).view(torch.bfloat16)
    off = torch.from_numpy(r.a_offsets.view(np.int32)).to(dev)
    ids = torch.from_numpy(r.expert_ids).to(dev)
    stats = torch.zeros(4, dtype=torch.int32, device=dev)
    flush_w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(FLUSH_BYTES // 4, dtype=torch.int32, device=dev)

    def flush_l2():
        flush_w.zero_()
        flush_r.sum()
    stream = torch.cuda.current_stream(dev)

    epi = {}
    if args.epilogue != "none":   # seeded epilogue operands, made on the device
        gen = torch.Generator(device=dev).manual_seed(1000 + rank)
        epi = {"bias": (0.1 * torch.randn((r.E, r.N), generator=gen, device=dev)).to(torch.bfloat16),
               "row_scale": torch.rand((r.rows,), generator=gen, device=dev) * 0.9 + 0.1,
               "activation": args.epilogue}

    def step(cc=c, aa=vals[akey], oo=off, ii=ids, ss=stats):
        if is_fp8(r):
            binding.gmm_run_fp8(h, cc, aa, oo, vals["w8"], ii, ss, vals["input_scale"], vals["weight_scale"],
                                fp8_gran(r), stream=stream, **epi)
        elif r.meta.get("planes"):
            binding.gmm_run_planes(h, cc, aa, oo, vals["b"], ii, ss, r.meta["planes"], stream=stream, **epi)
        elif r.name == "int4_dense":   # the dense quantised GEMM's own entry point
            binding.gmm_matmul_int4(h, cc, aa, vals["packed"][0], vals["scales"][0], group_size=r.group_size,
                                    stream=stream, **epi)
        elif r.int4:
            binding.gmm_run_int4_ex(h, cc, aa, oo, vals["packed"], vals["scales"], ii, ss,
                                    group_size=r.group_size, stream=stream, **epi)
        else:
            binding.gmm_run_ex(h, cc, aa, oo, vals["b"], ii, ss, stream=stream, **epi)

    for _ in range(args.warmup):
        flush_l2()
        step()
    torch.cuda.synchronize()
    status = binding.gmm_query_status(h)
    if status != binding.GMM_OK:
        raise RuntimeError(f"{r.name}: device status after warm-up: {binding.gmm_error_string(status)}")

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    w0 = time.time()
    for i in range(args.steps):
        flush_l2()
        evs[i][0].record(stream)
        step()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    w1 = time.time()
    sampler.stop()
    step_ms = [a.elapsed_time(b) for a, b in evs]
    mean_ms = statistics.mean(step_ms)
    status = binding.gmm_query_status(h)
    if status != binding.GMM_OK:
        raise RuntimeError(f"{r.name}: device status after timing: {binding.gmm_error_string(status)}")
    max_ms = reduce_max(mean_ms, world, dev)
    value = aggregate_tflops(world, flops, max_ms)

    # end to end through the public API with host buffers: H2D of the step's inputs
    # (activations, offsets, ids) from pinned memory, the kernel, D2H of C and stats.
    e2e = None
    if not args.no_e2e:
        a_h = vals[akey].cpu().pin_memory()
        off_h, ids_h = off.cpu().pin_memory(), ids.cpu().pin_memory()
        c_h = torch.empty_like(c, device="cpu").pin_memory()
        st_h = torch.empty_like(stats, device="cpu").pin_memory()
        a_d, off_d, ids_d = torch.empty_like(vals[akey]), torch.empty_like(off), torch.empty_like(ids)
        h2d = a_h.numel() * a_h.element_size() + off_h.numel() * 4 + ids_h.numel() * 4
        d2h = c_h.numel() * 2 + st_h.numel() * 4

        def e2e_step():
            a_d.copy_(a_h, non_blocking=True)
            off_d.copy_(off_h, non_blocking=True)
            ids_d.copy_(ids_h, non_blocking=True)
            step(c, a_d, off_d, ids_d, stats)
            c_h.copy_(c, non_blocking=True)
            st_h.copy_(stats, non_blocking=True)

        for _ in range(args.warmup):
            flush_l2()
            e2e_step()
        torch.cuda.synchronize()
        e_ms = []
        barrier(world)
        for _ in range(args.steps):
            flush_l2()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            e2e_step()
            e1.record(stream)
            e1.synchronize()
            e_ms.append(e0.elapsed_time(e1))
        e2e_max = reduce_max(statistics.mean(e_ms), world, dev)
        e2e = {"value": aggregate_tflops(world, flops, e2e_max), "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": e2e_max}
        del a_h, c_h, a_d

    # A library yardstick for context (never a reference for results): cuBLAS through
    # torch.matmul, one GEMM per active group, on the same resident operands.
    yardstick = None
    if args.yardstick and rank == 0 and not (r.int4 or is_fp8(r) or r.meta.get("planes")):
        segs = [(int(r.a_offsets[g]), int(r.a_offsets[g + 1]), int(r.expert_ids[g]))
                for g in np.flatnonzero(r.active_mask()) if r.a_offsets[g + 1] > r.a_offsets[g]]
        cy = torch.empty_like(c)

        def ystep():
            for r0, r1, e in segs:
                torch.matmul(vals["a"][r0:r1], vals["b"][e].t(), out=cy[r0:r1])
        for _ in range(args.warmup):
            flush_l2()
            ystep()
        y_ms = []
        for _ in range(min(args.steps, 50)):
            flush_l2()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            ystep()
            e1.record(stream)
            e1.synchronize()
            y_ms.append(e0.elapsed_time(e1))
        y = statistics.mean(y_ms)
        yardstick = {"kind": "torch.matmul per active group (cuBLAS, bf16), context only", "ms_per_step": y,
                     "value": flops / (y * 1e-3) / 1e12, "unit": "TFLOP/s", "launches_per_step": len(segs)}
        del cy

    cpu_baseline = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        nthreads = len(os.sched_getaffinity(0))
        s, t = pick_oracle_sample(r, vals, nthreads, args.oracle_seconds)
        # A workload whose whole oracle pass is short is timed over repeated passes,
        # so the baseline still rests on about half the target seconds of CPU work.
        passes, total = 1, t
        while total < 0.5 * args.oracle_seconds and passes < 1000:
            total += run_oracle(r, s, nthreads)
            passes += 1
        cpu_baseline = {"value": passes * s["flops"] / total / 1e12, "unit": "TFLOP/s", "cores": nthreads,
                        "kind": "oracle",
                        "sample": sample_desc(r, s) + f"; {passes} pass(es), {total:.2f} s"}
        if args.epilogue == "none":   # the timed run's output on the sample, after timing
            cpu_baseline["parity_after_timing"] = sample_parity(s, c)

    t_s = mean_ms * 1e-3
    peaks = d["peaks"]
    if d["bound"] == "hbm":
        achieved, peak, unit = nbytes / t_s / 1e9, peaks["hbm_gbs"], "GB/s"
    else:
        achieved, peak, unit = flops / t_s / 1e12, d["tensor_peak"], "TFLOP/s"
    roofline = {"bound": d["bound"], "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
                "traffic": profiled_traffic(r.name),
                "peak_source": f"{d['peaks_kind']} (burst)" + (" bf16 x 2, the nominal e4m3 : bf16 ratio"
                                                              if is_fp8(r) and d["bound"] == "tensor" else ""),
                "roofline_time_ms": max(d["t_tensor"], d["t_hbm"]) * 1e3,
                "frac_of_roofline_time": max(d["t_tensor"], d["t_hbm"]) / t_s,
                "kernel": kernel_name(r, args.variant)}
    out = {"value": value, "unit": "TFLOP/s", "ms_per_step": max_ms, "dtype": dtype_name(r),
           "config": d["config"], "roofline": roofline, "cpu_baseline": cpu_baseline, "e2e": e2e,
           "gpu_launches": args.steps, **({"yardstick": yardstick} if yardstick else {}),
           "clocks": sampler.summary(w0, w1), "region_wall_ms": (w1 - w0) * 1e3,
           "step_ms_min": min(step_ms), "step_ms_median": statistics.median(step_ms)}
    binding.gmm_destroy(h)
    del vals, c, flush_w, flush_r
    torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="all", choices=["all", *wl.WORKLOAD_NAMES],
                    help="'all' (default): the five configurations tiny, decode, prefill, fine_grained "
                         "and int4, then fp8_block_prefill, each timed in turn, prefill as the headline")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--oracle-seconds", type=float, default=3.0,
                    help="CPU oracle work per step of the reference arm / per cpu_baseline pass")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--groups", type=int, default=0,
                    help="profile-sized sub-workload: only the first G groups of the named routing")
    ap.add_argument("--rows", type=int, default=0,
                    help="redraw the named routing for this many rows (same groups and proportions)")
    ap.add_argument("--group-range", default=None,
                    help="sub-workload lo:hi - groups lo .. hi-1 of the named routing")
    ap.add_argument("--epilogue", default="none", choices=["none", "relu", "silu", "gelu_tanh"],
                    help="time the fused epilogue act(acc + bias[e, n]) * row_scale[r] with this activation "
                         "(seeded bias and per-row scales); 'none' is the plain GEMM")
    ap.add_argument("--yardstick", action="store_true",
                    help="also time torch.matmul per active group (cuBLAS, bf16 workloads) on the same data, "
                         "for context")
    ap.add_argument("--variant", default=None, choices=["pair", "single"],
                    help="kernel variant (default: the library's choice, CTA pairs)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    names = list(DEFAULT_CONFIGS) if args.workload == "all" else [args.workload]
    headline = HEADLINE if args.workload == "all" else args.workload

    world, rank, local = dist_env()
    import torch

    common = {"metric": METRIC, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
              "higher_is_better": True, "scaling": "weak", "vs_baseline": None}

    if args.impl == "reference":
        # The CPU oracle, timed on this host's cores; under torchrun only rank 0 works.
        if rank != 0:
            return
        per = {}
        for name in names:
            per[name] = reference_config(select_routing(name, args), args, len(names))
        head = per[headline]
        line = {"impl": "reference", **common, "n_gpus": 1, "value": head["value"], "unit": "TFLOP/s",
                "ms_per_step": head["ms_per_step"], "dtype": head["dtype"], "data": "synthetic (seeded)",
                "config": head["config"], "cpu_baseline": head["cpu_baseline"], "e2e": head["e2e"]}
        if len(names) > 1:
            line["headline"] = f"{headline}: the largest of the configurations in `configs`"
            line["configs"] = per
        print(json.dumps(line), flush=True)
        return

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    torch.cuda.set_device(local)
    dev = torch.device(f"cuda:{local}")

    from ragged_matmul_gb300 import build as gbuild
    if rank == 0:
        gbuild.build()
    barrier(world)
    if args.variant:
        os.environ["GMM_VARIANT"] = args.variant

    per = {}
    for name in names:
        per[name] = measure_config(select_routing(name, args), args, world, rank, local, dev)
    if rank == 0:
        head = per[headline]
        line = {**common, "value": head["value"], "unit": "TFLOP/s", "ms_per_step": head["ms_per_step"],
                "dtype": head["dtype"], "data": "synthetic (seeded, generated on device)",
                "config": head["config"], "roofline": head["roofline"], "cpu_baseline": head["cpu_baseline"],
                "e2e": head["e2e"], "gpu_launches": head["gpu_launches"], "clocks": head["clocks"],
                **({"yardstick": head["yardstick"]} if "yardstick" in head else {}),
                "region_wall_ms": head["region_wall_ms"], "step_ms_min": head["step_ms_min"],
                "step_ms_median": head["step_ms_median"]}
        if len(names) > 1:
            line["headline"] = f"{headline}: the largest of the configurations in `configs`"
            line["configs"] = per
            line["gpu_launches_all_configs"] = sum(x["gpu_launches"] for x in per.values())
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
