"""The bench's work counts, against closed forms written out per workload (CPU only).

The roofline fraction the bench reports is useful FLOPs (or algorithmic bytes) per launch
over the measured time and peak; these tests pin the per-launch counts of the default
run's configurations to their definitions:
  FLOPs  = 2 N K x (rows of active groups),
  bytes  = the weights of each distinct expert with rows, once (bf16 2NK; 4-bit NK/2 plus
           a bf16 scale per group_size of K; e4m3 NK plus an fp32 scale per (128 rows of N,
           128 of K)), plus the active rows of A (e4m3: K bytes and an fp32 scale per 128 of
           K) and of C (bf16) once, plus a_offsets and expert_ids and stats (4 (2G + 2)).
"""
import pytest

import bench
from ragged_matmul_gb300 import workloads as wl


def _active(r):
    rows = sum(int(r.loads[g]) for g in range(r.G) if 0 <= int(r.expert_ids[g]) < r.E)
    experts = {int(r.expert_ids[g]) for g in range(r.G) if 0 <= int(r.expert_ids[g]) < r.E and r.loads[g] > 0}
    return rows, len(experts)


def test_default_run_configurations():
    assert bench.DEFAULT_CONFIGS == ("tiny", "decode", "prefill", "fine_grained", "int4", "fp8_block_prefill")
    assert bench.HEADLINE == "prefill"


def test_decode_counts():
    r = wl.routing("decode")
    flops, nbytes, rows = bench.work_counts(r)
    assert rows == 2048
    assert flops == 2 * 2816 * 2048 * 2048
    # 64 experts' bf16 weights, A and C rows, offsets + ids + stats
    assert nbytes == 64 * 2816 * 2048 * 2 + 2048 * 2048 * 2 + 2048 * 2816 * 2 + 4 * (2 * 64 + 2) == 758_120_968


def test_prefill_counts():
    r = wl.routing("prefill")
    flops, nbytes, rows = bench.work_counts(r)
    assert rows == 32768
    assert flops == 2 * 14336 * 4096 * 32768
    assert nbytes == 8 * 14336 * 4096 * 2 + 32768 * 4096 * 2 + 32768 * 14336 * 2 + 4 * (2 * 8 + 2)


def test_fine_grained_counts():
    r = wl.routing("fine_grained")
    flops, nbytes, rows = bench.work_counts(r)
    active_rows, experts = _active(r)
    assert (rows, experts) == (active_rows, 115)      # 13 of 128 groups skipped
    assert flops == 2 * 4096 * 7168 * active_rows
    assert nbytes == experts * 4096 * 7168 * 2 + active_rows * 7168 * 2 + active_rows * 4096 * 2 + 4 * (2 * 128 + 2)


def test_int4_counts():
    r = wl.routing("int4")
    flops, nbytes, rows = bench.work_counts(r)
    assert r.group_size == 128 and rows == 8192
    assert flops == 2 * 4096 * 4096 * 8192
    packed = 4096 * 4096 // 2            # 8 four-bit values per 32-bit word
    scales = 4096 * (4096 // 128) * 2    # a bf16 scale per 128 of K per weight row
    assert nbytes == 64 * (packed + scales) + 8192 * 4096 * 2 + 8192 * 4096 * 2 + 4 * (2 * 64 + 2)


def test_fp8_block_prefill_counts():
    r = wl.routing("fp8_block_prefill")
    flops, nbytes, rows = bench.work_counts(r)
    assert tuple(r.meta["granularity"]) == (1, 128, 128)
    assert flops == 2 * 14336 * 4096 * 32768
    w = 14336 * 4096 + (14336 // 128) * (4096 // 128) * 4   # e4m3 weights, fp32 block scales
    a = 32768 * (4096 + 4 * (4096 // 128))                  # e4m3 rows and their per-block input scales
    assert nbytes == 8 * w + a + 32768 * 14336 * 2 + 4 * (2 * 8 + 2)


@pytest.mark.parametrize("name", ["decode", "prefill", "fine_grained", "int4", "fp8_block_prefill"])
def test_binding_bound_follows_the_measured_peaks(name):
    """The bound named in the roofline is the larger of the two times at the peaks."""
    r = wl.routing(name)

    class A:
        epilogue = "none"
    d = bench.describe(r, A())
    assert d["bound"] == ("tensor" if d["t_tensor"] >= d["t_hbm"] else "hbm")
    expected = {"decode": "hbm", "prefill": "tensor", "fine_grained": "hbm", "int4": "tensor",
                "fp8_block_prefill": "tensor"}
    assert d["bound"] == expected[name]
