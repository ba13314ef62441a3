"""Reduced shared-memory budgets: the kernels run shallower rings instead of failing.

The quantised GEMM page's launcher reduces pipeline stages or warp partitions when the
shared memory budget is exceeded (Modular "multistage_gemm_q", description).  Here the
budget is capped for testing with GMM_SMEM_BUDGET (read when a handle is created); the
library then sizes every ring for the smaller budget: fewer stages for the bf16, e4m3
and per-K-block e4m3 kernels, a fallback from CTA pairs to one CTA per tile when a
pair's minimum ring no longer fits, and for the 4-bit kernel a shallower token ring
and a packed-weight ring of half the slots.  Each case is checked against the oracle,
and the configuration in use is read from the library's GMM_DEBUG report on stderr.
"""
import os
import re

import numpy as np
import pytest

from ragged_matmul_gb300 import binding
from ragged_matmul_gb300 import workloads as wl

from gpu_util import check_against_oracle, check_fp8_against_oracle

pytestmark = pytest.mark.gpu

LOADS = [1, 130, 0, 257, 16, 40, 300, 7]
IDS = [5, 0, 1, -1, 3, 2, 4, 0]


def _create(E, budget, variant, capfd):
    """A handle created under the budget cap, with GMM_DEBUG on: the library then reports
    each grouped-kernel launch's layout on stderr (see _launches)."""
    capfd.readouterr()
    saved = {k: os.environ.get(k) for k in ("GMM_SMEM_BUDGET", "GMM_VARIANT", "GMM_DEBUG")}
    os.environ.update({"GMM_SMEM_BUDGET": str(budget), "GMM_VARIANT": variant, "GMM_DEBUG": "1"})
    try:
        h = binding.gmm_create(E, 0)
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    capfd.readouterr()
    return h


def _launches(capfd):
    """The layouts of the grouped-kernel launches since the last call, as
    [(kernel, groups, stages, packed slots)]."""
    err = capfd.readouterr().err
    return [(m.group(1), int(m.group(2)), int(m.group(3)), int(m.group(4))) for m in
            re.finditer(r"gmm: launch (\w+(?: pair)?), (\d+) groups: stages (\d+) packed slots (\d+)", err)]


@pytest.mark.parametrize("variant", ["pair", "single"])
def test_bf16_and_4bit_with_200kb(variant, capfd):
    """200 KB: one stage fewer for bf16 (3 instead of 4 for one CTA, 2 instead of 3 for a
    pair); the 4-bit kernels still fit their full layouts beside the prefix of 8 groups."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    h = _create(6, 200 * 1024, variant, capfd)
    try:
        r = wl.make_routing("b", 6, 384, 520, LOADS, IDS, a_dist=("normal", 1.0), b_dist=("normal", 1.0))
        _, _, status, _ = check_against_oracle(h, r, wl.host_values(r, 31), where=f"bf16 at 200 KB {variant}")
        assert status == binding.GMM_OK
        assert _launches(capfd) == [("bf16 pair", 8, 2, 0) if variant == "pair" else ("bf16", 8, 3, 0)]
        r4 = wl.make_routing("b4", 6, 384, 1024, LOADS, IDS, a_dist=("normal", 1.0), b_dist=None, int4=True,
                             group_size=128)
        _, _, status, _ = check_against_oracle(h, r4, wl.host_values(r4, 32), where=f"4-bit at 200 KB {variant}")
        assert status == binding.GMM_OK
        assert _launches(capfd) == [("int4 pair", 8, 6, 4) if variant == "pair" else ("int4", 8, 3, 4)]
    finally:
        binding.gmm_destroy(h)


def test_dense_4bit_and_e4m3_with_170kb(capfd):
    """170 KB: the 4-bit kernel fits only with the half packed ring; the dense 4-bit GEMM (one group) and both e4m3 kernels (3 stages instead of 4
    for one scale over K) run against the oracle."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    h = _create(4, 170 * 1024, "single", capfd)
    try:
        # the dense 4-bit GEMM (its own entry point): one group of 300 rows
        r4 = wl.make_routing("d4", 1, 256, 512, [300], [0], a_dist=("normal", 1.0), b_dist=None, int4=True,
                             group_size=128)
        v4 = wl.host_values(r4, 33)
        from gpu_util import assert_close, bits_of, sentinel_dev, to_dev_u16
        import oracle
        c = sentinel_dev(r4.rows, r4.N, "cuda:0")
        binding.gmm_matmul_int4(h, c, to_dev_u16(v4["a"], "cuda:0"),
                                torch.from_numpy(np.ascontiguousarray(v4["packed"][0]).view(np.int32)).cuda(),
                                to_dev_u16(v4["scales"][0], "cuda:0"), group_size=128)
        assert binding.gmm_query_status(h) == binding.GMM_OK
        assert _launches(capfd) == [("int4", 1, 3, 2)]
        ref = oracle.gmm_int4(v4["a"], r4.a_offsets, v4["packed"], v4["scales"], r4.expert_ids, group_size=128)
        assert_close(bits_of(c), ref.ref32, np.ones(r4.rows, bool), where="dense 4-bit at 170 KB")
        # e4m3, one scale over K and per-K-block scales
        r8 = wl.make_routing("e8", 4, 256, 512, [17, 0, 140, 33], [3, 1, -1, 0])
        for gran in ((1, 128, None), (1, 128, 128)):
            v8 = wl.fp8_host_values(r8, 34, gran)
            _, _, status, _ = check_fp8_against_oracle(h, r8, v8, gran, where=f"e4m3 {gran} at 170 KB")
            assert status == binding.GMM_OK
        assert _launches(capfd)[:1] == [("e4m3", 4, 3, 0)]   # one scale over K: the grouped kernel, 3 stages

    finally:
        binding.gmm_destroy(h)


def test_budget_too_small_for_a_launch_is_reported(capfd):
    """At 170 KB the 4-bit kernel's minimum ring does not fit beside the prefix of 4096
    groups: that launch is refused with GMM_ERR_UNSUPPORTED before anything runs."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    h = _create(2, 170 * 1024, "single", capfd)
    try:
        G = 4096
        dev = "cuda:0"
        a = torch.zeros((16, 128), dtype=torch.bfloat16, device=dev)
        c = torch.zeros((16, 128), dtype=torch.bfloat16, device=dev)
        off = torch.zeros(G + 1, dtype=torch.int32, device=dev)
        off[-1] = 16
        ids = torch.zeros(G, dtype=torch.int32, device=dev)
        st = torch.zeros(4, dtype=torch.int32, device=dev)
        q = torch.zeros((2, 128, 16), dtype=torch.int32, device=dev)
        s = torch.zeros((2, 128, 1), dtype=torch.bfloat16, device=dev)
        with pytest.raises(binding.GmmError) as e:
            binding.gmm_run_int4(h, c, a, off, q, s, ids, st, group_size=128)
        assert e.value.code == binding.GMM_ERR_UNSUPPORTED
    finally:
        binding.gmm_destroy(h)
