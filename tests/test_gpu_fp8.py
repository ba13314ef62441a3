"""Parity of the block-scaled e4m3 grouped GEMM (gmm_run_fp8, through the C ABI)
with the CPU oracle: small and ragged shapes element by element, the full-size
fp8 workloads on sampled rows and columns, and the argument checks.
"""
import numpy as np
import pytest

import oracle
from ragged_matmul_gb300 import binding
from ragged_matmul_gb300 import workloads as wl

from gpu_util import (VARIANTS, assert_close, bits_of, check_fp8_against_oracle, handle, live_row_mask,
                      run_gpu_fp8, sentinel_dev, to_dev_f32, to_dev_i32, to_dev_u8)

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


def case(E, N, K, loads, ids, seed, gran=(1, 128, None), base=0, rows=None):
    r = wl.make_routing("t", E, N, K, loads, ids, base=base)
    return r, wl.fp8_host_values(r, seed, gran, rows=rows)


@pytest.mark.parametrize("variant", VARIANTS)
def test_fp8_tiny(variant):
    r = wl.routing("tiny")
    v = wl.fp8_host_values(r, 1)
    _, _, status, _ = check_fp8_against_oracle(handle(r.E, variant), r, v, (1, 128, None), where="tiny")
    assert status == binding.GMM_OK


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("N,K", [(384, 320), (136, 208), (256, 128), (1024, 1104), (648, 512), (128, 16)])
def test_fp8_ragged_groups_tails(N, K, variant):
    """Group sizes around the token granules and tiles, N and K tails (K / 2 two-byte
    units not a multiple of 64: the last stage is part zero fill)."""
    loads = [1, 15, 16, 17, 31, 32, 33, 127, 128, 129, 255, 256, 257, 300, 513, 0, 2]
    ids = [3, 0, 5, 1, 7, 2, 6, 4, 3, 0, 1, 2, 6, 7, 5, 1, 4]
    r, v = case(8, N, K, loads, ids, 3)
    _, _, status, _ = check_fp8_against_oracle(handle(8, variant), r, v, (1, 128, None),
                                               where=f"fp8 ragged N={N} K={K} {variant}")
    assert status == binding.GMM_OK


@pytest.mark.parametrize("gran", [(1, 1, None), (3, 7, None), (128, 128, None), (1, 512, 4096), (2, 200, None)])
def test_fp8_scale_granularities(gran):
    """Row and column block sizes that divide nothing, one block, and gk > K."""
    r, v = case(4, 392, 256, [5, 130, 0, 77, 257], [2, 0, 1, 3, 1], 4, gran=gran)
    _, _, status, _ = check_fp8_against_oracle(handle(4), r, v, gran, where=f"granularity {gran}")
    assert status == binding.GMM_OK


@pytest.mark.parametrize("variant", VARIANTS)
def test_fp8_small_integers_bit_exact(variant):
    """e4m3 integers in [-3, 3] and power-of-two scales: every sum, scale product and
    bf16 rounding is exact, so the result must match bit for bit."""
    r = wl.make_routing("t", 3, 264, 64, [1, 40, 0, 200, 17], [2, 0, 1, 1, -1])
    rng = np.random.default_rng(5)
    to8 = wl._to_e4m3_bits
    v = {"a8": to8(rng.integers(-3, 4, (r.rows, 64)).astype(np.float32)),
         "w8": to8(rng.integers(-3, 4, (3, 264, 64)).astype(np.float32)),
         "input_scale": rng.choice([0.25, 0.5, 1.0], (r.rows, 1)).astype(np.float32),
         "weight_scale": rng.choice([0.5, 1.0, 2.0], (3, 3, 1)).astype(np.float32)}
    check_fp8_against_oracle(handle(3, variant), r, v, (1, 128, None), exact=True, where="fp8 exact")


def test_fp8_offset_base_skips_and_trailing_rows():
    r, v = case(4, 256, 192, [50, 300, 20, 64, 64], [-1, 2, -5, 2, 0], 6, base=37)
    rows_alloc = r.rows + 19
    v = wl.fp8_host_values(r, 6, rows=rows_alloc)
    _, _, status, _ = check_fp8_against_oracle(handle(4), r, v, (1, 128, None), rows_alloc=rows_alloc,
                                               where="fp8 skips")
    assert status == binding.GMM_OK


def test_fp8_bad_inputs_reported():
    r, v = case(4, 128, 64, [30, 40, 10], [0, 1, 2], 8)
    off = np.array([0, 30, 20, 80], np.uint32)
    got, stats, status = run_gpu_fp8(handle(4), v, off, r.expert_ids, (1, 128, None), N=128)
    assert np.all(got == wl.SENTINEL_BF16) and stats.tolist() == [0xFFFFFFFF, 3, 0xFFFFFFFF, 0xFFFFFFFF]
    assert status == binding.GMM_ERR_BAD_INPUT
    r2, v2 = case(4, 128, 64, [30, 40, 10], [0, 9, 2], 9)
    _, ref, status, _ = check_fp8_against_oracle(handle(4), r2, v2, (1, 128, None), where="fp8 bad id")
    assert ref.flags == oracle.BAD_EXPERT_ID and status == binding.GMM_ERR_BAD_INPUT


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("activation", ["none", "silu"])
def test_fp8_with_epilogue(activation, variant):
    """Scales first, then act(y + bias[e, n]) * row_scale[r]."""
    r, v = case(4, 392, 208, [1, 17, 0, 130, 33, 257, 7], [2, 0, 1, 3, -1, 1, 0], 10, gran=(2, 64, None))
    rng = np.random.default_rng(11)
    epi = {"bias_bits": wl._to_bf16_bits(rng.normal(0.0, 0.1, (4, 392)).astype(np.float32)),
           "row_scale": rng.uniform(0.1, 2.0, r.rows).astype(np.float32), "activation": activation}
    _, _, status, _ = check_fp8_against_oracle(handle(4, variant), r, v, (2, 64, None), epilogue=epi,
                                               where=f"fp8 epilogue {activation} {variant}")
    assert status == binding.GMM_OK


@pytest.mark.parametrize("variant", VARIANTS)
def test_fp8_with_epilogue_long_k(variant):
    """The same with K = 2080 e4m3 values (1040 two-byte units): the 4-epilogue-warp launch."""
    r, v = case(4, 392, 2080, [1, 17, 0, 130, 33, 257, 7], [2, 0, 1, 3, -1, 1, 0], 12, gran=(2, 64, None))
    rng = np.random.default_rng(13)
    epi = {"bias_bits": wl._to_bf16_bits(rng.normal(0.0, 0.1, (4, 392)).astype(np.float32)),
           "row_scale": rng.uniform(0.1, 2.0, r.rows).astype(np.float32), "activation": "gelu_tanh"}
    _, _, status, _ = check_fp8_against_oracle(handle(4, variant), r, v, (2, 64, None), epilogue=epi,
                                               where=f"fp8 epilogue long K {variant}")
    assert status == binding.GMM_OK


def test_fp8_accepts_float8_tensors():
    """The binding takes torch.float8_e4m3fn tensors as well as their uint8 bit patterns."""
    import torch
    r, v = case(2, 128, 64, [9, 20], [1, 0], 12)
    h = handle(2)
    c = sentinel_dev(r.rows, 128, DEV)
    st = to_dev_i32(np.zeros(4), DEV)
    binding.gmm_run_fp8(h, c, to_dev_u8(v["a8"], DEV).view(torch.float8_e4m3fn), to_dev_i32(r.a_offsets, DEV),
                        to_dev_u8(v["w8"], DEV).view(torch.float8_e4m3fn), to_dev_i32(r.expert_ids, DEV), st,
                        to_dev_f32(v["input_scale"], DEV), to_dev_f32(v["weight_scale"], DEV))
    ref = oracle.gmm_fp8(v["a8"], r.a_offsets, v["w8"], r.expert_ids, v["input_scale"], v["weight_scale"],
                         (1, 128, 64))
    assert_close(bits_of(c), ref.ref32, np.ones(r.rows, bool), "float8 tensors")


def test_fp8_argument_errors():
    """Nothing is launched (C stays sentinel) for each rejected argument."""
    import torch
    h = handle(4)
    r, v = case(4, 128, 64, [8], [1], 13)
    c = sentinel_dev(r.rows, 128, DEV)
    a, w = to_dev_u8(v["a8"], DEV), to_dev_u8(v["w8"], DEV)
    off, ids, st = to_dev_i32(r.a_offsets, DEV), to_dev_i32(r.expert_ids, DEV), to_dev_i32(np.zeros(4), DEV)
    s_in, s_w = to_dev_f32(v["input_scale"], DEV), to_dev_f32(v["weight_scale"], DEV)
    lib = binding.load_library()
    import ctypes
    P = ctypes.c_void_p
    stream = binding.stream_handle(0)

    def call(K=64, gran=(1, 128, 64), pin=s_in, pw=s_w):
        g = None if gran is None else (ctypes.c_int * 3)(*gran)
        return lib.gmm_run_fp8(h.ptr, P(c.data_ptr()), P(a.data_ptr()), P(off.data_ptr()), P(w.data_ptr()),
                               P(ids.data_ptr()), P(st.data_ptr()), 1, 128, K,
                               None if pin is None else P(pin.data_ptr()), None if pw is None else P(pw.data_ptr()),
                               g, None, stream)
    assert call(K=56) == binding.GMM_ERR_INVALID_ARG                  # K not a multiple of 16
    assert call(gran=(1, 128, 32)) == binding.GMM_ERR_UNSUPPORTED     # K blocks of less than 128
    assert call(K=256, gran=(1, 48, 128)) == binding.GMM_ERR_UNSUPPORTED   # per-K-block with gn % 32 != 0
    assert call(gran=(0, 128, 64)) == binding.GMM_ERR_INVALID_ARG
    assert call(gran=(1, 0, 64)) == binding.GMM_ERR_INVALID_ARG
    assert call(gran=None) == binding.GMM_ERR_INVALID_ARG
    assert call(pin=None) == binding.GMM_ERR_INVALID_ARG
    assert call(pw=None) == binding.GMM_ERR_INVALID_ARG
    assert lib.gmm_run_fp8(h.ptr, P(c.data_ptr()), P(a.data_ptr()), P(off.data_ptr()), P(w.data_ptr()),
                           P(ids.data_ptr()), P(st.data_ptr()), 1, 128, 64, P(s_in.data_ptr() + 2),
                           P(s_w.data_ptr()), (ctypes.c_int * 3)(1, 128, 64), None,
                           stream) == binding.GMM_ERR_INVALID_ARG    # misaligned input_scale
    torch.cuda.synchronize()
    assert np.all(bits_of(c) == wl.SENTINEL_BF16)
    with pytest.raises(binding.GmmError):   # per-K-block scales, shaped right, through the binding
        binding.gmm_run_fp8(h, c, a, off, w, ids, st, to_dev_f32(np.ones((8, 2), np.float32), DEV),
                            to_dev_f32(np.ones((4, 1, 2), np.float32), DEV), (1, 128, 32))


def _sampled_fp8(name, rows_per_group=2, ncols=96, seed=0):
    """The full fp8 workload on the GPU, checked on sampled rows and columns."""
    import torch
    r = wl.routing(name)
    gran = tuple(r.meta.get("granularity", (1, 128, None)))
    v = wl.fp8_device_values(r, seed, gran, device=DEV)
    h = handle(r.E)
    c = sentinel_dev(r.rows, r.N, DEV)
    stats = to_dev_i32(np.full(4, 0xFFFFFFFF, np.uint32), DEV)
    binding.gmm_run_fp8(h, c, v["a8"], to_dev_i32(r.a_offsets, DEV), v["w8"], to_dev_i32(r.expert_ids, DEV),
                        stats, v["input_scale"], v["weight_scale"], gran)
    assert binding.gmm_query_status(h) == binding.GMM_OK
    assert stats.cpu().numpy().view(np.uint32)[1] == int(r.active_mask().sum())
    live = live_row_mask(r.rows, r.a_offsets, r.expert_ids, r.E)
    assert bool((c.view(torch.int16)[torch.from_numpy(~live).to(DEV)] == wl.SENTINEL_BF16).all())
    rng = np.random.default_rng(seed + 200)
    rows, loads = [], []
    for g in range(r.G):
        lo, hi = int(r.a_offsets[g]), int(r.a_offsets[g + 1])
        pick = sorted(set([lo, hi - 1] + rng.integers(lo, hi, rows_per_group).tolist())) if hi > lo else []
        rows += pick
        loads.append(len(pick))
    rows = np.asarray(rows, np.int64)
    cols = np.unique(np.concatenate([[0, r.N - 1], rng.choice(r.N, ncols, replace=False)]))
    rows_t, cols_t = torch.from_numpy(rows).to(DEV), torch.from_numpy(cols).to(DEV)
    off_s = wl.offsets_from_loads(loads)
    # The sampled columns are weight rows of each expert; their scales keep their own
    # block: with one column per block (gn = 1) the scale is gathered per column.
    ws = v["weight_scale"][:, (cols_t // gran[1]), :].cpu().numpy()
    gk = r.K if gran[2] is None else gran[2]
    ref = oracle.gmm_fp8(v["a8"][rows_t].cpu().numpy(), off_s, v["w8"][:, cols_t, :].cpu().numpy(),
                         r.expert_ids, v["input_scale"][rows_t].cpu().numpy(), ws, (1, 1, gk))
    got = bits_of(c[rows_t][:, cols_t])
    live_s = live_row_mask(len(rows), off_s, r.expert_ids, r.E)
    err = assert_close(got, ref.ref32, live_s, where=name)
    assert np.all(got[~live_s] == wl.SENTINEL_BF16)
    return err


@pytest.mark.parametrize("name", ["fp8_decode", "fp8_prefill", "fp8_block_decode", "fp8_block_prefill"])
def test_fp8_full_size_sampled(name):
    _sampled_fp8(name)


# ---------------------------------------------------------------- per-K-block scales (gk < K)

@pytest.mark.parametrize("N,K,gran", [(384, 512, (1, 128, 128)), (264, 1104, (1, 32, 128)),
                                      (512, 768, (3, 64, 256)), (1024, 1024, (2, 256, 384)),
                                      (136, 256, (1, 32, 128)), (256, 4096, (1, 128, 128))])
def test_fp8_block_scales_ragged(N, K, gran):
    """Ragged groups (1 .. 513 rows, a skipped one), N and K tails (K = 1104: a partial last
    block), granularities that divide nothing, against the oracle's per-block sums."""
    loads = [1, 15, 16, 17, 127, 128, 129, 255, 257, 513, 0, 40]
    ids = [3, 0, 5, 1, 7, 2, 6, 4, -1, 0, 1, 2]
    r, v = case(8, N, K, loads, ids, 20, gran=gran)
    _, _, status, _ = check_fp8_against_oracle(handle(8), r, v, gran, where=f"fp8 block N={N} K={K} {gran}")
    assert status == binding.GMM_OK


def test_fp8_block_scales_bit_exact():
    """e4m3 integers in [-3, 3] and power-of-two block scales: every partial, scaled
    partial, sum and rounding is exact."""
    r = wl.make_routing("t", 3, 256, 512, [1, 40, 0, 200, 17], [2, 0, 1, 1, -1])
    rng = np.random.default_rng(21)
    to8 = wl._to_e4m3_bits
    v = {"a8": to8(rng.integers(-3, 4, (r.rows, 512)).astype(np.float32)),
         "w8": to8(rng.integers(-3, 4, (3, 256, 512)).astype(np.float32)),
         "input_scale": rng.choice([0.25, 0.5, 1.0], (r.rows, 4)).astype(np.float32),
         "weight_scale": rng.choice([0.125, 0.25, 0.5], (3, 2, 4)).astype(np.float32)}
    check_fp8_against_oracle(handle(3), r, v, (1, 128, 128), exact=True, where="fp8 block exact")


@pytest.mark.parametrize("activation", ["none", "gelu_tanh"])
def test_fp8_block_scales_with_epilogue(activation):
    r, v = case(4, 392, 640, [1, 17, 0, 130, 33, 257, 7], [2, 0, 1, 3, -1, 1, 0], 22, gran=(2, 64, 128))
    rng = np.random.default_rng(23)
    epi = {"bias_bits": wl._to_bf16_bits(rng.normal(0.0, 0.1, (4, 392)).astype(np.float32)),
           "row_scale": rng.uniform(0.1, 2.0, r.rows).astype(np.float32), "activation": activation}
    _, _, status, _ = check_fp8_against_oracle(handle(4), r, v, (2, 64, 128), epilogue=epi,
                                               where=f"fp8 block epilogue {activation}")
    assert status == binding.GMM_OK


def test_fp8_block_scales_edge_cases():
    """Offset base with trailing rows, bad offsets (nothing written), and no groups."""
    r, v = case(4, 256, 384, [50, 300, 20, 64], [-1, 2, 3, 0], 24, gran=(1, 128, 128), base=37)
    rows_alloc = r.rows + 19
    v = wl.fp8_host_values(r, 24, (1, 128, 128), rows=rows_alloc)
    check_fp8_against_oracle(handle(4), r, v, (1, 128, 128), rows_alloc=rows_alloc, where="fp8 block base")
    off = np.array([0, 30, 20, 80], np.uint32)
    r2, v2 = case(4, 128, 256, [30, 40, 10], [0, 1, 2], 25, gran=(1, 128, 128))
    got, stats, status = run_gpu_fp8(handle(4), v2, off, r2.expert_ids, (1, 128, 128), N=128)
    assert np.all(got == wl.SENTINEL_BF16) and status == binding.GMM_ERR_BAD_INPUT
    r3, v3 = case(4, 128, 256, [], [], 26, gran=(1, 128, 128), rows=16)
    got, stats, status = run_gpu_fp8(handle(4), v3, r3.a_offsets, r3.expert_ids, (1, 128, 128), N=128,
                                     rows_alloc=16)
    assert np.all(got == wl.SENTINEL_BF16) and stats[1] == 0 and status == binding.GMM_OK


@pytest.mark.parametrize("gran", [(1, 128, None), (1, 128, 128)])
def test_fp8_max_groups(gran):
    """4096 groups (the largest supported count) of 0..3 rows over 64 experts, both kernels."""
    rng = np.random.default_rng(70)
    G = 4096
    r, v = case(64, 256, 256, rng.integers(0, 4, G), rng.integers(-1, 64, G).astype(np.int32), 71, gran=gran)
    _, _, status, _ = check_fp8_against_oracle(handle(64), r, v, gran, where=f"fp8 max groups {gran}")
    assert status == binding.GMM_OK


@pytest.mark.parametrize("gran", [(1, 128, None), (1, 128, 128)])
def test_fp8_cuda_graph_replay(gran):
    """Both e4m3 kernels captured in a CUDA graph once and replayed on new inputs."""
    import torch
    h = handle(4)
    r = wl.make_routing("t", 4, 256, 512, [5, 130, 0, 77], [2, 0, -1, 3])
    v0 = wl.fp8_host_values(r, 90, gran)
    a8 = torch.empty(v0["a8"].shape, dtype=torch.uint8, device=DEV)
    w8 = torch.empty(v0["w8"].shape, dtype=torch.uint8, device=DEV)
    s_in = torch.empty(v0["input_scale"].shape, dtype=torch.float32, device=DEV)
    s_w = torch.empty(v0["weight_scale"].shape, dtype=torch.float32, device=DEV)
    c = sentinel_dev(r.rows, r.N, DEV)
    off, ids = to_dev_i32(r.a_offsets, DEV), to_dev_i32(r.expert_ids, DEV)
    st = to_dev_i32(np.zeros(4), DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    call = lambda: binding.gmm_run_fp8(h, c, a8, off, w8, ids, st, s_in, s_w, gran)
    with torch.cuda.stream(s):
        call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    live = live_row_mask(r.rows, r.a_offsets, r.expert_ids, r.E)
    gk = r.K if gran[2] is None else gran[2]
    for seed in (91, 92):
        v = wl.fp8_host_values(r, seed, gran)
        a8.copy_(to_dev_u8(v["a8"], DEV))
        w8.copy_(to_dev_u8(v["w8"], DEV))
        s_in.copy_(to_dev_f32(v["input_scale"], DEV))
        s_w.copy_(to_dev_f32(v["weight_scale"], DEV))
        g.replay()
        torch.cuda.synchronize()
        assert binding.gmm_query_status(h) == binding.GMM_OK
        ref = oracle.gmm_fp8(v["a8"], r.a_offsets, v["w8"], r.expert_ids, v["input_scale"], v["weight_scale"],
                             (gran[0], gran[1], gk))
        assert_close(bits_of(c), ref.ref32, live, f"graph replay fp8 {gran} seed {seed}")


@pytest.mark.parametrize("gran", [(1, 128, None), (1, 128, 128)])
def test_fp8_nan_codes_propagate_like_the_oracle(gran):
    """e4m3 NaN codes (S.1111.111) in A turn exactly the oracle's outputs into NaN."""
    r, v = case(3, 256, 256, [9, 40, 0, 17], [2, 0, 1, -1], 111, gran=gran)
    a8 = v["a8"].copy()
    a8[3, 5] = 0x7F
    a8[30, 200] = 0xFF
    v = dict(v, a8=a8)
    got, stats, status = run_gpu_fp8(handle(3), v, r.a_offsets, r.expert_ids, gran, N=r.N)
    gk = r.K if gran[2] is None else gran[2]
    ref = oracle.gmm_fp8(a8, r.a_offsets, v["w8"], r.expert_ids, v["input_scale"], v["weight_scale"],
                         (gran[0], gran[1], gk))
    live = live_row_mask(r.rows, r.a_offsets, r.expert_ids, r.E)
    gf = (got.astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(np.isnan(gf[live]), np.isnan(ref.ref32[live]))
    assert np.isnan(ref.ref32[3]).all() and np.isnan(ref.ref32[30]).all()
    finite_rows = live & np.isfinite(ref.ref32).all(axis=1)   # rows without a NaN input
    assert_close(got, ref.ref32, finite_rows, f"fp8 finite rows {gran}")
