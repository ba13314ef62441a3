// Block-scaled e4m3 grouped GEMM with per-K-block scales, for sm_103a.
//
// Operation (Modular "k_matmul_ragged_paged_scale" API page, section "Args":
// input_scale and weight_scale multiply the input and the weight; template
// parameter scales_granularity_mnk = (gm, gn, gk)), for each active group g with
// expert e and rows r of the group:
//   C[r, n] = bf16( sum_kb input_scale[r / gm, kb] * weight_scale[e, n / gn, kb]
//                          * sum_{k in block kb} a[r, k] * w[e, n, k] )
// then the optional epilogue, as in the grouped kernel.
//
// Each K block's partial sum is scaled before it joins the others, so the tensor
// core cannot accumulate over all of K.  The MMA writes each block's partial into
// one of two TMEM buffers; eight promotion warps per CTA fold it into a running fp32
// sum held in their registers, while the MMA fills the other buffer with the next
// block.
//
// Orientation.  Tokens are the MMA's M and weights its N (256 rows), unlike the
// grouped kernel: a TMEM lane is then a token row, so the input scale of a block is
// one value per thread, and with gn a multiple of 32 the weight scale is one value per
// 32-column TMEM load.  A promotion is one multiply-add per element.
//
// One CTA per tile of 128 token rows.  A K block of 128 is one stage, 512 cycles of
// tensor work at the e4m3 rate.  Two partial buffers leave the promotion little
// slack: the MMA of block kb + 2 waits for the release of block kb.  So a promotion
// warp reads a partial 64 columns per TMEM wait (two waits per block), releases the
// buffer as soon as its last load has landed, before that piece's multiply-adds, and
// folds two columns per paired fp32 FMA.  A microbenchmark of this pipeline alone
// (operands fixed in shared memory) runs a block in ~740 cycles with the promotion's
// loads and multiply-adds, against 512 with an immediate release: the fp32 work (one
// multiply-add per element, half the MMA time per block on each SM sub-partition)
// and the barrier round trips do not fit beside one block of MMAs.
// Tried and measured no better: 192- and 128-row tiles with 12 promotion warps or
// four partial buffers, a CTA-pair form (cta_group::2), whose every block crosses CTAs
// twice, N = 128 halves of each block with their own barriers, spinning instead of
// suspended barrier waits, a warp that stages the scales in shared memory, and
// 32-byte direct stores of C instead of the tensor stores.
//
// Roles (384 threads per CTA, three warpgroups):
//   warp 0       TMA producer: per stage (128 of K) a 128-row token slab (16 KB) and
//                the tile's 256 weight rows (32 KB), 128-byte swizzled.
//   warp 1       TMEM allocation (512 columns: two 256-column partial buffers) and the
//                MMA issue (kind::f8f6f4, M = 128, N = 256, 4 MMAs per stage).
//   warps 2, 3   idle.
//   warps 4..11  promotion and epilogue: warp w reads TMEM lane quadrant w % 4 and
//                weight columns 128 * ((w - 4) / 4) .. + 128 of each partial; every
//                thread owns one token row and 128 running sums.  After a tile's last
//                block they apply the epilogue and store their row's 128 columns.
//
// Registers: the launch gives every thread 168 (384 x 168 fills the register file).
// The first warpgroup then drops to 56 a thread and the two promotion warpgroups take
// 224: 128 running sums and a 64-column piece of a partial.  The host checks the
// launch register count before the first launch, since an increase the pool cannot
// cover would wait forever.
//
// Scheduling is the grouped kernel's static one (the same group scan and tile decode);
// every wait is bounded as there.
#pragma once

#include "gmm_kernel.cuh"

namespace gmm {

constexpr uint32_t kBwPromoWarps = 8;              // two per TMEM lane quadrant
constexpr uint32_t kBwFirstPromo = 4;              // warps 0..3: producer, MMA, two idle
constexpr int kBwThreads = 32 * (kBwFirstPromo + kBwPromoWarps);
constexpr uint32_t kBwLaunchRegs = 168;            // registers a thread at launch (the kernel's count)
constexpr uint32_t kBwRegsLow = 56;                // producer / MMA warpgroup after reallocation
constexpr uint32_t kBwRegsHigh = 224;              // promotion warpgroups after reallocation
static_assert(kBwLaunchRegs * kBwThreads <= 65536, "the launch fits the register file");
static_assert(128 * kBwRegsLow + 32 * kBwPromoWarps * kBwRegsHigh <= kBwLaunchRegs * kBwThreads,
              "the increase is covered by the launch's pool and the decrease");
constexpr uint32_t kBwCtaTok = 128;                // token rows per CTA (its TMEM lanes)
constexpr uint32_t kBwRows = 256;                  // weight rows per tile (MMA N)
constexpr uint32_t kBwBufs = kTmemCols / kBwRows;  // partial buffers in TMEM
constexpr uint32_t kBwTBytes = kBwCtaTok * 128;    // token slab of a stage: 128 rows x 128 e4m3
constexpr uint32_t kBwCols = kBwRows * 4 / kBwPromoWarps;   // weight columns per promotion warp
constexpr uint32_t kBwPiece = 64;                  // columns per TMEM wait
static_assert(kBwCols == 2 * kBwPiece, "a block is read in two pieces");
constexpr int kBwBiasBytes = kBwPromoWarps * kBwCols * 2;   // each promotion warp's bias columns (bf16)
constexpr uint32_t kBwStgBytes = 32 * 64;          // a promotion warp's C staging tile: 32 rows x 32 bf16
// Dynamic shared memory besides the stage ring and the group prefix: alignment slack,
// the C staging tiles and the bias columns.
constexpr int kBwFixedBytes = 1024 + static_cast<int>(kBwPromoWarps * kBwStgBytes) + kBwBiasBytes;

struct BwGeom {
  static constexpr uint32_t kRows = kBwRows;
  static constexpr uint32_t kMaxTok = kBwCtaTok;                 // token rows per tile
  static constexpr uint32_t kTokAlign = 16;
  static constexpr uint32_t kWBytes = kBwRows * 128;             // a stage's weight slab
  static constexpr uint32_t kStageBytes = kBwTBytes + kWBytes;   // shared memory per stage
};

// Each promotion thread keeps kBwCols running sums and a kBwPiece-column piece of a
// partial in registers.
__global__ void __launch_bounds__(kBwThreads, 1) gmm_fp8_block_kernel(const __grid_constant__ GmmParams p) {
  using G = BwGeom;
  __shared__ Ctrl ctl;
  __shared__ uint64_t part_full[kBwBufs];    // a block's partial is in the buffer (MMA commit)
  __shared__ uint64_t part_empty[kBwBufs];   // every promotion warp has read it
  extern __shared__ uint8_t dyn_smem[];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t ST = static_cast<uint32_t>(p.num_stages);
  const int KS = (p.K + kBK - 1) / kBK;   // stages per tile: 64 two-byte units = 128 e4m3 of K each
  const int SPB = p.kb_stages;            // stages per scale block (gk / 128)
  const int NKB = (KS + SPB - 1) / SPB;   // scale blocks per tile

  // Dynamic shared memory: the 1024-byte aligned rings, the promotion warps' C staging
  // tiles, their bias columns and the group prefix.
  const uint32_t dyn_base = smem_addr(dyn_smem);
  const uint32_t ring = (dyn_base + 1023u) & ~1023u;
  const uint32_t t_ring = ring;
  const uint32_t w_ring = ring + ST * kBwTBytes;
  const uint32_t c_stage = w_ring + ST * G::kWBytes;
  const uint32_t bias_stage = c_stage + kBwPromoWarps * kBwStgBytes;
  uint32_t *prefix = reinterpret_cast<uint32_t *>(dyn_smem + (bias_stage + kBwBiasBytes - dyn_base));

  if (tid == 0) {
    set_wait_limit(p.wait_limit_ns);
    for (uint32_t s = 0; s < ST; ++s) {
      mbar_init(smem_addr(&ctl.full[s]), 1);
      mbar_init(smem_addr(&ctl.empty[s]), 1);
    }
    for (uint32_t a = 0; a < kBwBufs; ++a) {
      mbar_init(smem_addr(&part_full[a]), 1);
      mbar_init(smem_addr(&part_empty[a]), kBwPromoWarps);
    }
    ctl.abort = 0;
    ctl.active = 0;
    ctl.flags = 0;
    ctl.max_group_tiles = 0;
    ctl.min_group_tiles = 0xffffffffu;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(&ctl.tmem_base), kTmemCols);
    tmem_relinquish();
    tc_fence_before_sync();
  }
  __syncthreads();
  build_schedule<G>(p, ctl, prefix, kBwThreads);
  if (blockIdx.x == 0 && tid == 0) {
    p.stats[1] = ctl.active;
    const uint32_t f = ctl.flags & (kStatusBadOffsets | kStatusBadExpert | kStatusTooLarge);
    if (f) atomicOr(p.status, f);
  }
  tc_fence_after_sync();
  const uint32_t tmem_base = ctl.tmem_base;
  const uint32_t total = ctl.total_tiles;
  volatile int *abort = &ctl.abort;
  const uint32_t unit0 = blockIdx.x;   // static share: tiles unit0, unit0 + units, ...
  const uint32_t units = gridDim.x;

  // Register reallocation: each setmaxnreg is executed by a whole warpgroup at one
  // place in the code, and the code after it is compiled for the new budget.  The
  // first warpgroup gives, the promotion warpgroups take.
  if (warp < static_cast<int>(kBwFirstPromo)) {
    warpgroup_regs_dec<kBwRegsLow>();
    if (warp == 0) {
      // ------------------------------------------------------------ TMA producer
      // The CTA's token map: the host's map with the row extent patched to a_offsets[G]
      // (rows past the end of A are zero-filled) and 128-row boxes.
      uint8_t *slot = p.map_slots + static_cast<size_t>(blockIdx.x) * kMapSlotBytes;
      if (total > 0 && lane == 0) {
        const uint4 *src = reinterpret_cast<const uint4 *>(&p.tok_map);
        uint4 *dst = reinterpret_cast<uint4 *>(slot);
#pragma unroll
        for (int i = 0; i < 8; ++i) dst[i] = src[i];
        tensormap_set_dim1(dst, __ldg(p.a_offsets + p.num_groups));
        tensormap_set_box1(dst, kBwCtaTok);
        tensormap_release();
        tensormap_acquire(slot);
        const CUtensorMap *tok = reinterpret_cast<const CUtensorMap *>(slot);
        prefetch_tensormap(&p.w_map);
        const uint64_t pol_first = l2_policy_evict_first();
        const uint64_t pol_last = l2_policy_evict_last();
        const uint64_t pol_normal = l2_policy_evict_normal();
        Ring rt;
        uint32_t pending = 0, pend_phase = 0;
        bool ok = true;
        for (uint32_t t = unit0; t < total && ok; t += units) {
          const Tile ti = decode_tile<G>(t, prefix, p);
          const uint64_t w_pol = (p.cache_hints && ti.single_block) ? pol_first : pol_normal;
          const uint64_t t_pol = p.cache_hints ? pol_last : pol_normal;
          const int32_t t_row = static_cast<int32_t>(ti.row0);
          const int32_t w_row = static_cast<int32_t>(ti.n0);
          for (int s = 0; s < KS; ++s) {
            const uint32_t full = smem_addr(&ctl.full[rt.slot]);
            if (!wait_phase(smem_addr(&ctl.empty[rt.slot]), rt.phase ^ 1u, abort)) { ok = false; break; }
            mbar_arrive_expect_tx(full, G::kStageBytes);
            const int32_t k0 = s * kBK;
            tma_load_2d_hint(t_ring + rt.slot * kBwTBytes, tok, full, k0, t_row, t_pol);
            tma_load_3d_hint(w_ring + rt.slot * G::kWBytes, &p.w_map, full, k0, w_row, ti.e, w_pol);
            pending |= 1u << rt.slot;
            pend_phase = (pend_phase & ~(1u << rt.slot)) | (rt.phase << rt.slot);
            rt.next(ST);
          }
        }
        if (!ok) {
          // Let the copies already issued land before the CTA can exit.
          for (uint32_t s = 0; s < ST; ++s)
            if (pending & (1u << s)) wait_phase_for(smem_addr(&ctl.full[s]), (pend_phase >> s) & 1u, kDrainLimitNs);
          atomicOr(p.status, kStatusTimeout);
        }
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issue (whole warp, one elected lane)
      if (total > 0) {
        Ring rt;
        uint32_t pb = 0, pb_phase = 0;   // partial buffer of the current block, and its use parity
        bool ok = true;
        const uint64_t t_desc0 = smem_desc_k_sw128(t_ring);
        const uint64_t w_desc0 = smem_desc_k_sw128(w_ring);
        const uint32_t t_lo = static_cast<uint32_t>(t_desc0), t_hi = static_cast<uint32_t>(t_desc0 >> 32);
        const uint32_t w_lo = static_cast<uint32_t>(w_desc0), w_hi = static_cast<uint32_t>(w_desc0 >> 32);
        const uint32_t idesc = idesc_e4m3_f32(kBwCtaTok, kBwRows);
        for (uint32_t t = unit0; t < total && ok; t += units) {
          int in_block = 0;   // stage within its scale block (s % SPB, counted)
          for (int s = 0; s < KS; ++s, in_block = (in_block + 1 == SPB) ? 0 : in_block + 1) {
            if (in_block == 0) {   // a new block starts in a free partial buffer
              const bool free_ =
                  __all_sync(0xffffffffu, wait_phase(smem_addr(&part_empty[pb]), pb_phase ^ 1u, abort));
              if (!free_) { ok = false; break; }
            }
            const bool staged = __all_sync(0xffffffffu, wait_phase(smem_addr(&ctl.full[rt.slot]), rt.phase, abort));
            if (!staged) { ok = false; break; }
            tc_fence_after_sync();
            // Four MMAs of K = 32 e4m3 (32 bytes) each, the stage's commit and, at the end of
            // a K block, the commit that hands its partial to the promotion warps.
            const bool block_end = in_block == SPB - 1 || s == KS - 1;
            mma_stage_f8_x4(tmem_base + pb * kBwRows, t_lo + ((rt.slot * kBwTBytes) >> 4), t_hi,
                            w_lo + ((rt.slot * G::kWBytes) >> 4), w_hi, idesc, in_block != 0,
                            smem_addr(&ctl.empty[rt.slot]), block_end, smem_addr(&part_full[pb]));
            rt.next(ST);
            if (block_end) {
              if (++pb == kBwBufs) {
                pb = 0;
                pb_phase ^= 1u;
              }
            }
          }
        }
        if (!ok && lane == 0) atomicOr(p.status, kStatusTimeout);
      }
    }
  } else {
    warpgroup_regs_inc<kBwRegsHigh>();
    // ------------------------------------------------------------ promotion and epilogue
    const uint32_t pw = static_cast<uint32_t>(warp) - kBwFirstPromo;   // promotion warp 0..7
    const uint32_t quad = static_cast<uint32_t>(warp & 3);
    const uint32_t part = pw >> 2;   // which kBwCols of the tile's columns
    // This thread's token row in the tile.
    const uint32_t trow = quad * 32 + static_cast<uint32_t>(lane);
    __nv_bfloat16 *bias_s = reinterpret_cast<__nv_bfloat16 *>(dyn_smem + (bias_stage - dyn_base)) + pw * kBwCols;
    const uint32_t stg = c_stage + pw * kBwStgBytes;   // this warp's C staging tile
    constexpr int kChunks = static_cast<int>(kBwCols / 32);
    const int wcols = p.w_scale_cols;
    // A tile's scale rows for this thread: its input scale row and the weight scale rows
    // of the warp's 32-column chunks (gn is a multiple of 32), as offsets from the
    // expert's first row (a column past N reads row 0 and is never stored).
    struct ScaleRows {
      const float *is_row;
      const float *ws_e;
      uint32_t ws_off[kChunks];
      bool row_ok;
    };
    auto scale_rows = [&](const Tile &x) {
      ScaleRows r;
      r.row_ok = trow < x.nrows;
      r.is_row = p.in_scale + static_cast<size_t>((x.row0 + trow) / static_cast<uint32_t>(p.scale_gm)) * p.scale_kb;
      r.ws_e = p.w_scale + static_cast<size_t>(x.e) * wcols * p.scale_kb;
#pragma unroll
      for (int c = 0; c < kChunks; ++c) {
        const uint32_t n = x.n0 + part * kBwCols + 32u * c;
        r.ws_off[c] = (n < static_cast<uint32_t>(p.N) ? n / static_cast<uint32_t>(p.scale_gn) : 0u) *
                      static_cast<uint32_t>(p.scale_kb);
      }
      return r;
    };
    // The scales of block kb + 1 are loaded while block kb is promoted, and those of the
    // next tile's first block (with the next tile's decode) before this tile's epilogue,
    // so no load's latency is waited for between blocks or between tiles.
    float isn = 0.0f, wsn[kChunks];
    auto load_scales = [&](const ScaleRows &r, int kb) {
      isn = r.row_ok ? __ldg(r.is_row + kb) : 0.0f;
#pragma unroll
      for (int c = 0; c < kChunks; ++c) wsn[c] = __ldg(r.ws_e + r.ws_off[c] + kb);
    };
    Tile tn{};
    ScaleRows sr{};   // the scale rows of the tile whose next block's scales are loaded
    if (unit0 < total) {
      tn = decode_tile<G>(unit0, prefix, p);
      sr = scale_rows(tn);
      load_scales(sr, 0);
    }
    uint32_t pb = 0, pb_phase = 0;
    bool ok = true;
    for (uint32_t t = unit0; t < total && ok; t += units) {
      const Tile ti = tn;
      const uint32_t ncol0 = ti.n0 + part * kBwCols;   // first of this warp's weight columns
      float acc[kBwCols];
#pragma unroll
      for (int j = 0; j < static_cast<int>(kBwCols); ++j) acc[j] = 0.0f;
      for (int kb = 0; kb < NKB; ++kb) {
        const float isv = isn;
        float wsv[kChunks];
#pragma unroll
        for (int c = 0; c < kChunks; ++c) wsv[c] = wsn[c];
        if (kb + 1 < NKB) load_scales(sr, kb + 1);
        int w_ok = 1;
        if (lane == 0) w_ok = wait_phase(smem_addr(&part_full[pb]), pb_phase, abort);
        if (!__shfl_sync(0xffffffffu, w_ok, 0)) { ok = false; break; }
        tc_fence_after_sync();
        const uint32_t taddr = tmem_base + ((quad * 32u) << 16) + pb * kBwRows + part * kBwCols;
#pragma unroll
        for (int h = 0; h < static_cast<int>(kBwCols / kBwPiece); ++h) {
          uint32_t v0[32], v1[32];
          tmem_ld_x32(taddr + kBwPiece * h, v0);
          tmem_ld_x32(taddr + kBwPiece * h + 32, v1);
          tmem_ld_wait();
          if (h == static_cast<int>(kBwCols / kBwPiece) - 1) {
            // Every load of the block has landed: release the buffer before the last
            // piece's multiply-adds.  Relaxed: the scale loads just issued stay in
            // flight instead of being waited for.
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive_relaxed(smem_addr(&part_empty[pb]));
          }
          const float f0 = isv * wsv[2 * h], f1 = isv * wsv[2 * h + 1];
          float *a = acc + kBwPiece * h;
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            fma_f32x2(a[j], a[j + 1], f0, __uint_as_float(v0[j]), __uint_as_float(v0[j + 1]));
            fma_f32x2(a[32 + j], a[33 + j], f1, __uint_as_float(v1[j]), __uint_as_float(v1[j + 1]));
          }
        }
        if (++pb == kBwBufs) {
          pb = 0;
          pb_phase ^= 1u;
        }
      }
      if (!ok) break;
      if (t + units < total) {   // the next tile, and its first block's scales (in flight during the epilogue)
        tn = decode_tile<G>(t + units, prefix, p);
        sr = scale_rows(tn);
        load_scales(sr, 0);
      }
      // Epilogue: act(y + bias[e, n]) * row_scale[r] on the finished sums, 32 columns at
      // a time.  When all 32 rows of the warp are in the group, a chunk is staged in
      // this warp's tile in TMA's 64-byte swizzle (16-byte block b of row r at
      // b ^ ((r >> 1) & 3)) and leaves through one tensor store of the 32 x 32 box,
      // which clips the columns past N; otherwise 16-byte stores masked to the group's
      // rows and to N (N is a multiple of 8: a group of 8 columns is in or past N whole).
      const bool fused = p.epi_bias != nullptr || p.epi_row_scale != nullptr || p.epi_act != kActNone;
      if (p.epi_bias != nullptr) {   // the warp's bias columns, staged once per tile
        __syncwarp();
#pragma unroll
        for (int i = 0; i < static_cast<int>(kBwCols / 32); ++i) {
          const uint32_t j = static_cast<uint32_t>(lane) * (kBwCols / 32) + i;
          const uint32_t n = ncol0 + j;
          bias_s[j] = n < static_cast<uint32_t>(p.N) ? p.epi_bias[static_cast<size_t>(ti.e) * p.N + n]
                                                      : __float2bfloat16_rn(0.0f);
        }
        __syncwarp();
      }
      const bool row_ok = trow < ti.nrows;
      const uint32_t grow = ti.row0 + trow;
      const float rs = (p.epi_row_scale != nullptr && row_ok) ? __ldg(p.epi_row_scale + grow) : 1.0f;
      const bool whole = p.c_tma && quad * 32u + 32u <= ti.nrows;
      __nv_bfloat16 *crow = p.c + static_cast<size_t>(grow) * p.N + ncol0;
#pragma unroll
      for (int cc = 0; cc < kChunks; ++cc) {
        uint32_t w[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          float y0 = acc[32 * cc + 2 * k], y1 = acc[32 * cc + 2 * k + 1];
          if (fused) {
            const float b0 = p.epi_bias != nullptr ? __bfloat162float(bias_s[32 * cc + 2 * k]) : 0.0f;
            const float b1 = p.epi_bias != nullptr ? __bfloat162float(bias_s[32 * cc + 2 * k + 1]) : 0.0f;
            y0 = epilogue_op(y0, b0, p.epi_act, rs);
            y1 = epilogue_op(y1, b1, p.epi_act, rs);
          }
          w[k] = pack_bf16x2(y0, y1);
        }
        if (whole && ncol0 + 32u * cc < static_cast<uint32_t>(p.N)) {   // (a box wholly past N: nothing to store)
          if (lane == 0) bulk_wait_read<0>();   // the previous store has read the staging tile
          __syncwarp();
          uint8_t *row_p = dyn_smem + (stg - dyn_base) + lane * 64;
#pragma unroll
          for (uint32_t b = 0; b < 4; ++b)
            *reinterpret_cast<uint4 *>(row_p + ((b ^ ((static_cast<uint32_t>(lane) >> 1) & 3u)) << 4)) =
                make_uint4(w[4 * b], w[4 * b + 1], w[4 * b + 2], w[4 * b + 3]);
          fence_async_smem();   // this thread's staging writes, before the async proxy reads them
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&p.c_map, stg, static_cast<int32_t>(ncol0 + 32u * cc), static_cast<int32_t>(ti.row0 + quad * 32u));
            bulk_commit();
          }
        } else if (row_ok) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (ncol0 + 32u * cc + 8u * q < static_cast<uint32_t>(p.N))
              *reinterpret_cast<uint4 *>(crow + 32 * cc + 8 * q) = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
        }
      }
    }
    if (lane == 0) bulk_wait_all();   // the tensor stores have read their staging tiles
    if (!ok && lane == 0) atomicOr(p.status, kStatusTimeout);
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace gmm
