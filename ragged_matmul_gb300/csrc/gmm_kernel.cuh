// Persistent, warp-specialised ragged grouped GEMM for sm_103a.
//
// Operation (Modular "grouped_matmul_sm100_persistent" API page, section
// "Args"): for each group g with expert e = expert_ids[g] in [0, E),
//   C[r, n] = bf16( sum_k A[r, k] * B[e, n, k] ),  r in [a_offsets[g], a_offsets[g+1]).
//
// Orientation.  The page's launcher swaps A and B so that the weights play the
// MMA's M role.  This kernel does the same for every tile: the MMA computes
//   D[n, t] = sum_k W[n, k] * T[t, k]      (M = 128 weight rows, N = tokens)
// so a tile holds 128 output columns of C and up to 256 token rows, and the
// token count of a tile only has to be a multiple of 16.  Small groups (decode)
// therefore pay for at most 15 padded tokens instead of a 128-row tile.
//
// Work decomposition.  A tile is (group g, n-block of 128 weight rows, token
// block of <= 256 rows of the group).  Every CTA scans a_offsets / expert_ids
// into a shared-memory prefix sum of tiles per group and walks tiles
// t = blockIdx.x, blockIdx.x + gridDim.x, ...; token blocks are the fastest
// index, so CTAs running at the same time share one weight panel in L2.
//
// Roles:
//   warp 0      TMA producer: weight slab [128 x 64] via a 3-D map over B
//               [E, N, K] (or the packed 4-bit words) and token slab [ntok x 64]
//               via 2-D maps over A, 128-byte swizzle, into an S-stage ring.
//   warp 1      TMEM allocation (512 columns = two 128 x 256 fp32 accumulators)
//               and the single MMA-issuing thread (tcgen05.mma kind::f16).
//   warps 2..5  epilogue: TMEM -> registers -> bf16 -> C, masking token rows past
//               the group's end and columns past N.  Two accumulators let the
//               epilogue of one tile overlap the main loop of the next.
//   warps 6..9  (4-bit variant only) dequantise the packed slab of each stage
//               into the bf16 weight slab the MMA reads.
//
// Row bounds.  The host does not know how many rows A has (that is
// a_offsets[G], on the device), so the token tensor maps are encoded with a
// placeholder extent and each CTA copies them into its own global slot and
// patches the row extent with tensormap.replace before its first copy.  Token
// rows past the end of A are then zero-filled by TMA instead of being read.
//
// Every wait is bounded (about 2 s of wall time); on expiry the kernel records
// a timeout in the status word, stops issuing work, drains its own copies and
// frees TMEM before returning.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "sm103_ptx.cuh"

namespace gmm {

constexpr int kBlockN = 128;                  // weight rows per tile (MMA M)
constexpr int kMaxTok = 256;                  // token rows per tile (MMA N, multiple of 16)
constexpr int kBK = 64;                       // K per stage: one 128-byte swizzle row of bf16
constexpr int kMaxStages = 8;
constexpr int kMaxGroups = 4096;
constexpr int kThreads = 192;                 // bf16 kernel: producer, MMA, 4 epilogue warps
constexpr int kInt4Threads = 320;             // 4-bit kernel: + 4 dequantisation warps
constexpr int kWBytes = kBlockN * kBK * 2;    // 16 KB weight slab
constexpr int kTBytes = kMaxTok * kBK * 2;    // 32 KB token slab
constexpr int kStageBytes = kWBytes + kTBytes;
constexpr int kQBytes = kBlockN * kBK / 2;    // 4 KB packed 4-bit slab (128 rows x 8 words)
constexpr int kInt4StageBytes = kStageBytes + kQBytes;
constexpr uint32_t kAccCols = 256;            // TMEM columns per accumulator
constexpr uint32_t kTmemCols = 2 * kAccCols;
constexpr int kMapSlotBytes = 256;            // per-CTA workspace: two patched 128-byte tensor maps

constexpr uint32_t kStatusBadOffsets = 1u;
constexpr uint32_t kStatusBadExpert = 2u;
constexpr uint32_t kStatusTimeout = 4u;
constexpr uint32_t kStatusTooLarge = 8u;

constexpr uint64_t kWaitLimitNs = 2000000000ull;   // give up on a pipeline wait after 2 s
constexpr uint64_t kDrainLimitNs = 200000000ull;   // and on draining copies after 0.2 s

struct alignas(128) GmmParams {
  CUtensorMap w_map;       // bf16 path: B {K, N, E}, box {64, 128, 1}, 128 B swizzle
                           // 4-bit path: packed words {K/8, N, E}, box {8, 128, 1}, no swizzle
  CUtensorMap tok_map128;  // A bf16 {K, rows}, box {64, 128} (rows patched on the device)
  CUtensorMap tok_map16;   // A bf16 {K, rows}, box {64, 16}  (rows patched on the device)
  __nv_bfloat16 *c;
  const uint32_t *a_offsets;
  const int32_t *expert_ids;
  uint32_t *stats;
  uint32_t *status;
  uint8_t *map_slots;
  int num_groups;
  int num_experts;
  int N;
  int K;
  int num_stages;
  const __nv_bfloat16 *scales;   // 4-bit path: [E, N, K / group_size]
  int group_size;                // 4-bit path: multiple of 64 dividing K
};

struct Tile {
  int32_t e;
  uint32_t row0;   // first token row of the tile
  uint32_t nrows;  // token rows that belong to the group (<= 256)
  uint32_t ntok;   // nrows rounded up to 16: the MMA's N
  uint32_t n0;     // first weight row / C column
};

struct __align__(8) Ctrl {
  uint64_t full[kMaxStages];    // TMA bytes of the stage landed
  uint64_t wfull[kMaxStages];   // 4-bit path: dequantised weight slab written
  uint64_t empty[kMaxStages];   // MMAs that read the stage completed
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint32_t tmem_base;
  int abort;
  uint32_t total_tiles;
  uint32_t active;
  uint32_t flags;
  unsigned long long warp_tiles[kInt4Threads / 32];
};

// Bounded wait on an mbarrier phase.  Returns false (and raises the CTA's abort
// flag) after kWaitLimitNs, or as soon as another role has aborted.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int *abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t spin = 1;; ++spin) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((spin & 63u) == 0) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        *abort = 1;
        return false;
      }
    }
  }
}

__device__ __forceinline__ bool wait_phase_for(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > limit_ns) return false;
  return true;
}

// Tiles of one group: token blocks of 256 rows times n-blocks of 128 columns.
__device__ __forceinline__ unsigned long long group_tiles(uint32_t rows, uint32_t n_blocks) {
  return static_cast<unsigned long long>((rows + kMaxTok - 1) / kMaxTok) * n_blocks;
}

// Scan a_offsets / expert_ids into prefix[g] = first tile of group g (all NT threads).
template <int NT>
__device__ void build_schedule(const GmmParams &p, Ctrl &ctl, uint32_t *prefix) {
  const int G = p.num_groups;
  const uint32_t n_blocks = static_cast<uint32_t>((p.N + kBlockN - 1) / kBlockN);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int chunk = (G + NT - 1) / NT;
  const int g_begin = min(G, tid * chunk), g_end = min(G, g_begin + chunk);

  unsigned long long mine = 0;
  uint32_t active = 0, flags = 0;
  for (int g = g_begin; g < g_end; ++g) {
    const uint32_t r0 = __ldg(p.a_offsets + g), r1 = __ldg(p.a_offsets + g + 1);
    const int32_t e = __ldg(p.expert_ids + g);
    if (r1 < r0) flags |= kStatusBadOffsets;
    if (e >= p.num_experts) flags |= kStatusBadExpert;
    if (e >= 0 && e < p.num_experts) {
      ++active;
      if (r1 > r0) mine += group_tiles(r1 - r0, n_blocks);
    }
    prefix[g + 1] = static_cast<uint32_t>(mine);   // running sum within the chunk, fixed up below
  }
  if (flags) atomicOr(&ctl.flags, flags);
  if (active) atomicAdd(&ctl.active, active);

  unsigned long long incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) ctl.warp_tiles[warp] = incl;
  __syncthreads();
  unsigned long long base = 0, total = 0;
  for (int w = 0; w < NT / 32; ++w) {
    if (w < warp) base += ctl.warp_tiles[w];
    total += ctl.warp_tiles[w];
  }
  base += incl - mine;
  for (int g = g_begin; g < g_end; ++g) prefix[g + 1] += static_cast<uint32_t>(base);
  if (tid == 0) {
    prefix[0] = 0;
    uint32_t t = static_cast<uint32_t>(total);
    if (total >= 0x7fffffffull) {
      atomicOr(&ctl.flags, kStatusTooLarge);
      t = 0;
    }
    ctl.total_tiles = t;
  }
  __syncthreads();
  if (tid == 0 && (ctl.flags & kStatusBadOffsets)) ctl.total_tiles = 0;   // reject the whole call
  __syncthreads();
}

__device__ __forceinline__ Tile decode_tile(uint32_t t, const uint32_t *prefix, const GmmParams &p) {
  int lo = 0, hi = p.num_groups - 1;   // last group whose first tile is <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const uint32_t local = t - prefix[lo];
  const uint32_t r0 = __ldg(p.a_offsets + lo);
  const uint32_t rows = __ldg(p.a_offsets + lo + 1) - r0;
  const uint32_t n_tok_blocks = (rows + kMaxTok - 1) / kMaxTok;
  const uint32_t nb = local / n_tok_blocks;
  const uint32_t tb = local - nb * n_tok_blocks;
  Tile x;
  x.e = __ldg(p.expert_ids + lo);
  x.row0 = r0 + tb * kMaxTok;
  x.nrows = min(static_cast<uint32_t>(kMaxTok), rows - tb * kMaxTok);
  x.ntok = (x.nrows + 15u) & ~15u;
  x.n0 = nb * kBlockN;
  return x;
}

// Dequantise one packed word (8 four-bit values, k = 8j .. 8j+7, low nibble first)
// into the 16-byte bf16 chunk the MMA expects: w_i = bf16((q_i - 8) * s).
// 0x4300 | q is the bf16 encoding of 128 + q (q < 16 fits the 7-bit mantissa at
// exponent 7), so subtracting 136 gives q - 8 exactly; the bf16x2 multiply then
// rounds the exact product (q - 8) * s once, to nearest even.
__device__ __forceinline__ uint4 dequant_word(uint32_t w, __nv_bfloat162 s2) {
  const __nv_bfloat162 bias = __floats2bfloat162_rn(136.0f, 136.0f);
  uint32_t pr[4];   // pr[i] = {w_i, w_{i+4}}
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t x = ((w >> (4 * i)) & 0x000F000Fu) | 0x43004300u;
    __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162 *>(&x);
    v = __hmul2(__hsub2(v, bias), s2);
    pr[i] = *reinterpret_cast<const uint32_t *>(&v);
  }
  uint4 out;
  out.x = __byte_perm(pr[0], pr[1], 0x5410);   // {w0, w1}
  out.y = __byte_perm(pr[2], pr[3], 0x5410);   // {w2, w3}
  out.z = __byte_perm(pr[0], pr[1], 0x7632);   // {w4, w5}
  out.w = __byte_perm(pr[2], pr[3], 0x7632);   // {w6, w7}
  return out;
}

// kInt4 = false: bf16 weights, 192 threads.  kInt4 = true: packed 4-bit weights
// dequantised by warps 6..9 into the stage's bf16 slab ahead of the MMA, 320 threads.
template <bool kInt4>
__global__ void __launch_bounds__(kInt4 ? kInt4Threads : kThreads, 1)
    gmm_grouped_kernel(const __grid_constant__ GmmParams p) {
  constexpr int NT = kInt4 ? kInt4Threads : kThreads;
  __shared__ Ctrl ctl;
  __shared__ uint32_t prefix[kMaxGroups + 1];
  extern __shared__ uint8_t dyn_smem[];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = p.num_stages;
  const int KB = (p.K + kBK - 1) / kBK;

  // 1024-byte aligned ring: S weight slabs, S token slabs, then (4-bit) S packed slabs.
  const uint32_t dyn_base = smem_addr(dyn_smem);
  const uint32_t ring = (dyn_base + 1023u) & ~1023u;
  const uint32_t w_ring = ring;
  const uint32_t t_ring = ring + S * kWBytes;
  const uint32_t q_ring = t_ring + S * kTBytes;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_addr(&ctl.full[s]), 1);
      mbar_init(smem_addr(&ctl.wfull[s]), 4 * 32);
      mbar_init(smem_addr(&ctl.empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_addr(&ctl.acc_full[a]), 1);
      mbar_init(smem_addr(&ctl.acc_empty[a]), 4 * 32);
    }
    ctl.abort = 0;
    ctl.active = 0;
    ctl.flags = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(&ctl.tmem_base), kTmemCols);
    tmem_relinquish();
    tc_fence_before_sync();
  }
  __syncthreads();
  build_schedule<NT>(p, ctl, prefix);

  if (blockIdx.x == 0 && tid == 0) {
    p.stats[1] = ctl.active;
    const uint32_t f = ctl.flags & (kStatusBadOffsets | kStatusBadExpert | kStatusTooLarge);
    if (f) atomicOr(p.status, f);
  }
  tc_fence_after_sync();
  const uint32_t tmem_base = ctl.tmem_base;
  const uint32_t total = ctl.total_tiles;
  volatile int *abort = &ctl.abort;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && total > 0) {
      uint8_t *slot = p.map_slots + static_cast<size_t>(blockIdx.x) * kMapSlotBytes;
      const uint4 *src128 = reinterpret_cast<const uint4 *>(&p.tok_map128);
      const uint4 *src16 = reinterpret_cast<const uint4 *>(&p.tok_map16);
      uint4 *dst = reinterpret_cast<uint4 *>(slot);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        dst[i] = src128[i];
        dst[8 + i] = src16[i];
      }
      const uint32_t rows = __ldg(p.a_offsets + p.num_groups);
      tensormap_set_dim1(slot, rows);
      tensormap_set_dim1(slot + 128, rows);
      tensormap_publish(slot);
      tensormap_publish(slot + 128);
      const CUtensorMap *tok128 = reinterpret_cast<const CUtensorMap *>(slot);
      const CUtensorMap *tok16 = reinterpret_cast<const CUtensorMap *>(slot + 128);
      prefetch_tensormap(&p.w_map);

      uint32_t stage = 0, phase = 0;
      uint32_t pending = 0;     // bit s: stage s has copies whose completion this thread has not seen
      uint32_t pend_phase = 0;  // bit s: the phase in which they complete
      bool ok = true;
      for (uint32_t t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const Tile ti = decode_tile(t, prefix, p);
        const uint32_t tx = (kInt4 ? kQBytes : kWBytes) + ti.ntok * (kBK * 2);
        for (int kb = 0; kb < KB; ++kb) {
          const uint32_t full = smem_addr(&ctl.full[stage]);
          if (!wait_phase(smem_addr(&ctl.empty[stage]), phase ^ 1u, abort)) { ok = false; break; }
          mbar_arrive_expect_tx(full, tx);
          const int32_t k0 = kb * kBK;
          if (kInt4)
            tma_load_3d(q_ring + stage * kQBytes, &p.w_map, full, k0 / 8, static_cast<int32_t>(ti.n0), ti.e);
          else
            tma_load_3d(w_ring + stage * kWBytes, &p.w_map, full, k0, static_cast<int32_t>(ti.n0), ti.e);
          uint32_t dst_t = t_ring + stage * kTBytes;
          int32_t r = static_cast<int32_t>(ti.row0);
          uint32_t left = ti.ntok;
          for (; left >= 128; left -= 128, r += 128, dst_t += 128 * kBK * 2)
            tma_load_2d(dst_t, tok128, full, k0, r);
          for (; left > 0; left -= 16, r += 16, dst_t += 16 * kBK * 2)
            tma_load_2d(dst_t, tok16, full, k0, r);
          pending |= 1u << stage;
          pend_phase = (pend_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == static_cast<uint32_t>(S)) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) {
        // Let the copies already issued land before the CTA can exit.
        for (int s = 0; s < S; ++s)
          if (pending & (1u << s))
            wait_phase_for(smem_addr(&ctl.full[s]), (pend_phase >> s) & 1u, kDrainLimitNs);
        atomicOr(p.status, kStatusTimeout);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && total > 0) {
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (uint32_t t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const Tile ti = decode_tile(t, prefix, p);
        if (!wait_phase(smem_addr(&ctl.acc_empty[acc]), acc_phase ^ 1u, abort)) { ok = false; break; }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + acc * kAccCols;
        const uint32_t idesc = idesc_bf16_f32(kBlockN, ti.ntok);
        for (int kb = 0; kb < KB; ++kb) {
          if (!wait_phase(smem_addr(&ctl.full[stage]), phase, abort)) { ok = false; break; }
          if (kInt4 && !wait_phase(smem_addr(&ctl.wfull[stage]), phase, abort)) { ok = false; break; }
          tc_fence_after_sync();
          const uint64_t a_desc = smem_desc_k_sw128(w_ring + stage * kWBytes);
          const uint64_t b_desc = smem_desc_k_sw128(t_ring + stage * kTBytes);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)   // +32 bytes along K per step: +2 in the >>4 address field
            mma_bf16(d_tmem, a_desc + 2u * k, b_desc + 2u * k, idesc, (kb | k) != 0);
          mma_commit(smem_addr(&ctl.empty[stage]));
          if (++stage == static_cast<uint32_t>(S)) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        mma_commit(smem_addr(&ctl.acc_full[acc]));
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      if (!ok) atomicOr(p.status, kStatusTimeout);
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------ epilogue
    const uint32_t quad = static_cast<uint32_t>(warp & 3);   // TMEM lanes this warp may read
    uint32_t acc = 0, acc_phase = 0;
    for (uint32_t t = blockIdx.x; t < total; t += gridDim.x) {
      const Tile ti = decode_tile(t, prefix, p);
      int ok = 1;
      if (lane == 0) ok = wait_phase(smem_addr(&ctl.acc_full[acc]), acc_phase, abort);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        if (lane == 0) atomicOr(p.status, kStatusTimeout);
        break;
      }
      tc_fence_after_sync();
      const uint32_t n = ti.n0 + quad * 32 + static_cast<uint32_t>(lane);
      const bool col_ok = n < static_cast<uint32_t>(p.N);
      __nv_bfloat16 *cp = p.c + static_cast<size_t>(ti.row0) * p.N + n;
      const uint32_t taddr = tmem_base + ((quad * 32u) << 16) + acc * kAccCols;
      for (uint32_t c0 = 0; c0 < ti.ntok; c0 += 16) {
        uint32_t v[16];
        tmem_ld_x16(taddr + c0, v);
        tmem_ld_wait();
        if (col_ok) {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (c0 + j < ti.nrows)
              cp[static_cast<size_t>(c0 + j) * p.N] = __float2bfloat16_rn(__uint_as_float(v[j]));
        }
      }
      tc_fence_before_sync();
      mbar_arrive(smem_addr(&ctl.acc_empty[acc]));
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
  } else if (kInt4) {
    // ------------------------------------------------------------ 4-bit dequantisation
    // Thread r (0..127) owns weight row n0 + r of every stage: 8 packed words in,
    // 8 swizzled 16-byte bf16 chunks out (chunk j of row r lands at j ^ (r % 8)).
    const uint32_t r = static_cast<uint32_t>(tid - 6 * 32);
    const int spr = p.K / p.group_size;   // scales per weight row
    uint32_t stage = 0, phase = 0;
    bool ok = true;
    for (uint32_t t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const Tile ti = decode_tile(t, prefix, p);
      const uint32_t n = ti.n0 + r;
      const bool row_ok = n < static_cast<uint32_t>(p.N);
      const __nv_bfloat16 *srow = p.scales + (static_cast<size_t>(ti.e) * p.N + (row_ok ? n : 0)) * spr;
      for (int kb = 0; kb < KB; ++kb) {
        const __nv_bfloat16 s = row_ok ? srow[(kb * kBK) / p.group_size] : __float2bfloat16_rn(0.0f);
        if (!wait_phase(smem_addr(&ctl.full[stage]), phase, abort)) { ok = false; break; }
        const uint4 *q = reinterpret_cast<const uint4 *>(dyn_smem + (q_ring - dyn_base) + stage * kQBytes + r * 32);
        const uint4 q0 = q[0], q1 = q[1];
        const uint32_t words[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        const __nv_bfloat162 s2 = __halves2bfloat162(s, s);
        uint8_t *wrow = dyn_smem + (w_ring - dyn_base) + stage * kWBytes + r * 128;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          *reinterpret_cast<uint4 *>(wrow + ((j ^ (r & 7)) << 4)) = dequant_word(words[j], s2);
        fence_async_smem();   // generic-proxy writes -> visible to the tensor core's reads
        mbar_arrive(smem_addr(&ctl.wfull[stage]));
        if (++stage == static_cast<uint32_t>(S)) { stage = 0; phase ^= 1u; }
      }
    }
    if (!ok) atomicOr(p.status, kStatusTimeout);
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace gmm
