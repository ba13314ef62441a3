// Persistent, warp-specialised ragged grouped GEMM for sm_103a.
//
// Operation (Modular "grouped_matmul_sm100_persistent" API page, section
// "Args"): for each group g with expert e = expert_ids[g] in [0, E),
//   C[r, n] = bf16( sum_k A[r, k] * B[e, n, k] ),  r in [a_offsets[g], a_offsets[g+1]).
//
// Orientation.  The page's launcher swaps A and B so that the weights play the
// MMA's M role.  This kernel does the same for every tile: the MMA computes
//   D[n, t] = sum_k W[n, k] * T[t, k]      (M = weight rows, N = tokens)
// so the token count of a tile only has to be a multiple of 16 (32 for a CTA
// pair).  Small groups (decode) pay for at most a few padded tokens instead of a
// 128-row tile.
//
// Work decomposition.  A tile is (group g, n-block of weight rows, token block of
// the group).  Every CTA scans a_offsets / expert_ids into a shared-memory prefix
// sum of tiles per group; within a group the token blocks are the fastest index
// (in L2-sized bands), so CTAs running at the same time share one weight panel in
// L2.  The producer thread (of the pair leader) decides the tile sequence and
// publishes it in a small shared-memory queue that every other role reads in order.
// With many tiles per CTA (at least kDynamicTilesPerUnit, or ...4) it claims tiles from a
// global counter, one tile ahead of its loads, so CTAs that draw cheaper tiles
// simply take more; with few tiles per CTA the claim costs more than the balance
// gains, and it takes the static round-robin share t = unit, unit + units, ...
//
// Variants (template parameters):
//   kPair = false  one CTA per tile, 128 weight rows, tcgen05 cta_group::1 (M = 128).
//   kPair = true   a cluster of two CTAs per tile, 256 weight rows, cta_group::2
//                  (M = 256): CTA r holds weight rows n0 + 128 r .. + 128 and half
//                  of the tokens; the leader (r = 0) issues the MMAs and commits to
//                  both CTAs' barriers; each CTA stores its own 128 columns of C.
//   kInt4 = false  bf16 weights, loaded by TMA into the stage together with tokens.
//   kInt4 = true   packed 4-bit weights: a dedicated TMA warp
//                  streams packed slabs through their own ring, and twelve warps
//                  dequantise them straight into tensor memory, where the MMA takes
//                  its A operand from (tcgen05.mma with A in TMEM).  The dequantised
//                  weights never touch shared memory, so shared memory carries only
//                  the token slabs and the packed slabs, and no proxy fence sits
//                  between the dequantisation and the MMA.
//   kFp8 = true    (with kInt4 = false) e4m3 operands, block-scaled (Modular
//                  "k_matmul_ragged_paged_scale", section "Args": input_scale and
//                  weight_scale; template parameter scales_granularity_mnk).  An
//                  e4m3 row of K elements is K bytes, i.e. the bf16 kernel's rows
//                  with K / 2 two-byte units: the host encodes the same tensor maps
//                  over the bytes, every stage carries 128 of K in the same
//                  128-byte swizzled rows, and the MMA is kind::f8f6f4 (K = 32 per
//                  instruction: the same 32 bytes per step).  The scales of the
//                  (gm, gn, K) granularity are applied in the epilogue:
//                    y = acc * input_scale[r / gm] * weight_scale[e, n / gn].
//
// Roles:
//   warp 0       TMA producer of token slabs (and of bf16 weight slabs).
//   warp 1       TMEM allocation (512 columns: two fp32 accumulators, and in the
//                4-bit kernel a ring of dequantised weight slabs between them) and
//                the MMA issue (the whole warp runs the loop, one elected lane
//                issues tcgen05.mma kind::f16, or kind::f8f6f4 for e4m3).
//   warps 2..5   epilogue: TMEM (16x256b loads) -> scales, optional bias /
//                activation / row scale -> bf16 -> stmatrix.trans into a
//                shared-memory staging tile (the transpose from weight-row lanes
//                to C rows) -> 16-byte stores to C, masking token rows past the
//                group's end and columns past N; two accumulators let it overlap
//                the next tile's main loop.  A 448-thread launch (bf16 / e4m3 with
//                short K) adds warps 6..13: the three warps of a TMEM lane quadrant
//                take every third 32-row chunk.
//   warp 6       (4-bit) TMA producer of packed slabs.
//   warps 7..18  (4-bit) dequantisation.
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

constexpr int kBlockN = 128;                  // weight rows per CTA and tile (MMA M of one CTA)
constexpr int kBK = 64;                       // K per stage: one 128-byte swizzle row of bf16
constexpr int kMaxStages = 12;                // deepest W+T stage ring
constexpr int kMaxGroups = 4096;
constexpr int kThreads = 192;                 // bf16 kernel: producer, MMA, 4 epilogue warps
// With short K a tile is a few stages, and storing its accumulator takes longer than
// computing it: the bf16 / e4m3 kernel then runs 12 epilogue warps, three per TMEM lane
// quadrant, each taking every third 32-row chunk (lora_qkv, K = 64: 0.0407 ms with 8
// warps, 0.0371 with 12; 16 would leave 96 registers a thread and spill).
constexpr int kThreadsWide = 448;
constexpr int kWideEpilogueMaxK = 512;
// 4-bit kernel: 64-wide K sub-slabs per stage, and the dequantisation warps.  The
// 12 warps form kDqGroups groups that take the stages in turn (stage s goes to group
// s % kDqGroups), so each warp has kDqGroups stage-times for its loop of waits,
// loads, arithmetic, TMEM store and arrive, whose fixed latency alone is longer
// than a stage.  Within a group, each TMEM lane quadrant gets kDqWarpsPerStage / 4
// warps with a thread per weight row, each covering kDqSubsPerWarp 64-K sub-slabs.
constexpr int kSub4 = 2;
constexpr int kDqGroups = 3;
constexpr int kDequantThreads = 384;
constexpr int kDqWarpsPerStage = kDequantThreads / 32 / kDqGroups;       // 4: one per quadrant
constexpr int kDqSubsPerWarp = kSub4 * 4 / kDqWarpsPerStage;             // 2: the whole 128 of K
static_assert(kDqWarpsPerStage % 4 == 0 && kDqSubsPerWarp >= 1, "every quadrant and sub-slab covered");
constexpr int kInt4Threads = kThreads + 32 + kDequantThreads;   // + one packed-slab producer warp
constexpr int kWBytes = kBlockN * kBK * 2;    // 16 KB bf16 weight slab
// 4-bit kernel, packed ring: a slot holds a chunk of kQChunkStages stages, 128 bytes of
// each weight row (one TMA box of 128 rows x 32 words, 128-byte swizzle).  Whole
// 128-byte rows make full-line DRAM requests, a quarter as many as 32-byte rows.
constexpr int kQChunkStages = 2;
constexpr int kQRowBytes = kQChunkStages * kSub4 * kBK / 2;   // 128
constexpr int kQSlotBytes = kBlockN * kQRowBytes;            // 16 KB
constexpr int kQStages = 4;                                  // slots (at most): 8 stages ahead
constexpr int kQRingBytes = kQStages * kQSlotBytes;
static_assert(kQRowBytes == 128, "the packed chunk is one 128-byte swizzle row per weight row");
// Epilogue staging: each epilogue warp transposes 32 token rows x its 32 C columns
// at a time through a bf16 tile in shared memory (stmatrix in, 16-byte row reads out),
// so that every thread stores 8 consecutive columns of one C row with one 16-byte
// store.  A tile row is 64 bytes (four 16-byte blocks); block b of row r sits at
// b ^ ((r >> 1) & 3), which keeps both the 8-row matrix writes and the row reads free
// of bank conflicts.
constexpr uint32_t kEpiRows = 32;
constexpr uint32_t kEpiRowBytes = 64;
constexpr int kEpiStageBytes = 12 * kEpiRows * kEpiRowBytes;   // up to 12 epilogue warps
template <bool kInt4>
constexpr uint32_t kEpiBytes = kInt4 ? 4 * kEpiRows * kEpiRowBytes : kEpiStageBytes;   // the 4-bit kernel has 4
constexpr uint32_t kAccCols = 256;            // TMEM columns per accumulator
constexpr uint32_t kTmemCols = 2 * kAccCols;
// 4-bit kernel: dequantised weight slabs live in TMEM (128 lanes = weight rows, 32
// columns = 64 bf16 of K per 64-wide slab) in the columns the accumulators leave
// free: an accumulator holds at most 160 token columns (kMaxTok), so columns
// 160..255 and 416..511 hold six slabs, kAStages = 6 / kSub4 stages of them: set s
// has its first 64 of K at column 160 + 32 s and its second at 256 columns further.  A
// stage is its token slab and its TMEM weight slabs together: one barrier tells the
// MMA that both are ready, one commit frees both.  The token ring is deeper than the
// slab ring (a multiple of kAStages, as deep as shared memory allows): stage s uses
// barriers and token slot s % depth, and TMEM slab set s % kAStages.  A token copy
// comes from L2 with about 1,900 cycles of latency under load, longer than the
// tensor work of two stages, so a ring of three token slots left the MMAs waiting for
// tokens at every stage.  128-K stages measured faster than 64-K stages: the MMA
// thread's fixed cost per stage outweighs a finer ring.
constexpr uint32_t kASlabs = 6;
constexpr uint32_t kAStages = kASlabs / kSub4;
constexpr uint32_t kASlab0 = 160;    // column of slab set 0's first 64 of K
__device__ __forceinline__ uint32_t a_slab_col(uint32_t set, uint32_t sub) {
  return kASlab0 + 32u * set + kAccCols * sub;
}
constexpr int kTokMaps = 16;                  // token maps per CTA: boxes of 16, 32, ..., 256 rows
constexpr int kMapSlotBytes = kTokMaps * 128; // per-CTA workspace: the patched 128-byte token maps
constexpr int kTileQueue = 8;                 // entries of the shared-memory tile queue
constexpr uint32_t kDynamicTilesPerUnit = 16; // bf16: dynamic tile claiming from this many tiles per CTA (pair)
constexpr uint32_t kDynamicTilesPerUnit4 = 8; // 4-bit: the same (its tiles are longer, measured better lower)
constexpr uint32_t kUnevenRatio = 4;          // groups this uneven get the two-ended claim order
constexpr uint32_t kNoTile = 0xffffffffu;     // queue entry meaning "no more tiles"

constexpr int kActNone = 0;       // activations of the optional epilogue (the C ABI's GMM_ACT_* values)
constexpr int kActRelu = 1;
constexpr int kActSilu = 2;
constexpr int kActGeluTanh = 3;

constexpr uint32_t kStatusBadOffsets = 1u;
constexpr uint32_t kStatusBadExpert = 2u;
constexpr uint32_t kStatusTimeout = 4u;
constexpr uint32_t kStatusTooLarge = 8u;

constexpr uint64_t kWaitLimitNs = 2000000000ull;   // give up on a pipeline wait after 2 s (by default)
constexpr uint32_t kSuspendNs = 1u << 20;            // longest suspension of one mbarrier test (~1 ms)
constexpr uint64_t kDrainLimitNs = 200000000ull;   // and on draining copies after 0.2 s

// Geometry of one kernel variant.
template <bool kInt4, bool kPair>
struct Geom {
  static constexpr uint32_t kRows = kPair ? 2 * kBlockN : kBlockN;   // weight rows (C columns) per tile
  static constexpr uint32_t kTokAlign = kPair ? 32 : 16;             // MMA N granule (pair: 2 x 16)
  // Token rows per tile.  The 4-bit path keeps slabs small so its token ring can be
  // deep: its MMA per stage is short (about 128 tokens), and the token copies come
  // from L2 with microsecond latency.
  static constexpr uint32_t kMaxTok = kInt4 ? 160 : 256;   // 4-bit: also bounded by the TMEM layout above
  static constexpr uint32_t kCtaTok = kPair ? kMaxTok / 2 : kMaxTok;   // token rows one CTA loads, at most
  static constexpr uint32_t kTSlot = kCtaTok * kBK * 2;                 // token slab per CTA
  static_assert(kCtaTok % 16 == 0 && kCtaTok / 16 <= kTokMaps, "a token map per 16-row slab height");
  static_assert(kTSlot % 1024 == 0, "token slabs must keep the 1024-byte swizzle alignment");
  // 64-wide K sub-slabs per pipeline stage.  The bf16 pair kernel takes 128 of K per
  // stage (8 MMAs per barrier wait and commit): the MMA thread's fixed cost per stage
  // (wait, fence, commit, loop) is then spread over twice the tensor work.  The 4-bit
  // kernel's width is kSub4 (see the TMEM layout above).
  static constexpr uint32_t kSub = kInt4 ? kSub4 : (kPair ? 2 : 1);
  // Shared memory of one stage of the W+T ring (the 4-bit kernel's weights are in TMEM).
  static constexpr uint32_t kStageBytes = kSub * ((kInt4 ? 0 : kWBytes) + kTSlot);
};

struct alignas(128) GmmParams {
  CUtensorMap w_map;       // bf16 path: B {K, N, E}, box {64, 128, 1}, 128 B swizzle
                           // 4-bit path: packed words {K/8, N, E}, box {8, 128, 1}, no swizzle
  CUtensorMap c_map;       // C bf16 {N, 2^31 rows}, box {32, 32}, 64-byte swizzle (valid when c_tma)
  CUtensorMap tok_map;     // A bf16 {K, rows}, box {64, 128}; each CTA derives from it one map per
                           // box height (16, 32, ... rows) and patches the row extent on the device
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
  int num_stages;                // depth of the W+T stage ring
  int q_stages;                  // 4-bit path: slots of the packed ring (kQStages, or 2 when shared memory is short)
  const __nv_bfloat16 *scales;   // 4-bit path: [E, N, K / group_size]
  int group_size;                // 4-bit path: multiple of 64 dividing K
  int scale_shift;               // 4-bit path: log2(group_size / 64) when that is a power of two, else -1
  int tok_band;                  // token blocks per band of the tile order (see decode_tile)
  uint32_t *tile_counter;        // workspace, 8-byte aligned, zero between launches: [0..1] one 64-bit claim
                                 // word (tiles claimed from the front | from the back << 32), [2] CTAs finished
  int cache_hints;               // 1: L2 eviction priorities on the TMA loads (see the producer)
  int c_tma;                     // 1: whole 32-row chunks of C leave through c_map (TMA stores)
  // Optional elementwise epilogue on the fp32 result before it is rounded to bf16:
  //   y = act(acc + bias[e, n]) * row_scale[r]      (each part optional)
  const __nv_bfloat16 *epi_bias;   // [E, N] or null
  const float *epi_row_scale;      // [rows of A] or null
  int epi_act;                     // kActNone, kActRelu, kActSilu, kActGeluTanh
  // Block scales of the e4m3 path, applied first: acc * in_scale[r / scale_gm] *
  // w_scale[e * w_scale_cols + n / scale_gn] (in_scale null: no scaling).
  const float *in_scale;           // [ceil(rows / scale_gm)]
  const float *w_scale;            // [E, w_scale_cols]
  int scale_gm;
  int scale_gn;
  int w_scale_cols;                // ceil(N / scale_gn)
  // Per-K-block scales (the block-scaled kernel): scale_kb = ceil(K / gk) values per
  // scale row, kb_stages = gk / 128 pipeline stages per block.
  int scale_kb;
  int kb_stages;
  // A-plane row offsetting (both 0: off): A holds three planes of M = a_offsets[G] rows;
  // C columns n < plane_s0 read plane 0, n < plane_s0 + plane_s1 plane 1, the rest plane 2.
  // Both are multiples of 256, so a tile's weight rows lie in one plane.
  int plane_s0;
  int plane_s1;
  // Test hooks of the timeout path, both off (0 / -1) in normal use: a shorter limit on
  // every pipeline wait, and (one-CTA bf16 kernel) a stage, counted from 0 over the
  // launch, for which the producer issues neither copies nor its arrival, so that the
  // stage never fills and the waits behind it give up with nothing in flight.
  unsigned long long wait_limit_ns;
  int test_stall_stage;
};

struct __align__(32) Tile {
  int32_t e;
  uint32_t single_block;   // the group fits one token block: its weight panels are read once
  uint32_t row0;           // first token row of the tile
  uint32_t nrows;          // token rows that belong to the group
  uint32_t ntok;           // nrows rounded up to the MMA granule: the MMA's N
  uint32_t n0;             // first weight row / C column of the tile
  uint32_t pad[2];         // to 32 bytes: a queue entry is read with two 16-byte loads
};

struct __align__(32) Ctrl {   // 32: the tile queue entries inside
  uint64_t full[kMaxStages];     // stage's TMA bytes landed (pair: both CTAs' bytes, on the leader);
                                 // 4-bit: and its TMEM weight slabs written by every dequantisation
                                 // warp (pair: of both CTAs)
  uint64_t empty[kMaxStages];    // MMAs that read the stage completed
  uint64_t qfull[kQStages];      // 4-bit: a packed chunk landed
  uint64_t qempty[kQStages];     // 4-bit: the dequantisation warps are done with a packed chunk
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t maps_ready;           // epilogue warp 2 has written this CTA's token maps
  uint64_t tq_full[kTileQueue];  // tile queue entry published
  uint64_t tq_empty[kTileQueue]; // every reader has taken the entry (pair: both CTAs', on the leader)
  uint32_t tq_tile[kTileQueue];
  Tile tq_info[kTileQueue];      // the entry's tile, decoded once by the publisher
  uint32_t tmem_base;
  int abort;
  uint32_t total_tiles;
  uint32_t max_group_tiles;      // largest and smallest non-zero tile count of a group
  uint32_t min_group_tiles;
  uint32_t active;
  uint32_t flags;
  unsigned long long warp_tiles[kInt4Threads / 32];
};

// A ring position: slot index and the parity of the slot's current use.
struct Ring {
  uint32_t slot = 0, phase = 0;
  __device__ __forceinline__ void next(uint32_t depth) {
    if (++slot == depth) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

// The CTA's limit on one pipeline wait: kWaitLimitNs, unless the launch asks for a
// shorter one (GmmParams::wait_limit_ns, a test of the timeout path).  Set by thread 0
// before the kernel's first block-wide barrier.
__shared__ uint64_t s_wait_limit_ns;

__device__ __forceinline__ void set_wait_limit(uint64_t requested) {
  s_wait_limit_ns = requested != 0 ? requested : kWaitLimitNs;
}

// Bounded wait on an mbarrier phase.  Returns false (and raises the CTA's abort
// flag) after s_wait_limit_ns, or as soon as another role has aborted.  Each test may
// suspend the thread for up to kSuspendNs (it resumes as soon as the phase
// completes), so a waiting role does not spin on the issue slots that the dequant,
// epilogue and MMA-issuing warps of its SM need; the abort flag and the clock are
// checked after every test.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int *abort) {
  if (mbar_test_wait(bar, parity)) return true;   // already complete: no potentially blocking test
  if (mbar_try_wait_hint(bar, parity, kSuspendNs)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (*abort) return false;
    if (global_timer_ns() - t0 > s_wait_limit_ns) {
      *abort = 1;
      return false;
    }
    if (mbar_try_wait_hint(bar, parity, kSuspendNs)) return true;
  }
}

// The same at cluster scope, for barriers the peer CTA arrives on: with acquire
// semantics, or relaxed (kRelaxed) where the phase publishes no generic-proxy writes.
template <bool kRelaxed = false>
__device__ __forceinline__ bool wait_phase_cluster(uint32_t bar, uint32_t parity, volatile int *abort) {
  auto test = [&]() {
    return kRelaxed ? mbar_test_wait_cluster_relaxed(bar, parity) : mbar_test_wait_cluster(bar, parity);
  };
  auto try_wait = [&]() {
    return kRelaxed ? mbar_try_wait_cluster_relaxed_hint(bar, parity, kSuspendNs)
                    : mbar_try_wait_cluster_hint(bar, parity, kSuspendNs);
  };
  if (test()) return true;
  if (try_wait()) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (*abort) return false;
    if (global_timer_ns() - t0 > s_wait_limit_ns) {
      *abort = 1;
      return false;
    }
    if (try_wait()) return true;
  }
}

__device__ __forceinline__ bool wait_phase_for(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait_hint(bar, parity, kSuspendNs))
    if (global_timer_ns() - t0 > limit_ns) return false;
  return true;
}

// Scan a_offsets / expert_ids into prefix[g] = first tile of group g (all nt threads).
template <class G>
__device__ void build_schedule(const GmmParams &p, Ctrl &ctl, uint32_t *prefix, int nt) {
  const int Gn = p.num_groups;
  const uint32_t n_blocks = static_cast<uint32_t>((p.N + G::kRows - 1) / G::kRows);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int chunk = (Gn + nt - 1) / nt;
  const int g_begin = min(Gn, tid * chunk), g_end = min(Gn, g_begin + chunk);

  unsigned long long mine = 0;
  uint32_t active = 0, flags = 0, gmax = 0, gmin = 0xffffffffu;
  for (int g = g_begin; g < g_end; ++g) {
    const uint32_t r0 = __ldg(p.a_offsets + g), r1 = __ldg(p.a_offsets + g + 1);
    const int32_t e = __ldg(p.expert_ids + g);
    if (r1 < r0) flags |= kStatusBadOffsets;
    if (e >= p.num_experts) flags |= kStatusBadExpert;
    if (e >= 0 && e < p.num_experts) {
      ++active;
      if (r1 > r0) {
        const uint32_t tb = (r1 - r0 + G::kMaxTok - 1) / G::kMaxTok;
        mine += static_cast<unsigned long long>(tb) * n_blocks;
        gmax = max(gmax, tb);
        gmin = min(gmin, tb);
      }
    }
    prefix[g + 1] = static_cast<uint32_t>(mine);   // running sum within the chunk, fixed up below
  }
  if (flags) atomicOr(&ctl.flags, flags);
  if (active) atomicAdd(&ctl.active, active);
  if (gmax) {
    atomicMax(&ctl.max_group_tiles, gmax);
    atomicMin(&ctl.min_group_tiles, gmin);
  }

  unsigned long long incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) ctl.warp_tiles[warp] = incl;
  __syncthreads();
  unsigned long long base = 0, total = 0;
  for (int w = 0; w < nt / 32; ++w) {
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

// Tile t -> (group, n-block, token block).  Within a group the token blocks are cut
// into bands of p.tok_band blocks; a band is walked n-block by n-block with its token
// blocks fastest.  CTAs running at the same time then share one weight panel, and the
// band's activations stay in L2 while the weight panels of the whole expert stream
// past.
template <class G>
__device__ __forceinline__ Tile decode_tile(uint32_t t, const uint32_t *prefix, const GmmParams &p) {
  int lo = 0, hi = p.num_groups - 1;   // last group whose first tile is <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const uint32_t local = t - prefix[lo];
  const uint32_t r0 = __ldg(p.a_offsets + lo);
  const uint32_t rows = __ldg(p.a_offsets + lo + 1) - r0;
  const uint32_t n_tok_blocks = (rows + G::kMaxTok - 1) / G::kMaxTok;
  const uint32_t n_blocks = (static_cast<uint32_t>(p.N) + G::kRows - 1) / G::kRows;
  const uint32_t band = static_cast<uint32_t>(p.tok_band);
  const uint32_t band_idx = local / (band * n_blocks);
  const uint32_t in_band = local - band_idx * band * n_blocks;
  const uint32_t band_len = min(band, n_tok_blocks - band_idx * band);
  const uint32_t nb = in_band / band_len;
  const uint32_t tb = band_idx * band + (in_band - nb * band_len);
  Tile x;
  x.e = __ldg(p.expert_ids + lo);
  x.single_block = n_tok_blocks == 1;
  x.row0 = r0 + tb * G::kMaxTok;
  x.nrows = min(G::kMaxTok, rows - tb * G::kMaxTok);
  x.ntok = (x.nrows + G::kTokAlign - 1) & ~(G::kTokAlign - 1);
  x.n0 = nb * G::kRows;
  return x;
}

// First A row of the plane that the tile's weight rows n0 .. read (A-plane row
// offsetting; 0 when it is off).
__device__ __forceinline__ uint32_t plane_row0(const GmmParams &p, uint32_t n0, uint32_t m_rows) {
  if ((p.plane_s0 | p.plane_s1) == 0) return 0u;
  const uint32_t plane = (n0 >= static_cast<uint32_t>(p.plane_s0) ? 1u : 0u) +
                         (n0 >= static_cast<uint32_t>(p.plane_s0 + p.plane_s1) ? 1u : 0u);
  return plane * m_rows;
}

// Two fp32 values -> one 32-bit word of two bf16 (round to nearest even), the lower
// column in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&v);
}

// The optional epilogue of one output element: bias, then activation, then row scale.
//   relu(y) = max(y, 0);  silu(y) = y / (1 + e^-y);
//   gelu(y) = y/2 * (1 + tanh(sqrt(2/pi) * (y + 0.044715 y^3)))   (the tanh form of GELU)
__device__ __forceinline__ float epilogue_op(float y, float bias, int act, float scale) {
  y += bias;
  if (act == kActRelu) {
    y = fmaxf(y, 0.0f);
  } else if (act == kActSilu) {
    y = __fdividef(y, 1.0f + __expf(-y));   // a huge denominator gives 0, the limit
  } else if (act == kActGeluTanh) {
    const float kSqrt2OverPi = 0.7978845608028654f;
    y = 0.5f * y * (1.0f + tanhf(kSqrt2OverPi * (y + 0.044715f * y * y * y)));
  }
  return y * scale;
}

// Dequantise one packed word (8 four-bit values, k = 8j .. 8j+7, low nibble first)
// into four bf16 pairs in K order (one TMEM column each): w_i = bf16((q_i - 8) * s).
// 0x4300 | q is the bf16 encoding of 128 + q (q < 16 fits the 7-bit mantissa at
// exponent 7), so subtracting 136 gives q - 8 exactly; the bf16x2 multiply then
// rounds the exact product (q - 8) * s once, to nearest even.  The bytes are put in
// place with byte permutes: the even nibbles (w & 0x0F0F0F0F) and the odd ones
// ((w >> 4) & 0x0F0F0F0F, the shift done as a high multiply) are interleaved into
// q0..q3 and q4..q7, and each pair then takes 0x43 as its high bytes.
__device__ __forceinline__ uint4 dequant_word(uint32_t w, __nv_bfloat162 s2) {
  const __nv_bfloat162 bias = __floats2bfloat162_rn(136.0f, 136.0f);
  const uint32_t ev = w & 0x0F0F0F0Fu;                       // q0 q2 q4 q6
  const uint32_t od = __umulhi(w, 1u << 28) & 0x0F0F0F0Fu;   // q1 q3 q5 q7
  const uint32_t a = __byte_perm(ev, od, 0x5140);            // q0 q1 q2 q3
  const uint32_t b = __byte_perm(ev, od, 0x7362);            // q4 q5 q6 q7
  constexpr uint32_t kHi = 0x43434343u;
  const uint32_t x[4] = {__byte_perm(a, kHi, 0x4140), __byte_perm(a, kHi, 0x4342),
                         __byte_perm(b, kHi, 0x4140), __byte_perm(b, kHi, 0x4342)};
  uint32_t out[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162 *>(&x[i]);
    v = __hmul2(__hsub2(v, bias), s2);
    out[i] = *reinterpret_cast<const uint32_t *>(&v);
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

// Reader of the tile queue (one thread).  Returns 1 with *tile and *info set (the
// publisher decodes each tile once and stores it with the entry, so readers need no
// global loads), 0 when the work is done, -1 when a wait gave up.  `empty0` is the
// address of the leader CTA's tq_empty[0] (a cluster address in the pair's second
// CTA, which then arrives remotely; that CTA's entries are published by the leader,
// so it waits with cluster scope).  The entry is copied out before the arrive that
// lets the publisher reuse it.
struct TileQueueReader {
  uint32_t pos = 0;
  __device__ __forceinline__ int next(Ctrl &ctl, uint32_t empty0, bool remote, volatile int *abort,
                                      uint32_t *tile, Tile *info) {
    const uint32_t slot = pos % kTileQueue, parity = (pos / kTileQueue) & 1u;
    const uint32_t full = smem_addr(&ctl.tq_full[slot]);
    if (!(remote ? wait_phase_cluster(full, parity, abort) : wait_phase(full, parity, abort))) return -1;
    *tile = *reinterpret_cast<volatile uint32_t *>(&ctl.tq_tile[slot]);
    if (*tile != kNoTile) {
      const volatile Tile &src = ctl.tq_info[slot];
      info->e = src.e;
      info->single_block = src.single_block;
      info->row0 = src.row0;
      info->nrows = src.nrows;
      info->ntok = src.ntok;
      info->n0 = src.n0;
    }
    const uint32_t empty = empty0 + slot * static_cast<uint32_t>(sizeof(uint64_t));
    if (remote) mbar_arrive_cluster(empty); else mbar_arrive(empty);
    ++pos;
    return *tile == kNoTile ? 0 : 1;
  }
};

// Where a role gets its tiles: with few tiles per CTA the static round-robin share
// (unit, unit + units, ...), computed and decoded by every role itself; with many,
// the queue.
struct TileSource {
  bool dynamic;
  uint32_t next_static, units, total;
  TileQueueReader q;
  __device__ __forceinline__ TileSource(bool dyn, uint32_t unit0, uint32_t units_, uint32_t total_)
      : dynamic(dyn), next_static(unit0), units(units_), total(total_) {}
  template <class G>
  __device__ __forceinline__ int next(Ctrl &ctl, uint32_t empty0, bool remote, volatile int *abort,
                                      const uint32_t *prefix, const GmmParams &p, Tile *info) {
    uint32_t tile;
    if (!dynamic) {
      if (next_static >= total) return 0;
      tile = next_static;
      next_static += units;
      *info = decode_tile<G>(tile, prefix, p);
      return 1;
    }
    return q.next(ctl, empty0, remote, abort, &tile, info);
  }
};

// The same for a whole warp: lane 0 waits for the entry, every lane reads it (two
// 16-byte loads of the same shared-memory words), then lane 0 releases it.
template <class G>
__device__ __forceinline__ int next_tile_warp(TileSource &src, Ctrl &ctl, uint32_t empty0, bool remote,
                                              volatile int *abort, const uint32_t *prefix, const GmmParams &p,
                                              Tile *info) {
  if (!src.dynamic) return src.next<G>(ctl, empty0, remote, abort, prefix, p, info);
  TileQueueReader &q = src.q;
  const uint32_t slot = q.pos % kTileQueue, parity = (q.pos / kTileQueue) & 1u;
  int ok = 1;
  if ((threadIdx.x & 31) == 0) {
    const uint32_t full = smem_addr(&ctl.tq_full[slot]);
    ok = remote ? wait_phase_cluster(full, parity, abort) : wait_phase(full, parity, abort);
  }
  if (!__shfl_sync(0xffffffffu, ok, 0)) return -1;
  __syncwarp();   // orders the other lanes' reads after lane 0's acquire
  const uint32_t tile = *reinterpret_cast<volatile uint32_t *>(&ctl.tq_tile[slot]);
  const uint4 w0 = ld_shared_v4(smem_addr(&ctl.tq_info[slot]));
  const uint4 w1 = ld_shared_v4(smem_addr(&ctl.tq_info[slot]) + 16u);
  __syncwarp();
  if ((threadIdx.x & 31) == 0) {
    const uint32_t empty = empty0 + slot * static_cast<uint32_t>(sizeof(uint64_t));
    if (remote) mbar_arrive_cluster(empty); else mbar_arrive(empty);
  }
  ++q.pos;
  if (tile == kNoTile) return 0;
  info->e = static_cast<int32_t>(w0.x);
  info->single_block = w0.y;
  info->row0 = w0.z;
  info->nrows = w0.w;
  info->ntok = w1.x;
  info->n0 = w1.y;
  return 1;
}

template <bool kInt4, bool kPair, bool kFp8 = false>
__global__ void __launch_bounds__(kInt4 ? kInt4Threads : kThreadsWide, 1)
    gmm_grouped_kernel(const __grid_constant__ GmmParams p) {
  static_assert(!(kInt4 && kFp8), "the e4m3 path has its weights in shared memory");
  using G = Geom<kInt4, kPair>;
  // Epilogue warps 2 .. 2 + n_epi - 1: 4, or 12 in a wide launch (bf16 / e4m3 only).
  const uint32_t n_epi = kInt4 ? 4u : blockDim.x / 32u - 2u;
  const uint32_t epi_arrivals = (kPair ? 2u : 1u) * n_epi;   // one per epilogue warp of each CTA
  constexpr uint32_t kDequantWarps = kDequantThreads / 32;
  // Arrivals per phase of a stage's `full` barrier: the token producer's (which also
  // sets the expected bytes) and, 4-bit, one per dequantisation warp of the stage's
  // group in each CTA.
  constexpr uint32_t kFullArrivals = 1 + (kInt4 ? (kPair ? 2 : 1) * kDqWarpsPerStage : 0);
  __shared__ Ctrl ctl;
  extern __shared__ uint8_t dyn_smem[];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t ST = static_cast<uint32_t>(p.num_stages);   // W+T stage ring (4-bit: tokens only)
  const int QS = kInt4 ? p.q_stages : 0;   // packed ring: 2 or 4 slots
  const uint32_t q_shift = QS == 4 ? 2u : 1u;
  const uint32_t SW = kInt4 ? 0u : ST;                         // weight slabs in shared memory
  const int KB = (p.K + static_cast<int>(G::kSub * kBK) - 1) / static_cast<int>(G::kSub * kBK);   // stages per tile
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;
  // Readers of each tile-queue entry: per CTA the MMA thread (leader only), the
  // epilogue warps and (4-bit) the packed-slab producer and the dequantisation
  // warps; in the pair's second CTA also its token producer.
  const uint32_t leader_readers = 1 + n_epi + (kInt4 ? 1 + kDequantWarps : 0);
  const uint32_t peer_readers = 1 + n_epi + (kInt4 ? 1 + kDequantWarps : 0);
  const uint32_t queue_arrivals = leader_readers + (kPair ? peer_readers : 0);

  // 1024-byte aligned rings, at identical offsets in both CTAs of a pair:
  // SW weight slabs (bf16), ST token slabs, then (4-bit) QS packed slabs, the epilogue
  // staging tiles, and the group prefix (as many entries as groups, G + 1).
  const uint32_t dyn_base = smem_addr(dyn_smem);
  const uint32_t ring = (dyn_base + 1023u) & ~1023u;
  const uint32_t w_ring = ring;
  const uint32_t t_ring = ring + SW * G::kSub * kWBytes;
  const uint32_t q_ring = t_ring + ST * G::kSub * G::kTSlot;   // 4-bit only
  const uint32_t epi_ring = q_ring + static_cast<uint32_t>(QS) * kQSlotBytes;   // epilogue staging tiles
  uint32_t *prefix = reinterpret_cast<uint32_t *>(dyn_smem + (epi_ring + kEpiBytes<kInt4> - dyn_base));

  if (tid == 0) {
    set_wait_limit(p.wait_limit_ns);
    for (uint32_t s = 0; s < ST; ++s) {
      mbar_init(smem_addr(&ctl.full[s]), kFullArrivals);
      mbar_init(smem_addr(&ctl.empty[s]), 1);
    }
    for (int s = 0; s < QS; ++s) {
      mbar_init(smem_addr(&ctl.qfull[s]), 1);
      mbar_init(smem_addr(&ctl.qempty[s]), kQChunkStages * kDqWarpsPerStage);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_addr(&ctl.acc_full[a]), 1);
      mbar_init(smem_addr(&ctl.acc_empty[a]), epi_arrivals);
    }
    mbar_init(smem_addr(&ctl.maps_ready), 1);
    for (int q = 0; q < kTileQueue; ++q) {
      mbar_init(smem_addr(&ctl.tq_full[q]), 1);
      mbar_init(smem_addr(&ctl.tq_empty[q]), queue_arrivals);
    }
    ctl.abort = 0;
    ctl.active = 0;
    ctl.flags = 0;
    ctl.max_group_tiles = 0;
    ctl.min_group_tiles = 0xffffffffu;
    fence_barrier_init();
  }
  if (warp == 1) {
    if constexpr (kPair) {
      tmem_alloc_pair(smem_addr(&ctl.tmem_base), kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_addr(&ctl.tmem_base), kTmemCols);
      tmem_relinquish();
    }
    tc_fence_before_sync();
  }
  __syncthreads();
  build_schedule<G>(p, ctl, prefix, static_cast<int>(blockDim.x));
  if constexpr (kPair) cluster_sync();   // the peer's barriers are initialised before anyone signals them

  if (blockIdx.x == 0 && tid == 0) {
    p.stats[1] = ctl.active;
    const uint32_t f = ctl.flags & (kStatusBadOffsets | kStatusBadExpert | kStatusTooLarge);
    if (f) atomicOr(p.status, f);
  }
  tc_fence_after_sync();
  const uint32_t tmem_base = ctl.tmem_base;
  const uint32_t total = ctl.total_tiles;
  volatile int *abort = &ctl.abort;
  // Tile-queue plumbing: readers arrive on the leader's tq_empty (remotely from the
  // pair's second CTA, which also waits on its entries with cluster scope).
  const uint32_t unit0 = kPair ? cluster_id_x() : blockIdx.x;   // this CTA's (pair's) static share
  const uint32_t units = kPair ? cluster_count_x() : gridDim.x;
  const bool dynamic = total >= (kInt4 ? kDynamicTilesPerUnit4 : kDynamicTilesPerUnit) * units;   // all CTAs agree
  const bool q_remote = kPair && rank != 0;
  const uint32_t q_empty0 = q_remote ? map_to_rank(smem_addr(&ctl.tq_empty[0]), 0) : smem_addr(&ctl.tq_empty[0]);

  if (warp == 0) {
    // ------------------------------------------------------------ token (and bf16 weight) producer
    // The token maps (one per copy height) are written by epilogue warp 2 while this
    // thread decodes its first tile; they are acquired before the first copy.
    constexpr int kMaps = static_cast<int>(G::kCtaTok / 16);
    uint8_t *slot = p.map_slots + static_cast<size_t>(blockIdx.x) * kMapSlotBytes;
    if (lane == 0 && total > 0) {
      bool maps_acquired = false;
      const CUtensorMap *tok_maps = reinterpret_cast<const CUtensorMap *>(slot);
      prefetch_tensormap(&p.w_map);
      const uint64_t pol_first = l2_policy_evict_first();
      const uint64_t pol_last = l2_policy_evict_last();
      const uint64_t pol_normal = l2_policy_evict_normal();

      const uint32_t m_rows = __ldg(p.a_offsets + p.num_groups);   // rows of one A plane
      Ring rt;
      int issued_stages = 0;    // stages of this launch so far (the timeout test's stall counts them)
      uint32_t pending = 0;     // bit s: stage s has copies whose completion this thread has not seen
      uint32_t pend_phase = 0;  // bit s: the phase in which they complete
      bool ok = true;
      // The leader's producer decides the tile sequence and publishes it one tile
      // ahead of its own loads, so the other roles (the packed-slab producer, the
      // pair's second CTA) can cross tile boundaries without waiting; dynamic claims
      // run two tiles ahead so the atomic's latency stays hidden.  Elsewhere the
      // producer reads the queue like every other role.
      TileSource reader(dynamic, unit0, units, total);
      uint32_t qpos = 0;
      // When group sizes are very uneven (the largest group has kUnevenRatio times the
      // token blocks of the smallest), half of the CTAs (pairs) claim from the back of
      // the tile order: they stream the weights of the small groups while the others
      // run the compute-heavy tiles of the large groups from the front, so the tensor
      // and HBM bounds overlap.  Both ends share one 64-bit claim word and meet
      // exactly; where they meet adapts to how fast each side goes.  With even groups
      // every claim comes from the front, which keeps more reuse in L2.
      const bool two_ended = ctl.max_group_tiles >= kUnevenRatio * ctl.min_group_tiles;
      const bool from_back = two_ended && (unit0 & 1u);
      // A claim is the atomic on the claim word (issued as early as possible) and,
      // once its old value is needed, the tile it names.
      auto claim_issue = [&]() -> unsigned long long {
        return atomicAdd(reinterpret_cast<unsigned long long *>(p.tile_counter), from_back ? (1ull << 32) : 1ull);
      };
      auto claim_tile = [&](unsigned long long old) -> uint32_t {
        const uint32_t front = static_cast<uint32_t>(old), back = static_cast<uint32_t>(old >> 32);
        if (static_cast<unsigned long long>(front) + back >= total) return kNoTile;
        return from_back ? total - 1u - back : front;
      };
      auto publish = [&](uint32_t t, Tile *info) -> bool {
        const uint32_t slot = qpos % kTileQueue, parity = (qpos / kTileQueue) & 1u;
        const uint32_t empty = smem_addr(&ctl.tq_empty[slot]);
        if (!(kPair ? wait_phase_cluster(empty, parity ^ 1u, abort) : wait_phase(empty, parity ^ 1u, abort)))
          return false;
        ctl.tq_tile[slot] = t;
        const Tile x = t == kNoTile ? Tile{} : decode_tile<G>(t, prefix, p);
        ctl.tq_info[slot] = x;
        *info = x;
        if constexpr (kPair) {   // the second CTA's copy of the entry, then its signal
          st_shared_cluster_u32(map_to_rank(smem_addr(&ctl.tq_tile[slot]), 1), t);
          const uint32_t *xw = reinterpret_cast<const uint32_t *>(&x);
          const uint32_t info1 = map_to_rank(smem_addr(&ctl.tq_info[slot]), 1);
#pragma unroll
          for (int i = 0; i < static_cast<int>(sizeof(Tile) / 4); ++i) st_shared_cluster_u32(info1 + 4u * i, xw[i]);
          mbar_arrive_cluster(map_to_rank(smem_addr(&ctl.tq_full[slot]), 1));
        }
        mbar_arrive(smem_addr(&ctl.tq_full[slot]));
        ++qpos;
        return true;
      };
      const bool publisher = dynamic && rank == 0;
      uint32_t cur = kNoTile, nxt = kNoTile;   // tile being loaded; tile already published after it
      Tile cur_info{}, nxt_info{};              // their decoded forms, kept from publishing
      if (publisher) {
        cur = claim_tile(claim_issue());
        nxt = cur == kNoTile ? kNoTile : claim_tile(claim_issue());
        ok = publish(cur, &cur_info) && (cur == kNoTile || publish(nxt, &nxt_info));
      }
      for (; ok;) {
        Tile ti;
        // The publisher claims the tile after `nxt` once this tile's first stage is
        // issued, and decodes and publishes it after the second: readers need it only a
        // tile later, and the copies of a new tile start without that work in between.
        uint32_t after = kNoTile;
        Tile after_info{};
        unsigned long long claim_old = 0;
        if (publisher) {
          if (cur == kNoTile) break;
          ti = cur_info;
        } else {
          const int got = reader.next<G>(ctl, q_empty0, q_remote, abort, prefix, p, &ti);
          if (got < 0) ok = false;
          if (got <= 0) break;
        }
        const uint32_t my_tok = kPair ? ti.ntok / 2 : ti.ntok;     // token rows this CTA loads
        const uint32_t tx =
            (kPair ? 2u : 1u) * G::kSub * ((kInt4 ? 0u : static_cast<uint32_t>(kWBytes)) + my_tok * (kBK * 2));
        const int32_t w_row = static_cast<int32_t>(ti.n0 + rank * kBlockN);
        // L2 priorities: a weight panel that only one token block of its group reads is
        // streamed once (evict first); token slabs are read again by every n-block of the
        // group (evict last), so streaming weights do not wash them out of L2.
        const uint64_t w_pol = (p.cache_hints && ti.single_block) ? pol_first : pol_normal;
        const uint64_t t_pol = p.cache_hints ? pol_last : pol_normal;
        if (!maps_acquired) {
          if (!wait_phase(smem_addr(&ctl.maps_ready), 0, abort)) { ok = false; break; }
          for (int i = 0; i < kMaps; ++i) tensormap_acquire(slot + i * 128);
          maps_acquired = true;
        }
        for (int kb = 0; kb < KB; ++kb, ++issued_stages) {
          const uint32_t full_local = smem_addr(&ctl.full[rt.slot]);
          if (!wait_phase(smem_addr(&ctl.empty[rt.slot]), rt.phase ^ 1u, abort)) { ok = false; break; }
          if (!kPair && !kInt4 && issued_stages == p.test_stall_stage) {   // test hook: this stage never fills
            rt.next(ST);
            continue;
          }
          if (rank == 0) mbar_arrive_expect_tx(full_local, tx);
          const int32_t r = static_cast<int32_t>(ti.row0 + rank * my_tok + plane_row0(p, ti.n0, m_rows));
          const CUtensorMap *tok = tok_maps + (my_tok / 16u - 1u);   // copies my_tok rows high
          if constexpr (kInt4) {
            // All kSub sub-slabs of the stage in one copy (3-D token map): sub-slab s
            // lands at +s * my_tok rows; one past K is zero-filled by TMA.
            const uint32_t dst_t = t_ring + rt.slot * G::kSub * G::kTSlot;
            const int32_t s0 = kb * static_cast<int32_t>(G::kSub);
            if constexpr (kPair) tma_load_3d_pair(dst_t, tok, map_to_rank(full_local, 0), 0, r, s0, t_pol);
            else tma_load_3d_hint(dst_t, tok, full_local, 0, r, s0, t_pol);
          }
#pragma unroll
          for (uint32_t sub = 0; sub < G::kSub && !kInt4; ++sub) {
            // Sub-slab `sub` of the stage: K from k0, weights at +sub*16 KB, tokens at
            // +sub*kTSlot.  A sub-slab past K is zero-filled by TMA and adds nothing.
            const int32_t k0 = (kb * static_cast<int32_t>(G::kSub) + static_cast<int32_t>(sub)) * kBK;
            const uint32_t dst_w = w_ring + (rt.slot * G::kSub + sub) * kWBytes;
            const uint32_t dst_t = t_ring + (rt.slot * G::kSub + sub) * G::kTSlot;
            if constexpr (kPair) {
              const uint32_t full_leader = map_to_rank(full_local, 0);
              tma_load_3d_pair(dst_w, &p.w_map, full_leader, k0, w_row, ti.e, w_pol);
              tma_load_2d_pair(dst_t, tok, full_leader, k0, r, t_pol);
            } else {
              tma_load_3d_hint(dst_w, &p.w_map, full_local, k0, w_row, ti.e, w_pol);
              tma_load_2d_hint(dst_t, tok, full_local, k0, r, t_pol);
            }
          }
          pending |= 1u << rt.slot;
          pend_phase = (pend_phase & ~(1u << rt.slot)) | (rt.phase << rt.slot);
          rt.next(ST);
          if (publisher && nxt != kNoTile) {
            if (kb == 0) claim_old = claim_issue();
            if (kb == (KB > 1 ? 1 : 0)) {
              after = claim_tile(claim_old);
              if (!publish(after, &after_info)) { ok = false; break; }
            }
          }
        }
        if (!ok) break;
        if (publisher) {
          cur = nxt;
          cur_info = nxt_info;
          if (cur != kNoTile) {
            nxt = after;
            nxt_info = after_info;
          }
        }
      }
      if (!ok) {
        // Let the copies already issued land before the CTA can exit.  In a pair only the
        // leader can observe `full` (it counts both CTAs' bytes); the peer is held at the
        // final cluster barrier until the leader has drained.
        for (uint32_t s = 0; s < ST; ++s)
          if ((pending & (1u << s)) && rank == 0)
            wait_phase_for(smem_addr(&ctl.full[s]), (pend_phase >> s) & 1u, kDrainLimitNs);
        atomicOr(p.status, kStatusTimeout);
      }
    }
  } else if (warp == 1) {
    if (total > 0 && rank == 0) {
      // ---------------------------------------------------------- MMA issuer (the leader of a pair)
      // The whole warp runs this loop with identical values in every lane, so the MMA
      // operands are warp-uniform; the tcgen05 wrappers issue from one elected lane.
      // Descriptors are a per-ring base plus a constant offset in the >>4 address field
      // (shared-memory addresses stay below 256 KB, so the 14-bit field never carries).
      Ring rt;
      uint32_t acc = 0, acc_phase = 0;
      uint32_t aset = 0;   // 4-bit: TMEM weight-slab set of the next stage (stage % kAStages)
      bool ok = true;
      TileSource reader(dynamic, unit0, units, total);
      const uint64_t t_desc0 = smem_desc_k_sw128(t_ring);
      const uint32_t t_lo = static_cast<uint32_t>(t_desc0), t_hi = static_cast<uint32_t>(t_desc0 >> 32);
      const uint32_t full0 = smem_addr(&ctl.full[0]), empty0 = smem_addr(&ctl.empty[0]);
      const uint64_t w_desc0 = smem_desc_k_sw128(w_ring);
      for (;;) {
        Tile ti;
        const int got = next_tile_warp<G>(reader, ctl, q_empty0, q_remote, abort, prefix, p, &ti);
        if (got < 0) ok = false;
        if (got <= 0) break;
        const bool acc_free = __all_sync(
            0xffffffffu, kPair ? wait_phase_cluster<true>(smem_addr(&ctl.acc_empty[acc]), acc_phase ^ 1u, abort)
                               : wait_phase(smem_addr(&ctl.acc_empty[acc]), acc_phase ^ 1u, abort));
        if (!acc_free) { ok = false; break; }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + acc * kAccCols;
        const uint32_t idesc = kFp8 ? idesc_e4m3_f32(G::kRows, ti.ntok) : idesc_bf16_f32(G::kRows, ti.ntok);
        if constexpr (kInt4) {
          // One instruction stream per stage (mma_stage_ts_x8): the wait for the stage,
          // its eight MMAs and the commit.  The pair's stage is also signalled by the
          // second CTA's dequantisation warps, so it is tested at cluster scope, relaxed:
          // their TMEM stores are ordered by tcgen05 fences and the token bytes by the
          // barrier.  The stage's two token sub-slabs sit my_tok rows apart (one 3-D
          // copy); its weight slabs are TMEM slab set `aset` (stage % kAStages).
          const uint32_t tok_step = ((kPair ? ti.ntok / 2 : ti.ntok) * (kBK * 2)) >> 4;
          for (int kb = 0; kb < KB; ++kb) {
            const uint32_t b0 = t_lo + rt.slot * ((G::kSub * G::kTSlot) >> 4);
            const uint32_t a0 = tmem_base + kASlab0 + 32u * aset;
            const uint32_t full = full0 + rt.slot * 8u, empty = empty0 + rt.slot * 8u;
            if (!mma_stage_ts_x8<kPair>(full, rt.phase, 4u, d_tmem, a0, a0 + kAccCols, b0, b0 + tok_step, t_hi, idesc,
                                        kb != 0, empty)) {
              // Not staged after a few suspended tests: check the clock and the abort
              // flag between further attempts, as every bounded wait does.
              const uint64_t t0 = global_timer_ns();
              bool issued = false;
              while (!issued) {
                if (*abort || global_timer_ns() - t0 > s_wait_limit_ns) break;
                issued = mma_stage_ts_x8<kPair>(full, rt.phase, 4u, d_tmem, a0, a0 + kAccCols, b0, b0 + tok_step,
                                                t_hi, idesc, kb != 0, empty);
              }
              if (!__all_sync(0xffffffffu, issued)) {
                *abort = 1;
                ok = false;
                break;
              }
            }
            if (++aset == kAStages) aset = 0;
            rt.next(ST);
          }
        } else {
        for (int kb = 0; kb < KB; ++kb) {
          const bool staged = __all_sync(0xffffffffu, wait_phase(smem_addr(&ctl.full[rt.slot]), rt.phase, abort));
          if (!staged) { ok = false; break; }
          tc_fence_after_sync();
          {
#pragma unroll
            for (uint32_t sub = 0; sub < G::kSub; ++sub) {
              const uint64_t b_desc = t_desc0 + (((rt.slot * G::kSub + sub) * G::kTSlot) >> 4);
              const uint64_t a_desc = w_desc0 + (((rt.slot * G::kSub + sub) * kWBytes) >> 4);
#pragma unroll
              for (int k = 0; k < kBK / 16; ++k) {   // +32 bytes along K per step: +2 in the >>4 address field
                const uint32_t accumulate = (kb | static_cast<int>(sub) | k) != 0;
                if constexpr (kPair && kFp8)
                  mma_f8_pair(d_tmem, a_desc + 2u * k, b_desc + 2u * k, idesc, accumulate);
                else if constexpr (kPair)
                  mma_bf16_pair(d_tmem, a_desc + 2u * k, b_desc + 2u * k, idesc, accumulate);
                else if constexpr (kFp8)
                  mma_f8(d_tmem, a_desc + 2u * k, b_desc + 2u * k, idesc, accumulate);
                else
                  mma_bf16(d_tmem, a_desc + 2u * k, b_desc + 2u * k, idesc, accumulate);
              }
            }
            if constexpr (kPair) mma_commit_pair(smem_addr(&ctl.empty[rt.slot]), 0x3);
            else mma_commit(smem_addr(&ctl.empty[rt.slot]));
          }
          rt.next(ST);
        }
        }
        if (!ok) break;
        if constexpr (kPair) mma_commit_pair(smem_addr(&ctl.acc_full[acc]), 0x3);
        else mma_commit(smem_addr(&ctl.acc_full[acc]));
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      if (!ok && lane == 0) atomicOr(p.status, kStatusTimeout);
    }
  } else if (warp < 2 + static_cast<int>(n_epi)) {
    // ------------------------------------------------------------ epilogue
    if (warp == 2) {
      // First, the producer's token maps: lane i builds the map whose copies are
      // 16 (i + 1) rows high (a tile's token slab, a multiple of 16 rows, is then one copy
      // per 64-K sub-slab), from the host's map with the row extent patched to
      // a_offsets[G] (three planes of it with A-plane row offsetting).  Done here, not in
      // the producer, so that it overlaps the producer's decode of its first tile.
      constexpr int kMaps = static_cast<int>(G::kCtaTok / 16);
      uint8_t *slot = p.map_slots + static_cast<size_t>(blockIdx.x) * kMapSlotBytes;
      if (total > 0 && lane < kMaps) {
        const uint4 *src = reinterpret_cast<const uint4 *>(&p.tok_map);
        uint4 *dst = reinterpret_cast<uint4 *>(slot + lane * 128);
#pragma unroll
        for (int i = 0; i < 8; ++i) dst[i] = src[i];
        const uint32_t planes = (p.plane_s0 | p.plane_s1) ? 3u : 1u;
        tensormap_set_dim1(dst, planes * __ldg(p.a_offsets + p.num_groups));
        tensormap_set_box1(dst, 16u * static_cast<uint32_t>(lane + 1));
        tensormap_release();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&ctl.maps_ready));
    }
    const uint32_t quad = static_cast<uint32_t>(warp & 3);   // TMEM lanes this warp may read
    // With 12 epilogue warps, warps 2 .. 5 take 32-row chunks 0, 3, 6 of a tile, warps
    // 6 .. 9 chunks 1, 4, 7 and warps 10 .. 13 chunks 2, 5.
    const uint32_t esub = static_cast<uint32_t>(warp - 2) >> 2, nsub = n_epi >> 2;
    // Staging buffers per warp: two with 4 epilogue warps (bf16 / e4m3: 16 of the 24 KB),
    // one with 12, and one in the 4-bit kernel (8 KB for its 4 warps).
    const uint32_t nbuf = kEpiBytes<kInt4> / (n_epi * kEpiRows * kEpiRowBytes) >= 2u ? 2u : 1u;
    uint32_t chunk_ctr = 0, outstanding = 0, last_buf = 0;   // this warp's TMA-store bookkeeping
    const uint32_t acc_empty0 = kPair ? map_to_rank(smem_addr(&ctl.acc_empty[0]), 0) : smem_addr(&ctl.acc_empty[0]);
    const uint32_t acc_empty1 = kPair ? map_to_rank(smem_addr(&ctl.acc_empty[1]), 0) : smem_addr(&ctl.acc_empty[1]);
    uint32_t acc = 0, acc_phase = 0;
    TileSource reader(dynamic, unit0, units, total);
    for (;;) {
      if (total == 0) break;
      Tile ti;
      const int got = next_tile_warp<G>(reader, ctl, q_empty0, q_remote, abort, prefix, p, &ti);
      if (got < 0 && lane == 0) atomicOr(p.status, kStatusTimeout);
      if (got <= 0) break;
      // Two views of a 32-row chunk.  Read from TMEM (16x256b shape, the stmatrix
      // fragment): thread l holds columns quad * 32 + 8i + l / 4 (i = 0 .. 3) of rows
      // 8g + 2(l % 4) + {0, 1} (g = 0 .. 3).  Stored to C: thread l writes 8
      // consecutive columns n8 .. n8 + 7 of row 8 pass + rsub (N is a multiple of 8, so
      // they are all in range or all past N).
      const uint32_t seg = static_cast<uint32_t>(lane) & 3u;
      const uint32_t rsub = static_cast<uint32_t>(lane) >> 2;
      const uint32_t ncta = ti.n0 + rank * kBlockN + quad * 32;   // this warp's first C column
      const uint32_t n8 = ncta + seg * 8;
      const bool cols_ok = n8 < static_cast<uint32_t>(p.N);
      __nv_bfloat16 *crow = p.c + static_cast<size_t>(ti.row0) * p.N + n8;
      const uint32_t taddr = tmem_base + ((quad * 32u) << 16) + acc * kAccCols;
      const bool scaled = kFp8 && p.in_scale != nullptr;
      const bool fused = p.epi_bias != nullptr || p.epi_row_scale != nullptr || p.epi_act != kActNone || scaled;
      // The fused epilogue's operands are loaded before the accumulator wait, so their
      // latency hides behind the tile's MMAs: the bias and (e4m3) weight scale of the
      // thread's 4 fragment columns, and the per-row factors of this warp's chunks, lane
      // l holding row l of each (row scale rs, e4m3 input scale sc).
      constexpr int kRowRegs = static_cast<int>(G::kMaxTok / 32);
      float rs[kRowRegs], sc[kRowRegs], bias4[4], wc4[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        bias4[i] = 0.0f;
        wc4[i] = 1.0f;
      }
      if (fused) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t n = ncta + 8u * i + (static_cast<uint32_t>(lane) >> 2);
          if (ncta + 8u * i < static_cast<uint32_t>(p.N)) {
            if (p.epi_bias != nullptr) bias4[i] = __bfloat162float(p.epi_bias[static_cast<size_t>(ti.e) * p.N + n]);
            if (scaled) wc4[i] = __ldg(p.w_scale + static_cast<size_t>(ti.e) * p.w_scale_cols + n / static_cast<uint32_t>(p.scale_gn));
          }
        }
#pragma unroll
        for (int q = 0; q < kRowRegs; ++q) {
          const uint32_t t = (static_cast<uint32_t>(q) * nsub + esub) * 32u + static_cast<uint32_t>(lane);
          const bool row_ok = t < ti.nrows;
          rs[q] = (p.epi_row_scale != nullptr && row_ok) ? __ldg(p.epi_row_scale + ti.row0 + t) : 1.0f;
          sc[q] = (scaled && row_ok) ? __ldg(p.in_scale + (ti.row0 + t) / static_cast<uint32_t>(p.scale_gm)) : 1.0f;
        }
      }
      int ok = 1;
      if (lane == 0) ok = wait_phase(smem_addr(&ctl.acc_full[acc]), acc_phase, abort);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        if (lane == 0) atomicOr(p.status, kStatusTimeout);
        break;
      }
      tc_fence_after_sync();
      // Per chunk: two TMEM loads (lanes +0 .. 15 and +16 .. 31), one wait; per 8-row
      // group g the four 8 x 8 matrices (fragment column blocks i) go to the staging
      // tile transposed, one stmatrix; then four row reads and 16-byte stores.  A chunk
      // may read TMEM columns past ntok (inside the accumulator); those rows are not
      // stored.  The row factors of rows c0 .. c0 + 31 are in rs[0] / sc[0] and move
      // down one register every chunk.
      const uint32_t stg0 = epi_ring + static_cast<uint32_t>(warp - 2) * nbuf * (kEpiRows * kEpiRowBytes);
      // stmatrix: thread l addresses row 8g + (l % 8) of matrix i = l / 8 (block i).
      const uint32_t st_row = static_cast<uint32_t>(lane) & 7u, st_blk = static_cast<uint32_t>(lane) >> 3;
      for (uint32_t c0 = esub * 32u; c0 < ti.ntok; c0 += 32u * nsub) {
        uint32_t va[16], vb[16];
        tmem_ld_16x256b_x4(taddr + c0, va);
        tmem_ld_16x256b_x4(taddr + (16u << 16) + c0, vb);
        // Staging buffer of this chunk; a TMA store that still reads it must finish first
        // (the newest group may stay in flight while it reads the other buffer).
        const uint32_t b = nbuf == 2u ? (chunk_ctr & 1u) : 0u;
        const uint32_t stg = stg0 + b * (kEpiRows * kEpiRowBytes);
        if (lane == 0 && ((outstanding >> b) & 1u)) {
          if (last_buf == b) bulk_wait_read<0>(); else bulk_wait_read<1>();
        }
        outstanding &= ~(1u << b);
        ++chunk_ctr;
        tmem_ld_wait();
        __syncwarp();   // the previous chunk's row reads are done, and the buffer is free
#pragma unroll
        for (uint32_t g = 0; g < 4; ++g) {
          // Row factors of this thread's two rows of the group.
          float s0 = 1.0f, s1 = 1.0f, q0 = 1.0f, q1 = 1.0f;
          if (fused) {
            const int r0 = static_cast<int>(8 * g + 2 * seg);
            s0 = __shfl_sync(0xffffffffu, rs[0], r0);
            s1 = __shfl_sync(0xffffffffu, rs[0], r0 + 1);
            if (kFp8) {
              q0 = __shfl_sync(0xffffffffu, sc[0], r0);
              q1 = __shfl_sync(0xffffffffu, sc[0], r0 + 1);
            }
          }
          uint32_t w[4];
#pragma unroll
          for (uint32_t i = 0; i < 4; ++i) {
            const uint32_t *v = (i >> 1) ? vb : va;
            float y0 = __uint_as_float(v[4 * g + 2 * (i & 1)]);
            float y1 = __uint_as_float(v[4 * g + 2 * (i & 1) + 1]);
            if (fused) {
              if (kFp8) {
                y0 *= q0 * wc4[i];
                y1 *= q1 * wc4[i];
              }
              y0 = epilogue_op(y0, bias4[i], p.epi_act, s0);
              y1 = epilogue_op(y1, bias4[i], p.epi_act, s1);
            }
            w[i] = pack_bf16x2(y0, y1);
          }
          const uint32_t row = 8 * g + st_row;
          stmatrix_x4_trans(stg + row * kEpiRowBytes + ((st_blk ^ ((row >> 1) & 3u)) << 4), w[0], w[1], w[2], w[3]);
        }
        if (p.c_tma && c0 + 32u <= ti.nrows && ncta < static_cast<uint32_t>(p.N)) {
          // A whole chunk of the group's rows: the staging tile is laid out in TMA's
          // 64-byte swizzle, so one store of the 32 x 32 box takes it to C (columns past
          // N are clipped by the map; a box wholly past N is not issued).  The warp's
          // memory queue then holds no C stores.
          fence_async_smem();   // this thread's stmatrix writes, before the async proxy reads them
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&p.c_map, stg, static_cast<int32_t>(ncta), static_cast<int32_t>(ti.row0 + c0));
            bulk_commit();
          }
          outstanding |= 1u << b;
          last_buf = b;
        } else {
          // The group's last, partial chunk (a TMA store would also write the rows after
          // the group's end): 16-byte stores masked to the group's rows.
          __syncwarp();
          const uint8_t *stg_ptr = dyn_smem + (stg - dyn_base);
#pragma unroll
          for (uint32_t pass = 0; pass < 4; ++pass) {
            const uint32_t rl = pass * 8u + rsub;   // row within the chunk
            const uint32_t row = c0 + rl;           // row within the tile
            const uint4 out =
                *reinterpret_cast<const uint4 *>(stg_ptr + rl * kEpiRowBytes + ((seg ^ ((rl >> 1) & 3u)) << 4));
            if (cols_ok && row < ti.nrows) *reinterpret_cast<uint4 *>(crow + static_cast<size_t>(row) * p.N) = out;
          }
        }
#pragma unroll
        for (int q = 0; q + 1 < kRowRegs; ++q) {
          rs[q] = rs[q + 1];
          sc[q] = sc[q + 1];
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        // Relaxed: the accumulator's loads are complete; the C stores need not be
        // visible to the MMA issuer.
        if constexpr (kPair) mbar_arrive_cluster_relaxed(acc ? acc_empty1 : acc_empty0);
        else mbar_arrive_relaxed(acc ? acc_empty1 : acc_empty0);
      }
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
    // The staging tiles must stay readable, and C written, before this warp moves on.
    if (lane == 0) bulk_wait_all();
  } else if (kInt4 && warp == 6) {
    // ------------------------------------------------------------ packed-slab producer (4-bit)
    if (lane == 0 && total > 0) {
      prefetch_tensormap(&p.w_map);
      const uint64_t pol_first = l2_policy_evict_first();
      const uint64_t pol_normal = l2_policy_evict_normal();
      Ring rq;
      uint32_t pending = 0, pend_phase = 0;
      bool ok = true;
      TileSource reader(dynamic, unit0, units, total);
      for (;;) {
        Tile ti;
        const int got = reader.next<G>(ctl, q_empty0, q_remote, abort, prefix, p, &ti);
        if (got < 0) ok = false;
        if (got <= 0) break;
        const int32_t w_row = static_cast<int32_t>(ti.n0 + rank * kBlockN);
        const uint64_t pol = (p.cache_hints && ti.single_block) ? pol_first : pol_normal;
        const int KC = (KB + kQChunkStages - 1) / kQChunkStages;   // chunks of the tile
        for (int kc = 0; kc < KC; ++kc) {
          if (!wait_phase(smem_addr(&ctl.qempty[rq.slot]), rq.phase ^ 1u, abort)) { ok = false; break; }
          const uint32_t qfull = smem_addr(&ctl.qfull[rq.slot]);
          mbar_arrive_expect_tx(qfull, kQSlotBytes);
          // One box of kQChunkStages stages; words past K are zero-filled by TMA.
          tma_load_3d_hint(q_ring + rq.slot * kQSlotBytes, &p.w_map, qfull, kc * (kQRowBytes / 4), w_row, ti.e, pol);
          pending |= 1u << rq.slot;
          pend_phase = (pend_phase & ~(1u << rq.slot)) | (rq.phase << rq.slot);
          rq.next(static_cast<uint32_t>(QS));
        }
        if (!ok) break;
      }
      if (!ok) {
        for (int s = 0; s < QS; ++s)
          if (pending & (1u << s)) wait_phase_for(smem_addr(&ctl.qfull[s]), (pend_phase >> s) & 1u, kDrainLimitNs);
        atomicOr(p.status, kStatusTimeout);
      }
    }
  } else if (kInt4) {
    // ------------------------------------------------------------ 4-bit dequantisation
    // Warp w (7 .. 18) may write the TMEM lanes of quadrant w % 4, so its thread `lane`
    // owns weight row r = 32 (w % 4) + lane.  The warp belongs to group
    // (w - 7) / kDqWarpsPerStage, which handles every kDqGroups-th stage (counted
    // across tiles); in a handled stage it converts kDqSubsPerWarp 64-K sub-slabs of
    // its row (8 packed words each) into 32 TMEM columns of bf16 pairs each.  The
    // arithmetic needs only the packed slab, so it runs as soon as the slab lands;
    // only the TMEM store waits, for the MMAs of stage s - kAStages, the last readers
    // of the slab set.  With as many groups as slab sets, group g always fills set g,
    // and its warps step straight from one of their stages to the next.  The barrier
    // of stage s - kAStages cannot move past the phase this warp waits for, because
    // its next phase needs the stage after it in this group, i.e. this warp's arrival.
    static_assert(kDqGroups == static_cast<int>(kAStages), "group g always fills TMEM slab set g");
    const uint32_t dw = static_cast<uint32_t>(warp - 7);
    const uint32_t quad = static_cast<uint32_t>(warp & 3);
    const uint32_t grp = dw / kDqWarpsPerStage;   // also the TMEM slab set this warp fills
    const uint32_t sub0 = ((dw % kDqWarpsPerStage) >> 2) * kDqSubsPerWarp;   // first sub-slab of this warp
    const uint32_t r = quad * 32u + static_cast<uint32_t>(lane);
    const int spr = p.K / p.group_size;   // scales per weight row
    const unsigned short *sbits = reinterpret_cast<const unsigned short *>(p.scales);
    const uint32_t lane_field = (quad * 32u) << 16;
    uint32_t s_next = grp;      // next stage (counted across tiles) of this warp's group
    uint32_t tile_base = 0;     // stages of earlier tiles
    // Barrier slot and phase of stage s_next (s_next % ST and its use count's parity), and
    // of this group's previous stage, s_next - kDqGroups, kept incrementally: ST is a
    // runtime multiple of kDqGroups, and a division by it costs tens of instructions.
    uint32_t fslot = grp, fphase = 0, eslot = 0, ephase = 0;
    bool has_prev = false;
    uint32_t chunk_base = 0;    // packed chunks of earlier tiles
    // A stage's `full` barrier lives in the leader CTA of a pair; `empty` in each CTA
    // (the leader's commit arrives on both).
    const uint32_t full0 = kPair ? map_to_rank(smem_addr(&ctl.full[0]), 0) : smem_addr(&ctl.full[0]);
    const uint32_t empty0 = smem_addr(&ctl.empty[0]);
    constexpr uint32_t kBarBytes = static_cast<uint32_t>(sizeof(uint64_t));
    bool ok = true;
    TileSource reader(dynamic, unit0, units, total);
    for (;;) {
      if (total == 0) break;
      Tile ti;
      const int got = next_tile_warp<G>(reader, ctl, q_empty0, q_remote, abort, prefix, p, &ti);
      if (got < 0) ok = false;
      if (got <= 0) break;
      const uint32_t n = ti.n0 + rank * kBlockN + r;
      const bool row_ok = n < static_cast<uint32_t>(p.N);
      const unsigned short *srow = sbits + (static_cast<size_t>(ti.e) * p.N + (row_ok ? n : 0)) * spr;
      // This group's stages of the tile: kb = s_next - tile_base, then every kDqGroups-th.
      for (; s_next < tile_base + static_cast<uint32_t>(KB) && ok; s_next += kDqGroups) {
        const int kb = static_cast<int>(s_next - tile_base);
        // Scales of this thread's sub-slabs; zero past K (the last stage's second
        // half when K is an odd multiple of 64) or past N, so the weights there are
        // zero, matching the zero-filled tokens.  Loaded first: the waits below
        // cover their latency.
        unsigned short sv[kDqSubsPerWarp];
#pragma unroll
        for (int i = 0; i < kDqSubsPerWarp; ++i) {
          const int sub = kb * kSub4 + static_cast<int>(sub0) + i;   // 64-K sub-slab along K
          const int idx = p.scale_shift >= 0 ? (sub >> p.scale_shift) : sub * kBK / p.group_size;
          sv[i] = (row_ok && sub * kBK < p.K) ? __ldg(srow + idx) : static_cast<unsigned short>(0);
        }
        // Packed chunk of this stage (slot and phase from the chunk count) and the
        // stage's half of it; 16-byte piece c of row r sits at piece c ^ (r % 8).
        const uint32_t chunk = chunk_base + static_cast<uint32_t>(kb) / kQChunkStages;
        const uint32_t qslot = chunk & static_cast<uint32_t>(QS - 1), qphase = (chunk >> q_shift) & 1u;
        const uint32_t piece0 = (static_cast<uint32_t>(kb) % kQChunkStages) * (kSub4 * 2);
        if (!__all_sync(0xffffffffu, wait_phase(smem_addr(&ctl.qfull[qslot]), qphase, abort))) {
          ok = false;   // the warp aborts together
          break;
        }
        const uint8_t *qrow = dyn_smem + (q_ring - dyn_base) + qslot * kQSlotBytes + r * kQRowBytes;
        uint32_t cols[kDqSubsPerWarp][32];
#pragma unroll
        for (int i = 0; i < kDqSubsPerWarp; ++i) {
          const uint32_t c = piece0 + (sub0 + i) * 2;
          const uint4 qa = *reinterpret_cast<const uint4 *>(qrow + (((c + 0) ^ (r & 7u)) << 4));
          const uint4 qb = *reinterpret_cast<const uint4 *>(qrow + (((c + 1) ^ (r & 7u)) << 4));
          const __nv_bfloat16 sb = __ushort_as_bfloat16(sv[i]);
          const __nv_bfloat162 s2v = __halves2bfloat162(sb, sb);
          const uint32_t words[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
#pragma unroll
          for (int j8 = 0; j8 < 8; ++j8) {
            const uint4 d = dequant_word(words[j8], s2v);
            cols[i][4 * j8 + 0] = d.x;
            cols[i][4 * j8 + 1] = d.y;
            cols[i][4 * j8 + 2] = d.z;
            cols[i][4 * j8 + 3] = d.w;
          }
        }
        __syncwarp();
        if (lane == 0) {   // the loads above are done; a chunk holding one stage gets both arrivals
          mbar_arrive(smem_addr(&ctl.qempty[qslot]));
          if (kb == KB - 1 && (KB % kQChunkStages) != 0) mbar_arrive(smem_addr(&ctl.qempty[qslot]));
        }
        if (has_prev) {   // the MMAs of stage s - kAStages (this group's previous) read this slab set
          if (!__all_sync(0xffffffffu, wait_phase(empty0 + eslot * kBarBytes, ephase, abort))) {
            ok = false;
            break;
          }
        }
        tc_fence_after_sync();   // the MMAs' reads of this TMEM slab set precede the overwrite
#pragma unroll
        for (int i = 0; i < kDqSubsPerWarp; ++i)
          tmem_st_x32(tmem_base + lane_field + a_slab_col(grp, sub0 + i), cols[i]);
        tmem_st_wait();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) {   // TMEM stores done
          const uint32_t fb = full0 + fslot * kBarBytes;
          if constexpr (kPair) mbar_arrive_cluster_relaxed(fb); else mbar_arrive_relaxed(fb);
        }
        eslot = fslot;
        ephase = fphase;
        has_prev = true;
        fslot += kDqGroups;
        if (fslot >= ST) {
          fslot -= ST;
          fphase ^= 1u;
        }
      }
      if (!ok) break;
      tile_base += static_cast<uint32_t>(KB);
      chunk_base += static_cast<uint32_t>((KB + kQChunkStages - 1) / kQChunkStages);
    }
    if (!ok) atomicOr(p.status, kStatusTimeout);
  }

  __syncthreads();
  if constexpr (kPair) cluster_sync();   // no CTA leaves while its peer may still signal it
  if (tid == 0) {
    // The last CTA to finish returns the tile counter to zero for the next launch
    // (launches through one workspace are stream-ordered, never concurrent).
    __threadfence();
    if (atomicAdd(p.tile_counter + 2, 1u) == gridDim.x - 1) {
      atomicExch(reinterpret_cast<unsigned long long *>(p.tile_counter), 0ull);
      atomicExch(p.tile_counter + 2, 0u);
    }
  }
  if (warp == 1) {
    tc_fence_after_sync();
    if constexpr (kPair) tmem_dealloc_pair(tmem_base, kTmemCols);
    else tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace gmm
