// Host side of the C ABI declared in include/gmm.h: handle management,
// argument validation, tensor-map encoding and the kernel launch.  No call
// here synchronises except gmm_query_status, and gmm_run / gmm_run_int4
// allocate nothing.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include "gmm.h"
#include "gmm_kernel.cuh"
#include "gmm_fp8_block.cuh"

namespace {

using gmm::GmmParams;

// Workspace layout: a 256-byte block with the status word at byte 0, the 64-bit
// tile-claim word (front count | back count << 32) at byte 64 and the finished-CTA
// counter at byte 72 (all zero between launches), the dense call's routing at 128 and
// its usage stats at 144; then one slot of tensor maps per CTA.
constexpr size_t kStatusBytes = 256;
constexpr size_t kTileCounterOffset = 64;
constexpr size_t kDenseRoutingOffset = 128;   // gmm_matmul_int4: a_offsets {0, M} and expert id 0
constexpr size_t kDenseStatsOffset = 144;     // and its usage stats (written, never read)

struct DeviceGuard {
  int prev = -1;
  bool switched = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) == cudaSuccess && prev != dev) switched = cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    if (switched) cudaSetDevice(prev);
  }
};

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// GMM_DEBUG=1: report the CUDA call behind a GMM_ERR_CUDA on stderr, and (when set as
// a handle is created) the handle's ring depths and each of its grouped-kernel launches'
// layout (diagnostics only).
void debug_report(const char *what, int code, const char *msg) {
  static const bool on = getenv("GMM_DEBUG") != nullptr;
  if (on) fprintf(stderr, "gmm: %s failed: %d %s\n", what, code, msg ? msg : "");
}

}  // namespace

// One launch configuration per kernel variant.  The grouped kernel keeps its group
// prefix (G + 1 words) in dynamic shared memory after the rings, so its configuration is
// chosen per launch: the first of its candidate layouts (in order of preference) whose
// minimum ring fits beside the prefix of that G, with as many stages as the rest holds.
struct gmm_variant {
  int stages = 0;           // depth of the W+T stage ring (grouped kernel: its first layout, one group)
  size_t smem = 0;          // dynamic shared memory of every launch
  size_t budget = 0;        // of which the kernel may use (the rest only keeps one CTA per SM)
  size_t stage_bytes = 0;   // grouped kernel: one stage of the ring
  int stage_mult = 1;       // grouped kernel: the ring depth is a multiple of this (4-bit: kAStages)
  int min_stages = 2;       // grouped kernel: the shallowest ring it runs with
  int layouts = 1;          // grouped kernel: candidate layouts, in order of preference
  size_t fixed[2] = {};     // per layout: everything but the stage ring and the prefix
  int q_stages[2] = {};     // per layout, 4-bit: packed-ring slots
  int grid = 0;             // CTAs: the SM count, or (pairs) twice the co-resident clusters of two
};

struct gmm_ctx {
  int device = 0;
  int num_experts = 0;
  int num_sms = 0;
  gmm_variant var[2][2];          // [4-bit][pair]
  gmm_variant var_fp8[2];         // e4m3 kernels, [pair]
  gmm_variant var_fp8_block;      // e4m3 with per-K-block scales (one CTA per tile)
  int smem_per_sm = 0;            // shared memory of one SM (a launch reserves more than half: one CTA per SM)
  bool debug = false;             // GMM_DEBUG was set when the handle was created
  int use_pairs = 1;              // bf16 path: 1 = CTA-pair kernels (cta_group::2), 0 = one CTA per tile
  int use_pairs_int4 = 1;         // 4-bit path: the same
  uint8_t *ws = nullptr;          // [status word | per-CTA tensor-map slots]
  size_t ws_bytes = 0;
  PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  PFN_cuMemsetD32Async_v3020 memset32 = nullptr;   // value writes that a captured CUDA graph replays as such
};

namespace {

int encode_map(gmm_ctx *h, CUtensorMap *m, CUtensorMapDataType type, uint32_t rank, const void *base,
               const cuuint64_t *dims, const cuuint64_t *strides, const cuuint32_t *box,
               CUtensorMapSwizzle swizzle) {
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = h->encode(m, type, rank, const_cast<void *>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) debug_report("cuTensorMapEncodeTiled", static_cast<int>(r), nullptr);
  return r == CUDA_SUCCESS ? GMM_OK : GMM_ERR_CUDA;
}

// Token (A) map, 128-byte swizzle.  The row extent and the box height written here
// are placeholders: each CTA derives one map per box height from it and patches the
// extent to a_offsets[G].
//   2-D {K, rows}, box {64, rows}: one 64-K sub-slab per copy (any K).
//   3-D {64, rows, K / 64} (strides: a row, then 128 bytes to the next 64 of K), box
//   {64, rows, sub}: `sub` sub-slabs of a stage in one copy, landing one after the
//   other in shared memory.  Only when K is a multiple of 64 (the 4-bit path).
int encode_token_maps(gmm_ctx *h, GmmParams &p, const void *a, int K, int sub_per_copy) {
  if (sub_per_copy == 1) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), 256};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
    cuuint32_t box[2] = {gmm::kBK, 128};
    return encode_map(h, &p.tok_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a, dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_128B);
  }
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(gmm::kBK), 256, static_cast<cuuint64_t>(K / gmm::kBK)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * 2, static_cast<cuuint64_t>(gmm::kBK) * 2};
  cuuint32_t box[3] = {gmm::kBK, 128, static_cast<cuuint32_t>(sub_per_copy)};
  return encode_map(h, &p.tok_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_128B);
}

// The optional epilogue: a known activation, and operands aligned for their element type.
int check_epilogue(const gmm_epilogue *e) {
  if (!e) return GMM_OK;
  if (e->activation < GMM_ACT_NONE || e->activation > GMM_ACT_GELU_TANH) return GMM_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(e->bias) & 1u) || (reinterpret_cast<uintptr_t>(e->row_scale) & 3u))
    return GMM_ERR_INVALID_ARG;
  return GMM_OK;
}

void set_epilogue(GmmParams &p, const gmm_epilogue *e) {
  static_assert(GMM_ACT_NONE == gmm::kActNone && GMM_ACT_RELU == gmm::kActRelu && GMM_ACT_SILU == gmm::kActSilu &&
                    GMM_ACT_GELU_TANH == gmm::kActGeluTanh,
                "activation codes of the C ABI and the kernel agree");
  p.epi_bias = e ? static_cast<const __nv_bfloat16 *>(e->bias) : nullptr;
  p.epi_row_scale = e ? e->row_scale : nullptr;
  p.epi_act = e ? e->activation : GMM_ACT_NONE;
}

int check_common(gmm_ctx *h, void *c, const void *a, const uint32_t *a_offsets, const int32_t *ids,
                 uint32_t *stats, int G, int N, int K) {
  if (!h || !c || !a || !a_offsets || !stats) return GMM_ERR_INVALID_ARG;
  if (!ids && G > 0) return GMM_ERR_INVALID_ARG;   // never read when there are no groups
  if (G < 0 || N < 8 || K < 8 || (N % 8) || (K % 8)) return GMM_ERR_INVALID_ARG;
  if (N > (1 << 24) || K > (1 << 24)) return GMM_ERR_UNSUPPORTED;
  if (G > gmm::kMaxGroups) return GMM_ERR_UNSUPPORTED;
  if (!aligned16(c) || !aligned16(a)) return GMM_ERR_INVALID_ARG;
  return GMM_OK;
}

// Token blocks per band of the tile order: as many 256-row blocks of A as fit in
// about 40 MB, a third of the GB300's L2, so a band's activations stay resident.
constexpr double kBandBytes = 40e6;

void fill_common(gmm_ctx *h, GmmParams &p, void *c, const uint32_t *a_offsets, const int32_t *ids,
                 uint32_t *stats, int G, int N, int K, uint32_t max_tok) {
  p.c = static_cast<__nv_bfloat16 *>(c);
  p.a_offsets = a_offsets;
  p.expert_ids = ids;
  p.stats = stats;
  p.status = reinterpret_cast<uint32_t *>(h->ws);
  p.tile_counter = reinterpret_cast<uint32_t *>(h->ws + kTileCounterOffset);
  p.map_slots = h->ws + kStatusBytes;
  p.num_groups = G;
  p.num_experts = h->num_experts;
  p.N = N;
  p.K = K;
  // C as a TMA store target: {N, 2^31} rows (the real row count is on the device; the
  // kernel only stores whole 32-row chunks inside a group through it), box 32 x 32,
  // 64-byte swizzle (the epilogue staging layout).  Without it every chunk takes the
  // 16-byte store path.
  p.c_tma = 0;
  if (h->encode != nullptr && aligned16(c)) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), 1ull << 31};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(N) * 2u};
    const cuuint32_t box[2] = {32, 32}, estr[2] = {1, 1};
    p.c_tma = h->encode(&p.c_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, c, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  }
  if (const char *env = getenv("GMM_TMA_STORE")) p.c_tma = p.c_tma && atoi(env) != 0;   // tuning override
  const double block_bytes = static_cast<double>(max_tok) * K * 2.0;
  const double band = kBandBytes / block_bytes;
  p.tok_band = band < 1.0 ? 1 : (band > 1e6 ? 1000000 : static_cast<int>(band));
  if (const char *env = getenv("GMM_TOK_BAND")) {   // tuning override
    const int v = atoi(env);
    if (v > 0) p.tok_band = v;
  }
  p.cache_hints = 1;
  if (const char *env = getenv("GMM_CACHE_HINTS")) p.cache_hints = atoi(env) != 0;   // tuning override
  // Test hooks of the device-timeout path (off unless set): GMM_TEST_WAIT_LIMIT_NS
  // shortens every pipeline wait, GMM_TEST_STALL_STAGE makes the one-CTA bf16 kernel's
  // producer skip that stage, so that the kernel gives up and reports a timeout.
  p.wait_limit_ns = 0;
  p.test_stall_stage = -1;
  if (const char *env = getenv("GMM_TEST_WAIT_LIMIT_NS")) p.wait_limit_ns = strtoull(env, nullptr, 10);
  if (const char *env = getenv("GMM_TEST_STALL_STAGE")) p.test_stall_stage = atoi(env);
}

// Stage-ring depth of a grouped-kernel launch with G groups in a layout: what the budget
// holds after the layout's fixed parts and the prefix, capped at kMaxStages, a multiple
// of stage_mult.
int stages_for(const gmm_variant &v, int G, int layout) {
  const size_t prefix = (static_cast<size_t>(G + 1) * 4 + 15) & ~static_cast<size_t>(15);
  const size_t fixed = v.fixed[layout];
  if (v.budget < fixed + prefix) return 0;
  long st = static_cast<long>((v.budget - fixed - prefix) / v.stage_bytes);
  if (st > gmm::kMaxStages) st = gmm::kMaxStages;
  st -= st % v.stage_mult;
  return static_cast<int>(st);
}

// Ring depths from the shared-memory budget (the pages' launchers likewise derive their
// pipeline depth from the shared memory available, and the quantised GEMM's launcher
// reduces stages or warp partitions when the budget is exceeded): as many stages as fit,
// and for the 4-bit kernel, if even its minimum ring does not fit with the full packed
// ring, a packed ring of half the slots.  The grid: one CTA per SM, or for pairs twice
// the number of clusters of two that fit at once.  `optin` is the budget (the device's
// opt-in shared memory per block, or less when capped for testing), `sm_smem` the SM's
// shared memory: a launch always reserves more than half of it, so one CTA runs per SM.
template <bool kInt4, bool kPair, bool kFp8 = false>
int configure(gmm_variant *v, int optin, int sm_smem, int device_optin, int num_sms) {
  using G = gmm::Geom<kInt4, kPair>;
  auto kernel = gmm::gmm_grouped_kernel<kInt4, kPair, kFp8>;
  cudaFuncAttributes attr;
  if (cudaFuncGetAttributes(&attr, reinterpret_cast<const void *>(kernel)) != cudaSuccess) return GMM_ERR_CUDA;
  const long avail = static_cast<long>(optin) - static_cast<long>(attr.sharedSizeBytes);
  if (avail <= 0) return GMM_ERR_UNSUPPORTED;
  v->budget = static_cast<size_t>(avail);
  v->stage_bytes = G::kStageBytes;
  v->stage_mult = kInt4 ? static_cast<int>(gmm::kAStages) : 1;
  // Candidate layouts.  4-bit, in order of preference: the full packed ring, then half
  // of it.  The variant is usable when at least one layout fits beside a one-group
  // prefix; a launch whose groups' prefix leaves no layout its minimum ring returns
  // GMM_ERR_UNSUPPORTED.
  v->min_stages = kInt4 ? static_cast<int>(gmm::kAStages) : 2;
  v->layouts = kInt4 ? 2 : 1;
  for (int c = 0; c < v->layouts; ++c) {
    v->q_stages[c] = kInt4 ? (c == 0 ? gmm::kQStages : 2) : 0;
    v->fixed[c] = 1024 + gmm::kEpiBytes<kInt4> + static_cast<size_t>(v->q_stages[c]) * gmm::kQSlotBytes;
  }
  v->stages = 0;
  for (int c = 0; c < v->layouts && v->stages < v->min_stages; ++c) v->stages = stages_for(*v, 1, c);
  if (v->stages < v->min_stages) return GMM_ERR_UNSUPPORTED;
  const long reserve = static_cast<long>(sm_smem) / 2 + 1024;   // more than half an SM: one CTA per SM
  const long cap = static_cast<long>(device_optin) - static_cast<long>(attr.sharedSizeBytes);
  v->smem = static_cast<size_t>(std::min(cap, std::max(avail, reserve)));
  if (cudaFuncSetAttribute(reinterpret_cast<const void *>(kernel), cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(v->smem)) != cudaSuccess)
    return GMM_ERR_CUDA;
  v->grid = num_sms;
  if (kPair) {
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cudaLaunchAttribute la[1];
    la[0].id = cudaLaunchAttributeClusterDimension;
    la[0].val.clusterDim.x = 2;
    la[0].val.clusterDim.y = 1;
    la[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(num_sms & ~1));
    cfg.blockDim = dim3(kInt4 ? gmm::kInt4Threads : gmm::kThreadsWide);   // the larger launch
    cfg.dynamicSmemBytes = v->smem;
    cfg.attrs = la;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg) != cudaSuccess || clusters < 1)
      return GMM_ERR_CUDA;
    v->grid = 2 * clusters < (num_sms & ~1) ? 2 * clusters : (num_sms & ~1);
  }
  return GMM_OK;
}

// The per-K-block e4m3 kernel: as many stages as fit beside the group prefix (sized at
// each launch, as for the grouped kernel), one CTA per SM.
int configure_fp8_block(gmm_variant *v, int optin, int sm_smem, int device_optin, int num_sms) {
  using G = gmm::BwGeom;
  auto kernel = gmm::gmm_fp8_block_kernel;
  cudaFuncAttributes attr;
  if (cudaFuncGetAttributes(&attr, reinterpret_cast<const void *>(kernel)) != cudaSuccess) return GMM_ERR_CUDA;
  // The kernel moves registers from its first warpgroup to the promotion warpgroups
  // (setmaxnreg).  The increase waits until the CTA's pool, the launch's registers a
  // thread times its threads, covers it, so a build whose register count left the pool
  // short would never finish: refuse it here instead.
  if (static_cast<long>(attr.numRegs) * gmm::kBwThreads <
      128L * gmm::kBwRegsLow + 32L * gmm::kBwPromoWarps * gmm::kBwRegsHigh)
    return GMM_ERR_UNSUPPORTED;
  const long avail = static_cast<long>(optin) - static_cast<long>(attr.sharedSizeBytes);
  if (avail <= 0) return GMM_ERR_UNSUPPORTED;
  v->budget = static_cast<size_t>(avail);
  v->stage_bytes = G::kStageBytes;
  v->stage_mult = 1;
  v->min_stages = 2;
  v->layouts = 1;
  v->q_stages[0] = 0;
  v->fixed[0] = static_cast<size_t>(gmm::kBwFixedBytes);
  v->stages = stages_for(*v, 1, 0);
  if (v->stages < v->min_stages) return GMM_ERR_UNSUPPORTED;
  const long reserve = static_cast<long>(sm_smem) / 2 + 1024;   // more than half an SM: one CTA per SM
  const long cap = static_cast<long>(device_optin) - static_cast<long>(attr.sharedSizeBytes);
  v->smem = static_cast<size_t>(std::min(cap, std::max(avail, reserve)));
  if (cudaFuncSetAttribute(reinterpret_cast<const void *>(kernel), cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(v->smem)) != cudaSuccess)
    return GMM_ERR_CUDA;
  v->grid = num_sms;
  return GMM_OK;
}

int launch_fp8_block(gmm_ctx *h, GmmParams &p, cudaStream_t stream) {
  DeviceGuard guard(h->device);
  const gmm_variant &v = h->var_fp8_block;
  p.num_stages = stages_for(v, p.num_groups, 0);
  if (p.num_stages < v.min_stages) return GMM_ERR_UNSUPPORTED;   // the prefix leaves no room for the ring
  if (h->debug)
    fprintf(stderr, "gmm: launch e4m3 block, %d groups: stages %d packed slots 0\n", p.num_groups, p.num_stages);
  gmm::gmm_fp8_block_kernel<<<v.grid, gmm::kBwThreads, v.smem, stream>>>(p);
  const cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) {
    debug_report("launch of the block-scaled kernel", static_cast<int>(err), cudaGetErrorString(err));
    return GMM_ERR_CUDA;
  }
  return GMM_OK;
}

template <bool kInt4, bool kFp8 = false>
int launch(gmm_ctx *h, GmmParams &p, cudaStream_t stream) {
  DeviceGuard guard(h->device);
  const int pairs = kInt4 ? h->use_pairs_int4 : h->use_pairs;
  const gmm_variant &v = kFp8 ? h->var_fp8[pairs] : h->var[kInt4][pairs];
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cudaLaunchAttribute attr[1];
  // Short K: 12 epilogue warps (the bf16 / e4m3 kernel reads its warp count from blockDim).
  cfg.blockDim = dim3(kInt4 ? gmm::kInt4Threads : (p.K <= gmm::kWideEpilogueMaxK ? gmm::kThreadsWide : gmm::kThreads));
  cfg.gridDim = dim3(static_cast<unsigned>(v.grid));
  cfg.dynamicSmemBytes = v.smem;
  cfg.stream = stream;
  int layout = 0;
  p.num_stages = 0;
  for (; layout < v.layouts; ++layout)
    if ((p.num_stages = stages_for(v, p.num_groups, layout)) >= v.min_stages) break;
  if (layout == v.layouts) return GMM_ERR_UNSUPPORTED;   // no layout's minimum ring fits beside this prefix
  p.q_stages = v.q_stages[layout];
  if (h->debug)
    fprintf(stderr, "gmm: launch %s%s, %d groups: stages %d packed slots %d\n", kInt4 ? "int4" : (kFp8 ? "e4m3" : "bf16"),
            pairs ? " pair" : "", p.num_groups, p.num_stages, p.q_stages);
  cudaError_t err;
  if (pairs) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    err = cudaLaunchKernelEx(&cfg, gmm::gmm_grouped_kernel<kInt4, true, kFp8>, p);
  } else {
    err = cudaLaunchKernelEx(&cfg, gmm::gmm_grouped_kernel<kInt4, false, kFp8>, p);
  }
  if (err != cudaSuccess) {
    debug_report("launch of the grouped kernel", static_cast<int>(err), cudaGetErrorString(err));
    cudaGetLastError();
    return GMM_ERR_CUDA;
  }
  return GMM_OK;
}

uint32_t max_tok(const gmm_ctx *h, bool int4) {
  if (int4) return h->use_pairs_int4 ? gmm::Geom<true, true>::kMaxTok : gmm::Geom<true, false>::kMaxTok;
  return h->use_pairs ? gmm::Geom<false, true>::kMaxTok : gmm::Geom<false, false>::kMaxTok;
}

}  // namespace

extern "C" {

const char *gmm_error_string(int code) {
  switch (code) {
    case GMM_OK: return "success";
    case GMM_ERR_INVALID_ARG: return "invalid argument";
    case GMM_ERR_UNSUPPORTED: return "unsupported shape or option";
    case GMM_ERR_CUDA: return "CUDA runtime or driver call failed";
    case GMM_ERR_DEVICE_TIMEOUT: return "kernel pipeline wait timed out";
    case GMM_ERR_BAD_INPUT: return "decreasing a_offsets or expert id out of range";
    case GMM_ERR_NO_DEVICE: return "no sm_103 device";
    default: return "unknown error code";
  }
}

int gmm_create(gmm_handle_t *out, int num_experts, int device) {
  if (!out) return GMM_ERR_INVALID_ARG;
  *out = nullptr;
  if (num_experts < 1) return GMM_ERR_INVALID_ARG;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) {
    cudaGetLastError();
    return GMM_ERR_NO_DEVICE;
  }
  int major = 0, minor = 0, sms = 0, optin = 0, sm_smem = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
  cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
  cudaDeviceGetAttribute(&sm_smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, device);
  if (major != 10 || minor != 3 || sms < 1) return GMM_ERR_NO_DEVICE;
  const int device_optin = optin;
  // Test override GMM_SMEM_BUDGET (bytes): size the rings as if a block could opt in to
  // no more shared memory than this, which exercises the reduced configurations.
  if (const char *env = getenv("GMM_SMEM_BUDGET")) {
    const int cap = atoi(env);
    if (cap > 0 && cap < optin) optin = cap;
  }

  gmm_ctx *h = new (std::nothrow) gmm_ctx;
  if (!h) return GMM_ERR_CUDA;
  h->device = device;
  h->num_experts = num_experts;
  h->num_sms = sms;

  DeviceGuard guard(device);
  void *fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
          cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn) {
    cudaGetLastError();
    delete h;
    return GMM_ERR_CUDA;
  }
  h->encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  fn = nullptr;
  if (cudaGetDriverEntryPointByVersion("cuMemsetD32Async", &fn, 3020, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn) {
    cudaGetLastError();
    delete h;
    return GMM_ERR_CUDA;
  }
  h->memset32 = reinterpret_cast<PFN_cuMemsetD32Async_v3020>(fn);

  h->smem_per_sm = sm_smem;
  const int single_ok = configure<false, false>(&h->var[0][0], optin, sm_smem, device_optin, sms) == GMM_OK &&
                        configure<true, false>(&h->var[1][0], optin, sm_smem, device_optin, sms) == GMM_OK &&
                        configure<false, false, true>(&h->var_fp8[0], optin, sm_smem, device_optin, sms) == GMM_OK &&
                        configure_fp8_block(&h->var_fp8_block, optin, sm_smem, device_optin, sms) == GMM_OK;
  // Tuning override GMM_VARIANT: "single" forces the one-CTA kernels, "pair" the pairs.
  const char *variant = getenv("GMM_VARIANT");
  const bool pairs_ok = sms >= 2 && configure<false, true>(&h->var[0][1], optin, sm_smem, device_optin, sms) == GMM_OK &&
                        configure<true, true>(&h->var[1][1], optin, sm_smem, device_optin, sms) == GMM_OK &&
                        configure<false, true, true>(&h->var_fp8[1], optin, sm_smem, device_optin, sms) == GMM_OK;
  h->use_pairs = pairs_ok && !(variant && std::strcmp(variant, "single") == 0);
  // The 4-bit path too: each CTA of a pair loads half of a stage's tokens (a 6-deep token
  // ring fits), and one MMA instruction covers both CTAs' 128 weight rows, half the
  // instructions per unit of work for the issuing warp, which shares its SM
  // sub-partition with dequantisation warps.
  h->use_pairs_int4 = h->use_pairs;
  if (!single_ok) {
    cudaGetLastError();
    delete h;
    return GMM_ERR_CUDA;
  }

  h->debug = getenv("GMM_DEBUG") != nullptr;
  if (h->debug) {
    const gmm_variant *vs[7] = {&h->var[0][0], &h->var[0][1], &h->var[1][0], &h->var[1][1],
                                &h->var_fp8[0], &h->var_fp8[1], &h->var_fp8_block};
    const char *names[7] = {"bf16", "bf16 pair", "int4", "int4 pair", "e4m3", "e4m3 pair", "e4m3 block"};
    for (int i = 0; i < 7; ++i)
      fprintf(stderr, "gmm: %-16s stages %d smem %zu grid %d\n", names[i], vs[i]->stages, vs[i]->smem, vs[i]->grid);
  }
  h->ws_bytes = kStatusBytes + static_cast<size_t>(sms) * gmm::kMapSlotBytes;
  if (cudaMalloc(&h->ws, h->ws_bytes) != cudaSuccess ||
      cudaMemset(h->ws, 0, h->ws_bytes) != cudaSuccess) {
    cudaGetLastError();
    if (h->ws) cudaFree(h->ws);
    delete h;
    return GMM_ERR_CUDA;
  }
  *out = h;
  return GMM_OK;
}

int gmm_destroy(gmm_handle_t h) {
  if (!h) return GMM_OK;
  DeviceGuard guard(h->device);
  int rc = GMM_OK;
  if (h->ws && cudaFree(h->ws) != cudaSuccess) rc = GMM_ERR_CUDA;
  delete h;
  return rc;
}

int gmm_run_ex(gmm_handle_t h, void *c, const void *a, const uint32_t *a_offsets, const void *b,
               const int32_t *expert_ids, uint32_t *expert_usage_stats, int num_groups, int N, int K,
               const gmm_epilogue *epilogue, cudaStream_t stream) {
  int rc = check_common(h, c, a, a_offsets, expert_ids, expert_usage_stats, num_groups, N, K);
  if (rc) return rc;
  rc = check_epilogue(epilogue);
  if (rc) return rc;
  if (!b || !aligned16(b)) return GMM_ERR_INVALID_ARG;

  GmmParams p;
  std::memset(&p, 0, sizeof(p));
  {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(N),
                          static_cast<cuuint64_t>(h->num_experts)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * 2, static_cast<cuuint64_t>(N) * K * 2};
    cuuint32_t box[3] = {gmm::kBK, gmm::kBlockN, 1};
    rc = encode_map(h, &p.w_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, b, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
  }
  rc = encode_token_maps(h, p, a, K, 1);
  if (rc) return rc;
  fill_common(h, p, c, a_offsets, expert_ids, expert_usage_stats, num_groups, N, K, max_tok(h, false));
  set_epilogue(p, epilogue);
  return launch<false>(h, p, stream);
}

int gmm_run(gmm_handle_t h, void *c, const void *a, const uint32_t *a_offsets, const void *b,
            const int32_t *expert_ids, uint32_t *expert_usage_stats, int num_groups, int N, int K,
            cudaStream_t stream) {
  return gmm_run_ex(h, c, a, a_offsets, b, expert_ids, expert_usage_stats, num_groups, N, K, nullptr, stream);
}

// A-plane row offsetting: the bf16 grouped kernel with the tile's token rows read from
// the plane its weight rows belong to (the producer adds plane * a_offsets[G]).
int gmm_run_planes(gmm_handle_t h, void *c, const void *a, const uint32_t *a_offsets, const void *b,
                   const int32_t *expert_ids, uint32_t *expert_usage_stats, int num_groups, int N, int K,
                   const int *a_plane_splits, const gmm_epilogue *epilogue, cudaStream_t stream) {
  if (!a_plane_splits) return GMM_ERR_INVALID_ARG;
  const int s0 = a_plane_splits[0], s1 = a_plane_splits[1];
  if (s0 < 0 || s1 < 0 || s0 > N || s1 > N - s0) return GMM_ERR_INVALID_ARG;
  if (s0 % 256 || s1 % 256) return GMM_ERR_UNSUPPORTED;   // a tile's 256 weight rows in one plane
  int rc = check_common(h, c, a, a_offsets, expert_ids, expert_usage_stats, num_groups, N, K);
  if (rc) return rc;
  rc = check_epilogue(epilogue);
  if (rc) return rc;
  if (!b || !aligned16(b)) return GMM_ERR_INVALID_ARG;
  GmmParams p;
  std::memset(&p, 0, sizeof(p));
  {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(N),
                          static_cast<cuuint64_t>(h->num_experts)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * 2, static_cast<cuuint64_t>(N) * K * 2};
    cuuint32_t box[3] = {gmm::kBK, gmm::kBlockN, 1};
    rc = encode_map(h, &p.w_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, b, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
  }
  rc = encode_token_maps(h, p, a, K, 1);
  if (rc) return rc;
  fill_common(h, p, c, a_offsets, expert_ids, expert_usage_stats, num_groups, N, K, max_tok(h, false));
  set_epilogue(p, epilogue);
  p.plane_s0 = s0;
  p.plane_s1 = s1;
  return launch<false>(h, p, stream);
}

// The e4m3 operands go through the bf16 kernel's tensor maps unchanged, over their
// bytes: a row of K e4m3 values is a row of K / 2 two-byte units, so the maps, the
// stage ring and the swizzled layout are the bf16 ones and only the MMA kind and the
// epilogue's scales differ (see the kernel's kFp8 variant).
int gmm_run_fp8(gmm_handle_t h, void *c, const void *a, const uint32_t *a_offsets, const void *b,
                const int32_t *expert_ids, uint32_t *expert_usage_stats, int num_groups, int N, int K,
                const float *input_scale, const float *weight_scale, const int *scales_granularity_mnk,
                const gmm_epilogue *epilogue, cudaStream_t stream) {
  if (K < 16 || K % 16) return GMM_ERR_INVALID_ARG;
  const int KU = K / 2;   // two-byte units per row
  int rc = check_common(h, c, a, a_offsets, expert_ids, expert_usage_stats, num_groups, N, KU);
  if (rc) return rc;
  rc = check_epilogue(epilogue);
  if (rc) return rc;
  if (!b || !aligned16(b)) return GMM_ERR_INVALID_ARG;
  if (!scales_granularity_mnk || !input_scale || !weight_scale) return GMM_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(input_scale) & 3u) || (reinterpret_cast<uintptr_t>(weight_scale) & 3u))
    return GMM_ERR_INVALID_ARG;
  const int gm = scales_granularity_mnk[0], gn = scales_granularity_mnk[1], gk = scales_granularity_mnk[2];
  if (gm < 1 || gn < 1 || gk < 1) return GMM_ERR_INVALID_ARG;
  // Per-K-block scales run the block-scaled kernel: whole 128-K stages per block, and
  // one weight scale per 32-column TMEM load.
  const bool blockwise = gk < K;
  if (blockwise && (gk % 128 || gn % 32)) return GMM_ERR_UNSUPPORTED;

  GmmParams p;
  std::memset(&p, 0, sizeof(p));
  {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(KU), static_cast<cuuint64_t>(N),
                          static_cast<cuuint64_t>(h->num_experts)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(N) * K};
    const cuuint32_t rows = !blockwise ? static_cast<cuuint32_t>(gmm::kBlockN) : gmm::BwGeom::kRows;
    cuuint32_t box[3] = {gmm::kBK, rows, 1};
    rc = encode_map(h, &p.w_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, b, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
  }
  rc = encode_token_maps(h, p, a, KU, 1);
  if (rc) return rc;
  fill_common(h, p, c, a_offsets, expert_ids, expert_usage_stats, num_groups, N, KU,
              !blockwise ? max_tok(h, false) : gmm::BwGeom::kMaxTok);
  set_epilogue(p, epilogue);
  p.in_scale = input_scale;
  p.w_scale = weight_scale;
  p.scale_gm = gm;
  p.scale_gn = gn;
  p.w_scale_cols = (N + gn - 1) / gn;
  p.scale_kb = (K + gk - 1) / gk;
  p.kb_stages = gk / 128;
  return blockwise ? launch_fp8_block(h, p, stream) : launch<false, true>(h, p, stream);
}

}  // extern "C"

namespace {

// The 4-bit path for `num_experts` experts of packed weights (the handle's E for the
// grouped calls, 1 for the dense one).
int run_int4(gmm_handle_t h, int num_experts, void *c, const void *a, const uint32_t *a_offsets,
             const uint32_t *b_packed, const void *b_scales, const int32_t *expert_ids,
             uint32_t *expert_usage_stats, int num_groups, int N, int K, int group_size,
             const gmm_epilogue *epilogue, cudaStream_t stream) {
  int rc = check_common(h, c, a, a_offsets, expert_ids, expert_usage_stats, num_groups, N, K);
  if (rc) return rc;
  rc = check_epilogue(epilogue);
  if (rc) return rc;
  if (!b_packed || !b_scales) return GMM_ERR_INVALID_ARG;
  if (!aligned16(b_packed) || (reinterpret_cast<uintptr_t>(b_scales) & 1u)) return GMM_ERR_INVALID_ARG;
  if (group_size < gmm::kBK || group_size % gmm::kBK || K % group_size) return GMM_ERR_UNSUPPORTED;

  GmmParams p;
  std::memset(&p, 0, sizeof(p));
  {
    // Packed weights as 32-bit words {K/8, N, E}; one box = 128 rows x 32 words (128 B,
    // two 128-K stages), 128-byte swizzle.
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(K / 8), static_cast<cuuint64_t>(N),
                          static_cast<cuuint64_t>(num_experts)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(K / 8) * 4, static_cast<cuuint64_t>(N) * (K / 8) * 4};
    cuuint32_t box[3] = {gmm::kQRowBytes / 4, gmm::kBlockN, 1};
    rc = encode_map(h, &p.w_map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, b_packed, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
  }
  rc = encode_token_maps(h, p, a, K, gmm::kSub4);
  if (rc) return rc;
  fill_common(h, p, c, a_offsets, expert_ids, expert_usage_stats, num_groups, N, K, max_tok(h, true));
  p.scales = static_cast<const __nv_bfloat16 *>(b_scales);
  // Scale index of 64-K sub-slab j is j / (group_size / 64): a shift when that is a power of two.
  p.scale_shift = -1;
  for (int s = 0, g64 = group_size / gmm::kBK; (1 << s) <= g64; ++s)
    if ((1 << s) == g64) p.scale_shift = s;
  p.group_size = group_size;
  p.num_experts = num_experts;
  set_epilogue(p, epilogue);
  return launch<true>(h, p, stream);
}

}  // namespace

extern "C" {

int gmm_run_int4_ex(gmm_handle_t h, void *c, const void *a, const uint32_t *a_offsets,
                    const uint32_t *b_packed, const void *b_scales, const int32_t *expert_ids,
                    uint32_t *expert_usage_stats, int num_groups, int N, int K, int group_size,
                    const gmm_epilogue *epilogue, cudaStream_t stream) {
  if (!h) return GMM_ERR_INVALID_ARG;
  return run_int4(h, h->num_experts, c, a, a_offsets, b_packed, b_scales, expert_ids, expert_usage_stats,
                  num_groups, N, K, group_size, epilogue, stream);
}

int gmm_matmul_int4(gmm_handle_t h, void *c, const void *a, const uint32_t *b_packed, const void *b_scales,
                    int M, int N, int K, int group_size, const gmm_epilogue *epilogue, cudaStream_t stream) {
  if (!h || M < 0) return GMM_ERR_INVALID_ARG;
  if (M == 0) return GMM_OK;
  // One group of M rows with expert 0: its offsets, id and (unread) usage stats live
  // in the handle's status block, written in stream order before the kernel by value
  // writes (memset nodes in a captured CUDA graph, so a replay needs no host memory).
  DeviceGuard guard(h->device);
  const CUdeviceptr routing = reinterpret_cast<CUdeviceptr>(h->ws + kDenseRoutingOffset);   // a_offsets[0..1], expert_ids[0]
  if (h->memset32(routing, 0u, 3, reinterpret_cast<CUstream>(stream)) != CUDA_SUCCESS ||
      h->memset32(routing + 4, static_cast<unsigned int>(M), 1, reinterpret_cast<CUstream>(stream)) != CUDA_SUCCESS) {
    cudaGetLastError();
    return GMM_ERR_CUDA;
  }
  const uint32_t *off = reinterpret_cast<const uint32_t *>(h->ws + kDenseRoutingOffset);
  const int32_t *ids = reinterpret_cast<const int32_t *>(h->ws + kDenseRoutingOffset + 8);
  uint32_t *stats = reinterpret_cast<uint32_t *>(h->ws + kDenseStatsOffset);
  return run_int4(h, 1, c, a, off, b_packed, b_scales, ids, stats, 1, N, K, group_size, epilogue, stream);
}

int gmm_run_int4(gmm_handle_t h, void *c, const void *a, const uint32_t *a_offsets,
                 const uint32_t *b_packed, const void *b_scales, const int32_t *expert_ids,
                 uint32_t *expert_usage_stats, int num_groups, int N, int K, int group_size,
                 cudaStream_t stream) {
  return gmm_run_int4_ex(h, c, a, a_offsets, b_packed, b_scales, expert_ids, expert_usage_stats, num_groups, N,
                         K, group_size, nullptr, stream);
}

int gmm_query_status(gmm_handle_t h, cudaStream_t stream) {
  if (!h) return GMM_ERR_INVALID_ARG;
  DeviceGuard guard(h->device);
  uint32_t status = 0;
  if (cudaMemcpyAsync(&status, h->ws, sizeof(status), cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      cudaMemsetAsync(h->ws, 0, sizeof(status), stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess) {
    cudaGetLastError();
    return GMM_ERR_CUDA;
  }
  if (status & gmm::kStatusTimeout) return GMM_ERR_DEVICE_TIMEOUT;
  if (status) return GMM_ERR_BAD_INPUT;
  return GMM_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free entry point (gmm_run_noalloc).
//
// Some callers cannot call cudaMalloc at the moment they need a grouped GEMM:
// code running inside a custom allocator or memory-pool callback, a framework
// that has reserved the whole device for its own pool, or an inference runtime
// that forbids allocations after start-up.  gmm_run_noalloc serves them: it
// launches the same bf16 kernel as gmm_run, but takes the kernel's scratch (its
// status word and the per-CTA patched tensor maps) from the fixed array below
// instead of a handle's cudaMalloc'd workspace, and it creates no handle.
//
// g_noalloc_scratch lives in every GPU that loads this library, until the
// process exits.  In host code its name is only a host-side stand-in, so the
// host never passes it to a kernel: it passes the device address obtained from
// cudaGetSymbolAddress once per device.
// ---------------------------------------------------------------------------
namespace {

constexpr int kNoAllocMaxCtas = 256;   // persistent grid = SM count; 152 on GB300
constexpr size_t kNoAllocScratchBytes = kStatusBytes + static_cast<size_t>(kNoAllocMaxCtas) * gmm::kMapSlotBytes;
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];   // 524,544 bytes

struct NoAllocDevice {
  bool ready = false;   // set-up succeeded; a failed set-up is retried by the next call
  gmm_ctx ctx;          // static storage; ctx.ws points into g_noalloc_scratch on this device
};

NoAllocDevice g_noalloc_devices[kNoAllocMaxDevices];
std::mutex g_noalloc_mutex;

// One-time set-up for the current device: resolve the scratch array's device
// address (which loads the library's module on this device, and with it the array,
// if that has not happened yet), the tensor-map encoder and the kernel's
// shared-memory configuration.  Only a successful set-up is kept: one that failed
// (for instance because it was attempted during a stream capture, where some of
// these calls are refused) is attempted again by the next call.
int noalloc_setup(int device, gmm_ctx **out) {
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  NoAllocDevice &d = g_noalloc_devices[device];
  if (d.ready) {
    *out = &d.ctx;
    return GMM_OK;
  }
  int major = 0, minor = 0, sms = 0, optin = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
  cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
  int rc = GMM_OK;
  if (major != 10 || minor != 3 || sms < 1) rc = GMM_ERR_NO_DEVICE;
  else if (sms > kNoAllocMaxCtas) rc = GMM_ERR_UNSUPPORTED;   // scratch holds 256 CTA slots
  void *scratch = nullptr;
  if (rc == GMM_OK && cudaGetSymbolAddress(&scratch, g_noalloc_scratch) != cudaSuccess) rc = GMM_ERR_CUDA;
  void *fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (rc == GMM_OK &&
      (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
           cudaSuccess ||
       q != cudaDriverEntryPointSuccess || !fn))
    rc = GMM_ERR_CUDA;
  if (rc == GMM_OK) {
    d.ctx.device = device;
    d.ctx.num_sms = sms;
    d.ctx.encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    d.ctx.use_pairs = 0;   // one CTA per tile: the grid is the SM count, one scratch slot per CTA
    int sm_smem = 0;
    cudaDeviceGetAttribute(&sm_smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, device);
    if (configure<false, false>(&d.ctx.var[0][0], optin, sm_smem, optin, sms) != GMM_OK) rc = GMM_ERR_CUDA;
    d.ctx.ws = static_cast<uint8_t *>(scratch);
    d.ctx.ws_bytes = kNoAllocScratchBytes;
  }
  if (rc != GMM_OK) {
    cudaGetLastError();
    return rc;
  }
  d.ready = true;
  *out = &d.ctx;
  return GMM_OK;
}

}  // namespace

extern "C" int gmm_run_noalloc(void *c, const void *a, const uint32_t *a_offsets, const void *b,
                               const int32_t *expert_ids, uint32_t *expert_usage_stats, int num_experts,
                               int num_groups, int N, int K, cudaStream_t stream) {
  if (num_experts < 1) return GMM_ERR_INVALID_ARG;
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess || device < 0) {
    cudaGetLastError();
    return GMM_ERR_NO_DEVICE;
  }
  if (device >= kNoAllocMaxDevices) return GMM_ERR_UNSUPPORTED;
  gmm_ctx *h = nullptr;
  int rc = noalloc_setup(device, &h);
  if (rc) return rc;
  rc = check_common(h, c, a, a_offsets, expert_ids, expert_usage_stats, num_groups, N, K);
  if (rc) return rc;
  if (!b || !aligned16(b)) return GMM_ERR_INVALID_ARG;

  GmmParams p;
  std::memset(&p, 0, sizeof(p));
  {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(N),
                          static_cast<cuuint64_t>(num_experts)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * 2, static_cast<cuuint64_t>(N) * K * 2};
    cuuint32_t box[3] = {gmm::kBK, gmm::kBlockN, 1};
    rc = encode_map(h, &p.w_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, b, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
  }
  rc = encode_token_maps(h, p, a, K, 1);
  if (rc) return rc;
  fill_common(h, p, c, a_offsets, expert_ids, expert_usage_stats, num_groups, N, K, max_tok(h, false));
  p.num_experts = num_experts;
  // The status word keeps the previous call's flags: clear it (stream-ordered, no allocation).
  if (cudaMemsetAsync(h->ws, 0, sizeof(uint32_t), stream) != cudaSuccess) {
    cudaGetLastError();
    return GMM_ERR_CUDA;
  }
  return launch<false>(h, p, stream);
}
