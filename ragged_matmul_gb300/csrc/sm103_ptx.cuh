// Inline-PTX building blocks for sm_103a: mbarriers, TMA tensor copies,
// tcgen05 (TMEM allocation, MMA, commit, TMEM loads) and device-side tensor-map
// patching.  Each wrapper is one PTX instruction (or a tiny fixed sequence) so
// that the kernels read as the pipeline they implement.
#pragma once

#include <cstdint>
#include <cuda.h>

namespace gmm {

// ----------------------------------------------------------------- misc

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ----------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async proxy (TMA, tcgen05.commit).
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Order this thread's generic-proxy shared-memory writes before later async-proxy
// reads of the same bytes (tcgen05.mma operand reads).
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// TMA store of a 2-D box from shared memory, in this thread's bulk async-group.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, uint32_t src, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(map), "r"(src),
               "r"(x), "r"(y)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until at most N of this thread's bulk groups still read their shared-memory source.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until all of this thread's bulk groups have completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Non-blocking test of a phase (returns at once).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// The same test, but a thread whose phase is not complete may be suspended in
// hardware until it completes or `hint_ns` nanoseconds pass, instead of returning at
// once; a waiting thread then takes no issue slots from the warps doing work.
__device__ __forceinline__ bool mbar_try_wait_hint(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return done != 0;
}

// 16-byte shared-memory load that the compiler keeps in place (after the wait that
// made the data visible).
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// ----------------------------------------------------------------- TMA

// L2 eviction-priority policies for TMA loads (.L2::cache_hint operands).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                                 int32_t x, int32_t y, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "l"(pol)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                                 int32_t x, int32_t y, int32_t z, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z), "l"(pol)
      : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Rewrite the extent of dimension 1 (rows) of a tensor map that lives in global memory.
__device__ __forceinline__ void tensormap_set_dim1(void *gmap, uint32_t extent) {
  asm volatile("tensormap.replace.tile.global_dim.global.b1024.b32 [%0], 1, %1;" ::"l"(
                   reinterpret_cast<uint64_t>(gmap)),
               "r"(extent)
               : "memory");
}

// Rewrite the box size of dimension 1 (rows per copy) of a tensor map in global memory.
__device__ __forceinline__ void tensormap_set_box1(void *gmap, uint32_t rows) {
  asm volatile("tensormap.replace.tile.box_dim.global.b1024.b32 [%0], 1, %1;" ::"l"(
                   reinterpret_cast<uint64_t>(gmap)),
               "r"(rows)
               : "memory");
}

// Make generic-proxy writes of global tensor maps (this thread's) visible to the
// tensor-map proxy, for any thread that acquires them afterwards.
__device__ __forceinline__ void tensormap_release() {
  asm volatile("fence.proxy.tensormap::generic.release.gpu;" ::: "memory");
}

// Acquire a global tensor map for this thread's later bulk tensor copies.
__device__ __forceinline__ void tensormap_acquire(const void *gmap) {
  asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(
                   reinterpret_cast<uint64_t>(gmap))
               : "memory");
}

// ----------------------------------------------------------------- tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// The tcgen05.mma and tcgen05.commit wrappers below are executed by a whole,
// converged warp with the same operands in every lane; one lane, chosen by
// elect.sync inside the wrapper, issues the instruction.  Operands computed by the
// whole warp are warp-uniform, so the compiler keeps them in uniform registers, which
// these instructions read, instead of moving them there before every issue.
//
// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulator (kind::f16).
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t.reg .b32 l;\n\t"
      "elect.sync l|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// One pipeline stage of the 4-bit kernel, from the wait for its operands to the commit
// that frees them: up to `tries` suspended tests of the stage's `full` barrier (phase
// `parity`; kPair: at cluster scope, relaxed), a warp vote so that every lane agrees,
// and, once it completed, a tcgen05 fence, eight MMAs over 128 of K (A in tensor
// memory: two 64-K slabs at a0 and a1, 8 columns per K step of 16; B in shared memory:
// two sub-slab descriptors whose low words are b0 and b1, high word bhi, +32 bytes per
// K step) and a commit of all of them to `empty` (kPair: cta_group::2, multicast to both
// CTAs' barriers).  Returns 1 when the stage was issued, 0 when the barrier had not
// completed after the tests (the caller checks its clock and tries again).
//
// Everything is one instruction stream with a single elect: the issuing warp shares its
// SM sub-partition with dequantisation warps that keep the issue port busy, and each
// instruction of its own costs it tens of cycles there.  A descriptor step adds to the
// low word only: the 14-bit start-address field holds shared-memory addresses >> 4,
// below 256 KB, so the step never carries out of it.  `accumulate` = 0 only for a
// tile's first stage: its first MMA then overwrites the accumulator.
#define GMM_TS_MMA(CG, A, B, P) "@e tcgen05.mma.cta_group::" CG ".kind::f16 [%1], [" A "], " B ", %7, " P ";\n\t"
#define GMM_TS_STAGE(CG, WAIT)                                                                 \
  "{\n\t.reg .pred e, p, t, r, v;\n\t.reg .b32 l, a, c, n;\n\t.reg .b64 b;\n\t"                      \
  "mov.u32 n, 0;\n\t"                                                                         \
  "GMM_W%=:\n\t" WAIT " r, [%10], %11, 1048576;\n\t"                                           \
  "vote.sync.all.pred v, r, 0xffffffff;\n\t"                                                 \
  "@v bra.uni GMM_G%=;\n\t"                                                                   \
  "add.u32 n, n, 1;\n\t"                                                                      \
  "setp.lt.u32 t, n, %12;\n\t"                                                                \
  "@t bra.uni GMM_W%=;\n\t"                                                                   \
  "mov.u32 %0, 0;\n\t"                                                                        \
  "bra.uni GMM_E%=;\n\t"                                                                      \
  "GMM_G%=:\n\t"                                                                              \
  "tcgen05.fence::after_thread_sync;\n\t"                                                     \
  "elect.sync l|e, 0xffffffff;\n\t"                                                          \
  "setp.ne.b32 p, %8, 0;\n\t"                                                                 \
  "setp.eq.b32 t, %8, %8;\n\t"                                                                \
  "mov.b64 b, {%4, %6};\n\t" GMM_TS_MMA(CG, "%2", "b", "p")                                  \
  "add.u32 a, %2, 8;\n\tadd.u32 c, %4, 2;\n\tmov.b64 b, {c, %6};\n\t" GMM_TS_MMA(CG, "a", "b", "t")  \
  "add.u32 a, %2, 16;\n\tadd.u32 c, %4, 4;\n\tmov.b64 b, {c, %6};\n\t" GMM_TS_MMA(CG, "a", "b", "t") \
  "add.u32 a, %2, 24;\n\tadd.u32 c, %4, 6;\n\tmov.b64 b, {c, %6};\n\t" GMM_TS_MMA(CG, "a", "b", "t") \
  "mov.b64 b, {%5, %6};\n\t" GMM_TS_MMA(CG, "%3", "b", "t")                                  \
  "add.u32 a, %3, 8;\n\tadd.u32 c, %5, 2;\n\tmov.b64 b, {c, %6};\n\t" GMM_TS_MMA(CG, "a", "b", "t")  \
  "add.u32 a, %3, 16;\n\tadd.u32 c, %5, 4;\n\tmov.b64 b, {c, %6};\n\t" GMM_TS_MMA(CG, "a", "b", "t") \
  "add.u32 a, %3, 24;\n\tadd.u32 c, %5, 6;\n\tmov.b64 b, {c, %6};\n\t" GMM_TS_MMA(CG, "a", "b", "t")

template <bool kPair>
__device__ __forceinline__ uint32_t mma_stage_ts_x8(uint32_t full, uint32_t parity, uint32_t tries, uint32_t d_tmem,
                                                    uint32_t a0, uint32_t a1, uint32_t b0, uint32_t b1, uint32_t bhi,
                                                    uint32_t idesc, uint32_t accumulate, uint32_t empty) {
  uint32_t issued;
  if constexpr (kPair) {
    asm volatile(GMM_TS_STAGE("2", "mbarrier.try_wait.parity.relaxed.cluster.shared::cta.b64")
                 "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
                 " [%9], %13;\n\t"
                 "mov.u32 %0, 1;\n\t"
                 "GMM_E%=:\n\t}"
                 : "=r"(issued)
                 : "r"(d_tmem), "r"(a0), "r"(a1), "r"(b0), "r"(b1), "r"(bhi), "r"(idesc), "r"(accumulate), "r"(empty),
                   "r"(full), "r"(parity), "r"(tries), "h"(static_cast<uint16_t>(3))
                 : "memory");
  } else {
    asm volatile(GMM_TS_STAGE("1", "mbarrier.try_wait.parity.shared::cta.b64")
                 "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%9];\n\t"
                 "mov.u32 %0, 1;\n\t"
                 "GMM_E%=:\n\t}"
                 : "=r"(issued)
                 : "r"(d_tmem), "r"(a0), "r"(a1), "r"(b0), "r"(b1), "r"(bhi), "r"(idesc), "r"(accumulate), "r"(empty),
                   "r"(full), "r"(parity), "r"(tries)
                 : "memory");
  }
  return issued;
}
#undef GMM_TS_STAGE
#undef GMM_TS_MMA

// Arrive once on `bar` when every tcgen05.mma issued so far (by this warp) has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t.reg .b32 l;\n\t"
      "elect.sync l|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
      : "memory");
}

// Each thread of the warp reads 16 consecutive 32-bit columns of its own TMEM lane.
__device__ __forceinline__ void tmem_ld_x16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
}

// The same for 32 columns.
__device__ __forceinline__ void tmem_ld_x32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]),
        "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]),
        "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
}

// Per-thread register budget of the calling warpgroup: every warp of the warpgroup
// executes the same instruction.  A decrease returns registers to the CTA's pool; an
// increase waits until the pool (registers a thread at launch x threads) has them.
template <uint32_t kRegs>
__device__ __forceinline__ void warpgroup_regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegs));
}
template <uint32_t kRegs>
__device__ __forceinline__ void warpgroup_regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegs));
}

// (d0, d1) = a * (b0, b1) + (d0, d1) in one paired fp32 instruction; each lane is
// rounded as fmaf.
__device__ __forceinline__ void fma_f32x2(float &d0, float &d1, float a, float b0, float b1) {
  asm("{\n\t.reg .b64 x, y, z;\n\t"
      "mov.b64 x, {%2, %2};\n\t"
      "mov.b64 y, {%3, %4};\n\t"
      "mov.b64 z, {%0, %1};\n\t"
      "fma.rn.f32x2 z, x, y, z;\n\t"
      "mov.b64 {%0, %1}, z;\n\t}"
      : "+f"(d0), "+f"(d1)
      : "f"(a), "f"(b0), "f"(b1));
}

// 16 TMEM lanes x 32 columns in the 16x256b shape (four repeats of 16 lanes x 8
// columns).  In repeat j (v[4j] .. v[4j + 3]) thread t holds lane t/4, columns
// 8j + 2(t%4) and 8j + 2(t%4) + 1 (v[4j], v[4j + 1]), and the same two columns of
// lane t/4 + 8 (v[4j + 2], v[4j + 3]), lanes counted from the lane of taddr.
__device__ __forceinline__ void tmem_ld_16x256b_x4(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
}

// Four 8x8 matrices of 16-bit values to shared memory, each transposed: thread t's
// word m (two values, row t/4 and columns 2(t%4), 2(t%4) + 1 of matrix m, the lower
// column in the low half) lands in rows 2(t%4) and 2(t%4) + 1, column t/4, of the
// stored matrix m, whose row r is the 16 bytes at the address of thread 8m + r.
__device__ __forceinline__ void stmatrix_x4_trans(uint32_t saddr, uint32_t r0, uint32_t r1, uint32_t r2,
                                                  uint32_t r3) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(saddr), "r"(r0),
               "r"(r1), "r"(r2), "r"(r3)
               : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Store 32 consecutive 32-bit columns from `taddr` (lane field: the warp's quadrant):
// thread t writes lane (taddr >> 16) + t, columns v[0..31].
__device__ __forceinline__ void tmem_st_x32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, "
      "%9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, "
      "%25, %26, %27, %28, %29, %30, %31, %32};"
      ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]),
        "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]),
        "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ----------------------------------------------------------------- clusters / CTA pairs

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_count_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}

// Address of the same shared-memory variable in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

// Store a 32-bit value into another CTA's shared memory (cluster address).
__device__ __forceinline__ void st_shared_cluster_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

// Whole-cluster barrier (every thread of every CTA in the cluster).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}

// Arrive on an mbarrier that may live in another CTA of the cluster.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Arrivals with relaxed semantics, for a signal that publishes no memory writes of
// this thread: the tensor-memory loads or stores it follows have already completed
// (tcgen05.wait::ld / wait::st, then tcgen05.fence::before_thread_sync).  A release
// arrive at cluster scope first waits until every earlier global store of the thread
// is visible across the cluster, which after an epilogue's stores takes about a
// microsecond.
__device__ __forceinline__ void mbar_arrive_relaxed(uint32_t bar) {
  asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

__device__ __forceinline__ bool mbar_test_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ bool mbar_try_wait_cluster_hint(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return done != 0;
}

// The cluster-scope test and wait without acquire semantics, for phases that publish
// no generic-proxy writes: tensor-memory accesses ordered by tcgen05 fences, and TMA
// bytes that the barrier itself counts.
__device__ __forceinline__ bool mbar_test_wait_cluster_relaxed(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.relaxed.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ bool mbar_try_wait_cluster_relaxed_hint(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.relaxed.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return done != 0;
}

// TMA loads of a CTA pair: the destination is this CTA's shared memory, the
// completion may be signalled on the leader CTA's mbarrier (a cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *map, uint32_t bar_cluster,
                                                 int32_t x, int32_t y, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y), "l"(pol)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap *map, uint32_t bar_cluster,
                                                 int32_t x, int32_t y, int32_t z, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y), "r"(z), "l"(pol)
      : "memory");
}

// TMEM allocation for a CTA pair: one warp of EACH CTA of the pair executes it.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// Pair MMA issued by the leader CTA: M = 256 rows split 128/128 over the two CTAs'
// shared memory (A operand) and TMEM (D); the N rows of the B operand come half
// from each CTA's shared memory at the same offsets.
__device__ __forceinline__ void mma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t.reg .b32 l;\n\t"
      "elect.sync l|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The same two forms for 8-bit operands (kind::f8f6f4): K = 32 elements, i.e. the
// same 32 bytes of each 128-byte swizzled row as one bf16 MMA, so the descriptors and
// their per-step advance are the bf16 ones; the formats are in the instruction
// descriptor.
__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t.reg .b32 l;\n\t"
      "elect.sync l|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_f8_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t.reg .b32 l;\n\t"
      "elect.sync l|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on the mbarrier at `bar` in every CTA of `cta_mask` when the pair MMAs
// issued so far have completed.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t.reg .b32 l;\n\t"
      "elect.sync l|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;\n\t}" ::"r"(bar),
      "h"(cta_mask)
      : "memory");
}

// One stage of the per-K-block e4m3 kernel (128 of K): four kind::f8f6f4 MMAs, A and B
// in shared memory (descriptors whose low words are a_lo and b_lo and high words a_hi
// and b_hi; +32 bytes per step of K = 32), then a commit of them to `empty` and, when
// `block_end` is non-zero, a second commit to `part` (the K block's partial is
// complete).  One elected lane issues everything; the issuing warp shares its SM
// sub-partition with the promotion warps.  `accumulate` = 0 for the first stage of a
// K block: its first MMA then overwrites the partial buffer.  A descriptor step adds
// to the low word only (shared-memory addresses >> 4 stay below 2^14: no carry).
__device__ __forceinline__ void mma_stage_f8_x4(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi, uint32_t b_lo,
                                                uint32_t b_hi, uint32_t idesc, uint32_t accumulate, uint32_t empty,
                                                uint32_t block_end, uint32_t part) {
  asm volatile(
      "{\n\t.reg .pred e, p, t, q;\n\t.reg .b32 l, x, y;\n\t.reg .b64 a, b;\n\t"
      "elect.sync l|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "setp.eq.b32 t, %6, %6;\n\t"
      "setp.ne.b32 q, %8, 0;\n\t"
      "mov.b64 a, {%1, %2};\n\tmov.b64 b, {%3, %4};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], a, b, %5, p;\n\t"
      "add.u32 x, %1, 2;\n\tadd.u32 y, %3, 2;\n\tmov.b64 a, {x, %2};\n\tmov.b64 b, {y, %4};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], a, b, %5, t;\n\t"
      "add.u32 x, %1, 4;\n\tadd.u32 y, %3, 4;\n\tmov.b64 a, {x, %2};\n\tmov.b64 b, {y, %4};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], a, b, %5, t;\n\t"
      "add.u32 x, %1, 6;\n\tadd.u32 y, %3, 6;\n\tmov.b64 a, {x, %2};\n\tmov.b64 b, {y, %4};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], a, b, %5, t;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%7];\n\t"
      "and.pred q, q, e;\n\t"
      "@q tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%9];\n\t}" ::"r"(d_tmem),
      "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate), "r"(empty), "r"(block_end),
      "r"(part)
      : "memory");
}

// ----------------------------------------------------------------- descriptors

// Shared-memory matrix descriptor for a K-major operand tile written by TMA with
// 128-byte swizzling: rows of 64 bf16 (128 B), 8-row swizzle atoms 1024 B apart.
// The tile base must be 1024-byte aligned; stepping K by 16 elements inside the
// 128-byte row adds 32 B to the start address.
__device__ __forceinline__ uint64_t smem_desc_k_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);   // [0,14)  start address >> 4
  d |= static_cast<uint64_t>(16u >> 4) << 16;            // [16,30) leading byte offset (unused here)
  d |= static_cast<uint64_t>(1024u >> 4) << 32;          // [32,46) stride byte offset: 8 rows x 128 B
  d |= static_cast<uint64_t>(1u) << 46;                  // [46,48) descriptor version
  d |= static_cast<uint64_t>(2u) << 61;                  // [61,64) swizzle: 128 B
  return d;
}

// Instruction descriptor, kind::f16: bf16 A and B (both K-major), fp32 D, shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(uint32_t M, uint32_t N) {
  return (1u << 4)              // D format: f32
         | (1u << 7)            // A format: bf16
         | (1u << 10)           // B format: bf16
         | ((N >> 3) << 17)     // N / 8
         | ((M >> 4) << 24);    // M / 16
}

// Instruction descriptor, kind::f8f6f4: e4m3 A and B (format code 0, both K-major),
// fp32 D, shape M x N.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(uint32_t M, uint32_t N) {
  return (1u << 4)              // D format: f32
         | (0u << 7)            // A format: e4m3
         | (0u << 10)           // B format: e4m3
         | ((N >> 3) << 17)     // N / 8
         | ((M >> 4) << 24);    // M / 16
}

}  // namespace gmm
