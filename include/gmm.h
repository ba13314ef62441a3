/*
 * gmm.h — C ABI of the GB300 (sm_103a) ragged grouped GEMM library (libgmm.so).
 *
 * The operation (Modular "grouped_matmul_sm100_persistent" API page, section
 * "Args"): for every group g whose expert id e = expert_ids[g] satisfies
 * 0 <= e < num_experts,
 *
 *     C[r, n] = bf16( sum_k A[r, k] * B[e, n, k] )
 *         for r in [a_offsets[g], a_offsets[g+1]), n in [0, N)
 *
 * accumulated in fp32 on the tensor cores and rounded to nearest even.
 *   - A  : bf16 [rows, K], row-major (K contiguous).  rows >= a_offsets[num_groups].
 *   - B  : bf16 [num_experts, N, K], row-major — the transposed-B convention of the
 *          page (each expert's weight matrix is stored N x K).
 *   - C  : bf16 [rows, N], row-major.
 *   - a_offsets          : uint32 [num_groups + 1], non-decreasing prefix sum of rows per group.
 *   - expert_ids         : int32  [num_groups]; a negative id skips the group.
 *   - expert_usage_stats : uint32 [>= 2]; index 1 receives the number of groups with
 *                          0 <= id < num_experts.  No other entry is read or written.
 * Rows of C that no active group covers keep their previous contents, bit for bit.
 *
 * Device-side conventions (checked on the device, reported by gmm_query_status):
 *   - a decreasing a_offsets entry: nothing is computed, stats[1] is still written,
 *     status GMM_ERR_BAD_INPUT;
 *   - an expert id >= num_experts: that group is skipped and not counted,
 *     status GMM_ERR_BAD_INPUT.
 *
 * All pointers passed to the run calls are DEVICE pointers on the handle's device
 * and are owned by the caller.  The run calls are asynchronous on `stream`: they
 * validate the arguments on the host, launch one persistent kernel and return;
 * they do not synchronise and allocate nothing.  They can be captured in a CUDA
 * graph and replayed (every device write they make before the kernel is a value
 * write, not a copy from host memory); gmm_query_status synchronises and must not
 * be called during a capture.
 *
 * A handle owns a small device workspace (a status word, a 64-bit tile-claim
 * word and a finished-CTA counter that each launch returns to zero, the routing of
 * gmm_matmul_int4's single group, and per-CTA tensor-map slots) that
 * every launch made through it rewrites.  Launches made through the
 * same handle must therefore not overlap on the GPU: issue them on one stream, or
 * use one handle per stream.
 */
#ifndef GMM_H_
#define GMM_H_

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes.  0 is success; everything else is negative. */
#define GMM_OK                  0
#define GMM_ERR_INVALID_ARG    -1  /* null pointer, negative size, misaligned or badly shaped operand */
#define GMM_ERR_UNSUPPORTED    -2  /* valid request outside what the kernels implement (e.g. too many groups) */
#define GMM_ERR_CUDA           -3  /* a CUDA runtime/driver call failed (allocation, launch, copy) */
#define GMM_ERR_DEVICE_TIMEOUT -4  /* a kernel gave up waiting on its own pipeline (reported by gmm_query_status) */
#define GMM_ERR_BAD_INPUT      -5  /* decreasing a_offsets or an expert id >= num_experts (gmm_query_status) */
#define GMM_ERR_NO_DEVICE      -6  /* the device is not an sm_103 GPU, or none is present */

typedef struct gmm_ctx *gmm_handle_t;

/*
 * Create a handle for `device` and `num_experts` experts (E, the leading
 * dimension of B; used for the id bounds check and the B tensor map).  This is
 * the host-side set-up that the grouped GEMM page's launcher does before its
 * persistent kernel (Modular "grouped_matmul_sm100_persistent", description: it
 * builds the TMA descriptors and picks the pipeline depth from the shared memory
 * available): here every kernel's shared-memory budget is read from the device's
 * opt-in shared memory once, each launch sizes its rings beside that call's group
 * prefix, and the tensor maps are built per call.
 * Allocates the handle's device workspace on `device` (cudaMalloc).  The
 * caller's current device is left unchanged.
 * Errors: GMM_ERR_INVALID_ARG (out == NULL, num_experts < 1),
 *         GMM_ERR_NO_DEVICE (no such device, or not compute capability 10.3),
 *         GMM_ERR_CUDA (allocation failed, or a kernel's launch configuration could
 *         not be set up).  *out is NULL on error.
 */
int gmm_create(gmm_handle_t *out, int num_experts, int device);

/*
 * bf16 ragged grouped GEMM (see the header comment for the operation).
 * N and K: multiples of 8 (16-byte rows, a TMA requirement), both >= 8.
 * c, a, b: 16-byte aligned.  num_groups: 0 .. 4096.
 * With num_groups == 0 only expert_usage_stats[1] = 0 is written (expert_ids may then be NULL).
 * Errors (nothing is launched): GMM_ERR_INVALID_ARG, GMM_ERR_UNSUPPORTED,
 *         GMM_ERR_CUDA (tensor-map encoding or launch failed).
 */
int gmm_run(gmm_handle_t h, void *c, const void *a, const uint32_t *a_offsets, const void *b,
            const int32_t *expert_ids, uint32_t *expert_usage_stats, int num_groups, int N, int K,
            cudaStream_t stream);

/*
 * Optional elementwise epilogue, applied to each fp32 result before it is rounded
 * to bf16 (the grouped and quantised GEMM pages both take an optional elementwise
 * function on the output: Modular "grouped_matmul_sm100_persistent" and
 * "multistage_gemm_q", section "Parameters", elementwise_lambda_fn; a C interface
 * takes these common steps instead of a function):
 *     y = act( acc[r, n] + bias[e, n] ) * row_scale[r]
 * where e is the group's expert and r the row of A.  Each part is optional:
 *   bias:       bf16 [num_experts, N] (2-byte aligned), or NULL for none;
 *   row_scale:  fp32 [rows of A] (4-byte aligned, e.g. routing weights), or NULL;
 *   activation: GMM_ACT_NONE, GMM_ACT_RELU (max(y, 0)), GMM_ACT_SILU (y / (1 + e^-y)),
 *               GMM_ACT_GELU_TANH (y/2 (1 + tanh(sqrt(2/pi) (y + 0.044715 y^3)))).
 * Rows that no active group covers stay untouched, as without the epilogue.
 */
#define GMM_ACT_NONE      0
#define GMM_ACT_RELU      1
#define GMM_ACT_SILU      2
#define GMM_ACT_GELU_TANH 3

typedef struct gmm_epilogue {
  const void *bias;
  const float *row_scale;
  int activation;
} gmm_epilogue;

/*
 * gmm_run with the optional epilogue (epilogue == NULL: exactly gmm_run).
 * Errors: as gmm_run, plus GMM_ERR_INVALID_ARG for an unknown activation or a
 * misaligned bias / row_scale.
 */
int gmm_run_ex(gmm_handle_t h, void *c, const void *a, const uint32_t *a_offsets, const void *b,
               const int32_t *expert_ids, uint32_t *expert_usage_stats, int num_groups, int N, int K,
               const gmm_epilogue *epilogue, cudaStream_t stream);

/*
 * 4-bit grouped GEMM (the grouped path with the weights of Modular's
 * "multistage_gemm_q", section "Parameters": pack_factor 4-bit values per uint32 and
 * one scale per group_size K elements).  B[e, n, k] is replaced by
 *     w = bf16( (q - 8) * scale[e, n, k / group_size] ),
 *     q = bits [4*(k%8), 4*(k%8)+4) of b_packed[e, n, k/8]   (low nibble first),
 * b_packed: uint32 [num_experts, N, K/8] (16-byte aligned);
 * b_scales: bf16 [num_experts, N, K/group_size] (2-byte aligned).
 * Requirements: those of gmm_run, plus group_size a multiple of 64 that divides K.
 * Errors: as gmm_run.
 */
int gmm_run_int4(gmm_handle_t h, void *c, const void *a, const uint32_t *a_offsets,
                 const uint32_t *b_packed, const void *b_scales, const int32_t *expert_ids,
                 uint32_t *expert_usage_stats, int num_groups, int N, int K, int group_size,
                 cudaStream_t stream);

/*
 * Dense rank-2 4-bit GEMM (Modular "multistage_gemm_q": C = A . B^T with B packed
 * 4-bit and group-quantised, section "Parameters": pack_factor, group_size):
 *     C[r, n] = sum_k A[r, k] * w[n, k],  w[n, k] = bf16( (q - 8) * scale[n, k / group_size] )
 * for r < M, with the nibble layout of gmm_run_int4.  It is the grouped path with one
 * group of M rows and one expert; the group's offsets and id are written into the
 * handle's workspace (stream-ordered), so the caller passes none.
 *   c: bf16 [M, N]; a: bf16 [M, K]; b_packed: uint32 [N, K/8]; b_scales: bf16 [N, K/group_size].
 * The page's function raises when an operand is not rank-2; here the ranks are fixed
 * by the signature (the Python binding raises for tensors of another rank).
 * M == 0 launches nothing.  Requirements and errors: as gmm_run_int4_ex, plus
 * GMM_ERR_INVALID_ARG for M < 0.  Calls through one handle share its workspace, so
 * they must be stream-ordered, as for every call through a handle.
 */
int gmm_matmul_int4(gmm_handle_t h, void *c, const void *a, const uint32_t *b_packed, const void *b_scales,
                    int M, int N, int K, int group_size, const gmm_epilogue *epilogue, cudaStream_t stream);

/* gmm_run_int4 with the optional epilogue (epilogue == NULL: exactly gmm_run_int4). */
int gmm_run_int4_ex(gmm_handle_t h, void *c, const void *a, const uint32_t *a_offsets,
                    const uint32_t *b_packed, const void *b_scales, const int32_t *expert_ids,
                    uint32_t *expert_usage_stats, int num_groups, int N, int K, int group_size,
                    const gmm_epilogue *epilogue, cudaStream_t stream);

/*
 * The bf16 grouped GEMM with A-plane row offsetting (Modular
 * "grouped_matmul_sm100_persistent", section "Parameters": a_plane_splits, per-plane
 * split sizes for fused LoRA QKV A-plane row offsetting, (0, 0) disabling it).  The
 * reading taken: a holds three planes of M = a_offsets[G] rows, stacked along its rows
 * ([3 M, K], e.g. the q, k and v inputs of a fused QKV projection), and
 * (s0, s1) = a_plane_splits cut the N columns into three parts:
 *     C[r, n] = bf16( sum_k a[p(n) * M + r, k] * b[e, n, k] ),
 *     p(n) = 0 for n < s0, 1 for s0 <= n < s0 + s1, 2 otherwise,
 * for the rows and groups of gmm_run, then the optional epilogue.  (0, 0) is gmm_run_ex.
 * a must hold 3 * a_offsets[G] rows (any a_offsets[G] rows when the splits are (0, 0)).
 * Requirements: those of gmm_run, s0 and s1 multiples of 256 (a tile's 256 weight rows
 * lie in one plane; else GMM_ERR_UNSUPPORTED), 0 <= s0, 0 <= s1, s0 + s1 <= N (else
 * GMM_ERR_INVALID_ARG, also for a NULL a_plane_splits).  Errors: as gmm_run_ex.
 */
int gmm_run_planes(gmm_handle_t h, void *c, const void *a, const uint32_t *a_offsets, const void *b,
                   const int32_t *expert_ids, uint32_t *expert_usage_stats, int num_groups, int N, int K,
                   const int *a_plane_splits, const gmm_epilogue *epilogue, cudaStream_t stream);

/*
 * Block-scaled e4m3 grouped GEMM (Modular "k_matmul_ragged_paged_scale", section
 * "Args": input_scale and weight_scale multiply the input and the weight; template
 * parameter scales_granularity_mnk; without the page's paged KV-cache write, the
 * result goes to C as in gmm_run).  With (gm, gn, gk) = scales_granularity_mnk and
 * kb = k / gk the K block of k:
 *     C[r, n] = bf16( sum_kb input_scale[r / gm, kb] * weight_scale[e, n / gn, kb]
 *                            * sum_{k in block kb} a[r, k] * b[e, n, k] )
 * for the rows and groups of gmm_run, a and b e4m3 (1 sign, 4 exponent bits with
 * bias 7, 3 mantissa bits), sums in fp32.  Then the optional epilogue.
 *   a: e4m3 bytes [rows, K] (16-byte aligned); b: e4m3 bytes [num_experts, N, K]
 *   (16-byte aligned); input_scale: fp32 [ceil(rows / gm), ceil(K / gk)];
 *   weight_scale: fp32 [num_experts, ceil(N / gn), ceil(K / gk)] (both row-major,
 *   4-byte aligned, read only for active groups); c and the rest as gmm_run.
 * Requirements: those of gmm_run with K a multiple of 16 (an e4m3 row is K bytes, a
 * multiple of 16 for TMA), gm, gn, gk >= 1, and either gk >= K (one scale over the
 * whole reduction, applied to the finished sum) or gk a multiple of 128 with gn a
 * multiple of 32 (per-K-block scales, a kernel of their own); other granularities
 * return GMM_ERR_UNSUPPORTED.
 * Errors: as gmm_run_ex, plus GMM_ERR_INVALID_ARG for NULL or misaligned scales,
 * a NULL scales_granularity_mnk or a granularity below 1.
 */
int gmm_run_fp8(gmm_handle_t h, void *c, const void *a, const uint32_t *a_offsets, const void *b,
                const int32_t *expert_ids, uint32_t *expert_usage_stats, int num_groups, int N, int K,
                const float *input_scale, const float *weight_scale, const int *scales_granularity_mnk,
                const gmm_epilogue *epilogue, cudaStream_t stream);

/*
 * Allocation-free variant of gmm_run, for callers that cannot call cudaMalloc when
 * they need the GEMM: code running inside an allocator or memory-pool callback, a
 * framework that has reserved all device memory for its own pool, or a runtime that
 * forbids allocations after start-up.  The pages have no counterpart to this call.
 *
 * It computes exactly what gmm_run computes, with the same kernel, on the CALLER'S
 * CURRENT DEVICE (all pointers must live there), and needs no handle: num_experts is
 * passed directly.  The caller still provides every input and output buffer.  The
 * kernel's scratch (a status word and one 2 KB slot of tensor maps per CTA) comes from
 * a fixed array compiled into the library, 524,544 bytes on every GPU that loads it,
 * held until the process exits.  That array has slots for at most 256 CTAs; the grid
 * is one CTA per SM, so a device with more than 256 SMs gets GMM_ERR_UNSUPPORTED.
 *
 * The first call on a device does a one-time set-up (looks up the array's device
 * address, the tensor-map encoder, and the kernel's shared-memory setting); make that
 * first call before any stream capture.  A set-up that fails is not remembered: the
 * next call tries it again.  No call allocates or frees device memory itself, but
 * note that CUDA loads a library's device code lazily by default: the array is
 * reserved on a device when the library's module is first loaded there, which is
 * the first call into this library on that device (this one or any other).  A
 * caller that later hands all free device memory to its own pool should make one
 * call at start-up, before it does so.
 *
 * Every call shares the one array and finds the previous call's contents in it; the
 * call clears the status word itself (stream-ordered on `stream`), rewrites the
 * tensor-map slots, and its kernel returns the array's tile-claim word and
 * finished-CTA counter to zero when it finishes (they are zero when the library is loaded).  Calls whose kernels overlap on the GPU (different streams, or
 * concurrent threads) race on the array: order them on one stream.  The device
 * status (bad offsets / ids) is not reported by this call; the device still applies
 * the same rules (see the header comment).
 * Errors (nothing is launched): those of gmm_run, plus GMM_ERR_INVALID_ARG
 * (num_experts < 1), GMM_ERR_NO_DEVICE (current device is not sm_103),
 * GMM_ERR_UNSUPPORTED (more than 256 SMs, or a device index >= 64).
 */
int gmm_run_noalloc(void *c, const void *a, const uint32_t *a_offsets, const void *b,
                    const int32_t *expert_ids, uint32_t *expert_usage_stats, int num_experts,
                    int num_groups, int N, int K, cudaStream_t stream);

/*
 * The error report of the quantised GEMM page (Modular "multistage_gemm_q", section
 * "Raises": the function raises an error on invalid input) for the conditions that
 * only the device sees: decreasing offsets and out-of-range expert ids, and a
 * kernel that gave up on a pipeline wait.
 * Synchronise `stream`, then read and clear the device status that the kernels of
 * this handle accumulated since the last query.  Returns GMM_OK,
 * GMM_ERR_BAD_INPUT or GMM_ERR_DEVICE_TIMEOUT (timeout wins when both are set),
 * or GMM_ERR_CUDA when the synchronisation or the copy fails (for instance after
 * an earlier asynchronous fault).
 */
int gmm_query_status(gmm_handle_t h, cudaStream_t stream);

/* Static, NUL-terminated description of a return code. */
const char *gmm_error_string(int code);

/*
 * Release the handle and its workspace.  The caller must make sure no launch made
 * through the handle is still running (synchronise first).  NULL is accepted.
 */
int gmm_destroy(gmm_handle_t h);

#ifdef __cplusplus
}
#endif

#endif /* GMM_H_ */
