/*
 * CPU oracle for the ragged grouped GEMM behind a mixture-of-experts layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: it exists so the test suite, the smoke check and the
 * bench's CPU-baseline leg have an independent, obviously correct answer to
 * compare the CUDA kernels against.  It shares no code, header, table or
 * helper with the CUDA library.
 *
 * What it computes (Modular "grouped_matmul_sm100_persistent" API page,
 * section "Args": a_offsets is the per-group prefix sum of A rows, b holds the
 * weights in the transposed-B convention, expert_ids picks the expert of a
 * group and negative entries skip it, expert_usage_stats[1] holds the active
 * count):
 *
 *   for every group g with e = expert_ids[g], 0 <= e < E:
 *     for every row r in [a_offsets[g], a_offsets[g+1]) and column n in [0, N):
 *       ref[r, n] = sum_{k=0}^{K-1} A[r, k] * B[e, n, k]
 *       C[r, n]   = bf16 round-to-nearest-even of ref[r, n]
 *
 *   A is [rows, K] bf16, B is [E, N, K] bf16 (K contiguous, i.e. the
 *   transposed-B layout), C is [rows, N] bf16.  Rows that no active group
 *   covers keep whatever bits C held before the call.
 *
 * Conventions the pages leave open and this library fixes:
 *   - The sum is accumulated in fp32 in ascending k (products of two bf16
 *     values are exact in fp32).  An fp64 accumulation is also offered, for
 *     diagnostics and for pinning the fp32 result against its error bound.
 *   - expert_usage_stats[1] = number of groups with 0 <= expert_ids[g] < E
 *     (an empty group with a valid id counts).  No other entry is touched.
 *   - a_offsets must be non-decreasing.  If any a_offsets[g+1] < a_offsets[g]
 *     the call computes nothing (no C row is written), still writes
 *     expert_usage_stats[1], and reports ORACLE_BAD_OFFSETS.
 *   - A group whose id is >= E is skipped, is not counted, and is reported
 *     with ORACLE_BAD_EXPERT_ID.
 *
 * The 4-bit variant (Modular "multistage_gemm_q" API page, section
 * "Parameters": pack_factor 4-bit values per uint32, one scale per group_size
 * K elements) replaces B[e, n, k] by
 *     q = bits [4*(k%8), 4*(k%8)+4) of word k/8 of row (e, n)   (low nibble first)
 *     w = bf16_rne( (float)(q - 8) * scale[e, n, k / group_size] )
 * with zero point 8 and bf16 scales [E, N, K/group_size].  (q - 8) * scale is
 * exact in fp32 and is rounded to bf16 once, as the weight that feeds the MMA.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_BAD_OFFSETS   1
#define ORACLE_BAD_EXPERT_ID 2

/* ---- bf16 <-> fp32, written from the IEEE-754 binary16-brain-float layout ---- */

/* bf16 is the upper 16 bits of an fp32 value: widening is exact. */
static float bf16_bits_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round an fp32 value to the nearest bf16, ties to even.  NaN stays NaN (quiet). */
static uint16_t f32_to_bf16_bits_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u)          /* NaN: keep sign and payload top, set quiet bit */
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lower = u & 0xffffu;                 /* the 16 bits that are dropped */
    uint32_t upper = u >> 16;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))
        upper += 1u;                               /* carries into the exponent correctly, inf included */
    return (uint16_t)upper;
}

void oracle_round_bf16_array(uint16_t *out, const float *in, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = f32_to_bf16_bits_rne(in[i]);
}

/* ---- validation shared by both variants ---- */

int oracle_validate(const uint32_t *a_offsets, const int32_t *expert_ids, int num_groups,
                    int num_experts, uint32_t *active_count)
{
    int flags = 0;
    uint32_t active = 0;
    for (int g = 0; g < num_groups; ++g) {
        if (a_offsets[g + 1] < a_offsets[g]) flags |= ORACLE_BAD_OFFSETS;
        int32_t e = expert_ids[g];
        if (e >= num_experts) flags |= ORACLE_BAD_EXPERT_ID;
        if (e >= 0 && e < num_experts) active += 1;
    }
    *active_count = active;
    return flags;
}

/* ---- the row loop ---- */

/* One unit of work: an output row r computed with weights W (N x K, bf16 bits). */
typedef struct {
    int64_t row;
    const uint16_t *w;   /* points at B[e] (or a dequantised copy of it) */
} row_job;

typedef struct {
    const row_job *jobs;
    int64_t first, last;                 /* [first, last) */
    const uint16_t *a;
    uint16_t *c;
    float *ref32;
    double *ref64;
    int N, K;
} worker_arg;

static void compute_rows(const worker_arg *w)
{
    const int N = w->N, K = w->K;
    for (int64_t j = w->first; j < w->last; ++j) {
        const int64_t r = w->jobs[j].row;
        const uint16_t *arow = w->a + r * (int64_t)K;
        for (int n = 0; n < N; ++n) {
            const uint16_t *wrow = w->jobs[j].w + (int64_t)n * K;
            float acc32 = 0.0f;
            double acc64 = 0.0;
            for (int k = 0; k < K; ++k) {
                float x = bf16_bits_to_f32(arow[k]);
                float y = bf16_bits_to_f32(wrow[k]);
                acc32 += x * y;                    /* x * y is exact in fp32 */
                if (w->ref64) acc64 += (double)x * (double)y;
            }
            const int64_t o = r * (int64_t)N + n;
            if (w->c) w->c[o] = f32_to_bf16_bits_rne(acc32);
            if (w->ref32) w->ref32[o] = acc32;
            if (w->ref64) w->ref64[o] = acc64;
        }
    }
}

static void *worker_main(void *p)
{
    compute_rows((const worker_arg *)p);
    return NULL;
}

/* Run the jobs on up to nthreads threads; each output row is owned by exactly one thread. */
static void run_jobs(const row_job *jobs, int64_t njobs, const uint16_t *a, uint16_t *c,
                     float *ref32, double *ref64, int N, int K, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > njobs) nthreads = (int)(njobs > 0 ? njobs : 1);
    pthread_t tids[256];
    worker_arg args[256];
    int started[256];
    for (int t = 0; t < nthreads; ++t) {
        args[t].jobs = jobs;
        args[t].first = njobs * t / nthreads;
        args[t].last = njobs * (t + 1) / nthreads;
        args[t].a = a;
        args[t].c = c;
        args[t].ref32 = ref32;
        args[t].ref64 = ref64;
        args[t].N = N;
        args[t].K = K;
        started[t] = (t > 0) && pthread_create(&tids[t], NULL, worker_main, &args[t]) == 0;
        if (t > 0 && !started[t]) compute_rows(&args[t]);   /* no thread: do it here */
    }
    compute_rows(&args[0]);
    for (int t = 1; t < nthreads; ++t)
        if (started[t]) pthread_join(tids[t], NULL);
}

/*
 * bf16 grouped GEMM.
 *   c      : [rows_alloc, N] bf16 bits, written only for rows of active groups (may be NULL)
 *   ref32  : [rows_alloc, N] fp32 sums, same rows (may be NULL)
 *   ref64  : [rows_alloc, N] fp64 sums, same rows (may be NULL)
 *   stats  : expert_usage_stats; only index 1 is written (may be NULL)
 * Returns the ORACLE_* flags (0 when the input is valid), or -1 on allocation failure.
 */
int oracle_gmm_bf16(uint16_t *c, float *ref32, double *ref64, const uint16_t *a,
                    const uint32_t *a_offsets, const uint16_t *b, const int32_t *expert_ids,
                    uint32_t *stats, int num_groups, int num_experts, int N, int K, int nthreads)
{
    uint32_t active = 0;
    int flags = oracle_validate(a_offsets, expert_ids, num_groups, num_experts, &active);
    if (stats) stats[1] = active;
    if (flags & ORACLE_BAD_OFFSETS) return flags;

    int64_t njobs = 0;
    for (int g = 0; g < num_groups; ++g)
        if (expert_ids[g] >= 0 && expert_ids[g] < num_experts)
            njobs += (int64_t)a_offsets[g + 1] - (int64_t)a_offsets[g];
    row_job *jobs = (row_job *)malloc(sizeof(row_job) * (size_t)(njobs > 0 ? njobs : 1));
    if (!jobs) return -1;
    int64_t j = 0;
    for (int g = 0; g < num_groups; ++g) {
        int32_t e = expert_ids[g];
        if (e < 0 || e >= num_experts) continue;                 /* skipped group */
        for (int64_t r = a_offsets[g]; r < (int64_t)a_offsets[g + 1]; ++r) {
            jobs[j].row = r;
            jobs[j].w = b + (int64_t)e * N * K;
            ++j;
        }
    }
    run_jobs(jobs, njobs, a, c, ref32, ref64, N, K, nthreads);
    free(jobs);
    return flags;
}

/* Dequantise one expert's packed 4-bit weights into bf16 bits w[N, K]. */
void oracle_dequant_int4(uint16_t *w, const uint32_t *packed, const uint16_t *scales, int N, int K,
                         int group_size)
{
    const int words_per_row = K / 8;
    const int scales_per_row = K / group_size;
    for (int n = 0; n < N; ++n) {
        for (int k = 0; k < K; ++k) {
            uint32_t word = packed[(int64_t)n * words_per_row + k / 8];
            int q = (int)((word >> (4 * (k % 8))) & 0xfu);
            float s = bf16_bits_to_f32(scales[(int64_t)n * scales_per_row + k / group_size]);
            w[(int64_t)n * K + k] = f32_to_bf16_bits_rne((float)(q - 8) * s);
        }
    }
}

/*
 * 4-bit grouped GEMM: packed [E, N, K/8] uint32, scales [E, N, K/group_size] bf16 bits.
 * Same outputs and conventions as oracle_gmm_bf16.  Returns flags, -1 on allocation
 * failure, -2 when K or group_size do not divide as the packing requires.
 */
int oracle_gmm_int4(uint16_t *c, float *ref32, double *ref64, const uint16_t *a,
                    const uint32_t *a_offsets, const uint32_t *packed, const uint16_t *scales,
                    const int32_t *expert_ids, uint32_t *stats, int num_groups, int num_experts,
                    int N, int K, int group_size, int nthreads)
{
    if (K % 8 != 0 || group_size <= 0 || K % group_size != 0) return -2;
    uint32_t active = 0;
    int flags = oracle_validate(a_offsets, expert_ids, num_groups, num_experts, &active);
    if (stats) stats[1] = active;
    if (flags & ORACLE_BAD_OFFSETS) return flags;

    /* Dequantise every expert that an active group uses, once. */
    uint16_t **wq = (uint16_t **)calloc((size_t)(num_experts > 0 ? num_experts : 1), sizeof(uint16_t *));
    if (!wq) return -1;
    int64_t njobs = 0;
    int failed = 0;
    for (int g = 0; g < num_groups && !failed; ++g) {
        int32_t e = expert_ids[g];
        if (e < 0 || e >= num_experts) continue;
        njobs += (int64_t)a_offsets[g + 1] - (int64_t)a_offsets[g];
        if (wq[e]) continue;
        wq[e] = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)N * (size_t)K);
        if (!wq[e]) { failed = 1; break; }
        oracle_dequant_int4(wq[e], packed + (int64_t)e * N * (K / 8),
                            scales + (int64_t)e * N * (K / group_size), N, K, group_size);
    }
    row_job *jobs = failed ? NULL : (row_job *)malloc(sizeof(row_job) * (size_t)(njobs > 0 ? njobs : 1));
    if (jobs) {
        int64_t j = 0;
        for (int g = 0; g < num_groups; ++g) {
            int32_t e = expert_ids[g];
            if (e < 0 || e >= num_experts) continue;
            for (int64_t r = a_offsets[g]; r < (int64_t)a_offsets[g + 1]; ++r) {
                jobs[j].row = r;
                jobs[j].w = wq[e];
                ++j;
            }
        }
        run_jobs(jobs, njobs, a, c, ref32, ref64, N, K, nthreads);
        free(jobs);
    }
    for (int e = 0; e < num_experts; ++e) free(wq[e]);
    free(wq);
    return jobs ? flags : -1;
}
