/*
 * w4a16_oracle.c -- CPU oracle for the weight-only INT4 (W4A16) GEMM.
 *
 * TEST INFRASTRUCTURE.  Only the test-suite, the smoke check and the CPU-baseline leg of the
 * benchmark load this file.  The product (the CUDA library and its Python binding) never
 * calls it and shares no code with it.
 *
 * It is deliberately plain and slow: every quantity is computed from its definition in double
 * precision, from the exact fp16 input values, with loops a reader can check by eye against
 * the pages.  The pages are four docs.rs source listings:
 *   [marlin.rs]      ferrum-kernels 0.8.5 src/backend/cuda/marlin.rs
 *   [vllm_marlin.rs] ferrum-kernels 0.8.4 src/backend/cuda/vllm_marlin.rs
 *   [mmq_ffi.rs]     memra-engine 0.122.0 mmq_ffi.rs
 *   [transformer.rs] ferrum-kernels 0.8.6 src/backend/cuda/vnext_ops/transformer.rs
 *
 * What is computed (the plain definition the method reaches up to rounding):
 *   q[k][n]  = 4-bit code of logical weight row k, column n (GPTQ [K/8, N] int32 words,
 *              row 8r+i at bits 4i..4i+3 -- "low nibble first", the reading the pages imply)
 *   g(k)     = g_idx[k] with act-order, else k / group_size (group_size -1: one group)
 *   zp       = 8 for u4b8, zeros[g(k)][n] for u4
 *   W[k][n]  = (q[k][n] - zp) * scales[g(k)][n]
 *   C[m][n]  = sum_k A[m][k] * W[k][n]
 *
 * Pins: every function here is checked in tests/test_oracle_pins.py against closed forms,
 * brute force, library routines and the worked examples the pages print; none is
 * "parity unpinned".
 */
#ifndef M_PI
#define M_PI 3.14159265358979323846
#endif
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_U4 4   /* [vllm_marlin.rs] FERRUM_MARLIN_SCALAR_U4: codes with a zero point  */
#define ORC_U4B8 5 /* [vllm_marlin.rs] FERRUM_MARLIN_SCALAR_U4B8: codes with bias 8     */

/* ---------------------------------------------------------------------------------------
 * IEEE 754 binary16 -> double, from the format's definition (1 sign bit, 5 exponent bits
 * with bias 15, 10 fraction bits; exponent 0 = subnormal, exponent 31 = inf/NaN).
 * ------------------------------------------------------------------------------------- */
double orc_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1F;
    int frac = h & 0x3FF;
    double v;
    if (expo == 0)
        v = ldexp((double)frac, -24);                 /* 0.frac * 2^-14 */
    else if (expo == 31)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp(1.0 + frac / 1024.0, expo - 15);
    return sign ? -v : v;
}

/* bfloat16 -> double, from the format's definition: the top half of an IEEE binary32 (1 sign
 * bit, 8 exponent bits with bias 127, 7 fraction bits; exponent 0 = subnormal, 255 = inf/NaN).
 * The BF16-activation GEMM reads its activations, scales and zeros this way. */
double orc_bf16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 7) & 0xFF;
    int frac = h & 0x7F;
    double v;
    if (expo == 0)
        v = ldexp((double)frac, -133);                /* 0.frac * 2^-126 */
    else if (expo == 255)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp(1.0 + frac / 128.0, expo - 127);
    return sign ? -v : v;
}

/* A 16-bit input value: binary16, or bfloat16 when `bf16` is set. */
static double orc_h16(uint16_t h, int bf16)
{
    return bf16 ? orc_bf16_to_double(h) : orc_half_to_double(h);
}

void orc_halves_to_doubles(const uint16_t *h, long count, double *out)
{
    for (long i = 0; i < count; ++i)
        out[i] = orc_half_to_double(h[i]);
}

/* ---------------------------------------------------------------------------------------
 * GPTQ logical layout.  [vllm_marlin.rs] `load_stacked_gptq_vllm_marlin` doc: qweight is
 * `[K/8, N]` i32; eight K-consecutive codes share one word.  Within the word the pages never
 * print the INT4 order; the zero-point packer there (`repack_gptq_qzeros_to_marlin`) puts
 * lane i at bits 4*i, and we read the weight words the same way (low nibble first).
 * ------------------------------------------------------------------------------------- */
static int orc_code(const int32_t *qweight, int n, int row, int col)
{
    uint32_t word = (uint32_t)qweight[(long)(row / 8) * n + col];
    return (int)((word >> (4 * (row % 8))) & 0xFu);
}

void orc_unpack_gptq(const int32_t *qweight, int k, int n, uint8_t *codes)
{
    for (int row = 0; row < k; ++row)
        for (int col = 0; col < n; ++col)
            codes[(long)row * n + col] = (uint8_t)orc_code(qweight, n, row, col);
}

void orc_pack_gptq(const uint8_t *codes, int k, int n, int32_t *qweight)
{
    for (int r = 0; r < k / 8; ++r)
        for (int col = 0; col < n; ++col) {
            uint32_t word = 0;
            for (int i = 0; i < 8; ++i)
                word |= (uint32_t)(codes[(long)(8 * r + i) * n + col] & 0xF) << (4 * i);
            qweight[(long)r * n + col] = (int32_t)word;
        }
}

/* ---------------------------------------------------------------------------------------
 * Group count.  [transformer.rs] `marlin_num_groups`: group_size -1 = one channelwise group;
 * otherwise a positive size that divides K.  Returns the count, or -1 on a rejected pair.
 * [marlin.rs] `validate` of the Marlin-MoE launch adds that a positive size is a multiple
 * of 16; we keep that rule as well.
 * ------------------------------------------------------------------------------------- */
int orc_group_count(int k, int group_size)
{
    if (k <= 0)
        return -1;
    if (group_size == -1)
        return 1;
    if (group_size <= 0 || group_size % 16 != 0 || k % group_size != 0)
        return -1;
    return k / group_size;
}

/* Group of logical row k.  [marlin.rs] `MarlinWeight` doc: with act-order (desc_act) each
 * row carries its own group in g_idx; otherwise rows g*group_size .. are group g. */
static int orc_group_of(int row, int k, int group_size, const int32_t *g_idx)
{
    if (g_idx)
        return g_idx[row];
    if (group_size == -1)
        return 0;
    (void)k;
    return row / group_size;
}

/* Dequantised weight W[k][n] = (q - zp) * s.  [vllm_marlin.rs] scalar ids U4 / U4B8;
 * [marlin.rs] `ferrum_vllm_marlin_moe_f16`: has_zp = 0 is the symmetric U4B8 code (zero 8),
 * has_zp = 1 carries explicit zero points.  (q - zp) is exact; the product is exact in
 * double as both factors have at most 11 significant bits. */
static double orc_weight(const int32_t *qweight, const uint16_t *scales, const uint16_t *zeros,
                         const int32_t *g_idx, int k, int n, int group_size, int weight_type,
                         int row, int col, int bf16)
{
    int g = orc_group_of(row, k, group_size, g_idx);
    double s = orc_h16(scales[(long)g * n + col], bf16);
    double zp = (weight_type == ORC_U4B8) ? 8.0 : orc_h16(zeros[(long)g * n + col], bf16);
    double q = (double)orc_code(qweight, n, row, col);
    return (q - zp) * s;
}

/* Materialised dequantised matrix W [K][N] in double. */
void orc_dequant(const int32_t *qweight, const uint16_t *scales, const uint16_t *zeros,
                 const int32_t *g_idx, int k, int n, int group_size, int weight_type, double *w)
{
    for (int row = 0; row < k; ++row)
        for (int col = 0; col < n; ++col)
            w[(long)row * n + col] = orc_weight(qweight, scales, zeros, g_idx, k, n, group_size,
                                                weight_type, row, col, 0);
}

/* Plain triple loop C = A * W over double matrices (A [M][K] with row stride lda). */
void orc_matmul(const double *a, long lda, const double *w, int m, int k, int n, double *c)
{
    for (int i = 0; i < m; ++i)
        for (int j = 0; j < n; ++j) {
            double acc = 0.0;
            for (int kk = 0; kk < k; ++kk)
                acc += a[(long)i * lda + kk] * w[(long)kk * n + j];
            c[(long)i * n + j] = acc;
        }
}

/* ---------------------------------------------------------------------------------------
 * The W4A16 GEMM.  [marlin.rs] `marlin_gemm` doc: C[m, n] = A[m, k] @ dequant(B[k, n]).
 * A is fp16 [M][lda], C is returned in double [M][N].  Columns are split across threads;
 * each output is one plain k-ordered sum of A[m][k] * W[k][n], with W from its definition.
 * W does not depend on the row of A, so a thread writes out the W entries of a band of its
 * columns once (every entry by `orc_weight`) and then forms the sums of every row of A over
 * that band; each sum is the same k-ordered double sum of the same products as when W is
 * re-derived for every row.
 * ------------------------------------------------------------------------------------- */
#define ORC_BAND 256 /* columns of W held at a time by one thread */

struct orc_gemm_job {
    const uint16_t *a; long lda; int m;
    const int32_t *qweight; const uint16_t *scales; const uint16_t *zeros; const int32_t *g_idx;
    int k, n, group_size, weight_type;
    double *c;
    int col_begin, col_end;
    int bf16; /* A, scales and zeros are bfloat16 (else binary16) */
};

static void *orc_gemm_worker(void *arg)
{
    struct orc_gemm_job *jb = (struct orc_gemm_job *)arg;
    if (jb->col_end <= jb->col_begin)
        return NULL;
    double *w = (double *)malloc(sizeof(double) * (size_t)jb->k * ORC_BAND);
    double *acc = (double *)malloc(sizeof(double) * ORC_BAND);
    for (int c0 = jb->col_begin; c0 < jb->col_end; c0 += ORC_BAND) {
        int width = jb->col_end - c0 < ORC_BAND ? jb->col_end - c0 : ORC_BAND;
        for (int row = 0; row < jb->k; ++row)
            for (int j = 0; j < width; ++j)
                w[(long)row * width + j] = orc_weight(jb->qweight, jb->scales, jb->zeros, jb->g_idx,
                                                      jb->k, jb->n, jb->group_size,
                                                      jb->weight_type, row, c0 + j, jb->bf16);
        for (int i = 0; i < jb->m; ++i) {
            for (int j = 0; j < width; ++j)
                acc[j] = 0.0;
            for (int row = 0; row < jb->k; ++row) {
                double av = orc_h16(jb->a[(long)i * jb->lda + row], jb->bf16);
                const double *wr = w + (long)row * width;
                for (int j = 0; j < width; ++j)
                    acc[j] += av * wr[j];
            }
            for (int j = 0; j < width; ++j)
                jb->c[(long)i * jb->n + c0 + j] = acc[j];
        }
    }
    free(acc);
    free(w);
    return NULL;
}

static void orc_gemm_fmt(const uint16_t *a, long lda, int m, const int32_t *qweight,
                         const uint16_t *scales, const uint16_t *zeros, const int32_t *g_idx, int k,
                         int n, int group_size, int weight_type, double *c, int nthreads, int bf16);

void orc_gemm(const uint16_t *a, long lda, int m, const int32_t *qweight, const uint16_t *scales,
              const uint16_t *zeros, const int32_t *g_idx, int k, int n, int group_size,
              int weight_type, double *c, int nthreads)
{
    orc_gemm_fmt(a, lda, m, qweight, scales, zeros, g_idx, k, n, group_size, weight_type, c,
                 nthreads, 0);
}

/* The same GEMM with bfloat16 activations, scales and zeros (BF16 activations). */
void orc_gemm_bf16(const uint16_t *a, long lda, int m, const int32_t *qweight,
                   const uint16_t *scales, const uint16_t *zeros, const int32_t *g_idx, int k,
                   int n, int group_size, int weight_type, double *c, int nthreads)
{
    orc_gemm_fmt(a, lda, m, qweight, scales, zeros, g_idx, k, n, group_size, weight_type, c,
                 nthreads, 1);
}

static void orc_gemm_fmt(const uint16_t *a, long lda, int m, const int32_t *qweight,
                         const uint16_t *scales, const uint16_t *zeros, const int32_t *g_idx, int k,
                         int n, int group_size, int weight_type, double *c, int nthreads, int bf16)
{
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > n)
        nthreads = n;
    if (nthreads > 256)
        nthreads = 256;
    pthread_t tid[256];
    struct orc_gemm_job jobs[256];
    for (int t = 0; t < nthreads; ++t) {
        struct orc_gemm_job jb = {a, lda, m, qweight, scales, zeros, g_idx, k, n, group_size,
                                  weight_type, c, (int)((long)n * t / nthreads),
                                  (int)((long)n * (t + 1) / nthreads), bf16};
        jobs[t] = jb;
    }
    for (int t = 1; t < nthreads; ++t)
        pthread_create(&tid[t], NULL, orc_gemm_worker, &jobs[t]);
    orc_gemm_worker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t)
        pthread_join(tid[t], NULL);
}

/* A second formulation of the same GEMM, used only to cross-check the first: collect, per
 * group g, the exact sums T_g[m][n] = sum_{k in g} (q - zp) * A[m][k], then
 * C = sum_g s_g[n] * T_g.  It differs from `orc_gemm` only by fp64 rounding. */
void orc_gemm_by_groups(const uint16_t *a, long lda, int m, const int32_t *qweight,
                        const uint16_t *scales, const uint16_t *zeros, const int32_t *g_idx,
                        int k, int n, int group_size, int weight_type, int num_groups, double *c)
{
    double *t = (double *)malloc(sizeof(double) * (size_t)n);
    for (int i = 0; i < m; ++i) {
        for (int j = 0; j < n; ++j)
            c[(long)i * n + j] = 0.0;
        for (int g = 0; g < num_groups; ++g) {
            for (int j = 0; j < n; ++j)
                t[j] = 0.0;
            for (int row = 0; row < k; ++row) {
                if (orc_group_of(row, k, group_size, g_idx) != g)
                    continue;
                double av = orc_half_to_double(a[(long)i * lda + row]);
                for (int j = 0; j < n; ++j) {
                    double zp = (weight_type == ORC_U4B8)
                                    ? 8.0 : orc_half_to_double(zeros[(long)g * n + j]);
                    t[j] += ((double)orc_code(qweight, n, row, j) - zp) * av;
                }
            }
            for (int j = 0; j < n; ++j)
                c[(long)i * n + j] += orc_half_to_double(scales[(long)g * n + j]) * t[j];
        }
    }
    free(t);
}

/* ---------------------------------------------------------------------------------------
 * The library's packed tile layout, written out as nested loops from its definition (the
 * layout is this project's own; the pages say only that the kernel layout is a permutation
 * of the GPTQ words with the same byte count -- [marlin.rs] module doc, [vllm_marlin.rs]
 * `ferrum_vllm_gptq_marlin_repack` doc).
 *
 * Definition.  Rows are taken in "sorted" order: sorted row r is logical row perm[r] when a
 * permutation is given ([marlin.rs] `MarlinWeight::perm`: qweight rows permuted by
 * argsort(g_idx)), else row r.  The K x N code matrix is cut into tiles of 64 sorted rows x
 * 128 columns; tile (column tile nt, row block kb) is 1024 consecutive words starting at
 * word (nt * K/64 + kb) * 1024.  Inside a tile, word (h, c, j) for h in {0,1},
 * c in [0,128), j in [0,4) sits at h*512 + c*4 + j and holds 8 codes of column nt*128 + c:
 * for p in 0..3 and e in 0..1, the code of sorted row kb*64 + h*32 + 2*j + 8*p + e sits at
 * bit 4*p + 16*e.
 * ------------------------------------------------------------------------------------- */
void orc_repack_tiles(const int32_t *qweight, const int32_t *perm, int k, int n, int32_t *out)
{
    int kblocks = k / 64, ntiles = n / 128;
    for (int nt = 0; nt < ntiles; ++nt)
        for (int kb = 0; kb < kblocks; ++kb) {
            long base = ((long)nt * kblocks + kb) * 1024;
            for (int h = 0; h < 2; ++h)
                for (int c = 0; c < 128; ++c)
                    for (int j = 0; j < 4; ++j) {
                        uint32_t word = 0;
                        for (int p = 0; p < 4; ++p)
                            for (int e = 0; e < 2; ++e) {
                                int sorted_row = kb * 64 + h * 32 + 2 * j + 8 * p + e;
                                int row = perm ? perm[sorted_row] : sorted_row;
                                uint32_t code = (uint32_t)orc_code(qweight, n, row, nt * 128 + c);
                                word |= code << (4 * p + 16 * e);
                            }
                        out[base + h * 512 + c * 4 + j] = (int32_t)word;
                    }
        }
}

/* Inverse of `orc_repack_tiles` (without undoing a permutation): GPTQ words of sorted rows. */
void orc_unpack_tiles(const int32_t *tiles, int k, int n, int32_t *qweight)
{
    int kblocks = k / 64, ntiles = n / 128;
    memset(qweight, 0, sizeof(int32_t) * (size_t)(k / 8) * (size_t)n);
    for (int nt = 0; nt < ntiles; ++nt)
        for (int kb = 0; kb < kblocks; ++kb) {
            long base = ((long)nt * kblocks + kb) * 1024;
            for (int h = 0; h < 2; ++h)
                for (int c = 0; c < 128; ++c)
                    for (int j = 0; j < 4; ++j) {
                        uint32_t word = (uint32_t)tiles[base + h * 512 + c * 4 + j];
                        for (int p = 0; p < 4; ++p)
                            for (int e = 0; e < 2; ++e) {
                                int row = kb * 64 + h * 32 + 2 * j + 8 * p + e;
                                uint32_t code = (word >> (4 * p + 16 * e)) & 0xFu;
                                long at = (long)(row / 8) * n + nt * 128 + c;
                                qweight[at] = (int32_t)((uint32_t)qweight[at] | (code << (4 * (row % 8))));
                            }
                    }
        }
}

/* ---------------------------------------------------------------------------------------
 * Expert-major CSR schedule.  [mmq_ffi.rs] `ExpertCsr::from_pair_rows`: count routes per
 * expert, prefix-sum, list active experts in increasing order with their segment offsets,
 * and place every pair id into its expert's segment in pair order.  Rejections follow the
 * same function and `from_parts`.  Returns the number of active experts, or -1.
 * ------------------------------------------------------------------------------------- */
int orc_csr_from_pair_rows(int n_expert, int n_tokens, int n_pairs, const int32_t *selected,
                           const int32_t *pair_tok, int32_t *ex_ids, int32_t *ex_off,
                           int32_t *ex_pairs, int32_t *pair_tok_out)
{
    if (n_expert <= 0 || n_tokens <= 0 || n_pairs <= 0)
        return -1;
    long *count = (long *)calloc((size_t)n_expert, sizeof(long));
    long *cursor = (long *)calloc((size_t)n_expert + 1, sizeof(long));
    int active = -1;
    for (int p = 0; p < n_pairs; ++p) {
        if (selected[p] < 0 || selected[p] >= n_expert)
            goto done;
        count[selected[p]]++;
    }
    for (int p = 0; p < n_pairs; ++p)
        if (pair_tok[p] < 0 || pair_tok[p] >= n_tokens)
            goto done;
    for (int e = 0; e < n_expert; ++e)
        cursor[e + 1] = cursor[e] + count[e];
    active = 0;
    for (int e = 0; e < n_expert; ++e)
        if (count[e]) {
            ex_ids[active] = e;
            ex_off[active] = (int32_t)cursor[e];
            ++active;
        }
    ex_off[active] = n_pairs;
    for (int p = 0; p < n_pairs; ++p)
        ex_pairs[cursor[selected[p]]++] = p;
    for (int p = 0; p < n_pairs; ++p)
        pair_tok_out[p] = pair_tok[p];
done:
    free(count);
    free(cursor);
    return active;
}

/* [mmq_ffi.rs] `ExpertCsr::from_token_routes`: token-major routes, pair p reads token
 * p / experts_per_token. */
int orc_csr_from_token_routes(int n_expert, int n_tokens, int experts_per_token,
                              const int32_t *selected, int n_selected, int32_t *ex_ids,
                              int32_t *ex_off, int32_t *ex_pairs, int32_t *pair_tok_out)
{
    if (experts_per_token <= 0 || (long)n_tokens * experts_per_token != n_selected)
        return -1;
    int32_t *rows = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n_selected > 0 ? n_selected : 1));
    for (int p = 0; p < n_selected; ++p)
        rows[p] = p / experts_per_token;
    int r = orc_csr_from_pair_rows(n_expert, n_tokens, n_selected, selected, rows, ex_ids, ex_off,
                                   ex_pairs, pair_tok_out);
    free(rows);
    return r;
}

/* [mmq_ffi.rs] `ExpertCsr::from_parts` checks: offsets start at 0 and end at n_pairs with
 * non-empty increasing segments, expert ids strictly increasing and in range, every pair id
 * exactly once, every activation row in range.  Returns 0 when valid, else -1. */
int orc_csr_validate(int n_expert, int n_tokens, int n_active, int n_pairs, const int32_t *ex_ids,
                     const int32_t *ex_off, const int32_t *ex_pairs, const int32_t *pair_tok)
{
    if (n_expert <= 0 || n_tokens <= 0 || n_active <= 0 || n_pairs <= 0)
        return -1;
    if (ex_off[0] != 0 || ex_off[n_active] != n_pairs)
        return -1;
    for (int i = 0; i + 1 < n_active; ++i)
        if (ex_ids[i] >= ex_ids[i + 1])
            return -1;
    for (int i = 0; i < n_active; ++i) {
        if (ex_ids[i] < 0 || ex_ids[i] >= n_expert)
            return -1;
        if (ex_off[i] >= ex_off[i + 1])
            return -1;
    }
    char *seen = (char *)calloc((size_t)n_pairs, 1);
    int ok = 0;
    for (int r = 0; r < n_pairs; ++r) {
        int p = ex_pairs[r];
        if (p < 0 || p >= n_pairs || seen[p] || pair_tok[p] < 0 || pair_tok[p] >= n_tokens) {
            ok = -1;
            break;
        }
        seen[p] = 1;
    }
    free(seen);
    return ok;
}

/* ---------------------------------------------------------------------------------------
 * Grouped (MoE) GEMM over the CSR schedule.  [mmq_ffi.rs] expert-segmented entry points:
 * pairs are grouped by expert, pair_tok gathers the activation row, and the output is
 * pair-major: Y[pair][:] = A[pair_tok[pair]][:] @ dequant(B_expert).  No routing weight is
 * applied.  Weights are stacked per expert: the GPTQ words of expert e start at
 * e*(K/8)*N, its scales/zeros at e*G*N.
 * ------------------------------------------------------------------------------------- */
void orc_grouped(const uint16_t *a, long lda, const int32_t *qweight_stack,
                 const uint16_t *scales_stack, const uint16_t *zeros_stack, const int32_t *ex_ids,
                 const int32_t *ex_off, const int32_t *ex_pairs, const int32_t *pair_tok,
                 int n_active, int k, int n, int group_size, int weight_type, double *y,
                 int nthreads)
{
    int groups = orc_group_count(k, group_size);
    long words_per_expert = (long)(k / 8) * n;
    long scales_per_expert = (long)groups * n;
    for (int i = 0; i < n_active; ++i) {
        int e = ex_ids[i];
        int rows = ex_off[i + 1] - ex_off[i];
        if (rows <= 0)
            continue;
        const int32_t *qw = qweight_stack + (long)e * words_per_expert;
        const uint16_t *sc = scales_stack + (long)e * scales_per_expert;
        const uint16_t *zp = zeros_stack ? zeros_stack + (long)e * scales_per_expert : NULL;
        /* The segment's activation rows, in segment order, then one GEMM with this expert's
         * weights; row r of its result is pair ex_pairs[ex_off[i] + r]. */
        uint16_t *a_seg = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)rows * k);
        double *y_seg = (double *)malloc(sizeof(double) * (size_t)rows * n);
        for (int r = 0; r < rows; ++r) {
            int pair = ex_pairs[ex_off[i] + r];
            memcpy(a_seg + (long)r * k, a + (long)pair_tok[pair] * lda, sizeof(uint16_t) * (size_t)k);
        }
        orc_gemm(a_seg, k, rows, qw, sc, zp, NULL, k, n, group_size, weight_type, y_seg, nthreads);
        for (int r = 0; r < rows; ++r) {
            int pair = ex_pairs[ex_off[i] + r];
            memcpy(y + (long)pair * n, y_seg + (long)r * n, sizeof(double) * (size_t)n);
        }
        free(a_seg);
        free(y_seg);
    }
}

/* ---------------------------------------------------------------------------------------
 * FP8 E4M3 weights (W8A16).  [vllm_marlin.rs] scalar id FERRUM_MARLIN_SCALAR_FE4M3FN and
 * `vllm_fp8_marlin_repack_raw_bits`: the weights arrive as [K/4, N] 32-bit words, each holding
 * four consecutive K-axis E4M3 bytes of one output column, little-endian (row 4r+i at byte i
 * of word (r, n)); [marlin.rs] Marlin-MoE validation: E4M3 takes group_size -1 or 128 and no
 * zero points.  W[k][n] = e4m3(code) * scales[g(k)][n].
 *
 * E4M3 ("fn" variant) from its definition: 1 sign bit, 4 exponent bits with bias 7, 3 fraction
 * bits; exponent 0 is subnormal (fraction/8 * 2^-6); exponent 15 with fraction 7 is NaN, and
 * there are no infinities (exponent 15 with fraction 0..6 is an ordinary value up to 448).
 * ------------------------------------------------------------------------------------- */
double orc_e4m3_to_double(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int expo = (code >> 3) & 0xF;
    int frac = code & 0x7;
    double v;
    if (expo == 15 && frac == 7)
        return NAN;
    if (expo == 0)
        v = ldexp((double)frac / 8.0, -6);
    else
        v = ldexp(1.0 + frac / 8.0, expo - 7);
    return sign ? -v : v;
}

static int orc_fp8_code(const int32_t *qweight, int n, int row, int col)
{
    uint32_t word = (uint32_t)qweight[(long)(row / 4) * n + col];
    return (int)((word >> (8 * (row % 4))) & 0xFFu);
}

/* Dequantised FP8 matrix W [K][N] in double. */
void orc_dequant_fp8(const int32_t *qweight, const uint16_t *scales, int k, int n, int group_size,
                     double *w)
{
    for (int row = 0; row < k; ++row) {
        int g = group_size == -1 ? 0 : row / group_size;
        for (int col = 0; col < n; ++col)
            w[(long)row * n + col] = orc_e4m3_to_double((uint8_t)orc_fp8_code(qweight, n, row, col)) *
                                     orc_half_to_double(scales[(long)g * n + col]);
    }
}

/* C = A W with the FP8 weights: W derived once, then the plain k-ordered double sums (one
 * thread per band of columns, as orc_gemm). */
struct orc_fp8_job {
    const uint16_t *a; long lda; int m; const double *w; int k, n; double *c; int c0, c1;
};

static void *orc_fp8_worker(void *arg)
{
    struct orc_fp8_job *jb = (struct orc_fp8_job *)arg;
    int width = jb->c1 - jb->c0;
    if (width <= 0)
        return NULL;
    double *acc = (double *)malloc(sizeof(double) * (size_t)width);
    for (int i = 0; i < jb->m; ++i) {
        for (int j = 0; j < width; ++j)
            acc[j] = 0.0;
        /* Row by row of W, so that the band's entries are read in memory order; every output
         * is still the k-ordered sum of its products. */
        for (int row = 0; row < jb->k; ++row) {
            double a_ik = orc_half_to_double(jb->a[(long)i * jb->lda + row]);
            const double *wrow = jb->w + (long)row * jb->n + jb->c0;
            for (int j = 0; j < width; ++j)
                acc[j] += a_ik * wrow[j];
        }
        for (int j = 0; j < width; ++j)
            jb->c[(long)i * jb->n + jb->c0 + j] = acc[j];
    }
    free(acc);
    return NULL;
}

void orc_gemm_fp8(const uint16_t *a, long lda, int m, const int32_t *qweight, const uint16_t *scales,
                  int k, int n, int group_size, double *c, int nthreads)
{
    double *w = (double *)malloc(sizeof(double) * (size_t)k * (size_t)n);
    orc_dequant_fp8(qweight, scales, k, n, group_size, w);
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > n)
        nthreads = n;
    if (nthreads > 256)
        nthreads = 256;
    pthread_t tid[256];
    struct orc_fp8_job jobs[256];
    for (int t = 0; t < nthreads; ++t) {
        struct orc_fp8_job jb = {a, lda, m, w, k, n, c, (int)((long)n * t / nthreads),
                                 (int)((long)n * (t + 1) / nthreads)};
        jobs[t] = jb;
    }
    for (int t = 1; t < nthreads; ++t)
        pthread_create(&tid[t], NULL, orc_fp8_worker, &jobs[t]);
    orc_fp8_worker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t)
        pthread_join(tid[t], NULL);
    free(w);
}

/* The library's FP8 tile layout, from its definition (the pages' own FP8 Marlin tiles are
 * another layout; this one is this project's).  Tile (nt, kb): rows kb*64 .. kb*64+63, columns
 * nt*128 .. nt*128+127, 2048 words at word (nt * K/64 + kb) * 2048.  Word (q, c, t) at
 * q*512 + c*4 + t, q and t in 0..3, c in 0..127, holds rows kb*64 + 16q + 4t + i of column
 * nt*128 + c at byte i (i in 0..3). */
void orc_repack_fp8_tiles(const int32_t *qweight, int k, int n, int32_t *out)
{
    int kblocks = k / 64, ntiles = n / 128;
    for (int nt = 0; nt < ntiles; ++nt)
        for (int kb = 0; kb < kblocks; ++kb) {
            long base = ((long)nt * kblocks + kb) * 2048;
            for (int q = 0; q < 4; ++q)
                for (int c = 0; c < 128; ++c)
                    for (int t = 0; t < 4; ++t) {
                        uint32_t word = 0;
                        for (int i = 0; i < 4; ++i) {
                            int row = kb * 64 + 16 * q + 4 * t + i;
                            word |= (uint32_t)orc_fp8_code(qweight, n, row, nt * 128 + c) << (8 * i);
                        }
                        out[base + q * 512 + c * 4 + t] = (int32_t)word;
                    }
        }
}

/* ---------------------------------------------------------------------------------------
 * The vLLM Marlin-MoE routing.  [marlin.rs] `ferrum_vllm_marlin_moe_f16` declaration and
 * `marlin_gemm_moe_vllm` doc: the caller first runs `moe_align_block_size`, which lists, for
 * each expert in turn, the flattened (token, slot) ids routed to it -- id = token * top_k + slot
 * -- padded to a multiple of moe_block_size with the sentinel prob_m * top_k; expert_ids gives
 * the expert of every block of moe_block_size rows and num_tokens_past_padded the padded
 * length.  The launch then computes, for every non-sentinel row r of block b,
 *     c[id][:] = A[id / top_k][:] @ dequant(B_{expert_ids[b]})  (times topk_weights[id] when
 *     mul_topk_weights is set),
 * and leaves c's other rows alone; with is_ep, a block whose expert id is -1 (an expert another
 * rank holds) is skipped.  The page test that runs it puts a batch's tokens in the prefix of
 * one block and fills the rest with the sentinel.
 *
 * moe_align_block_size as read here: experts in increasing order; inside an expert its ids in
 * increasing order; experts with no ids get no block.  Writes at most `capacity` entries;
 * returns num_tokens_past_padded, or -1 on an expert id out of range or a too small capacity.
 * ------------------------------------------------------------------------------------- */
int orc_moe_align_block_size(const int32_t *topk_ids, int m, int top_k, int n_experts,
                             int block_size, int capacity, int32_t *sorted_ids,
                             int32_t *expert_ids)
{
    int n_ids = m * top_k;
    for (int i = 0; i < n_ids; ++i)
        if (topk_ids[i] < 0 || topk_ids[i] >= n_experts)
            return -1;
    int len = 0;
    for (int e = 0; e < n_experts; ++e) {
        int count = 0;
        for (int i = 0; i < n_ids; ++i)
            if (topk_ids[i] == e) {
                if (len + count >= capacity)
                    return -1;
                sorted_ids[len + count] = i;
                ++count;
            }
        if (count == 0)
            continue;
        int padded = (count + block_size - 1) / block_size * block_size;
        if (len + padded > capacity)
            return -1;
        for (int r = count; r < padded; ++r)
            sorted_ids[len + r] = n_ids; /* the sentinel */
        for (int b = 0; b < padded / block_size; ++b)
            expert_ids[len / block_size + b] = e;
        len += padded;
    }
    return len;
}

/* The launch's result in double: c [m * top_k][n], rows that no non-sentinel entry names are
 * not written.  Returns 0, or -1 on an expert id out of range (or -1 without is_ep). */
int orc_moe_blocks(const uint16_t *a, long lda, const int32_t *qweight_stack,
                   const uint16_t *scales_stack, const uint16_t *zeros_stack,
                   const int32_t *sorted_ids, const int32_t *expert_ids, int padded,
                   const float *topk_weights, int block_size, int top_k, int is_ep,
                   int n_experts, int m, int k, int n, int group_size, int weight_type, double *c,
                   int nthreads)
{
    int groups = orc_group_count(k, group_size);
    long words_per_expert = (long)(k / 8) * n;
    long scales_per_expert = (long)groups * n;
    double *row = (double *)malloc(sizeof(double) * (size_t)n);
    for (int b = 0; b < padded / block_size; ++b) {
        int e = expert_ids[b];
        if (e == -1 && is_ep)
            continue;
        if (e < 0 || e >= n_experts) {
            free(row);
            return -1;
        }
        for (int r = b * block_size; r < (b + 1) * block_size; ++r) {
            int id = sorted_ids[r];
            if (id < 0 || id >= m * top_k)
                continue; /* sentinel (or padding beyond the ids) */
            orc_gemm(a + (long)(id / top_k) * lda, lda, 1, qweight_stack + (long)e * words_per_expert,
                     scales_stack + (long)e * scales_per_expert,
                     zeros_stack ? zeros_stack + (long)e * scales_per_expert : NULL, NULL, k, n,
                     group_size, weight_type, row, nthreads);
            double w = topk_weights ? (double)topk_weights[id] : 1.0;
            for (int j = 0; j < n; ++j)
                c[(long)id * n + j] = row[j] * w;
        }
    }
    free(row);
    return 0;
}

/* ---------------------------------------------------------------------------------------
 * Gated activations after the gate and up projections.  [transformer.rs]
 * `encode_compressed_tensors_dense_swiglu`: gate = A Wg and up = A Wu are two W4A16 GEMMs,
 * then the planar SiLU-multiply (`launch_planar_silu_mul`) gives h = silu(gate) * up, which the
 * down projection consumes; the symmetric U4B8 GeGLU pipeline beside it uses the tanh form of
 * GELU instead.  Textbook definitions, in double:
 *   silu(x)      = x / (1 + exp(-x))                     (x times the logistic sigmoid)
 *   gelu_tanh(x) = x/2 * (1 + tanh(sqrt(2/pi) * (x + 0.044715 x^3)))
 * kind 1 = SiLU, 2 = GELU (tanh form).  h[i] = act(gate[i]) * up[i].
 * ------------------------------------------------------------------------------------- */
double orc_act(double x, int kind)
{
    if (kind == 1)
        return x / (1.0 + exp(-x));
    const double c = sqrt(2.0 / M_PI);
    return 0.5 * x * (1.0 + tanh(c * (x + 0.044715 * x * x * x)));
}

void orc_glu(const double *gate, const double *up, long count, int kind, double *h)
{
    for (long i = 0; i < count; ++i)
        h[i] = orc_act(gate[i], kind) * up[i];
}

/* ---------------------------------------------------------------------------------------
 * AutoGPTQ zero-point words.  [vllm_marlin.rs] `repack_gptq_qzeros_to_marlin`: on-disk
 * qzeros are `[groups, N/8]` words holding `zero - 1` at bits 4*lane; the runtime zero is
 * the stored code + 1, and code 15 is rejected.  This writes the runtime zeros as doubles
 * [groups][N]; returns 0, or -1 on a code 15.
 * `gptq_qzeros_are_symmetric_code7`: every lane of every word is 7 (zero 8).
 * ------------------------------------------------------------------------------------- */
int orc_qzeros_to_zero_points(const int32_t *qzeros, int groups, int n, double *zero_points)
{
    for (int g = 0; g < groups; ++g)
        for (int col = 0; col < n; ++col) {
            uint32_t word = (uint32_t)qzeros[(long)g * (n / 8) + col / 8];
            uint32_t raw = (word >> (4 * (col % 8))) & 0xFu;
            if (raw == 15)
                return -1;
            zero_points[(long)g * n + col] = (double)raw + 1.0;
        }
    return 0;
}

int orc_qzeros_symmetric_code7(const int32_t *qzeros, long count)
{
    if (count <= 0)
        return 0;
    for (long i = 0; i < count; ++i)
        for (int lane = 0; lane < 8; ++lane)
            if ((((uint32_t)qzeros[i] >> (4 * lane)) & 0xFu) != 7)
                return 0;
    return 1;
}
