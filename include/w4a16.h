/*
 * w4a16.h -- C ABI of the GB300 (sm_103a) weight-only INT4 GEMM library (libw4a16.so).
 *
 * The operation (ferrum-kernels 0.8.5 src/backend/cuda/marlin.rs, doc of `marlin_gemm`):
 *     C[M, N] = A[M, K] (fp16) x dequant(B)[K, N],   fp32 accumulation, fp16 output,
 * where B holds 4-bit codes q with one fp16 scale s per group of `group_size` rows of K:
 *     u4b8:  w = (q - 8) * s                  (ferrum-kernels 0.8.4 vllm_marlin.rs, scalar U4B8)
 *     u4:    w = (q - z) * s, z an fp16 zero  (same page, scalar U4; marlin.rs Marlin-MoE `has_zp`)
 * with an optional act-order permutation (marlin.rs, `MarlinWeight::perm`: rows of B are
 * permuted by argsort(g_idx) at load time and the columns of A are gathered by the same
 * permutation at run time).
 *
 * Conventions shared by every entry point
 *   - Pointers named "device" must be CUDA device (or managed) memory; "host" ones host memory.
 *   - fp16 buffers are IEEE binary16, passed as `void*`.
 *   - All matrices are row-major.  The caller owns every allocation and keeps it alive until
 *     the work enqueued on `stream` has finished (marlin.rs, Marlin-MoE raw launch arguments).
 *   - Calls are asynchronous on `stream` and never synchronise, allocate, or fall back to the
 *     CPU.  The stream may be a capturing stream (CUDA graphs).
 *   - Return value: 0 on success, else a staged status `(stage << 16) | detail`, after the
 *     convention of marlin.rs (`marlin_moe_ffi_status`):
 *       stage 1  invalid argument      detail = W4A16_ARG_*
 *       stage 2  unsupported shape     detail = W4A16_ARG_*
 *       stage 3  device query/resource detail = cudaError_t
 *       stage 6  kernel launch         detail = cudaError_t
 *       stage 7  device-side error     detail = W4A16_DEV_* bits (read with w4a16_status)
 *     Argument checks run before any CUDA call, so they work on a machine without a GPU.
 */
#ifndef W4A16_H
#define W4A16_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define W4A16_ABI_VERSION 1

/* Weight types: the scalar ids of ferrum-kernels 0.8.4 vllm_marlin.rs (FERRUM_MARLIN_SCALAR_*). */
#define W4A16_TYPE_U4 4   /* codes with an explicit fp16 zero point per (group, column) */
#define W4A16_TYPE_U4B8 5 /* symmetric codes, zero point 8                              */
#define W4A16_TYPE_FE4M3 8 /* 8-bit FP8 E4M3 ("fn") weights, W8A16: w = e4m3(code) * s,
                              no zero points (scalar FERRUM_MARLIN_SCALAR_FE4M3FN)      */

/* Flags.  Bits 1..3 keep the positions of the page's FERRUM_MARLIN_HAS_ACT_ORDER,
 * FERRUM_MARLIN_IS_K_FULL and FERRUM_MARLIN_HAS_ZERO_POINTS (vllm_marlin.rs). */
#define W4A16_FLAG_ACT_ORDER (1u << 1)  /* g_idx and perm given; A is gathered by perm       */
#define W4A16_FLAG_IS_K_FULL (1u << 2)  /* this call sees the whole K (always true here)     */
#define W4A16_FLAG_HAS_ZP (1u << 3)     /* zeros given; required exactly for W4A16_TYPE_U4   */
#define W4A16_FLAG_FORCE_SIMT (1u << 8) /* run the CUDA-core reference kernel (diagnostics)  */
#define W4A16_FLAG_A_SMEM (1u << 9)     /* stage dequantised weights in shared memory instead
                                           of tensor memory (diagnostics / comparison)       */
#define W4A16_FLAG_FORCE_TC (1u << 10)  /* always use the tcgen05 kernel (diagnostics)      */
#define W4A16_FLAG_FORCE_MMA (1u << 11) /* always use the small-M split-K register-fragment
                                           kernel; M above 64 is then rejected
                                           (unsupported-shape)                               */
#define W4A16_FLAG_STATIC_WEIGHTS (1u << 12) /* b_packed, scales and zeros are not written by the
                                           work that precedes this call on its stream, so the
                                           kernel may start reading them before that work has
                                           finished (it still waits before reading A or
                                           writing C or the workspace).  Without the flag
                                           weights are only prefetched into L2 early.        */
#define W4A16_FLAG_FORCE_SLICE (1u << 13) /* always use the small-M column-slice kernel (each
                                           CTA owns 16-column slices over all of K, no
                                           split-K); M above 32 or a group size that is not
                                           -1 or a multiple of 64 is then rejected
                                           (unsupported-shape)                               */

#define W4A16_FLAG_SWIGLU (1u << 14) /* gated FFN epilogue: the weight's 2I columns are gate
                                           and up projections interleaved by
                                           w4_gate_up_interleave, and C receives
                                           H[M][I] = silu(A Wg) * (A Wu) (ldc >= I) instead of
                                           the product (tcgen05 kernel only: _FORCE_SIMT,
                                           _FORCE_MMA and _FORCE_SLICE are rejected)        */
#define W4A16_FLAG_GEGLU (1u << 15)  /* the same with gelu_tanh(x) = x/2 (1 + tanh(sqrt(2/pi)
                                           (x + 0.044715 x^3))) in place of silu; exclusive
                                           with W4A16_FLAG_SWIGLU.  Both activations are
                                           evaluated in fp32 as x sigmoid(y) (y = x for silu,
                                           2 sqrt(2/pi) (x + 0.044715 x^3) for gelu_tanh)
                                           with a fast exponential: within the gated
                                           tolerance, not correctly rounded               */
#define W4A16_FLAG_BF16 (1u << 16)   /* a, scales, zeros and c are bfloat16 instead of fp16
                                           (marlin.rs declares bf16 A and C for its
                                           `ferrum_vllm_marlin_moe_mxfp4_bf16` entry point;
                                           here with the 4-bit codes).  4-bit weight types
                                           only (not W4A16_TYPE_FE4M3); the tcgen05 kernel and,
                                           for group_size -1 or a multiple of 64, the small-M
                                           kernels (_FORCE_SIMT is rejected, _FORCE_MMA with
                                           other groups is unsupported-shape; the default choice
                                           sends those groups to the tcgen05 kernel).  (q - z)
                                           is exact in bf16 for integer
                                           zero points, the product with the scale is rounded
                                           once to bf16 (8 significant bits), products sum in
                                           fp32 and C is rounded once to bf16               */

/* Detail codes of stage-1/2 statuses. */
#define W4A16_ARG_NULL 1        /* a required pointer is NULL                                  */
#define W4A16_ARG_ALIGN 2       /* a pointer or leading dimension breaks its alignment rule    */
#define W4A16_ARG_SHAPE 3       /* a size is negative, or K % 128 / N % 256 is violated        */
#define W4A16_ARG_FLAGS 4       /* flags disagree with the pointers or the weight type         */
#define W4A16_ARG_OVERFLOW 5    /* an extent does not fit the index types                      */
#define W4A16_ARG_WORKSPACE 6   /* workspace missing or smaller than w4a16_*_workspace_size    */
#define W4A16_ARG_GROUP 7       /* group_size not -1 or a positive multiple of 16 dividing K  */
#define W4A16_ARG_TYPE 8        /* unknown weight type                                         */
#define W4A16_ARG_SCHEDULE 9    /* grouped schedule sizes out of range                         */
#define W4A16_ARG_SCRATCH 10    /* w4a16_gemm_noalloc: the call needs more scratch than it has */
#define W4A16_ARG_QZERO 11      /* a packed GPTQ zero code of 15 (its zero point would be 16)  */

/* Device-side error bits (stage 7), accumulated in the workspace status word. */
#define W4A16_DEV_TIMEOUT 1     /* a bounded wait inside a kernel ran out; the workspace's
                                   split-tile counters may then be left non-zero, so zero-fill
                                   the whole workspace again before its next use             */
#define W4A16_DEV_PERM 2        /* a perm entry was outside [0, K)                             */
#define W4A16_DEV_GIDX 4        /* g_idx[perm[i]] != i / group_size (groups not equal-sized)   */
#define W4A16_DEV_SCHEDULE 8    /* a CSR entry was outside its range                           */
#define W4A16_DEV_ZERO 16       /* w4a16_zero_points_check: a zero point is not an integer in
                                   [0, 15]                                                   */

/* ------------------------------------------------------------------------------------------
 * Packed tile layout (this library's own; the pages only say the kernel layout is a
 * permutation of the GPTQ words with the same byte count: marlin.rs module doc,
 * vllm_marlin.rs `ferrum_vllm_gptq_marlin_repack` doc).
 *
 * Input ("GPTQ") layout: int32 [K/8][N]; word (r, n) holds the codes of rows 8r..8r+7 of
 * column n, row 8r+i at bits 4i..4i+3 (low nibble first).
 *
 * Tile layout: K*N/8 int32 words.  "Sorted row" r is logical row perm[r] when a permutation
 * is given, else r.  Tile (nt, kb) covers sorted rows kb*64 .. kb*64+63 and columns
 * nt*128 .. nt*128+127 and occupies the 1024 words starting at (nt * K/64 + kb) * 1024.
 * Word h*512 + c*4 + j of a tile (h in {0,1}, c in [0,128), j in [0,4)) holds eight codes
 * of column nt*128 + c: for p in 0..3 and e in 0..1, the code of sorted row
 * kb*64 + h*32 + 8p + 2j + e sits at bit 4p + 16e.  One mask then turns the row pair
 * (8p + 2j, 8p + 2j + 1) into two fp16 lanes, a word is exactly what one thread of an
 * m16n8k16 register fragment needs for two 16-row k steps, the four words of one
 * (half, column) are one 16-byte load of 32 rows, and each 64x128 tile is one contiguous
 * 4 KiB bulk copy.
 * ---------------------------------------------------------------------------------------- */

/* GPTQ words -> tile layout.
 *   qweight   device int32 [K/8][N], read only
 *   perm      device int32 [K] or NULL; sorted row r takes logical row perm[r]
 *   b_packed  device int32 [K*N/8], written; must not overlap qweight
 *   status    device int32 or NULL; W4A16_DEV_PERM is OR-ed in when a perm entry is out of
 *             range (that row's codes are then written as 0)
 *   k, n      K % 128 == 0, N % 256 == 0 (marlin.rs module doc), both > 0
 * Alignment: qweight, b_packed 16 bytes; perm, status 4 bytes.
 * Source: vllm_marlin.rs `ferrum_vllm_gptq_marlin_repack` (GPTQ -> kernel tiles, has_perm). */
int w4_repack(const int32_t *qweight, const int32_t *perm, int32_t *b_packed, int32_t *status,
              int k, int n, cudaStream_t stream);

/* Gate/up interleave for the gated FFN epilogue (W4A16_FLAG_SWIGLU / _GEGLU).
 * transformer.rs, `encode_compressed_tensors_dense_swiglu` and the U4B8 GeGLU pipeline beside
 * it: gate = A Wg and up = A Wu are two W4A16 GEMMs over the same A, then h = act(gate) * up
 * feeds the down projection.  Here both run as one GEMM over a [K][2I] weight whose columns
 * alternate in blocks of 16 -- destination column 32b + r is gate column 16b + r for r < 16
 * and up column 16b + r - 16 for r >= 16 -- so each 128-column tile of the kernel holds 64
 * features' gate and up sums side by side and its epilogue writes act(gate) * up.
 * This permutes the columns of a row-major [rows][n2] array, n2 = 2I, from the planar order
 * (the I gate columns, then the I up columns) into that order; apply it to the GPTQ words
 * [K/8][2I] (elem_bytes 4) before w4_repack, and to the scales and zeros [G][2I]
 * (elem_bytes 2).  For w4a16_gemm, I must be a multiple of 128 (so 2I % 256 == 0).
 *   src, dst  device arrays of rows x n2 elements, not overlapping, aligned to elem_bytes
 *   n2        a positive multiple of 32;  elem_bytes 2 or 4 */
int w4_gate_up_interleave(const void *src, void *dst, int rows, int n2, int elem_bytes,
                          cudaStream_t stream);

/* FP8 E4M3 weights (W8A16).  Input: int32 [K/4][N], each word holding four K-consecutive E4M3
 * codes of one column, row 4r+i at byte i (little-endian) -- the input ABI of vllm_marlin.rs
 * `vllm_fp8_marlin_repack_raw_bits`; a checkpoint's row-major [N][K] bytes are transposed into
 * it.  Output (this library's FP8 tile layout, K*N/4 words): tile (nt, kb) covers rows
 * kb*64 .. kb*64+63 and columns nt*128 .. nt*128+127 at word (nt * K/64 + kb) * 2048; word
 * q*512 + c*4 + t (q, t in 0..3, c in 0..127) is the input word of rows kb*64 + 16q + 4t .. +3
 * of column nt*128 + c, so each thread of the kernel reads its column's 64 rows as four 16-byte
 * loads.  K % 128 == 0, N % 256 == 0; 16-byte aligned; the buffers must not overlap.
 * W4A16_TYPE_FE4M3 GEMMs (w4a16_gemm, _grouped, _moe_blocks) take these tiles, fp16 scales
 * [G][N] with group_size -1 or a positive multiple of 64 dividing K (the pages' FP8 Marlin
 * takes -1 or 128), no zero points, no act-order, fp16 activations.  They run on the
 * column-slice kernel for M <= 16 with N / 16 >= the SM count (W4A16_FLAG_FORCE_SLICE forces it;
 * M above 16 is then unsupported-shape)
 * and otherwise on the tcgen05 kernel; forcing the split-K small-M or the CUDA-core kernel is
 * rejected (those are 4-bit only).  Each code becomes its exact fp16 value
 * (cvt.rn.f16x2.e4m3x2); the product with the scale is rounded once. */
int w8_repack(const int32_t *qweight, int32_t *b_packed, int k, int n, cudaStream_t stream);

/* FP8 tiles -> the [K/4][N] input words (the inverse of w8_repack). */
int w8_unpack(const int32_t *b_packed, int32_t *qweight, int k, int n, cudaStream_t stream);

/* Tile layout -> GPTQ words of the sorted rows (the inverse of w4_repack; a permutation
 * applied at repack time is not undone).  Same shape, alignment and overlap rules. */
int w4_unpack(const int32_t *b_packed, int32_t *qweight, int k, int n, cudaStream_t stream);

/* Workspace bytes that w4a16_gemm needs for these sizes on a device with `num_sms`
 * multiprocessors (num_sms <= 0: query the current device; returns 0 if that fails or the
 * sizes are invalid).  The workspace holds a status word, the split-K tile counters, the
 * fp32 partial tiles and, with act-order, the gathered copy of A.  It must be zero-filled
 * once after allocation; the kernels leave it ready for the next call (counters reset
 * themselves), so no per-call memset is needed.  The one exception: after w4a16_status has
 * reported W4A16_DEV_TIMEOUT, a CTA that gave up may have left its tile counters part-way, and
 * the next call would then reduce the wrong partials -- zero-fill the whole workspace again
 * (cudaMemsetAsync over its size) before reusing it.  Calls that run concurrently need
 * separate workspaces. */
size_t w4a16_workspace_size(int m, int n, int k, int group_size, unsigned flags, int num_sms);

/* The W4A16 GEMM.
 *   a          device fp16 [M][lda], lda >= K, lda % 8 == 0, 16-byte aligned
 *   b_packed   device int32 tile layout of the [K][N] codes (from w4_repack)
 *   c          device fp16 [M][ldc], ldc >= N, ldc % 8 == 0; written
 *   scales     device fp16 [G][N], G = K / group_size (1 for group_size -1)
 *   zeros      device fp16 [G][N] integer zero points in [0, 15], or NULL (u4b8).  The
 *              kernels form (q - z) exactly by integer arithmetic inside fp16 and do not check
 *              the values: a zero point that is not an integer in [0, 15] gives unspecified
 *              results (w4a16_zero_points_check reports such values)
 *   g_idx      device int32 [K] or NULL: group of each logical row (act-order)
 *   perm       device int32 [K] or NULL: the permutation that w4_repack applied, one that
 *              sorts g_idx (argsort; any order of the rows inside a group is accepted).
 *              Groups must be equal-sized (g_idx[perm[i]] == i/group_size, as GPTQ's desc_act
 *              layout is); a violation sets W4A16_DEV_GIDX.
 *   workspace  device, >= w4a16_workspace_size(...) bytes, 256-byte aligned, zero-filled once
 *   m          >= 0 (0 is a no-op);  n % 256 == 0;  k % 128 == 0
 *   group_size -1 (one group) or a positive multiple of 16 dividing K
 *              (transformer.rs `marlin_num_groups`; marlin.rs Marlin-MoE validation)
 *   weight_type W4A16_TYPE_U4B8 (zeros NULL), W4A16_TYPE_U4 (zeros and W4A16_FLAG_HAS_ZP) or
 *              W4A16_TYPE_FE4M3 (FP8 tiles from w8_repack; zeros NULL, see there)
 *   flags      W4A16_FLAG_*; ACT_ORDER exactly when g_idx and perm are given.  With
 *              W4A16_FLAG_SWIGLU or _GEGLU, N = 2I columns of interleaved gate/up weights
 *              (w4_gate_up_interleave) and c receives H [M][ldc], ldc >= I, with
 *              H[m][f] = act(gate[m][f]) * up[m][f] computed in fp32 from the fp32 sums and
 *              rounded once to fp16
 * Kernel choice (unless a W4A16_FLAG_FORCE_* flag picks one): M <= 8 -- and M <= 32 while
 * N / 16 <= 2 x the SM count -- with group_size -1 or a multiple of 64 and N / 16 >= the SM
 * count runs the column-slice kernel (no split-K); the rest of M <= 32 the split-K
 * register-fragment kernel; larger M the tcgen05 kernel.  All three give results within the
 * same tolerance of the exact product; they round differently, so their bits may differ.
 * Results are deterministic: a fixed reduction order makes repeated calls on the same device
 * with the same sizes and flags bit-identical.  Tuning overrides read once from the
 * environment (W4A16_STAGE_BLOCKS, W4A16_DECODE_ROWS, W4A16_DECODE_GRID, W4A16_TILE_TOKENS,
 * W4A16_SLICE, W4A16_PAIR_HALF; unset by default) change the kernel choice and tiling, and with them the
 * rounding order: results stay within tolerance but their bits can differ between processes
 * whose environments differ. */
int w4a16_gemm(const void *a, int lda, const int32_t *b_packed, void *c, int ldc,
               const void *scales, const void *zeros, const int32_t *g_idx, const int32_t *perm,
               void *workspace, size_t workspace_bytes, int m, int n, int k, int group_size,
               int weight_type, unsigned flags, cudaStream_t stream);

/* Which kernel w4a16_gemm runs for these sizes and flags on a device with `num_sms`
 * multiprocessors (num_sms <= 0: the current device): 0 the tcgen05 kernel, 1 the split-K
 * small-M kernel, 2 the column-slice small-M kernel; -1 for sizes or flags that w4a16_gemm
 * rejects.  Host code only (with num_sms > 0 it touches no GPU).  For tests and benchmarks:
 * the pages check the tile geometry a launch picked (marlin.rs, the profile-sink test of the
 * vLLM Marlin-MoE path). */
int w4a16_kernel_for(int m, int n, int k, int group_size, unsigned flags, int num_sms);

/* Device scratch of w4a16_gemm_noalloc, per GPU that loads the library (held until exit). */
#define W4A16_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/* w4a16_gemm without a workspace argument, for callers that cannot allocate device memory
 * (code running inside a host callback or an allocator hook, under a framework's sealed
 * memory pool, or in a plug-in whose host offers neither an allocator nor a workspace).  It
 * allocates nothing: the scratch that w4a16_gemm keeps in the caller's workspace lives in a
 * fixed device array of W4A16_NOALLOC_SCRATCH_BYTES inside the library.  The pages have no
 * counterpart of this entry point; it is this library's own.
 *   Arguments as w4a16_gemm, minus workspace / workspace_bytes, plus
 *   status_out  device int32 or NULL, 4-byte aligned: receives (stream-ordered) the call's
 *               device-side error bits (W4A16_DEV_*), 0 when all went well
 * It holds the tcgen05 kernel's token tiles to at most 192 rows (w4a16_gemm goes up to 256),
 * so that their partial-tile slots stay small; M above 192 then runs in tiles of 192 rows, a
 * little slower than w4a16_gemm where that would pick taller tiles.  The scratch a call needs
 * is the status header, one counter per output tile, two fp32 partial slots per CTA (SM count
 * x tile rows x 128 columns each) and, with act-order, the copy of A (M*K*2 bytes); a call for
 * which these exceed W4A16_NOALLOC_SCRATCH_BYTES (an act-order call with a large M*K, a very
 * large M, or a part with many more SMs) returns stage 2 with detail W4A16_ARG_SCRATCH and
 * launches nothing.
 * The first call on a device looks up the array's device address (once per device, cached
 * for the life of the process); make that first call before any stream capture.  A
 * cudaDeviceReset makes the cached address stale: calling this entry point after one is not
 * supported.  Each call clears the status word and tile
 * counters it needs on `stream` before its kernels run.  All calls on one device share the
 * array: calls whose work overlaps on the GPU (other streams, other host threads) race and
 * produce wrong results, so serialise them. */
int w4a16_gemm_noalloc(const void *a, int lda, const int32_t *b_packed, void *c, int ldc,
                       const void *scales, const void *zeros, const int32_t *g_idx,
                       const int32_t *perm, int32_t *status_out, int m, int n, int k,
                       int group_size, int weight_type, unsigned flags, cudaStream_t stream);

/* Workspace bytes for w4a16_gemm_grouped (same rules as w4a16_workspace_size). */
size_t w4a16_grouped_workspace_size(int n_pairs, int n_active, int n, int k, int group_size,
                                    unsigned flags, int num_sms);

/* Grouped (MoE) W4A16 GEMM over an expert-major CSR schedule (memra-engine mmq_ffi.rs,
 * `ExpertCsr`): for every active expert i (ex_ids[i], strictly increasing) and every pair p in
 * ex_pairs[ex_off[i] .. ex_off[i+1]):
 *     y[p][:] = a[pair_tok[p]][:] x dequant(B_{ex_ids[i]})
 * Output rows are pair-major; no routing weight is applied.
 *   a             device fp16 [n_tokens][lda]
 *   b_packed_stack device int32, expert e's tiles at word e*K*N/8
 *   y             device fp16 [n_pairs][ldy]
 *   scales_stack  device fp16, expert e's [G][N] scales at element e*G*N; zeros_stack alike
 *   ex_ids        device int32 [n_active];  ex_off device int32 [n_active+1];
 *   ex_pairs      device int32 [n_pairs];   pair_tok device int32 [n_pairs]
 *   n_active      1..W4A16_MAX_SEGMENTS; n_experts bounds ex_ids
 * Act-order is not supported here (W4A16_FLAG_ACT_ORDER is rejected), and every call runs the
 * tcgen05 kernel (W4A16_FLAG_FORCE_SIMT, _FORCE_MMA and _FORCE_SLICE are rejected).  With
 * W4A16_FLAG_SWIGLU / _GEGLU the experts' weights are interleaved gate/up projections of
 * N = 2I columns and y receives [n_pairs][ldy], ldy >= I, of act(gate) * up, as for
 * w4a16_gemm.
 * Out-of-range schedule entries are skipped and reported as W4A16_DEV_SCHEDULE. */
#define W4A16_MAX_SEGMENTS 1024
int w4a16_gemm_grouped(const void *a, int lda, const int32_t *b_packed_stack, void *y, int ldy,
                       const void *scales_stack, const void *zeros_stack, const int32_t *ex_ids,
                       const int32_t *ex_off, const int32_t *ex_pairs, const int32_t *pair_tok,
                       int n_active, int n_experts, int n_pairs, int n_tokens, int n, int k,
                       int group_size, int weight_type, unsigned flags, void *workspace,
                       size_t workspace_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------------------------
 * Block-routed MoE: the vLLM Marlin-MoE routing interface (ferrum-kernels 0.8.5 marlin.rs,
 * `ferrum_vllm_marlin_moe_f16` and `marlin_gemm_moe_vllm`), on the same tcgen05 kernel as
 * w4a16_gemm_grouped.  Rows are flattened (token, slot) ids, id = token * top_k + slot:
 *   sorted_token_ids  [num_tokens_past_padded] ids listed per expert, each expert's run
 *                     padded to a multiple of moe_block_size with the sentinel prob_m * top_k
 *   expert_ids        [num_tokens_past_padded / moe_block_size] expert of each block; with
 *                     is_ep, -1 marks an expert another rank holds (the block is skipped)
 *   num_tokens_past_padded  one device int32, the padded length (read on the device, so the
 *                     call needs no host synchronisation)
 * and for every non-sentinel row r of block b:
 *     c[id][:] = a[id / top_k][:] x dequant(B_{expert_ids[b]})   (x topk_weights[id] when
 *     mul_topk_weights is 1), rounded once to fp16;
 * rows of c that no entry names are not written.
 * ---------------------------------------------------------------------------------------- */
#define W4A16_MOE_MAX_BLOCKS 4096

/* Host builder of the routing above (vLLM's `moe_align_block_size`, as marlin.rs's doc has the
 * caller run it first): topk_ids [m * top_k] host int32, token-major (id t * top_k + j is token
 * t's j-th expert).  Experts in increasing order, each expert's ids in increasing order, an
 * expert with no ids gets no block.  sorted_token_ids needs `capacity` entries
 * (m * top_k + n_experts * (block_size - 1) always suffices), expert_ids capacity / block_size.
 * Returns num_tokens_past_padded, or -1 on an expert id out of range, a too small capacity or
 * bad sizes. */
int w4a16_moe_align_block_size(const int32_t *topk_ids, int m, int top_k, int n_experts,
                               int block_size, int capacity, int32_t *sorted_token_ids,
                               int32_t *expert_ids);

/* Workspace bytes for w4a16_gemm_moe_blocks (same rules as w4a16_workspace_size). */
size_t w4a16_moe_blocks_workspace_size(int max_padded, int moe_block_size, int n_experts, int n,
                                       int k, int group_size, unsigned flags, int num_sms);

/* The block-routed grouped GEMM.
 *   a               device fp16 [prob_m][lda]
 *   b_packed_stack, scales_stack, zeros_stack  as w4a16_gemm_grouped (expert e's tiles at word
 *                   e*K*N/8, its [G][N] scales / zeros at element e*G*N); zeros for U4 only
 *   c               device fp16 [prob_m * top_k][ldc] (ldc >= N, or >= N/2 with the gated flags)
 *   sorted_token_ids, expert_ids, num_tokens_past_padded  device int32, 4-byte aligned
 *   topk_weights    device fp32 [prob_m * top_k] (4-byte aligned), required when
 *                   mul_topk_weights is 1
 *   max_padded      capacity of sorted_token_ids: a multiple of moe_block_size, at most
 *                   W4A16_MOE_MAX_BLOCKS blocks; num_tokens_past_padded must not exceed it
 *   moe_block_size  8, 16, 32, 48 or 64;  top_k, prob_m, n_experts positive
 *   mul_topk_weights, is_ep  0 or 1
 *   flags           as w4a16_gemm_grouped (W4A16_FLAG_HAS_ZP, W4A16_FLAG_SWIGLU / _GEGLU, ...)
 *   workspace       >= w4a16_moe_blocks_workspace_size(...) bytes, 256-byte aligned,
 *                   zero-filled once (as w4a16_gemm's)
 * Three launches on `stream`: a one-CTA routing kernel that turns the blocks into the grouped
 * kernel's segments (runs of blocks of one expert, blocks of expert -1 dropped) in the
 * workspace, a gather of the rows' activations, and the grouped tcgen05 GEMM.  A padded length
 * that is negative, larger than max_padded or not a whole number of blocks, an expert id out of
 * range (or -1 without is_ep), an id other than a valid one or the sentinel, or more runs than
 * the schedule holds (min(blocks, 1024)) set W4A16_DEV_SCHEDULE; the affected rows are not
 * written. */
int w4a16_gemm_moe_blocks(const void *a, int lda, const int32_t *b_packed_stack, void *c, int ldc,
                          const void *scales_stack, const void *zeros_stack,
                          const int32_t *sorted_token_ids, const int32_t *expert_ids,
                          const int32_t *num_tokens_past_padded, const float *topk_weights,
                          int max_padded, int moe_block_size, int top_k, int mul_topk_weights,
                          int is_ep, int n_experts, int prob_m, int n, int k, int group_size,
                          int weight_type, unsigned flags, void *workspace, size_t workspace_bytes,
                          cudaStream_t stream);

/* Host-side schedule builder (memra-engine mmq_ffi.rs `ExpertCsr::from_token_routes`):
 * token-major routes selected[t*experts_per_token + j] -> expert-major CSR.  Host pointers;
 * ex_ids needs n_expert entries, ex_off n_expert+1, ex_pairs and pair_tok n_tokens*experts_per_token.
 * Returns the number of active experts, or a negative value on rejected input. */
int w4a16_csr_from_token_routes(int n_expert, int n_tokens, int experts_per_token,
                                const int32_t *selected, int32_t *ex_ids, int32_t *ex_off,
                                int32_t *ex_pairs, int32_t *pair_tok);

/* ------------------------------------------------------------------------------------------
 * Checkpoint loading helpers (off the GEMM's path).
 * ---------------------------------------------------------------------------------------- */

/* AutoGPTQ packed zero points -> the fp16 zero points w4a16_gemm takes (host memory, host
 * code).  ferrum-kernels 0.8.4 vllm_marlin.rs, `repack_gptq_qzeros_to_marlin`: a checkpoint
 * stores `zero - 1`, eight 4-bit codes per int32 word along N, column 8w + i at bits 4i..4i+3,
 * so the runtime zero point is the stored code + 1, and a stored 15 (zero point 16, not a
 * 4-bit value) is rejected.
 *   qzeros  host int32 [groups][n / 8]
 *   zeros   host uint16 [groups][n], written: IEEE binary16 bit patterns of the zero points
 *           (integers 1..15), ready to copy to the device
 *   n       a positive multiple of 8
 * Returns 0, or stage 1 with W4A16_ARG_QZERO if any code is 15 (then nothing is written),
 * W4A16_ARG_SHAPE or W4A16_ARG_NULL. */
int w4_qzeros_to_zero_points(const int32_t *qzeros, int groups, int n, uint16_t *zeros);

/* Whether a checkpoint's packed zero words say "symmetric": every 4-bit code of every word is
 * 7 (zero point 8), so the weights can run as W4A16_TYPE_U4B8 without zero points
 * (vllm_marlin.rs, `gptq_qzeros_are_symmetric_code7`).  Host memory; returns 1 or 0 (0 for
 * an empty or NULL array). */
int w4_qzeros_symmetric_code7(const int32_t *qzeros, long long count);

/* Device check of fp16 zero points before they are handed to w4a16_gemm (whose kernels assume
 * integers in [0, 15] and do not check): ORs W4A16_DEV_ZERO into *status (device int32,
 * 4-byte aligned) if any of the `count` values is not an integer in [0, 15] or is NaN.
 * Asynchronous on `stream`; `zeros` is device fp16, 2-byte aligned.  Returns 0, a stage-1
 * status for bad arguments, or a stage-6 launch status. */
int w4a16_zero_points_check(const void *zeros, long long count, int32_t *status,
                            cudaStream_t stream);

/* Reads (synchronously, on `stream`) the device-side status word of a workspace and clears
 * it.  *device_bits receives the W4A16_DEV_* bits seen since the last read.  Returns 0, or a
 * stage-3 status if the copy failed. */
int w4a16_status(void *workspace, int *device_bits, cudaStream_t stream);

/* Self-test of the bounded wait used by every kernel: launches one block that waits on a
 * barrier nobody arrives at, for at most `limit_ns` nanoseconds, then records
 * W4A16_DEV_TIMEOUT in the workspace status word and returns normally.  The context stays
 * usable.  `workspace` needs 256 bytes. */
int w4a16_selftest_timeout(void *workspace, long long limit_ns, cudaStream_t stream);

/* Human-readable name of a status's stage ("ok", "invalid-argument", ...). */
const char *w4a16_status_string(int status);

/* ABI version of the loaded library (W4A16_ABI_VERSION). */
int w4a16_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* W4A16_H */
