// w4a16_aux.cu -- the layout, gather, diagnostic and self-test kernels.
//
//   repack / unpack   GPTQ words <-> the library's tile layout (integer bit moves)
//   gather_cols       act-order: a_perm[m][i] = A[m][perm[i]], and the equal-group check
//   gather_rows       grouped:   a_sorted[r] = A[pair_tok[ex_pairs[r]]]
//   gemm_simt         a CUDA-core reference of the GEMM (diagnostics; same dequant arithmetic)
//   selftest_timeout  exercises the bounded wait on a barrier that never completes
#include "ptx.cuh"
#include "w4a16_internal.h"
#include "w4a16.h"

namespace w4 {

// Tile words (include/w4a16.h, "Packed tile layout"): word (h, c, j) of a 64 x 128 tile holds,
// for p in 0..3 and e in 0..1, the code of row 32h + 2j + 8p + e at bit 4p + 16e.

// One thread per output word.  Word o: tile = o / 1024; inside the tile h = w / 512,
// column c = (w / 4) % 128, j = w % 4.
__global__ void repack_kernel(const int32_t *__restrict__ qweight, const int32_t *__restrict__ perm,
                              int32_t *__restrict__ out, int32_t *status, int k, int n)
{
    const long long total = (long long)k * n / 8;
    const int kblocks = k / KBLK;
    for (long long o = blockIdx.x * (long long)blockDim.x + threadIdx.x; o < total;
         o += (long long)gridDim.x * blockDim.x) {
        const long long tile = o / TILE_WORDS;
        const int w = (int)(o - tile * TILE_WORDS);
        const int nt = (int)(tile / kblocks);
        const int kb = (int)(tile - (long long)nt * kblocks);
        const int h = w >> 9;
        const int c = (w >> 2) & 127;
        const int j = w & 3;
        const int col = nt * TILE_N + c;
        const int r0 = kb * KBLK + h * 32 + 2 * j;
        uint32_t word = 0;
        if (perm == nullptr) {
            // rows r0 + 8p + {0,1} are nibbles 2j, 2j+1 of GPTQ word (r0 + 8p) / 8
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const uint32_t src = (uint32_t)qweight[(long long)((r0 >> 3) + p) * n + col];
                word |= ((src >> (8 * j)) & 0xFu) << (4 * p);
                word |= ((src >> (8 * j + 4)) & 0xFu) << (4 * p + 16);
            }
        } else {
#pragma unroll
            for (int p = 0; p < 4; ++p)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int row = perm[r0 + 8 * p + e];
                    if (row < 0 || row >= k) {
                        if (status)
                            atomicOr(status, W4A16_DEV_PERM);
                        continue;
                    }
                    const uint32_t src = (uint32_t)qweight[(long long)(row >> 3) * n + col];
                    word |= ((src >> (4 * (row & 7))) & 0xFu) << (4 * p + 16 * e);
                }
        }
        out[o] = (int32_t)word;
    }
}

// One thread per GPTQ word (rows 8r..8r+7 of one column): they are pair p = r % 4 of the four
// tile words j = 0..3 of their (block, half, column).
__global__ void unpack_kernel(const int32_t *__restrict__ tiles, int32_t *__restrict__ qweight, int k,
                              int n)
{
    const long long total = (long long)k * n / 8;
    const int kblocks = k / KBLK;
    for (long long o = blockIdx.x * (long long)blockDim.x + threadIdx.x; o < total;
         o += (long long)gridDim.x * blockDim.x) {
        const int r = (int)(o / n);
        const int col = (int)(o - (long long)r * n);
        const int kb = r / 8;
        const int h = (r % 8) / 4;
        const int p = r % 4;
        const int nt = col / TILE_N;
        const int c = col % TILE_N;
        const int32_t *src = tiles + ((long long)nt * kblocks + kb) * TILE_WORDS + h * 512 + c * 4;
        uint32_t word = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t t = (uint32_t)src[j];
            word |= ((t >> (4 * p)) & 0xFu) << (8 * j);
            word |= ((t >> (4 * p + 16)) & 0xFu) << (8 * j + 4);
        }
        qweight[o] = (int32_t)word;
    }
}

// FP8 tiles: tile (nt, kb) holds 2048 words; word (q, c, t) at q*512 + c*4 + t is the source
// word of rows kb*64 + 16q + 4t .. +3 of column nt*128 + c (four K-consecutive E4M3 codes,
// already in the source's byte order), so the repack only moves whole words.
__global__ void repack_fp8_kernel(const int32_t *__restrict__ qweight, int32_t *__restrict__ out,
                                  int k, int n)
{
    const long long total = (long long)k * n / 4;
    const int kblocks = k / KBLK;
    for (long long o = blockIdx.x * (long long)blockDim.x + threadIdx.x; o < total;
         o += (long long)gridDim.x * blockDim.x) {
        const long long tile = o / TILE_WORDS_FP8;
        const int w = (int)(o - tile * TILE_WORDS_FP8);
        const int nt = (int)(tile / kblocks);
        const int kb = (int)(tile - (long long)nt * kblocks);
        const int q = w >> 9, c = (w >> 2) & 127, t = w & 3;
        out[o] = qweight[(long long)(kb * 16 + 4 * q + t) * n + nt * TILE_N + c];
    }
}

__global__ void unpack_fp8_kernel(const int32_t *__restrict__ tiles, int32_t *__restrict__ qweight,
                                  int k, int n)
{
    const long long total = (long long)k * n / 4;
    const int kblocks = k / KBLK;
    for (long long o = blockIdx.x * (long long)blockDim.x + threadIdx.x; o < total;
         o += (long long)gridDim.x * blockDim.x) {
        const int r = (int)(o / n);              // source word row: rows 4r .. 4r+3
        const int col = (int)(o - (long long)r * n);
        const int kb = r / 16, q = (r % 16) / 4, t = r % 4;
        const int nt = col / TILE_N, c = col % TILE_N;
        qweight[o] = tiles[((long long)nt * kblocks + kb) * TILE_WORDS_FP8 + q * 512 + c * 4 + t];
    }
}

// The same gather for tall A: one row at a time is staged whole in shared memory with 16-byte
// loads, then each thread forms eight consecutive outputs from it and writes them as one
// 16-byte store (K % 8 == 0, lda % 8 == 0, both checked by the caller).  A row costs one read
// and one write of its bytes instead of a scattered 2-byte load per element.
__global__ void gather_cols_staged_kernel(const __half *__restrict__ a, int lda,
                                          const int32_t *__restrict__ perm,
                                          const int32_t *__restrict__ g_idx, int group_size,
                                          __half *__restrict__ out, int m, int k, int *status)
{
    extern __shared__ __align__(16) uint16_t rowbuf[];
    pdl_launch_dependents();
    pdl_wait();
    const int chunks = k / 8;
    for (int row = blockIdx.x; row < m; row += gridDim.x) {
        const uint4 *src = reinterpret_cast<const uint4 *>(a + (long long)row * lda);
        for (int i = threadIdx.x; i < chunks; i += blockDim.x)
            reinterpret_cast<uint4 *>(rowbuf)[i] = src[i];
        __syncthreads();
        uint4 *dst = reinterpret_cast<uint4 *>(out + (long long)row * k);
        for (int i = threadIdx.x; i < chunks; i += blockDim.x) {
            uint32_t w[4];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int col = 8 * i + j;
                const int sc = perm[col];
                uint32_t v = 0;
                if (sc >= 0 && sc < k) {
                    v = rowbuf[sc];
                    if (row == 0 && g_idx != nullptr && g_idx[sc] != col / group_size)
                        atomicOr(status, W4A16_DEV_GIDX);
                } else if (row == 0) {
                    atomicOr(status, W4A16_DEV_PERM);
                }
                if (j & 1)
                    w[j >> 1] |= v << 16;
                else
                    w[j >> 1] = v;
            }
            dst[i] = make_uint4(w[0], w[1], w[2], w[3]);
        }
        __syncthreads();
    }
}

// a_perm[m][i] = a[m][perm[i]].  Row 0's threads also check the equal-group property
// g_idx[perm[i]] == i / group_size that the GEMM relies on.
__global__ void gather_cols_kernel(const __half *__restrict__ a, int lda,
                                   const int32_t *__restrict__ perm, const int32_t *__restrict__ g_idx,
                                   int group_size, __half *__restrict__ out, int m, int k, int *status)
{
    pdl_launch_dependents();
    pdl_wait();
    for (int row = blockIdx.y; row < m; row += gridDim.y)
        for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < k; i += gridDim.x * blockDim.x) {
            const int src = perm[i];
            __half v = __float2half(0.0f);
            if (src >= 0 && src < k) {
                v = a[(long long)row * lda + src];
                if (row == 0 && g_idx != nullptr && g_idx[src] != i / group_size)
                    atomicOr(status, W4A16_DEV_GIDX);
            } else if (row == 0) {
                atomicOr(status, W4A16_DEV_PERM);
            }
            out[(long long)row * k + i] = v;
        }
}

// a_sorted[r][:] = a[pair_tok[ex_pairs[r]]][:], 16-byte vectors (K % 8 == 0, lda % 8 == 0).
__global__ void gather_rows_kernel(const __half *__restrict__ a, int lda,
                                   const int32_t *__restrict__ ex_pairs,
                                   const int32_t *__restrict__ pair_tok, __half *__restrict__ out,
                                   int n_pairs, int n_tokens, int k, int *status)
{
    pdl_launch_dependents();
    pdl_wait();
    const int r = blockIdx.x;
    const int pair = ex_pairs[r];
    int tok = -1;
    if (pair >= 0 && pair < n_pairs)
        tok = pair_tok[pair];
    uint4 *dst = reinterpret_cast<uint4 *>(out + (long long)r * k);
    if (tok < 0 || tok >= n_tokens) {
        if (threadIdx.x == 0)
            atomicOr(status, W4A16_DEV_SCHEDULE);
        for (int i = threadIdx.x; i < k / 8; i += blockDim.x)
            dst[i] = make_uint4(0, 0, 0, 0);
        return;
    }
    const uint4 *src = reinterpret_cast<const uint4 *>(a + (long long)tok * lda);
    for (int i = threadIdx.x; i < k / 8; i += blockDim.x)
        dst[i] = src[i];
}

// ---------------------------------------------------------------------------------------
// Block-routed MoE (the vLLM Marlin-MoE interface) -> the grouped kernel's segment schedule,
// on the device (the padded length is a device value).  One CTA: blocks of `block_size` sorted
// rows with a valid expert are compacted in order (blocks of expert -1 with is_ep drop out),
// runs of consecutive blocks of one expert become segments, and every compacted row maps to
// its output row id, or -1 for a sentinel.  Segment slots past the last hold empty segments at
// the end offset, so the kernel can be told the slot count, not the segment count.
// ---------------------------------------------------------------------------------------
constexpr int ROUTE_THREADS = 1024;
constexpr int ROUTE_PER_THREAD = MOE_MAX_BLOCKS / ROUTE_THREADS;

// Exclusive scan of up to MOE_MAX_BLOCKS flags (ROUTE_PER_THREAD consecutive per thread);
// returns the total.  `warp_sums` holds 32 ints of shared memory.
static __device__ int block_exclusive_scan(const int (&flag)[ROUTE_PER_THREAD],
                                           int (&pos)[ROUTE_PER_THREAD], int *warp_sums)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int local = 0;
#pragma unroll
    for (int i = 0; i < ROUTE_PER_THREAD; ++i)
        local += flag[i];
    int incl = local;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d)
            incl += v;
    }
    if (lane == 31)
        warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = warp_sums[lane];
        int wi = w;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, wi, d);
            if (lane >= d)
                wi += v;
        }
        warp_sums[lane] = wi - w; // exclusive prefix of warp sums
        if (lane == 31)
            warp_sums[32] = wi;   // total
    }
    __syncthreads();
    int run = warp_sums[warp] + incl - local;
#pragma unroll
    for (int i = 0; i < ROUTE_PER_THREAD; ++i) {
        pos[i] = run;
        run += flag[i];
    }
    const int total = warp_sums[32];
    __syncthreads();
    return total;
}

__global__ void __launch_bounds__(ROUTE_THREADS)
    moe_route_kernel(const int32_t *__restrict__ sorted_ids, const int32_t *__restrict__ expert_ids,
                     const int32_t *__restrict__ ntpp, int max_padded, int block_size, int n_ids,
                     int n_experts, int is_ep, int seg_cap, int32_t *__restrict__ ex_off,
                     int32_t *__restrict__ ex_ids, int32_t *__restrict__ ex_pairs, int *status)
{
    __shared__ int cexp[MOE_MAX_BLOCKS]; // expert of compacted block c
    __shared__ int cblk[MOE_MAX_BLOCKS]; // its block in the caller's order
    __shared__ int warp_sums[33];
    pdl_launch_dependents();
    pdl_wait();
    int padded = *ntpp;
    if (padded < 0 || padded > max_padded || padded % block_size != 0) {
        if (threadIdx.x == 0)
            atomicOr(status, W4A16_DEV_SCHEDULE);
        padded = 0;
    }
    const int n_blocks = padded / block_size;
    const int b0 = threadIdx.x * ROUTE_PER_THREAD;
    int flag[ROUTE_PER_THREAD], pos[ROUTE_PER_THREAD], exp_[ROUTE_PER_THREAD];
    bool bad = false;
#pragma unroll
    for (int i = 0; i < ROUTE_PER_THREAD; ++i) {
        const int b = b0 + i;
        exp_[i] = b < n_blocks ? expert_ids[b] : -1;
        flag[i] = (b < n_blocks && exp_[i] >= 0 && exp_[i] < n_experts) ? 1 : 0;
        bad |= b < n_blocks && !flag[i] && !(is_ep && exp_[i] == -1);
    }
    if (bad)
        atomicOr(status, W4A16_DEV_SCHEDULE);
    const int n_valid = block_exclusive_scan(flag, pos, warp_sums);
#pragma unroll
    for (int i = 0; i < ROUTE_PER_THREAD; ++i)
        if (flag[i]) {
            cexp[pos[i]] = exp_[i];
            cblk[pos[i]] = b0 + i;
        }
    __syncthreads();
    // Segment starts among the compacted blocks.
#pragma unroll
    for (int i = 0; i < ROUTE_PER_THREAD; ++i) {
        const int c = b0 + i;
        flag[i] = (c < n_valid && (c == 0 || cexp[c] != cexp[c - 1])) ? 1 : 0;
    }
    int n_seg = block_exclusive_scan(flag, pos, warp_sums);
    const bool overflow = n_seg > seg_cap;
    if (overflow) {
        if (threadIdx.x == 0)
            atomicOr(status, W4A16_DEV_SCHEDULE);
        n_seg = 0;
    }
    const int rows = overflow ? 0 : n_valid * block_size;
    if (!overflow) {
#pragma unroll
        for (int i = 0; i < ROUTE_PER_THREAD; ++i)
            if (flag[i]) {
                ex_ids[pos[i]] = cexp[b0 + i];
                ex_off[pos[i]] = (b0 + i) * block_size;
            }
    }
    for (int sidx = n_seg + (int)threadIdx.x; sidx <= seg_cap; sidx += ROUTE_THREADS) {
        ex_off[sidx] = rows;
        if (sidx < seg_cap)
            ex_ids[sidx] = 0;
    }
    for (int r = threadIdx.x; r < max_padded; r += ROUTE_THREADS) {
        int id = -1;
        if (r < rows) {
            const int src = sorted_ids[cblk[r / block_size] * block_size + r % block_size];
            if (src >= 0 && src < n_ids)
                id = src;
            else if (src != n_ids)
                atomicOr(status, W4A16_DEV_SCHEDULE);
        }
        ex_pairs[r] = id;
    }
}

// a_sorted[r] = a[ex_pairs[r] / top_k] for the rows of the routed schedule (ex_off_end holds
// their count), a zero row for a sentinel; rows past the count are left alone.
__global__ void moe_gather_kernel(const __half *__restrict__ a, int lda,
                                  const int32_t *__restrict__ ex_off_end,
                                  const int32_t *__restrict__ ex_pairs, int top_k,
                                  __half *__restrict__ out, int k)
{
    pdl_launch_dependents();
    pdl_wait();
    const int r = blockIdx.x;
    if (r >= *ex_off_end)
        return;
    const int id = ex_pairs[r];
    uint4 *dst = reinterpret_cast<uint4 *>(out + (long long)r * k);
    if (id < 0) {
        for (int i = threadIdx.x; i < k / 8; i += blockDim.x)
            dst[i] = make_uint4(0, 0, 0, 0);
        return;
    }
    const uint4 *src = reinterpret_cast<const uint4 *>(a + (long long)(id / top_k) * lda);
    for (int i = threadIdx.x; i < k / 8; i += blockDim.x)
        dst[i] = src[i];
}

// Gate/up interleave of a row-major [rows][2I] array: destination column j takes source
// column 16b + r (gate) for j = 32b + r, r < 16, and I + 16b + r - 16 (up) for r >= 16.
template <typename T>
__global__ void gate_up_interleave_kernel(const T *__restrict__ src, T *__restrict__ dst, int rows,
                                          int n2)
{
    const int half_n = n2 / 2;
    const long long total = (long long)rows * n2;
    for (long long o = blockIdx.x * (long long)blockDim.x + threadIdx.x; o < total;
         o += (long long)gridDim.x * blockDim.x) {
        const long long row = o / n2;
        const int j = (int)(o - row * n2);
        const int b = j >> 5, r = j & 31;
        const int from = r < 16 ? 16 * b + r : half_n + 16 * b + r - 16;
        dst[o] = src[row * n2 + from];
    }
}

// CUDA-core reference GEMM: one thread per output, fp32 accumulation in k order, weights
// dequantised with the same fp16 arithmetic as the tensor-core path ((q - z) exact, then one
// rounding of the product with the scale).
__global__ void gemm_simt_kernel(GemmParams p, const __half *__restrict__ a, int lda)
{
    const int col = blockIdx.x * blockDim.x + threadIdx.x;
    if (col >= p.n)
        return;
    const int nt = col / TILE_N, c = col % TILE_N;
    for (int row = blockIdx.y; row < p.m; row += gridDim.y) {
    float acc = 0.0f;
    for (int r = 0; r < p.k; ++r) {
        const int kb = r / KBLK, h = (r % KBLK) / 32, r32 = r % 32;
        const int pp = r32 / 8, j = (r32 % 8) / 2, e = r32 % 2;
        const uint32_t w =
            (uint32_t)p.b[((long long)nt * p.kblocks + kb) * TILE_WORDS + h * 512 + c * 4 + j];
        const int q = (w >> (4 * pp + 16 * e)) & 0xF;
        const int g = r / p.group_size;
        const __half s = p.scales[(long long)g * p.n + col];
        const __half z = p.zeros ? p.zeros[(long long)g * p.n + col] : __float2half(8.0f);
        const __half d = __hsub(__hadd(__float2half(1024.0f), __int2half_rn(q)),
                                __hadd(__float2half(1024.0f), z));
        const __half wv = __hmul(d, s);
        acc = fmaf(__half2float(a[(long long)row * lda + r]), __half2float(wv), acc);
    }
    p.c[(long long)row * p.ldc + col] = __float2half_rn(acc);
    }
}

__global__ void selftest_timeout_kernel(int *status, unsigned long long limit_ns)
{
    __shared__ uint64_t bar;
    __shared__ volatile int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        abort_flag = 0;
    }
    __syncthreads();
    WaitCtl ctl{&abort_flag, status, limit_ns};
    if (threadIdx.x == 0)
        mbar_wait(&bar, 0, ctl, W4A16_DEV_TIMEOUT); // nobody arrives: must time out
    __syncthreads();
}

static int grid_for(long long work, int block)
{
    long long g = (work + block - 1) / block;
    if (g < 1)
        g = 1;
    if (g > 65535LL * 32)
        g = 65535LL * 32;
    return (int)g;
}

int launch_repack(const int32_t *qweight, const int32_t *perm, int32_t *out, int32_t *status, int k,
                  int n, cudaStream_t stream)
{
    const long long total = (long long)k * n / 8;
    repack_kernel<<<grid_for(total, 256), 256, 0, stream>>>(qweight, perm, out, status, k, n);
    return cudaGetLastError();
}

int launch_unpack(const int32_t *tiles, int32_t *qweight, int k, int n, cudaStream_t stream)
{
    const long long total = (long long)k * n / 8;
    unpack_kernel<<<grid_for(total, 256), 256, 0, stream>>>(tiles, qweight, k, n);
    return cudaGetLastError();
}

int launch_repack_fp8(const int32_t *qweight, int32_t *out, int k, int n, cudaStream_t stream)
{
    const long long total = (long long)k * n / 4;
    repack_fp8_kernel<<<grid_for(total, 256), 256, 0, stream>>>(qweight, out, k, n);
    return cudaGetLastError();
}

int launch_unpack_fp8(const int32_t *tiles, int32_t *qweight, int k, int n, cudaStream_t stream)
{
    const long long total = (long long)k * n / 4;
    unpack_fp8_kernel<<<grid_for(total, 256), 256, 0, stream>>>(tiles, qweight, k, n);
    return cudaGetLastError();
}

int launch_gather_cols(const __half *a, int lda, const int32_t *perm, const int32_t *g_idx,
                       int group_size, __half *out, int m, int k, int *status, cudaStream_t stream)
{
    // Tall A with rows that fit the default shared-memory window: staged rows, one CTA per row
    // (up to 4096 CTAs, each looping).  Short A keeps the element-wise kernel, whose grid also
    // spreads each row over CTAs.
    if (m >= 64 && k * 2 <= 48 * 1024 && k % 8 == 0 && lda % 8 == 0) {
        const int grid = m < 4096 ? m : 4096;
        gather_cols_staged_kernel<<<grid, 256, k * 2, stream>>>(a, lda, perm, g_idx, group_size,
                                                                out, m, k, status);
        return cudaGetLastError();
    }
    const int bx = (k + 255) / 256;
    dim3 grid(bx, m < 65535 ? m : 65535);
    gather_cols_kernel<<<grid, 256, 0, stream>>>(a, lda, perm, g_idx, group_size, out, m, k, status);
    return cudaGetLastError();
}

int launch_gather_rows(const __half *a, int lda, const int32_t *ex_pairs, const int32_t *pair_tok,
                       __half *out, int n_pairs, int n_tokens, int k, int *status,
                       cudaStream_t stream)
{
    gather_rows_kernel<<<n_pairs, 128, 0, stream>>>(a, lda, ex_pairs, pair_tok, out, n_pairs,
                                                    n_tokens, k, status);
    return cudaGetLastError();
}

int launch_moe_route(const int32_t *sorted_ids, const int32_t *expert_ids, const int32_t *ntpp,
                     int max_padded, int block_size, int n_ids, int n_experts, int is_ep,
                     int seg_cap, int32_t *ex_off, int32_t *ex_ids, int32_t *ex_pairs, int *status,
                     cudaStream_t stream)
{
    moe_route_kernel<<<1, ROUTE_THREADS, 0, stream>>>(sorted_ids, expert_ids, ntpp, max_padded,
                                                      block_size, n_ids, n_experts, is_ep, seg_cap,
                                                      ex_off, ex_ids, ex_pairs, status);
    return cudaGetLastError();
}

int launch_moe_gather(const __half *a, int lda, const int32_t *ex_off_end, const int32_t *ex_pairs,
                      int top_k, __half *out, int max_padded, int k, cudaStream_t stream)
{
    moe_gather_kernel<<<max_padded, 128, 0, stream>>>(a, lda, ex_off_end, ex_pairs, top_k, out, k);
    return cudaGetLastError();
}

int launch_gate_up_interleave(const void *src, void *dst, int rows, int n2, int elem_bytes,
                              cudaStream_t stream)
{
    const long long total = (long long)rows * n2;
    if (elem_bytes == 4)
        gate_up_interleave_kernel<int32_t><<<grid_for(total, 256), 256, 0, stream>>>(
            static_cast<const int32_t *>(src), static_cast<int32_t *>(dst), rows, n2);
    else
        gate_up_interleave_kernel<uint16_t><<<grid_for(total, 256), 256, 0, stream>>>(
            static_cast<const uint16_t *>(src), static_cast<uint16_t *>(dst), rows, n2);
    return cudaGetLastError();
}

int launch_gemm_simt(const GemmParams &p, const __half *a, int lda, cudaStream_t stream)
{
    dim3 grid((p.n + 127) / 128, p.m < 65535 ? p.m : 65535);
    gemm_simt_kernel<<<grid, 128, 0, stream>>>(p, a, lda);
    return cudaGetLastError();
}

int launch_selftest_timeout(int *status, unsigned long long limit_ns, cudaStream_t stream)
{
    selftest_timeout_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
    return cudaGetLastError();
}

} // namespace w4
