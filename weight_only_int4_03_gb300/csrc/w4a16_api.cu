// w4a16_api.cu -- the C ABI of include/w4a16.h: argument checks, tile planning, workspace
// carving, tensor-map encoding and launches.  No entry point allocates, synchronises (except
// w4a16_status, whose job is to read back) or falls back to the CPU.
#include <cudaTypedefs.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>

#include "w4a16_internal.h"
#include "w4a16.h"

using namespace w4;

namespace {

constexpr int STAGE_ARG = 1;
constexpr int STAGE_UNSUPPORTED = 2;
constexpr int STAGE_RESOURCE = 3;
constexpr int STAGE_LAUNCH = 6;

inline int status_of(int stage, int detail)
{
    return (stage << 16) | (detail & 0xFFFF);
}

inline bool aligned(const void *p, uintptr_t a)
{
    return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

inline long long round_up(long long v, long long a)
{
    return (v + a - 1) / a * a;
}

constexpr long long HEADER_BYTES = 256;
constexpr unsigned long long WAIT_LIMIT_NS = 2000000000ull; // 2 s per bounded wait

// Group-size rule: transformer.rs `marlin_num_groups` (-1 or a positive divisor of K) with
// marlin.rs's Marlin-MoE rule that a positive size is a multiple of 16.  Returns G or -1.
int num_groups(int k, int group_size)
{
    if (k <= 0)
        return -1;
    if (group_size == -1)
        return 1;
    if (group_size <= 0 || group_size % 16 != 0 || k % group_size != 0)
        return -1;
    return k / group_size;
}

struct Plan {
    int nt_max, m_tiles, tiles_bound, grid;
    int kbs, sg_box, act_kb_bytes, packed_off, scales_off, zeros_off;
    int stages, stage_bytes, acc_bufs, acc_col0, tmem_cols, smem_bytes, seg_off, epi_off, a_slots;
    bool a_tmem, mma; // mma: a small-M register-fragment kernel instead of tcgen05
    bool slice = false; // ... the column-slice one (no split-K)
    int act_rows = 0;   // rows of one activation box (slice kernel: M; pairs: a half-tile;
                        // others: nt_max)
    int halves = 1, nt_half = 0; // tcgen05: token tile as a pair of half-tiles (halves 2)
    int tile_bytes = TILE_BYTES; // one packed 64 x 128 tile (FP8: twice as large)
    int split = 0;    // tile-aligned split factor (0: stream-K)
    int n_slices = 0, slice_per = 0;
    long long counters_off, partials_off, a_off, total;
};

// Workspace carving (byte offsets), shared by the size queries and the launches.  The
// partial-tile area holds two [slot_rows x 128] fp32 slots per CTA: slot_cta_rows is the
// largest (CTAs x tile rows) of the kernels the call may pick.
void carve(Plan &pl, long long slot_cta_rows, long long a_bytes)
{
    pl.counters_off = HEADER_BYTES;
    pl.partials_off = round_up(pl.counters_off + 4LL * pl.tiles_bound, 256);
    pl.a_off = round_up(pl.partials_off + slot_cta_rows * 2 * TILE_N * 4, 256);
    pl.total = round_up(pl.a_off + a_bytes, 256);
}

// L2 bytes of the current device (cached; 0 if the query fails).
long long l2_bytes()
{
    static std::mutex mu;
    static long long cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrL2CacheSize, dev) != cudaSuccess)
            return 0;
        cache[dev] = v;
    }
    return cache[dev];
}

int sm_count(int *out)
{
    static std::mutex mu;
    static int cache[64];
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 64 && cache[dev] > 0) {
        *out = cache[dev];
        return cudaSuccess;
    }
    int v = 0;
    err = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess)
        return err;
    if (dev >= 0 && dev < 64)
        cache[dev] = v;
    *out = v;
    return cudaSuccess;
}

int env_int(const char *name, int lo, int hi, int dflt)
{
    const char *s = getenv(name);
    if (!s)
        return dflt;
    const int v = atoi(s);
    return (v >= lo && v <= hi) ? v : dflt;
}

// 64-row blocks per pipeline stage.  A TMA copy has a large fixed cost, so the packed codes
// of a stage travel as one bulk copy of kbs * 4 KiB; 8 blocks (32 KiB) is the default,
// W4A16_STAGE_BLOCKS overrides it for tuning.
int stage_blocks_default()
{
    static int v = env_int("W4A16_STAGE_BLOCKS", 1, MAX_STAGES, 8);
    return v;
}

// Largest M the small-M kernel takes by default (W4A16_DECODE_ROWS overrides, 0..64).
int decode_rows_default()
{
    static int v = env_int("W4A16_DECODE_ROWS", 0, 64, 32);
    return v;
}

// CTAs per SM that one small-M launch fills (W4A16_DECODE_GRID overrides, 1..2).  Each CTA is
// sized for half an SM either way; a launch that fills one leaves the other free for the next
// launch of the stream, whose CTAs then start their weight copies while this one drains.
int decode_grid_per_sm()
{
    static int v = env_int("W4A16_DECODE_GRID", 1, decode_ctas_per_sm(), decode_ctas_per_sm());
    return v;
}

// Token-tile height of the tcgen05 kernel (a multiple of 16, at most cap rows): one tile for
// M <= cap; above that M is cut into ceil(M / 224) tiles of equal height rounded up to 16, but
// never below 192 rows.  Prefill is bound by the dequantisation of each weight tile, which is
// done once per token tile, so fewer, taller tiles win while the tile count stays the same or
// drops: M=1024 runs 5 tiles of 208 (6 of 192 before), M=4096 19 of 224 (22 of 192).  Up to
// 192 rows two accumulator buffers fit in tensor memory beside the dequantised-weight ring
// (the epilogue overlaps the next tile's MMAs); taller tiles trade that overlap for the
// smaller tile count.  Below 192 rows per tile the kernel slows sharply (160-row tiles run at
// two thirds of the rate), so M just above a multiple of 192 keeps 192-row tiles.
// W4A16_TILE_TOKENS overrides for tuning.
int pick_nt(int m, int cap)
{
    static int env = [] {
        const int v = env_int("W4A16_TILE_TOKENS", 16, MAX_TOK, 0);
        return v % 16 == 0 ? v : 0;
    }();
    if (env > 0) {
        const int e = env < cap ? env : cap;
        return m <= e ? (int)round_up(m, 16) : e;
    }
    if (m <= cap)
        return (int)round_up(m, 16);
    const int hi = cap < TALL_TILE_TOK ? cap : TALL_TILE_TOK;
    const int lo = hi < TWO_BUF_TILE_TOK ? hi : TWO_BUF_TILE_TOK;
    const int tiles = (m + hi - 1) / hi;
    const int nt = (int)round_up((m + tiles - 1) / tiles, 16);
    return nt < lo ? lo : nt;
}

// The tcgen05 kernel's token tile: pick_nt's single tile, or -- for w4a16_gemm's full tile cap,
// when it lowers the number of tiles -- a pair of half-tiles of equal height (a multiple of 16,
// at most PAIR_HALF_TOK) whose MMAs share each dequantised weight block.  The dequantisation
// bounds the kernel at large M, and a pair dequantises once for up to 384 tokens where a single
// tile does for at most 256: M=4096 runs 11 pairs of 2 x 192 (19 tiles of 224 before), M=2048
// 6 of 2 x 176, M=1024 3 of 2 x 176.
struct TcTile {
    int rows, halves, half;
};

int pair_half_max()
{
    static int v = [] {
        const int e = env_int("W4A16_PAIR_HALF", 0, PAIR_HALF_TOK, PAIR_HALF_TOK);
        return e % 16 == 0 ? e : PAIR_HALF_TOK;
    }();
    return v;
}

TcTile pick_tc_tile(int m, int cap, bool allow_pairs)
{
    TcTile t{pick_nt(m, cap), 1, 0};
    t.half = t.rows;
    const int hmax = pair_half_max();
    if (!allow_pairs || m <= cap || cap < MAX_TOK || hmax == 0)
        return t;
    const int tiles = (m + t.rows - 1) / t.rows;
    const int pairs = (m + 2 * hmax - 1) / (2 * hmax);
    if (pairs >= tiles)
        return t;
    const int per_pair = (m + pairs - 1) / pairs;
    t.half = (int)round_up((per_pair + 1) / 2, 16);
    t.halves = 2;
    t.rows = 2 * t.half;
    return t;
}

// Token-tile height of the small-M kernel: the smallest of 8, 16, 32, 64 rows that holds M.
int pick_nt_mma(int m)
{
    int nt = 8;
    while (nt < m)
        nt <<= 1;
    return nt;
}

// Stage geometry: [activations kbs x nt_max x 128 B | packed kbs x 4 KiB | scales | zeros].
// The activation part starts the stage (1024-byte aligned for the 128-byte swizzle); the
// scale rows a stage touches are at most ceil(kbs*64 / gs) + 1 (a group may straddle the
// stage start), never more than the tensor's rows.
void stage_layout(Plan &pl, int kbs, int group_size, int g_rows, bool has_zp)
{
    pl.kbs = kbs;
    const int halves = pl.halves > 1 ? pl.halves : 1;
    pl.act_kb_bytes = (halves > 1 ? pl.nt_half : pl.nt_max) * 128; // per half-tile and block
    const int sg = (kbs * KBLK + group_size - 1) / group_size + 1;
    pl.sg_box = sg < g_rows ? sg : g_rows;
    pl.packed_off = halves * kbs * pl.act_kb_bytes; // [half][block][rows x 128 B]
    pl.scales_off = pl.packed_off + kbs * pl.tile_bytes;
    pl.zeros_off = pl.scales_off + (int)round_up((long long)pl.sg_box * SG_BYTES, 128);
    const int end = has_zp ? pl.zeros_off + pl.sg_box * SG_BYTES : pl.zeros_off;
    pl.stage_bytes = (int)round_up(end, 1024);
}

// Dynamic shared memory a CTA may use: the tcgen05 kernel (one CTA per SM) or the small-M
// kernel (several per SM).  Cached per device.
int smem_limit(int *limit, bool mma)
{
    static std::mutex mu;
    static int limit_cache[2][64];
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 64 && limit_cache[mma][dev] > 0) {
        *limit = limit_cache[mma][dev];
        return cudaSuccess;
    }
    err = (cudaError_t)(mma ? decode_smem_limit(limit) : gemm_smem_limit(limit));
    if (err != cudaSuccess)
        return err;
    if (dev >= 0 && dev < 64)
        limit_cache[mma][dev] = *limit;
    return cudaSuccess;
}

// Shared-memory plan: the largest stage (up to the default block count, and for the tcgen05
// kernel no more blocks than the dequantised-weight ring holds) that still leaves three
// stages in flight; two at the very least.
int plan_smem(Plan &pl, bool grouped, bool has_zp, int group_size, int g_rows)
{
    int limit = 0;
    int err = smem_limit(&limit, pl.mma);
    if (err != cudaSuccess)
        return err;
    const int extra = pl.mma ? decode_extra_smem(pl.nt_max) : gemm_extra_smem(pl.a_tmem, grouped);
    if (pl.slice) {
        // Column-slice stage: [activations kbs x M rows x 128 B | codes kbs x 512 B | scale
        // rows x 16 columns | zero rows], kbs = 8 warps x slice_bpw(nt_max) blocks.  The
        // activation box is exactly M rows (the token rows an 8-token MMA tile has beyond M read
        // a zero row instead).  After the stages: two buffers for the cross-warp sum of a slice
        // (8 warps x nt_max/8 x 4 x 32 fp32 each), then the 128-byte zero row.
        const int kbs = SLICE_WARPS * slice_bpw(pl.nt_max, pl.tile_bytes == TILE_BYTES_FP8);
        pl.kbs = kbs;
        pl.act_kb_bytes = pl.act_rows * 128;
        const int sg = (kbs * KBLK + group_size - 1) / group_size + 1;
        pl.sg_box = sg < g_rows ? sg : g_rows;
        pl.packed_off = (int)round_up((long long)kbs * pl.act_kb_bytes, 1024);
        const int block_bytes = pl.tile_bytes == TILE_BYTES_FP8 ? 2 * SLICE_BLOCK_BYTES : SLICE_BLOCK_BYTES;
        pl.scales_off = pl.packed_off + kbs * block_bytes;
        pl.zeros_off = pl.scales_off + (int)round_up((long long)pl.sg_box * SLICE_N * 2, 128);
        const int end = has_zp ? pl.zeros_off + pl.sg_box * SLICE_N * 2 : pl.zeros_off;
        pl.stage_bytes = (int)round_up(end, 1024);
        const int red = 2 * SLICE_WARPS * (pl.nt_max / 8) * 4 * 32 * 4 + 128;
        pl.stages = (limit - extra - red) / pl.stage_bytes;
        if (pl.stages < 2)
            return cudaErrorInvalidConfiguration;
        if (pl.stages > MAX_STAGES)
            pl.stages = MAX_STAGES;
        pl.epi_off = pl.stages * pl.stage_bytes;
        pl.seg_off = pl.epi_off;
        pl.smem_bytes = pl.stages * pl.stage_bytes + red + extra;
        return cudaSuccess;
    }
    if (pl.mma) {
        int kbs = stage_blocks_default();
        for (;; kbs = kbs > 1 ? kbs / 2 : 0) {
            if (kbs == 0)
                return cudaErrorInvalidConfiguration;
            stage_layout(pl, kbs, group_size, g_rows, has_zp);
            pl.stages = (limit - extra) / pl.stage_bytes;
            if (pl.stages >= 3 || (kbs == 1 && pl.stages >= 2))
                break;
        }
        if (pl.stages > MAX_STAGES)
            pl.stages = MAX_STAGES;
    } else {
        // The tcgen05 kernel gives each stage its own kbs weight slots, so stages x kbs <=
        // a_slots.  The largest stage (from the default block count down) that leaves three
        // stages in flight, else the one with the most stages (two at the least).
        int best_kbs = 0, best_stages = 0;
        for (int kbs = stage_blocks_default(); kbs >= 1; kbs /= 2) {
            stage_layout(pl, kbs, group_size, g_rows, has_zp);
            int st = (limit - extra) / pl.stage_bytes;
            if (st > MAX_STAGES)
                st = MAX_STAGES;
            if (st * kbs > pl.a_slots)
                st = pl.a_slots / kbs;
            if (st > best_stages) {
                best_kbs = kbs;
                best_stages = st;
            }
            if (st >= 3)
                break;
        }
        if (best_stages < 2)
            return cudaErrorInvalidConfiguration;
        stage_layout(pl, best_kbs, group_size, g_rows, has_zp);
        pl.stages = best_stages;
    }
    pl.epi_off = pl.stages * pl.stage_bytes + (!pl.mma && !pl.a_tmem ? SMEM_A_SLOTS * A_SLOT_BYTES : 0);
    pl.seg_off = pl.epi_off + (pl.mma ? 0 : EPI_STAGE_BYTES);
    pl.smem_bytes = pl.stages * pl.stage_bytes + extra;
    return cudaSuccess;
}

// Tensor memory of the tcgen05 kernel: accumulators (two buffers when they fit next to a
// 4-slot weight ring) and, in tensor-memory mode, as many 32-column weight slots as the rest
// of the 512 columns hold (at most MAX_A_SLOTS).
void plan_tmem(Plan &pl)
{
    if (pl.mma) {
        pl.acc_bufs = 1;
        pl.a_slots = 0;
        pl.acc_col0 = 0;
        pl.tmem_cols = 0;
        return;
    }
    const int min_ring = pl.a_tmem ? 4 * A_SLOT_COLS : 0;
    pl.acc_bufs = (min_ring + 2 * pl.nt_max <= 512) ? 2 : 1;
    if (pl.a_tmem) {
        const int slots = (512 - pl.acc_bufs * pl.nt_max) / A_SLOT_COLS;
        pl.a_slots = slots > MAX_A_SLOTS ? MAX_A_SLOTS : slots;
    } else {
        pl.a_slots = SMEM_A_SLOTS;
    }
    pl.acc_col0 = pl.a_tmem ? pl.a_slots * A_SLOT_COLS : 0;
    const int need = pl.acc_col0 + pl.acc_bufs * pl.nt_max;
    int cols = 32;
    while (cols < need)
        cols <<= 1;
    pl.tmem_cols = cols;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Activation rows [rows][ld] fp16 viewed as [K/64][rows][64]: one copy brings kbs column
// blocks of nt_max rows, each landing as an [nt_max x 128 B] tile in the 128-byte swizzle.
int encode_act_map(CUtensorMap *map, const void *base, int rows, int k, int ld, int nt, int kbs)
{
    auto fn = encode_fn();
    if (!fn)
        return cudaErrorNotSupported;
    cuuint64_t dims[3] = {(cuuint64_t)KBLK, (cuuint64_t)rows, (cuuint64_t)(k / KBLK)};
    cuuint64_t strides[2] = {(cuuint64_t)ld * 2, (cuuint64_t)KBLK * 2};
    cuuint32_t box[3] = {KBLK, (cuuint32_t)nt, (cuuint32_t)kbs};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Scale (or zero) rows [g_rows][n] fp16: boxes of box_n columns (128, or 16 for the
// column-slice kernel) x sg_box group rows.
int encode_group_map(CUtensorMap *map, const void *base, int g_rows, int n, int sg_box,
                     int box_n = TILE_N)
{
    auto fn = encode_fn();
    if (!fn)
        return cudaErrorNotSupported;
    cuuint64_t dims[2] = {(cuuint64_t)n, (cuuint64_t)g_rows};
    cuuint64_t strides[1] = {(cuuint64_t)n * 2};
    cuuint32_t box[2] = {(cuuint32_t)box_n, (cuuint32_t)sg_box};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Packed tiles viewed as [tiles x K/64 x 2][512] int32 rows (a row is one 32-row half of a
// 64-row block of a 128-column tile: 128 columns x 4 words): a box of 64 words x 2*kbs rows
// brings the codes of one 16-column slice for kbs consecutive blocks, 256 bytes per row.
int encode_slice_weight_map(CUtensorMap *map, const void *base, int n, int k, int kbs, bool w8)
{
    auto fn = encode_fn();
    if (!fn)
        return cudaErrorNotSupported;
    // Rows of 512 words: the two 32-row halves of a 4-bit tile, or the four 16-row quarters of
    // an FP8 tile; a slice's block is 64 words of 2 (or 4) consecutive rows.
    const int rows_per_block = w8 ? 4 : 2;
    cuuint64_t dims[2] = {(cuuint64_t)(TILE_WORDS / 2),
                          (cuuint64_t)(n / TILE_N) * (cuuint64_t)(k / KBLK) * rows_per_block};
    cuuint64_t strides[1] = {(cuuint64_t)TILE_BYTES / 2};
    cuuint32_t box[2] = {(cuuint32_t)(SLICE_N * 4), (cuuint32_t)(rows_per_block * kbs)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, const_cast<void *>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Checks shared by both GEMM entry points.  Returns 0 or a stage-1/2 status.
int check_weights(const void *b, const void *scales, const void *zeros, int n, int k, int group_size,
                  int weight_type, unsigned flags)
{
    if (weight_type != W4A16_TYPE_U4 && weight_type != W4A16_TYPE_U4B8 &&
        weight_type != W4A16_TYPE_FE4M3)
        return status_of(STAGE_ARG, W4A16_ARG_TYPE);
    if (n <= 0 || k <= 0)
        return status_of(STAGE_ARG, W4A16_ARG_SHAPE);
    if (!b || !scales)
        return status_of(STAGE_ARG, W4A16_ARG_NULL);
    if (!aligned(b, 16) || !aligned(scales, 16) || (zeros && !aligned(zeros, 16)))
        return status_of(STAGE_ARG, W4A16_ARG_ALIGN);
    if (k % 128 != 0 || n % 256 != 0)
        return status_of(STAGE_UNSUPPORTED, W4A16_ARG_SHAPE);
    if (num_groups(k, group_size) < 0)
        return status_of(STAGE_ARG, W4A16_ARG_GROUP);
    // FP8 weights: groups of whole 64-row blocks (the pages' Marlin-MoE rule is -1 or 128).
    if (weight_type == W4A16_TYPE_FE4M3 && group_size != -1 && group_size % KBLK != 0)
        return status_of(STAGE_ARG, W4A16_ARG_GROUP);
    const bool has_zp_flag = (flags & W4A16_FLAG_HAS_ZP) != 0;
    if (has_zp_flag != (zeros != nullptr))
        return status_of(STAGE_ARG, W4A16_ARG_FLAGS);
    if ((weight_type == W4A16_TYPE_U4) != (zeros != nullptr))
        return status_of(STAGE_ARG, W4A16_ARG_FLAGS);
    if ((long long)k * n / 4 > (1LL << 40))
        return status_of(STAGE_ARG, W4A16_ARG_OVERFLOW);
    return 0;
}

// FP8 weights run on the tcgen05 kernel only, without act-order (the pages' FP8 Marlin has
// neither zero points nor act-order), and with fp16 activations.
int check_fp8_flags(int weight_type, unsigned flags)
{
    if (weight_type != W4A16_TYPE_FE4M3)
        return 0;
    if (flags & (W4A16_FLAG_ACT_ORDER | W4A16_FLAG_FORCE_SIMT | W4A16_FLAG_FORCE_MMA |
                 W4A16_FLAG_BF16))
        return status_of(STAGE_ARG, W4A16_ARG_FLAGS);
    return 0;
}

int tile_bytes_of(int weight_type)
{
    return weight_type == W4A16_TYPE_FE4M3 ? TILE_BYTES_FP8 : TILE_BYTES;
}

// The packed-tile geometry of a call's weight type, after fill_params.
void set_weight_type(GemmParams &p, int weight_type, unsigned flags)
{
    const bool w8 = weight_type == W4A16_TYPE_FE4M3;
    p.w8 = w8 ? 1 : 0;
    p.bf16 = (flags & W4A16_FLAG_BF16) ? 1 : 0;
    p.tile_words = w8 ? TILE_WORDS_FP8 : TILE_WORDS;
    p.tile_bytes = w8 ? TILE_BYTES_FP8 : TILE_BYTES;
}

int launch_status(int err)
{
    return err == cudaSuccess ? 0 : status_of(STAGE_LAUNCH, err);
}

// CTA count for `tiles` output tiles of `kblocks` 64-row blocks on `ctas` CTA slots, and the
// split factor (0: stream-K).  When every tile can take s >= 1 CTAs (s <= kblocks), each with
// one near-equal K-range, and tiles * s CTAs cover at least 80 % of the slots, launch exactly
// that: no CTA's range then straddles two tiles, so none runs two split-tile protocols back to
// back (M=8, 4096x4096: 9.9 -> 7.6 us).  Otherwise stream-K over all slots.
int aligned_grid(int tiles, int kblocks, int ctas, int *split)
{
    *split = 0;
    const long long units = (long long)tiles * kblocks;
    if (units <= ctas)
        return (int)(units > 0 ? units : 1);
    int s = tiles > 0 ? ctas / tiles : 0;
    if (s > kblocks)
        s = kblocks;
    if (s >= 1 && (long long)tiles * s * 5 >= (long long)ctas * 4) {
        *split = s;
        return tiles * s;
    }
    return ctas;
}

// Whether the column-slice kernel is picked by default where it applies (W4A16_SLICE=0 turns
// it off, for comparison).
bool slice_default()
{
    static int v = env_int("W4A16_SLICE", 0, 1, 1);
    return v != 0;
}

// Gated-activation epilogue selected by the flags: 0 none, 1 SwiGLU, 2 GeGLU (tanh form), -1
// both (rejected).
int glu_kind(unsigned flags)
{
    const bool sw = (flags & W4A16_FLAG_SWIGLU) != 0, ge = (flags & W4A16_FLAG_GEGLU) != 0;
    return sw && ge ? -1 : sw ? 1 : ge ? 2 : 0;
}

// Kernel flags of a dense call, checked before anything touches the device: 0, or the status
// of flags that conflict or force a small-M kernel beyond what it takes.  The column-slice
// kernel needs M <= 32 and groups of whole 64-row blocks (`gs` resolved: K for one group); the
// split-K small-M kernel M <= 64.
int check_kernel_flags(int m, int gs, unsigned flags)
{
    // The gated epilogue lives in the tcgen05 kernel (and its split-tile reduction) only; the
    // bfloat16 operand formats in the tcgen05 kernel and, for groups of whole 64-row blocks,
    // the small-M kernels (not the CUDA-core reference kernel).
    const int glu = glu_kind(flags);
    const bool bf16 = (flags & W4A16_FLAG_BF16) != 0;
    if (glu < 0 || (glu > 0 && (flags & (W4A16_FLAG_FORCE_SIMT | W4A16_FLAG_FORCE_MMA |
                                         W4A16_FLAG_FORCE_SLICE))))
        return status_of(STAGE_ARG, W4A16_ARG_FLAGS);
    if (bf16 && (flags & W4A16_FLAG_FORCE_SIMT))
        return status_of(STAGE_ARG, W4A16_ARG_FLAGS);
    if (bf16 && (flags & W4A16_FLAG_FORCE_MMA) && gs % KBLK != 0)
        return status_of(STAGE_UNSUPPORTED, W4A16_ARG_SHAPE);
    const unsigned other = W4A16_FLAG_FORCE_TC | W4A16_FLAG_A_SMEM | W4A16_FLAG_FORCE_SIMT;
    if (flags & W4A16_FLAG_FORCE_SLICE) {
        if (flags & (other | W4A16_FLAG_FORCE_MMA))
            return status_of(STAGE_ARG, W4A16_ARG_FLAGS);
        if (m > SLICE_MAX_ROWS || gs % KBLK != 0)
            return status_of(STAGE_UNSUPPORTED, W4A16_ARG_SHAPE);
    }
    if (flags & W4A16_FLAG_FORCE_MMA) {
        if (flags & other)
            return status_of(STAGE_ARG, W4A16_ARG_FLAGS);
        if (m > decode_max_rows())
            return status_of(STAGE_UNSUPPORTED, W4A16_ARG_SHAPE);
    }
    return 0;
}

// Kernel of a dense call whose flags passed check_kernel_flags: 2 = column-slice small-M
// kernel, 1 = split-K small-M register-fragment kernel, 0 = tcgen05.  By default the
// column-slice kernel takes M <= 32 with whole-block groups when there is at least one
// 16-column slice per SM (measured at 4096x4096: M=1 5.3 us against 8.1 split-K; at
// 4096x12288: 11.9 against 13.5); the split-K one the rest up to 32 rows.
int choose_kernel(int m, int n, int gs, unsigned flags, int num_sms)
{
    if (flags & W4A16_FLAG_FORCE_SLICE)
        return 2;
    if (flags & W4A16_FLAG_FORCE_MMA)
        return 1;
    if (flags & (W4A16_FLAG_FORCE_TC | W4A16_FLAG_A_SMEM | W4A16_FLAG_FORCE_SIMT |
                 W4A16_FLAG_SWIGLU | W4A16_FLAG_GEGLU))
        return 0;
    // bf16 small-M kernels take groups of whole 64-row blocks only.
    if ((flags & W4A16_FLAG_BF16) && gs % KBLK != 0)
        return 0;
    // 9..32 tokens (two or four 8-token tiles, a shallower ring) only while each CTA gets one
    // slice: at N=12288 (3 slices per CTA) the split-K kernel is faster at M=16.
    const int slices = n / SLICE_N;
    const bool fits = m <= 8 || slices <= num_sms * decode_grid_per_sm();
    if (m <= SLICE_MAX_ROWS && gs % KBLK == 0 && slice_default() && slices >= num_sms && fits)
        return 2;
    return m <= decode_rows_default() ? 1 : 0;
}

// Dense plan.  The workspace is carved for the larger tile of the two kernels, so a size
// query answers for whichever kernel the call then picks.
void dense_plan(Plan &pl, int m, int n, int k, unsigned flags, int num_sms, int kernel,
                int tile_cap)
{
    const bool mma = kernel != 0;
    pl.mma = mma;
    pl.slice = kernel == 2;
    pl.a_tmem = (flags & W4A16_FLAG_A_SMEM) == 0;
    const bool mma_ok = m <= decode_max_rows();
    const TcTile tc = pick_tc_tile(m, tile_cap, (flags & W4A16_FLAG_A_SMEM) == 0);
    const int nt_tc = tc.rows;
    const int nt_mma = mma_ok || pl.slice ? pick_nt_mma(m) : nt_tc;
    const int nt_small = nt_tc < nt_mma ? nt_tc : nt_mma;
    pl.nt_max = mma ? nt_mma : nt_tc;
    pl.halves = mma ? 1 : tc.halves;
    pl.nt_half = mma ? nt_mma : tc.half;
    pl.m_tiles = (m + pl.nt_max - 1) / pl.nt_max;
    const long long units = (long long)pl.m_tiles * (n / TILE_N) * (k / KBLK);
    const int ctas = mma ? num_sms * decode_grid_per_sm() : num_sms;
    pl.grid = aligned_grid(pl.m_tiles * (n / TILE_N), k / KBLK, ctas, &pl.split);
    pl.act_rows = pl.slice ? m : pl.halves > 1 ? pl.nt_half : pl.nt_max;
    if (pl.slice) {
        // Consecutive slices per CTA, as evenly as the CTA slots allow (N=12288: 768 slices,
        // 3 each on 256 CTAs); no split-K, so no partial slots or counters are used.
        pl.n_slices = n / SLICE_N;
        pl.slice_per = (pl.n_slices + ctas - 1) / ctas;
        pl.grid = (pl.n_slices + pl.slice_per - 1) / pl.slice_per;
        pl.split = 0;
    }
    // The workspace serves whichever kernel a call picks: counters for the smaller tile
    // height, partial slots for the larger CTA count x tile height.
    pl.tiles_bound = ((m + nt_small - 1) / nt_small) * (n / TILE_N);
    long long slot_rows = (long long)num_sms * nt_tc;
    if (mma_ok) {
        const long long r = (long long)num_sms * decode_ctas_per_sm() * nt_mma;
        if (r > slot_rows)
            slot_rows = r;
    }
    const long long a_bytes = (flags & W4A16_FLAG_ACT_ORDER) ? (long long)m * k * 2 : 0;
    carve(pl, slot_rows, a_bytes);
}

// Token-tile height of a grouped call: the average pairs per active expert plus an eighth
// (segment sizes spread around the average), rounded up to 16 and capped at 192 -- a tile
// per segment, little padding (8 experts, 1024 pairs: 144 rows, +12 % over 192-row tiles).
int pick_nt_grouped(int n_pairs, int n_active)
{
    static const int env = env_int("W4A16_TILE_TOKENS", 16, MAX_TOK, 0) % 16 == 0
                               ? env_int("W4A16_TILE_TOKENS", 16, MAX_TOK, 0)
                               : 0;
    if (env > 0)
        return env;
    const long long avg = (n_pairs + (long long)n_active - 1) / n_active;
    const long long want = round_up(avg + avg / 8, 16);
    return (int)(want < 16 ? 16 : want > 192 ? 192 : want);
}

void grouped_plan(Plan &pl, int n_pairs, int n_active, int n, int k, unsigned flags, int num_sms)
{
    pl.mma = false;
    pl.a_tmem = (flags & W4A16_FLAG_A_SMEM) == 0;
    pl.nt_max = pick_nt_grouped(n_pairs, n_active);
    pl.act_rows = pl.nt_max;
    pl.halves = 1;
    pl.nt_half = pl.nt_max;
    pl.m_tiles = 0;
    pl.tiles_bound = ((n_pairs + pl.nt_max - 1) / pl.nt_max + n_active) * (n / TILE_N);
    pl.grid = num_sms;
    carve(pl, (long long)num_sms * pl.nt_max, (long long)n_pairs * k * 2);
}

// Block-routed MoE plan: the sorted activation copy has max_padded rows cut into at most
// seg_cap segments (one per run of blocks of one expert); the token tile follows the average
// rows per expert.  After the activation copy the workspace holds the routing the device
// builds: ex_off [seg_cap + 1], ex_ids [seg_cap], ex_pairs [max_padded].
struct MoePlan {
    int seg_cap;
    long long off_off, ids_off, pairs_off, total;
};

void moe_blocks_plan(Plan &pl, MoePlan &mp, int max_padded, int block_size, int n_experts, int n,
                     int k, unsigned flags, int num_sms)
{
    const int n_blocks = max_padded / block_size;
    mp.seg_cap = n_blocks < MAX_SEGMENTS ? n_blocks : MAX_SEGMENTS;
    pl.mma = false;
    pl.a_tmem = (flags & W4A16_FLAG_A_SMEM) == 0;
    const int per = n_experts < mp.seg_cap ? n_experts : mp.seg_cap;
    pl.nt_max = pick_nt_grouped(max_padded, per > 0 ? per : 1);
    pl.act_rows = pl.nt_max;
    pl.halves = 1;
    pl.nt_half = pl.nt_max;
    pl.m_tiles = 0;
    pl.tiles_bound = ((max_padded + pl.nt_max - 1) / pl.nt_max + mp.seg_cap) * (n / TILE_N);
    pl.grid = num_sms;
    carve(pl, (long long)num_sms * pl.nt_max, (long long)max_padded * k * 2);
    mp.off_off = pl.total;
    mp.ids_off = round_up(mp.off_off + 4LL * (mp.seg_cap + 1), 256);
    mp.pairs_off = round_up(mp.ids_off + 4LL * mp.seg_cap, 256);
    mp.total = round_up(mp.pairs_off + 4LL * max_padded, 256);
}

// Size checks of the block-routed interface (marlin.rs, `MarlinMoeRawLaunchArgs::validate`:
// moe_block_size in {8, 16, 32, 48, 64}, positive top_k and prob_m, prob_m * top_k within
// int32) plus this library's capacity: whole blocks, at most MOE_MAX_BLOCKS of them.
int check_moe_sizes(int max_padded, int block_size, int top_k, int prob_m, int n_experts)
{
    if (!(block_size == 8 || block_size == 16 || block_size == 32 || block_size == 48 ||
          block_size == 64))
        return status_of(STAGE_ARG, W4A16_ARG_SCHEDULE);
    if (top_k <= 0 || prob_m <= 0 || n_experts <= 0 || max_padded <= 0 ||
        max_padded % block_size != 0)
        return status_of(STAGE_ARG, W4A16_ARG_SCHEDULE);
    if ((long long)prob_m * top_k > 0x7FFFFFFFLL)
        return status_of(STAGE_ARG, W4A16_ARG_OVERFLOW);
    if (max_padded / block_size > MOE_MAX_BLOCKS)
        return status_of(STAGE_UNSUPPORTED, W4A16_ARG_SCHEDULE);
    return 0;
}

void fill_params(GemmParams &p, const Plan &pl, int m, int n, int k, int group_size)
{
    memset(&p, 0, sizeof(p));
    p.limit_ns = WAIT_LIMIT_NS;
    p.m = m;
    p.n = n;
    p.k = k;
    p.group_size = group_size == -1 ? k : group_size;
    p.num_groups = num_groups(k, group_size);
    p.nt_max = pl.nt_max;
    p.m_tiles = pl.m_tiles;
    p.n_tiles = n / TILE_N;
    p.kblocks = k / KBLK;
    p.stages = pl.stages;
    p.stage_bytes = pl.stage_bytes;
    p.kbs = pl.kbs;
    p.act_kb_bytes = pl.act_kb_bytes;
    p.packed_off = pl.packed_off;
    p.scales_off = pl.scales_off;
    p.zeros_off = pl.zeros_off;
    p.sg_box = pl.sg_box;
    p.acc_bufs = pl.acc_bufs;
    p.halves = pl.halves > 1 ? pl.halves : 1;
    p.nt_half = pl.halves > 1 ? pl.nt_half : pl.nt_max;
    p.acc_col0 = pl.acc_col0;
    p.tmem_cols = pl.tmem_cols;
    p.a_slots = pl.a_slots;
    p.seg_smem_off = pl.seg_off;
    p.epi_smem_off = pl.epi_off;
    p.static_weights = 0;
    p.split = pl.split;
    p.n_slices = pl.n_slices;
    p.slice_per = pl.slice_per;
    p.tile_words = TILE_WORDS;
    p.tile_bytes = TILE_BYTES;
}

// Tensor maps of one launch: activations (3-D, swizzled) and the scale / zero rows.  With no
// zero points the zero map is a copy of the scale map that the kernels never read.
int encode_maps(const Plan &pl, const void *act, int rows, int k, int ld, const void *scales,
                const void *zeros, int g_rows, int n, CUtensorMap *ma, CUtensorMap *ms,
                CUtensorMap *mz)
{
    const int box_n = pl.slice ? SLICE_N : TILE_N;
    int err = encode_act_map(ma, act, rows, k, ld, pl.act_rows, pl.kbs);
    if (err == cudaSuccess)
        err = encode_group_map(ms, scales, g_rows, n, pl.sg_box, box_n);
    if (err == cudaSuccess) {
        if (zeros)
            err = encode_group_map(mz, zeros, g_rows, n, pl.sg_box, box_n);
        else
            *mz = *ms;
    }
    return err;
}

} // namespace

namespace w4 {

size_t dense_workspace_size(int m, int n, int k, int group_size, unsigned flags, int num_sms,
                            int tile_cap)
{
    if (m < 0 || n <= 0 || k <= 0 || n % 256 != 0 || k % 128 != 0 || num_groups(k, group_size) < 0)
        return 0;
    if (num_sms <= 0 && sm_count(&num_sms) != cudaSuccess)
        return 0;
    Plan pl;
    dense_plan(pl, m > 0 ? m : 1, n, k, flags, num_sms, 0, tile_cap);
    return (size_t)pl.total;
}

int dense_gemm(const void *a, int lda, const int32_t *b_packed, void *c, int ldc,
               const void *scales, const void *zeros, const int32_t *g_idx, const int32_t *perm,
               void *workspace, size_t workspace_bytes, int m, int n, int k, int group_size,
               int weight_type, unsigned flags, cudaStream_t stream, int tile_cap)
{
    int st = check_weights(b_packed, scales, zeros, n, k, group_size, weight_type, flags);
    if (st)
        return st;
    if (m < 0)
        return status_of(STAGE_ARG, W4A16_ARG_SHAPE);
    const bool act_order = (flags & W4A16_FLAG_ACT_ORDER) != 0;
    if (act_order != (g_idx != nullptr && perm != nullptr) || ((g_idx != nullptr) != (perm != nullptr)))
        return status_of(STAGE_ARG, W4A16_ARG_FLAGS);
    if (m == 0)
        return 0; // empty input: nothing to compute
    if (!a || !c || !workspace)
        return status_of(STAGE_ARG, W4A16_ARG_NULL);
    const int glu = glu_kind(flags);
    if (glu < 0)
        return status_of(STAGE_ARG, W4A16_ARG_FLAGS);
    if (lda < k || ldc < (glu > 0 ? n / 2 : n))
        return status_of(STAGE_ARG, W4A16_ARG_SHAPE);
    if (lda % 8 != 0 || ldc % 8 != 0 || !aligned(a, 16) || !aligned(c, 16) ||
        !aligned(workspace, 256) || (g_idx && !aligned(g_idx, 4)) || (perm && !aligned(perm, 4)))
        return status_of(STAGE_ARG, W4A16_ARG_ALIGN);
    if ((long long)m * lda > (1LL << 40) || (long long)m * ldc > (1LL << 40))
        return status_of(STAGE_ARG, W4A16_ARG_OVERFLOW);
    if ((flags & W4A16_FLAG_FORCE_SIMT) && m > (1 << 20))
        return status_of(STAGE_UNSUPPORTED, W4A16_ARG_SHAPE);

    const int gs_resolved = group_size == -1 ? k : group_size;
    st = check_kernel_flags(m, gs_resolved, flags);
    if (st)
        return st;
    st = check_fp8_flags(weight_type, flags);
    if (st)
        return st;

    int num_sms = 0;
    int err = sm_count(&num_sms);
    if (err != cudaSuccess)
        return status_of(STAGE_RESOURCE, err);
    // FP8 weights: the column-slice kernel where the 4-bit rule picks it, else the tcgen05
    // kernel (the split-K small-M kernel is 4-bit only).
    int kernel = choose_kernel(m, n, gs_resolved, flags, num_sms);
    if (weight_type == W4A16_TYPE_FE4M3) {
        // FP8 column slices: two stages of their doubled code bytes fit up to 16 tokens.  By
        // default they take M <= 16 with at least one slice per SM (measured at N = 4096 …
        // 12288: 4.8-14.6 us against 11.1-22.0 us on the tcgen05 kernel), else the tcgen05
        // kernel (the split-K small-M kernel is 4-bit only).
        if (m > 16 && (flags & W4A16_FLAG_FORCE_SLICE))
            return status_of(STAGE_UNSUPPORTED, W4A16_ARG_SHAPE);
        const unsigned tc_flags = W4A16_FLAG_FORCE_TC | W4A16_FLAG_A_SMEM | W4A16_FLAG_SWIGLU |
                                  W4A16_FLAG_GEGLU;
        if (!(flags & W4A16_FLAG_FORCE_SLICE))
            kernel = (!(flags & tc_flags) && m <= 16 && n / SLICE_N >= num_sms && slice_default()) ? 2 : 0;
    }
    Plan pl;
    dense_plan(pl, m, n, k, flags, num_sms, kernel, tile_cap);
    if (workspace_bytes < (size_t)pl.total)
        return status_of(STAGE_ARG, W4A16_ARG_WORKSPACE);
    const int g = num_groups(k, group_size);
    plan_tmem(pl);
    pl.tile_bytes = tile_bytes_of(weight_type);
    err = plan_smem(pl, false, zeros != nullptr, group_size == -1 ? k : group_size, g);
    if (err != cudaSuccess)
        return status_of(STAGE_RESOURCE, err);

    char *ws = static_cast<char *>(workspace);
    GemmParams p;
    fill_params(p, pl, m, n, k, group_size);
    set_weight_type(p, weight_type, flags);
    p.b = b_packed;
    p.scales = static_cast<const __half *>(scales);
    p.zeros = static_cast<const __half *>(zeros);
    p.c = static_cast<__half *>(c);
    p.ldc = ldc;
    p.static_weights = (flags & W4A16_FLAG_STATIC_WEIGHTS) ? 1 : 0;
    p.glu = glu;
    // Tile order: walk token tiles outermost when the activations outweigh the weights and
    // would not stay in L2 while every column tile passes over them (e.g. M=4096, K=11008:
    // 90 MB of A, read 4.6 times from DRAM column-tile-major).
    {
        const long long a_bytes = (long long)m * k * 2, w_bytes = (long long)k * n / 2;
        p.m_outer = (a_bytes > w_bytes && a_bytes * 2 > l2_bytes()) ? 1 : 0;
    }
    p.status = reinterpret_cast<int *>(ws);
    p.counters = reinterpret_cast<int *>(ws + pl.counters_off);
    p.partials = reinterpret_cast<float *>(ws + pl.partials_off);

    const __half *a_src = static_cast<const __half *>(a);
    int a_ld = lda;
    if (act_order) {
        __half *a_perm = reinterpret_cast<__half *>(ws + pl.a_off);
        err = launch_gather_cols(a_src, lda, perm, g_idx, p.group_size, a_perm, m, k, p.status,
                                 stream);
        if (err != cudaSuccess)
            return status_of(STAGE_LAUNCH, err);
        a_src = a_perm;
        a_ld = k;
    }
    if (flags & W4A16_FLAG_FORCE_SIMT)
        return launch_status(launch_gemm_simt(p, a_src, a_ld, stream));

    CUtensorMap ma, ms, mz;
    err = encode_maps(pl, a_src, m, k, a_ld, scales, zeros, g, n, &ma, &ms, &mz);
    if (err != cudaSuccess)
        return status_of(STAGE_RESOURCE, err);
    GemmConfig cfg{pl.grid, pl.smem_bytes, pl.a_tmem};
    if (pl.slice) {
        CUtensorMap mw;
        err = encode_slice_weight_map(&mw, b_packed, n, k, pl.kbs, p.w8 != 0);
        if (err != cudaSuccess)
            return status_of(STAGE_RESOURCE, err);
        return launch_status(launch_slice(p, ma, mw, ms, mz, cfg, stream));
    }
    if (pl.mma)
        return launch_status(launch_decode(p, ma, ms, mz, cfg, stream));
    return launch_status(launch_gemm(p, ma, ms, mz, cfg, stream));
}

} // namespace w4

extern "C" {

int w4a16_abi_version(void)
{
    return W4A16_ABI_VERSION;
}

const char *w4a16_status_string(int status)
{
    switch (status >> 16) {
    case 0:
        return status == 0 ? "ok" : "unknown";
    case STAGE_ARG:
        return "invalid-argument";
    case STAGE_UNSUPPORTED:
        return "unsupported-shape";
    case STAGE_RESOURCE:
        return "device-resource";
    case STAGE_LAUNCH:
        return "kernel-launch";
    case 7:
        return "device-error";
    default:
        return "unknown";
    }
}

int w4_repack(const int32_t *qweight, const int32_t *perm, int32_t *b_packed, int32_t *status, int k,
              int n, cudaStream_t stream)
{
    if (k <= 0 || n <= 0)
        return status_of(STAGE_ARG, W4A16_ARG_SHAPE);
    if (!qweight || !b_packed)
        return status_of(STAGE_ARG, W4A16_ARG_NULL);
    if (!aligned(qweight, 16) || !aligned(b_packed, 16) || (perm && !aligned(perm, 4)) ||
        (status && !aligned(status, 4)))
        return status_of(STAGE_ARG, W4A16_ARG_ALIGN);
    if (k % 128 != 0 || n % 256 != 0)
        return status_of(STAGE_UNSUPPORTED, W4A16_ARG_SHAPE);
    const long long bytes = (long long)k * n / 2;
    const char *qa = reinterpret_cast<const char *>(qweight);
    const char *ob = reinterpret_cast<const char *>(b_packed);
    if (qa < ob + bytes && ob < qa + bytes)
        return status_of(STAGE_ARG, W4A16_ARG_FLAGS);
    return launch_status(launch_repack(qweight, perm, b_packed, status, k, n, stream));
}

int w8_repack(const int32_t *qweight, int32_t *b_packed, int k, int n, cudaStream_t stream)
{
    if (k <= 0 || n <= 0)
        return status_of(STAGE_ARG, W4A16_ARG_SHAPE);
    if (!qweight || !b_packed)
        return status_of(STAGE_ARG, W4A16_ARG_NULL);
    if (!aligned(qweight, 16) || !aligned(b_packed, 16))
        return status_of(STAGE_ARG, W4A16_ARG_ALIGN);
    if (k % 128 != 0 || n % 256 != 0)
        return status_of(STAGE_UNSUPPORTED, W4A16_ARG_SHAPE);
    const long long bytes = (long long)k * n;
    const char *qa = reinterpret_cast<const char *>(qweight);
    const char *ob = reinterpret_cast<const char *>(b_packed);
    if (qa < ob + bytes && ob < qa + bytes)
        return status_of(STAGE_ARG, W4A16_ARG_FLAGS);
    return launch_status(launch_repack_fp8(qweight, b_packed, k, n, stream));
}

int w8_unpack(const int32_t *b_packed, int32_t *qweight, int k, int n, cudaStream_t stream)
{
    if (k <= 0 || n <= 0)
        return status_of(STAGE_ARG, W4A16_ARG_SHAPE);
    if (!qweight || !b_packed)
        return status_of(STAGE_ARG, W4A16_ARG_NULL);
    if (!aligned(qweight, 16) || !aligned(b_packed, 16))
        return status_of(STAGE_ARG, W4A16_ARG_ALIGN);
    if (k % 128 != 0 || n % 256 != 0)
        return status_of(STAGE_UNSUPPORTED, W4A16_ARG_SHAPE);
    const long long bytes = (long long)k * n;
    const char *qa = reinterpret_cast<const char *>(qweight);
    const char *ob = reinterpret_cast<const char *>(b_packed);
    if (qa < ob + bytes && ob < qa + bytes)
        return status_of(STAGE_ARG, W4A16_ARG_FLAGS);
    return launch_status(launch_unpack_fp8(b_packed, qweight, k, n, stream));
}

int w4_gate_up_interleave(const void *src, void *dst, int rows, int n2, int elem_bytes,
                          cudaStream_t stream)
{
    if (rows <= 0 || n2 <= 0 || n2 % 32 != 0 || (elem_bytes != 2 && elem_bytes != 4))
        return status_of(STAGE_ARG, W4A16_ARG_SHAPE);
    if (!src || !dst)
        return status_of(STAGE_ARG, W4A16_ARG_NULL);
    if (!aligned(src, elem_bytes) || !aligned(dst, elem_bytes))
        return status_of(STAGE_ARG, W4A16_ARG_ALIGN);
    const long long bytes = (long long)rows * n2 * elem_bytes;
    if (bytes > (1LL << 40))
        return status_of(STAGE_ARG, W4A16_ARG_OVERFLOW);
    const char *sa = static_cast<const char *>(src);
    const char *da = static_cast<const char *>(dst);
    if (sa < da + bytes && da < sa + bytes)
        return status_of(STAGE_ARG, W4A16_ARG_FLAGS);
    return launch_status(launch_gate_up_interleave(src, dst, rows, n2, elem_bytes, stream));
}

int w4_unpack(const int32_t *b_packed, int32_t *qweight, int k, int n, cudaStream_t stream)
{
    if (k <= 0 || n <= 0)
        return status_of(STAGE_ARG, W4A16_ARG_SHAPE);
    if (!qweight || !b_packed)
        return status_of(STAGE_ARG, W4A16_ARG_NULL);
    if (!aligned(qweight, 16) || !aligned(b_packed, 16))
        return status_of(STAGE_ARG, W4A16_ARG_ALIGN);
    if (k % 128 != 0 || n % 256 != 0)
        return status_of(STAGE_UNSUPPORTED, W4A16_ARG_SHAPE);
    const long long bytes = (long long)k * n / 2;
    const char *qa = reinterpret_cast<const char *>(qweight);
    const char *ob = reinterpret_cast<const char *>(b_packed);
    if (qa < ob + bytes && ob < qa + bytes)
        return status_of(STAGE_ARG, W4A16_ARG_FLAGS);
    return launch_status(launch_unpack(b_packed, qweight, k, n, stream));
}

size_t w4a16_workspace_size(int m, int n, int k, int group_size, unsigned flags, int num_sms)
{
    return w4::dense_workspace_size(m, n, k, group_size, flags, num_sms, w4::MAX_TOK);
}

size_t w4a16_grouped_workspace_size(int n_pairs, int n_active, int n, int k, int group_size,
                                    unsigned flags, int num_sms)
{
    if (n_pairs <= 0 || n_active <= 0 || n_active > W4A16_MAX_SEGMENTS || n <= 0 || k <= 0 ||
        n % 256 != 0 || k % 128 != 0 || num_groups(k, group_size) < 0)
        return 0;
    if (num_sms <= 0 && sm_count(&num_sms) != cudaSuccess)
        return 0;
    Plan pl;
    grouped_plan(pl, n_pairs, n_active, n, k, flags, num_sms);
    return (size_t)pl.total;
}

int w4a16_gemm(const void *a, int lda, const int32_t *b_packed, void *c, int ldc, const void *scales,
               const void *zeros, const int32_t *g_idx, const int32_t *perm, void *workspace,
               size_t workspace_bytes, int m, int n, int k, int group_size, int weight_type,
               unsigned flags, cudaStream_t stream)
{
    return w4::dense_gemm(a, lda, b_packed, c, ldc, scales, zeros, g_idx, perm, workspace,
                          workspace_bytes, m, n, k, group_size, weight_type, flags, stream,
                          w4::MAX_TOK);
}
int w4a16_kernel_for(int m, int n, int k, int group_size, unsigned flags, int num_sms)
{
    if (m <= 0 || n <= 0 || k <= 0 || n % 256 != 0 || k % 128 != 0 || num_groups(k, group_size) < 0)
        return -1;
    const int gs_resolved = group_size == -1 ? k : group_size;
    if (check_kernel_flags(m, gs_resolved, flags) != 0)
        return -1;
    if (num_sms <= 0 && sm_count(&num_sms) != cudaSuccess)
        return -1;
    return choose_kernel(m, n, gs_resolved, flags, num_sms);
}

int w4a16_gemm_grouped(const void *a, int lda, const int32_t *b_packed_stack, void *y, int ldy,
                       const void *scales_stack, const void *zeros_stack, const int32_t *ex_ids,
                       const int32_t *ex_off, const int32_t *ex_pairs, const int32_t *pair_tok,
                       int n_active, int n_experts, int n_pairs, int n_tokens, int n, int k,
                       int group_size, int weight_type, unsigned flags, void *workspace,
                       size_t workspace_bytes, cudaStream_t stream)
{
    int st = check_weights(b_packed_stack, scales_stack, zeros_stack, n, k, group_size, weight_type,
                           flags);
    if (st)
        return st;
    if (flags & (W4A16_FLAG_ACT_ORDER | W4A16_FLAG_FORCE_SIMT | W4A16_FLAG_FORCE_MMA |
                 W4A16_FLAG_FORCE_SLICE))
        return status_of(STAGE_ARG, W4A16_ARG_FLAGS);
    const int glu = glu_kind(flags);
    if (glu < 0)
        return status_of(STAGE_ARG, W4A16_ARG_FLAGS);
    st = check_fp8_flags(weight_type, flags);
    if (st)
        return st;
    if (n_active <= 0 || n_active > W4A16_MAX_SEGMENTS || n_experts <= 0 || n_pairs <= 0 ||
        n_tokens <= 0 || n_active > n_experts)
        return status_of(STAGE_ARG, W4A16_ARG_SCHEDULE);
    if (!a || !y || !workspace || !ex_ids || !ex_off || !ex_pairs || !pair_tok)
        return status_of(STAGE_ARG, W4A16_ARG_NULL);
    if (lda < k || ldy < (glu > 0 ? n / 2 : n))
        return status_of(STAGE_ARG, W4A16_ARG_SHAPE);
    if (lda % 8 != 0 || ldy % 8 != 0 || !aligned(a, 16) || !aligned(y, 16) ||
        !aligned(workspace, 256) || !aligned(ex_ids, 4) || !aligned(ex_off, 4) ||
        !aligned(ex_pairs, 4) || !aligned(pair_tok, 4))
        return status_of(STAGE_ARG, W4A16_ARG_ALIGN);
    if ((long long)n_tokens * lda > (1LL << 40) || (long long)n_pairs * ldy > (1LL << 40) ||
        (long long)n_experts * k * n / 8 > (1LL << 40))
        return status_of(STAGE_ARG, W4A16_ARG_OVERFLOW);

    int num_sms = 0;
    int err = sm_count(&num_sms);
    if (err != cudaSuccess)
        return status_of(STAGE_RESOURCE, err);
    Plan pl;
    grouped_plan(pl, n_pairs, n_active, n, k, flags, num_sms);
    if (workspace_bytes < (size_t)pl.total)
        return status_of(STAGE_ARG, W4A16_ARG_WORKSPACE);
    const int g = num_groups(k, group_size);
    plan_tmem(pl);
    pl.tile_bytes = tile_bytes_of(weight_type);
    err = plan_smem(pl, true, zeros_stack != nullptr, group_size == -1 ? k : group_size,
                    g * n_experts);
    if (err != cudaSuccess)
        return status_of(STAGE_RESOURCE, err);

    char *ws = static_cast<char *>(workspace);
    GemmParams p;
    fill_params(p, pl, n_pairs, n, k, group_size);
    set_weight_type(p, weight_type, flags);
    p.b = b_packed_stack;
    p.scales = static_cast<const __half *>(scales_stack);
    p.zeros = static_cast<const __half *>(zeros_stack);
    p.c = static_cast<__half *>(y);
    p.ldc = ldy;
    p.glu = glu;
    p.status = reinterpret_cast<int *>(ws);
    p.counters = reinterpret_cast<int *>(ws + pl.counters_off);
    p.partials = reinterpret_cast<float *>(ws + pl.partials_off);
    p.ex_off = ex_off;
    p.ex_ids = ex_ids;
    p.ex_pairs = ex_pairs;
    p.n_active = n_active;
    p.n_experts = n_experts;
    p.n_pairs = n_pairs;
    p.n_rows = n_pairs;
    p.b_expert_words = (long long)k * n / (p.w8 ? 4 : 8);
    p.s_expert_elems = (long long)p.num_groups * n;

    __half *a_sorted = reinterpret_cast<__half *>(ws + pl.a_off);
    err = launch_gather_rows(static_cast<const __half *>(a), lda, ex_pairs, pair_tok, a_sorted,
                             n_pairs, n_tokens, k, p.status, stream);
    if (err != cudaSuccess)
        return status_of(STAGE_LAUNCH, err);
    CUtensorMap ma, ms, mz;
    err = encode_maps(pl, a_sorted, n_pairs, k, k, scales_stack, zeros_stack, g * n_experts, n, &ma,
                      &ms, &mz);
    if (err != cudaSuccess)
        return status_of(STAGE_RESOURCE, err);
    GemmConfig cfg{pl.grid, pl.smem_bytes, pl.a_tmem};
    return launch_status(launch_gemm(p, ma, ms, mz, cfg, stream));
}

size_t w4a16_moe_blocks_workspace_size(int max_padded, int moe_block_size, int n_experts, int n,
                                       int k, int group_size, unsigned flags, int num_sms)
{
    if (check_moe_sizes(max_padded, moe_block_size, 1, 1, n_experts) != 0 || n <= 0 || k <= 0 ||
        n % 256 != 0 || k % 128 != 0 || num_groups(k, group_size) < 0)
        return 0;
    if (num_sms <= 0 && sm_count(&num_sms) != cudaSuccess)
        return 0;
    Plan pl;
    MoePlan mp;
    moe_blocks_plan(pl, mp, max_padded, moe_block_size, n_experts, n, k, flags, num_sms);
    return (size_t)mp.total;
}

int w4a16_gemm_moe_blocks(const void *a, int lda, const int32_t *b_packed_stack, void *c, int ldc,
                          const void *scales_stack, const void *zeros_stack,
                          const int32_t *sorted_token_ids, const int32_t *expert_ids,
                          const int32_t *num_tokens_past_padded, const float *topk_weights,
                          int max_padded, int moe_block_size, int top_k, int mul_topk_weights,
                          int is_ep, int n_experts, int prob_m, int n, int k, int group_size,
                          int weight_type, unsigned flags, void *workspace, size_t workspace_bytes,
                          cudaStream_t stream)
{
    int st = check_weights(b_packed_stack, scales_stack, zeros_stack, n, k, group_size, weight_type,
                           flags);
    if (st)
        return st;
    if (flags & (W4A16_FLAG_ACT_ORDER | W4A16_FLAG_FORCE_SIMT | W4A16_FLAG_FORCE_MMA |
                 W4A16_FLAG_FORCE_SLICE))
        return status_of(STAGE_ARG, W4A16_ARG_FLAGS);
    const int glu = glu_kind(flags);
    if (glu < 0 || (mul_topk_weights != 0 && topk_weights == nullptr) ||
        (mul_topk_weights != 0 && mul_topk_weights != 1) || (is_ep != 0 && is_ep != 1))
        return status_of(STAGE_ARG, W4A16_ARG_FLAGS);
    st = check_fp8_flags(weight_type, flags);
    if (st)
        return st;
    st = check_moe_sizes(max_padded, moe_block_size, top_k, prob_m, n_experts);
    if (st)
        return st;
    if (!a || !c || !workspace || !sorted_token_ids || !expert_ids || !num_tokens_past_padded)
        return status_of(STAGE_ARG, W4A16_ARG_NULL);
    if (lda < k || ldc < (glu > 0 ? n / 2 : n))
        return status_of(STAGE_ARG, W4A16_ARG_SHAPE);
    if (lda % 8 != 0 || ldc % 8 != 0 || !aligned(a, 16) || !aligned(c, 16) ||
        !aligned(workspace, 256) || !aligned(sorted_token_ids, 4) || !aligned(expert_ids, 4) ||
        !aligned(num_tokens_past_padded, 4) || (topk_weights && !aligned(topk_weights, 4)))
        return status_of(STAGE_ARG, W4A16_ARG_ALIGN);
    const long long n_ids = (long long)prob_m * top_k;
    if (n_ids * ldc > (1LL << 40) || (long long)prob_m * lda > (1LL << 40) ||
        (long long)n_experts * k * n / 8 > (1LL << 40) || (long long)max_padded * k > (1LL << 40))
        return status_of(STAGE_ARG, W4A16_ARG_OVERFLOW);

    int num_sms = 0;
    int err = sm_count(&num_sms);
    if (err != cudaSuccess)
        return status_of(STAGE_RESOURCE, err);
    Plan pl;
    MoePlan mp;
    moe_blocks_plan(pl, mp, max_padded, moe_block_size, n_experts, n, k, flags, num_sms);
    if (workspace_bytes < (size_t)mp.total)
        return status_of(STAGE_ARG, W4A16_ARG_WORKSPACE);
    const int g = num_groups(k, group_size);
    plan_tmem(pl);
    pl.tile_bytes = tile_bytes_of(weight_type);
    err = plan_smem(pl, true, zeros_stack != nullptr, group_size == -1 ? k : group_size,
                    g * n_experts);
    if (err != cudaSuccess)
        return status_of(STAGE_RESOURCE, err);

    char *ws = static_cast<char *>(workspace);
    int32_t *ex_off = reinterpret_cast<int32_t *>(ws + mp.off_off);
    int32_t *ex_ids = reinterpret_cast<int32_t *>(ws + mp.ids_off);
    int32_t *ex_pairs = reinterpret_cast<int32_t *>(ws + mp.pairs_off);
    GemmParams p;
    fill_params(p, pl, max_padded, n, k, group_size);
    set_weight_type(p, weight_type, flags);
    p.b = b_packed_stack;
    p.scales = static_cast<const __half *>(scales_stack);
    p.zeros = static_cast<const __half *>(zeros_stack);
    p.c = static_cast<__half *>(c);
    p.ldc = ldc;
    p.glu = glu;
    p.status = reinterpret_cast<int *>(ws);
    p.counters = reinterpret_cast<int *>(ws + pl.counters_off);
    p.partials = reinterpret_cast<float *>(ws + pl.partials_off);
    p.ex_off = ex_off;
    p.ex_ids = ex_ids;
    p.ex_pairs = ex_pairs;
    p.n_active = mp.seg_cap;
    p.n_experts = n_experts;
    p.n_pairs = (int)n_ids;
    p.n_rows = max_padded;
    p.skip_sentinel = 1;
    p.row_weight = mul_topk_weights ? topk_weights : nullptr;
    p.b_expert_words = (long long)k * n / (p.w8 ? 4 : 8);
    p.s_expert_elems = (long long)p.num_groups * n;

    err = launch_moe_route(sorted_token_ids, expert_ids, num_tokens_past_padded, max_padded,
                           moe_block_size, (int)n_ids, n_experts, is_ep, mp.seg_cap, ex_off, ex_ids,
                           ex_pairs, p.status, stream);
    if (err != cudaSuccess)
        return status_of(STAGE_LAUNCH, err);
    __half *a_sorted = reinterpret_cast<__half *>(ws + pl.a_off);
    err = launch_moe_gather(static_cast<const __half *>(a), lda, ex_off + mp.seg_cap, ex_pairs, top_k,
                            a_sorted, max_padded, k, stream);
    if (err != cudaSuccess)
        return status_of(STAGE_LAUNCH, err);
    CUtensorMap ma, ms, mz;
    err = encode_maps(pl, a_sorted, max_padded, k, k, scales_stack, zeros_stack, g * n_experts, n,
                      &ma, &ms, &mz);
    if (err != cudaSuccess)
        return status_of(STAGE_RESOURCE, err);
    GemmConfig cfg{pl.grid, pl.smem_bytes, pl.a_tmem};
    return launch_status(launch_gemm(p, ma, ms, mz, cfg, stream));
}

int w4a16_moe_align_block_size(const int32_t *topk_ids, int m, int top_k, int n_experts,
                               int block_size, int capacity, int32_t *sorted_token_ids,
                               int32_t *expert_ids)
{
    if (m <= 0 || top_k <= 0 || n_experts <= 0 || block_size <= 0 || capacity < 0)
        return -1;
    const long long n_ids_ll = (long long)m * top_k;
    if (n_ids_ll > 0x7FFFFFFF)
        return -1;
    const int n_ids = (int)n_ids_ll;
    if (!topk_ids || !sorted_token_ids || !expert_ids)
        return -1;
    // Counting sort: ids per expert, each expert's run padded to whole blocks, experts in
    // order, ids in increasing order inside a run; padding rows hold the sentinel n_ids.
    long long *start = static_cast<long long *>(calloc((size_t)n_experts + 1, sizeof(long long)));
    if (!start)
        return -1;
    int ret = -1;
    for (int i = 0; i < n_ids; ++i) {
        const int e = topk_ids[i];
        if (e < 0 || e >= n_experts)
            goto out;
        start[e + 1]++;
    }
    for (int e = 0; e < n_experts; ++e)
        start[e + 1] = start[e] + (start[e + 1] + block_size - 1) / block_size * block_size;
    if (start[n_experts] > capacity)
        goto out;
    {
        long long *cursor = static_cast<long long *>(malloc(sizeof(long long) * (size_t)n_experts));
        if (!cursor)
            goto out;
        for (long long r = 0; r < start[n_experts]; ++r)
            sorted_token_ids[r] = n_ids;
        for (int e = 0; e < n_experts; ++e) {
            cursor[e] = start[e];
            for (long long b = start[e] / block_size; b < start[e + 1] / block_size; ++b)
                expert_ids[b] = e;
        }
        for (int i = 0; i < n_ids; ++i)
            sorted_token_ids[cursor[topk_ids[i]]++] = i;
        free(cursor);
        ret = (int)start[n_experts];
    }
out:
    free(start);
    return ret;
}

int w4a16_csr_from_token_routes(int n_expert, int n_tokens, int experts_per_token,
                                const int32_t *selected, int32_t *ex_ids, int32_t *ex_off,
                                int32_t *ex_pairs, int32_t *pair_tok)
{
    if (n_expert <= 0 || n_tokens <= 0 || experts_per_token <= 0)
        return -1;
    const long long n_pairs_ll = (long long)n_tokens * experts_per_token;
    if (n_pairs_ll > 0x7FFFFFFF)
        return -1;
    const int n_pairs = (int)n_pairs_ll;
    if (!selected || !ex_ids || !ex_off || !ex_pairs || !pair_tok)
        return -1;
    // Counting sort of pair ids by expert: segment starts are the prefix sums of the counts;
    // pairs keep their relative order inside a segment.
    int *start = static_cast<int *>(calloc((size_t)n_expert + 1, sizeof(int)));
    if (!start)
        return -1;
    for (int p = 0; p < n_pairs; ++p) {
        const int e = selected[p];
        if (e < 0 || e >= n_expert) {
            free(start);
            return -1;
        }
        start[e + 1]++;
    }
    for (int e = 0; e < n_expert; ++e)
        start[e + 1] += start[e];
    int active = 0;
    for (int e = 0; e < n_expert; ++e)
        if (start[e + 1] > start[e]) {
            ex_ids[active] = e;
            ex_off[active] = start[e];
            ++active;
        }
    ex_off[active] = n_pairs;
    for (int p = 0; p < n_pairs; ++p) {
        ex_pairs[start[selected[p]]++] = p;
        pair_tok[p] = p / experts_per_token;
    }
    free(start);
    return active;
}

int w4a16_status(void *workspace, int *device_bits, cudaStream_t stream)
{
    if (!workspace || !device_bits)
        return status_of(STAGE_ARG, W4A16_ARG_NULL);
    int bits = 0;
    cudaError_t err = cudaMemcpyAsync(&bits, workspace, sizeof(int), cudaMemcpyDeviceToHost, stream);
    if (err == cudaSuccess)
        err = cudaStreamSynchronize(stream);
    if (err == cudaSuccess)
        err = cudaMemsetAsync(workspace, 0, sizeof(int), stream);
    if (err == cudaSuccess)
        err = cudaStreamSynchronize(stream);
    if (err != cudaSuccess)
        return status_of(STAGE_RESOURCE, err);
    *device_bits = bits;
    return 0;
}

int w4a16_selftest_timeout(void *workspace, long long limit_ns, cudaStream_t stream)
{
    if (!workspace)
        return status_of(STAGE_ARG, W4A16_ARG_NULL);
    if (!aligned(workspace, 256))
        return status_of(STAGE_ARG, W4A16_ARG_ALIGN);
    if (limit_ns <= 0 || limit_ns > 10000000000LL)
        return status_of(STAGE_ARG, W4A16_ARG_SHAPE);
    return launch_status(launch_selftest_timeout(static_cast<int *>(workspace),
                                                 (unsigned long long)limit_ns, stream));
}

} // extern "C"
