// w4a16_common.cuh -- device code shared by the W4A16 GEMM kernels: dequantisation of a tile
// word, the data-parallel + stream-K work schedule, the grouped schedule table, the TMA
// producer and the fixed-order split-K reduction.
#pragma once

#include <cuda_bf16.h>

#include "ptx.cuh"
#include "w4a16_internal.h"
#include "w4a16.h"

namespace w4 {

// ---------------------------------------------------------------------------------------
// Dequantisation of one tile word (8 codes, 4 pairs) into 4 fp16 pairs (q - z) * s.
// Pair p sits at bits (4p, 16+4p).  OR-ing a code into the mantissa of 1024.0 (0x6400) gives
// 1024 + q exactly; a code in the upper nibble of a byte gives 1024 + 16 q, which one FMA by
// 1/16 turns into 64 + q.  Subtracting (1024 + z) or (64 + z) is exact for integer zero
// points, so the only rounding is the final product with the scale.  Each pair takes its own
// scale and zero (the pairs of one word belong to two groups when group_size is 16).
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ __half2 u32_as_h2(uint32_t v)
{
    return *reinterpret_cast<__half2 *>(&v);
}

__device__ __forceinline__ uint32_t h2_as_u32(__half2 v)
{
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ void dequant_word(uint32_t x, const __half2 (&zlo)[4],
                                             const __half2 (&zhi)[4], const __half2 (&s2)[4],
                                             uint32_t (&out)[4])
{
    const uint32_t magic = 0x64006400u;
    const __half2 sixteenth = __halves2half2(__ushort_as_half(0x2C00), __ushort_as_half(0x2C00));
    const uint32_t t0 = (x & 0x000F000Fu) | magic;
    const uint32_t t1 = (x & 0x00F000F0u) | magic;
    const uint32_t x8 = __umulhi(x, 1u << 24); // x >> 8, on the FMA pipe (the integer pipe is the busy one)
    const uint32_t t2 = (x8 & 0x000F000Fu) | magic;
    const uint32_t t3 = (x8 & 0x00F000F0u) | magic;
    const __half2 v0 = __hsub2(u32_as_h2(t0), zlo[0]);
    const __half2 v1 = __hfma2(u32_as_h2(t1), sixteenth, zhi[1]);
    const __half2 v2 = __hsub2(u32_as_h2(t2), zlo[2]);
    const __half2 v3 = __hfma2(u32_as_h2(t3), sixteenth, zhi[3]);
    out[0] = h2_as_u32(__hmul2(v0, s2[0]));
    out[1] = h2_as_u32(__hmul2(v1, s2[1]));
    out[2] = h2_as_u32(__hmul2(v2, s2[2]));
    out[3] = h2_as_u32(__hmul2(v3, s2[3]));
}

// Scales (and zeros) of the four 8-row pairs p of half h of a 64-row block, each pair looking
// up its own group (general group sizes; one division per pair).
__device__ __forceinline__ void load_scales(const GemmParams &p, const __half *ssm, const __half *zsm,
                                            bool has_zp, int kb, int h, int g_first, int col,
                                            __half2 (&s2)[4], __half2 (&zlo)[4], __half2 (&zhi)[4])
{
#pragma unroll
    for (int pp = 0; pp < 4; ++pp) {
        const int gl = (kb * KBLK + h * 32 + pp * 8) / p.group_size - g_first;
        const int idx = gl * TILE_N + col;
        s2[pp] = __half2half2(ssm[idx]);
        if (has_zp) {
            const __half z = zsm[idx];
            zlo[pp] = __half2half2(__hadd(__ushort_as_half(0x6400), z));
            zhi[pp] = __half2half2(__hneg(__hadd(__ushort_as_half(0x5400), z)));
        } else {
            zlo[pp] = __half2half2(__ushort_as_half(0x6408));
            zhi[pp] = __half2half2(__ushort_as_half(0xD480));
        }
    }
}

// Uniform case (a group spans whole 64-row blocks): scale and zero offsets of one group row
// `grp_rel` (relative to the stage's first group row), the same for all four pairs.
__device__ __forceinline__ void load_scales_row(const __half *ssm, const __half *zsm, bool has_zp,
                                                int grp_rel, int col, __half2 (&s2)[4],
                                                __half2 (&zlo)[4], __half2 (&zhi)[4])
{
    const int idx = grp_rel * TILE_N + col;
    const __half2 s = __half2half2(ssm[idx]);
    __half2 lo = __half2half2(__ushort_as_half(0x6408)); // 1032
    __half2 hi = __half2half2(__ushort_as_half(0xD480)); // -72
    if (has_zp) {
        const __half z = zsm[idx];
        lo = __half2half2(__hadd(__ushort_as_half(0x6400), z));         // 1024 + z
        hi = __half2half2(__hneg(__hadd(__ushort_as_half(0x5400), z))); // -(64 + z)
    }
#pragma unroll
    for (int pp = 0; pp < 4; ++pp) {
        s2[pp] = s;
        zlo[pp] = lo;
        zhi[pp] = hi;
    }
}

// Two fp32 results rounded to the output's 16-bit format (fp16, or bf16), packed low-first.
__device__ __forceinline__ uint32_t pack_out2(float lo, float hi, bool bf16)
{
    if (bf16) {
        const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<const uint32_t *>(&v);
    }
    const __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

__device__ __forceinline__ uint16_t to_out16(float x, bool bf16)
{
    return bf16 ? __bfloat16_as_ushort(__float2bfloat16_rn(x)) : __half_as_ushort(__float2half_rn(x));
}

// log2 of the blocks per group when that is a power of two, else -1.
__device__ __forceinline__ int group_shift(int gs_kb)
{
    return (gs_kb > 0 && (gs_kb & (gs_kb - 1)) == 0) ? __ffs(gs_kb) - 1 : -1;
}

// ---------------------------------------------------------------------------------------
// Work schedule shared by every role: whole tiles round-robin while at least two full waves
// remain, then contiguous ranges of (tile, 64-row block) units ("stream-K").
// ---------------------------------------------------------------------------------------

// 64-bit division is a long software sequence on the GPU; use 32 bits when the operands fit.
__device__ __forceinline__ long long div_fast(long long a, long long b, bool small)
{
    return small ? (long long)((uint32_t)a / (uint32_t)b) : a / b;
}

struct Sched {
    int grid, cta, tiles, kblocks, dp_tiles, dp_next;
    long long sk_units, u, u_end, u_begin;
    bool small; // sk_units * (grid + 1) fits in 32 bits
    // Split mode (split > 0, grid = tiles * split): CTA c takes the (c % split)-th of `split`
    // near-equal K-ranges of tile c / split -- one segment, never straddling two tiles.
    int split, split_tile, kb_lo, kb_hi;
    bool split_done;

    // CTAs beyond the number of work units get nothing, so that the CTAs sharing a split
    // tile are always consecutive (the fixed-order reduction walks them by index).
    __device__ void init(int tiles_, int kblocks_, int split_ = 0)
    {
        tiles = tiles_;
        kblocks = kblocks_;
        split = split_;
        if (split > 0) {
            grid = (int)gridDim.x;
            cta = (int)blockIdx.x;
            dp_tiles = dp_next = 0;
            sk_units = u = u_end = u_begin = 0;
            small = true;
            const int r = cta % split;
            split_tile = cta / split;
            kb_lo = (int)((long long)r * kblocks / split);
            kb_hi = (int)((long long)(r + 1) * kblocks / split);
            split_done = split_tile >= tiles || kb_lo >= kb_hi;
            return;
        }
        const long long units = (long long)tiles * kblocks;
        grid = (int)min((long long)gridDim.x, max(units, 1LL));
        cta = blockIdx.x;
        const int waves = tiles / grid;
        if (tiles % grid == 0)
            dp_tiles = tiles;
        else
            dp_tiles = waves >= 2 ? (waves - 1) * grid : 0;
        dp_next = cta;
        sk_units = (long long)(tiles - dp_tiles) * kblocks;
        small = sk_units * (long long)(grid + 1) < (1LL << 32);
        const bool idle = cta >= grid;
        u = (sk_units && !idle) ? begin_of(cta) : 0;
        u_end = (sk_units && !idle) ? begin_of(cta + 1) : 0;
        u_begin = u;
        if (idle)
            dp_next = dp_tiles;
    }

    // First stream-K unit of CTA c.
    __device__ __forceinline__ long long begin_of(int c) const
    {
        return div_fast((long long)c * sk_units, grid, small);
    }

    // Next segment of work: tile index and its 64-row block range [kb0, kb1).
    __device__ bool next(int &tile, int &kb0, int &kb1)
    {
        if (split > 0) {
            if (split_done)
                return false;
            tile = split_tile;
            kb0 = kb_lo;
            kb1 = kb_hi;
            split_done = true;
            return true;
        }
        if (dp_next < dp_tiles) {
            tile = dp_next;
            kb0 = 0;
            kb1 = kblocks;
            dp_next += grid;
            return true;
        }
        if (u < u_end) {
            const long long t = div_fast(u, kblocks, small);
            kb0 = (int)(u - t * kblocks);
            const long long stop = min((t + 1) * kblocks, u_end);
            kb1 = kb0 + (int)(stop - u);
            tile = dp_tiles + (int)t;
            u = stop;
            return true;
        }
        return false;
    }

    // CTA that owns stream-K unit `unit`.
    __device__ int owner(long long unit) const
    {
        return (int)div_fast((unit + 1) * grid - 1, sk_units, small);
    }
};

struct TileInfo {
    int n0;      // first weight column
    int row0;    // first activation row (in the tensor map's row space)
    int rows;    // valid rows
    int ntok;    // rows rounded up to 16 (tcgen05 N)
    int expert;  // weight stack index
};

// Grouped schedule table in shared memory: tile prefix, row offsets, expert ids.
struct SegTable {
    int *tile_prefix; // [n_active + 1]
    int *row_off;     // [n_active + 1]
    int *expert;      // [n_active]
};

__device__ __forceinline__ TileInfo tile_info(const GemmParams &p, const SegTable &seg, int tile)
{
    TileInfo ti;
    if (p.ex_off == nullptr) {
        // Column-tile-major by default (the tiles running at once share weight columns);
        // token-tile-major when A is the operand that would otherwise fall out of L2.
        const int nt = p.m_outer ? tile % p.n_tiles : tile / p.m_tiles;
        const int mt = p.m_outer ? tile / p.n_tiles : tile - nt * p.m_tiles;
        ti.n0 = nt * TILE_N;
        ti.row0 = mt * p.nt_max;
        ti.rows = min(p.nt_max, p.m - ti.row0);
        ti.expert = 0;
    } else {
        int lo = 0, hi = p.n_active - 1; // last segment with tile_prefix <= tile
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (seg.tile_prefix[mid] <= tile)
                lo = mid;
            else
                hi = mid - 1;
        }
        const int local = tile - seg.tile_prefix[lo];
        const int cnt = seg.row_off[lo + 1] - seg.row_off[lo];
        const int mtiles = max(1, (cnt + p.nt_max - 1) / p.nt_max);
        const int nt = local / mtiles;
        const int mt = local - nt * mtiles;
        ti.n0 = nt * TILE_N;
        ti.row0 = seg.row_off[lo] + mt * p.nt_max;
        ti.rows = min(p.nt_max, cnt - mt * p.nt_max);
        ti.expert = seg.expert[lo];
    }
    ti.ntok = (ti.rows + 15) & ~15;
    return ti;
}

// Ring position and phase, advanced incrementally (no division in the loops).
struct Ring {
    int idx = 0;
    uint32_t phase = 0;
    __device__ __forceinline__ void advance(int size)
    {
        if (++idx == size) {
            idx = 0;
            phase ^= 1u;
        }
    }
};

// The position `steps` entries after r in a ring of `size`.
__device__ __forceinline__ Ring ring_after(Ring r, int steps, int size)
{
    for (int i = 0; i < steps; ++i)
        r.advance(size);
    return r;
}

// ---------------------------------------------------------------------------------------
// TMA producer (one thread).  A stage holds up to p.kbs consecutive 64-row blocks of one
// segment: their packed codes (one contiguous bulk copy -- copies have a large fixed cost, so
// they are made as big as the stage allows), the scale/zero rows they touch (one tensor copy
// each) and their activation rows (one 3-D tensor copy, p.kbs blocks deep).
// ---------------------------------------------------------------------------------------
// The weight part of one stage (packed codes, scale rows, zero rows), arming its barrier for
// the whole stage including the activation rows that follow separately.
static __device__ __forceinline__ void issue_stage_weights(const GemmParams &p,
                                                           const CUtensorMap *tmap_s,
                                                           const CUtensorMap *tmap_z,
                                                           const TileInfo &ti, int kb, int nkb,
                                                           uint8_t *st, uint64_t *full)
{
    const bool has_zp = p.zeros != nullptr;
    const uint32_t fixed_bytes = (uint32_t)p.sg_box * SG_BYTES * (has_zp ? 2u : 1u) +
                                 (uint32_t)(p.halves * p.kbs) * (uint32_t)p.act_kb_bytes;
    const int32_t *bw = p.b + ti.expert * p.b_expert_words +
                        ((long long)(ti.n0 / TILE_N) * p.kblocks) * p.tile_words;
    mbar_arrive_expect_tx(full, fixed_bytes + nkb * (uint32_t)p.tile_bytes);
    // The codes are read once per call: first to leave L2, so that what is re-read (the
    // activations, scales, split partials, the kernel's own instructions) stays.
    bulk_load_hint(st + p.packed_off, bw + (long long)kb * p.tile_words, nkb * p.tile_bytes, full,
                   policy_evict_first());
    const int g_first = ti.expert * p.num_groups + (kb * KBLK) / p.group_size;
    tensor_load_2d(st + p.scales_off, tmap_s, ti.n0, g_first, full);
    if (has_zp)
        tensor_load_2d(st + p.zeros_off, tmap_z, ti.n0, g_first, full);
}

// With static weights (W4A16_FLAG_STATIC_WEIGHTS) the weight part of the first ring's worth
// of stages is issued before the programmatic-dependency wait: nothing the preceding kernel
// writes is read.  Returns the number of stages so issued (their activation rows are still
// to come, from run_producer).
template <class SCHED>
static __device__ int issue_static_weights(const GemmParams &p, const CUtensorMap *tmap_s,
                                           const CUtensorMap *tmap_z, const SegTable &seg,
                                           SCHED sched, uint8_t *smem, uint64_t *full_bars)
{
    int n = 0;
    int tile, kb0, kb1;
    while (n < p.stages && sched.next(tile, kb0, kb1)) {
        const TileInfo ti = tile_info(p, seg, tile);
        for (int kb = kb0; kb < kb1 && n < p.stages; kb += p.kbs, ++n)
            issue_stage_weights(p, tmap_s, tmap_z, ti, kb, min(p.kbs, kb1 - kb),
                                smem + (size_t)n * p.stage_bytes, &full_bars[n]);
    }
    return n;
}

// `pre`: leading stages whose weight part issue_static_weights already issued.  `dep_wait`:
// the caller has not yet waited on the preceding kernel; wait before the first copy that may
// read its output (any copy, unless the weights are static; else the first activation copy).
template <class SCHED>
static __device__ void run_producer(const GemmParams &p, const CUtensorMap *tmap_a,
                                    const CUtensorMap *tmap_s, const CUtensorMap *tmap_z,
                                    const SegTable &seg, SCHED sched, uint8_t *smem,
                                    uint64_t *full_bars, uint64_t *empty_bars, const WaitCtl &ctl,
                                    int pre = 0, bool dep_wait = false)
{
    if (dep_wait && !p.static_weights)
        pdl_wait();
    Ring ring;
    uint32_t issued = 0;
    int tile, kb0, kb1;
    bool ok = true;
    while (ok && sched.next(tile, kb0, kb1)) {
        const TileInfo ti = tile_info(p, seg, tile);
        for (int kb = kb0; kb < kb1; kb += p.kbs) {
            const int nkb = min(p.kbs, kb1 - kb);
            uint64_t *full = &full_bars[ring.idx];
            uint8_t *st = smem + (size_t)ring.idx * p.stage_bytes;
            if ((int)issued >= pre) {
                if (!mbar_wait(&empty_bars[ring.idx], ring.phase ^ 1u, ctl, W4A16_DEV_TIMEOUT)) {
                    ok = false;
                    break;
                }
                issue_stage_weights(p, tmap_s, tmap_z, ti, kb, nkb, st, full);
            }
            if (dep_wait && issued == 0 && p.static_weights)
                pdl_wait();
            // 64 columns x (half-)tile rows x kbs column blocks, landing as kbs consecutive
            // [rows x 128 B] tiles in the 128-byte swizzle; a paired tile loads its second
            // half-tile's rows after the first's.  Activation rows are read again for every
            // column tile: last to leave L2.
            for (int h = 0; h < p.halves; ++h)
                tensor_load_3d_hint(st + h * p.kbs * p.act_kb_bytes, tmap_a, 0,
                                    ti.row0 + h * p.nt_half, kb, full, policy_evict_last());
            ring.advance(p.stages);
            ++issued;
        }
    }
    // Leave no copy in flight: wait (bounded, ignoring the abort flag) for the last stages.
    WaitCtl drain_ctl = ctl;
    volatile int no_abort = 0;
    drain_ctl.abort_flag = &no_abort;
    const uint32_t n = issued < (uint32_t)p.stages ? issued : (uint32_t)p.stages;
    for (uint32_t i = 0; i < n; ++i) {
        int idx = ring.idx - 1 - (int)i;
        uint32_t ph = ring.phase;
        if (idx < 0) {
            idx += p.stages;
            ph ^= 1u;
        }
        mbar_wait(&full_bars[idx], ph, drain_ctl, W4A16_DEV_TIMEOUT);
    }
}

// L2 prefetch of the packed codes of this CTA's first `budget` bytes of work (dense schedule
// only).  The weights never depend on the kernel that precedes this one on the stream, so the
// prefetch may run before the programmatic-dependency wait and overlap that kernel's tail; it
// only warms L2 (the coherence point), and the real loads still come after the wait.
template <class SCHED>
static __device__ void prefetch_first_codes(const GemmParams &p, SCHED sched, uint32_t budget)
{
    SegTable no_seg{nullptr, nullptr, nullptr};
    int tile, kb0, kb1;
    while (budget > 0 && sched.next(tile, kb0, kb1)) {
        const TileInfo ti = tile_info(p, no_seg, tile);
        const int32_t *bw = p.b + ((long long)(ti.n0 / TILE_N) * p.kblocks + kb0) * TILE_WORDS;
        uint32_t bytes = (uint32_t)(kb1 - kb0) * TILE_BYTES;
        if (bytes > budget)
            bytes = budget;
        bulk_prefetch_l2(bw, bytes);
        budget -= bytes;
    }
}

// Builds the grouped schedule table (warp-wide): per active segment its row range, expert
// and number of tiles; returns the total tile count.  The offsets must form a non-decreasing
// chain inside [0, n_pairs] and the expert ids must be in range; otherwise the whole schedule
// is treated as empty and W4A16_DEV_SCHEDULE is reported, so no tile can index past the
// workspace's counters.
static __device__ int build_segments(const GemmParams &p, SegTable &seg, int lane)
{
    bool bad = false;
    for (int base = 0; base < p.n_active; base += 32) {
        const int i = base + lane;
        bool b = false;
        if (i < p.n_active) {
            const int lo = p.ex_off[i], hi = p.ex_off[i + 1], e = p.ex_ids[i];
            b = lo < 0 || hi < lo || hi > p.n_rows || e < 0 || e >= p.n_experts;
        }
        bad |= __any_sync(0xffffffffu, b);
    }
    if (bad) {
        if (lane == 0)
            atomicOr(p.status, W4A16_DEV_SCHEDULE);
        return 0;
    }
    int running = 0;
    for (int base = 0; base < p.n_active; base += 32) {
        const int i = base + lane;
        int tiles_i = 0;
        if (i < p.n_active) {
            const int lo = p.ex_off[i], hi = p.ex_off[i + 1];
            seg.row_off[i] = lo;
            seg.expert[i] = p.ex_ids[i];
            if (i == p.n_active - 1)
                seg.row_off[i + 1] = hi;
            tiles_i = ((hi - lo + p.nt_max - 1) / p.nt_max) * p.n_tiles;
        }
        int incl = tiles_i; // inclusive warp scan
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d)
                incl += v;
        }
        if (i < p.n_active)
            seg.tile_prefix[i] = running + incl - tiles_i;
        running += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0)
        seg.tile_prefix[p.n_active] = running;
    __syncwarp();
    return running;
}

// ---------------------------------------------------------------------------------------
// Split (stream-K) tiles.  Every CTA that covers part of a tile's 64-row blocks writes an
// fp32 partial into one of its two workspace slots (0: the tile where its range starts,
// 1: its last tile); the last of them to arrive sums all partials in CTA order.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ float *partial_slot(const GemmParams &p, int cta, int slot)
{
    return p.partials + ((long long)(cta * 2 + slot) * p.nt_max) * TILE_N;
}

// This CTA's slot for stream-K tile st_tile.
__device__ __forceinline__ int own_slot(const GemmParams &p, const Sched &sched, long long st_tile)
{
    if (sched.split > 0)
        return 0; // one segment per CTA
    return sched.u_begin >= st_tile * p.kblocks ? 0 : 1;
}

// Output row of tile row `row`: dense rows are in place; grouped rows go to pair ex_pairs[.].
// Returns -1 for a row that writes nothing: a padding row of the block-routed interface
// (entry -1), or an out-of-range entry, which is reported.
__device__ __forceinline__ int output_row(const GemmParams &p, const TileInfo &ti, int row)
{
    int out_row = ti.row0 + row;
    if (p.ex_off != nullptr) {
        out_row = p.ex_pairs[out_row];
        if (out_row < 0 || out_row >= p.n_pairs) {
            if (!(p.skip_sentinel && out_row == -1))
                atomicOr(p.status, W4A16_DEV_SCHEDULE);
            return -1;
        }
    }
    return out_row;
}

// Scale of an output row (the block-routed interface's top-k weight), 1 otherwise.
__device__ __forceinline__ float row_scale(const GemmParams &p, int out_row)
{
    return p.row_weight != nullptr ? p.row_weight[out_row] : 1.0f;
}

// Contributors c_lo..c_hi of stream-K tile st_tile and the slot of the first one (the others
// start inside the tile, so they use slot 0).
struct Contributors {
    int lo, hi, lo_slot;
};

__device__ __forceinline__ Contributors contributors(const GemmParams &p, const Sched &sched,
                                                     long long st_tile)
{
    Contributors c;
    if (sched.split > 0) {
        c.lo = (int)st_tile * sched.split;
        c.hi = c.lo + sched.split - 1;
        c.lo_slot = 0;
        return c;
    }
    const long long u0 = st_tile * p.kblocks;
    c.lo = sched.owner(u0);
    c.hi = sched.owner(u0 + p.kblocks - 1);
    c.lo_slot = sched.begin_of(c.lo) >= u0 ? 0 : 1;
    return c;
}

// Split-tile counter: one acquire-release atomic at GPU scope.  The CTA's partial stores
// happen before it through the CTA-wide rendezvous that precedes it, and release is
// cumulative, so they are visible to whoever reads the counter's later value; the acquire half
// makes the other contributors' partials visible to the last arriver (and, through the
// rendezvous that follows, to the rest of its CTA).
__device__ __forceinline__ int split_counter_arrive(int *counter)
{
    int old;
    asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], 1;" : "=r"(old) : "l"(counter) : "memory");
    return old;
}

// Sum the partials of a split tile and write fp16 C.  Work items are (row, 4-column quad).
// With fewer items than threads, `ways` consecutive threads share an item, thread j summing
// contributors lo + j, lo + j + ways, ... and a fixed shuffle tree combining the ways; with more
// items than threads, each thread takes RB items per round and keeps their loads (up to
// RB x CB partial quads) in flight together -- the partials sit in L2, so the reduction is
// bound by load latency, not bandwidth.  Every order is fixed, so results are bit-identical from
// run to run.  `nthreads` must be a multiple of 32.
static __device__ __forceinline__ void store_quad(const GemmParams &p, const TileInfo &ti, int row,
                                                  int cq, float4 acc)
{
    const int out_row = output_row(p, ti, row);
    if (out_row < 0)
        return;
    const float w = row_scale(p, out_row);
    uint2 packed;
    packed.x = pack_out2(acc.x * w, acc.y * w, p.bf16);
    packed.y = pack_out2(acc.z * w, acc.w * w, p.bf16);
    *reinterpret_cast<uint2 *>(p.c + (long long)out_row * p.ldc + ti.n0 + 4 * cq) = packed;
}

__device__ __forceinline__ const float4 *partial_quads(const GemmParams &p, const Contributors &cb,
                                                       int c)
{
    return reinterpret_cast<const float4 *>(partial_slot(p, c, c == cb.lo ? cb.lo_slot : 0));
}

// ---------------------------------------------------------------------------------------
// Gated activation epilogue (W4A16_FLAG_SWIGLU / _GEGLU).  The weight's columns are gate and up
// projections interleaved in blocks of 16: packed columns 32b .. 32b+15 are gate features
// 16b .. 16b+15 and packed columns 32b+16 .. 32b+31 the up features of the same indices, so a
// 128-column tile holds features n0/2 .. n0/2 + 63 and writes act(gate) * up there.
// ---------------------------------------------------------------------------------------
// Both are g * sigmoid(x): silu with x = g; gelu_tanh, 0.5 g (1 + tanh t) with
// t = sqrt(2/pi) (g + 0.044715 g^3), since 1 + tanh t = 2 sigmoid(2t).  One fast exponential and
// one reciprocal per element: the epilogue warps share their SM sub-partitions with the MMA-
// issuing thread, and accurate expf / division / tanhf there slowed the gated MoE GEMM by 5 %.
// (x -> -inf: the exponential is inf, its reciprocal 0; x -> +inf: the result is g.)
__device__ __forceinline__ float glu_act(float g, int kind)
{
    float x = g;
    if (kind != 1) {
        const float c = 0.7978845608028654f; // sqrt(2 / pi)
        x = 2.0f * c * (g + 0.044715f * g * g * g);
    }
    return g * __frcp_rn(1.0f + __expf(-x));
}

// Split tile of a gated call: items are (row, gate quad); each sums its gate quad and the up
// quad 16 columns on over the contributors in index order, then writes 4 features.
static __device__ void reduce_tile_glu(const GemmParams &p, const TileInfo &ti, const Contributors &cb,
                                       int tid, int nthreads)
{
    constexpr int QUADS = TILE_N / 4;
    constexpr int OUTQ = TILE_N / 8; // 16 gate quads per row
    const int items = ti.rows * OUTQ;
    for (int item = tid; item < items; item += nthreads) {
        const int row = item / OUTQ, gq = item - (item / OUTQ) * OUTQ;
        const int qg = row * QUADS + (gq >> 2) * 8 + (gq & 3);
        float4 g = make_float4(0.f, 0.f, 0.f, 0.f), u = g;
        for (int c0 = cb.lo; c0 <= cb.hi; c0 += 4) {
            float4 vg[4], vu[4];
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                const bool ok = c0 + x <= cb.hi;
                const float4 *src = partial_quads(p, cb, ok ? c0 + x : cb.lo);
                vg[x] = ok ? __ldcg(src + qg) : make_float4(0.f, 0.f, 0.f, 0.f);
                vu[x] = ok ? __ldcg(src + qg + 4) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                g.x += vg[x].x; g.y += vg[x].y; g.z += vg[x].z; g.w += vg[x].w;
                u.x += vu[x].x; u.y += vu[x].y; u.z += vu[x].z; u.w += vu[x].w;
            }
        }
        const int out_row = output_row(p, ti, row);
        if (out_row < 0)
            continue;
        const float w = row_scale(p, out_row);
        uint2 packed;
        packed.x = pack_out2(glu_act(g.x, p.glu) * u.x * w, glu_act(g.y, p.glu) * u.y * w, p.bf16);
        packed.y = pack_out2(glu_act(g.z, p.glu) * u.z * w, glu_act(g.w, p.glu) * u.w * w, p.bf16);
        *reinterpret_cast<uint2 *>(p.c + (long long)out_row * p.ldc + ti.n0 / 2 + 4 * gq) = packed;
    }
}

template <int RB = 4, int CB = 4>
static __device__ void reduce_tile(const GemmParams &p, const TileInfo &ti, const Contributors &cb,
                                   int tid, int nthreads)
{
    constexpr int QUADS = TILE_N / 4;
    const int items = ti.rows * QUADS;
    const int ncontrib = cb.hi - cb.lo + 1;
    if (items * 2 <= nthreads) {
        int ways = 1;
        while (ways < 16 && ways * 2 <= ncontrib && items * ways * 2 <= nthreads)
            ways *= 2;
        const int slot = tid;
        const bool active = slot < items * ways;
        const int item = slot / ways;
        const int j = slot - item * ways;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (active) {
            for (int c0 = cb.lo + j; c0 <= cb.hi; c0 += 8 * ways) {
                float4 v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int c = c0 + u * ways;
                    v[u] = c <= cb.hi ? __ldcg(partial_quads(p, cb, c) + item)
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    acc.x += v[u].x;
                    acc.y += v[u].y;
                    acc.z += v[u].z;
                    acc.w += v[u].w;
                }
            }
        }
        for (int off = 1; off < ways; off <<= 1) {
            acc.x += __shfl_xor_sync(0xffffffffu, acc.x, off);
            acc.y += __shfl_xor_sync(0xffffffffu, acc.y, off);
            acc.z += __shfl_xor_sync(0xffffffffu, acc.z, off);
            acc.w += __shfl_xor_sync(0xffffffffu, acc.w, off);
        }
        if (active && j == 0)
            store_quad(p, ti, item / QUADS, item % QUADS, acc);
        return;
    }
    // RB items per round x CB contributors per batch: RB * CB independent 16-byte loads in
    // flight per thread (the reduction is bound by their latency).
    for (int base = tid; base < items; base += nthreads * RB) {
        float4 acc[RB];
#pragma unroll
        for (int r = 0; r < RB; ++r)
            acc[r] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int c0 = cb.lo; c0 <= cb.hi; c0 += CB) {
            float4 v[RB][CB];
#pragma unroll
            for (int r = 0; r < RB; ++r)
#pragma unroll
                for (int u = 0; u < CB; ++u) {
                    const int item = base + r * nthreads, c = c0 + u;
                    v[r][u] = (item < items && c <= cb.hi) ? __ldcg(partial_quads(p, cb, c) + item)
                                                          : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
            for (int r = 0; r < RB; ++r)
#pragma unroll
                for (int u = 0; u < CB; ++u) {
                    acc[r].x += v[r][u].x;
                    acc[r].y += v[r][u].y;
                    acc[r].z += v[r][u].z;
                    acc[r].w += v[r][u].w;
                }
        }
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            const int item = base + r * nthreads;
            if (item < items)
                store_quad(p, ti, item / QUADS, item % QUADS, acc[r]);
        }
    }
}

} // namespace w4
