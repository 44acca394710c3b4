// w4a16_gemm.cu -- the tcgen05 W4A16 GEMM kernel for sm_103a.
//
// Computes C[M,N] = A[M,K] x dequant(B)[K,N] (ferrum-kernels 0.8.5 marlin.rs, `marlin_gemm`
// doc) with the weights on the tcgen05 M side ("swap-AB"):
//     D[n, t] = sum_k W^T[n, k] * A^T[k, t],   D = C^T tile of 128 weight columns x T tokens.
// One persistent CTA per SM, warp-specialised:
//   warp 0       TMA producer: one 4 KiB bulk copy of packed codes, the group scales/zeros
//                and T/16 tensor copies of activation rows (128-byte swizzle) per 64-row stage
//   warp 1       tcgen05.mma issuer (one thread) and tensor-memory owner
//   warps 4..7   epilogue: tensor memory -> registers -> fp16 C, or fp32 split-K partials
//   warps 8..15  dequant: codes -> (q - z) * s in fp16 -> tensor memory (the MMA's A operand)
// Work is split "data-parallel + stream-K": whole tiles round-robin while at least two full
// waves remain, the rest as contiguous ranges of (tile, 64-row block) units.  Tiles cut by
// a range boundary are summed from fp32 partials in a fixed order by the last contributor
// to finish (an atomic counter that resets itself), so results are deterministic and no CTA
// ever waits for another.
#include "ptx.cuh"
#include "w4a16_internal.h"
#include "../../include/w4a16.h"

namespace w4 {

// ---------------------------------------------------------------------------------------
// Dequantisation of one tile word (8 codes) into 4 fp16 pairs (q - z) * s.
// Codes 2i and 2i+1 sit at bits 4i and 16+4i.  OR-ing a code into the mantissa of 1024.0
// (0x6400) gives 1024 + q exactly; a code in the upper nibble of a byte gives 1024 + 16 q,
// which one FMA by 1/16 turns into 64 + q.  Subtracting (1024 + z) or (64 + z) is exact for
// integer zero points, so the only rounding is the final product with the scale.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ __half2 u32_as_h2(uint32_t v)
{
    return *reinterpret_cast<__half2 *>(&v);
}

__device__ __forceinline__ uint32_t h2_as_u32(__half2 v)
{
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ void dequant_word(uint32_t x, __half2 zlo, __half2 zhi, __half2 s2,
                                             uint32_t *out)
{
    const uint32_t magic = 0x64006400u;
    const __half2 sixteenth = __halves2half2(__ushort_as_half(0x2C00), __ushort_as_half(0x2C00));
    const uint32_t t0 = (x & 0x000F000Fu) | magic;
    const uint32_t t1 = (x & 0x00F000F0u) | magic;
    const uint32_t x8 = x >> 8;
    const uint32_t t2 = (x8 & 0x000F000Fu) | magic;
    const uint32_t t3 = (x8 & 0x00F000F0u) | magic;
    const __half2 v0 = __hsub2(u32_as_h2(t0), zlo);
    const __half2 v1 = __hfma2(u32_as_h2(t1), sixteenth, zhi);
    const __half2 v2 = __hsub2(u32_as_h2(t2), zlo);
    const __half2 v3 = __hfma2(u32_as_h2(t3), sixteenth, zhi);
    out[0] = h2_as_u32(__hmul2(v0, s2));
    out[1] = h2_as_u32(__hmul2(v1, s2));
    out[2] = h2_as_u32(__hmul2(v2, s2));
    out[3] = h2_as_u32(__hmul2(v3, s2));
}

// ---------------------------------------------------------------------------------------
// Work schedule shared by every role.
// ---------------------------------------------------------------------------------------
struct Sched {
    int grid, cta, tiles, kblocks, dp_tiles, dp_next;
    long long sk_units, u, u_end;

    // CTAs beyond the number of work units get nothing, so that the CTAs sharing a split
    // tile are always consecutive (the fixed-order reduction walks them by index).
    __device__ void init(int tiles_, int kblocks_)
    {
        tiles = tiles_;
        kblocks = kblocks_;
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
        const bool idle = cta >= grid;
        u = (sk_units && !idle) ? (long long)cta * sk_units / grid : 0;
        u_end = (sk_units && !idle) ? (long long)(cta + 1) * sk_units / grid : 0;
        if (idle)
            dp_next = dp_tiles;
    }

    // Next segment of work: tile index and its 64-row block range [kb0, kb1).
    __device__ bool next(int &tile, int &kb0, int &kb1)
    {
        if (dp_next < dp_tiles) {
            tile = dp_next;
            kb0 = 0;
            kb1 = kblocks;
            dp_next += grid;
            return true;
        }
        if (u < u_end) {
            const long long t = u / kblocks;
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
        return (int)(((unit + 1) * grid - 1) / sk_units);
    }

    // Partial slot (0 = first stream-K tile of CTA c, 1 = its last) used for stream-K tile st.
    __device__ int slot_of(int c, long long st) const
    {
        const long long first = ((long long)c * sk_units / grid) / kblocks;
        return st == first ? 0 : 1;
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
        const int nt = tile / p.m_tiles;
        const int mt = tile - nt * p.m_tiles;
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

struct Bars {
    uint64_t full[MAX_STAGES];
    uint64_t empty[MAX_STAGES];
    uint64_t afull[MAX_A_SLOTS];
    uint64_t aempty[MAX_A_SLOTS];
    uint64_t accfull[2];
    uint64_t accempty[2];
    uint64_t drain;
    uint64_t epi;       // epilogue-group rendezvous (bounded, unlike a named barrier)
};

// ---------------------------------------------------------------------------------------
// Roles
// ---------------------------------------------------------------------------------------
__device__ void run_producer(const GemmParams &p, const CUtensorMap *tmap, const SegTable &seg,
                             Sched sched, uint8_t *smem, Bars &bars, const WaitCtl &ctl)
{
    const int has_zp = p.zeros != nullptr;
    uint32_t it = 0;
    int tile, kb0, kb1;
    bool ok = true;
    while (ok && sched.next(tile, kb0, kb1)) {
        const TileInfo ti = tile_info(p, seg, tile);
        const int nt = ti.n0 / TILE_N;
        const int32_t *bw = p.b + ti.expert * p.b_expert_words +
                            ((long long)nt * p.kblocks) * TILE_WORDS;
        const __half *sc = p.scales + ti.expert * p.s_expert_elems + ti.n0;
        const __half *zp = has_zp ? p.zeros + ti.expert * p.s_expert_elems + ti.n0 : nullptr;
        const int boxes = ti.ntok / BOX_ROWS;
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
            const int stage = it % p.stages;
            const uint32_t ph = (it / p.stages) & 1u;
            if (!mbar_wait(&bars.empty[stage], ph ^ 1u, ctl, W4A16_DEV_TIMEOUT)) {
                ok = false;
                break;
            }
            uint8_t *st = smem + (size_t)stage * p.stage_bytes;
            const int r0 = kb * KBLK;
            const int g0 = r0 / p.group_size;
            const int g1 = (r0 + KBLK - 1) / p.group_size;
            const int nsg = g1 - g0 + 1;
            const uint32_t bytes = TILE_BYTES + nsg * SG_BYTES * (1 + has_zp) + boxes * BOX_ROWS * 128;
            mbar_arrive_expect_tx(&bars.full[stage], bytes);
            bulk_load(st + p.act_bytes, bw + (long long)kb * TILE_WORDS, TILE_BYTES,
                      &bars.full[stage]);
            for (int g = 0; g < nsg; ++g) {
                bulk_load(st + p.act_bytes + TILE_BYTES + g * SG_BYTES,
                          sc + (long long)(g0 + g) * p.n, SG_BYTES, &bars.full[stage]);
                if (has_zp)
                    bulk_load(st + p.act_bytes + TILE_BYTES + (MAX_SG + g) * SG_BYTES,
                              zp + (long long)(g0 + g) * p.n, SG_BYTES, &bars.full[stage]);
            }
            for (int bx = 0; bx < boxes; ++bx)
                tensor_load_2d(st + bx * BOX_ROWS * 128, tmap, r0, ti.row0 + bx * BOX_ROWS,
                               &bars.full[stage]);
        }
    }
    // Leave no copy in flight: wait (bounded) for the last stages issued.
    WaitCtl drain_ctl = ctl;
    volatile int no_abort = 0;
    drain_ctl.abort_flag = &no_abort;
    const uint32_t first = it > (uint32_t)p.stages ? it - p.stages : 0;
    for (uint32_t i = first; i < it; ++i)
        mbar_wait(&bars.full[i % p.stages], (i / p.stages) & 1u, drain_ctl, W4A16_DEV_TIMEOUT);
}

template <bool A_TMEM>
__device__ void run_mma(const GemmParams &p, const SegTable &seg, Sched sched, uint8_t *smem,
                        uint8_t *aring, Bars &bars, uint32_t tmem_base, const WaitCtl &ctl)
{
    uint32_t it = 0, seg_i = 0;
    int tile, kb0, kb1;
    bool ok = true;
    while (ok && sched.next(tile, kb0, kb1)) {
        const TileInfo ti = tile_info(p, seg, tile);
        const uint32_t idesc = idesc_f16_f32(TILE_N, ti.ntok);
        const int abuf = seg_i % p.acc_bufs;
        const uint32_t acc_ph = (seg_i / p.acc_bufs) & 1u;
        if (!mbar_wait(&bars.accempty[abuf], acc_ph ^ 1u, ctl, W4A16_DEV_TIMEOUT))
            break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + p.acc_col0 + abuf * p.nt_max;
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
            const int stage = it % p.stages;
            const uint32_t ph = (it / p.stages) & 1u;
            const int aslot = it % p.a_slots;
            const uint32_t aph = (it / p.a_slots) & 1u;
            if (!mbar_wait(&bars.full[stage], ph, ctl, W4A16_DEV_TIMEOUT) ||
                !mbar_wait(&bars.afull[aslot], aph, ctl, W4A16_DEV_TIMEOUT)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t act = smem_u32(smem + (size_t)stage * p.stage_bytes);
#pragma unroll
            for (int kk = 0; kk < KBLK / 16; ++kk) {
                const uint64_t bdesc = desc_sw128(act + kk * 32);
                const uint32_t acc = (kb > kb0 || kk > 0) ? 1u : 0u;
                if (A_TMEM) {
                    mma_ts(d_tmem, tmem_base + aslot * A_SLOT_COLS + kk * 8, bdesc, idesc, acc);
                } else {
                    const uint64_t adesc =
                        desc_sw128(smem_u32(aring + aslot * A_SLOT_BYTES) + kk * 32);
                    mma_ss(d_tmem, adesc, bdesc, idesc, acc);
                }
            }
            mma_commit(&bars.empty[stage]);
            mma_commit(&bars.aempty[aslot]);
        }
        if (!ok)
            break;
        mma_commit(&bars.accfull[abuf]);
        ++seg_i;
    }
    // Leave no MMA in flight before tensor memory is released.
    mma_commit(&bars.drain);
    WaitCtl drain_ctl = ctl;
    volatile int no_abort = 0;
    drain_ctl.abort_flag = &no_abort;
    mbar_wait(&bars.drain, 0, drain_ctl, W4A16_DEV_TIMEOUT);
}

template <bool A_TMEM>
__device__ void run_dequant(const GemmParams &p, Sched sched, uint8_t *smem, uint8_t *aring,
                            Bars &bars, uint32_t tmem_base, const WaitCtl &ctl, int warp, int lane)
{
    const int q = warp & 3;
    const int h = (warp - DQ_WARP0) >> 2;
    const int nl = q * 32 + lane;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    const bool has_zp = p.zeros != nullptr;
    const __half2 zlo8 = __float2half2_rn(1032.0f);
    const __half2 zhi8 = __float2half2_rn(-72.0f);
    uint32_t it = 0;
    int tile, kb0, kb1;
    while (sched.next(tile, kb0, kb1)) {
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
            const int stage = it % p.stages;
            const uint32_t ph = (it / p.stages) & 1u;
            const int aslot = it % p.a_slots;
            const uint32_t aph = (it / p.a_slots) & 1u;
            if (!mbar_wait(&bars.full[stage], ph, ctl, W4A16_DEV_TIMEOUT) ||
                !mbar_wait(&bars.aempty[aslot], aph ^ 1u, ctl, W4A16_DEV_TIMEOUT))
                return;
            tc_fence_after();
            const uint8_t *st = smem + (size_t)stage * p.stage_bytes;
            const uint4 wv =
                *reinterpret_cast<const uint4 *>(st + p.act_bytes + (h * 512 + nl * 4) * 4);
            const __half *ssm = reinterpret_cast<const __half *>(st + p.act_bytes + TILE_BYTES);
            const __half *zsm = ssm + MAX_SG * TILE_N;
            const int r0 = kb * KBLK;
            const int g0 = r0 / p.group_size;
            uint32_t out[16];
            const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int gl = (r0 + h * 32 + j * 8) / p.group_size - g0;
                const __half s = ssm[gl * TILE_N + nl];
                __half2 zlo = zlo8, zhi = zhi8;
                if (has_zp) {
                    const __half z = zsm[gl * TILE_N + nl];
                    zlo = __half2half2(__hadd(__float2half(1024.0f), z));
                    zhi = __half2half2(__hneg(__hadd(__float2half(64.0f), z)));
                }
                dequant_word(words[j], zlo, zhi, __half2half2(s), &out[j * 4]);
            }
            if (A_TMEM) {
                tmem_st16(tmem_base + lane_base + aslot * A_SLOT_COLS + h * 16, out);
                tmem_st_wait();
                tc_fence_before();
            } else {
                uint8_t *slot = aring + aslot * A_SLOT_BYTES + nl * 128;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int chunk = h * 4 + j;
                    *reinterpret_cast<uint4 *>(slot + ((chunk ^ (nl & 7)) << 4)) =
                        make_uint4(out[j * 4], out[j * 4 + 1], out[j * 4 + 2], out[j * 4 + 3]);
                }
                fence_proxy_async_smem();
            }
            // One arrival per warp: the warp's tensor-memory (or shared-memory) writes are
            // complete and fenced in every lane before the warp converges here.
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&bars.afull[aslot]);
                mbar_arrive(&bars.empty[stage]);
            }
        }
    }
}

__device__ void run_epilogue(const GemmParams &p, const SegTable &seg, Sched sched, Bars &bars,
                             uint32_t tmem_base, const WaitCtl &ctl, int warp, int lane,
                             volatile int *last_flag)
{
    const int q = warp & 3;
    const int nl = q * 32 + lane;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    const bool grouped = p.ex_off != nullptr;
    uint32_t seg_i = 0, nsync = 0;
    int tile, kb0, kb1;
    // All 128 epilogue threads meet here; gives up (false) on abort instead of hanging.
    auto rendezvous = [&]() -> bool {
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&bars.epi);
        const bool ok = mbar_wait(&bars.epi, nsync & 1u, ctl, W4A16_DEV_TIMEOUT);
        ++nsync;
        return ok;
    };
    while (sched.next(tile, kb0, kb1)) {
        const TileInfo ti = tile_info(p, seg, tile);
        const int abuf = seg_i % p.acc_bufs;
        const uint32_t acc_ph = (seg_i / p.acc_bufs) & 1u;
        if (!mbar_wait(&bars.accfull[abuf], acc_ph, ctl, W4A16_DEV_TIMEOUT))
            return;
        tc_fence_after();
        const uint32_t taddr = tmem_base + lane_base + p.acc_col0 + abuf * p.nt_max;
        const bool whole = (kb0 == 0 && kb1 == p.kblocks);
        const int col = ti.n0 + nl;
        const long long st_tile = (long long)tile - sched.dp_tiles;
        float *part = nullptr;
        if (!whole)
            part = p.partials +
                   ((long long)(sched.cta * 2 + sched.slot_of(sched.cta, st_tile)) * p.nt_max) * TILE_N;
        for (int c0 = 0; c0 < ti.ntok; c0 += 16) {
            uint32_t v[16];
            tmem_ld16(taddr + c0, v);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int row = c0 + j;
                if (row < ti.rows) {
                    const float f = __uint_as_float(v[j]);
                    if (whole) {
                        int out_row = ti.row0 + row;
                        if (grouped) {
                            out_row = p.ex_pairs[out_row];
                            if (out_row < 0 || out_row >= p.n_pairs) {
                                atomicOr(p.status, W4A16_DEV_SCHEDULE);
                                continue;
                            }
                        }
                        p.c[(long long)out_row * p.ldc + col] = __float2half_rn(f);
                    } else {
                        __stcg(part + row * TILE_N + nl, f);
                    }
                }
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&bars.accempty[abuf]);
        ++seg_i;
        if (whole)
            continue;
        // Split tile: publish the partial, and let the last contributor reduce.
        __threadfence();
        if (!rendezvous())
            return;
        const long long u0 = st_tile * p.kblocks;
        const int c_lo = sched.owner(u0);
        const int c_hi = sched.owner(u0 + p.kblocks - 1);
        if (warp == EPI_WARP0 && lane == 0) {
            __threadfence();
            const int old = atomicAdd(&p.counters[tile], 1);
            const int last = old == (c_hi - c_lo);
            if (last)
                __threadfence();
            *last_flag = last;
        }
        if (!rendezvous())
            return;
        if (!*last_flag)
            continue;
        // Fixed-order sum over the contributors c_lo..c_hi.  Thread (row phase rph, column
        // quad cq) owns rows rph, rph+4, ... and columns 4cq..4cq+3; loads are batched (four
        // contributors x four rows) so that they overlap.
        const int rph = warp - EPI_WARP0;
        const int cq = lane;
        for (int rb = rph; rb < ti.rows; rb += 16) {
            float4 acc[4];
#pragma unroll
            for (int u4 = 0; u4 < 4; ++u4)
                acc[u4] = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int c0 = c_lo; c0 <= c_hi; c0 += 4) {
                float4 v[4][4];
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const int c = c0 + cc;
                    const float4 *pc = reinterpret_cast<const float4 *>(
                        p.partials + ((long long)(c * 2 + sched.slot_of(c, st_tile)) * p.nt_max) * TILE_N);
#pragma unroll
                    for (int u4 = 0; u4 < 4; ++u4) {
                        const int row = rb + 4 * u4;
                        v[cc][u4] = (c <= c_hi && row < ti.rows) ? __ldcg(pc + row * (TILE_N / 4) + cq)
                                                                : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    if (c0 + cc > c_hi)
                        break;
#pragma unroll
                    for (int u4 = 0; u4 < 4; ++u4) {
                        acc[u4].x += v[cc][u4].x;
                        acc[u4].y += v[cc][u4].y;
                        acc[u4].z += v[cc][u4].z;
                        acc[u4].w += v[cc][u4].w;
                    }
                }
            }
#pragma unroll
            for (int u4 = 0; u4 < 4; ++u4) {
                const int row = rb + 4 * u4;
                if (row >= ti.rows)
                    break;
                int out_row = ti.row0 + row;
                if (grouped) {
                    out_row = p.ex_pairs[out_row];
                    if (out_row < 0 || out_row >= p.n_pairs) {
                        atomicOr(p.status, W4A16_DEV_SCHEDULE);
                        continue;
                    }
                }
                const __half2 lo = __floats2half2_rn(acc[u4].x, acc[u4].y);
                const __half2 hi = __floats2half2_rn(acc[u4].z, acc[u4].w);
                uint2 packed;
                packed.x = *reinterpret_cast<const uint32_t *>(&lo);
                packed.y = *reinterpret_cast<const uint32_t *>(&hi);
                *reinterpret_cast<uint2 *>(p.c + (long long)out_row * p.ldc + ti.n0 + 4 * cq) = packed;
            }
        }
        if (warp == EPI_WARP0 && lane == 0)
            p.counters[tile] = 0;
    }
}

// Builds the grouped schedule table (warp-wide): per active segment its row range, expert
// and number of tiles; returns the total tile count.  The offsets must form a non-decreasing
// chain inside [0, n_pairs] and the expert ids must be in range; otherwise the whole schedule
// is treated as empty and W4A16_DEV_SCHEDULE is reported (so no tile can index past the
// workspace's counters).
__device__ int build_segments(const GemmParams &p, SegTable &seg, int lane)
{
    bool bad = false;
    for (int base = 0; base < p.n_active; base += 32) {
        const int i = base + lane;
        bool b = false;
        if (i < p.n_active) {
            const int lo = p.ex_off[i], hi = p.ex_off[i + 1], e = p.ex_ids[i];
            b = lo < 0 || hi < lo || hi > p.n_pairs || e < 0 || e >= p.n_experts;
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

template <bool A_TMEM>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    w4a16_gemm_kernel(const __grid_constant__ GemmParams p, const __grid_constant__ CUtensorMap tmap_a)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ Bars bars;
    __shared__ uint32_t tmem_base_sh;
    __shared__ volatile int abort_sh;
    __shared__ volatile int last_sh;
    __shared__ int total_tiles_sh;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint8_t *aring = smem + (size_t)p.stages * p.stage_bytes;
    SegTable seg;
    int *segmem = reinterpret_cast<int *>(smem + p.seg_smem_off);
    seg.tile_prefix = segmem;
    seg.row_off = segmem + (MAX_SEGMENTS + 1);
    seg.expert = segmem + 2 * (MAX_SEGMENTS + 1);

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&bars.full[s], 1);
            mbar_init(&bars.empty[s], DQ_WARPS + 1);
        }
        for (int s = 0; s < p.a_slots; ++s) {
            mbar_init(&bars.afull[s], DQ_WARPS);
            mbar_init(&bars.aempty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars.accfull[s], 1);
            mbar_init(&bars.accempty[s], EPI_THREADS / 32);
        }
        mbar_init(&bars.drain, 1);
        mbar_init(&bars.epi, EPI_THREADS / 32);
        fence_mbar_init();
        abort_sh = 0;
        last_sh = 0;
        prefetch_tensormap(&tmap_a);
    }
    if (warp == MMA_WARP) {
        tmem_alloc(&tmem_base_sh, p.tmem_cols);
        tmem_relinquish();
    }
    if (warp == SEG_WARP) {
        int total = p.m_tiles * p.n_tiles;
        if (p.ex_off != nullptr)
            total = build_segments(p, seg, lane);
        if (lane == 0)
            total_tiles_sh = total;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = tmem_base_sh;
    WaitCtl ctl{&abort_sh, p.status, p.limit_ns};
    Sched sched;
    sched.init(total_tiles_sh, p.kblocks);

    if (warp == PRODUCER_WARP) {
        if (lane == 0)
            run_producer(p, &tmap_a, seg, sched, smem, bars, ctl);
    } else if (warp == MMA_WARP) {
        if (lane == 0)
            run_mma<A_TMEM>(p, seg, sched, smem, aring, bars, tmem_base, ctl);
        __syncwarp();
    } else if (warp >= EPI_WARP0 && warp < EPI_WARP0 + 4) {
        run_epilogue(p, seg, sched, bars, tmem_base, ctl, warp, lane, &last_sh);
    } else if (warp >= DQ_WARP0) {
        run_dequant<A_TMEM>(p, sched, smem, aring, bars, tmem_base, ctl, warp, lane);
    }
    __syncwarp();

    tc_fence_before();
    __syncthreads();
    if (warp == MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem_base, p.tmem_cols);
    }
}

int gemm_extra_smem(bool a_tmem, bool grouped)
{
    int bytes = 1024; // alignment slack
    if (!a_tmem)
        bytes += SMEM_A_SLOTS * A_SLOT_BYTES;
    if (grouped)
        bytes += (3 * MAX_SEGMENTS + 2) * (int)sizeof(int);
    return bytes;
}

int launch_gemm(const GemmParams &p, const CUtensorMap &tmap_a, const GemmConfig &cfg,
                cudaStream_t stream)
{
    static int attr_done[2][64];
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    const int variant = cfg.a_tmem ? 1 : 0;
    auto kernel = cfg.a_tmem ? w4a16_gemm_kernel<true> : w4a16_gemm_kernel<false>;
    if (dev < 64 && attr_done[variant][dev] < cfg.smem_bytes) {
        err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   cfg.smem_bytes);
        if (err != cudaSuccess)
            return err;
        attr_done[variant][dev] = cfg.smem_bytes;
    }
    kernel<<<cfg.grid, NUM_THREADS, cfg.smem_bytes, stream>>>(p, tmap_a);
    return cudaGetLastError();
}

int gemm_smem_limit(int *bytes)
{
    int dev = 0, optin = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    err = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (err != cudaSuccess)
        return err;
    cudaFuncAttributes fa;
    err = cudaFuncGetAttributes(&fa, w4a16_gemm_kernel<true>);
    if (err != cudaSuccess)
        return err;
    *bytes = optin - (int)fa.sharedSizeBytes;
    return cudaSuccess;
}

} // namespace w4
