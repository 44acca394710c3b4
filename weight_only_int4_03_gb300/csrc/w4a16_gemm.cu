// w4a16_gemm.cu -- the tcgen05 W4A16 GEMM kernel for sm_103a (used for larger M).
//
// Computes C[M,N] = A[M,K] x dequant(B)[K,N] (ferrum-kernels 0.8.5 marlin.rs, `marlin_gemm`
// doc) with the weights on the tcgen05 M side ("swap-AB"):
//     D[n, t] = sum_k W^T[n, k] * A^T[k, t],   D = C^T tile of 128 weight columns x T tokens.
// One persistent CTA per SM, warp-specialised:
//   warp 0       TMA producer (w4a16_common.cuh): per stage one bulk copy of packed codes,
//                one tensor copy of scales (and zeros), one 3-D copy of activation rows
//   warp 1       tcgen05.mma issuer (one thread) and tensor-memory owner
//   warps 4..7   epilogue: tensor memory -> registers -> fp16 C, or fp32 split-K partials
//   warps 8..15  dequant, two sets of four: codes -> (q - z) * s in fp16 -> tensor memory,
//                the MMA's A operand
// Work is split "data-parallel + stream-K"; tiles cut by a range boundary are summed from
// fp32 partials in a fixed order by the last contributor to finish (a self-resetting atomic
// counter), so results are deterministic and no CTA ever waits for another.
#include <cuda_fp8.h>

#include "w4a16_common.cuh"

namespace w4 {

struct Bars {
    uint64_t full[MAX_STAGES];
    uint64_t empty[MAX_STAGES];
    uint64_t afull[MAX_STAGES]; // a stage's weight slots dequantised (its dequant set)
    uint64_t accfull[2];
    uint64_t accempty[2];
    uint64_t drain;
    uint64_t split_done[2]; // the epilogue warps' partial stores of the CTA's split tiles
};

// The four k steps of one 64-row block: MMAs on the dequantised weight slot (tensor memory at
// a_tmem, or shared memory at a_smem) against the block's activation rows, into d_tmem; with
// PAIR, the second half-tile's rows (half_bytes on) into d_tmem + nt_half with the same weights.
template <bool A_TMEM, bool PAIR>
__device__ __forceinline__ void issue_block_mmas(uint32_t d_tmem, int nt_half, uint32_t a_tmem,
                                                 const uint8_t *a_smem, uint32_t act,
                                                 uint32_t half_bytes, uint32_t idesc,
                                                 uint32_t idesc2, bool accumulate)
{
    // The k steps advance the B descriptors' start address by 32 bytes (2 in its 16-byte
    // units); shared-memory addresses stay below 2^18, so the 14-bit field never carries.
    const uint64_t b0 = desc_sw128(act), b1 = desc_sw128(act + half_bytes);
#pragma unroll
    for (int kk = 0; kk < KBLK / 16; ++kk) {
        const uint32_t acc = (accumulate || kk > 0) ? 1u : 0u;
        if (A_TMEM) {
            mma_ts(d_tmem, a_tmem + kk * 8, b0 + (uint64_t)(kk * 2), idesc, acc);
            if (PAIR)
                mma_ts(d_tmem + nt_half, a_tmem + kk * 8, b1 + (uint64_t)(kk * 2), idesc2, acc);
        } else {
            const uint64_t adesc = desc_sw128(smem_u32(a_smem) + kk * 32);
            mma_ss(d_tmem, adesc, desc_sw128(act + kk * 32), idesc, acc);
            if (PAIR)
                mma_ss(d_tmem + nt_half, adesc, desc_sw128(act + half_bytes + kk * 32), idesc2, acc);
        }
    }
}

template <bool A_TMEM>
__device__ void run_mma(const GemmParams &p, const SegTable &seg, Sched sched, uint8_t *smem,
                        uint8_t *aring, Bars &bars, uint32_t tmem_base, const WaitCtl &ctl)
{
    Ring ring;
    uint32_t seg_i = 0;
    int tile, kb0, kb1;
    bool ok = true;
    while (ok && sched.next(tile, kb0, kb1)) {
        const TileInfo ti = tile_info(p, seg, tile);
        // A paired tile runs its two half-tiles as two MMAs per k step on the same weight
        // operand, into adjacent accumulator columns (half 1 starts nt_half columns on).
        const int n_first = ti.ntok < p.nt_half ? ti.ntok : p.nt_half;
        const int n_second = ti.ntok - n_first;
        const uint32_t idesc = p.bf16 ? idesc_bf16_f32(TILE_N, n_first) : idesc_f16_f32(TILE_N, n_first);
        const int n2 = n_second > 0 ? n_second : 16;
        const uint32_t idesc2 = p.bf16 ? idesc_bf16_f32(TILE_N, n2) : idesc_f16_f32(TILE_N, n2);
        const uint32_t half_bytes = (uint32_t)(p.kbs * p.act_kb_bytes);
        const int abuf = seg_i % p.acc_bufs;
        const uint32_t acc_ph = (seg_i / p.acc_bufs) & 1u;
        if (!mbar_wait(&bars.accempty[abuf], acc_ph ^ 1u, ctl, W4A16_DEV_TIMEOUT))
            break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + p.acc_col0 + abuf * p.nt_max;
        for (int kb = kb0; ok && kb < kb1; kb += p.kbs) {
            const int nkb = min(p.kbs, kb1 - kb);
            // One wait per stage: the stage's dequant set signals all of its blocks at once,
            // after waiting for the stage itself, so the activation rows have landed too.
            if (!mbar_wait(&bars.afull[ring.idx], ring.phase, ctl, W4A16_DEV_TIMEOUT)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t st = smem_u32(smem + (size_t)ring.idx * p.stage_bytes);
            const int slot0 = ring.idx * p.kbs;
            for (int j = 0; j < nkb; ++j) {
                const int aslot = slot0 + j;
                const uint32_t act = st + j * p.act_kb_bytes;
                // The single / paired choice is made per block, outside the k steps: a branch
                // between the MMAs of a block, even one never taken, slowed the kernel by 40 %.
                if (n_second > 0)
                    issue_block_mmas<A_TMEM, true>(d_tmem, p.nt_half, tmem_base + aslot * A_SLOT_COLS,
                                                   aring + aslot * A_SLOT_BYTES, act, half_bytes,
                                                   idesc, idesc2, kb + j > kb0);
                else
                    issue_block_mmas<A_TMEM, false>(d_tmem, p.nt_half, tmem_base + aslot * A_SLOT_COLS,
                                                    aring + aslot * A_SLOT_BYTES, act, half_bytes,
                                                    idesc, idesc2, kb + j > kb0);
            }
            // One commit releases the stage: its shared memory to the producer and its weight
            // slots to the dequant set that next fills the stage.
            mma_commit(&bars.empty[ring.idx]);
            ring.advance(p.stages);
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

// Dequant: two sets of four warps (one warp per tensor-memory lane quarter).  Consecutive
// stages alternate between the sets; a set converts all of its stage's blocks into the stage's
// own weight slots (slot stage * kbs + j), issues their tensor-memory stores and waits for them
// once.  Each thread owns one weight column (lane) and turns the 8 words of its column in a
// block into 64 fp16 values: 32 tensor-memory columns.
constexpr int DQ_SETS = DQ_WARPS / 4;

// grp_rel >= 0: the block lies in one group, row grp_rel of the stage's scales; otherwise
// each 8-row pair looks up its own group.
template <bool A_TMEM>
__device__ __forceinline__ void dequant_block(const GemmParams &p, const uint8_t *packed,
                                              const __half *ssm, const __half *zsm, int kb,
                                              int g_first, int grp_rel, int nl, bool has_zp,
                                              uint32_t dst_tmem, uint8_t *dst_smem)
{
    __half2 s2[4], zlo[4], zhi[4];
    if (grp_rel >= 0)
        load_scales_row(ssm, zsm, has_zp, grp_rel, nl, s2, zlo, zhi);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        if (grp_rel < 0)
            load_scales(p, ssm, zsm, has_zp, kb, h, g_first, nl, s2, zlo, zhi);
        const uint4 wv = *reinterpret_cast<const uint4 *>(packed + (h * 512 + nl * 4) * 4);
        const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
        uint32_t out[16];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            // word jj holds rows 2jj + 8pp + {0,1}: tensor-memory column jj + 4pp of the half
            uint32_t o4[4];
            dequant_word(words[jj], zlo, zhi, s2, o4);
#pragma unroll
            for (int pp = 0; pp < 4; ++pp)
                out[jj + 4 * pp] = o4[pp];
        }
        if (A_TMEM) {
            tmem_st16(dst_tmem + h * 16, out);
        } else {
            uint8_t *rowp = dst_smem + nl * 128;
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                const int chunk = h * 4 + q4;
                *reinterpret_cast<uint4 *>(rowp + ((chunk ^ (nl & 7)) << 4)) =
                    make_uint4(out[q4 * 4], out[q4 * 4 + 1], out[q4 * 4 + 2], out[q4 * 4 + 3]);
            }
        }
    }
}

// FP8 E4M3: the thread's column holds its block's 64 rows as 16 words of four K-consecutive
// codes (word (q, t) = rows 16q + 4t .. 16q + 4t + 3, at q*512 + c*4 + t); each 16-bit half
// converts exactly to an fp16 pair (rows 2p, 2p+1 -> tensor-memory column p), and one multiply
// by the group's scale rounds it.  The block lies in one group (group_size -1 or a multiple of
// 64 for FP8).
template <bool A_TMEM>
__device__ __forceinline__ void dequant_block_fp8(const uint8_t *packed, const __half *ssm, int grp_rel,
                                                  int nl, uint32_t dst_tmem, uint8_t *dst_smem)
{
    const __half2 s = __half2half2(ssm[grp_rel * TILE_N + nl]);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        uint32_t out[16];
#pragma unroll
        for (int qq = 0; qq < 2; ++qq) {
            const int q = hh * 2 + qq;
            const uint4 wv = *reinterpret_cast<const uint4 *>(packed + (q * 512 + nl * 4) * 4);
            const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(
                    (__nv_fp8x2_storage_t)(words[t] & 0xFFFFu), __NV_E4M3);
                const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(
                    (__nv_fp8x2_storage_t)(words[t] >> 16), __NV_E4M3);
                out[qq * 8 + 2 * t] = h2_as_u32(__hmul2(__half2(lo), s));
                out[qq * 8 + 2 * t + 1] = h2_as_u32(__hmul2(__half2(hi), s));
            }
        }
        if (A_TMEM) {
            tmem_st16(dst_tmem + hh * 16, out);
        } else {
            uint8_t *rowp = dst_smem + nl * 128;
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                const int chunk = hh * 4 + q4;
                *reinterpret_cast<uint4 *>(rowp + ((chunk ^ (nl & 7)) << 4)) =
                    make_uint4(out[q4 * 4], out[q4 * 4 + 1], out[q4 * 4 + 2], out[q4 * 4 + 3]);
            }
        }
    }
}

// bfloat16 operands (7 fraction bits).
__device__ __forceinline__ __nv_bfloat162 u32_as_bf2(uint32_t v)
{
    return *reinterpret_cast<__nv_bfloat162 *>(&v);
}

__device__ __forceinline__ uint32_t bf2_as_u32(__nv_bfloat162 v)
{
    return *reinterpret_cast<uint32_t *>(&v);
}

// Scale and -(128 + zero) of one (group, column), as bf16 pairs.
__device__ __forceinline__ void bf16_scale_zero(const uint16_t *ssm, const uint16_t *zsm, bool has_zp,
                                                int idx, __nv_bfloat162 &s2, __nv_bfloat162 &z2)
{
    s2 = __bfloat162bfloat162(__ushort_as_bfloat16(ssm[idx]));
    __nv_bfloat16 zb = __ushort_as_bfloat16((uint16_t)0xC308); // -136 = -(128 + 8)
    if (has_zp)
        zb = __hneg(__hadd(__ushort_as_bfloat16((uint16_t)0x4300), __ushort_as_bfloat16(zsm[idx])));
    z2 = __bfloat162bfloat162(zb);
}

// One word's four row pairs (bits 4p, 16 + 4p) as bf16 pairs (q - z) * s.  The fraction of a
// bf16 has 7 bits (bit 7 is the exponent's lowest), so each nibble is first moved to bits 0-3
// (shifts as high halves of products, on the FMA pipe) and OR-ed into 128.0 (0x4300, spacing
// 1): 128 + q exactly.  Adding -(128 + z) is exact for integer zero points; the product with
// the scale rounds once.
__device__ __forceinline__ void dequant_word_bf16(uint32_t x, const __nv_bfloat162 (&z2)[4],
                                                  const __nv_bfloat162 (&s2)[4], uint32_t (&out)[4])
{
    const uint32_t xs[4] = {x, __umulhi(x, 1u << 28), __umulhi(x, 1u << 24), __umulhi(x, 1u << 20)};
#pragma unroll
    for (int pp = 0; pp < 4; ++pp) {
        const uint32_t t = (xs[pp] & 0x000F000Fu) | 0x43004300u;
        out[pp] = bf2_as_u32(__hmul2(__hadd2(u32_as_bf2(t), z2[pp]), s2[pp]));
    }
}

// grp_rel >= 0: the block lies in one group, row grp_rel of the stage's scales; otherwise
// each 8-row pair looks up its own group.
template <bool A_TMEM>
__device__ __forceinline__ void dequant_block_bf16(const GemmParams &p, const uint8_t *packed,
                                                   const uint16_t *ssm, const uint16_t *zsm, int kb,
                                                   int g_first, int grp_rel, int nl, bool has_zp,
                                                   uint32_t dst_tmem, uint8_t *dst_smem)
{
    __nv_bfloat162 s2[4], z2[4];
    if (grp_rel >= 0) {
        bf16_scale_zero(ssm, zsm, has_zp, grp_rel * TILE_N + nl, s2[0], z2[0]);
#pragma unroll
        for (int pp = 1; pp < 4; ++pp) {
            s2[pp] = s2[0];
            z2[pp] = z2[0];
        }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        if (grp_rel < 0) {
#pragma unroll
            for (int pp = 0; pp < 4; ++pp) {
                const int gl = (kb * KBLK + h * 32 + pp * 8) / p.group_size - g_first;
                bf16_scale_zero(ssm, zsm, has_zp, gl * TILE_N + nl, s2[pp], z2[pp]);
            }
        }
        const uint4 wv = *reinterpret_cast<const uint4 *>(packed + (h * 512 + nl * 4) * 4);
        const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
        uint32_t out[16];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            // word jj holds rows 2jj + 8pp + {0,1} at bits (4pp, 16 + 4pp): column jj + 4pp
            uint32_t o4[4];
            dequant_word_bf16(words[jj], z2, s2, o4);
#pragma unroll
            for (int pp = 0; pp < 4; ++pp)
                out[jj + 4 * pp] = o4[pp];
        }
        if (A_TMEM) {
            tmem_st16(dst_tmem + h * 16, out);
        } else {
            uint8_t *rowp = dst_smem + nl * 128;
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                const int chunk = h * 4 + q4;
                *reinterpret_cast<uint4 *>(rowp + ((chunk ^ (nl & 7)) << 4)) =
                    make_uint4(out[q4 * 4], out[q4 * 4 + 1], out[q4 * 4 + 2], out[q4 * 4 + 3]);
            }
        }
    }
}

// Weight kinds of the tcgen05 kernel: 4-bit codes with fp16 operands, FP8 E4M3 codes with
// fp16 operands, 4-bit codes with bf16 operands.
constexpr int WK_U4_F16 = 0, WK_FP8_F16 = 1, WK_U4_BF16 = 2;

template <bool A_TMEM, int WK>
__device__ void run_dequant(const GemmParams &p, Sched sched, uint8_t *smem, uint8_t *aring,
                            Bars &bars, uint32_t tmem_base, const WaitCtl &ctl, int warp, int lane)
{
    const int q = warp & 3;
    const int set = (warp - DQ_WARP0) >> 2;
    const int nl = q * 32 + lane;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    const bool has_zp = p.zeros != nullptr;
    const int gs = p.group_size;
    const int gs_kb = (gs % KBLK == 0) ? gs / KBLK : 0; // 64-row blocks per group, or 0
    const int gs_sh = group_shift(gs_kb);
    Ring ring;
    // Stages of several blocks are shared: set s converts blocks s, s + DQ_SETS, ... of every
    // stage, and both sets arrive on the stage's barrier (count 8), whether they had a block in
    // it or not.  Stages of one block (the tall paired tiles) go to the sets in turn (count 4).
    // With an even stage count a ring slot then always belongs to the same set, which so sees
    // every phase of that slot's barrier in order and skips the other set's stages altogether;
    // with an odd count ownership of a slot alternates, and a set that skipped could wait on a
    // phase two ahead of the barrier, which a parity test cannot tell from the one before, so
    // both sets then wait for every stage.
    const bool shared = p.kbs > 1;
    const bool lockstep = shared || (p.stages % DQ_SETS) != 0;
    int owner_set = 0; // dequant set of the next one-block stage
    int tile, kb0, kb1;
    while (sched.next(tile, kb0, kb1)) {
        for (int kb = kb0; kb < kb1; kb += p.kbs) {
            const int nkb = min(p.kbs, kb1 - kb);
            // A stage's weight slots are free once the stage has landed: the producer refilled
            // it only after the MMAs that last read those slots completed.
            bool mine = set < nkb;
            if (!shared) {
                mine = owner_set == set;
                owner_set = (owner_set + 1 == DQ_SETS) ? 0 : owner_set + 1;
            }
            if (!mine && !lockstep) {
                ring.advance(p.stages);
                continue;
            }
            if (!mbar_wait(&bars.full[ring.idx], ring.phase, ctl, W4A16_DEV_TIMEOUT))
                return;
            if (!mine) {
                if (shared) {
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&bars.afull[ring.idx]);
                }
                ring.advance(p.stages);
                continue;
            }
            tc_fence_after();
            const uint8_t *st = smem + (size_t)ring.idx * p.stage_bytes;
            const __half *ssm = reinterpret_cast<const __half *>(st + p.scales_off);
            const __half *zsm = reinterpret_cast<const __half *>(st + p.zeros_off);
            const int g_first = (kb * KBLK) / gs;
            const int slot0 = ring.idx * p.kbs;
            const int jstep = shared ? DQ_SETS : 1;
            for (int j = shared ? set : 0; j < nkb; j += jstep) {
                const int slot = slot0 + j;
                const int kbj = kb + j;
                const int grp_rel = gs_kb == 0   ? -1
                                    : gs_sh >= 0 ? (kbj >> gs_sh) - g_first
                                                 : kbj / gs_kb - g_first;
                if (WK == WK_FP8_F16)
                    dequant_block_fp8<A_TMEM>(st + p.packed_off + j * TILE_BYTES_FP8, ssm, grp_rel,
                                              nl, tmem_base + lane_base + slot * A_SLOT_COLS,
                                              aring + slot * A_SLOT_BYTES);
                else if (WK == WK_U4_BF16)
                    dequant_block_bf16<A_TMEM>(p, st + p.packed_off + j * TILE_BYTES,
                                               reinterpret_cast<const uint16_t *>(ssm),
                                               reinterpret_cast<const uint16_t *>(zsm), kbj,
                                               g_first, grp_rel, nl, has_zp,
                                               tmem_base + lane_base + slot * A_SLOT_COLS,
                                               aring + slot * A_SLOT_BYTES);
                else
                    dequant_block<A_TMEM>(p, st + p.packed_off + j * TILE_BYTES, ssm, zsm, kbj,
                                          g_first, grp_rel, nl, has_zp,
                                          tmem_base + lane_base + slot * A_SLOT_COLS,
                                          aring + slot * A_SLOT_BYTES);
            }
            if (A_TMEM) {
                tmem_st_wait();
                tc_fence_before();
            } else {
                fence_proxy_async_smem();
            }
            // One arrival per warp and stage: every lane's writes are complete and fenced first.
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&bars.afull[ring.idx]);
            ring.advance(p.stages);
        }
    }
}

// Split tiles get only their fp32 partial here.  The segment that starts a stream-K range
// arrives on its tile's counter as soon as the four epilogue warps have stored it, long before
// the contributor whose range ends in that tile, which so is the tile's last arriver and a CTA
// is last for at most one tile; the other split segments arrive, and every reduction runs,
// once the whole CTA is done (see the kernel's end), when all of its threads can share it.
__device__ void run_epilogue(const GemmParams &p, const SegTable &seg, Sched sched, Bars &bars,
                             uint32_t tmem_base, uint8_t *smem, const WaitCtl &ctl, int warp,
                             int lane, int *split_tiles, volatile int *split_last, int *n_split)
{
    const int q = warp & 3;
    __half *stg = reinterpret_cast<__half *>(smem + p.epi_smem_off) + q * EPI_ROWS * 32;
    uint16_t *stg16 = reinterpret_cast<uint16_t *>(stg); // fp16 or bf16 bits
    const int nl = q * 32 + lane;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    uint32_t seg_i = 0, n_seen = 0; // n_seen: split segments so far
    int tile, kb0, kb1;
    while (sched.next(tile, kb0, kb1)) {
        const TileInfo ti = tile_info(p, seg, tile);
        const int abuf = seg_i % p.acc_bufs;
        const uint32_t acc_ph = (seg_i / p.acc_bufs) & 1u;
        if (!mbar_wait(&bars.accfull[abuf], acc_ph, ctl, W4A16_DEV_TIMEOUT))
            return;
        tc_fence_after();
        const uint32_t taddr = tmem_base + lane_base + p.acc_col0 + abuf * p.nt_max;
        const bool whole = (kb0 == 0 && kb1 == p.kblocks);
        const long long st_tile = (long long)tile - sched.dp_tiles;
        float *part = whole ? nullptr : partial_slot(p, sched.cta, own_slot(p, sched, st_tile));
        // Batches of 32 token rows: two tensor-memory loads and their wait (tens of cycles),
        // then the batch's output.  A split tile's fp32 partial goes straight from the registers
        // (each store a coalesced 128-byte row of the slot).  A whole tile goes out through this
        // warp's staging buffer (its 32 columns x 32 rows as 16-bit values), so that each lane
        // writes 16-byte runs of a C row instead of single halves.  Each path is its own short
        // loop with the per-call choices (gating, row weights, row mapping) made outside the
        // unrolled parts: the accumulator is held until the last batch has been read, and a
        // loop carrying every case, with the next batch's loads issued early, took twice as
        // long per batch in place.
        const bool weighted = p.row_weight != nullptr;
        const bool dense = p.ex_off == nullptr;
        // The accumulator is released as soon as the last batch has been read from tensor
        // memory, before that batch is written out.
        bool released = false;
        auto release = [&]() {
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&bars.accempty[abuf]);
            released = true;
        };
        if (whole && p.glu) {
            // Gated tiles keep the next batch's loads issued as soon as this batch is staged:
            // measured faster for them (MoE gate_up with SwiGLU 397 -> 344 us).
            uint32_t v[32];
            auto load_batch = [&](int c0) {
                tmem_ld16(taddr + c0, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
                if (c0 + 16 < ti.ntok)
                    tmem_ld16(taddr + c0 + 16, *reinterpret_cast<uint32_t(*)[16]>(&v[16]));
            };
            load_batch(0);
            for (int c0 = 0; c0 < ti.ntok; c0 += EPI_ROWS) {
                const bool more = c0 + EPI_ROWS < ti.ntok;
                const int nr = ti.rows - c0;
                tmem_ld_wait();
                if (!more)
                    release();
                float rw = 1.0f;
                if (weighted && lane < nr) {
                    const int orow = p.ex_pairs[ti.row0 + c0 + lane];
                    if (orow >= 0 && orow < p.n_pairs)
                        rw = p.row_weight[orow];
                }
                // Lanes 0..15 hold gate features n0/2 + 16q + lane, lanes 16..31 the up values
                // of the same features: 32 rows x 16 features through the staging buffer.
#pragma unroll
                for (int j = 0; j < EPI_ROWS; ++j) {
                    const float g = __uint_as_float(v[j]);
                    const float u = __shfl_down_sync(0xffffffffu, g, 16);
                    const float w = weighted ? __shfl_sync(0xffffffffu, rw, j) : 1.0f;
                    if (lane < 16)
                        stg16[j * 16 + lane] = to_out16(glu_act(g, p.glu) * u * w, p.bf16);
                }
                __syncwarp();
                if (more)
                    load_batch(c0 + EPI_ROWS);
#pragma unroll
                for (int i = 0; i < EPI_ROWS / 16; ++i) {
                    const int r = i * 16 + (lane >> 1);
                    const int cseg = (lane & 1) * 8;
                    const uint4 val = *reinterpret_cast<const uint4 *>(stg + r * 16 + cseg);
                    if (r < nr) {
                        const int out_row = output_row(p, ti, c0 + r);
                        if (out_row >= 0)
                            __stcs(reinterpret_cast<uint4 *>(p.c + (long long)out_row * p.ldc +
                                                             ti.n0 / 2 + q * 16 + cseg),
                                   val);
                    }
                }
                __syncwarp();
            }
        } else {
            for (int c0 = 0; c0 < ti.ntok; c0 += EPI_ROWS) {
                uint32_t v[32];
                tmem_ld16(taddr + c0, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
                if (c0 + 16 < ti.ntok)
                    tmem_ld16(taddr + c0 + 16, *reinterpret_cast<uint32_t(*)[16]>(&v[16]));
                tmem_ld_wait();
                if (c0 + EPI_ROWS >= ti.ntok)
                    release();
                const int nr = ti.rows - c0; // rows of this batch that exist (all 32 when >= 32)
                if (!whole) {
                    float *dst = part + c0 * TILE_N + nl;
                    if (nr >= EPI_ROWS) {
#pragma unroll
                        for (int j = 0; j < EPI_ROWS; ++j)
                            __stcg(dst + j * TILE_N, __uint_as_float(v[j]));
                    } else {
#pragma unroll
                        for (int j = 0; j < EPI_ROWS; ++j)
                            if (j < nr)
                                __stcg(dst + j * TILE_N, __uint_as_float(v[j]));
                    }
                    continue;
                }
                // Block-routed calls may scale each output row (top-k weights): lane j holds the
                // weight of row c0 + j, handed to every lane by a shuffle.
                float rw = 1.0f;
                if (weighted && lane < nr) {
                    const int orow = p.ex_pairs[ti.row0 + c0 + lane];
                    if (orow >= 0 && orow < p.n_pairs)
                        rw = p.row_weight[orow];
                }
                if (weighted) {
#pragma unroll
                    for (int j = 0; j < EPI_ROWS; ++j)
                        stg16[j * 32 + lane] =
                            to_out16(__uint_as_float(v[j]) * __shfl_sync(0xffffffffu, rw, j), p.bf16);
                } else {
#pragma unroll
                    for (int j = 0; j < EPI_ROWS; ++j)
                        stg16[j * 32 + lane] = to_out16(__uint_as_float(v[j]), p.bf16);
                }
                __syncwarp();
                if (dense) {
                    // Rows map to C rows row0 + row: written once, streaming stores (first out of L2).
                    const long long row_base = (long long)(ti.row0 + c0);
#pragma unroll
                    for (int i = 0; i < EPI_ROWS / 8; ++i) {
                        const int r = i * 8 + (lane >> 2);
                        const int cseg = (lane & 3) * 8;
                        const uint4 val = *reinterpret_cast<const uint4 *>(stg + r * 32 + cseg);
                        if (r < nr)
                            __stcs(reinterpret_cast<uint4 *>(p.c + (row_base + r) * p.ldc + ti.n0 +
                                                             q * 32 + cseg),
                                   val);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < EPI_ROWS / 8; ++i) {
                        const int r = i * 8 + (lane >> 2);
                        const int cseg = (lane & 3) * 8;
                        const uint4 val = *reinterpret_cast<const uint4 *>(stg + r * 32 + cseg);
                        if (r < nr) {
                            const int out_row = output_row(p, ti, c0 + r);
                            if (out_row >= 0)
                                __stcs(reinterpret_cast<uint4 *>(p.c + (long long)out_row * p.ldc +
                                                                 ti.n0 + q * 32 + cseg),
                                       val);
                        }
                    }
                }
                __syncwarp();
            }
        }
        if (!released)
            release();
        ++seg_i;
        if (!whole && kb1 == p.kblocks && sched.split == 0 && n_seen < 2) {
            // A stream-K segment that ends at its tile's end: the start of this CTA's range,
            // done long before the range's end.  Arrive now: every lane's partial stores are
            // made visible at GPU scope, each warp arrives on this split tile's rendezvous (a
            // barrier of its own, used once), and one thread, once all four have (a bounded
            // wait: no thread waits on a warp that gave up), makes the acquire-release arrival.
            __threadfence();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&bars.split_done[n_seen]);
            if (warp == EPI_WARP0 && lane == 0) {
                if (!mbar_wait(&bars.split_done[n_seen], 0, ctl, W4A16_DEV_TIMEOUT))
                    return;
                const Contributors cb = contributors(p, sched, st_tile);
                const int old = split_counter_arrive(&p.counters[tile]);
                split_tiles[*n_split] = tile;
                split_last[*n_split] = old == (cb.hi - cb.lo);
                ++*n_split;
            }
            ++n_seen;
        } else if (!whole && warp == EPI_WARP0 && lane == 0) {
            split_tiles[*n_split] = tile; // arrives at the CTA's end
            split_last[*n_split] = -1;
            ++*n_split;
        }
    }
}

template <bool A_TMEM, int WK>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    w4a16_gemm_kernel(const __grid_constant__ GemmParams p, const __grid_constant__ CUtensorMap tmap_a,
                      const __grid_constant__ CUtensorMap tmap_s, const __grid_constant__ CUtensorMap tmap_z)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ Bars bars;
    __shared__ uint32_t tmem_base_sh;
    __shared__ volatile int abort_sh;
    __shared__ volatile int last_sh[2];
    __shared__ int split_tiles_sh[2];
    __shared__ int n_split_sh;
    __shared__ int total_tiles_sh;
    __shared__ int pre_sh;

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
            mbar_init(&bars.empty[s], 1); // the MMA warp's commit
        }
        for (int s = 0; s < p.stages; ++s)   // the warps of the sets converting the stage
            mbar_init(&bars.afull[s], p.kbs > 1 ? 4 * DQ_SETS : 4);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars.accfull[s], 1);
            mbar_init(&bars.accempty[s], EPI_THREADS / 32);
        }
        mbar_init(&bars.drain, 1);
        mbar_init(&bars.split_done[0], EPI_THREADS / 32);
        mbar_init(&bars.split_done[1], EPI_THREADS / 32);
        fence_mbar_init();
        abort_sh = 0;
        last_sh[0] = last_sh[1] = 0;
        n_split_sh = 0;
        prefetch_tensormap(&tmap_a);
        prefetch_tensormap(&tmap_s);
        if (p.zeros != nullptr)
            prefetch_tensormap(&tmap_z);
        // Static weights of a dense call: the codes and scales of the first stages go out
        // before the dependency wait, overlapping the preceding kernel's tail (the schedule of
        // a dense call reads nothing from memory; a grouped one needs its segment table).
        pre_sh = 0;
        if (p.static_weights && p.ex_off == nullptr) {
            Sched first;
            first.init(p.m_tiles * p.n_tiles, p.kblocks, p.split);
            pre_sh = issue_static_weights(p, &tmap_s, &tmap_z, seg, first, smem, bars.full);
        }
    }
    if (warp == MMA_WARP) {
        tmem_alloc(&tmem_base_sh, p.tmem_cols);
        tmem_relinquish();
    }
    // Everything above touches only this CTA's resources, so it may overlap the previous
    // kernel; from here on global memory written by earlier work is read.
    if (threadIdx.x == 0)
        pdl_launch_dependents();
    pdl_wait();
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
    sched.init(total_tiles_sh, p.kblocks, p.split);

    if (warp == PRODUCER_WARP) {
        if (lane == 0)
            run_producer(p, &tmap_a, &tmap_s, &tmap_z, seg, sched, smem, bars.full, bars.empty, ctl,
                         pre_sh);
    } else if (warp == MMA_WARP) {
        if (lane == 0)
            run_mma<A_TMEM>(p, seg, sched, smem, aring, bars, tmem_base, ctl);
    } else if (warp >= EPI_WARP0 && warp < EPI_WARP0 + 4) {
        run_epilogue(p, seg, sched, bars, tmem_base, smem, ctl, warp, lane, split_tiles_sh,
                     last_sh, &n_split_sh);
    } else if (warp >= DQ_WARP0) {
        run_dequant<A_TMEM, WK>(p, sched, smem, aring, bars, tmem_base, ctl, warp, lane);
    }
    __syncwarp();

    tc_fence_before();
    __syncthreads();
    if (warp == MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem_base, p.tmem_cols);
    }

    // Split tiles of this CTA (at most two: where its range starts and ends).  The one that
    // starts the range was counted in by the epilogue; the others arrive here (the barrier
    // above orders the partial stores before the atomics; release is cumulative).  The last
    // contributor of a tile sums the partials with all of the CTA's threads (the acquire half
    // of its arrival, and a barrier, make the other contributors' partials visible to all).
    const int n_split = n_split_sh;
    if (n_split == 0 || abort_sh)
        return;
    if (threadIdx.x < n_split && last_sh[threadIdx.x] < 0) {
        const int tile = split_tiles_sh[threadIdx.x];
        const Contributors cb = contributors(p, sched, (long long)tile - sched.dp_tiles);
        const int old = split_counter_arrive(&p.counters[tile]);
        last_sh[threadIdx.x] = old == (cb.hi - cb.lo);
    }
    __syncthreads();
    for (int i = 0; i < n_split; ++i) {
        if (!last_sh[i])
            continue;
        const int tile = split_tiles_sh[i];
        const TileInfo ti = tile_info(p, seg, tile);
        const Contributors cb = contributors(p, sched, (long long)tile - sched.dp_tiles);
        if (p.glu)
            reduce_tile_glu(p, ti, cb, threadIdx.x, NUM_THREADS);
        else if (ti.rows * (TILE_N / 4) <= 4 * NUM_THREADS)
            // A short tile (up to 64 rows, typically 4+ contributors): one round of 4 items per
            // thread covers it, with 4 contributors' loads in flight.
            reduce_tile<4, 4>(p, ti, cb, threadIdx.x, NUM_THREADS);
        else
            // Taller tiles (2-3 contributors): 8 items x 2 contributors in flight per thread.
            reduce_tile<8, 2>(p, ti, cb, threadIdx.x, NUM_THREADS);
        if (threadIdx.x == 0)
            p.counters[tile] = 0;
    }
}

int gemm_extra_smem(bool a_tmem, bool grouped)
{
    int bytes = 1024 + EPI_STAGE_BYTES; // alignment slack, epilogue staging
    if (!a_tmem)
        bytes += SMEM_A_SLOTS * A_SLOT_BYTES;
    if (grouped)
        bytes += (3 * MAX_SEGMENTS + 2) * (int)sizeof(int);
    return bytes;
}

static int launch_pdl(const void *kernel_fn, int grid, int threads, int smem, cudaStream_t stream,
                      void **args)
{
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(grid);
    lc.blockDim = dim3(threads);
    lc.dynamicSmemBytes = smem;
    lc.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    return cudaLaunchKernelExC(&lc, kernel_fn, args);
}

int launch_gemm(const GemmParams &p, const CUtensorMap &tmap_a, const CUtensorMap &tmap_s,
                const CUtensorMap &tmap_z, const GemmConfig &cfg, cudaStream_t stream)
{
    static int attr_done[6][64];
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    const int wk = p.w8 ? WK_FP8_F16 : p.bf16 ? WK_U4_BF16 : WK_U4_F16;
    const int variant = (cfg.a_tmem ? 1 : 0) + 2 * wk;
    void (*kernels[6])(GemmParams, CUtensorMap, CUtensorMap, CUtensorMap) = {
        w4a16_gemm_kernel<false, WK_U4_F16>,  w4a16_gemm_kernel<true, WK_U4_F16>,
        w4a16_gemm_kernel<false, WK_FP8_F16>, w4a16_gemm_kernel<true, WK_FP8_F16>,
        w4a16_gemm_kernel<false, WK_U4_BF16>, w4a16_gemm_kernel<true, WK_U4_BF16>};
    auto kernel = kernels[variant];
    if (dev < 64 && attr_done[variant][dev] < cfg.smem_bytes) {
        err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   cfg.smem_bytes);
        if (err != cudaSuccess)
            return err;
        attr_done[variant][dev] = cfg.smem_bytes;
    }
    // Programmatic stream serialisation: the kernel may be scheduled while the previous
    // kernel of the stream drains; it waits (griddepcontrol.wait) before reading its inputs.
    void *args[] = {const_cast<GemmParams *>(&p), const_cast<CUtensorMap *>(&tmap_a),
                    const_cast<CUtensorMap *>(&tmap_s), const_cast<CUtensorMap *>(&tmap_z)};
    return launch_pdl(reinterpret_cast<const void *>(kernel), cfg.grid, NUM_THREADS, cfg.smem_bytes,
                      stream, args);
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
    err = cudaFuncGetAttributes(&fa, w4a16_gemm_kernel<true, WK_U4_F16>);
    if (err != cudaSuccess)
        return err;
    *bytes = optin - (int)fa.sharedSizeBytes - 256;
    return cudaSuccess;
}

} // namespace w4
