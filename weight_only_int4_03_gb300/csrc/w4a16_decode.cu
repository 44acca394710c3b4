// w4a16_decode.cu -- the small-M W4A16 GEMMs: weights dequantised in registers straight into
// warp-level mma.sync (m16n8k16), for decode-sized M (up to 64 rows).  Two kernels share the
// per-lane fragment work described here: the split-K kernel (w4a16_decode_kernel, below) and
// the column-slice kernel (w4a16_slice_kernel, at the end of the file; no split-K).
//
// Why a second kernel: at small M the job is to stream the packed weights at HBM speed, which
// leaves a budget of roughly 20 warp instructions per 32-bit word of codes.  The tcgen05
// kernel stages every dequantised weight in tensor (or shared) memory and reads it back as an
// MMA operand, and a 128x16x16 tcgen05.mma costs about as much as a 128x64x16 one; both cap
// the weight rate well below the HBM rate.  Here the weights never leave registers.
//
// Operand roles ("swap-AB", as in the tcgen05 kernel): the weights are the MMA's A operand
// (16 weight columns x 16 k), the activations its B operand (16 k x 8 tokens), so one MMA
// consumes 256 weights whatever M is, and one B fragment (loaded from the swizzled stage by
// ldmatrix) serves a whole warp's 16 columns.  The tile layout puts in each 32-bit word
// exactly what one lane needs of an A fragment for two 16-row k steps: word j of column c
// holds rows 8p + 2j + {0,1}, p = 0..3, i.e. fragment registers a0 / a2 of step 0 (p = 0, 1)
// and of step 1 (p = 2, 3); column c + 8 gives a1 / a3.
//
// Budget: the loop is kept to the dequantisation proper, one shared load per word, one
// ldmatrix per 32 rows and one MMA per word.  When a group covers whole blocks
// (group_size % 64 == 0) a lane's scale and zero change only where a group ends, which a
// per-stage bit mask marks, and the scale leaves the loop altogether: the MMAs of a group
// take the exact integers (q - z) and accumulate sum_k (q - z) a in fp32, and at the group's
// end that sum is multiplied by the column's scale and added to the output accumulator --
// the same product regrouped, since the scale is constant along K within a group (on the
// MMA's M side, one per accumulator row).  That leaves 9 instructions per 8 codes (an
// integer shift, four and-or, four fp16 add/fma) instead of 13, and it drops a rounding:
// (q - z) s is never rounded to fp16.  Groups smaller than a block, and tiles of more than
// 16 tokens (whose accumulators leave no registers for a second set), keep the scale in the
// dequantisation.
//
// Split-K kernel CTA: one TMA producer warp (the producer of w4a16_common.cuh) and 8 compute
// warps; warp w owns 16 weight columns of every 64-row block (16 columns x 64 rows = 4 words
// per lane).
// Two CTAs share an SM, so one CTA's segment epilogue (partials, the split counter, the
// reduction) overlaps the other's streaming.  Work is split over CTAs with the same
// data-parallel + stream-K schedule as the tcgen05 kernel; split tiles are reduced in a fixed
// order by the last contributor.
#include <cuda_fp8.h>
#include <type_traits>

#include "w4a16_common.cuh"

namespace w4 {

constexpr int DEC_WARPS = 8; // compute warps
constexpr int DEC_THREADS = (DEC_WARPS + 1) * 32;
constexpr int DEC_CTAS_PER_SM = 2;

struct DecBars {
    uint64_t full[MAX_STAGES];
    uint64_t empty[MAX_STAGES];
    uint64_t epi;
};

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// A plain shared-memory load (not inline assembly), so the compiler may schedule the code
// words of later blocks early; the stage's mbarrier wait (a memory clobber) keeps them after
// the data has landed.
__device__ __forceinline__ uint32_t lds32(uint32_t addr)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (uint32_t)__cvta_generic_to_shared(smem_raw);
    return *reinterpret_cast<const uint32_t *>(smem_raw + (addr - base));
}

__device__ __forceinline__ uint16_t lds16(uint32_t addr)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (uint32_t)__cvta_generic_to_shared(smem_raw);
    return *reinterpret_cast<const uint16_t *>(smem_raw + (addr - base));
}

// D (f32 16x8) += A (16x16, row) * B (16x8, col), fp16 or (BF) bf16 operands.  Registers
// only, so the compiler may schedule it freely.
template <bool BF>
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1)
{
    if (BF)
        asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
            "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    else
        asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
            "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D (f32 16x8) = A * B with no accumulator input, fp16 or (BF) bf16 operands.
template <bool BF>
__device__ __forceinline__ void mma_16816_z(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                            uint32_t a3, uint32_t b0, uint32_t b1)
{
    if (BF)
        asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
            "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%10, %10, %10, %10};"
            : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
    else
        asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
            "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%10, %10, %10, %10};"
            : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

__device__ __forceinline__ __nv_bfloat162 u32_as_bf2(uint32_t v)
{
    return *reinterpret_cast<__nv_bfloat162 *>(&v);
}

__device__ __forceinline__ uint32_t bf2_as_u32(__nv_bfloat162 v)
{
    return *reinterpret_cast<uint32_t *>(&v);
}

// Codes -> pairs (q - z) for one column (one zero for all 8 codes), exact: pair p of word x
// sits at bits (4p, 16 + 4p).  fp16: the nibbles at bits 0-3 go into 1024.0 (spacing 1) and
// those at bits 4-7 into 1024.0 at spacing 16 (undone by an fma with 1/16); zlo = 1024 + z,
// zhi = -(64 + z).  bf16 (7 fraction bits): every nibble is first shifted to bits 0-3 and
// OR-ed into 128.0; zlo = -(128 + z).
template <bool BF>
__device__ __forceinline__ void dequant_word_int(uint32_t x, uint32_t zlo, uint32_t zhi,
                                                 uint32_t (&out)[4])
{
    if (BF) {
        const uint32_t xs[4] = {x, __umulhi(x, 1u << 28), __umulhi(x, 1u << 24), __umulhi(x, 1u << 20)};
#pragma unroll
        for (int pp = 0; pp < 4; ++pp)
            out[pp] = bf2_as_u32(__hadd2(u32_as_bf2((xs[pp] & 0x000F000Fu) | 0x43004300u),
                                         u32_as_bf2(zlo)));
        return;
    }
    const uint32_t magic = 0x64006400u;
    const __half2 sixteenth = __halves2half2(__ushort_as_half(0x2C00), __ushort_as_half(0x2C00));
    const uint32_t x8 = __umulhi(x, 1u << 24); // x >> 8, on the FMA pipe (the integer pipe is the busy one)
    out[0] = h2_as_u32(__hsub2(u32_as_h2((x & 0x000F000Fu) | magic), u32_as_h2(zlo)));
    out[1] = h2_as_u32(__hfma2(u32_as_h2((x & 0x00F000F0u) | magic), sixteenth, u32_as_h2(zhi)));
    out[2] = h2_as_u32(__hsub2(u32_as_h2((x8 & 0x000F000Fu) | magic), u32_as_h2(zlo)));
    out[3] = h2_as_u32(__hfma2(u32_as_h2((x8 & 0x00F000F0u) | magic), sixteenth, u32_as_h2(zhi)));
}

// The same pairs times the column's scale s: (q - z) is exact; the product is rounded once.
template <bool BF>
__device__ __forceinline__ void dequant_word_col(uint32_t x, uint32_t zlo, uint32_t zhi, uint32_t s,
                                                 uint32_t (&out)[4])
{
    uint32_t v[4];
    dequant_word_int<BF>(x, zlo, zhi, v);
#pragma unroll
    for (int pp = 0; pp < 4; ++pp)
        out[pp] = BF ? bf2_as_u32(__hmul2(u32_as_bf2(v[pp]), u32_as_bf2(s)))
                     : h2_as_u32(__hmul2(u32_as_h2(v[pp]), u32_as_h2(s)));
}

// Scale (as a broadcast pair of 16-bit values, and as a float) and the zero offsets of column
// `col` in group row `grp` of a stage (dequant_word_int); constants for u4b8 (z = 8).
struct ColGroup {
    uint32_t s, zlo, zhi;
    float sf;
};

// The same from shared addresses of the scale and zero elements (explicit shared loads).
template <bool BF>
__device__ __forceinline__ ColGroup col_group_sh(bool has_zp, uint32_t s_addr, uint32_t z_addr)
{
    ColGroup cgp;
    const uint16_t sb = lds16(s_addr);
    cgp.s = (uint32_t)sb * 0x10001u;
    if (BF) {
        cgp.sf = __bfloat162float(__ushort_as_bfloat16(sb));
        __nv_bfloat16 zn = __ushort_as_bfloat16((uint16_t)0xC308); // -136 = -(128 + 8)
        if (has_zp)
            zn = __hneg(__hadd(__ushort_as_bfloat16((uint16_t)0x4300), __ushort_as_bfloat16(lds16(z_addr))));
        cgp.zlo = (uint32_t)__bfloat16_as_ushort(zn) * 0x10001u;
        cgp.zhi = 0;
        return cgp;
    }
    cgp.sf = __half2float(__ushort_as_half(sb));
    if (has_zp) {
        const __half z = __ushort_as_half(lds16(z_addr));
        cgp.zlo = (uint32_t)__half_as_ushort(__hadd(__ushort_as_half(0x6400), z)) * 0x10001u;          // 1024 + z
        cgp.zhi = (uint32_t)__half_as_ushort(__hneg(__hadd(__ushort_as_half(0x5400), z))) * 0x10001u; // -(64 + z)
    } else {
        cgp.zlo = 0x64086408u; // 1032
        cgp.zhi = 0xD480D480u; // -72
    }
    return cgp;
}

template <bool BF>
__device__ __forceinline__ ColGroup col_group(bool has_zp, const __half *ssm, const __half *zsm,
                                              int idx)
{
    ColGroup cgp;
    if (BF) {
        const uint16_t sb = reinterpret_cast<const uint16_t *>(ssm)[idx];
        cgp.s = (uint32_t)sb * 0x10001u;
        cgp.sf = __bfloat162float(__ushort_as_bfloat16(sb));
        __nv_bfloat16 zn = __ushort_as_bfloat16((uint16_t)0xC308); // -136 = -(128 + 8)
        if (has_zp)
            zn = __hneg(__hadd(__ushort_as_bfloat16((uint16_t)0x4300),
                               __ushort_as_bfloat16(reinterpret_cast<const uint16_t *>(zsm)[idx])));
        cgp.zlo = (uint32_t)__bfloat16_as_ushort(zn) * 0x10001u;
        cgp.zhi = 0;
        return cgp;
    }
    const __half sh = ssm[idx];
    cgp.s = (uint32_t)__half_as_ushort(sh) * 0x10001u;
    cgp.sf = __half2float(sh);
    if (has_zp) {
        const __half z = zsm[idx];
        cgp.zlo = (uint32_t)__half_as_ushort(__hadd(__ushort_as_half(0x6400), z)) * 0x10001u;          // 1024 + z
        cgp.zhi = (uint32_t)__half_as_ushort(__hneg(__hadd(__ushort_as_half(0x5400), z))) * 0x10001u; // -(64 + z)
    } else {
        cgp.zlo = 0x64086408u; // 1032
        cgp.zhi = 0xD480D480u; // -72
    }
    return cgp;
}

// One 64-row block of a warp's 16 columns: per lane four code words (columns col0 and
// col0 + 8, rows 0..31 and 32..63), dequantised into A fragments for four k steps -- exact
// (q - z) when the scale is applied per group (SCALED false), else (q - z) s -- times the B
// fragments of every 8-token tile.  `w_addr` is the shared address of the lane's first word,
// `act0` / `act1` of its ldmatrix rows for the two 32-row halves, which accumulate into acc0 /
// acc1 (two independent MMA chains when they differ).
// HALF: bytes from a block's first 32-row half to its second (2048 in a 128-column tile, 256
// in a 16-column slice); column col + 8 is always 128 bytes on.
template <int NT, bool SCALED, int HALF = 2048, bool BF = false>
__device__ __forceinline__ void block_mma(uint32_t w_addr, uint32_t act0, uint32_t act1,
                                          const ColGroup &c0, const ColGroup &c1,
                                          float (&acc0)[NT][4], float (&acc1)[NT][4])
{
    uint32_t a0[4], a1[4], a2[4], a3[4];
    if (SCALED) {
        dequant_word_col<BF>(lds32(w_addr), c0.zlo, c0.zhi, c0.s, a0);
        dequant_word_col<BF>(lds32(w_addr + 128), c1.zlo, c1.zhi, c1.s, a1);
        dequant_word_col<BF>(lds32(w_addr + HALF), c0.zlo, c0.zhi, c0.s, a2);
        dequant_word_col<BF>(lds32(w_addr + HALF + 128), c1.zlo, c1.zhi, c1.s, a3);
    } else {
        dequant_word_int<BF>(lds32(w_addr), c0.zlo, c0.zhi, a0);
        dequant_word_int<BF>(lds32(w_addr + 128), c1.zlo, c1.zhi, a1);
        dequant_word_int<BF>(lds32(w_addr + HALF), c0.zlo, c0.zhi, a2);
        dequant_word_int<BF>(lds32(w_addr + HALF + 128), c1.zlo, c1.zhi, a3);
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        uint32_t b[4], e[4];
        ldmatrix_x4(act0 + nt * 1024, b);
        ldmatrix_x4(act1 + nt * 1024, e);
        mma_16816<BF>(acc0[nt], a0[0], a1[0], a0[1], a1[1], b[0], b[1]);
        mma_16816<BF>(acc1[nt], a2[0], a3[0], a2[1], a3[1], e[0], e[1]);
        mma_16816<BF>(acc0[nt], a0[2], a1[2], a0[3], a1[3], b[2], b[3]);
        mma_16816<BF>(acc1[nt], a2[2], a3[2], a2[3], a3[3], e[2], e[3]);
    }
}

// End of a group: acc += s (g0 + g1) per accumulator row (registers 0, 1: column col0, scale
// s0; 2, 3: column col0 + 8, scale s1), and the group accumulators restart from zero.
template <int NT>
__device__ __forceinline__ void flush_group(float (&acc)[NT][4], float (&g0)[NT][4],
                                            float (&g1)[NT][4], float s0, float s1)
{
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float sc = i < 2 ? s0 : s1;
            acc[nt][i] = fmaf(g1[nt][i], sc, fmaf(g0[nt][i], sc, acc[nt][i]));
            g0[nt][i] = 0.f;
            g1[nt][i] = 0.f;
        }
}

constexpr int DEC_UNROLL = 4; // stages of exactly this many blocks take the unrolled path

// NT: 8-token tiles per CTA tile (nt_max = 8 * NT).  BLOCK_GROUPS: group_size is a multiple
// of 64, so a group covers whole blocks and one scale serves all of a lane's codes in a
// block; otherwise each 8-row pair looks up its own group (slow, general path).
template <int NT, bool BLOCK_GROUPS, bool BF>
__device__ void run_compute(const GemmParams &p, Sched sched, uint8_t *smem, DecBars &bars,
                            const WaitCtl &ctl, int w, int lane, volatile int *last_flag)
{
    const bool has_zp = p.zeros != nullptr;
    const int gs = p.group_size;
    const int gs_kb = BLOCK_GROUPS ? gs / KBLK : 1;
    const bool gs_pow2 = (gs_kb & (gs_kb - 1)) == 0;
    // Bit b of ends64: block b (counted from a group start) is the last of its group.
    unsigned long long ends64 = 0;
    if (gs_kb <= 32)
        for (int b = gs_kb - 1; b < 64; b += gs_kb)
            ends64 |= 1ull << b;
    const int t = lane & 3;
    const int col0 = w * 16 + (lane >> 2); // this lane's weight columns: col0 and col0 + 8
    const uint32_t w_off = (uint32_t)(col0 * 4 + t) * 4u;
    // ldmatrix.x4: matrix i = lane / 8 is 16-byte chunk 4h + i of token rows 0..7 of an
    // 8-token tile, so registers (0, 1) are the B fragment of k step 2h and (2, 3) of 2h + 1.
    const uint32_t lm_off0 = (uint32_t)((lane & 7) * 128 + ((((lane >> 3)) ^ (lane & 7)) << 4));
    const uint32_t lm_off1 = (uint32_t)((lane & 7) * 128 + (((4 + (lane >> 3)) ^ (lane & 7)) << 4));
    Ring ring;
    uint32_t nsync = 0;
    auto rendezvous = [&]() -> bool {
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&bars.epi);
        const bool ok = mbar_wait(&bars.epi, nsync & 1u, ctl, W4A16_DEV_TIMEOUT);
        ++nsync;
        return ok;
    };
    SegTable no_seg{nullptr, nullptr, nullptr};
    int tile, kb0, kb1;
    while (sched.next(tile, kb0, kb1)) {
        const TileInfo ti = tile_info(p, no_seg, tile);
        // acc: the output accumulators.  With DEFER (whole-block groups, NT <= 2) the block
        // MMAs go into g0 / g1, the unscaled sums of the current group, one per 32-row half so
        // that two MMA chains run side by side; taller tiles (enough independent chains, and
        // no registers to spare for a second set) scale in the dequantisation and accumulate
        // straight into acc.
        constexpr bool DEFER = BLOCK_GROUPS && NT <= 2;
        float acc[NT][4], g0_own[NT][4], g1_own[NT][4];
        float(&g0)[NT][4] = DEFER ? g0_own : acc;
        float(&g1)[NT][4] = DEFER ? g1_own : acc;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc[nt][i] = 0.f;
                g0_own[nt][i] = 0.f;
                g1_own[nt][i] = 0.f;
            }
        float s0 = 0.f, s1 = 0.f; // the current group's scales of columns col0, col0 + 8
        int in_grp = BLOCK_GROUPS ? kb0 % gs_kb : 0; // blocks of the current group before kb
        for (int kb = kb0; kb < kb1; kb += p.kbs) {
            const int nkb = min(p.kbs, kb1 - kb);
            if (!mbar_wait(&bars.full[ring.idx], ring.phase, ctl, W4A16_DEV_TIMEOUT))
                return;
            const uint8_t *st = smem + (size_t)ring.idx * p.stage_bytes;
            const __half *ssm = reinterpret_cast<const __half *>(st + p.scales_off);
            const __half *zsm = reinterpret_cast<const __half *>(st + p.zeros_off);
            const uint32_t w_addr = smem_u32(st + p.packed_off) + w_off;
            const uint32_t act0 = smem_u32(st) + lm_off0;
            const uint32_t act1 = smem_u32(st) + lm_off1;
            if (BLOCK_GROUPS) {
                // Bit j of gend: block kb + j is the last of its group.
                uint32_t gend;
                if (gs_kb <= 32) {
                    gend = (uint32_t)(ends64 >> in_grp);
                } else {
                    const int e = gs_kb - 1 - in_grp;
                    gend = e < 32 ? 1u << e : 0u;
                }
                in_grp += nkb;
                if (in_grp >= gs_kb)
                    in_grp = gs_pow2 ? (in_grp & (gs_kb - 1)) : in_grp % gs_kb;
                int gidx = col0; // scale index of the current group (relative to the stage's)
                ColGroup c0 = col_group<BF>(has_zp, ssm, zsm, gidx);
                ColGroup c1 = col_group<BF>(has_zp, ssm, zsm, gidx + 8);
                s0 = c0.sf;
                s1 = c1.sf;
                auto next_group = [&]() {
                    gidx += TILE_N;
                    c0 = col_group<BF>(has_zp, ssm, zsm, gidx);
                    c1 = col_group<BF>(has_zp, ssm, zsm, gidx + 8);
                    s0 = c0.sf;
                    s1 = c1.sf;
                };
                if (nkb == DEC_UNROLL) {
                    // Taller tiles keep more accumulators live: unroll less there.
                    constexpr int UNROLL = NT <= 2 ? DEC_UNROLL : 2;
#pragma unroll UNROLL
                    for (int j = 0; j < DEC_UNROLL; ++j) {
                        block_mma<NT, !DEFER, 2048, BF>(w_addr + j * TILE_BYTES, act0 + j * p.act_kb_bytes,
                                                        act1 + j * p.act_kb_bytes, c0, c1, g0, g1);
                        if (gend & (1u << j)) {
                            if (DEFER)
                                flush_group<NT>(acc, g0, g1, s0, s1);
                            if (j + 1 < DEC_UNROLL)
                                next_group();
                        }
                    }
                } else {
                    for (int j = 0; j < nkb; ++j) {
                        block_mma<NT, !DEFER, 2048, BF>(w_addr + j * TILE_BYTES, act0 + j * p.act_kb_bytes,
                                                        act1 + j * p.act_kb_bytes, c0, c1, g0, g1);
                        if (gend & (1u << j)) {
                            if (DEFER)
                                flush_group<NT>(acc, g0, g1, s0, s1);
                            if (j + 1 < nkb)
                                next_group();
                        }
                    }
                }
            } else {
                const int g_first = (kb * KBLK) / gs;
                const uint32_t *pw = reinterpret_cast<const uint32_t *>(st + p.packed_off) + w_off / 4;
                for (int j = 0; j < nkb; ++j) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t a0[4], a1[4];
                        __half2 s2[4], zl[4], zh[4];
                        load_scales(p, ssm, zsm, has_zp, kb + j, h, g_first, col0, s2, zl, zh);
                        dequant_word(pw[h * 512], zl, zh, s2, a0);
                        load_scales(p, ssm, zsm, has_zp, kb + j, h, g_first, col0 + 8, s2, zl, zh);
                        dequant_word(pw[h * 512 + 32], zl, zh, s2, a1);
                        const uint32_t actj = (h ? act1 : act0) + j * p.act_kb_bytes;
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            uint32_t b[4];
                            ldmatrix_x4(actj + nt * 1024, b);
                            mma_16816<BF>(acc[nt], a0[0], a1[0], a0[1], a1[1], b[0], b[1]);
                            mma_16816<BF>(acc[nt], a0[2], a1[2], a0[3], a1[3], b[2], b[3]);
                        }
                    }
                    pw += TILE_WORDS;
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&bars.empty[ring.idx]);
            ring.advance(p.stages);
        }

        // A segment may end inside a group: add what it holds of that group.
        if (DEFER)
            flush_group<NT>(acc, g0, g1, s0, s1);

        // Segment end: fp16 C for a whole tile, else an fp32 partial and the split protocol.
        // (Nothing of the preceding kernel may still read C or this workspace.)
        pdl_wait();
        const bool whole = (kb0 == 0 && kb1 == p.kblocks);
        const long long st_tile = (long long)tile - sched.dp_tiles;
        float *part = whole ? nullptr : partial_slot(p, sched.cta, own_slot(p, sched, st_tile));
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int row = nt * 8 + 2 * t + (i & 1);
                const int col = col0 + 8 * (i >> 1);
                const float v = acc[nt][i];
                if (row >= ti.rows)
                    continue;
                if (whole)
                    reinterpret_cast<uint16_t *>(p.c)[(long long)(ti.row0 + row) * p.ldc + ti.n0 + col] =
                        to_out16(v, BF);
                else
                    __stcg(part + row * TILE_N + col, v);
            }
        if (whole)
            continue;
        if (!rendezvous())
            return;
        const Contributors cb = contributors(p, sched, st_tile);
        if (w == 0 && lane == 0) {
            const int old = split_counter_arrive(&p.counters[tile]);
            const int last = old == (cb.hi - cb.lo);
            *last_flag = last;
        }
        if (!rendezvous())
            return;
        if (!*last_flag)
            continue;
        reduce_tile<(NT <= 2 ? 2 : 1)>(p, ti, cb, w * 32 + lane, DEC_WARPS * 32); // lighter: no spills
        if (w == 0 && lane == 0)
            p.counters[tile] = 0;
    }
}

template <int NT, bool BLOCK_GROUPS, bool BF = false>
__global__ void __launch_bounds__(DEC_THREADS, DEC_CTAS_PER_SM)
    w4a16_decode_kernel(const __grid_constant__ GemmParams p, const __grid_constant__ CUtensorMap tmap_a,
                        const __grid_constant__ CUtensorMap tmap_s, const __grid_constant__ CUtensorMap tmap_z)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ DecBars bars;
    __shared__ volatile int abort_sh;
    __shared__ volatile int last_sh;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);

    int pre = 0; // stages whose weight part went out before the dependency wait (thread 0)
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&bars.full[s], 1);
            mbar_init(&bars.empty[s], DEC_WARPS);
        }
        mbar_init(&bars.epi, DEC_WARPS);
        fence_mbar_init();
        abort_sh = 0;
        last_sh = 0;
        prefetch_tensormap(&tmap_a);
        prefetch_tensormap(&tmap_s);
        if (p.zeros != nullptr)
            prefetch_tensormap(&tmap_z);
        pdl_launch_dependents();
        Sched first;
        first.init(p.m_tiles * p.n_tiles, p.kblocks, p.split);
        SegTable none{nullptr, nullptr, nullptr};
        if (p.static_weights)
            pre = issue_static_weights(p, &tmap_s, &tmap_z, none, first, smem, bars.full);
        else
            prefetch_first_codes(p, first, (uint32_t)p.stages * p.kbs * TILE_BYTES);
    }
    // No programmatic-dependency wait here: the set-up below reads nothing the preceding
    // kernel writes, so it overlaps that kernel's tail.  The producer waits before its first
    // activation copy (and, without static weights, before any copy), the compute warps
    // before their first global write.
    __syncthreads();
    WaitCtl ctl{&abort_sh, p.status, p.limit_ns};
    Sched sched;
    sched.init(p.m_tiles * p.n_tiles, p.kblocks, p.split);
    SegTable no_seg{nullptr, nullptr, nullptr};

    if (warp == 0) {
        if (lane == 0)
            run_producer(p, &tmap_a, &tmap_s, &tmap_z, no_seg, sched, smem, bars.full, bars.empty,
                         ctl, pre, true);
    } else {
        run_compute<NT, BLOCK_GROUPS, BF>(p, sched, smem, bars, ctl, warp - 1, lane, &last_sh);
    }
    __syncwarp();
    __syncthreads();
}

// ---------------------------------------------------------------------------------------
// Column-slice kernel (M <= 32, groups of whole blocks).  The kernel above splits K across
// CTAs, and the split tiles cost every call a tail of two L2 round trips (partial stores, the
// counter, the last contributor's reduction) that sits on the critical path of back-to-back
// calls.  Here a work item is one 16-column slice over all of K: a CTA takes a run of
// consecutive slices, its 8 compute warps take 4 consecutive blocks each (2 for 9..16 tokens,
// 1 for 17..32) of every stage, and the warps' fp32 sums of a slice meet in shared memory (fixed order, so
// repeated calls are bit-identical) and are written as fp16 C.  No partials, counters or
// workspace traffic.  The per-lane work is the same as block_mma above, on the slice's 16
// columns; a stage's activation box is exactly M rows, so little shared memory goes to the
// token rows an 8-token MMA tile has past M.
// ---------------------------------------------------------------------------------------
static_assert(DEC_WARPS == SLICE_WARPS, "slice reduction buffers are sized for 8 warps");

// One stage's codes and scale (and zero) rows, arming its barrier for the whole stage
// including the activation rows that follow separately.
static __device__ __forceinline__ void slice_issue_weights(const GemmParams &p,
                                                           const CUtensorMap *tmap_w,
                                                           const CUtensorMap *tmap_s,
                                                           const CUtensorMap *tmap_z, int slice,
                                                           int kb0, uint8_t *st, uint64_t *full)
{
    const bool has_zp = p.zeros != nullptr;
    const uint32_t sg_bytes = (uint32_t)p.sg_box * SLICE_N * 2;
    // A block of a slice is 2 rows of the weight view (4-bit) or 4 (FP8), 256 bytes each.
    const int rows_per_block = p.w8 ? 4 : 2;
    mbar_arrive_expect_tx(full, (uint32_t)p.kbs * (uint32_t)p.act_kb_bytes +
                                    (uint32_t)(p.kbs * rows_per_block) * 256u +
                                    sg_bytes * (has_zp ? 2u : 1u));
    constexpr int SLICES_PER_TILE = TILE_N / SLICE_N;
    const int tile = slice / SLICES_PER_TILE;
    const int x = (slice % SLICES_PER_TILE) * SLICE_N * 4; // word offset inside a view row
    const int row = (tile * p.kblocks + kb0) * rows_per_block;
    tensor_load_2d_hint(st + p.packed_off, tmap_w, x, row, full, policy_evict_first());
    const int g0 = (kb0 * KBLK) / p.group_size;
    tensor_load_2d(st + p.scales_off, tmap_s, slice * SLICE_N, g0, full);
    if (has_zp)
        tensor_load_2d(st + p.zeros_off, tmap_z, slice * SLICE_N, g0, full);
}

static __device__ void slice_producer(const GemmParams &p, const CUtensorMap *tmap_a,
                                      const CUtensorMap *tmap_w, const CUtensorMap *tmap_s,
                                      const CUtensorMap *tmap_z, int s_begin, int s_end, int n_st,
                                      uint8_t *smem, DecBars &bars, const WaitCtl &ctl, int pre)
{
    if (!p.static_weights)
        pdl_wait();
    Ring ring;
    int issued = 0;
    bool ok = true;
    for (int sl = s_begin; ok && sl < s_end; ++sl) {
        for (int st = 0; st < n_st; ++st) {
            uint64_t *full = &bars.full[ring.idx];
            uint8_t *stp = smem + (size_t)ring.idx * p.stage_bytes;
            if (issued >= pre) {
                if (!mbar_wait(&bars.empty[ring.idx], ring.phase ^ 1u, ctl, W4A16_DEV_TIMEOUT)) {
                    ok = false;
                    break;
                }
                slice_issue_weights(p, tmap_w, tmap_s, tmap_z, sl, st * p.kbs, stp, full);
            }
            if (issued == 0 && p.static_weights)
                pdl_wait();
            // The M rows of A for the stage's blocks; blocks past K read zeros.
            tensor_load_3d_hint(stp, tmap_a, 0, 0, st * p.kbs, full, policy_evict_last());
            ring.advance(p.stages);
            ++issued;
        }
    }
    // Leave no copy in flight: wait (bounded, ignoring the abort flag) for the last stages.
    WaitCtl drain_ctl = ctl;
    volatile int no_abort = 0;
    drain_ctl.abort_flag = &no_abort;
    const int n = issued < p.stages ? issued : p.stages;
    for (int i = 0; i < n; ++i) {
        int idx = ring.idx - 1 - i;
        uint32_t ph = ring.phase;
        if (idx < 0) {
            idx += p.stages;
            ph ^= 1u;
        }
        mbar_wait(&bars.full[idx], ph, drain_ctl, W4A16_DEV_TIMEOUT);
    }
}

// One 64-row block of the lane's two slice columns (c and c + 8) against NT 8-token tiles:
// `w_addr` is the lane's first code word, act0[nt] / act1[nt] its ldmatrix row addresses for
// the block's two 32-row halves.
template <int NT, bool BF>
__device__ __forceinline__ void slice_block_mma(uint32_t w_addr, const uint32_t (&act0)[NT],
                                                const uint32_t (&act1)[NT], const ColGroup &c0,
                                                const ColGroup &c1, float (&acc0)[NT][4],
                                                float (&acc1)[NT][4])
{
    constexpr uint32_t HALF = SLICE_N * 4 * 4; // 256 bytes: one 32-row half of the slice
    uint32_t a0[4], a1[4], a2[4], a3[4];
    dequant_word_col<BF>(lds32(w_addr), c0.zlo, c0.zhi, c0.s, a0);
    dequant_word_col<BF>(lds32(w_addr + 128), c1.zlo, c1.zhi, c1.s, a1);
    dequant_word_col<BF>(lds32(w_addr + HALF), c0.zlo, c0.zhi, c0.s, a2);
    dequant_word_col<BF>(lds32(w_addr + HALF + 128), c1.zlo, c1.zhi, c1.s, a3);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        uint32_t b[4], e[4];
        ldmatrix_x4(act0[nt], b);
        ldmatrix_x4(act1[nt], e);
        mma_16816<BF>(acc0[nt], a0[0], a1[0], a0[1], a1[1], b[0], b[1]);
        mma_16816<BF>(acc1[nt], a2[0], a3[0], a2[1], a3[1], e[0], e[1]);
        mma_16816<BF>(acc0[nt], a0[2], a1[2], a0[3], a1[3], b[2], b[3]);
        mma_16816<BF>(acc1[nt], a2[2], a3[2], a2[3], a3[3], e[2], e[3]);
    }
}

// The same block with the scale applied in fp32 per block: the MMAs take the exact (q - z)
// (fp16: 9 instructions per 8 codes instead of 13; bf16: 12 instead of 16), start from zero,
// and the block's sums are multiplied by the column's s into the output accumulators --
// (q - z) s is never rounded to 16 bits (for a one-hot row of A the result is the exact
// product, rounded once on output).
template <int NT, bool BF>
__device__ __forceinline__ void slice_block_mma_bs(uint32_t w_addr, const uint32_t (&act0)[NT],
                                                   const uint32_t (&act1)[NT], const ColGroup &c0,
                                                   const ColGroup &c1, float (&acc0)[NT][4],
                                                   float (&acc1)[NT][4])
{
    constexpr uint32_t HALF = SLICE_N * 4 * 4;
    uint32_t a0[4], a1[4], a2[4], a3[4];
    dequant_word_int<BF>(lds32(w_addr), c0.zlo, c0.zhi, a0);
    dequant_word_int<BF>(lds32(w_addr + 128), c1.zlo, c1.zhi, a1);
    dequant_word_int<BF>(lds32(w_addr + HALF), c0.zlo, c0.zhi, a2);
    dequant_word_int<BF>(lds32(w_addr + HALF + 128), c1.zlo, c1.zhi, a3);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        uint32_t b[4], e[4];
        ldmatrix_x4(act0[nt], b);
        ldmatrix_x4(act1[nt], e);
        float d0[4], d1[4];
        mma_16816_z<BF>(d0, a0[0], a1[0], a0[1], a1[1], b[0], b[1]);
        mma_16816_z<BF>(d1, a2[0], a3[0], a2[1], a3[1], e[0], e[1]);
        mma_16816<BF>(d0, a0[2], a1[2], a0[3], a1[3], b[2], b[3]);
        mma_16816<BF>(d1, a2[2], a3[2], a2[3], a3[3], e[2], e[3]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float sc = i < 2 ? c0.sf : c1.sf;
            acc0[nt][i] = fmaf(d0[i], sc, acc0[nt][i]);
            acc1[nt][i] = fmaf(d1[i], sc, acc1[nt][i]);
        }
    }
}

// FP8 E4M3 codes: one 64-row block of the lane's two slice columns.  In shared memory the block
// is four 256-byte rows, one per 16-row quarter q (= k step), each holding the slice's 16
// columns x 4 words of four K-consecutive codes.  For k step q the lane's A fragment needs rows
// 2t, 2t+1 and 2t+8, 2t+9 of columns c and c+8: the 16-bit halves at `w_addr` + q*256 (+ 8 for
// the rows 8 on, + 128 for column c + 8), each converting exactly to an fp16 pair; the product
// with the column's scale is rounded once.
template <int NT>
__device__ __forceinline__ void slice_block_mma_fp8(uint32_t w_addr, const uint32_t (&act0)[NT],
                                                    const uint32_t (&act1)[NT], uint32_t s0,
                                                    uint32_t s1, float (&acc0)[NT][4],
                                                    float (&acc1)[NT][4])
{
    uint32_t a[4][4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint32_t base = w_addr + q * 256;
        const uint16_t h[4] = {lds16(base), lds16(base + 128), lds16(base + 8), lds16(base + 136)};
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const __half2_raw v = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)h[r], __NV_E4M3);
            a[q][r] = h2_as_u32(__hmul2(__half2(v), u32_as_h2((r & 1) ? s1 : s0)));
        }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        uint32_t b[4], e[4];
        ldmatrix_x4(act0[nt], b);
        ldmatrix_x4(act1[nt], e);
        mma_16816<false>(acc0[nt], a[0][0], a[0][1], a[0][2], a[0][3], b[0], b[1]);
        mma_16816<false>(acc0[nt], a[1][0], a[1][1], a[1][2], a[1][3], b[2], b[3]);
        mma_16816<false>(acc1[nt], a[2][0], a[2][1], a[2][2], a[2][3], e[0], e[1]);
        mma_16816<false>(acc1[nt], a[3][0], a[3][1], a[3][2], a[3][3], e[2], e[3]);
    }
}

// FP8 with the scale applied in fp32 per block: each code converts exactly to fp16, the MMAs
// start from zero, and the block's sums times the column's s go into the output accumulators.
template <int NT>
__device__ __forceinline__ void slice_block_mma_fp8_bs(uint32_t w_addr, const uint32_t (&act0)[NT],
                                                       const uint32_t (&act1)[NT], float s0, float s1,
                                                       float (&acc0)[NT][4], float (&acc1)[NT][4])
{
    uint32_t a[4][4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint32_t base = w_addr + q * 256;
        const uint16_t h[4] = {lds16(base), lds16(base + 128), lds16(base + 8), lds16(base + 136)};
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const __half2_raw v = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)h[r], __NV_E4M3);
            a[q][r] = h2_as_u32(__half2(v));
        }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        uint32_t b[4], e[4];
        ldmatrix_x4(act0[nt], b);
        ldmatrix_x4(act1[nt], e);
        float d0[4], d1[4];
        mma_16816_z<false>(d0, a[0][0], a[0][1], a[0][2], a[0][3], b[0], b[1]);
        mma_16816_z<false>(d1, a[2][0], a[2][1], a[2][2], a[2][3], e[0], e[1]);
        mma_16816<false>(d0, a[1][0], a[1][1], a[1][2], a[1][3], b[2], b[3]);
        mma_16816<false>(d1, a[3][0], a[3][1], a[3][2], a[3][3], e[2], e[3]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float sc = i < 2 ? s0 : s1;
            acc0[nt][i] = fmaf(d0[i], sc, acc0[nt][i]);
            acc1[nt][i] = fmaf(d1[i], sc, acc1[nt][i]);
        }
    }
}

// Compute warp w of the column-slice kernel: blocks w*BPW .. w*BPW + BPW - 1 of every stage.
// A stage's activations are kbs blocks x M rows of 128 bytes in the 128-byte swizzle (16-byte
// chunk c of row j at j*128 + ((c ^ (j & 7)) << 4) from the 1024-aligned stage start); the
// lanes of a token row at or past M point ldmatrix at the zero row instead.
template <int NT, bool BF, bool W8>
__device__ __forceinline__ void slice_compute(const GemmParams &p, uint8_t *smem, DecBars &bars,
                              const WaitCtl &ctl, int w, int lane, int s_begin, int s_end,
                              int n_st)
{
    constexpr int BPW = slice_bpw(8 * NT, W8);
    constexpr int KBS = SLICE_WARPS * BPW;
    const bool has_zp = p.zeros != nullptr;
    const int t = lane & 3;
    const int c = lane >> 2; // this lane's slice columns: c and c + 8
    // 4-bit: word t of column c, half 0, of block bl (row 2*bl of 16 columns x 4 words).
    // FP8: the 16-bit half (t & 1) of word t >> 1 of column c, quarter 0 (row 4*bl).
    const uint32_t w_lane = W8 ? (uint32_t)(c * 16 + (t >> 1) * 4 + (t & 1) * 2)
                               : (uint32_t)((c * 4 + t) * 4);
    constexpr uint32_t BLOCK_STRIDE = W8 ? 1024u : 2u * SLICE_N * 4 * 4;
    constexpr int VALS = NT * 4 * 32; // one warp's accumulators
    float *red = reinterpret_cast<float *>(smem + p.epi_smem_off);
    const uint32_t zero_row = smem_u32(smem + p.epi_smem_off + 2 * SLICE_WARPS * VALS * 4);
    const int m = p.m;
    // ldmatrix row offsets (from the stage start) of this lane for block j of the warp's run,
    // token tile nt and the block's two 32-row halves; valid bit (j, nt) clear: token row >= M.
    uint32_t act_off0[BPW][NT], act_off1[BPW][NT];
    uint32_t valid = 0;
#pragma unroll
    for (int j = 0; j < BPW; ++j)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int tok = nt * 8 + (lane & 7);
            const int row = (w * BPW + j) * m + tok;
            const uint32_t ch = (uint32_t)(lane >> 3);
            const uint32_t sw = (uint32_t)(row & 7);
            act_off0[j][nt] = (uint32_t)row * 128u + ((ch ^ sw) << 4);
            act_off1[j][nt] = (uint32_t)row * 128u + (((4u + ch) ^ sw) << 4);
            if (tok < m)
                valid |= 1u << (j * NT + nt);
        }
    // Group of block kb relative to the stage's first group: a shift when the blocks per group
    // are a power of two.
    const int gs_kb = p.group_size / KBLK;
    const int gsh = group_shift(gs_kb);
    Ring ring;
    uint32_t nsync = 0;
    bool dep_done = false;
    for (int sl = s_begin; sl < s_end; ++sl) {
        float acc0[NT][4], acc1[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc0[nt][i] = 0.f;
                acc1[nt][i] = 0.f;
            }
        for (int st = 0; st < n_st; ++st) {
            if (!mbar_wait(&bars.full[ring.idx], ring.phase, ctl, W4A16_DEV_TIMEOUT))
                return;
            const uint8_t *stp = smem + (size_t)ring.idx * p.stage_bytes;
            const uint32_t act_base = smem_u32(stp);
            const uint32_t w_base = smem_u32(stp + p.packed_off) + w_lane;
            const uint32_t s_sh = act_base + (uint32_t)p.scales_off;
            const uint32_t z_sh = act_base + (uint32_t)p.zeros_off;
            const int kb0 = st * KBS;
            // Group of each of the warp's blocks relative to the stage's first group (the
            // stage's scale rows start there), stepped along the blocks: no division per block.
            int gj[BPW];
            {
                const int kbw = kb0 + w * BPW;
                const int gw = gsh >= 0 ? kbw >> gsh : kbw / gs_kb;
                const int g_stage = gsh >= 0 ? kb0 >> gsh : kb0 / gs_kb;
                int g = gw - g_stage, r = kbw - gw * gs_kb;
#pragma unroll
                for (int j = 0; j < BPW; ++j) {
                    gj[j] = g;
                    if (++r == gs_kb) {
                        r = 0;
                        ++g;
                    }
                }
            }
            // ZP: the zero-point branch resolved at compile time, outside the unrolled blocks.
            auto block = [&](int j, auto zp_c) {
                constexpr bool ZP = decltype(zp_c)::value;
                const int bl = w * BPW + j;
                const uint32_t so = (uint32_t)(gj[j] * SLICE_N + c) * 2u;
                const ColGroup c0 = col_group_sh<BF>(ZP, s_sh + so, z_sh + so);
                const ColGroup c1 = col_group_sh<BF>(ZP, s_sh + so + 16, z_sh + so + 16);
                uint32_t act0[NT], act1[NT];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const bool ok = (valid >> (j * NT + nt)) & 1u;
                    act0[nt] = ok ? act_base + act_off0[j][nt] : zero_row;
                    act1[nt] = ok ? act_base + act_off1[j][nt] : zero_row;
                }
                if (W8 && NT <= 2)
                    slice_block_mma_fp8_bs<NT>(w_base + (uint32_t)bl * BLOCK_STRIDE, act0, act1,
                                               c0.sf, c1.sf, acc0, acc1);
                else if (W8)
                    slice_block_mma_fp8<NT>(w_base + (uint32_t)bl * BLOCK_STRIDE, act0, act1, c0.s,
                                            c1.s, acc0, acc1);
                else if (NT <= 2)
                    slice_block_mma_bs<NT, BF>(w_base + (uint32_t)bl * BLOCK_STRIDE, act0, act1, c0,
                                               c1, acc0, acc1);
                else
                    slice_block_mma<NT, BF>(w_base + (uint32_t)bl * BLOCK_STRIDE, act0, act1, c0,
                                            c1, acc0, acc1);
            };
            auto blocks = [&](auto zp_c) {
                if (kb0 + KBS <= p.kblocks) {
                    // A full stage: no per-block bound in the unrolled loop.
#pragma unroll
                    for (int j = 0; j < BPW; ++j)
                        block(j, zp_c);
                } else {
                    // The last, partial stage of a slice: blocks past K are skipped (their
                    // scale rows were never loaded).
#pragma unroll
                    for (int j = 0; j < BPW; ++j)
                        if (kb0 + w * BPW + j < p.kblocks)
                            block(j, zp_c);
                }
            };
            if (!W8 && has_zp)
                blocks(std::true_type{});
            else
                blocks(std::false_type{});
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&bars.empty[ring.idx]);
            ring.advance(p.stages);
        }
        // The warp's sums into this slice's buffer (two buffers alternate: a warp can be one
        // slice ahead of the slowest reader, never two, since the rendezvous below needs all).
        float *buf = red + ((sl - s_begin) & 1) * (SLICE_WARPS * VALS);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i)
                buf[(w * NT * 4 + nt * 4 + i) * 32 + lane] = acc0[nt][i] + acc1[nt][i];
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&bars.epi);
        if (!mbar_wait(&bars.epi, nsync & 1u, ctl, W4A16_DEV_TIMEOUT))
            return;
        ++nsync;
        if (!dep_done) {
            pdl_wait(); // nothing of the preceding kernel may still read C
            dep_done = true;
        }
        // Thread `id` sums values (register reg, lane ln) over the 8 warps in a fixed order;
        // with four token tiles (512 values) each of the 256 threads takes two.
        for (int id = w * 32 + lane; id < VALS; id += SLICE_WARPS * 32) {
            const int reg = id >> 5, ln = id & 31;
            float v = 0.f;
#pragma unroll
            for (int q = 0; q < SLICE_WARPS; ++q)
                v += buf[(q * NT * 4 + reg) * 32 + ln];
            const int nt = reg >> 2, i = reg & 3;
            const int row = nt * 8 + 2 * (ln & 3) + (i & 1);
            const int col = sl * SLICE_N + (ln >> 2) + 8 * (i >> 1);
            if (row < m)
                reinterpret_cast<uint16_t *>(p.c)[(long long)row * p.ldc + col] = to_out16(v, BF);
        }
    }
}

template <int NT, bool BF = false, bool W8 = false>
__global__ void __launch_bounds__(DEC_THREADS, DEC_CTAS_PER_SM)
    w4a16_slice_kernel(const __grid_constant__ GemmParams p, const __grid_constant__ CUtensorMap tmap_a,
                       const __grid_constant__ CUtensorMap tmap_w,
                       const __grid_constant__ CUtensorMap tmap_s,
                       const __grid_constant__ CUtensorMap tmap_z)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ DecBars bars;
    __shared__ volatile int abort_sh;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const int s_begin = blockIdx.x * p.slice_per;
    const int s_end = min(s_begin + p.slice_per, p.n_slices);
    const int n_st = (p.kblocks + p.kbs - 1) / p.kbs; // stages per slice

    int pre = 0; // stages whose weight part went out before the dependency wait (thread 0)
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&bars.full[s], 1);
            mbar_init(&bars.empty[s], DEC_WARPS);
        }
        mbar_init(&bars.epi, DEC_WARPS);
        fence_mbar_init();
        abort_sh = 0;
        prefetch_tensormap(&tmap_a);
        prefetch_tensormap(&tmap_w);
        prefetch_tensormap(&tmap_s);
        if (p.zeros != nullptr)
            prefetch_tensormap(&tmap_z);
        pdl_launch_dependents();
        if (p.static_weights) {
            const int total = (s_end - s_begin) * n_st;
            for (; pre < p.stages && pre < total; ++pre)
                slice_issue_weights(p, &tmap_w, &tmap_s, &tmap_z, s_begin + pre / n_st,
                                    (pre % n_st) * p.kbs, smem + (size_t)pre * p.stage_bytes,
                                    &bars.full[pre]);
        }
    }
    // The zero row that ldmatrix reads for token rows past M.
    if (warp == 1)
        reinterpret_cast<uint32_t *>(smem + p.epi_smem_off + 2 * SLICE_WARPS * NT * 4 * 32 * 4)[lane] = 0u;
    // As in the kernel above: no dependency wait before the set-up; the producer waits before
    // its first activation copy (without static weights, before any copy), the compute warps
    // before their first write of C.
    __syncthreads();
    WaitCtl ctl{&abort_sh, p.status, p.limit_ns};
    if (warp == 0) {
        if (lane == 0)
            slice_producer(p, &tmap_a, &tmap_w, &tmap_s, &tmap_z, s_begin, s_end, n_st, smem, bars,
                           ctl, pre);
    } else {
        slice_compute<NT, BF, W8>(p, smem, bars, ctl, warp - 1, lane, s_begin, s_end, n_st);
    }
    __syncwarp();
    __syncthreads();
}

int decode_max_rows()
{
    return 64;
}

// Alignment slack only (the stages are all the dynamic shared memory).
int decode_extra_smem(int nt_max)
{
    (void)nt_max;
    return 1024;
}

// CTAs of the small-M kernel per SM, and the dynamic shared memory each may use so that they
// all fit: the SM's shared memory split evenly, less each CTA's reserved and static part.
int decode_ctas_per_sm()
{
    return DEC_CTAS_PER_SM;
}

int decode_smem_limit(int *bytes)
{
    int dev = 0, per_sm = 0, reserved = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err == cudaSuccess)
        err = cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    if (err == cudaSuccess)
        err = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
    cudaFuncAttributes fa, fs;
    if (err == cudaSuccess)
        err = cudaFuncGetAttributes(&fa, w4a16_decode_kernel<1, true>);
    if (err == cudaSuccess)
        err = cudaFuncGetAttributes(&fs, w4a16_slice_kernel<1>);
    if (err != cudaSuccess)
        return err;
    const int stat = (int)(fa.sharedSizeBytes > fs.sharedSizeBytes ? fa.sharedSizeBytes
                                                                     : fs.sharedSizeBytes);
    *bytes = per_sm / DEC_CTAS_PER_SM - reserved - stat - 256;
    return cudaSuccess;
}

int launch_decode(const GemmParams &p, const CUtensorMap &tmap_a, const CUtensorMap &tmap_s,
                  const CUtensorMap &tmap_z, const GemmConfig &cfg, cudaStream_t stream)
{
    static int attr_done[12][64];
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    int v;
    switch (p.nt_max) {
    case 8: v = 0; break;
    case 16: v = 1; break;
    case 32: v = 2; break;
    case 64: v = 3; break;
    default: return cudaErrorInvalidValue;
    }
    // bf16 operands: whole-block groups only (the host sends smaller groups to the tcgen05
    // kernel).
    if (p.bf16 && p.group_size % KBLK != 0)
        return cudaErrorInvalidValue;
    void (*kernels[12])(GemmParams, CUtensorMap, CUtensorMap, CUtensorMap) = {
        w4a16_decode_kernel<1, true>,  w4a16_decode_kernel<2, true>,  w4a16_decode_kernel<4, true>,
        w4a16_decode_kernel<8, true>,  w4a16_decode_kernel<1, false>, w4a16_decode_kernel<2, false>,
        w4a16_decode_kernel<4, false>, w4a16_decode_kernel<8, false>,
        w4a16_decode_kernel<1, true, true>, w4a16_decode_kernel<2, true, true>,
        w4a16_decode_kernel<4, true, true>, w4a16_decode_kernel<8, true, true>};
    const int variant = p.bf16 ? 8 + v : v + (p.group_size % KBLK == 0 ? 0 : 4);
    auto kernel = kernels[variant];
    if (dev < 64 && attr_done[variant][dev] < cfg.smem_bytes) {
        err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   cfg.smem_bytes);
        if (err != cudaSuccess)
            return err;
        attr_done[variant][dev] = cfg.smem_bytes;
    }
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(cfg.grid);
    lc.blockDim = dim3(DEC_THREADS);
    lc.dynamicSmemBytes = cfg.smem_bytes;
    lc.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    return cudaLaunchKernelEx(&lc, kernel, p, tmap_a, tmap_s, tmap_z);
}

int launch_slice(const GemmParams &p, const CUtensorMap &tmap_a, const CUtensorMap &tmap_w,
                 const CUtensorMap &tmap_s, const CUtensorMap &tmap_z, const GemmConfig &cfg,
                 cudaStream_t stream)
{
    static int attr_done[9][64];
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    int v;
    switch (p.nt_max) {
    case 8: v = 0; break;
    case 16: v = 1; break;
    case 32: v = 2; break;
    default: return cudaErrorInvalidValue;
    }
    if (p.bf16)
        v += 3;
    else if (p.w8)
        v += 6;
    void (*kernels[9])(GemmParams, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap) = {
        w4a16_slice_kernel<1>,       w4a16_slice_kernel<2>,       w4a16_slice_kernel<4>,
        w4a16_slice_kernel<1, true>, w4a16_slice_kernel<2, true>, w4a16_slice_kernel<4, true>,
        w4a16_slice_kernel<1, false, true>, w4a16_slice_kernel<2, false, true>,
        w4a16_slice_kernel<4, false, true>};
    auto kernel = kernels[v];
    if (dev < 64 && attr_done[v][dev] < cfg.smem_bytes) {
        err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   cfg.smem_bytes);
        if (err != cudaSuccess)
            return err;
        attr_done[v][dev] = cfg.smem_bytes;
    }
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(cfg.grid);
    lc.blockDim = dim3(DEC_THREADS);
    lc.dynamicSmemBytes = cfg.smem_bytes;
    lc.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    return cudaLaunchKernelEx(&lc, kernel, p, tmap_a, tmap_w, tmap_s, tmap_z);
}

} // namespace w4
