// w4a16_decode.cu -- the small-M W4A16 GEMM: weights dequantised in registers straight into
// warp-level mma.sync (m16n8k16), for decode-sized M (up to 64 rows).
//
// Why a second kernel: at small M the job is to stream the packed weights at HBM speed.  The
// tcgen05 kernel stages every dequantised weight in tensor (or shared) memory and reads it
// back as an MMA operand, and a 128x16x16 tcgen05.mma costs about as much as a 128x64x16 one;
// both cap the weight rate well below the HBM rate.  Here each thread converts the 8 codes of
// one tile word -- which the tile layout makes exactly its m16n8k16 B fragment for two 16-row
// steps -- and feeds the fp16 registers to mma.sync directly; the activations (A, m16 x k16 per
// step) come from shared memory through ldmatrix.  Only the 4-bit codes, scales and
// activations move on chip.
//
// CTA: one TMA producer warp (the producer of w4a16_common.cuh) and 16 compute warps, warp g
// owning the 8 weight columns 8g..8g+7 of the 128-column tile.  Work is split over CTAs with
// the same data-parallel + stream-K schedule; split tiles are reduced in a fixed order by the
// last contributor.
#include "w4a16_common.cuh"

namespace w4 {

constexpr int DEC_WARPS = 16;                 // compute warps (one 8-column group each)
constexpr int DEC_THREADS = (DEC_WARPS + 1) * 32;

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

__device__ __forceinline__ void ldmatrix_x2(uint32_t addr, uint32_t &r0, uint32_t &r1)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
                 : "=r"(r0), "=r"(r1)
                 : "r"(addr));
}

// D (f32 16x8) += A (f16 16x16, row) * B (f16 16x8, col)
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
                 "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// MT m16 row tiles; HALF: at most 8 rows, held as 8-row activation tiles (the MMA's rows
// 8..15 are zero registers).
template <int MT, bool HALF>
__device__ void run_compute(const GemmParams &p, Sched sched, uint8_t *smem, DecBars &bars,
                            const WaitCtl &ctl, int g, int lane, volatile int *last_flag)
{
    const bool has_zp = p.zeros != nullptr;
    const int gs = p.group_size;
    const int gs_kb = (gs % KBLK == 0) ? gs / KBLK : 0;
    const int col_in_tile = 8 * g + (lane >> 2);   // B / scale column of this thread
    // ldmatrix: matrix i = lane / 8 covers rows 8*(i&1).. and 16-byte chunk (i>>1) of a step
    // (x4); for the 8-row tiles, matrix i = lane / 8 (0, 1) is chunk i of rows 0..7 (x2).
    const int lm_row = HALF ? (lane & 7) : (lane & 7) + 8 * ((lane >> 3) & 1);
    const int lm_chunk = HALF ? ((lane >> 3) & 1) : (lane >> 4);
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
        float acc[MT][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int i = 0; i < 4; ++i)
                acc[mt][i] = 0.f;
        for (int kb = kb0; kb < kb1; kb += p.kbs) {
            const int nkb = min(p.kbs, kb1 - kb);
            if (!mbar_wait(&bars.full[ring.idx], ring.phase, ctl, W4A16_DEV_TIMEOUT))
                return;
            const uint8_t *st = smem + (size_t)ring.idx * p.stage_bytes;
            const __half *ssm = reinterpret_cast<const __half *>(st + p.scales_off);
            const __half *zsm = reinterpret_cast<const __half *>(st + p.zeros_off);
            const int g_first = (kb * KBLK) / gs;
            for (int j = 0; j < nkb; ++j) {
                const int kbj = kb + j;
                const uint32_t act = smem_u32(st + j * p.act_kb_bytes);
                const uint32_t *packed =
                    reinterpret_cast<const uint32_t *>(st + p.packed_off + j * TILE_BYTES);
                const uint32_t w0 = packed[32 * g + lane];
                const uint32_t w1 = packed[512 + 32 * g + lane];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    __half2 s2[4], zlo[4], zhi[4];
                    load_scales(p, ssm, zsm, has_zp, kbj, h, g_first, gs_kb, col_in_tile, s2, zlo,
                                zhi);
                    uint32_t b[4];
                    dequant_word(h ? w1 : w0, zlo, zhi, s2, b);
#pragma unroll
                    for (int step = 0; step < 2; ++step) {
                        const int chunk = (h * 2 + step) * 2 + lm_chunk;
#pragma unroll
                        for (int mt = 0; mt < MT; ++mt) {
                            const int r = mt * 16 + lm_row;
                            const uint32_t addr = act + r * 128 + ((chunk ^ (r & 7)) << 4);
                            uint32_t a[4];
                            if (HALF) {
                                ldmatrix_x2(addr, a[0], a[2]);
                                a[1] = 0u;
                                a[3] = 0u;
                            } else {
                                ldmatrix_x4(addr, a);
                            }
                            mma_16816(acc[mt], a, b[2 * step], b[2 * step + 1]);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&bars.empty[ring.idx]);
            ring.advance(p.stages);
        }

        // Segment end: fp16 C for a whole tile, else an fp32 partial and the split protocol.
        const bool whole = (kb0 == 0 && kb1 == p.kblocks);
        const long long st_tile = (long long)tile - sched.dp_tiles;
        const int col = ti.n0 + 8 * g + 2 * (lane & 3);
        float *part = whole ? nullptr : partial_slot(p, sched.cta, own_slot(p, sched, st_tile));
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int row = mt * 16 + (lane >> 2) + 8 * hr;
                if (row >= ti.rows)
                    continue;
                if (whole) {
                    const int out_row = output_row(p, ti, row);
                    if (out_row >= 0)
                        *reinterpret_cast<__half2 *>(p.c + (long long)out_row * p.ldc + col) =
                            __floats2half2_rn(acc[mt][2 * hr], acc[mt][2 * hr + 1]);
                } else {
                    __stcg(reinterpret_cast<float2 *>(part + row * TILE_N + (col - ti.n0)),
                           make_float2(acc[mt][2 * hr], acc[mt][2 * hr + 1]));
                }
            }
        if (whole)
            continue;
        if (!rendezvous())
            return;
        const Contributors cb = contributors(p, sched, st_tile);
        if (g == 0 && lane == 0) {
            __threadfence();
            const int old = atomicAdd(&p.counters[tile], 1);
            const int last = old == (cb.hi - cb.lo);
            if (last)
                __threadfence();
            *last_flag = last;
        }
        if (!rendezvous())
            return;
        if (!*last_flag)
            continue;
        reduce_tile(p, ti, cb, g * 32 + lane, DEC_WARPS * 32);
        if (g == 0 && lane == 0)
            p.counters[tile] = 0;
    }
}

template <int MT, bool HALF>
__global__ void __launch_bounds__(DEC_THREADS, 1)
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
    }
    pdl_wait();
    __syncthreads();
    WaitCtl ctl{&abort_sh, p.status, p.limit_ns};
    Sched sched;
    sched.init(p.m_tiles * p.n_tiles, p.kblocks);
    SegTable no_seg{nullptr, nullptr, nullptr};

    if (warp == 0) {
        if (lane == 0)
            run_producer(p, &tmap_a, &tmap_s, &tmap_z, no_seg, sched, smem, bars.full, bars.empty,
                         ctl);
    } else {
        run_compute<MT, HALF>(p, sched, smem, bars, ctl, warp - 1, lane, &last_sh);
    }
    __syncwarp();
    __syncthreads();
}

int decode_max_rows()
{
    return 64;
}

int decode_extra_smem()
{
    return 1024; // alignment slack
}

int launch_decode(const GemmParams &p, const CUtensorMap &tmap_a, const CUtensorMap &tmap_s,
                  const CUtensorMap &tmap_z, const GemmConfig &cfg, cudaStream_t stream)
{
    static int attr_done[5][64];
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    // variant 0: 8-row tiles; 1..4: MT m16 tiles
    const int variant = p.nt_max == 8 ? 0 : p.nt_max / 16;
    if (variant < 0 || variant > 4 || (variant > 0 && p.nt_max % 16 != 0))
        return cudaErrorInvalidValue;
    void (*kernels[5])(GemmParams, CUtensorMap, CUtensorMap, CUtensorMap) = {
        w4a16_decode_kernel<1, true>, w4a16_decode_kernel<1, false>, w4a16_decode_kernel<2, false>,
        w4a16_decode_kernel<3, false>, w4a16_decode_kernel<4, false>};
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

} // namespace w4
