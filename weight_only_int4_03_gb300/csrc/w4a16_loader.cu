// w4a16_loader.cu -- checkpoint-loading helpers around the GEMM: AutoGPTQ packed zero points
// into the fp16 zero points the GEMM takes, detection of symmetric checkpoints whose zero
// words are all code 7, and a device check that fp16 zero points are what the kernels assume.
//
// The two qzeros helpers run on the host: a loader holds the checkpoint's qzeros words in
// host memory when it converts them (ferrum-kernels 0.8.4 vllm_marlin.rs,
// `load_stacked_gptq_vllm_marlin`, converts them on the host before upload).
#include <stdint.h>

#include "w4a16.h"
#include "w4a16_internal.h"

namespace {

// fp16 bit pattern of an integer v in [0, 2048] (exact: at most 11 significant bits).
uint16_t half_bits_of_int(uint32_t v)
{
    if (v == 0)
        return 0;
    int e = 31 - __builtin_clz(v); // floor(log2 v)
    const uint32_t frac = (v << (10 - e)) & 0x3FFu;
    return (uint16_t)(((uint32_t)(e + 15) << 10) | frac);
}

// One thread per zero point: anything but an integer in [0, 15] (NaN included) is reported.
__global__ void zero_points_check_kernel(const __half *zeros, long long count, int *status)
{
    bool bad = false;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < count;
         i += (long long)gridDim.x * blockDim.x) {
        const float z = __half2float(zeros[i]);
        bad |= !(z >= 0.f && z <= 15.f && z == truncf(z));
    }
    if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0)
        atomicOr(status, W4A16_DEV_ZERO);
}

} // namespace

extern "C" {

int w4_qzeros_to_zero_points(const int32_t *qzeros, int groups, int n, uint16_t *zeros)
{
    if (groups <= 0 || n <= 0 || n % 8 != 0)
        return (1 << 16) | W4A16_ARG_SHAPE;
    if (!qzeros || !zeros)
        return (1 << 16) | W4A16_ARG_NULL;
    // Check every code first, so that a rejected input leaves `zeros` untouched.
    const long long words = (long long)groups * (n / 8);
    for (long long w = 0; w < words; ++w)
        for (int lane = 0; lane < 8; ++lane)
            if ((((uint32_t)qzeros[w] >> (4 * lane)) & 0xFu) == 0xFu)
                return (1 << 16) | W4A16_ARG_QZERO;
    for (long long w = 0; w < words; ++w) {
        const long long g = w / (n / 8), col0 = (w % (n / 8)) * 8;
        for (int lane = 0; lane < 8; ++lane) {
            const uint32_t stored = ((uint32_t)qzeros[w] >> (4 * lane)) & 0xFu;
            zeros[g * n + col0 + lane] = half_bits_of_int(stored + 1);
        }
    }
    return 0;
}

int w4_qzeros_symmetric_code7(const int32_t *qzeros, long long count)
{
    if (!qzeros || count <= 0)
        return 0;
    for (long long i = 0; i < count; ++i)
        if ((uint32_t)qzeros[i] != 0x77777777u)
            return 0;
    return 1;
}

int w4a16_zero_points_check(const void *zeros, long long count, int32_t *status,
                            cudaStream_t stream)
{
    if (count < 0)
        return (1 << 16) | W4A16_ARG_SHAPE;
    if (count == 0)
        return 0;
    if (!zeros || !status)
        return (1 << 16) | W4A16_ARG_NULL;
    if ((reinterpret_cast<uintptr_t>(zeros) & 1u) || (reinterpret_cast<uintptr_t>(status) & 3u))
        return (1 << 16) | W4A16_ARG_ALIGN;
    long long blocks = (count + 255) / 256;
    if (blocks > 4096)
        blocks = 4096;
    zero_points_check_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
        static_cast<const __half *>(zeros), count, reinterpret_cast<int *>(status));
    const cudaError_t err = cudaGetLastError();
    return err == cudaSuccess ? 0 : (6 << 16) | (err & 0xFFFF);
}

} // extern "C"
