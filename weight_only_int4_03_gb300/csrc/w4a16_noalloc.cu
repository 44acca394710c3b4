// w4a16_noalloc.cu -- w4a16_gemm_noalloc: the dense W4A16 GEMM with its scratch memory (status
// word, split-K tile counters, fp32 partial tiles, act-order copy of A) in a fixed array that
// the library owns, for callers that cannot allocate device memory.
//
// Who needs it: code that runs where cudaMalloc is off limits -- inside a host callback or
// another library's allocator hook, under a memory pool that a framework has sealed, or in a
// plug-in whose host gives it no allocator and no workspace argument -- still has to pass a
// workspace to w4a16_gemm.  This entry point takes none.  Nothing here calls cudaMalloc,
// cudaFree or any routine that allocates.
//
// The array is W4A16_NOALLOC_SCRATCH_BYTES (32 MiB) of device memory per GPU that loads the
// library, held until the process exits.  Every call on a device shares it, so calls whose
// kernels overlap on the GPU (two streams, or two host threads) race and give wrong results;
// serialise them.
#include <mutex>

#include "w4a16.h"
#include "w4a16_internal.h"

static __device__ __align__(256) unsigned char g_scratch[W4A16_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int MAX_DEVICES = 64;
constexpr size_t HEADER_BYTES = 256; // the workspace starts with the status word ...
constexpr int TILE_COLS = 128;       // ... then one counter per (token tile, 128-column tile)
constexpr int MIN_TILE_ROWS = 8;     // the smallest token tile either kernel uses

std::mutex g_mu;
void *g_scratch_ptr[MAX_DEVICES];

// Device address of g_scratch on the current device (host code cannot use the symbol's name
// as an address).  Looked up once per device, on that device's first call.
int scratch_address(void **out)
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    if (dev < 0 || dev >= MAX_DEVICES)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        err = cudaGetSymbolAddress(&p, g_scratch);
        if (err != cudaSuccess)
            return err;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

} // namespace

extern "C" int w4a16_gemm_noalloc(const void *a, int lda, const int32_t *b_packed, void *c, int ldc,
                                  const void *scales, const void *zeros, const int32_t *g_idx,
                                  const int32_t *perm, int32_t *status_out, int m, int n, int k,
                                  int group_size, int weight_type, unsigned flags,
                                  cudaStream_t stream)
{
    if (m == 0 || m < 0 || n <= 0 || k <= 0)
        // Same answers as w4a16_gemm for an empty or invalid shape (no scratch needed).
        return w4a16_gemm(a, lda, b_packed, c, ldc, scales, zeros, g_idx, perm, nullptr, 0, m, n, k,
                          group_size, weight_type, flags, stream);
    // The tallest token tiles (up to 256 rows) take more partial-slot room than the scratch
    // holds; tiles of at most 192 rows -- two accumulator buffers, the kernel's former default
    // -- fit for every shape, so only an act-order copy of A can push a call over.
    const int tile_cap = w4::TWO_BUF_TILE_TOK;
    const size_t need = w4::dense_workspace_size(m, n, k, group_size, flags, 0, tile_cap);
    if (need == 0)
        // Invalid sizes: let the full argument checks of w4a16_gemm name the problem.
        return w4a16_gemm(a, lda, b_packed, c, ldc, scales, zeros, g_idx, perm, nullptr, 0, m, n, k,
                          group_size, weight_type, flags, stream);
    if (need > (size_t)W4A16_NOALLOC_SCRATCH_BYTES)
        return (2 << 16) | W4A16_ARG_SCRATCH;
    if (status_out && (reinterpret_cast<uintptr_t>(status_out) & 3u))
        return (1 << 16) | W4A16_ARG_ALIGN;

    void *ws = nullptr;
    int err = scratch_address(&ws);
    if (err != cudaSuccess)
        return (3 << 16) | (err & 0xFFFF);

    // The status word and the tile counters must start at zero.  A call that completes leaves
    // them so, but one that gave up on a bounded wait may not: clear them on every call.
    const size_t tiles_bound =
        (size_t)((m + MIN_TILE_ROWS - 1) / MIN_TILE_ROWS) * (size_t)(n / TILE_COLS);
    size_t clear = HEADER_BYTES + 4 * tiles_bound;
    if (clear > need)
        clear = need;
    err = cudaMemsetAsync(ws, 0, clear, stream);
    if (err != cudaSuccess)
        return (6 << 16) | (err & 0xFFFF);

    const int st = w4::dense_gemm(a, lda, b_packed, c, ldc, scales, zeros, g_idx, perm, ws,
                                  (size_t)W4A16_NOALLOC_SCRATCH_BYTES, m, n, k, group_size,
                                  weight_type, flags, stream, tile_cap);
    if (st != 0 || !status_out)
        return st;
    // Hand the call's device-side error bits to the caller (stream-ordered, no host wait).
    err = cudaMemcpyAsync(status_out, ws, sizeof(int32_t), cudaMemcpyDeviceToDevice, stream);
    return err == cudaSuccess ? 0 : ((6 << 16) | (err & 0xFFFF));
}
