// w4a16_internal.h -- shared definitions of the library's translation units (not installed).
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "w4a16.h"

namespace w4 {

// Packed tile geometry (see include/w4a16.h, "Packed tile layout").
constexpr int TILE_N = 128;      // weight columns per tile = tcgen05 M (weights are the A operand)
constexpr int KBLK = 64;         // K rows per tile
constexpr int TILE_WORDS = 1024; // 32-bit words per tile
constexpr int TILE_BYTES = 4096;
constexpr int TILE_WORDS_FP8 = 2048; // the same tile of FP8 E4M3 codes
constexpr int TILE_BYTES_FP8 = 8192;

// Pipeline geometry.
constexpr int SG_BYTES = TILE_N * 2; // one scale (or zero) row of a column tile
constexpr int MAX_A_SLOTS = 12;      // dequantised-weight ring in tensor memory (runtime size)
constexpr int SMEM_A_SLOTS = 4;      // ... or in shared memory
constexpr int A_SLOT_COLS = 32;      // tensor-memory columns per slot: 64 fp16 per lane
constexpr int A_SLOT_BYTES = TILE_N * KBLK * 2;
constexpr int MAX_STAGES = 16;
constexpr int MAX_TOK = 256;         // activation rows per tile = tcgen05 N upper bound
constexpr int TALL_TILE_TOK = 224;   // tallest token tile chosen for M above one tile
constexpr int TWO_BUF_TILE_TOK = 192; // tallest token tile with two accumulator buffers
constexpr int PAIR_HALF_TOK = 192;    // tallest half-tile of a paired token tile

// Warp roles of the tcgen05 GEMM kernel.
constexpr int NUM_THREADS = 512;
constexpr int PRODUCER_WARP = 0;
constexpr int MMA_WARP = 1;
constexpr int SEG_WARP = 2;      // builds the grouped schedule table at start-up
constexpr int EPI_WARP0 = 4;     // warps 4..7: one per tensor-memory lane quarter
constexpr int DQ_WARP0 = 8;      // warps 8..15: two sets of four (one warp per lane quarter)
constexpr int DQ_WARPS = 8;
constexpr int EPI_THREADS = 128;
constexpr int EPI_ROWS = 32;                               // token rows per epilogue batch
constexpr int EPI_STAGE_BYTES = 4 * EPI_ROWS * 32 * 2;     // per warp: 32 rows x 32 columns fp16

constexpr int MAX_SEGMENTS = 1024;

// Column-slice small-M kernel: 16 weight columns over all of K per work item; a pipeline
// stage holds slice_bpw consecutive blocks for each of the 8 compute warps.
constexpr int SLICE_N = 16;
__host__ __device__ constexpr int slice_bpw(int nt_max, bool w8 = false)
{
    // FP8 blocks carry twice the code bytes: half as many per warp (at least one).
    return (nt_max <= 8 ? 4 : nt_max <= 16 ? 2 : 1) / (w8 && nt_max <= 16 ? 2 : 1);
}
constexpr int SLICE_BLOCK_BYTES = SLICE_N * KBLK / 2; // codes of one block of a slice
constexpr int SLICE_MAX_ROWS = 32;
constexpr int SLICE_WARPS = 8; // compute warps of the small-M kernels

struct GemmParams {
    const int32_t *b;         // packed tiles (expert 0)
    const __half *scales;     // [G][N] (expert 0)
    const __half *zeros;      // [G][N] or null (u4b8)
    __half *c;                // output rows
    int ldc;
    float *partials;          // [grid][2][nt_max][128] fp32 split-K partial tiles
    int *counters;            // one per tile
    int *status;              // device status word
    unsigned long long limit_ns;
    int m, n, k;
    int group_size;           // resolved: K for a single group
    int num_groups;
    int nt_max;               // activation rows per tile (multiple of 16, <= 256)
    int m_tiles;              // dense: ceil(m / nt_max)
    int n_tiles, kblocks;
    int stages, stage_bytes;
    int kbs;                  // 64-row blocks per pipeline stage
    int act_kb_bytes;         // activation bytes per block in a stage (nt_max rows x 128 B)
    int packed_off, scales_off, zeros_off; // byte offsets inside a stage
    int sg_box;               // scale rows copied per stage
    int acc_bufs, acc_col0, tmem_cols;
    int w8;                   // FP8 E4M3 weights (tcgen05 kernel only)
    int bf16;                 // bfloat16 activations, scales, zeros and output (tcgen05 only)
    int tile_words, tile_bytes; // one packed 64 x 128 tile: 1024 words (4-bit) or 2048 (FP8)
    int halves;               // tcgen05 kernel: 1, or 2 when a tile is a pair of token half-tiles
                              // that share each dequantised weight block
    int nt_half;              // rows of a half-tile (= nt_max when halves is 1)
    int a_slots;              // dequantised-weight ring slots (<= MAX_A_SLOTS)
    int seg_smem_off;         // grouped: byte offset of the schedule table in dynamic smem
    int epi_smem_off;         // tcgen05 kernel: byte offset of the epilogue's staging buffer
    int static_weights;       // weights may be read before the preceding kernel completes
    int split;                // > 0: tile-aligned split schedule (grid = tiles * split)
    int m_outer;              // dense: tile index runs token-tile-major
    int n_slices, slice_per;  // column-slice kernel: N / 16 slices, consecutive slices per CTA
    int glu;                  // 0: C = the product; 1 / 2: C[., f] = silu / gelu_tanh(gate) * up
                              // over gate/up columns interleaved in 16-column blocks
    // grouped schedule (null ex_off = dense)
    const int *ex_off;
    const int *ex_ids;
    const int *ex_pairs;
    int n_active, n_experts, n_pairs;
    int n_rows;               // grouped: rows of the sorted activation copy (segments end there)
    int skip_sentinel;        // grouped: an ex_pairs entry of -1 is a padding row, not an error
    const float *row_weight;  // grouped: output row o is scaled by row_weight[o] (or null)
    long long b_expert_words;
    long long s_expert_elems;
};

struct GemmConfig {
    int grid;
    int smem_bytes;
    bool a_tmem;
};

// Launchers (return a cudaError_t value).
int launch_gemm(const GemmParams &p, const CUtensorMap &tmap_a, const CUtensorMap &tmap_s,
                const CUtensorMap &tmap_z, const GemmConfig &cfg, cudaStream_t stream);
int launch_decode(const GemmParams &p, const CUtensorMap &tmap_a, const CUtensorMap &tmap_s,
                  const CUtensorMap &tmap_z, const GemmConfig &cfg, cudaStream_t stream);
int launch_slice(const GemmParams &p, const CUtensorMap &tmap_a, const CUtensorMap &tmap_w,
                 const CUtensorMap &tmap_s, const CUtensorMap &tmap_z, const GemmConfig &cfg,
                 cudaStream_t stream);
int launch_gemm_simt(const GemmParams &p, const __half *a, int lda, cudaStream_t stream);
int launch_repack(const int32_t *qweight, const int32_t *perm, int32_t *out, int32_t *status, int k,
                  int n, cudaStream_t stream);
int launch_unpack(const int32_t *tiles, int32_t *qweight, int k, int n, cudaStream_t stream);
int launch_repack_fp8(const int32_t *qweight, int32_t *out, int k, int n, cudaStream_t stream);
int launch_unpack_fp8(const int32_t *tiles, int32_t *qweight, int k, int n, cudaStream_t stream);
int launch_gather_cols(const __half *a, int lda, const int32_t *perm, const int32_t *g_idx,
                       int group_size, __half *out, int m, int k, int *status, cudaStream_t stream);
int launch_gather_rows(const __half *a, int lda, const int32_t *ex_pairs, const int32_t *pair_tok,
                       __half *out, int n_pairs, int n_tokens, int k, int *status,
                       cudaStream_t stream);
int launch_selftest_timeout(int *status, unsigned long long limit_ns, cudaStream_t stream);
constexpr int MOE_MAX_BLOCKS = W4A16_MOE_MAX_BLOCKS; // blocks per block-routed MoE call
int launch_moe_route(const int32_t *sorted_ids, const int32_t *expert_ids, const int32_t *ntpp,
                     int max_padded, int block_size, int n_ids, int n_experts, int is_ep,
                     int seg_cap, int32_t *ex_off, int32_t *ex_ids, int32_t *ex_pairs, int *status,
                     cudaStream_t stream);
int launch_moe_gather(const __half *a, int lda, const int32_t *ex_off_end, const int32_t *ex_pairs,
                      int top_k, __half *out, int max_padded, int k, cudaStream_t stream);
int launch_gate_up_interleave(const void *src, void *dst, int rows, int n2, int elem_bytes,
                              cudaStream_t stream);
int gemm_smem_limit(int *bytes);

// Dynamic shared memory the kernels need beyond the stages.
int gemm_extra_smem(bool a_tmem, bool grouped);
int decode_extra_smem(int nt_max);
int decode_max_rows();
int decode_ctas_per_sm();
int decode_smem_limit(int *bytes);

// The dense entry points with the tcgen05 kernel's token tile held to at most tile_cap rows (a
// multiple of 16, TWO_BUF_TILE_TOK..MAX_TOK): w4a16_workspace_size / w4a16_gemm use MAX_TOK;
// a caller with a fixed scratch may ask for shorter tiles, whose partial slots take less.
size_t dense_workspace_size(int m, int n, int k, int group_size, unsigned flags, int num_sms,
                            int tile_cap);
int dense_gemm(const void *a, int lda, const int32_t *b_packed, void *c, int ldc,
               const void *scales, const void *zeros, const int32_t *g_idx, const int32_t *perm,
               void *workspace, size_t workspace_bytes, int m, int n, int k, int group_size,
               int weight_type, unsigned flags, cudaStream_t stream, int tile_cap);

} // namespace w4
