// Internal declarations shared by the CUDA translation units of libw4.
// Not part of the public ABI (that is include/w4.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "w4.h"

namespace w4 {

constexpr int kGroup = 128;      // weights per (row, scale, zero) group along K
constexpr int kTileRows = 16;    // rows per tile = M of one m16n8k16 tensor-core op
constexpr int kChunkK = 64;      // K covered by one 16-byte load of every lane of a warp
constexpr int kBlockTiles = 8;   // tiles per row block (one per consumer warp)
constexpr int kBlockRows = kTileRows * kBlockTiles;   // 128
constexpr int kMaxSplits = 8;    // thread blocks per cluster (portable cluster size)
// Bytes of one (row block, group) record in each of the three buffers.
constexpr int kRecWeights = kBlockTiles * 1024;      // 8 tiles x 2 chunks x 32 lanes x 16 B
constexpr int kRecScales = kBlockTiles * 8 * 4;      // 8 tiles x 8 lane groups x 2 fp16
constexpr int kRecZeros = kBlockTiles * 8;           // 8 tiles x 8 lane groups x 2 nibbles

// First W4_HEADER_BYTES of a repacked qweight buffer.
struct Header {
    char magic[8];          // "W4G128KL"
    uint32_t layout_id;     // W4_LAYOUT_ID
    uint32_t version;       // W4_LAYOUT_VERSION
    int32_t K;
    int32_t N;
    uint32_t bad_zeros;     // set by w4_repack when a zero point > 15 was seen
    uint32_t kernel_error;  // set by w4_gemv if a wait gave up (never in normal operation)
    uint32_t reserved[24];
};
static_assert(sizeof(Header) == W4_HEADER_BYTES, "header size");

__host__ __device__ inline int row_blocks(int N) { return (N + kBlockRows - 1) / kBlockRows; }

// Rows of the gate/up-interleaved layout for I outputs: every 16-row tile
// holds 8 gate rows and the 8 matching up rows (see w4_repack.cu).
__host__ __device__ inline int swiglu_rows(int I) { return 16 * ((I + 7) / 8); }
constexpr size_t kErrorOffset = 28;   // byte offset of Header::kernel_error

// Kernel-layout byte sizes (see w4_repack.cu for the layout itself).
inline size_t packed_qweight_bytes(int K, int N) {
    return (size_t)W4_HEADER_BYTES + (size_t)row_blocks(N) * (K / kGroup) * kRecWeights;
}
inline size_t packed_scales_bytes(int K, int N) {
    return (size_t)row_blocks(N) * (K / kGroup) * kRecScales;
}
inline size_t packed_zeros_bytes(int K, int N) {
    return (size_t)row_blocks(N) * (K / kGroup) * kRecZeros;
}

// swiglu_I = 0: plain layout of an N x K weight.  swiglu_I = I > 0: the
// input is a fused [2I][K] gate/up weight and N must be swiglu_rows(I).
cudaError_t launch_repack(const uint32_t *qweight, const uint16_t *scales,
                          const uint8_t *zeros, int K, int N, int swiglu_I, void *qweight_out,
                          void *scales_out, void *zeros_out, cudaStream_t stream);

cudaError_t launch_dequant(const uint32_t *qweight, const uint16_t *scales,
                           const uint8_t *zeros, int K, int N, uint16_t *w_out,
                           cudaStream_t stream);

struct GemvShape {
    int warps;    // consumer warps per block; each owns one 16-row tile
    int splits;   // K splits = blocks per cluster
    int stages;   // depth of the shared-memory weight ring
    bool fold;    // zero point folded out of the inner product (see w4_gemv.cu)
};

// Launch shape for an N x K weight (independent of M).  Returns false if no
// shape fits the shared-memory budget.
bool gemv_shape(int K, int N, int num_sms, GemvShape *out);

// What launch_gemv will launch for (M, K, N): which kernel instance, the
// grid, shared memory and whether it overlaps the previous kernel.
struct GemvLaunch {
    GemvShape shape;
    int variant;        // 0: two blocks per SM, 6 stages; 1: three, 6; 2: three, 5
    int arith;          // 0: exact q - z; 1: folded; 2: folded, wide x prologue
    bool persistent;    // blocks take row blocks in turn
    bool capped;        // shared memory padded to cap blocks per SM
    bool overlap;       // programmatic dependent launch
    dim3 grid;
    size_t smem_bytes;
    int stages;
};

cudaError_t plan_gemv(bool f32_out, int M, int K, int N, const GemvShape &shape, int num_sms,
                      GemvLaunch *out);

// swiglu_I = 0: y[M][N] = W x.  swiglu_I = I > 0: W is a gate/up-interleaved
// weight of N = swiglu_rows(I) rows and y[M][I] = silu(gate x) * (up x).
cudaError_t launch_gemv(const void *qweight, const void *scales, const void *zeros,
                        const uint16_t *x, void *y, bool f32_out, int M, int K, int N,
                        const GemvShape &shape, int swiglu_I, int num_sms,
                        cudaStream_t stream);

// Tensor-core (tcgen05) product for more than W4_MAX_TOKENS tokens
// (w4_gemm_tc.cu): one pass over the weight, blocks of 128 rows x 128 tokens.
int gemm_tc_splits(int K, int N, int num_sms);
cudaError_t launch_gemm_tc(const void *qweight, const void *scales, const void *zeros,
                           const uint16_t *x, void *y, bool f32_out, int M, int K, int N,
                           int num_sms, cudaStream_t stream);

// Workspace path (w4_gemv_sk.cu): grid size, workspace bytes, launch.
int gemv_ws_blocks(int K, int N, int num_sms);
size_t gemv_ws_bytes(int K, int N, int num_sms);
cudaError_t launch_quantize(const uint16_t *w, int K, int N, bool symmetric, uint32_t *qweight,
                            uint16_t *scales, uint8_t *zeros, int num_sms, cudaStream_t stream);
cudaError_t launch_gemv_ws(const void *qweight, const void *scales, const void *zeros,
                           const uint16_t *x, void *y, bool f32_out, int M, int K, int N,
                           void *workspace, int num_sms, cudaStream_t stream);

}  // namespace w4
