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
constexpr int kMaxSplits = 8;    // thread blocks per cluster (portable cluster size)

// First W4_HEADER_BYTES of a repacked qweight buffer.
struct Header {
    char magic[8];          // "W4G128KL"
    uint32_t layout_id;     // W4_LAYOUT_ID
    uint32_t version;       // W4_LAYOUT_VERSION
    int32_t K;
    int32_t N;
    uint32_t bad_zeros;     // set by w4_repack when a zero point > 15 was seen
    uint32_t reserved[25];
};
static_assert(sizeof(Header) == W4_HEADER_BYTES, "header size");

inline int row_tiles(int N) { return (N + kTileRows - 1) / kTileRows; }

// Kernel-layout byte sizes (see w4_repack.cu for the layout itself).
inline size_t packed_qweight_bytes(int K, int N) {
    return (size_t)W4_HEADER_BYTES + (size_t)row_tiles(N) * kTileRows * (size_t)K / 2;
}
inline size_t packed_scales_bytes(int K, int N) {
    return (size_t)row_tiles(N) * (K / kGroup) * 8 * sizeof(uint32_t);
}
inline size_t packed_zeros_bytes(int K, int N) {
    return (size_t)row_tiles(N) * (K / kGroup) * 8;
}

cudaError_t launch_repack(const uint32_t *qweight, const uint16_t *scales,
                          const uint8_t *zeros, int K, int N, void *qweight_out,
                          void *scales_out, void *zeros_out, cudaStream_t stream);

cudaError_t launch_dequant(const uint32_t *qweight, const uint16_t *scales,
                           const uint8_t *zeros, int K, int N, uint16_t *w_out,
                           cudaStream_t stream);

struct GemvShape {
    int warps;    // warps per block; each owns one 16-row tile
    int splits;   // K splits = blocks per cluster
};

// Launch shape for an N x K weight (independent of M).  Returns false if no
// shape fits the shared-memory budget.
bool gemv_shape(int K, int N, int num_sms, GemvShape *out);

cudaError_t launch_gemv(const void *qweight, const void *scales, const void *zeros,
                        const uint16_t *x, void *y, bool f32_out, int M, int K, int N,
                        const GemvShape &shape, cudaStream_t stream);

}  // namespace w4
