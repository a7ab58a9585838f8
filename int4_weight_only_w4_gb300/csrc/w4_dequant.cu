// w4_dequant: canonical INT4 weights -> fp16 W[N][K], for checking.
//
// One thread per 16-byte piece of a row (four packed words = 32 weights of one
// group): read once, unpack all 32 nibbles, write 64 bytes.  This is the
// "one thread per packed word" shape of "Custom AWQ Dequantization Kernel",
// section "Kernel versions" (v2), widened to 16-byte loads.
//
// Each value is (q - z) * s computed in fp32 -- exact, since |q - z| needs at
// most 8 bits for any uint8 z and an fp16 significand 11 -- and rounded once
// to fp16, nearest-even.
#include <cuda_fp16.h>

#include "w4_internal.cuh"

namespace w4 {
namespace {

__global__ void dequant_kernel(const uint4 *__restrict__ qw, const uint16_t *__restrict__ sc,
                               const uint8_t *__restrict__ zp, int K, int N,
                               uint4 *__restrict__ out) {
    const int G = K / kGroup;
    const int pieces_per_row = K / 32;
    const size_t total = (size_t)N * pieces_per_row;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (size_t)gridDim.x * blockDim.x) {
        const size_t n = i / pieces_per_row;
        const int k0 = (int)(i % pieces_per_row) * 32;
        const size_t gi = n * G + k0 / kGroup;
        const float s = __half2float(__ushort_as_half(sc[gi]));
        const int z = zp[gi];
        const uint4 w = qw[i];
        const uint32_t words[4] = {w.x, w.y, w.z, w.w};
        uint32_t packed[16];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const int qa = (int)((words[j] >> (8 * p)) & 0xFu);
                const int qb = (int)((words[j] >> (8 * p + 4)) & 0xFu);
                const __half ha = __float2half_rn((float)(qa - z) * s);
                const __half hb = __float2half_rn((float)(qb - z) * s);
                packed[4 * j + p] = (uint32_t)__half_as_ushort(ha) |
                                    ((uint32_t)__half_as_ushort(hb) << 16);
            }
        }
        uint4 *dst = out + (n * (size_t)K + k0) / 8;
#pragma unroll
        for (int v = 0; v < 4; ++v)
            dst[v] = make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2],
                                packed[4 * v + 3]);
    }
}

}  // namespace

cudaError_t launch_dequant(const uint32_t *qweight, const uint16_t *scales, const uint8_t *zeros,
                           int K, int N, uint16_t *w_out, cudaStream_t stream) {
    const size_t work = (size_t)N * (K / 32);
    size_t blocks = (work + 255) / 256;
    if (blocks > 65535u * 8u) blocks = 65535u * 8u;
    dequant_kernel<<<(int)blocks, 256, 0, stream>>>(reinterpret_cast<const uint4 *>(qweight),
                                                    scales, zeros, K, N,
                                                    reinterpret_cast<uint4 *>(w_out));
    return cudaGetLastError();
}

}  // namespace w4
