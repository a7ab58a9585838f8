// w4_repack: canonical layout -> kernel layout (offline, once per weight).
//
// The kernel layout feeds the bf16 tensor-core operation mma.m16n8k16 with
// weights as its A operand (16 rows x 16 k) and up to 8 tokens as its B
// operand, and is cut into records that one bulk copy can move: rows are
// grouped in tiles of 16 and row blocks of 8 tiles (128 rows, padded with
// zero weights past N); K in groups of 128.  Record (b, g) -- row block b,
// group g -- holds, in each of the three buffers:
//   qweight: 8 KB at 128 + (b*G + g) * 8192: tile w (0..7), chunk c (0..1,
//            64 k each, kc = 128g + 64c), lane l = 4*gq + tq: 16 bytes at
//            w*1024 + c*512 + l*16, four 32-bit words v = 0..3.  The sum over
//            k does not depend on the order of k, so inside a chunk the four
//            k-steps j of the tensor-core operation take a permuted k: column
//            pair (2tq, 2tq+1) of step j is k = kc + 16tq + 4j + {0, 1} and
//            column pair (2tq+8, 2tq+9) is k = kc + 16tq + 4j + {2, 3}.  With
//            that order the B registers a lane needs for the chunk are the
//            eight consecutive x pairs starting at kc + 16tq: two 16-byte loads
//            straight from x as copied, no rearranging.  With
//            k0 = kc + 16tq + 4*(v >> 1) + 2*(v & 1), word v holds the pairs
//            (first k of a pair in the low half-word, second in the high one):
//              bits  0- 3 / 16-19 : row 16t+gq,   k = k0     / k0 + 1
//              bits  4- 7 / 20-23 : row 16t+gq,   k = k0 + 8 / k0 + 9
//              bits  8-11 / 24-27 : row 16t+gq+8, k = k0     / k0 + 1
//              bits 12-15 / 28-31 : row 16t+gq+8, k = k0 + 8 / k0 + 9
//            with t = 8b + w.  Steps 0 and 1 of the chunk take their A
//            registers from the nibbles at bits 0-3 and 8-11 of words
//            (0, 1) and (2, 3); steps 2 and 3 from bits 4-7 and 12-15.  So
//            word & 0x000F000F, word & 0x00F000F0, (word >> 8) & 0x000F000F
//            and (word >> 8) & 0x00F000F0 are A registers as they stand: one
//            shift per word (the second pair of each half-word sits four bits
//            higher, which an fp16 mantissa absorbs as a factor 16; see
//            w4_device.cuh).  This is the even/odd pair interleave of
//            "Building an LLM Inference Runtime ...", section "Bug #3"
//            (nibble slots hold w0,w2,w4,w6 in the low half-word and
//            w1,w3,w5,w7 in the high one), extended to the two rows and the
//            two step pairs of a fragment.
//   scales:  256 B at (b*G + g) * 256: uint32 [w][gq] = fp16 scale of row
//            16t+gq (low half) and of row 16t+gq+8 (high half).
//   zeros:   64 B at (b*G + g) * 64: byte [w][gq] = z of row 16t+gq (low
//            nibble) | z of row 16t+gq+8 (high nibble).
// Padded rows have q = z = 0 and s = 0, so they contribute exact zeros.
//
// Gate/up-interleaved layout (layout id W4_LAYOUT_ID_SWIGLU): the input is a
// fused [2I][K] weight (gate rows 0..I-1, up rows I..2I-1) and kernel row
// r = 16 t + i holds gate row 8t + i for i < 8 and up row 8t + i - 8 for
// i >= 8 (zero past I).  Each lane of the tensor-core operation then holds,
// for rows gq and gq + 8 of a tile, the gate and the up product of the same
// output, so the activation runs in registers ("qengine", section "How it
// works": gate and up projections interleaved so SwiGLU runs in registers).
#include <string.h>

#include "w4_internal.cuh"

namespace w4 {
namespace {

__global__ void write_header_kernel(Header *h, int K, int N, uint32_t layout_id) {
    const char magic[8] = {'W', '4', 'G', '1', '2', '8', 'K', 'L'};
    for (int i = 0; i < 8; ++i) h->magic[i] = magic[i];
    h->layout_id = layout_id;
    h->version = W4_LAYOUT_VERSION;
    h->K = K;
    h->N = N;
    h->bad_zeros = 0;
    h->kernel_error = 0;
    for (int i = 0; i < 24; ++i) h->reserved[i] = 0;
}

__device__ __forceinline__ uint32_t nib(uint32_t w, int i) { return (w >> (4 * i)) & 0xFu; }

// Canonical row of kernel row r, or -1 for a zero row.
__device__ __forceinline__ int src_row(int r, int N, int swiglu_I) {
    if (swiglu_I == 0) return r < N ? r : -1;
    const int j = 8 * (r >> 4) + (r & 7);
    if (j >= swiglu_I) return -1;
    return (r & 8) ? swiglu_I + j : j;
}

__global__ void repack_weights_kernel(const uint32_t *__restrict__ qw, int K, int N, int NB,
                                      int swiglu_I, uint4 *__restrict__ out) {
    const int G = K / kGroup;
    const size_t words_per_row = (size_t)K / 8;
    const size_t total = (size_t)NB * G * (kRecWeights / 16);
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (size_t)gridDim.x * blockDim.x) {
        const int lane = (int)(i & 31);
        const int c = (int)((i >> 5) & 1);
        const int w = (int)((i >> 6) & 7);
        const size_t bg = i >> 9;
        const int g = (int)(bg % G);
        const int b = (int)(bg / G);
        const int gq = lane >> 2, tq = lane & 3;
        const int r0 = (b * kBlockTiles + w) * kTileRows + gq;
        const int s0 = src_row(r0, N, swiglu_I), s1 = src_row(r0 + 8, N, swiglu_I);
        const uint32_t *ra = s0 >= 0 ? qw + (size_t)s0 * words_per_row : nullptr;
        const uint32_t *rb = s1 >= 0 ? qw + (size_t)s1 * words_per_row : nullptr;
        // nibble of canonical row r (base pointer) at k; 0 for a zero row
        auto q = [](const uint32_t *r, int k) -> uint32_t {
            return r ? nib(r[k / 8], k % 8) : 0u;
        };
        uint32_t res[4];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const int k0 = g * kGroup + c * kChunkK + 16 * tq + 4 * (v >> 1) + 2 * (v & 1);
            res[v] = q(ra, k0) | (q(ra, k0 + 8) << 4) | (q(rb, k0) << 8) | (q(rb, k0 + 8) << 12) |
                     (q(ra, k0 + 1) << 16) | (q(ra, k0 + 9) << 20) | (q(rb, k0 + 1) << 24) |
                     (q(rb, k0 + 9) << 28);
        }
        out[i] = make_uint4(res[0], res[1], res[2], res[3]);
    }
}

__global__ void repack_meta_kernel(const uint16_t *__restrict__ sc, const uint8_t *__restrict__ zp,
                                   int K, int N, int NB, int swiglu_I,
                                   uint32_t *__restrict__ sc_out,
                                   uint8_t *__restrict__ zp_out, Header *h) {
    const int G = K / kGroup;
    const size_t total = (size_t)NB * G * 64;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (size_t)gridDim.x * blockDim.x) {
        const int gq = (int)(i & 7);
        const int w = (int)((i >> 3) & 7);
        const size_t bg = i >> 6;
        const int g = (int)(bg % G);
        const int b = (int)(bg / G);
        const int r0 = (b * kBlockTiles + w) * kTileRows + gq;
        const int c0 = src_row(r0, N, swiglu_I), c1 = src_row(r0 + 8, N, swiglu_I);
        const uint32_t s0 = c0 >= 0 ? sc[(size_t)c0 * G + g] : 0u;
        const uint32_t s1 = c1 >= 0 ? sc[(size_t)c1 * G + g] : 0u;
        const uint32_t z0 = c0 >= 0 ? zp[(size_t)c0 * G + g] : 0u;
        const uint32_t z1 = c1 >= 0 ? zp[(size_t)c1 * G + g] : 0u;
        if (z0 > 15u || z1 > 15u) atomicOr(&h->bad_zeros, 1u);
        sc_out[i] = s0 | (s1 << 16);
        zp_out[i] = (uint8_t)((z0 & 0xFu) | ((z1 & 0xFu) << 4));
    }
}

int grid_for(size_t work, int threads) {
    size_t blocks = (work + threads - 1) / threads;
    if (blocks > 65535u * 8u) blocks = 65535u * 8u;
    return blocks ? (int)blocks : 1;
}

}  // namespace

cudaError_t launch_repack(const uint32_t *qweight, const uint16_t *scales, const uint8_t *zeros,
                          int K, int N, int swiglu_I, void *qweight_out, void *scales_out,
                          void *zeros_out, cudaStream_t stream) {
    const int NB = row_blocks(N);
    const int G = K / kGroup;
    Header *h = static_cast<Header *>(qweight_out);
    write_header_kernel<<<1, 1, 0, stream>>>(h, K, swiglu_I ? swiglu_I : N,
                                             swiglu_I ? W4_LAYOUT_ID_SWIGLU : W4_LAYOUT_ID);
    const size_t pieces = (size_t)NB * G * (kRecWeights / 16);
    repack_weights_kernel<<<grid_for(pieces, 256), 256, 0, stream>>>(
        qweight, K, N, NB, swiglu_I,
        reinterpret_cast<uint4 *>(static_cast<char *>(qweight_out) + W4_HEADER_BYTES));
    const size_t metas = (size_t)NB * G * 64;
    repack_meta_kernel<<<grid_for(metas, 256), 256, 0, stream>>>(
        scales, zeros, K, N, NB, swiglu_I, static_cast<uint32_t *>(scales_out),
        static_cast<uint8_t *>(zeros_out), h);
    return cudaGetLastError();
}

}  // namespace w4
