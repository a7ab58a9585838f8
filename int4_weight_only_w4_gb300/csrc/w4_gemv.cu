// w4_gemv: fused INT4-dequantise + matrix-vector product for sm_103a.
//
// Work split.  A thread block of `warps` warps owns `warps` consecutive
// 16-row tiles (one per warp) and one slice of K.  With `splits` > 1 the
// K slices of the same tiles are handled by the `splits` blocks of one thread
// block cluster, which combine their fp32 partial sums through distributed
// shared memory in a fixed rank order: deterministic, no workspace, no float
// atomics ("qengine", section "Learnings": float atomics made one run in fifty
// differ; a fixed summation order fixed it).
//
// Per warp.  Each lane streams its 16-byte pieces of the packed weights (see
// w4_repack.cu for the layout) with L1-bypassing 128-bit loads, keeping kInFlight
// pieces in flight.  A piece holds 64 k of its fragment rows; each of its four
// words is turned into the four bf16x2 registers of a tensor-core A fragment
// without any conversion instruction: (word >> 4p) & 0x000F000F | 0x43004300
// is the bf16 pair (128 + q_even, 128 + q_odd) exactly (bf16 has 7 fraction
// bits, so 128 + q for q < 128 is exact), and one bf16x2 subtraction of
// (128 + z) leaves q - z exactly.  mma.m16n8k16 (bf16 inputs, fp32
// accumulation) then multiplies the 16 x 16 weight block with up to 8 token
// columns of x.  The products q - z times x are exact; the scale is applied
// once per group of 128 in fp32: acc += s * sum_group (q - z) x.
//
// x staging.  Each block copies its K slice of x (bf16 pairs, no arithmetic)
// to shared memory, permuted so that each lane's eight B-fragment registers
// for one 64-k piece are two consecutive 16-byte words.  Lanes whose token
// column is >= M feed zeros.  The shape (warps, splits) depends only on K and N,
// so the result for one token does not depend on M (batch invariance,
// "qengine", section "How it works": identical results for row r whether 1 or
// 8 rows are processed).
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "w4_internal.cuh"

namespace cg = cooperative_groups;

namespace w4 {
namespace {

constexpr int kInFlight = 8;      // 16-byte pieces per lane in flight (even)
constexpr int kWarps = 8;         // warps (16-row tiles) per block
constexpr size_t kMaxXBytes = 200 * 1024;   // shared-memory budget for staged x

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t ld_nc_u32(const uint32_t *p) {
    uint32_t r;
    asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(r) : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t ld_nc_u8(const uint8_t *p) {
    uint16_t r;
    asm volatile("ld.global.nc.u8 %0, [%1];" : "=h"(r) : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
    __nv_bfloat162 va = *reinterpret_cast<__nv_bfloat162 *>(&a);
    __nv_bfloat162 vb = *reinterpret_cast<__nv_bfloat162 *>(&b);
    __nv_bfloat162 r = __hsub2(va, vb);
    return *reinterpret_cast<uint32_t *>(&r);
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// One 16-byte piece: four k-steps of 16.
__device__ __forceinline__ void piece_mma(float (&d)[4], const uint4 &w, const uint32_t (&b)[8],
                                          uint32_t czl, uint32_t czh) {
    const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t wd = words[j];
        uint32_t a0 = (wd & 0x000F000Fu) | 0x43004300u;
        uint32_t a1 = ((wd >> 4) & 0x000F000Fu) | 0x43004300u;
        uint32_t a2 = ((wd >> 8) & 0x000F000Fu) | 0x43004300u;
        uint32_t a3 = ((wd >> 12) & 0x000F000Fu) | 0x43004300u;
        a0 = bf16x2_sub(a0, czl);
        a1 = bf16x2_sub(a1, czh);
        a2 = bf16x2_sub(a2, czl);
        a3 = bf16x2_sub(a3, czh);
        mma_bf16_16816(d, a0, a1, a2, a3, b[2 * j], b[2 * j + 1]);
    }
}

template <bool F32OUT>
__device__ __forceinline__ void store_tile(void *yv, const float (&acc)[4], int t, int lane,
                                           int M, int N) {
    const int gq = lane >> 2, tq = lane & 3;
    const int r0 = t * kTileRows + gq, r1 = r0 + 8;
    const int m0 = 2 * tq, m1 = m0 + 1;
    const float v[4] = {acc[0], acc[1], acc[2], acc[3]};
    const int ms[4] = {m0, m1, m0, m1};
    const int rs[4] = {r0, r0, r1, r1};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (ms[i] < M && rs[i] < N) {
            const size_t o = (size_t)ms[i] * N + rs[i];
            if (F32OUT)
                static_cast<float *>(yv)[o] = v[i];
            else
                static_cast<__nv_bfloat16 *>(yv)[o] = __float2bfloat16_rn(v[i]);
        }
    }
}

template <bool F32OUT>
__global__ void __launch_bounds__(kWarps * 32)
gemv_kernel(const uint4 *__restrict__ qw, const uint32_t *__restrict__ sc,
            const uint8_t *__restrict__ zp, const uint32_t *__restrict__ x32,
            void *__restrict__ yv, int M, int K, int N, int T, int S) {
    extern __shared__ __align__(16) uint32_t smem[];
    const int G = K / kGroup;
    const int C = K / kChunkK;
    const int split = blockIdx.y;
    const int g0 = (int)((long long)split * G / S);
    const int g1 = (int)((long long)(split + 1) * G / S);
    const int c0 = 2 * g0;
    const int nch = 2 * (g1 - g0);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gq = lane >> 2, tq = lane & 3;
    const int t = blockIdx.x * kWarps + warp;
    const bool active = t < T;

    // Issue the first weight and group-metadata loads before staging x.
    const uint4 *wp = qw + ((size_t)t * C + c0) * 32 + lane;
    const size_t meta0 = ((size_t)t * G + g0) * 8 + gq;
    uint4 ring[kInFlight];
    uint32_t sring[kInFlight / 2], zring[kInFlight / 2];
#pragma unroll
    for (int i = 0; i < kInFlight / 2; ++i) sring[i] = zring[i] = 0u;
#pragma unroll
    for (int i = 0; i < kInFlight; ++i) {
        ring[i] = make_uint4(0u, 0u, 0u, 0u);
        if (active && i < nch) {
            ring[i] = ld_stream(wp + (size_t)i * 32);
            if ((i & 1) == 0) {
                sring[i / 2] = ld_nc_u32(sc + meta0 + (size_t)(i / 2) * 8);
                zring[i / 2] = ld_nc_u8(zp + meta0 + (size_t)(i / 2) * 8);
            }
        }
    }

    // Stage this block's K slice of x: xs[(piece * M + m) * 4 + tq][8 words].
    uint32_t *xs = smem;
    {
        const int per_row = nch * 32;            // bf16 pairs of one token in the slice
        const size_t row_words = (size_t)K / 2;
        for (int i = threadIdx.x; i < M * per_row; i += kWarps * 32) {
            const int m = i / per_row, r = i - m * per_row;
            const int cl = r >> 5, u = r & 31;
            const int j = u >> 3, o = u & 7;
            const uint32_t v = x32[(size_t)m * row_words + (size_t)(c0 + cl) * 32 + u];
            xs[((cl * M + m) * 4 + (o & 3)) * 8 + 2 * j + (o >> 2)] = v;
        }
    }
    __syncthreads();

    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if (active) {
        const uint32_t *xl = xs + (gq * 4 + tq) * 8;
        const bool has_x = gq < M;
        const int piece_stride = M * 32;
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t czl = 0u, czh = 0u;
        float sl = 0.f, sh = 0.f;
        for (int base = 0; base < nch; base += kInFlight) {
#pragma unroll
            for (int i = 0; i < kInFlight; ++i) {
                const int ci = base + i;
                if (ci < nch) {
                    const uint4 w = ring[i];
                    if ((i & 1) == 0) {
                        const uint32_t zb = zring[i / 2], sp = sring[i / 2];
                        czl = ((zb & 0xFu) | 0x4300u) * 0x10001u;
                        czh = (((zb >> 4) & 0xFu) | 0x4300u) * 0x10001u;
                        sl = __half2float(__ushort_as_half((unsigned short)(sp & 0xFFFFu)));
                        sh = __half2float(__ushort_as_half((unsigned short)(sp >> 16)));
                        d[0] = d[1] = d[2] = d[3] = 0.f;
                    }
                    const int nx = ci + kInFlight;
                    if (nx < nch) {
                        ring[i] = ld_stream(wp + (size_t)nx * 32);
                        if ((i & 1) == 0) {
                            sring[i / 2] = ld_nc_u32(sc + meta0 + (size_t)(nx / 2) * 8);
                            zring[i / 2] = ld_nc_u8(zp + meta0 + (size_t)(nx / 2) * 8);
                        }
                    }
                    uint32_t b[8];
                    if (has_x) {
                        const uint4 *bp = reinterpret_cast<const uint4 *>(xl + ci * piece_stride);
                        const uint4 b0 = bp[0], b1 = bp[1];
                        b[0] = b0.x; b[1] = b0.y; b[2] = b0.z; b[3] = b0.w;
                        b[4] = b1.x; b[5] = b1.y; b[6] = b1.z; b[7] = b1.w;
                    } else {
#pragma unroll
                        for (int q = 0; q < 8; ++q) b[q] = 0u;
                    }
                    piece_mma(d, w, b, czl, czh);
                    if (i & 1) {
                        acc[0] = fmaf(d[0], sl, acc[0]);
                        acc[1] = fmaf(d[1], sl, acc[1]);
                        acc[2] = fmaf(d[2], sh, acc[2]);
                        acc[3] = fmaf(d[3], sh, acc[3]);
                    }
                }
            }
        }
    }

    if (S == 1) {
        if (active) store_tile<F32OUT>(yv, acc, t, lane, M, N);
        return;
    }
    // Combine the K slices of the cluster in rank order 0, 1, ..., S-1.
    float4 *red = reinterpret_cast<float4 *>(reinterpret_cast<char *>(smem) +
                                             (size_t)(2 * ((G + S - 1) / S)) * M * 128);
    red[warp * 32 + lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    if (active && (warp % S) == split) {
        float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
        for (int r = 0; r < S; ++r) {
            const float4 v = *cluster.map_shared_rank(&red[warp * 32 + lane], r);
            s0 += v.x; s1 += v.y; s2 += v.z; s3 += v.w;
        }
        const float tot[4] = {s0, s1, s2, s3};
        store_tile<F32OUT>(yv, tot, t, lane, M, N);
    }
    cluster.sync();
}

size_t x_bytes(int K, int S, int M) {
    const int G = K / kGroup;
    return (size_t)2 * ((G + S - 1) / S) * M * 128;
}

size_t smem_bytes(int K, int S, int M) {
    return x_bytes(K, S, M) + (S > 1 ? (size_t)kWarps * 32 * sizeof(float4) : 0);
}

}  // namespace

bool gemv_shape(int K, int N, int num_sms, GemvShape *out) {
    const int T = row_tiles(N);
    const int G = K / kGroup;
    const int blocks_n = (T + kWarps - 1) / kWarps;
    const long long slots = 2LL * (num_sms > 0 ? num_sms : 1);
    int best_s = 0;
    long long best_cost = 0;
    for (int S = 1; S <= kMaxSplits && S <= G; ++S) {
        if (x_bytes(K, S, W4_MAX_TOKENS) > kMaxXBytes) continue;
        const long long ctas = (long long)blocks_n * S;
        const long long waves = (ctas + slots - 1) / slots;
        const long long cost = waves * ((G + S - 1) / S);
        if (best_s == 0 || cost < best_cost) {
            best_s = S;
            best_cost = cost;
        }
    }
    if (best_s == 0) return false;
    out->warps = kWarps;
    out->splits = best_s;
    return true;
}

cudaError_t launch_gemv(const void *qweight, const void *scales, const void *zeros,
                        const uint16_t *x, void *y, bool f32_out, int M, int K, int N,
                        const GemvShape &shape, cudaStream_t stream) {
    const int T = row_tiles(N);
    const int S = shape.splits;
    const size_t smem = smem_bytes(K, S, M);
    static bool attr_done[2][64] = {};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    auto kern = f32_out ? gemv_kernel<true> : gemv_kernel<false>;
    if (dev < 64 && !attr_done[f32_out][dev]) {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)(kMaxXBytes + kWarps * 32 * sizeof(float4)));
        if (err != cudaSuccess) return err;
        attr_done[f32_out][dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((T + kWarps - 1) / kWarps), (unsigned)S, 1);
    cfg.blockDim = dim3(kWarps * 32, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = (unsigned)S;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = S > 1 ? 1 : 0;
    const uint4 *qw = reinterpret_cast<const uint4 *>(static_cast<const char *>(qweight) +
                                                      W4_HEADER_BYTES);
    return cudaLaunchKernelEx(&cfg, kern, qw, static_cast<const uint32_t *>(scales),
                              static_cast<const uint8_t *>(zeros),
                              reinterpret_cast<const uint32_t *>(x), y, M, K, N, T, S);
}

}  // namespace w4
