// w4_stream_read: the read bandwidth this GPU delivers to a kernel that only
// reads, measured with the GEMV kernels' own streaming method ("qengine",
// section "Learnings": the roofline a decode kernel is judged against should
// come from a plain read benchmark on the same GPU, not from the data sheet
// or from a copy, which also writes).
//
// Mode 0 (bulk-copy ring): each block streams a contiguous share of the
// buffer in 8 KB records through a ring of shared-memory stages, one producer
// lane issuing cp.async.bulk copies (completion counted in bytes on the
// stage's mbarrier) and one consumer warp releasing each stage after touching
// one word per lane -- the GEMV's weight path without its arithmetic.
// Mode 1 (128-bit loads): every thread reads 16-byte words with streaming
// loads in a grid-stride loop.  Both fold what they read into one word
// (xor), so nothing can be optimised away.
#include "w4_device.cuh"

namespace w4 {
namespace {

constexpr int kSrRecord = 8192;
constexpr int kSrStages = 12;
constexpr int kSrThreads = 64;   // warp 0: producer (lane 0); warp 1: consumer

__global__ void __launch_bounds__(kSrThreads, 2)
stream_read_ring(const char *__restrict__ src, size_t records, uint32_t *out) {
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kSrStages * kSrRecord);
    uint64_t *empty = full + kSrStages;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kSrStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const size_t r0 = (size_t)blockIdx.x * records / gridDim.x;
    const size_t r1 = (size_t)(blockIdx.x + 1) * records / gridDim.x;
    uint32_t acc = 0;
    bool ok = true;
    if (warp == 0) {
        if (lane == 0) {
            size_t issued = 0;
            for (size_t r = r0; r < r1 && ok; ++r, ++issued) {
                const int s = (int)(issued % kSrStages);
                const uint32_t round = (uint32_t)(issued / kSrStages);
                if (round > 0) {
                    if (!mbar_wait(&empty[s], (round - 1) & 1u)) {
                        ok = false;
                        break;
                    }
                    fence_proxy_async();
                }
                mbar_expect_tx(&full[s], kSrRecord);
                bulk_g2s(smem + s * kSrRecord, src + r * kSrRecord, kSrRecord, &full[s]);
            }
            // let the copies still in flight land (bounded) before exit
            for (size_t q = issued > kSrStages ? issued - kSrStages : 0; q < issued; ++q)
                mbar_wait(&full[q % kSrStages], (uint32_t)((q / kSrStages) & 1));
        }
    } else {
        size_t n = 0;
        for (size_t r = r0; r < r1; ++r, ++n) {
            const int s = (int)(n % kSrStages);
            if (!__all_sync(0xFFFFFFFFu, mbar_wait(&full[s], (uint32_t)((n / kSrStages) & 1)))) {
                ok = false;
                break;
            }
            acc ^= reinterpret_cast<const uint32_t *>(smem + s * kSrRecord)[lane * 64];
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
        for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(0xFFFFFFFFu, acc, o);
    }
    if (threadIdx.x == 32) atomicXor(out, acc);
    if (!ok) atomicOr(out + 1, 1u);
}

__global__ void __launch_bounds__(512) stream_read_ld128(const uint4 *__restrict__ src, size_t n16,
                                                        uint32_t *out) {
    uint32_t acc = 0;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < n16; i += 4 * stride) {
        const uint4 a = __ldcs(src + i), b = __ldcs(src + i + stride);
        const uint4 c = __ldcs(src + i + 2 * stride), d = __ldcs(src + i + 3 * stride);
        acc ^= a.x ^ b.y ^ c.z ^ d.w;
    }
    for (; i < n16; i += stride) acc ^= __ldcs(src + i).x;
    for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(0xFFFFFFFFu, acc, o);
    if ((threadIdx.x & 31) == 0) atomicXor(out, acc);
}

}  // namespace
}  // namespace w4

extern "C" w4_status w4_stream_read(const void *src, size_t bytes, int mode, uint32_t *out,
                                    w4_stream_t stream) {
    if (!src || !out || (uintptr_t)src % 16 != 0 || (uintptr_t)out % 4 != 0 || bytes == 0)
        return W4_ERR_INVALID_ARG;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms <= 0)
        return W4_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (mode == W4_STREAM_READ_RING) {
        if (bytes % w4::kSrRecord != 0) return W4_ERR_INVALID_ARG;
        const size_t smem = (size_t)w4::kSrStages * (w4::kSrRecord + 16);
        if (cudaFuncSetAttribute(w4::stream_read_ring, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem) != cudaSuccess)
            return W4_ERR_CUDA;
        w4::stream_read_ring<<<2 * sms, w4::kSrThreads, smem, s>>>(
            static_cast<const char *>(src), bytes / w4::kSrRecord, out);
    } else if (mode == W4_STREAM_READ_LD128) {
        if (bytes % 16 != 0) return W4_ERR_INVALID_ARG;
        w4::stream_read_ld128<<<4 * sms, 512, 0, s>>>(static_cast<const uint4 *>(src), bytes / 16,
                                                       out);
    } else {
        return W4_ERR_INVALID_ARG;
    }
    return cudaGetLastError() == cudaSuccess ? W4_OK : W4_ERR_CUDA;
}
