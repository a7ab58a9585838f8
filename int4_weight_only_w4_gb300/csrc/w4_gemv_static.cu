// w4_gemv_ws_static: the workspace-split GEMV (w4_gemv_sk.cu) with its scratch
// in a static device array, for callers that cannot allocate device memory.
// Nothing here allocates: the array is part of the library's device image and
// exists on a GPU from the moment the library's code is loaded there.
#include <mutex>

#include "w4_internal.cuh"

namespace {

// The scratch: row-block counters (zeroed by each call before the launch),
// then the partial-sum slots.  In host code `g_scratch` is the runtime's
// host-side stand-in for the array, not a device address; the device address
// comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_scratch[W4_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_device[kMaxDevices] = {};

// Device address of g_scratch on device `dev` (the current device), looked
// up once per device.
cudaError_t scratch_on(int dev, void **out) {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_device[dev] == nullptr) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_device[dev] = p;
    }
    *out = g_scratch_device[dev];
    return cudaSuccess;
}

bool aligned_to(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

}  // namespace

extern "C" w4_status w4_gemv_ws_static(const void *qweight, const void *scales,
                                       const void *zeros, const uint16_t *x, uint16_t *y,
                                       int M, int K, int N, w4_stream_t stream) {
    if (K <= 0 || K % w4::kGroup != 0 || N <= 0) return W4_ERR_INVALID_ARG;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return W4_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return W4_ERR_UNSUPPORTED;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms <= 0)
        return W4_ERR_CUDA;
    // The size limit is checked first, so that a product too large for the
    // array is refused whatever else is wrong with the call.
    if (w4::gemv_ws_bytes(K, N, sms) > (size_t)W4_STATIC_SCRATCH_BYTES)
        return W4_ERR_SCRATCH_LIMIT;
    if (!qweight || !scales || !zeros || !x || !y) return W4_ERR_INVALID_ARG;
    if (M < 1 || M > W4_MAX_TOKENS) return W4_ERR_UNSUPPORTED;
    if (!aligned_to(qweight, 16) || !aligned_to(scales, 16) || !aligned_to(zeros, 16) ||
        !aligned_to(x, 16) || !aligned_to(y, 2))
        return W4_ERR_INVALID_ARG;
    void *scratch = nullptr;
    if (scratch_on(dev, &scratch) != cudaSuccess) return W4_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // The counters must start at zero; a completed call leaves them so, but a
    // call that failed may not have.
    const size_t counter_bytes = ((size_t)w4::row_blocks(N) * 4 + 255) / 256 * 256;
    if (cudaMemsetAsync(scratch, 0, counter_bytes, s) != cudaSuccess) return W4_ERR_CUDA;
    const cudaError_t e =
        w4::launch_gemv_ws(qweight, scales, zeros, x, y, false, M, K, N, scratch, sms, s);
    return e == cudaSuccess ? W4_OK : W4_ERR_CUDA;
}
