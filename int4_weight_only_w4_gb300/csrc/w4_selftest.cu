// w4_selftest_bounded_wait: the bounded mbarrier wait of the GEMV kernels
// (mbar_wait in w4_device.cuh) run against a barrier that nothing completes.
// The wait must give up after its limit and report it, without faulting or
// hanging the GPU.
#include "w4_device.cuh"

namespace w4 {
namespace {

__global__ void bounded_wait_kernel(uint32_t *status) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);               // one arrival expected; none ever comes
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0) *status = mbar_wait(&bar, 0) ? 0u : 1u;
}

}  // namespace
}  // namespace w4

extern "C" w4_status w4_selftest_bounded_wait(uint32_t *status, w4_stream_t stream) {
    if (!status || (uintptr_t)status % 4 != 0) return W4_ERR_INVALID_ARG;
    w4::bounded_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(status);
    return cudaGetLastError() == cudaSuccess ? W4_OK : W4_ERR_CUDA;
}
