// C ABI of libw4 (declared in include/w4.h): argument checks on the host,
// then the launches.  Nothing here allocates device or pinned memory.
#include <string.h>

#include <atomic>

#include "w4_internal.cuh"

namespace {

bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

bool valid_kn(int K, int N) { return K > 0 && K % w4::kGroup == 0 && N > 0; }

w4_status cuda_status(cudaError_t e) { return e == cudaSuccess ? W4_OK : W4_ERR_CUDA; }

// SM count of the current device, cached per device.  The cache entries are
// atomic: host threads that race on a first call both read the attribute and
// store the same value.
int device_sms() {
    static std::atomic<int> cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (dev >= 0 && dev < 64) {
        const int c = cached[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return -1;
    if (dev >= 0 && dev < 64) cached[dev].store(sms, std::memory_order_relaxed);
    return sms;
}

w4_status gemv_common(const void *qweight, const void *scales, const void *zeros,
                      const uint16_t *x, void *y, bool f32_out, int M, int K, int N,
                      w4_stream_t stream) {
    if (!qweight || !scales || !zeros || !x || !y) return W4_ERR_INVALID_ARG;
    if (!valid_kn(K, N)) return W4_ERR_INVALID_ARG;
    if (M < 1 || M > W4_MAX_TOKENS) return W4_ERR_UNSUPPORTED;
    if (!aligned(qweight, 16) || !aligned(scales, 16) || !aligned(zeros, 16) ||
        !aligned(x, 16) || !aligned(y, f32_out ? 4 : 2))
        return W4_ERR_INVALID_ARG;
    const int sms = device_sms();
    if (sms <= 0) return W4_ERR_CUDA;
    w4::GemvShape shape;
    if (!w4::gemv_shape(K, N, sms, &shape)) return W4_ERR_UNSUPPORTED;
    return cuda_status(w4::launch_gemv(qweight, scales, zeros, x, y, f32_out, M, K, N, shape, 0,
                                       sms, reinterpret_cast<cudaStream_t>(stream)));
}

w4_status repack_common(const uint32_t *qweight, const uint16_t *scales, const uint8_t *zeros,
                        int K, int N, int swiglu_I, void *qweight_out, void *scales_out,
                        void *zeros_out, w4_stream_t stream) {
    if (!qweight || !scales || !zeros || !qweight_out || !scales_out || !zeros_out)
        return W4_ERR_INVALID_ARG;
    if (!valid_kn(K, N)) return W4_ERR_INVALID_ARG;
    if (!aligned(qweight, 4) || !aligned(scales, 2) || !aligned(qweight_out, 16) ||
        !aligned(scales_out, 16) || !aligned(zeros_out, 16))
        return W4_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) return W4_ERR_CUDA;
    if (cap != cudaStreamCaptureStatusNone) return W4_ERR_UNSUPPORTED;
    cudaError_t e = w4::launch_repack(qweight, scales, zeros, K, N, swiglu_I, qweight_out,
                                      scales_out, zeros_out, s);
    if (e != cudaSuccess) return W4_ERR_CUDA;
    w4::Header h;
    e = cudaMemcpyAsync(&h, qweight_out, sizeof h, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return W4_ERR_CUDA;
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return W4_ERR_CUDA;
    return h.bad_zeros ? W4_ERR_INVALID_ARG : W4_OK;
}

w4_status check_header_common(const void *header, int K, int N, uint32_t layout_id) {
    if (!header) return W4_ERR_INVALID_ARG;
    w4::Header h;
    memcpy(&h, header, sizeof h);
    if (memcmp(h.magic, "W4G128KL", 8) != 0 || h.layout_id != layout_id ||
        h.version != W4_LAYOUT_VERSION || h.K != K || h.N != N || h.bad_zeros != 0)
        return W4_ERR_LAYOUT;
    if (h.kernel_error != 0) return W4_ERR_CUDA;
    return W4_OK;
}

// Up to 16 tokens: the GEMV in passes of 8 tokens (one or two passes over
// the weight; each row bit-identical to the single-token GEMV).  More: one
// pass over the weight on the tensor cores (w4_gemm_tc.cu), in tiles of 128
// tokens.  Measured on the 7B shapes: two passes for 16 tokens against the
// tensor cores for 17, gate_up 32.0 vs 44.0 us, qkv 9.5 vs 10.4, down 24.6 vs
// 24.3 (even); a third pass (17-24 tokens) would cost about 47, 14 and 37 us.
constexpr int kGemmPassMaxTokens = 2 * W4_MAX_TOKENS;

w4_status gemm_common(const void *qweight, const void *scales, const void *zeros,
                      const uint16_t *x, void *y, bool f32_out, int M, int K, int N,
                      w4_stream_t stream) {
    if (M < 1) return W4_ERR_UNSUPPORTED;
    if (!valid_kn(K, N)) return W4_ERR_INVALID_ARG;
    if (M <= kGemmPassMaxTokens) {
        const size_t ybytes = f32_out ? 4 : 2;
        for (int m0 = 0; m0 < M; m0 += W4_MAX_TOKENS) {
            const int mp = M - m0 < W4_MAX_TOKENS ? M - m0 : W4_MAX_TOKENS;
            const w4_status st = gemv_common(
                qweight, scales, zeros, x ? x + (size_t)m0 * K : x,
                y ? static_cast<char *>(y) + (size_t)m0 * N * ybytes : y, f32_out, mp, K, N,
                stream);
            if (st != W4_OK) return st;
        }
        return W4_OK;
    }
    if (!qweight || !scales || !zeros || !x || !y) return W4_ERR_INVALID_ARG;
    if (!aligned(qweight, 16) || !aligned(scales, 16) || !aligned(zeros, 16) ||
        !aligned(x, 16) || !aligned(y, f32_out ? 4 : 2))
        return W4_ERR_INVALID_ARG;
    // tensor-copy coordinates are 32-bit: x rows, and the weight records seen
    // as 128-byte rows (64 per record)
    if ((long long)M * K >= (1LL << 40) || (M + 127) / 128 > 65535 ||
        (long long)w4::row_blocks(N) * (K / 128) * 64 >= (1LL << 31))
        return W4_ERR_UNSUPPORTED;
    const int sms = device_sms();
    if (sms <= 0) return W4_ERR_CUDA;
    return cuda_status(w4::launch_gemm_tc(qweight, scales, zeros, x, y, f32_out, M, K, N, sms,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

w4_status gemv_swiglu_common(const void *qweight, const void *scales, const void *zeros,
                             const uint16_t *x, void *y, bool f32_out, int M, int K, int I,
                             w4_stream_t stream) {
    if (!qweight || !scales || !zeros || !x || !y) return W4_ERR_INVALID_ARG;
    if (!valid_kn(K, I)) return W4_ERR_INVALID_ARG;
    if (M < 1 || M > W4_MAX_TOKENS) return W4_ERR_UNSUPPORTED;
    if (!aligned(qweight, 16) || !aligned(scales, 16) || !aligned(zeros, 16) ||
        !aligned(x, 16) || !aligned(y, f32_out ? 4 : 2))
        return W4_ERR_INVALID_ARG;
    const int sms = device_sms();
    if (sms <= 0) return W4_ERR_CUDA;
    const int rows = w4::swiglu_rows(I);
    w4::GemvShape shape;
    if (!w4::gemv_shape(K, rows, sms, &shape)) return W4_ERR_UNSUPPORTED;
    return cuda_status(w4::launch_gemv(qweight, scales, zeros, x, y, f32_out, M, K, rows, shape,
                                       I, sms, reinterpret_cast<cudaStream_t>(stream)));
}

w4_status gemv_ws_common(const void *qweight, const void *scales, const void *zeros,
                         const uint16_t *x, void *y, bool f32_out, int M, int K, int N,
                         void *workspace, size_t workspace_bytes, w4_stream_t stream) {
    if (!qweight || !scales || !zeros || !x || !y || !workspace) return W4_ERR_INVALID_ARG;
    if (!valid_kn(K, N)) return W4_ERR_INVALID_ARG;
    if (M < 1 || M > W4_MAX_TOKENS) return W4_ERR_UNSUPPORTED;
    if (!aligned(qweight, 16) || !aligned(scales, 16) || !aligned(zeros, 16) ||
        !aligned(x, 16) || !aligned(y, f32_out ? 4 : 2) || !aligned(workspace, 256))
        return W4_ERR_INVALID_ARG;
    const int sms = device_sms();
    if (sms <= 0) return W4_ERR_CUDA;
    if (workspace_bytes < w4::gemv_ws_bytes(K, N, sms)) return W4_ERR_INVALID_ARG;
    return cuda_status(w4::launch_gemv_ws(qweight, scales, zeros, x, y, f32_out, M, K, N,
                                          workspace, sms, reinterpret_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

const char *w4_status_string(w4_status status) {
    switch (status) {
        case W4_OK: return "W4_OK";
        case W4_ERR_INVALID_ARG: return "W4_ERR_INVALID_ARG";
        case W4_ERR_UNSUPPORTED: return "W4_ERR_UNSUPPORTED";
        case W4_ERR_LAYOUT: return "W4_ERR_LAYOUT";
        case W4_ERR_CUDA: return "W4_ERR_CUDA";
        case W4_ERR_SCRATCH_LIMIT: return "W4_ERR_SCRATCH_LIMIT";
    }
    return "W4_ERR_UNKNOWN";
}

int w4_version(void) { return 10000; }

w4_status w4_repacked_sizes(int K, int N, size_t *qweight_bytes, size_t *scales_bytes,
                            size_t *zeros_bytes) {
    if (!valid_kn(K, N) || !qweight_bytes || !scales_bytes || !zeros_bytes)
        return W4_ERR_INVALID_ARG;
    *qweight_bytes = w4::packed_qweight_bytes(K, N);
    *scales_bytes = w4::packed_scales_bytes(K, N);
    *zeros_bytes = w4::packed_zeros_bytes(K, N);
    return W4_OK;
}

w4_status w4_repack(const uint32_t *qweight, const uint16_t *scales, const uint8_t *zeros, int K,
                    int N, void *qweight_out, void *scales_out, void *zeros_out,
                    w4_stream_t stream) {
    return repack_common(qweight, scales, zeros, K, N, 0, qweight_out, scales_out, zeros_out,
                         stream);
}

w4_status w4_check_header(const void *header, int K, int N) {
    return check_header_common(header, K, N, W4_LAYOUT_ID);
}

w4_status w4_repacked_sizes_swiglu(int K, int I, size_t *qweight_bytes, size_t *scales_bytes,
                                   size_t *zeros_bytes) {
    if (!valid_kn(K, I) || I > (1 << 29)) return W4_ERR_INVALID_ARG;
    return w4_repacked_sizes(K, w4::swiglu_rows(I), qweight_bytes, scales_bytes, zeros_bytes);
}

w4_status w4_repack_swiglu(const uint32_t *qweight, const uint16_t *scales, const uint8_t *zeros,
                           int K, int I, void *qweight_out, void *scales_out, void *zeros_out,
                           w4_stream_t stream) {
    if (!valid_kn(K, I) || I > (1 << 29)) return W4_ERR_INVALID_ARG;
    return repack_common(qweight, scales, zeros, K, w4::swiglu_rows(I), I, qweight_out,
                         scales_out, zeros_out, stream);
}

w4_status w4_check_header_swiglu(const void *header, int K, int I) {
    return check_header_common(header, K, I, W4_LAYOUT_ID_SWIGLU);
}

w4_status w4_gemv_swiglu(const void *qweight, const void *scales, const void *zeros,
                         const uint16_t *x, uint16_t *y, int M, int K, int I,
                         w4_stream_t stream) {
    return gemv_swiglu_common(qweight, scales, zeros, x, y, false, M, K, I, stream);
}

w4_status w4_gemv_swiglu_f32(const void *qweight, const void *scales, const void *zeros,
                             const uint16_t *x, float *y, int M, int K, int I,
                             w4_stream_t stream) {
    return gemv_swiglu_common(qweight, scales, zeros, x, y, true, M, K, I, stream);
}

w4_status w4_dequant(const uint32_t *qweight, const uint16_t *scales, const uint8_t *zeros, int K,
                     int N, uint16_t *w_out, w4_stream_t stream) {
    if (!qweight || !scales || !zeros || !w_out) return W4_ERR_INVALID_ARG;
    if (!valid_kn(K, N)) return W4_ERR_INVALID_ARG;
    if (!aligned(qweight, 16) || !aligned(scales, 2) || !aligned(w_out, 16))
        return W4_ERR_INVALID_ARG;
    return cuda_status(w4::launch_dequant(qweight, scales, zeros, K, N, w_out,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

w4_status w4_gemv(const void *qweight, const void *scales, const void *zeros, const uint16_t *x,
                  uint16_t *y, int M, int K, int N, w4_stream_t stream) {
    return gemv_common(qweight, scales, zeros, x, y, false, M, K, N, stream);
}

w4_status w4_gemv_f32(const void *qweight, const void *scales, const void *zeros,
                      const uint16_t *x, float *y, int M, int K, int N, w4_stream_t stream) {
    return gemv_common(qweight, scales, zeros, x, y, true, M, K, N, stream);
}

w4_status w4_gemm(const void *qweight, const void *scales, const void *zeros, const uint16_t *x,
                  uint16_t *y, int M, int K, int N, w4_stream_t stream) {
    return gemm_common(qweight, scales, zeros, x, y, false, M, K, N, stream);
}

w4_status w4_gemm_f32(const void *qweight, const void *scales, const void *zeros,
                      const uint16_t *x, float *y, int M, int K, int N, w4_stream_t stream) {
    return gemm_common(qweight, scales, zeros, x, y, true, M, K, N, stream);
}

w4_status w4_gemv_workspace_bytes(int K, int N, size_t *bytes) {
    if (!valid_kn(K, N) || !bytes) return W4_ERR_INVALID_ARG;
    const int sms = device_sms();
    if (sms <= 0) return W4_ERR_CUDA;
    *bytes = w4::gemv_ws_bytes(K, N, sms);
    return W4_OK;
}

w4_status w4_gemv_ws(const void *qweight, const void *scales, const void *zeros,
                     const uint16_t *x, uint16_t *y, int M, int K, int N, void *workspace,
                     size_t workspace_bytes, w4_stream_t stream) {
    return gemv_ws_common(qweight, scales, zeros, x, y, false, M, K, N, workspace,
                          workspace_bytes, stream);
}

w4_status w4_gemv_ws_f32(const void *qweight, const void *scales, const void *zeros,
                         const uint16_t *x, float *y, int M, int K, int N, void *workspace,
                         size_t workspace_bytes, w4_stream_t stream) {
    return gemv_ws_common(qweight, scales, zeros, x, y, true, M, K, N, workspace,
                          workspace_bytes, stream);
}

w4_status w4_quantize(const uint16_t *w, int K, int N, int mode, uint32_t *qweight,
                      uint16_t *scales, uint8_t *zeros, w4_stream_t stream) {
    if (!w || !qweight || !scales || !zeros) return W4_ERR_INVALID_ARG;
    if (!valid_kn(K, N)) return W4_ERR_INVALID_ARG;
    if (mode != W4_QUANT_ASYMMETRIC && mode != W4_QUANT_SYMMETRIC) return W4_ERR_INVALID_ARG;
    if (!aligned(w, 16) || !aligned(qweight, 4) || !aligned(scales, 2))
        return W4_ERR_INVALID_ARG;
    const int sms = device_sms();
    if (sms <= 0) return W4_ERR_CUDA;
    return cuda_status(w4::launch_quantize(w, K, N, mode == W4_QUANT_SYMMETRIC, qweight, scales,
                                           zeros, sms, reinterpret_cast<cudaStream_t>(stream)));
}

w4_status w4_gemv_config(int K, int N, int *tiles_per_block, int *k_splits,
                         int *zero_point_folded) {
    if (!valid_kn(K, N)) return W4_ERR_INVALID_ARG;
    const int sms = device_sms();
    if (sms <= 0) return W4_ERR_CUDA;
    w4::GemvShape shape;
    if (!w4::gemv_shape(K, N, sms, &shape)) return W4_ERR_UNSUPPORTED;
    if (tiles_per_block) *tiles_per_block = shape.warps;
    if (k_splits) *k_splits = shape.splits;
    if (zero_point_folded) *zero_point_folded = shape.fold ? 1 : 0;
    return W4_OK;
}

w4_status w4_gemv_plan(int M, int K, int N, w4_gemv_launch_info *info) {
    if (!valid_kn(K, N) || !info) return W4_ERR_INVALID_ARG;
    if (M < 1 || M > W4_MAX_TOKENS) return W4_ERR_UNSUPPORTED;
    const int sms = device_sms();
    if (sms <= 0) return W4_ERR_CUDA;
    w4::GemvShape shape;
    if (!w4::gemv_shape(K, N, sms, &shape)) return W4_ERR_UNSUPPORTED;
    w4::GemvLaunch L;
    if (w4::plan_gemv(false, M, K, N, shape, sms, &L) != cudaSuccess) return W4_ERR_CUDA;
    memset(info, 0, sizeof *info);
    info->k_splits = shape.splits;
    info->zero_point_folded = shape.fold ? 1 : 0;
    info->grid_x = (int)L.grid.x;
    info->grid_y = (int)L.grid.y;
    info->persistent = L.persistent ? 1 : 0;
    info->overlap = L.overlap ? 1 : 0;
    info->capped = L.capped ? 1 : 0;
    info->ring_stages = L.stages;
    info->wide_prologue = L.arith == 2 ? 1 : 0;
    info->blocks_per_sm_max = L.variant == 0 ? 2 : 3;
    info->smem_bytes = L.smem_bytes;
    return W4_OK;
}

}  // extern "C"
