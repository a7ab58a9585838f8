// w4_quantize: binary16 W -> canonical (q, s, z), one group of 128 weights of
// one row at a time (the grouping of the matrix-vector product).
//
// Rule (fp32 from the exact binary16 values, every operation rounded to
// nearest, ties to even; the codes are taken against the stored fp16 scale):
//   asymmetric: lo = min(0, min w), hi = max(0, max w), s = fp16((hi - lo) / 15),
//               z = clamp(rint(-lo / s), 0, 15), q = clamp(rint(w / s) + z, 0, 15)
//   symmetric:  s = fp16(max |w| / 7), z = 8, q = clamp(rint(w / s), -8, 7) + 8
//               (scale = absmax / 7: "Building an LLM Inference Runtime ...",
//               section "The Stack Architecture: A One-Page Overview"; values
//               in [-8, 7]: "CodeAlign-Runtime", section "Level 3 -- INT4
//               Quantization + Fused Kernel")
// A group whose scale rounds to 0 stores s = 0 and q = z.
//
// The rows are contiguous, so group t = n * G + g is the 256 bytes at
// w + 128 t and owns qweight words 16 t .. 16 t + 15, scales[t], zeros[t]:
// the work is a one-dimensional stream over N * G groups.  Sixteen lanes take
// one group: each loads 16 bytes (eight weights) and produces one packed
// word, the group's range comes from a 16-lane shuffle reduction, and every
// lane derives the same scale and zero point from it.  Each warp keeps
// several groups' loads in flight; the grid covers every SM.
//
// rint(w / s) without a division per weight: t = w * rcp(s), with rcp(s) and
// the product each rounded to nearest, is within |w/s| * 2^-22.4 of the
// correctly rounded quotient the rule asks for, so the two round to different
// integers only if t lies within that distance of a half-integer.  Where t is
// within T * 2^-21 of one (T = the group's largest |w| times rcp(s), rounded
// the same way, so T >= |t|), the quotient is taken with the correctly
// rounded division instead; elsewhere rint(t) is the rule's value.  rint(t)
// comes from one addition: t + 1.5 * 2^23 rounds to nearest (ties to even)
// at unit spacing for |t| < 2^22 (here |t| <= 32), so its low bits are
// rint(t) as an integer and subtracting 1.5 * 2^23 again gives it exactly as
// a float.
#include <cuda_fp16.h>

#include "w4_internal.cuh"

namespace w4 {
namespace {

constexpr int kQuantThreads = 256;
constexpr int kQuantUnroll = 4;          // group pairs per warp in flight

__device__ __forceinline__ float clampf(float v, float a, float b) {
    return fminf(fmaxf(v, a), b);
}

// rint(x / s) as an integer, with r = rcp_rn(s) and tol = T * 2^-21 (see above).
__device__ __forceinline__ int rint_div(float x, float s, float r, float tol) {
    constexpr float kMagic = 12582912.f;                // 1.5 * 2^23
    const float t = __fmul_rn(x, r);
    const float y = __fadd_rn(t, kMagic);
    const float n = __fsub_rn(y, kMagic);
    // distance from t to the nearest half-integer is 0.5 - |t - n|
    if (0.5f - fabsf(t - n) <= tol) return (int)rintf(__fdiv_rn(x, s));
    return (int)(__float_as_uint(y) - __float_as_uint(kMagic));
}

template <bool SYMMETRIC>
__global__ void __launch_bounds__(kQuantThreads)
quantize_kernel(const uint4 *__restrict__ w, long long groups,
                uint32_t *__restrict__ qweight, __half *__restrict__ scales,
                uint8_t *__restrict__ zeros) {
    constexpr bool symmetric = SYMMETRIC;
    const int lane = threadIdx.x & 31;
    const int sub = lane & 15;                          // 16-byte piece of the group
    const long long warp = ((long long)blockIdx.x * kQuantThreads + threadIdx.x) >> 5;
    const long long warps = ((long long)gridDim.x * kQuantThreads) >> 5;
    // warp w handles group pairs p = w, w + warps, ...; lanes 0-15 take group
    // 2p, lanes 16-31 group 2p + 1
    for (long long p0 = warp; 2 * p0 < groups; p0 += warps * kQuantUnroll) {
        uint4 v[kQuantUnroll];
#pragma unroll
        for (int u = 0; u < kQuantUnroll; ++u) {
            const long long t = 2 * (p0 + u * warps) + (lane >> 4);
            v[u] = t < groups ? __ldcs(&w[t * 16 + sub]) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kQuantUnroll; ++u) {
            const long long t = 2 * (p0 + u * warps) + (lane >> 4);
            // every lane of the warp takes part in the shuffles below
            const uint32_t words[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
            float x[8];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                x[2 * j] = __half2float(__ushort_as_half((unsigned short)(words[j] & 0xFFFFu)));
                x[2 * j + 1] = __half2float(__ushort_as_half((unsigned short)(words[j] >> 16)));
            }
            float lo = 0.f, hi = 0.f, amax = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if constexpr (SYMMETRIC) {
                    amax = fmaxf(amax, fabsf(x[j]));
                } else {
                    lo = fminf(lo, x[j]);
                    hi = fmaxf(hi, x[j]);
                }
            }
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) {
                if constexpr (SYMMETRIC) {
                    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
                } else {
                    lo = fminf(lo, __shfl_xor_sync(0xFFFFFFFFu, lo, o));
                    hi = fmaxf(hi, __shfl_xor_sync(0xFFFFFFFFu, hi, o));
                }
            }
            const float s32 = symmetric ? __fdiv_rn(amax, 7.f) : __fdiv_rn(__fsub_rn(hi, lo), 15.f);
            const __half sh = __float2half_rn(s32);
            const float s = __half2float(sh);
            const float r = s == 0.f ? 0.f : __frcp_rn(s);
            // T * 2^-21 with T = rcp(s) times the largest |w| (rounded as t is)
            const float tol =
                __fmul_rn(symmetric ? amax : fmaxf(-lo, hi), r) * 0x1p-21f;
            float z;
            if (s == 0.f)
                z = symmetric ? 8.f : 0.f;
            else
                z = symmetric ? 8.f : clampf(rintf(__fdiv_rn(-lo, s)), 0.f, 15.f);
            const int zi = (int)z;
            uint32_t word = 0u;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                int q;
                if (s == 0.f) {
                    q = zi;
                } else {
                    const int c = rint_div(x[j], s, r, tol);
                    q = symmetric ? min(max(c, -8), 7) + 8
                                  : min(max(min(max(c, -16), 16) + zi, 0), 15);
                }
                word |= (uint32_t)q << (4 * j);
            }
            if (t < groups) {
                __stcs(&qweight[t * 16 + sub], word);
                if (sub == 0) {
                    scales[t] = sh;
                    zeros[t] = (uint8_t)z;
                }
            }
        }
    }
}

}  // namespace

cudaError_t launch_quantize(const uint16_t *w, int K, int N, bool symmetric, uint32_t *qweight,
                            uint16_t *scales, uint8_t *zeros, int num_sms, cudaStream_t stream) {
    const long long groups = (long long)N * (K / kGroup);
    const long long pairs = (groups + 1) / 2;
    const long long warps_needed = (pairs + kQuantUnroll - 1) / kQuantUnroll;
    const long long blocks_needed = (warps_needed * 32 + kQuantThreads - 1) / kQuantThreads;
    // eight 256-thread blocks per SM fill it; never more blocks than work
    const long long cap = 8LL * (num_sms > 0 ? num_sms : 1);
    const int grid = (int)(blocks_needed < cap ? blocks_needed : cap);
    if (symmetric)
        quantize_kernel<true><<<grid, kQuantThreads, 0, stream>>>(
            reinterpret_cast<const uint4 *>(w), groups, qweight,
            reinterpret_cast<__half *>(scales), zeros);
    else
        quantize_kernel<false><<<grid, kQuantThreads, 0, stream>>>(
            reinterpret_cast<const uint4 *>(w), groups, qweight,
            reinterpret_cast<__half *>(scales), zeros);
    return cudaGetLastError();
}

}  // namespace w4
