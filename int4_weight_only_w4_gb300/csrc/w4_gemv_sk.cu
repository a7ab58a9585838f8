// w4_gemv_ws: the W4 GEMV as an even split of the whole product over a
// persistent grid, with a caller-provided workspace ("stream-K" split).
//
// Units of work are (row block, group) records (w4_repack.cu), numbered
// u = row_block * G + group, which is also their order in memory.  The grid
// is P = min(units, 3 * SMs) blocks; block c streams the contiguous units
// [c*W/P, (c+1)*W/P) (W = all units) through the same producer / consumer
// ring as w4_gemv, with the group's slice of x (256 bytes per token) copied
// into each stage next to the weights.  So every block does the same amount of
// work, all blocks are resident at once (three per SM), and there is no
// cluster and no tail wave.
//
// A row block whose units all fall in one block's range is stored directly.
// A row block cut between consecutive blocks is combined deterministically:
// each contributing block writes its fp32 partial (4 KB) into its own slot of
// the workspace, makes it visible (__threadfence) and increments the row
// block's counter; the block that brings the counter to the number of
// contributors adds all partials in block order, stores the result and
// resets the counter to zero.  Nobody waits for anybody, and no float
// atomics are used ("qengine", section "Learnings": a fixed summation order
// made results bit-identical).  The split depends only on K, N and the SM
// count, never on M, so the result for a token does not depend on M.
//
// Workspace (device, 256-byte aligned, zero-filled before its first use): NB
// counters (uint32, padded to 256 bytes), which every completed call leaves at
// zero, then 2 * P partial slots of 4 KB (scratch, overwritten before read).
#include <atomic>

#include "w4_device.cuh"

namespace w4 {
namespace {

constexpr int kSkStages = 6;
constexpr int kSkBlocksPerSm = 3;
constexpr int kXSlice = kGroup * 2;                  // bytes of one token's x per group
// Token slices sit 272 bytes apart, so the two tokens read by one quarter-warp
// (rows gq, gq+1 of the B fragment) fall in disjoint shared-memory banks.
constexpr int kXStride = kXSlice + 16;
constexpr int kXOff = kRecWeights + kRecScales + kRecZeros;
constexpr int kSkStageBytes = kXOff + W4_MAX_TOKENS * kXStride;  // 10688
constexpr int kPartialFloats4 = kWarps * 32;         // float4 per partial slot (4 KB)

struct SkPlan {
    size_t flag_off, bar_off, total;
};

__host__ __device__ inline SkPlan sk_plan() {
    SkPlan p;
    p.flag_off = (size_t)kSkStages * kSkStageBytes;
    p.bar_off = p.flag_off + 16;
    p.total = p.bar_off + (size_t)(2 * kSkStages) * 8;
    return p;
}

// First unit of block c.
__host__ __device__ inline long long sk_u0(long long c, long long W, long long P) {
    return c * W / P;
}

// The block whose range holds unit a (the largest c with sk_u0(c) <= a).
__device__ __forceinline__ int sk_block_of(long long a, long long W, long long P) {
    return (int)(((a + 1) * P + W - 1) / W - 1);
}

// This block's part of row block rb is complete (all eight consumer warps
// call this together).  Stores the row block if the block covered it whole;
// otherwise publishes the partial and, if it is the last contributor, adds all
// contributors' partials in block order and stores the sum.  Not inlined: it
// runs once per row block, and keeping it out of the unrolled stage loop keeps
// that loop small.
template <bool F32OUT>
__device__ __noinline__ void finish_row_block(float a0, float a1, float a2, float a3, int rb,
                                              bool whole, int G, long long W, int P, int c,
                                              int first_rb, uint32_t *counters,
                                              float4 *partials, volatile int *s_last, void *yv,
                                              int M, int N) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = rb * kWarps + warp;
    if (whole) {
        const float acc[4] = {a0, a1, a2, a3};
        store_tile<F32OUT>(yv, acc, t, lane, M, N);
        return;
    }
    const int slot = 2 * c + (rb == first_rb ? 0 : 1);
    partials[(size_t)slot * kPartialFloats4 + warp * 32 + lane] = make_float4(a0, a1, a2, a3);
    __threadfence();
    consumer_sync();
    const long long ru0 = (long long)rb * G;
    const int cf = sk_block_of(ru0, W, P), cl = sk_block_of(ru0 + G - 1, W, P);
    if (threadIdx.x == 0) {
        const unsigned prev = atomicAdd(&counters[rb], 1u);
        *s_last = prev == (unsigned)(cl - cf) ? 1 : 0;
    }
    consumer_sync();
    if (*s_last) {
        __threadfence();
        // Contributor cc's slot: 0 if rb is the first row block it touches,
        // which for every contributor after cf means it starts inside rb.
        float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 *base = partials + warp * 32 + lane;
        for (int c0 = cf; c0 <= cl; c0 += 8) {
            float4 v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int cc = c0 + j;
                if (cc <= cl) {
                    const int sl = 2 * cc + ((cc == cf && sk_u0(cc, W, P) < ru0) ? 1 : 0);
                    v[j] = __ldcg(base + (size_t)sl * kPartialFloats4);
                }
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (c0 + j <= cl) {
                    sum.x += v[j].x;
                    sum.y += v[j].y;
                    sum.z += v[j].z;
                    sum.w += v[j].w;
                }
            }
        }
        const float tot[4] = {sum.x, sum.y, sum.z, sum.w};
        store_tile<F32OUT>(yv, tot, t, lane, M, N);
        if (threadIdx.x == 0) counters[rb] = 0u;   // ready for the next call
    }
}

template <bool F32OUT>
__global__ void __launch_bounds__(kThreads, kSkBlocksPerSm)
gemv_sk_kernel(const char *__restrict__ qw, const char *__restrict__ sc,
               const char *__restrict__ zp, const __nv_bfloat16 *__restrict__ x,
               void *__restrict__ yv, uint32_t *err, int M, int K, int N, int P,
               uint32_t *__restrict__ counters, float4 *__restrict__ partials,
               uint32_t nib_mask, uint32_t bf16_magic) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int G = K / kGroup;
    const long long W = (long long)row_blocks(N) * G;
    const int c = blockIdx.x;
    const long long u0 = sk_u0(c, W, P), u1 = sk_u0(c + 1, W, P);
    const int n = (int)(u1 - u0);
    const int first_rb = (int)(u0 / G);
    const int g0 = (int)(u0 - (long long)first_rb * G);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const SkPlan plan = sk_plan();
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + plan.bar_off);
    uint64_t *empty = full + kSkStages;
    volatile int *s_last = reinterpret_cast<volatile int *>(smem + plan.flag_off);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kSkStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        reinterpret_cast<uint32_t *>(smem + plan.flag_off)[1] = nib_mask;
        reinterpret_cast<uint32_t *>(smem + plan.flag_off)[2] = bf16_magic;
    }
    __syncthreads();
    allow_dependents();

    bool ok = true;
    if (warp == kWarps) {
        // ---- producer: the block's records in order, with x next to them ----
        if (lane == 0) {
            const uint32_t stage_tx = (uint32_t)(kXOff + M * kXSlice);
            const char *qp = qw + W4_HEADER_BYTES + (size_t)u0 * kRecWeights;
            const char *sp = sc + (size_t)u0 * kRecScales;
            const char *zq = zp + (size_t)u0 * kRecZeros;
            // The first records (up to two) do not depend on the previous
            // kernel in the stream; their x slices follow once it has ended.
            const int first = n < 2 ? n : 2;
            int g = g0, i = 0, issued = 0;
            uint32_t phase = 0;
            for (int s = 0; s < n; ++s) {
                if (s == first) {
                    wait_prerequisites();
                    for (int f = 0; f < first; ++f) {
                        const int gf = g0 + f < G ? g0 + f : g0 + f - G;
                        for (int m = 0; m < M; ++m)
                            bulk_g2s(smem + f * kSkStageBytes + kXOff + m * kXStride,
                                     x + (size_t)m * K + (size_t)gf * kGroup, kXSlice, &full[f]);
                    }
                }
                if (s >= kSkStages && !mbar_wait(&empty[i], phase ^ 1u)) {
                    ok = false;
                    break;
                }
                if (s >= kSkStages) fence_proxy_async();
                unsigned char *st = smem + i * kSkStageBytes;
                mbar_expect_tx(&full[i], stage_tx);
                bulk_g2s(st, qp, kRecWeights, &full[i]);
                bulk_g2s(st + kRecWeights, sp, kRecScales, &full[i]);
                bulk_g2s(st + kRecWeights + kRecScales, zq, kRecZeros, &full[i]);
                if (s >= first)
                    for (int m = 0; m < M; ++m)
                        bulk_g2s(st + kXOff + m * kXStride, x + (size_t)m * K + (size_t)g * kGroup,
                                 kXSlice, &full[i]);
                ++issued;
                qp += kRecWeights;
                sp += kRecScales;
                zq += kRecZeros;
                if (++g == G) g = 0;
                if (++i == kSkStages) {
                    i = 0;
                    phase ^= 1u;
                }
            }
            if (ok && n == first) {
                wait_prerequisites();
                for (int f = 0; f < first; ++f) {
                    const int gf = g0 + f < G ? g0 + f : g0 + f - G;
                    for (int m = 0; m < M; ++m)
                        bulk_g2s(smem + f * kSkStageBytes + kXOff + m * kXStride,
                                 x + (size_t)m * K + (size_t)gf * kGroup, kXSlice, &full[f]);
                }
            }
            if (!ok) {
                for (int s = issued > kSkStages ? issued - kSkStages : 0; s < issued; ++s)
                    mbar_wait(&full[s % kSkStages], (s / kSkStages) & 1);
                atomicOr(err, 1u);
            }
        }
    } else {
        // ---- consumers: warp w owns tile w of whichever row block is current ----
        // Token slots M..7 of every stage are never written by the copies:
        // zero them once, so tokens past M multiply zeros.
        for (int w = threadIdx.x; w < kSkStages * (W4_MAX_TOKENS - M) * (kXSlice / 4);
             w += kWarps * 32) {
            const int per_stage = (W4_MAX_TOKENS - M) * (kXSlice / 4);
            const int st_i = w / per_stage, r = w - st_i * per_stage;
            const int m = M + r / (kXSlice / 4), o = r % (kXSlice / 4);
            reinterpret_cast<uint32_t *>(smem + st_i * kSkStageBytes + kXOff + m * kXStride)[o] =
                0u;
        }
        consumer_sync();
        wait_prerequisites();           // x and y belong to the previous kernel until it ends
        const int gq = lane >> 2, tq = lane & 3;
        const int xoff = kXOff + gq * kXStride + tq * 32;   // this lane's B words in a stage
        const float zq[4] = {0.f, 0.f, 0.f, 0.f};
        // The two conversion constants, read from shared memory so that they
        // sit in ordinary registers: left as kernel parameters they are kept
        // in uniform registers, and a three-input logic operation takes only
        // one of those, which costs a register move per extraction.
        const uint32_t mask = reinterpret_cast<volatile uint32_t *>(smem + plan.flag_off)[1];
        const uint32_t magic = reinterpret_cast<volatile uint32_t *>(smem + plan.flag_off)[2];
        int i = 0, s = 0, rb = first_rb, g = g0;
        uint32_t phase = 0;
        // The block's units, one row-block segment at a time.  A warp whose
        // wait gives up stops computing but keeps taking part in every barrier
        // and counter step, so no other warp waits for it and the counters
        // stay consistent; the error word reports the failure.
        while (s < n) {
            const int seg = n - s < G - g ? n - s : G - g;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            for (int k = 0; k < seg; ++k) {
                if (ok && !mbar_wait(&full[i], phase)) ok = false;
                if (ok) {
                    const unsigned char *st = smem + i * kSkStageBytes;
                    const GroupData gd = read_group(st, warp, lane);
                    const GroupB gb = load_b(reinterpret_cast<const uint32_t *>(st + xoff));
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[i]);   // stage copied to registers
                    group_mma(acc, gd, gb, zq, mask, magic);
                }
                if (++i == kSkStages) {
                    i = 0;
                    phase ^= 1u;
                }
            }
            finish_row_block<F32OUT>(acc[0], acc[1], acc[2], acc[3], rb, seg == G, G, W, P, c,
                                     first_rb, counters, partials, s_last, yv, M, N);
            s += seg;
            ++rb;
            g = 0;
        }
        if (!ok && lane == 0) atomicOr(err, 1u);
    }
}

}  // namespace

int gemv_ws_blocks(int K, int N, int num_sms) {
    const long long W = (long long)row_blocks(N) * (K / kGroup);
    const long long cap = (long long)kSkBlocksPerSm * (num_sms > 0 ? num_sms : 1);
    return (int)(W < cap ? W : cap);
}

size_t gemv_ws_bytes(int K, int N, int num_sms) {
    const size_t counters = ((size_t)row_blocks(N) * 4 + 255) / 256 * 256;
    return counters + (size_t)2 * gemv_ws_blocks(K, N, num_sms) * kPartialFloats4 * 16;
}

cudaError_t launch_gemv_ws(const void *qweight, const void *scales, const void *zeros,
                           const uint16_t *x, void *y, bool f32_out, int M, int K, int N,
                           void *workspace, int num_sms, cudaStream_t stream) {
    const int P = gemv_ws_blocks(K, N, num_sms);
    const SkPlan plan = sk_plan();
    // Set once per (output type, device); atomic flags, so host threads that
    // race on a first call both set the (idempotent) attribute.
    static std::atomic<bool> attr_done[2][64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    auto kern = f32_out ? gemv_sk_kernel<true> : gemv_sk_kernel<false>;
    if (!attr_done[f32_out][dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)plan.total);
        if (e != cudaSuccess) return e;
        attr_done[f32_out][dev].store(true, std::memory_order_release);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)P, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = plan.total;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const char *q = static_cast<const char *>(qweight);
    uint32_t *err = reinterpret_cast<uint32_t *>(const_cast<char *>(q) + kErrorOffset);
    uint32_t *counters = static_cast<uint32_t *>(workspace);
    float4 *partials = reinterpret_cast<float4 *>(
        static_cast<char *>(workspace) + ((size_t)row_blocks(N) * 4 + 255) / 256 * 256);
    return cudaLaunchKernelEx(&cfg, kern, q, static_cast<const char *>(scales),
                              static_cast<const char *>(zeros),
                              reinterpret_cast<const __nv_bfloat16 *>(x), y, err, M, K, N, P,
                              counters, partials, 0x000F000Fu, 0x43004300u);
}

}  // namespace w4
