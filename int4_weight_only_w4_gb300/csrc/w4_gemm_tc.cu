// w4_gemm for more than 16 tokens: one pass over the weight on the 5th-generation
// tensor cores (tcgen05: accumulators and the dequantised weight operand in
// tensor memory).
//
// Passes of 8 tokens ("qengine", section "How the numbers were measured")
// stream and unpack the weight once per pass; prefill batches need the weight
// read once.  Here a thread block owns one 128-row block of W and a tile of up
// to 128 tokens and walks its K groups once, with one role per warp (20):
//   weight producer (warp 0, one lane): per group, the record's 8 KB of
//     nibbles with one 2-D tensor copy (the record seen as 64 rows of 128 B,
//     128-byte swizzle, so that the converters' row reads below hit every
//     bank), plus its 256 B of scales and 64 B of zero points (plain bulk
//     copies), into a ring of 12 stages;
//   x producer (warp 19, one lane): per group, the tile's tokens x 128 k of x
//     as two 2-D tensor copies of 64 k (128-byte swizzled, K-major: the layout
//     the tensor cores read), tokens past M filled with zeros by the copy,
//     into a ring of 3 to 16 stages (more for smaller tiles);
//   converters (warps 1..8): warp w owns tensor-memory lanes 32 (w mod 4) ..
//     +31, i.e. one weight row per thread, and the groups g with g mod 2 ==
//     (w - 1) / 4.  Per group a thread reads its row's 128 nibbles (eight
//     16-byte loads, half of each belonging to the row eight below), forms
//     bf16 (q - z) -- exact: (nibble | 0x4300) read as bf16 is 128 + q, one
//     bf16 add of -(128 + z) -- and writes the 128 values into one of four
//     operand buffers in tensor memory (two tcgen05.st); the row's fp32
//     scale goes to a 16-deep ring in shared memory;
//   issuers (warps 17, 18, one lane each): the groups alternate between them;
//     per group eight tcgen05.mma.kind::f16 with the weight operand from
//     tensor memory and x from shared memory (M = 128 rows, N = the token
//     tile rounded up to 16, K = 16 each) into one of 2 to 8 accumulators
//     (32, 64 or 128 columns wide: the tile rounded up), then tcgen05.commit
//     to the barriers that free the operand buffers and publish the sums.  A
//     tensor-core instruction holds its issuing thread for about 100 cycles
//     whatever N is (up to 128), so two issuers on independent accumulators
//     double the rate;
//   readback (warps 9..16): warp w reads lanes 32 (w mod 4) .. +31 and the
//     16-column units u of the token columns with u mod 2 == (w - 9) / 4: per
//     group tcgen05.ld of the row's fp32 group sums and acc += s * sum in
//     registers; then the epilogue (or, with a K split, the cluster combine).
// The group's scale multiplies the group's fp32 sum, exactly the arithmetic of
// the GEMV's exact path: per group sum_k (q - z) x accumulated in fp32 by the
// tensor cores, then acc = fma(s, sum, acc) group by group in order.  A
// token's result does not depend on the other tokens of the tile or on M.
//
// Every wait is bounded (about 2 s of clock cycles): a role that gives up sets
// the header's error word and the block winds down; the producers wait
// (bounded) for their copies in flight and the issuers for their last
// tensor-core work before the tensor memory is freed.
#include <cuda.h>   // CUtensorMap and the tensor-map encoder's types (resolved at run time)
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cooperative_groups.h>

#include <atomic>
#include <mutex>

#include "w4_device.cuh"

namespace cg = cooperative_groups;

namespace w4 {
namespace {

constexpr int kTcRows = 128;                        // weight rows per block (one row block)
constexpr int kTcTokens = 128;                      // tokens per block at most
constexpr int kWRing = 12;                          // weight-record stages
constexpr int kXRegion = 3 * 32768;                 // x stages: 96 KB, 3 stages of 128 tokens
constexpr int kMaxXStages = 16;                     // ... up to 16 stages of fewer tokens
constexpr int kABufs = 4;                           // weight operands in tensor memory
constexpr int kDCols = 256;                         // tensor-memory columns for accumulators
constexpr int kMaxDStages = 8;                      // accumulators: kDCols / their width
constexpr int kSRing = 16;                          // per-group scales handed to the readback
constexpr int kSzBytes = kRecScales + kRecZeros;    // 320: scales and zero points of a record
constexpr int kConv = 8;                            // converter warps 1..8
constexpr int kRead = 8;                            // readback warps 9..16
constexpr int kIssuers = 2;                         // issuer warps 17, 18 (alternate groups)
constexpr int kTcIssuer = 1 + kConv + kRead;        // first issuer warp
constexpr int kXProducer = kTcIssuer + kIssuers;    // warp 19
constexpr int kTcThreads = (kXProducer + 1) * 32;   // 640
// tensor memory: accumulators d at columns dcols d (dcols = 32, 64 or 128:
// the token tile rounded up), weight operands a at kDCols + 64 a (128 k of
// bf16 = 64 32-bit columns)
constexpr uint32_t kACol = kDCols;
constexpr int kTcTmemCols = 512;
static_assert(kACol + kABufs * 64 <= kTcTmemCols, "tensor memory budget");

struct TcSmem {
    // offsets from the 1024-byte-aligned base
    static constexpr int w0 = 0;                               // weight nibbles [kWRing]
    static constexpr int x0 = w0 + kWRing * kRecWeights;       // x tiles [nX]
    static constexpr int sz0 = x0 + kXRegion;                  // scales + zeros [kWRing]
    static constexpr int scl0 = sz0 + kWRing * kSzBytes;       // fp32 scales [kSRing][128]
    static constexpr int bars = scl0 + kSRing * kTcRows * 4;
    // barriers: w_full[W], w_empty[W], x_full[X], x_empty[X], a_full[A],
    // a_empty[A], d_full[D], d_empty[D], s_full[S], s_empty[S]
    static constexpr int nbars = 2 * (kWRing + kMaxXStages + kABufs + kMaxDStages + kSRing);
    static constexpr int tmem_slot = bars + nbars * 8;
    static constexpr int total = tmem_slot + 16;
    static constexpr int alloc = total + 1024;                 // + alignment slack
};
static_assert(TcSmem::alloc <= 232448, "shared memory per block");
static_assert(kXRegion >= kTcTokens * kTcRows * 4, "combine buffer fits the x ring");

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 2-D tensor copy global -> shared, completion counted in bytes on `bar`.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int c0, int c1,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];"
        ::"r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1),
        "r"(smem_addr(bar))
        : "memory");
}

// Shared-memory matrix descriptor (tcgen05): K-major operand in the 128-byte
// swizzled layout; start address and the 1024-byte stride between 8-row
// groups in 16-byte units, descriptor version 1, swizzle mode 128 B.
__device__ __forceinline__ uint64_t tc_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);          // start address
    d |= (uint64_t)1u << 16;                          // leading offset (unused for this layout)
    d |= (uint64_t)(1024u >> 4) << 32;                // stride offset: 8 rows x 128 B
    d |= (uint64_t)1u << 46;                          // version
    d |= (uint64_t)2u << 61;                          // 128-byte swizzle
    return d;
}

// Instruction descriptor for kind::f16: fp32 accumulators, bf16 A and B, both
// K-major, N x M = n x 128.
__device__ __forceinline__ uint32_t tc_idesc(int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(kTcRows >> 4) << 24);
}

// D (tensor memory) [+]= A (tensor memory) x B (shared memory)^T.
__device__ __forceinline__ void tc_mma_ts(uint32_t dtmem, uint32_t atmem, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        ::"r"(dtmem), "r"(atmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(smem_addr(bar))
                 : "memory");
}

// 16 consecutive fp32 columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tc_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Two 16-column loads of this thread's lane (columns c .. c + 15 and c + 32 ..
// c + 47), one wait.
__device__ __forceinline__ void tc_ld16_pair(uint32_t taddr, float (&v)[16], float (&u)[16]) {
    uint32_t r[16], q[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(q[0]), "=r"(q[1]), "=r"(q[2]), "=r"(q[3]), "=r"(q[4]), "=r"(q[5]), "=r"(q[6]),
          "=r"(q[7]), "=r"(q[8]), "=r"(q[9]), "=r"(q[10]), "=r"(q[11]), "=r"(q[12]),
          "=r"(q[13]), "=r"(q[14]), "=r"(q[15])
        : "r"(taddr + 32u));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        v[i] = __uint_as_float(r[i]);
        u[i] = __uint_as_float(q[i]);
    }
}

// (a0, a1) = fma(s, (v0, v1), (a0, a1)) as one packed instruction: each lane
// is the IEEE fused multiply-add rounded to nearest, the same bits as fmaf.
__device__ __forceinline__ void fma2(float &a0, float &a1, float s, float v0, float v1) {
    asm("{\n\t.reg .b64 a, b, c;\n\t"
        "mov.b64 a, {%0, %1};\n\t"
        "mov.b64 b, {%2, %2};\n\t"
        "mov.b64 c, {%3, %4};\n\t"
        "fma.rn.f32x2 a, b, c, a;\n\t"
        "mov.b64 {%0, %1}, a;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "f"(s), "f"(v0), "f"(v1));
}

// This thread's 32 words into 32 consecutive columns of its tensor-memory lane.
__device__ __forceinline__ void tc_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
        "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]),
        "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]),
        "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
        "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

template <bool F32OUT>
__global__ void __launch_bounds__(kTcThreads, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap xmap,
               const char *__restrict__ sc, const char *__restrict__ zp, void *__restrict__ yv,
               uint32_t *err, int M, int K, int N, int xrows) {
    extern __shared__ unsigned char smem_raw[];
    // 1024-byte-aligned base (the swizzle atoms are 1024-byte aligned)
    const uint32_t raw = smem_addr(smem_raw);
    unsigned char *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const int Gall = K / kGroup;
    const int S = (int)gridDim.z;                    // K split: blocks of one cluster
    const int split = (int)blockIdx.z;
    const int gbeg = (int)((long long)split * Gall / S);
    const int G = (int)((long long)(split + 1) * Gall / S) - gbeg;   // groups of this block
    const int rb = blockIdx.x;                       // row block
    const int m0 = blockIdx.y * kTcTokens;           // first token of the tile
    const int mt = M - m0 < kTcTokens ? M - m0 : kTcTokens;   // tokens in the tile
    const int n_mma = (mt + 15) / 16 * 16;           // MMA N: tokens rounded up to 16
    // accumulator width and count: 32, 64 or 128 columns, kDCols in all
    const int dcols = n_mma <= 32 ? 32 : n_mma <= 64 ? 64 : 128;
    const int nD = kDCols / dcols;                   // 8, 4 or 2: a multiple of kIssuers
    // x stages: two 64-k boxes of xrows tokens each, as many as fit (up to 16)
    const int xstage = 2 * xrows * 128;
    const int nX = kXRegion / xstage < kMaxXStages ? kXRegion / xstage : kMaxXStages;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + TcSmem::bars);
    uint64_t *w_full = bars, *w_empty = w_full + kWRing;
    uint64_t *x_full = w_empty + kWRing, *x_empty = x_full + kMaxXStages;
    uint64_t *a_full = x_empty + kMaxXStages;   // [A]: weight operand written
    uint64_t *a_empty = a_full + kABufs;        // [A]: weight operand read by the MMAs
    uint64_t *d_full = a_empty + kABufs;        // [D]: accumulator holds the sums
    uint64_t *d_empty = d_full + kMaxDStages;   // [D]: accumulator read back
    uint64_t *s_full = d_empty + kMaxDStages;   // [S]: a group's scales written
    uint64_t *s_empty = s_full + kSRing;        // [S]: a group's scales read
    float *scl = reinterpret_cast<float *>(smem + TcSmem::scl0);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + TcSmem::tmem_slot);
    volatile uint32_t *failed = tmem_slot + 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kWRing; ++s) {
            mbar_init(&w_full[s], 1);
            mbar_init(&w_empty[s], kConv / 2);   // the four converters of the group
        }
        for (int s = 0; s < kMaxXStages; ++s) {
            mbar_init(&x_full[s], 1);
            mbar_init(&x_empty[s], 1);
        }
        for (int b = 0; b < kABufs; ++b) {
            mbar_init(&a_full[b], kConv / 2);
            mbar_init(&a_empty[b], 1);
        }
        for (int b = 0; b < kMaxDStages; ++b) {
            mbar_init(&d_full[b], 1);
            mbar_init(&d_empty[b], kRead);
        }
        for (int b = 0; b < kSRing; ++b) {
            mbar_init(&s_full[b], kConv / 2);
            mbar_init(&s_empty[b], kRead);
        }
        *failed = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kTcIssuer) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_addr(tmem_slot)), "r"(kTcTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---- weight producer: the row block's G records ----
        if (lane == 0) {
            const size_t rec0 = (size_t)rb * Gall + gbeg;
            int g = 0;
            for (; g < G; ++g) {
                const int s = g % kWRing;
                if (g >= kWRing) {
                    if (!mbar_wait(&w_empty[s], ((g / kWRing) - 1) & 1)) break;
                    fence_proxy_async();
                }
                const size_t rec = rec0 + g;
                unsigned char *sz = smem + TcSmem::sz0 + s * kSzBytes;
                mbar_expect_tx(&w_full[s], kRecWeights + kSzBytes);
                tma_load_2d(smem + TcSmem::w0 + s * kRecWeights, &wmap, 0,
                            (int)(rec * (kRecWeights / 128)), &w_full[s]);
                bulk_g2s(sz, sc + rec * kRecScales, kRecScales, &w_full[s]);
                bulk_g2s(sz + kRecScales, zp + rec * kRecZeros, kRecZeros, &w_full[s]);
            }
            if (g < G) {
                *failed = 1;
                atomicOr(err, 1u);
            }
            // let the copies still in flight land (bounded) before exit
            for (int q = g > kWRing ? g - kWRing : 0; q < g; ++q)
                mbar_wait(&w_full[q % kWRing], (q / kWRing) & 1);
        }
    } else if (warp == kXProducer) {
        // ---- x producer: the tile's tokens, 128 k per group ----
        if (lane == 0) {
            int g = 0;
            for (; g < G; ++g) {
                const int b = g % nX;
                if (g >= nX) {
                    if (!mbar_wait(&x_empty[b], ((g / nX) - 1) & 1)) break;
                    fence_proxy_async();
                }
                unsigned char *xb = smem + TcSmem::x0 + b * xstage;
                const int k0 = (gbeg + g) * kGroup;
                mbar_expect_tx(&x_full[b], 2 * xrows * 128);
                tma_load_2d(xb, &xmap, k0, m0, &x_full[b]);
                tma_load_2d(xb + xrows * 128, &xmap, k0 + 64, m0, &x_full[b]);
            }
            if (g < G) {
                *failed = 1;
                atomicOr(err, 1u);
            }
            for (int q = g > nX ? g - nX : 0; q < g; ++q)
                mbar_wait(&x_full[q % nX], (q / nX) & 1);
        }
    } else if (warp >= kTcIssuer && warp < kTcIssuer + kIssuers) {
        // ---- issuers: issuer i takes the groups g = i mod kIssuers, eight
        // MMAs each into accumulator g mod nD (a tensor-core instruction
        // holds its issuing thread for about 100 cycles whatever N is, so
        // two issuers on independent accumulators double the rate) ----
        if (lane == 0) {
            const int i0 = warp - kTcIssuer;
            const uint32_t idesc = tc_idesc(n_mma);
            const uint32_t x_base = smem_addr(smem + TcSmem::x0);
            int g = i0;
            for (; g < G; g += kIssuers) {
                const int a = g % kABufs, b = g % nX, d = g % nD;
                if (!mbar_wait(&a_full[a], (g / kABufs) & 1)) break;
                if (!mbar_wait(&x_full[b], (g / nX) & 1)) break;
                if (g >= nD && !mbar_wait(&d_empty[d], ((g / nD) - 1) & 1)) break;
                tc_fence_after();
                const uint32_t dt = tmem + (uint32_t)(d * dcols);
                const uint32_t at = tmem + kACol + (uint32_t)(a * 64);
                const uint32_t xb = x_base + (uint32_t)(b * xstage);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    // k-step j: 16 k = 8 columns of the weight operand; 32 bytes
                    // into the j/4-th 64-k atom of x
                    const uint32_t bo = (uint32_t)((j >> 2) * xrows * 128 + (j & 3) * 32);
                    tc_mma_ts(dt, at + (uint32_t)(8 * j), tc_desc(xb + bo), idesc,
                              j > 0 ? 1u : 0u);
                }
                tc_commit(&a_empty[a]);    // weight operand a may be rewritten
                tc_commit(&x_empty[b]);    // x stage b may be refilled
                tc_commit(&d_full[d]);     // accumulator d holds the group's sums
            }
            if (g < G) {
                *failed = 1;
                atomicOr(err, 1u);
            }
            // before the tensor memory is freed: this issuer's last groups'
            // work has ended
            for (int q = i0; q < g; q += kIssuers)
                if (q + nD >= g) mbar_wait(&d_full[q % nD], (q / nD) & 1);
        }
    } else if (warp <= kConv) {
        // ---- converters: warps 1..8; warp w converts the groups g with
        // g mod 2 == (w - 1) / 4, all 128 k of its quarter's 32 rows ----
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;     // this thread's weight row in the block
        const int par = (warp - 1) >> 2;         // group parity
        const int tile = row >> 4, gq = row & 7, hi = (row >> 3) & 1;
        // The record's nibbles of row `row`, k = 64 h .. 64 h + 63 (h = 0, 1):
        // chunk tq = 0..3 (16 k each) at byte tile * 1024 + h * 512 + gq * 64 +
        // tq * 16 of the record (the kernel layout, w4_repack.cu), which the
        // 128-byte swizzle of the tensor copy moved to chunk ((gq & 1) * 4 +
        // tq) ^ (row128 & 7) of 128-byte row row128.  A chunk's word v holds,
        // for row 16 tile + gq (hi = 0) in bits 0-7 and 16-23 and for row
        // 16 tile + gq + 8 (hi = 1) in bits 8-15 and 24-31: k = 2v, 2v + 1
        // (low nibbles) and 2v + 8, 2v + 9 (high nibbles) of the chunk.
        uint32_t woff[2][4];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int row128 = tile * 8 + h * 4 + (gq >> 1);
#pragma unroll
            for (int tq = 0; tq < 4; ++tq)
                woff[h][tq] =
                    (uint32_t)(row128 * 128 + (((((gq & 1) << 2) | tq) ^ (row128 & 7)) << 4));
        }
        const int shift = 8 * hi;
        const uint32_t mask = 0x000F000Fu, magic = 0x43004300u;
        const uint32_t t_op = tmem + ((uint32_t)(quarter * 32) << 16) + kACol;
        int g = par;
        for (; g < G; g += 2) {
            const int s = g % kWRing, a = g % kABufs, sr = g % kSRing;
            bool w = mbar_wait(&w_full[s], (g / kWRing) & 1);
            if (g >= kABufs) w = w && mbar_wait(&a_empty[a], ((g / kABufs) - 1) & 1);
            if (g >= kSRing) w = w && mbar_wait(&s_empty[sr], ((g / kSRing) - 1) & 1);
            if (!__all_sync(0xFFFFFFFFu, w)) break;
            tc_fence_after();
            const unsigned char *wst = smem + TcSmem::w0 + s * kRecWeights;
            const unsigned char *sz = smem + TcSmem::sz0 + s * kSzBytes;
            uint4 wv[2][4];
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int tq = 0; tq < 4; ++tq)
                    wv[h][tq] = *reinterpret_cast<const uint4 *>(wst + woff[h][tq]);
            // scale: fp16 pair (row 16 tile + gq, + 8) at tile * 32 + gq * 4;
            // zero points: nibble pair at tile * 8 + gq
            const uint32_t spair = *reinterpret_cast<const uint32_t *>(sz + tile * 32 + gq * 4);
            const uint32_t zb = sz[kRecScales + tile * 8 + gq];
            scl[sr * kTcRows + row] = __half2float(
                __ushort_as_half((unsigned short)(hi ? (spair >> 16) : (spair & 0xFFFFu))));
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&w_empty[s]);   // the stage's bytes are in registers
                mbar_arrive(&s_full[sr]);
            }
            const uint32_t z = hi ? (zb >> 4) : (zb & 0xFu);
            const uint32_t nz = (z | 0xC300u) * 0x10001u;   // -(128 + z), bf16 pair
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t r[32];
#pragma unroll
                for (int tq = 0; tq < 4; ++tq) {
                    const uint32_t words[4] = {wv[h][tq].x, wv[h][tq].y, wv[h][tq].z, wv[h][tq].w};
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        const uint32_t wd = words[v] >> shift;
                        r[8 * tq + v] = bf16x2_add(and_or(wd, mask, magic), nz);
                        r[8 * tq + 4 + v] = bf16x2_add(and_or(wd >> 4, mask, magic), nz);
                    }
                }
                tc_st32(t_op + (uint32_t)(a * 64 + 32 * h), r);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&a_full[a]);
        }
        if (g < G) {
            if (lane == 0) atomicOr(err, 1u);
            *failed = 1;
        }
    } else {
        // ---- readback: warps 9..16; warp w reads tensor-memory lanes 32 (w mod 4)
        // .. +31 (one weight row per thread) and the 16-column units u of the
        // token columns with u mod 2 == half: unit u = 2 l + half (l = 0..3)
        // goes to acc[16 l ..] ----
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const int half = (warp - 1 - kConv) >> 2;
        const uint32_t t_acc = tmem + ((uint32_t)(quarter * 32) << 16) + 16u * half;
        float acc[kTcTokens / 2];
#pragma unroll
        for (int i = 0; i < kTcTokens / 2; ++i) acc[i] = 0.f;
        int g = 0;
        for (; g < G; ++g) {
            const int d = g % nD, sr = g % kSRing;
            // warp-uniform: every lane waits, and they give up together before
            // the warp-wide tensor-memory loads
            const bool w = mbar_wait(&d_full[d], (g / nD) & 1) &&
                           mbar_wait(&s_full[sr], (g / kSRing) & 1);
            if (!__all_sync(0xFFFFFFFFu, w)) break;
            tc_fence_after();
            const float s_g = scl[sr * kTcRows + row];
#pragma unroll
            for (int l = 0; l < 4; l += 2) {
                if (16 * (2 * (l + 1) + half) < n_mma) {
                    // units 2 l + half and 2 (l + 1) + half in one wait
                    float v[16], u[16];
                    tc_ld16_pair(t_acc + (uint32_t)(d * dcols + 32 * l), v, u);
#pragma unroll
                    for (int i = 0; i < 16; i += 2) {
                        fma2(acc[16 * l + i], acc[16 * l + i + 1], s_g, v[i], v[i + 1]);
                        fma2(acc[16 * (l + 1) + i], acc[16 * (l + 1) + i + 1], s_g, u[i],
                             u[i + 1]);
                    }
                } else if (16 * (2 * l + half) < n_mma) {
                    float v[16];
                    tc_ld16(t_acc + (uint32_t)(d * dcols + 32 * l), v);
#pragma unroll
                    for (int i = 0; i < 16; i += 2)
                        fma2(acc[16 * l + i], acc[16 * l + i + 1], s_g, v[i], v[i + 1]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&d_empty[d]);
                mbar_arrive(&s_empty[sr]);
            }
        }
        if (g < G) {
            if (lane == 0) atomicOr(err, 1u);
            *failed = 1;
        } else if (S == 1) {
            // y[m0 + m][rb * 128 + row] for the tile's tokens; rows past N are padding
            const int n = rb * kTcRows + row;
            if (n < N) {
#pragma unroll
                for (int i = 0; i < kTcTokens / 2; ++i) {
                    const int m = 16 * (2 * (i >> 4) + half) + (i & 15);
                    if (m < mt) {
                        const size_t o = (size_t)(m0 + m) * N + n;
                        if (F32OUT)
                            static_cast<float *>(yv)[o] = acc[i];
                        else
                            static_cast<__nv_bfloat16 *>(yv)[o] = __float2bfloat16_rn(acc[i]);
                    }
                }
            }
        } else {
            // K split: this block's partial sums, [token][row] fp32, into its own
            // shared memory (the x ring, idle now: every MMA has completed) for
            // the cluster's combine
            float *red = reinterpret_cast<float *>(smem + TcSmem::x0);
#pragma unroll
            for (int i = 0; i < kTcTokens / 2; ++i) {
                const int m = 16 * (2 * (i >> 4) + half) + (i & 15);
                if (m < mt) red[m * kTcRows + row] = acc[i];
            }
        }
    }

    if (S > 1) {
        // Combine the S partial sums of each output in rank order 0, 1, ..., S-1
        // through distributed shared memory: block `split` of the cluster adds
        // and stores the tokens i with i mod S == split.  No float atomics.
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();
        if (warp > kConv && warp <= kConv + kRead && *failed == 0) {
            const int row = (warp & 3) * 32 + lane;
            const int half = (warp - 1 - kConv) >> 2;
            const int n = rb * kTcRows + row;
            float *red = reinterpret_cast<float *>(smem + TcSmem::x0);
            // tokens i = split + S j, alternating between the two warps of a quarter
            for (int i = split + S * half; i < mt; i += 2 * S) {
                float v = 0.f;
                for (int q = 0; q < S; ++q)
                    v += cluster.map_shared_rank(red, (unsigned)q)[i * kTcRows + row];
                if (n < N) {
                    const size_t o = (size_t)(m0 + i) * N + n;
                    if (F32OUT)
                        static_cast<float *>(yv)[o] = v;
                    else
                        static_cast<__nv_bfloat16 *>(yv)[o] = __float2bfloat16_rn(v);
                }
            }
        }
        cluster.sync();   // no block leaves while another still reads its shared memory
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kTcIssuer) {
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTcTmemCols));
    }
}

// cuTensorMapEncodeTiled, resolved once from the driver through the runtime.
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

}  // namespace

namespace {

std::atomic<bool> g_attr_done[2][64] = {};

// The kernel's dynamic shared memory limit, set once per device and variant.
cudaError_t prepare_tc(bool f32_out, int dev) {
    if (g_attr_done[f32_out][dev].load(std::memory_order_acquire)) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(
        f32_out ? gemm_tc_kernel<true> : gemm_tc_kernel<false>,
        cudaFuncAttributeMaxDynamicSharedMemorySize, TcSmem::alloc);
    if (e == cudaSuccess) g_attr_done[f32_out][dev].store(true, std::memory_order_release);
    return e;
}

// How many clusters of s blocks of the kernel can be resident at once on the
// device (clusters are placed whole, within one GPC); cached per device and
// size, -1 when the query failed (also cached, so that a device's choice
// never changes between calls).
std::atomic<int> g_max_clusters[64][9] = {};

int max_active_clusters(int dev, int s) {
    int n = g_max_clusters[dev][s].load(std::memory_order_acquire);
    if (n != 0) return n;
    n = -1;
    if (prepare_tc(false, dev) == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(1, 1, (unsigned)s);
        cfg.blockDim = dim3(kTcThreads, 1, 1);
        cfg.dynamicSmemBytes = TcSmem::alloc;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = (unsigned)s;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int q = 0;
        if (cudaOccupancyMaxActiveClusters(&q, (const void *)gemm_tc_kernel<false>, &cfg) ==
                cudaSuccess &&
            q > 0)
            n = q;
        else
            (void)cudaGetLastError();   // clear the error the failed query left
    }
    g_max_clusters[dev][s].store(n, std::memory_order_release);
    return n;
}

}  // namespace

int gemm_tc_splits(int K, int N, int num_sms) {
    // The largest S of 1..8 that gives every block at least four groups and
    // keeps the row blocks' clusters of S blocks within one wave (one block
    // per SM; as many clusters resident as there are row blocks; where the
    // runtime cannot tell, powers of two only).  It depends on K, N and the
    // device only, never on M, so a token's result is the same whatever M is.
    const int NB = row_blocks(N), G = K / kGroup;
    int smax = num_sms > 0 ? num_sms / NB : 1;
    if (smax > 8) smax = 8;
    if (smax > G / 4) smax = G / 4;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    for (int S = smax; S >= 2; --S) {
        const int n = max_active_clusters(dev, S);
        if (n < 0 ? (S & (S - 1)) == 0 : n >= NB) return S;
    }
    return 1;
}

// Tokens per x tile copy: 128, or M rounded up to 16 when M is smaller.
int gemm_tc_x_rows(int M) {
    return M >= kTcTokens ? kTcTokens : (M + 15) / 16 * 16;
}

cudaError_t launch_gemm_tc(const void *qweight, const void *scales, const void *zeros,
                           const uint16_t *x, void *y, bool f32_out, int M, int K, int N,
                           int num_sms, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    const EncodeTiledFn encode = encode_tiled();
    if (!encode) return cudaErrorNotSupported;
    auto kern = f32_out ? gemm_tc_kernel<true> : gemm_tc_kernel<false>;
    if ((e = prepare_tc(f32_out, dev)) != cudaSuccess) return e;
    const int NB = row_blocks(N), Gall = K / kGroup;
    const int xrows = gemm_tc_x_rows(M);
    const char *q = static_cast<const char *>(qweight);
    CUtensorMap wmap, xmap;
    {
        // the weight records' nibbles as rows of 128 bytes, 64 rows per record
        const cuuint64_t dims[2] = {128, (cuuint64_t)NB * Gall * (kRecWeights / 128)};
        const cuuint64_t strides[1] = {128};
        const cuuint32_t box[2] = {128, kRecWeights / 128};
        const cuuint32_t estr[2] = {1, 1};
        if (encode(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                   const_cast<char *>(q) + W4_HEADER_BYTES, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        // x [M][K] bf16: boxes of 64 k x xrows tokens; tokens past M read as zeros
        const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
        const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
        const cuuint32_t box[2] = {64, (cuuint32_t)xrows};
        const cuuint32_t estr[2] = {1, 1};
        if (encode(&xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(x), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    const int S = gemm_tc_splits(K, N, num_sms);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)NB, (unsigned)((M + kTcTokens - 1) / kTcTokens), (unsigned)S);
    cfg.blockDim = dim3(kTcThreads, 1, 1);
    cfg.dynamicSmemBytes = TcSmem::alloc;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = (unsigned)S;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    uint32_t *err = reinterpret_cast<uint32_t *>(const_cast<char *>(q) + kErrorOffset);
    return cudaLaunchKernelEx(&cfg, kern, wmap, xmap, static_cast<const char *>(scales),
                              static_cast<const char *>(zeros), y, err, M, K, N, xrows);
}

}  // namespace w4
