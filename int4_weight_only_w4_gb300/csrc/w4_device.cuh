// Device-side building blocks shared by the GEMV kernels (w4_gemv.cu,
// w4_gemv_sk.cu): PTX wrappers for mbarriers, bulk copies and programmatic
// dependent launch, the nibble-to-bf16 / -fp16 conversions and the
// tensor-core steps.
// Internal to libw4.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "w4_internal.cuh"

namespace w4 {
namespace {

constexpr int kWarps = kBlockTiles;                 // consumer warps (one per 16-row tile)
constexpr int kThreads = (kWarps + 1) * 32;         // + one producer warp
constexpr long long kWaitLimit = 4000000000LL;      // clock cycles (~2 s)

// ---- PTX wrappers ---------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

// Orders this thread's view of shared memory in the generic proxy (the
// consumers' reads of a stage, acquired through its "empty" barrier) before
// its following async-proxy operations (the bulk copy that refills the
// stage).  Without it the refill can land while the last reads of the stage
// are still being served: an mbarrier release/acquire pair orders memory
// within one proxy only.
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of `bar` to complete; false if the wait gave up.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > kWaitLimit) return false;
    }
    return true;
}

// Programmatic dependent launch: let the next kernel in the stream start its
// prologue now / wait until the previous kernel in the stream has completed
// and its writes are visible.
__device__ __forceinline__ void allow_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void wait_prerequisites() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// a * 1 + c on a bf16 pair; with c = -(128 + z) this is (128 + q) - (128 + z)
// = q - z, exact.
__device__ __forceinline__ uint32_t bf16x2_add(uint32_t a, uint32_t c) {
    uint32_t r;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(0x3F803F80u), "r"(c));
    return r;
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

// d = A * B (accumulator starts from the zero registers zq).
__device__ __forceinline__ void mma_bf16_16816_first(float (&d)[4], uint32_t a0, uint32_t a1,
                                                     uint32_t a2, uint32_t a3, uint32_t b0,
                                                     uint32_t b1, const float (&zq)[4]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%10, %11, %12, %13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(zq[0]), "f"(zq[1]),
          "f"(zq[2]), "f"(zq[3]));
}

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                              uint32_t a2, uint32_t a3, uint32_t b0,
                                              uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_f16_16816_first(float (&d)[4], uint32_t a0, uint32_t a1,
                                                    uint32_t a2, uint32_t a3, uint32_t b0,
                                                    uint32_t b1, const float (&zq)[4]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%10, %11, %12, %13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(zq[0]), "f"(zq[1]),
          "f"(zq[2]), "f"(zq[3]));
}

// Packed pairs of fp32 values (one 64-bit register pair, element 0 in the low
// half): one instruction for two independent correctly rounded operations.
__device__ __forceinline__ unsigned long long f32x2_mul(unsigned long long a,
                                                        unsigned long long b) {
    unsigned long long r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ unsigned long long f32x2_add(unsigned long long a,
                                                        unsigned long long b) {
    unsigned long long r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ float f32x2_lo(unsigned long long v) {
    return __uint_as_float((uint32_t)v);
}
__device__ __forceinline__ float f32x2_hi(unsigned long long v) {
    return __uint_as_float((uint32_t)(v >> 32));
}

// (w & mask) | magic in one three-input logic operation.
__device__ __forceinline__ uint32_t and_or(uint32_t w, uint32_t mask, uint32_t magic) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(w), "r"(mask), "r"(magic));
    return r;
}

// Barrier over the eight consumer warps only (the producer warp is busy).
__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"r"(kWarps * 32) : "memory");
}

// A lane's four words of one 64-k chunk as A registers (layout of
// w4_repack.cu): for word v, r[0][v] and r[2][v] carry the first pair of rows
// gq and gq + 8 (steps 0, 1), r[1][v] and r[3][v] the second (steps 2, 3).
// The tensor-core steps of the chunk are then
//   step 0: (r0[0], r2[0], r0[1], r2[1])   step 1: (r0[2], r2[2], r0[3], r2[3])
//   step 2: (r1[0], r3[0], r1[1], r3[1])   step 3: (r1[2], r3[2], r1[3], r3[3])
// with B registers 2j, 2j+1 of the lane's eight (x pairs 8tq .. 8tq+7 of the
// chunk); steps 0, 1 accumulate into d[0] and steps 2, 3 into d[1] (two
// independent chains).  FIRST: the chains start from the zero registers zq.
template <bool FIRST, bool HALF>
__device__ __forceinline__ void chunk_steps(float (&d)[2][4], const uint32_t (&r)[4][4],
                                            const uint4 &bl, const uint4 &bh,
                                            const float (&zq)[4]) {
    const uint32_t b[8] = {bl.x, bl.y, bl.z, bl.w, bh.x, bh.y, bh.z, bh.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int p = j >> 1;                 // 0: first pairs (r0, r2), 1: second (r1, r3)
        const int v = 2 * (j & 1);            // words v, v + 1
        const uint32_t a0 = r[p][v], a1 = r[2 + p][v], a2 = r[p][v + 1], a3 = r[2 + p][v + 1];
        if (FIRST && (j & 1) == 0) {
            if (HALF)
                mma_f16_16816_first(d[p], a0, a1, a2, a3, b[2 * j], b[2 * j + 1], zq);
            else
                mma_bf16_16816_first(d[p], a0, a1, a2, a3, b[2 * j], b[2 * j + 1], zq);
        } else {
            if (HALF)
                mma_f16_16816(d[p], a0, a1, a2, a3, b[2 * j], b[2 * j + 1]);
            else
                mma_bf16_16816(d[p], a0, a1, a2, a3, b[2 * j], b[2 * j + 1]);
        }
    }
}

// bf16 operands, exact q - z: (word >> 4i) & 0x000F000F | 0x43004300 is the
// bf16 pair (128 + q, 128 + q') exactly (bf16 has 7 fraction bits, so 128 + q
// is exact for q < 128), and one bf16x2 fma adding -(128 + z) leaves q - z
// exactly.  ncl, nch = -(128 + z) for rows gq and gq + 8 as bf16 pairs; mask
// and magic are 0x000F000F and 0x43004300 in registers, so that each
// extraction is one three-input logic operation.
template <bool FIRST>
__device__ __forceinline__ void chunk_mma(float (&d)[2][4], const uint4 &w, const uint4 &bl,
                                          const uint4 &bh, uint32_t ncl, uint32_t nch,
                                          const float (&zq)[4], uint32_t mask, uint32_t magic) {
    const uint32_t words[4] = {w.x, w.y, w.z, w.w};
    uint32_t r[4][4];
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        const uint32_t wd = words[v];
        r[0][v] = bf16x2_add(and_or(wd, mask, magic), ncl);
        r[1][v] = bf16x2_add(and_or(wd >> 4, mask, magic), ncl);
        r[2][v] = bf16x2_add(and_or(wd >> 8, mask, magic), nch);
        r[3][v] = bf16x2_add(and_or(wd >> 12, mask, magic), nch);
    }
    chunk_steps<FIRST, false>(d, r, bl, bh, zq);
}

// fp16 operands, zero point folded out: with magic 0x64006400 (fp16 1024),
// word & 0x000F000F | magic is (1024 + q, 1024 + q') and
// word & 0x00F000F0 | magic is (1024 + 16 q, 1024 + 16 q') (fp16 has 10
// fraction bits, so both are exact); the same for word >> 8.  One shift per
// word.  d[0] = sum (1024 + q) x over the chunk's steps 0, 1 and
// d[1] = sum (1024 + 16 q) x over steps 2, 3; x is fp16 here.
template <bool FIRST>
__device__ __forceinline__ void chunk_mma_half(float (&d)[2][4], const uint4 &w, const uint4 &bl,
                                               const uint4 &bh, const float (&zq)[4],
                                               uint32_t mask, uint32_t mask_hi, uint32_t magic) {
    const uint32_t words[4] = {w.x, w.y, w.z, w.w};
    uint32_t r[4][4];
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        const uint32_t wd = words[v], wd8 = words[v] >> 8;
        r[0][v] = and_or(wd, mask, magic);
        r[1][v] = and_or(wd, mask_hi, magic);
        r[2][v] = and_or(wd8, mask, magic);
        r[3][v] = and_or(wd8, mask_hi, magic);
    }
    chunk_steps<FIRST, true>(d, r, bl, bh, zq);
}

// What a consumer lane takes out of one stage: its two 16-byte weight pieces,
// the scale pair of its rows and their zero-point pair.
struct GroupData {
    uint4 w0, w1;
    uint32_t sp, zb;
};

__device__ __forceinline__ GroupData read_group(const unsigned char *st, int warp, int lane) {
    GroupData g;
    g.w0 = *reinterpret_cast<const uint4 *>(st + warp * 1024 + lane * 16);
    g.w1 = *reinterpret_cast<const uint4 *>(st + warp * 1024 + 512 + lane * 16);
    g.sp = *reinterpret_cast<const uint32_t *>(st + kRecWeights + warp * 32 + (lane >> 2) * 4);
    g.zb = st[kRecWeights + kRecScales + warp * 8 + (lane >> 2)];
    return g;
}

// This lane's B registers for one group: the x pairs 8tq .. 8tq+7 of each of
// the group's two 64-k chunks (xg points at word 8tq of the group's first
// chunk of the lane's token row).
struct GroupB {
    uint4 b0l, b0h, b1l, b1h;
};

__device__ __forceinline__ GroupB load_b(const uint32_t *xg) {
    const uint4 *bp = reinterpret_cast<const uint4 *>(xg);
    GroupB b;
    b.b0l = bp[0];
    b.b0h = bp[1];
    b.b1l = bp[8];
    b.b1h = bp[9];
    return b;
}

// One group (two 64-k chunks), bf16 operands q - z, into the lane's four fp32
// accumulators: acc += s * sum_group (q - z) x for its two rows and two
// token columns.
__device__ __forceinline__ void group_mma(float (&acc)[4], const GroupData &g, const GroupB &b,
                                          const float (&zq)[4], uint32_t mask, uint32_t magic) {
    // -(128 + z) as a bf16 pair, for rows gq and gq + 8
    const uint32_t ncl = ((g.zb & 0xFu) | 0xC300u) * 0x10001u;
    const uint32_t nch = ((g.zb >> 4) | 0xC300u) * 0x10001u;
    const float sl = __half2float(__ushort_as_half((unsigned short)(g.sp & 0xFFFFu)));
    const float sh = __half2float(__ushort_as_half((unsigned short)(g.sp >> 16)));
    float d[2][4];
    chunk_mma<true>(d, g.w0, b.b0l, b.b0h, ncl, nch, zq, mask, magic);
    chunk_mma<false>(d, g.w1, b.b1l, b.b1h, ncl, nch, zq, mask, magic);
    acc[0] = fmaf(d[0][0] + d[1][0], sl, acc[0]);
    acc[1] = fmaf(d[0][1] + d[1][1], sl, acc[1]);
    acc[2] = fmaf(d[0][2] + d[1][2], sh, acc[2]);
    acc[3] = fmaf(d[0][3] + d[1][3], sh, acc[3]);
}

// One group with fp16 operands and the zero point folded out of the inner
// product.  Over the group, d[0] = sum_{k in S01} (1024 + q) x and
// d[1] / 16 = sum_{k in S23} (64 + q) x, where S01 = {k : k mod 16 < 8} (the
// steps 0, 1 of every chunk) and S23 = {k : k mod 16 >= 8}; so
//   sum_k (q - z) x = d[0] + d[1] / 16 - (1024 + z) X01 - (64 + z) X23
// with X01, X23 the sums of x over S01 and S23.  xs = (X01 of token 2tq,
// X01 of 2tq + 1, X23 of 2tq, X23 of 2tq + 1).  Scaling by 1/16 is exact and
// (1024 + z) X, (64 + z) X are exact inside the fma.
__device__ __forceinline__ void group_mma_half_folded(float (&acc)[4], const GroupData &g,
                                                      const GroupB &b, float4 xs,
                                                      const float (&zq)[4], uint32_t mask,
                                                      uint32_t mask_hi, uint32_t magic) {
    // -(1024 + z) and -(64 + z) in fp32: 0xC4800000 is -1024 (z << 13 adds z),
    // 0xC2800000 is -64 (z << 17 adds z)
    const uint32_t zl = g.zb & 0xFu, zh = g.zb >> 4;
    const float n1l = __uint_as_float(0xC4800000u | (zl << 13));
    const float n1h = __uint_as_float(0xC4800000u | (zh << 13));
    const float n16l = __uint_as_float(0xC2800000u | (zl << 17));
    const float n16h = __uint_as_float(0xC2800000u | (zh << 17));
    const float sl = __half2float(__ushort_as_half((unsigned short)(g.sp & 0xFFFFu)));
    const float sh = __half2float(__ushort_as_half((unsigned short)(g.sp >> 16)));
    float d[2][4];
    chunk_mma_half<true>(d, g.w0, b.b0l, b.b0h, zq, mask, mask_hi, magic);
    chunk_mma_half<false>(d, g.w1, b.b1l, b.b1h, zq, mask, mask_hi, magic);
    acc[0] = fmaf(fmaf(n16l, xs.z, fmaf(n1l, xs.x, fmaf(d[1][0], 0.0625f, d[0][0]))), sl, acc[0]);
    acc[1] = fmaf(fmaf(n16l, xs.w, fmaf(n1l, xs.y, fmaf(d[1][1], 0.0625f, d[0][1]))), sl, acc[1]);
    acc[2] = fmaf(fmaf(n16h, xs.z, fmaf(n1h, xs.x, fmaf(d[1][2], 0.0625f, d[0][2]))), sh, acc[2]);
    acc[3] = fmaf(fmaf(n16h, xs.w, fmaf(n1h, xs.y, fmaf(d[1][3], 0.0625f, d[0][3]))), sh, acc[3]);
}

// The SwiGLU epilogue of the gate/up-interleaved layout: tile t holds gate
// rows 8t..8t+7 in its rows gq and the matching up rows in gq + 8, so the
// lane's acc[0], acc[2] (token 2tq) and acc[1], acc[3] (token 2tq + 1) are
// (gate, up) pairs of output j = 8t + gq: y[m][j] = silu(gate) * up in fp32.
template <bool F32OUT>
__device__ __forceinline__ void store_swiglu(void *yv, const float (&acc)[4], int t, int lane,
                                             int M, int I) {
    const int gq = lane >> 2, tq = lane & 3;
    const int j = 8 * t + gq;
    if (j >= I) return;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int m = 2 * tq + h;
        if (m < M) {
            const float g = acc[h], u = acc[2 + h];
            const float v = g / (1.f + expf(-g)) * u;
            const size_t o = (size_t)m * I + j;
            if (F32OUT)
                static_cast<float *>(yv)[o] = v;
            else
                static_cast<__nv_bfloat16 *>(yv)[o] = __float2bfloat16_rn(v);
        }
    }
}

template <bool F32OUT>
__device__ __forceinline__ void store_tile(void *yv, const float (&acc)[4], int t, int lane,
                                           int M, int N) {
    const int gq = lane >> 2, tq = lane & 3;
    const int r0 = t * kTileRows + gq, r1 = r0 + 8;
    const int m0 = 2 * tq, m1 = m0 + 1;
    const int ms[4] = {m0, m1, m0, m1};
    const int rs[4] = {r0, r0, r1, r1};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (ms[i] < M && rs[i] < N) {
            const size_t o = (size_t)ms[i] * N + rs[i];
            if (F32OUT)
                static_cast<float *>(yv)[o] = acc[i];
            else
                static_cast<__nv_bfloat16 *>(yv)[o] = __float2bfloat16_rn(acc[i]);
        }
    }
}


}  // namespace
}  // namespace w4
