// Device-side building blocks shared by the GEMV kernels (w4_gemv.cu,
// w4_gemv_sk.cu): PTX wrappers for mbarriers, bulk copies and programmatic
// dependent launch, the nibble-to-bf16 conversion and the tensor-core step.
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

// One 64-k chunk: four k-steps j; steps 0, 1 go to accumulator d[0] and steps
// 2, 3 to d[1] (two independent chains).  bl, bh hold this lane's eight B
// registers for the chunk: x pairs 8tq .. 8tq+7 of the chunk, register 2j
// for the step's first column pair and 2j+1 for its second (the permuted k
// order of w4_repack.cu).
// ncl, nch = -(128 + z) for rows gq and gq + 8 as bf16 pairs.  mask and magic
// are 0x000F000F and 0x43004300, passed in registers so that each extraction
// is one three-input logic operation.  FIRST: the accumulators start from zero.
// SUBZ: subtract 128 + z from every A register (A = q - z exactly); without
// it A = 128 + q and the caller removes (128 + z) * sum(x) per group.
template <bool FIRST, bool SUBZ = true>
__device__ __forceinline__ void chunk_mma(float (&d)[2][4], const uint4 &w, const uint4 &bl,
                                          const uint4 &bh, uint32_t ncl, uint32_t nch,
                                          const float (&zq)[4], uint32_t mask, uint32_t magic) {
    const uint32_t words[4] = {w.x, w.y, w.z, w.w};
    const uint32_t b[8] = {bl.x, bl.y, bl.z, bl.w, bh.x, bh.y, bh.z, bh.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t wd = words[j];
        uint32_t a0 = and_or(wd, mask, magic);
        uint32_t a1 = and_or(wd >> 4, mask, magic);
        uint32_t a2 = and_or(wd >> 8, mask, magic);
        uint32_t a3 = and_or(wd >> 12, mask, magic);
        if (SUBZ) {
            a0 = bf16x2_add(a0, ncl);
            a1 = bf16x2_add(a1, nch);
            a2 = bf16x2_add(a2, ncl);
            a3 = bf16x2_add(a3, nch);
        }
        if (FIRST && (j & 1) == 0)
            mma_bf16_16816_first(d[j >> 1], a0, a1, a2, a3, b[2 * j], b[2 * j + 1], zq);
        else
            mma_bf16_16816(d[j >> 1], a0, a1, a2, a3, b[2 * j], b[2 * j + 1]);
    }
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
// chunk of one token row, or at a zero patch).
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

// One group (two 64-k chunks) into the lane's four fp32 accumulators:
// acc += s * sum_group (q - z) x for its two rows and two token columns.
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

// group_mma with the zero point folded out of the inner product:
//   sum_k (q - z) x = sum_k (128 + q) x - (128 + z) * sum_k x,
// so the A registers are the extracted 128 + q as they are (no per-register
// subtraction) and each of the lane's four outputs takes one fp32 fma with
// xs = (sum of the group's x for token 2tq, for token 2tq + 1).  The
// product (128 + z) * sum_k x is exact inside the fma.
__device__ __forceinline__ void group_mma_folded(float (&acc)[4], const GroupData &g,
                                                 const GroupB &b, float2 xs,
                                                 const float (&zq)[4], uint32_t mask,
                                                 uint32_t magic) {
    // -(128 + z) in fp32: 0xC3000000 is -128, and z << 16 adds z to it.
    const float nzl = __uint_as_float(0xC3000000u | ((g.zb & 0xFu) << 16));
    const float nzh = __uint_as_float(0xC3000000u | ((g.zb >> 4) << 16));
    const float sl = __half2float(__ushort_as_half((unsigned short)(g.sp & 0xFFFFu)));
    const float sh = __half2float(__ushort_as_half((unsigned short)(g.sp >> 16)));
    float d[2][4];
    chunk_mma<true, false>(d, g.w0, b.b0l, b.b0h, 0u, 0u, zq, mask, magic);
    chunk_mma<false, false>(d, g.w1, b.b1l, b.b1h, 0u, 0u, zq, mask, magic);
    acc[0] = fmaf(fmaf(nzl, xs.x, d[0][0] + d[1][0]), sl, acc[0]);
    acc[1] = fmaf(fmaf(nzl, xs.y, d[0][1] + d[1][1]), sl, acc[1]);
    acc[2] = fmaf(fmaf(nzh, xs.x, d[0][2] + d[1][2]), sh, acc[2]);
    acc[3] = fmaf(fmaf(nzh, xs.y, d[0][3] + d[1][3]), sh, acc[3]);
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
