// w4_gemv: fused INT4-dequantise + matrix-vector product for sm_103a.
//
// Work split.  One thread block owns one row block (8 tiles of 16 rows, see
// w4_repack.cu) and one slice of K.  With `splits` > 1 the K slices of a row
// block are handled by the `splits` blocks of one thread-block cluster, which
// combine their fp32 partial sums through distributed shared memory in a fixed
// rank order: deterministic, no workspace, no float atomics ("qengine",
// section "Learnings": float atomics made one run in fifty differ; a fixed
// summation order fixed it).
//
// Streaming.  A producer warp moves the block's weights group by group
// (one 8 KB weight record + 256 B of scales + 64 B of zeros per group) into a
// ring of shared-memory stages with bulk asynchronous copies (cp.async.bulk,
// completion counted in bytes on an mbarrier), and the block's K slice of x
// once at the start.  Eight consumer warps (one per 16-row tile) wait on a
// stage's "full" barrier, copy their part of it into registers and release it
// on the stage's "empty" barrier, so the producer keeps kStages groups (51 KB
// per block) in flight: the copy engine, not per-thread loads,
// carries the bytes in flight that HBM needs.  This is the one-producer,
// several-consumers, transaction-counted-barrier arrangement of "Building an
// LLM Inference Runtime ...", section "Bug #1", applied to weight streaming.
//
// Per consumer warp and group.  The 16-byte piece a lane owns in each 64-k
// chunk holds four k-steps of its tensor-core A fragment, and each word
// becomes A registers without a conversion instruction.  Exact operand:
// (word >> 4p) & 0x000F000F | 0x43004300 is the bf16 pair (128 + q, 128 + q')
// exactly (bf16 has 7 fraction bits), and one bf16x2 fma adding -(128 + z)
// leaves q - z exactly; mma.m16n8k16 (bf16, fp32 accumulation) multiplies
// the 16 x 16 weight block with up to 8 token columns of x, the products
// (q - z) * x are exact, and acc += s * sum_group (q - z) x.  Folded (blocks
// of at least kFoldMinGroups groups): word & 0x000F000F and word & 0x00F000F0
// (and the same of word >> 8) OR 0x64006400 are the fp16 pairs (1024 + q) and
// (1024 + 16 q) exactly, one shift per word; x enters as fp16 scaled per
// token by a power of two, and the zero point is removed once per group and
// output through the group's half sums of x (group_mma_half_folded).  Token
// columns >= M read token 0's row and are never stored.
//
// Batch invariance ("qengine", section "How it works"): the K split and the
// arithmetic depend on K, N and the SM count only.  What else depends on M
// -- shared-memory residency, the persistent grid of several-wave products
// (one block per slot taking row blocks in turn), which of two x prologues
// runs -- changes who computes a tile, not how, so a token's result is the
// same for any M and any other tokens.
//
// Waits are bounded: a wait that exceeds ~2 s of clock cycles gives up, the
// block records the failure in the header's kernel_error word and skips the
// rest of its work; it never spins forever.
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>
#include <map>
#include <mutex>
#include <tuple>

#include "w4_device.cuh"

namespace cg = cooperative_groups;

namespace w4 {
namespace {

constexpr int kStageBytes = kRecWeights + kRecScales + kRecZeros;   // 8512
constexpr int kStages = 6;                          // shared-memory ring depth
constexpr int kStagesShort = 5;                     // ring depth that lets a third block fit
constexpr size_t kBlockSmemBudget = 113 * 1024;     // two blocks per SM
constexpr size_t kBlockSmemBudget3 = 74 * 1024;     // three blocks per SM
constexpr int kFoldMinGroups = 8;                   // see gemv_shape
constexpr size_t kOverlapBelowBytes = 16u << 20;    // packed weights of a "short" product
constexpr int kPersistMinTokens = 3;                // see plan_gemv
constexpr int kWideMinTokens = 5;                   // see plan_gemv
// Weight records a block requests before waiting for the previous kernel
// (programmatic dependent launch); fewer than any ring holds, so that those
// copies need no ring waits.
constexpr int kPreIssue = 2;
static_assert(kPreIssue < kStagesShort && kPreIssue < kStages, "pre-issued copies fit one round");

struct SmemPlan {
    size_t x_off, x_row_bytes, red_off, xsum_off, tok_off, bar_off, total;
};

// Shared memory: [stages][weights | scales | zeros] [x rows as copied]
// [partials] [per-group sums of x] [per-token maxima] [barriers]
__host__ __device__ inline SmemPlan smem_plan(int K, int S, int M, int stages) {
    const int G = K / kGroup;
    const int gmax = (G + S - 1) / S;
    SmemPlan p;
    p.x_off = (size_t)stages * kStageBytes;
    p.x_row_bytes = (size_t)gmax * kGroup * 2 + 16;      // +16 B: rows land on other banks
    p.red_off = p.x_off + (size_t)M * p.x_row_bytes;
    // Receive slots for the tiles this block reduces: ceil(8 / S) tiles, one
    // 512-byte partial from each of the S blocks of the cluster.
    p.xsum_off = p.red_off + (S > 1 ? (size_t)S * ((kWarps + S - 1) / S) * 32 * 16 : 0);
    p.tok_off = p.xsum_off + (size_t)gmax * 16 * 4;     // float [gmax][4 token pairs][4]
    p.bar_off = p.tok_off + 64;                         // uint32 [8] (+ padding)
    p.total = p.bar_off + (size_t)(2 * stages + 1) * 8 + 8;   // + the two constants
    return p;
}

// 2^e (or 2^-e for inverse) with e chosen so that 2^e times the bf16 value
// whose magnitude bits are maxbits lies in [2^14, 2^15) (e clamped to
// [-126, 126]): the scale of a token's slice of x that brings it into fp16
// range.  1 when the slice is all zero.
__device__ __forceinline__ float token_scale(uint32_t maxbits, bool inverse) {
    if (maxbits == 0) return 1.f;
    int e = 141 - (int)(maxbits >> 7);                  // 14 - (bf16 exponent - 127)
    e = e > 126 ? 126 : (e < -126 ? -126 : e);
    return __uint_as_float((uint32_t)((inverse ? -e : e) + 127) << 23);
}


// Final store of a tile: y = W x, or the SwiGLU of the interleaved pairs.
template <bool F32OUT>
__device__ __forceinline__ void store_out(void *yv, const float (&acc)[4], int t, int lane, int M,
                                          int N, int swiglu_I) {
    if (swiglu_I)
        store_swiglu<F32OUT>(yv, acc, t, lane, M, swiglu_I);
    else
        store_tile<F32OUT>(yv, acc, t, lane, M, N);
}

// Combine the K slices of a cluster in rank order 0, 1, ..., S-1 (all
// threads of every block of the cluster call this once, after their loop).
// Tile w is reduced by block w % S: every block first stores its partial of
// tile w into that block's receive slot (rank, w / S) through distributed
// shared memory, then one cluster barrier (release / acquire) makes all
// partials visible, and each reducing warp adds its S slots from its own
// shared memory.  No block reads another block's memory after the barrier,
// so none has to wait for the others before exiting.
template <bool F32OUT>
__device__ __forceinline__ void cluster_combine(float a0, float a1, float a2, float a3, void *yv,
                                             unsigned char *red_bytes, int t, int S, int split,
                                             int M, int N, int swiglu_I) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int J = (kWarps + S - 1) / S;                 // tiles reduced per block
    float4 *red = reinterpret_cast<float4 *>(red_bytes);
    cg::cluster_group cluster = cg::this_cluster();
    if (warp < kWarps) {
        float4 *dst = cluster.map_shared_rank(red, (unsigned)(warp % S));
        dst[(split * J + warp / S) * 32 + lane] = make_float4(a0, a1, a2, a3);
    }
    cluster.sync();
    if (warp < kWarps && (warp % S) == split) {
        float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
        for (int r = 0; r < S; ++r) {
            const float4 v = red[(r * J + warp / S) * 32 + lane];
            s0 += v.x;
            s1 += v.y;
            s2 += v.z;
            s3 += v.w;
        }
        const float tot[4] = {s0, s1, s2, s3};
        store_out<F32OUT>(yv, tot, t, lane, M, N, swiglu_I);
    }
}

// PERSIST (split S = 1 only): block c takes row blocks c, c + gridDim.x, ...
// in turn through one ring and one x prologue; otherwise block (b, split)
// takes row block b's K slice `split`.  WIDE (FOLD only): the x prologue's
// work is spread over (group, token) pairs (see plan_gemv for its use).
template <bool F32OUT, int MIN_BLOCKS, bool FOLD, int STAGES, bool PERSIST, bool WIDE>
__global__ void __launch_bounds__(kThreads, MIN_BLOCKS)
gemv_kernel(const char *__restrict__ qw, const char *__restrict__ sc,
            const char *__restrict__ zp, const __nv_bfloat16 *__restrict__ x,
            void *__restrict__ yv, uint32_t *err, int M, int K, int N, int S, int pre,
            int swiglu_I,
            uint32_t nib_mask, uint32_t bf16_magic) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int G = K / kGroup;
    const int b = blockIdx.x;
    const int split = blockIdx.y;
    const int g0 = (int)((long long)split * G / S);
    const int g1 = (int)((long long)(split + 1) * G / S);
    const int ng = g1 - g0;
    // units (row block, group) this block streams, row block by row block
    const int nrb = PERSIST ? (row_blocks(N) - b + (int)gridDim.x - 1) / (int)gridDim.x : 1;
    const int U = nrb * ng;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int kStages = STAGES;
    const SmemPlan plan = smem_plan(K, S, M, kStages);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + plan.bar_off);
    uint64_t *empty = full + kStages;
    uint64_t *xbar = empty + kStages;
    unsigned char *xs = smem + plan.x_off;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kWarps);
        }
        mbar_init(xbar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (FOLD && WIDE)   // per-token maxima of |x| (the prologue's atomicMax)
            for (int m = 0; m < W4_MAX_TOKENS; ++m)
                reinterpret_cast<uint32_t *>(smem + plan.tok_off)[m] = 0u;
        reinterpret_cast<uint32_t *>(xbar + 1)[0] = nib_mask;
        reinterpret_cast<uint32_t *>(xbar + 1)[1] = bf16_magic;
    }
    __syncthreads();

    bool ok = true;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    // A following launch that opted into programmatic dependent launch may
    // start its prologue (and its own weight copies) from here on.
    allow_dependents();
    if (warp == kWarps) {
        // ---- producer ----
        if (lane == 0) {
            // The weights do not depend on the previous kernel in the stream:
            // under programmatic dependent launch, request the first `pre`
            // groups before waiting for it; then x (which the consumers need
            // first), then the rest.  Launched normally (pre = 0), the wait
            // returns at once and x goes ahead of every weight copy.
            int issued = 0;
            int pb = b, ps = 0;                     // row block and group of the next unit
            const int first = U < pre ? U : pre;    // < kStages: no ring waits needed
            for (int s = 0; s < first; ++s) {
                unsigned char *st = smem + s * kStageBytes;
                const size_t rec = PERSIST ? (size_t)pb * G + g0 + ps : (size_t)b * G + g0 + s;
                if (PERSIST && ++ps == ng) {
                    ps = 0;
                    pb += (int)gridDim.x;
                }
                mbar_expect_tx(&full[s], kStageBytes);
                bulk_g2s(st, qw + W4_HEADER_BYTES + rec * kRecWeights, kRecWeights, &full[s]);
                bulk_g2s(st + kRecWeights, sc + rec * kRecScales, kRecScales, &full[s]);
                bulk_g2s(st + kRecWeights + kRecScales, zp + rec * kRecZeros, kRecZeros,
                         &full[s]);
                ++issued;
            }
            wait_prerequisites();
            mbar_expect_tx(xbar, (uint32_t)(M * ng * kGroup * 2));
            for (int m = 0; m < M; ++m)
                bulk_g2s(xs + m * plan.x_row_bytes, x + (size_t)m * K + (size_t)g0 * kGroup,
                         (uint32_t)(ng * kGroup * 2), xbar);
            uint32_t phase = 0;                     // round of the ring, mod 2
            for (int base = 0; base < U && ok; base += kStages) {
#pragma unroll
                for (int i = 0; i < kStages; ++i) {
                    const int s = base + i;
                    if (s >= first && s < U && ok) {
                        if (base > 0 && !mbar_wait(&empty[i], phase ^ 1u)) {
                            ok = false;
                        } else {
                            if (base > 0) fence_proxy_async();
                            unsigned char *st = smem + i * kStageBytes;
                            const size_t rec =
                                PERSIST ? (size_t)pb * G + g0 + ps : (size_t)b * G + g0 + s;
                            if (PERSIST && ++ps == ng) {
                                ps = 0;
                                pb += (int)gridDim.x;
                            }
                            mbar_expect_tx(&full[i], kStageBytes);
                            bulk_g2s(st, qw + W4_HEADER_BYTES + rec * kRecWeights, kRecWeights,
                                     &full[i]);
                            bulk_g2s(st + kRecWeights, sc + rec * kRecScales, kRecScales,
                                     &full[i]);
                            bulk_g2s(st + kRecWeights + kRecScales, zp + rec * kRecZeros,
                                     kRecZeros, &full[i]);
                            ++issued;
                        }
                    }
                }
                phase ^= 1u;
            }
            if (!ok) {
                // Give the copies already issued a bounded chance to land before exit.
                for (int s = issued > kStages ? issued - kStages : 0; s < issued; ++s)
                    mbar_wait(&full[s % kStages], (s / kStages) & 1);
                atomicOr(err, 1u);
            }
        }
    } else {
        // ---- consumers: warp w owns tile 8b + w ----
        const int gq = lane >> 2, tq = lane & 3;
        // Fold only: per group and token X01, X23 (float [gmax][4 token
        // pairs][4]), and per token the largest |x| of the slice (bf16 bits).
        // Sums of tokens >= M are never written: the accumulators they feed
        // belong to token columns that are not stored.
        float *xsum = reinterpret_cast<float *>(smem + plan.xsum_off);
        uint32_t *tok_max = reinterpret_cast<uint32_t *>(smem + plan.tok_off);
        if (FOLD && !WIDE) {
            // sums of tokens >= M stay zero; maxima start at zero
            for (int i = threadIdx.x; i < ng * 16; i += kWarps * 32) xsum[i] = 0.f;
            if (threadIdx.x < W4_MAX_TOKENS) tok_max[threadIdx.x] = 0u;
            consumer_sync();
        }
        // x is used as copied: the kernel layout orders k inside each 64-k chunk
        // so that lane tq's eight B registers are the x pairs at
        // 64c + 16tq .. 64c + 16tq + 15 (see w4_repack.cu).
        // Token columns gq >= M read token 0's row: column n of a tensor-core
        // product depends on column n of B alone, and those columns are never
        // stored.
        const uint32_t *xrow =
            reinterpret_cast<const uint32_t *>(xs + (size_t)(gq < M ? gq : 0) * plan.x_row_bytes) +
            tq * 8;    // words 8tq .. 8tq+7 of each 32-word chunk
        const float zq[4] = {0.f, 0.f, 0.f, 0.f};
        // The conversion constants, read from shared memory so that they sit
        // in ordinary registers: left as kernel parameters, the compiler may
        // keep them in uniform registers, and a three-input logic operation
        // takes only one of those, which costs a register move per extraction.
        const uint32_t mask = reinterpret_cast<volatile uint32_t *>(xbar + 1)[0];
        const uint32_t magic = reinterpret_cast<volatile uint32_t *>(xbar + 1)[1];
        const uint32_t mask_hi = mask << 4;
        // Sleep (no polling) until the previous kernel in the stream is done:
        // x may be its output, and a block launched early must not take issue
        // slots from that kernel's still-running blocks.
        wait_prerequisites();
        {
            // Every consumer thread takes part in the barriers below even if
            // its wait gave up.
            const bool x_ok = mbar_wait(xbar, 0);
            if constexpr (FOLD && WIDE) {
                // The folded product runs on fp16 operands: x is scaled per
                // token by a power of two 2^e (exact) that brings the largest
                // |x| of the token's slice into [2^14, 2^15), then rounded to
                // fp16 in place; per group and token the two sums X01
                // (k mod 16 < 8) and X23 (k mod 16 >= 8) of the scaled values
                // feed the zero-point term of group_mma_half_folded (the fp16
                // values equal them except below the fp16 normal range, 2^28
                // under the token's largest).  The fp32 arithmetic is fixed:
                // per 16-aligned block of the group and half (first or last
                // eight values), the values at even and at odd positions are
                // summed left to right in two packed lanes and the two lane
                // sums added; then over the eight blocks the pairwise tree
                // ((p0+p1)+(p2+p3))+((p4+p5)+(p6+p7)).  Only the assignment
                // of that work to threads depends on the number of (group,
                // token) pairs: tpp threads per pair, each with per = 8 / tpp
                // consecutive blocks, joined by shuffles that follow the same
                // tree.  (The wide prologue; the narrow one below takes the
                // maxima token by token.  Both compute the same numbers.)
                const int pairs = ng * M;
                int tpp = 8;
                while (tpp > 1 && pairs * tpp > kWarps * 32) tpp >>= 1;
                const int per = 8 / tpp;
                // (1) the largest magnitude of each token's slice, as bf16 bits
                // (whose integer order is the order of the magnitudes)
                if (x_ok) {
                    for (int base = 0; base < pairs * tpp; base += kWarps * 32) {
                        const int idx = base + (int)threadIdx.x;
                        const int pair = idx / tpp, sub = idx - pair * tpp;
                        const bool live = pair < pairs;
                        const int gl = live ? pair / M : 0, m = live ? pair - gl * M : 0;
                        const uint4 *blk = reinterpret_cast<const uint4 *>(
                            xs + (size_t)m * plan.x_row_bytes + (size_t)gl * kGroup * 2 +
                            (size_t)sub * per * 32);
                        uint32_t mx2 = 0u;              // two 16-bit maxima
                        if (live) {
#pragma unroll
                            for (int j = 0; j < 2 * per; ++j) {
                                const uint4 v = blk[j];
                                mx2 = __vmaxu2(mx2, v.x & 0x7FFF7FFFu);
                                mx2 = __vmaxu2(mx2, v.y & 0x7FFF7FFFu);
                                mx2 = __vmaxu2(mx2, v.z & 0x7FFF7FFFu);
                                mx2 = __vmaxu2(mx2, v.w & 0x7FFF7FFFu);
                            }
                        }
                        uint32_t mx = max(mx2 & 0xFFFFu, mx2 >> 16);
                        for (int o = 1; o < tpp; o <<= 1)
                            mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
                        if (sub == 0 && live && mx) atomicMax(&tok_max[m], mx);
                    }
                }
                consumer_sync();
                // (2) scale, convert in place, sum
                if (x_ok) {
                    for (int base = 0; base < pairs * tpp; base += kWarps * 32) {
                        const int idx = base + (int)threadIdx.x;
                        const int pair = idx / tpp, sub = idx - pair * tpp;
                        const bool live = pair < pairs;
                        const int gl = live ? pair / M : 0, m = live ? pair - gl * M : 0;
                        uint4 *blk = reinterpret_cast<uint4 *>(
                            xs + (size_t)m * plan.x_row_bytes + (size_t)gl * kGroup * 2 +
                            (size_t)sub * per * 32);
                        float v01 = 0.f, v23 = 0.f;
                        if (live) {
                            const float sc = token_scale(tok_max[m], false);
                            const unsigned long long sc2 =
                                ((unsigned long long)__float_as_uint(sc) << 32) | __float_as_uint(sc);
                            float l01[3], l23[3];   // pending subtree sums, levels 0..2
#pragma unroll
                            for (int j = 0; j < per; ++j) {
                                const uint4 u0 = blk[2 * j], u1 = blk[2 * j + 1];
                                const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w,
                                                       u1.x, u1.y, u1.z, u1.w};
                                uint32_t h[8];
                                unsigned long long a01 = 0ull, a23 = 0ull;
#pragma unroll
                                for (int e = 0; e < 8; ++e) {
                                    // the pair as fp32 (bf16 is the top half of fp32), scaled
                                    const unsigned long long f = f32x2_mul(
                                        ((unsigned long long)(w[e] & 0xFFFF0000u) << 32) |
                                            (unsigned long long)(w[e] << 16),
                                        sc2);
                                    const __half2 hv = __floats2half2_rn(f32x2_lo(f), f32x2_hi(f));
                                    h[e] = *reinterpret_cast<const uint32_t *>(&hv);
                                    if (e < 4)
                                        a01 = e == 0 ? f : f32x2_add(a01, f);
                                    else
                                        a23 = e == 4 ? f : f32x2_add(a23, f);
                                }
                                blk[2 * j] = make_uint4(h[0], h[1], h[2], h[3]);
                                blk[2 * j + 1] = make_uint4(h[4], h[5], h[6], h[7]);
                                // leaf j of the pairwise tree over this thread's
                                // blocks; after the last leaf v is the subtree
                                v01 = f32x2_lo(a01) + f32x2_hi(a01);
                                v23 = f32x2_lo(a23) + f32x2_hi(a23);
                                if (j & 1) {
                                    v01 = l01[0] + v01;
                                    v23 = l23[0] + v23;
                                    if (j & 2) {
                                        v01 = l01[1] + v01;
                                        v23 = l23[1] + v23;
                                        if (j & 4) {
                                            v01 = l01[2] + v01;
                                            v23 = l23[2] + v23;
                                        } else {
                                            l01[2] = v01;
                                            l23[2] = v23;
                                        }
                                    } else {
                                        l01[1] = v01;
                                        l23[1] = v23;
                                    }
                                } else {
                                    l01[0] = v01;
                                    l23[0] = v23;
                                }
                            }
                        }
                        // the pair's tpp subtrees
                        for (int o = 1; o < tpp; o <<= 1) {
                            v01 += __shfl_xor_sync(0xFFFFFFFFu, v01, o);
                            v23 += __shfl_xor_sync(0xFFFFFFFFu, v23, o);
                        }
                        if (sub == 0 && live) {
                            float *xg = xsum + gl * 16 + (m >> 1) * 4 + (m & 1);
                            xg[0] = v01;
                            xg[2] = v23;
                        }
                    }
                }
                consumer_sync();
            }
            if constexpr (FOLD && !WIDE) {
                // The folded product runs on fp16 operands: x is scaled per
                // token by a power of two (exact) into fp16 range.  (1) The
                // largest |x| of each token's slice, as bf16 magnitude bits
                // (whose integer order is the order of the values).
                if (x_ok) {
                    for (int m = 0; m < M; ++m) {
                        const uint4 *row =
                            reinterpret_cast<const uint4 *>(xs + (size_t)m * plan.x_row_bytes);
                        uint32_t mx2 = 0u;              // two 16-bit maxima
                        for (int i = threadIdx.x; i < ng * 16; i += kWarps * 32) {
                            const uint4 v = row[i];
                            mx2 = __vmaxu2(mx2, v.x & 0x7FFF7FFFu);
                            mx2 = __vmaxu2(mx2, v.y & 0x7FFF7FFFu);
                            mx2 = __vmaxu2(mx2, v.z & 0x7FFF7FFFu);
                            mx2 = __vmaxu2(mx2, v.w & 0x7FFF7FFFu);
                        }
                        const uint32_t mx =
                            __reduce_max_sync(0xFFFFFFFFu, max(mx2 & 0xFFFFu, mx2 >> 16));
                        if (lane == 0 && mx) atomicMax(&tok_max[m], mx);
                    }
                }
                consumer_sync();
                // (2) x -> fp16 (scaled, rounded to nearest), in place, and per
                // group and token the two sums X01 (k mod 16 < 8) and X23
                // (k mod 16 >= 8) of the scaled values for the zero-point term
                // of group_mma_half_folded (the fp16 values equal them except
                // below the fp16 normal range, 2^28 under the token's largest).
                // The fp32 arithmetic is fixed: per 16-aligned block of the
                // group and half (first or last eight values), the values at
                // even and at odd positions are summed left to right in two
                // packed lanes and the two lane sums added; then over the
                // eight blocks the pairwise tree ((p0+p1)+(p2+p3))+((p4+p5)+
                // (p6+p7)).  Only the assignment of that work to threads
                // depends on the number of (group, token) pairs: tpp threads
                // per pair, each with 8 / tpp blocks, joined by shuffles that
                // follow the same tree.
                if (x_ok) {
                    const int pairs = ng * M;
                    int tpp = 8;
                    while (tpp > 1 && pairs * tpp > kWarps * 32) tpp >>= 1;
                    const int per = 8 / tpp;
                    for (int base = 0; base < pairs * tpp; base += kWarps * 32) {
                        const int idx = base + (int)threadIdx.x;
                        const int pair = idx / tpp, sub = idx - pair * tpp;
                        const int gl = pair / M, m = pair - gl * M;
                        float p01[8], p23[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) p01[j] = p23[j] = 0.f;
                        if (pair < pairs) {
                            const float sc = token_scale(tok_max[m], false);
                            const unsigned long long sc2 =
                                ((unsigned long long)__float_as_uint(sc) << 32) | __float_as_uint(sc);
                            uint4 *blk = reinterpret_cast<uint4 *>(
                                xs + (size_t)m * plan.x_row_bytes + (size_t)gl * kGroup * 2 +
                                (size_t)sub * per * 32);
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                if (j < per) {
                                    const uint4 u0 = blk[2 * j], u1 = blk[2 * j + 1];
                                    const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w,
                                                           u1.x, u1.y, u1.z, u1.w};
                                    uint32_t h[8];
                                    unsigned long long a01 = 0ull, a23 = 0ull;
#pragma unroll
                                    for (int e = 0; e < 8; ++e) {
                                        // the pair as fp32 (bf16 is the top half of fp32),
                                        // scaled
                                        const unsigned long long f = f32x2_mul(
                                            ((unsigned long long)(w[e] & 0xFFFF0000u) << 32) |
                                                (unsigned long long)(w[e] << 16),
                                            sc2);
                                        const __half2 v = __floats2half2_rn(f32x2_lo(f), f32x2_hi(f));
                                        h[e] = *reinterpret_cast<const uint32_t *>(&v);
                                        if (e < 4)
                                            a01 = e == 0 ? f : f32x2_add(a01, f);
                                        else
                                            a23 = e == 4 ? f : f32x2_add(a23, f);
                                    }
                                    blk[2 * j] = make_uint4(h[0], h[1], h[2], h[3]);
                                    blk[2 * j + 1] = make_uint4(h[4], h[5], h[6], h[7]);
                                    p01[j] = f32x2_lo(a01) + f32x2_hi(a01);
                                    p23[j] = f32x2_lo(a23) + f32x2_hi(a23);
                                }
                            }
                        }
                        // this thread's subtree over its `per` blocks, then the
                        // shuffles over the pair's tpp threads
                        if (per >= 2) {
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                if (2 * j + 1 < per) {
                                    p01[2 * j] = p01[2 * j] + p01[2 * j + 1];
                                    p23[2 * j] = p23[2 * j] + p23[2 * j + 1];
                                }
                            }
                        }
                        if (per >= 4) {
                            p01[0] = p01[0] + p01[2];
                            p23[0] = p23[0] + p23[2];
                            if (per == 8) {
                                p01[4] = p01[4] + p01[6];
                                p23[4] = p23[4] + p23[6];
                            }
                        }
                        if (per == 8) {
                            p01[0] = p01[0] + p01[4];
                            p23[0] = p23[0] + p23[4];
                        }
                        float v01 = p01[0], v23 = p23[0];
                        for (int o = 1; o < tpp; o <<= 1) {
                            v01 += __shfl_xor_sync(0xFFFFFFFFu, v01, o);
                            v23 += __shfl_xor_sync(0xFFFFFFFFu, v23, o);
                        }
                        if (sub == 0 && pair < pairs) {
                            float *xg = xsum + gl * 16 + (m >> 1) * 4 + (m & 1);
                            xg[0] = v01;
                            xg[2] = v23;
                        }
                    }
                }
                consumer_sync();
            }
            if (!x_ok) goto consumer_failed;
        }
        {
            // (X01, X01, X23, X23) of tokens 2tq, 2tq+1 for each group
            const float4 *xs4 = reinterpret_cast<const float4 *>(xsum) + tq;
            uint32_t phase = 0;                 // round of the ring, mod 2
            int s = 0;
            if constexpr (PERSIST) {
                // the per-token scale of x, undone on each row block's
                // accumulators before its store (a power of two: exact)
                float us0 = 1.f, us1 = 1.f;
                if constexpr (FOLD) {
                    if (2 * tq < M) us0 = token_scale(tok_max[2 * tq], true);
                    if (2 * tq + 1 < M) us1 = token_scale(tok_max[2 * tq + 1], true);
                }
                int gi = 0;                     // group of the unit in its row block
                int rb = b;                     // the unit's row block
                auto unit = [&](int i) {
                    const GroupData g = read_group(smem + i * kStageBytes, warp, lane);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[i]);   // stage copied to registers
                    if constexpr (FOLD)
                        group_mma_half_folded(acc, g, load_b(xrow + gi * 64), xs4[gi * 4], zq,
                                              mask, mask_hi, magic);
                    else
                        group_mma(acc, g, load_b(xrow + gi * 64), zq, mask, magic);
                    if (++gi == ng) {           // row block rb done: store it
                        gi = 0;
                        acc[0] *= us0;
                        acc[1] *= us1;
                        acc[2] *= us0;
                        acc[3] *= us1;
                        store_out<F32OUT>(yv, acc, rb * kWarps + warp, lane, M, N, swiglu_I);
                        acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
                        rb += (int)gridDim.x;
                    }
                };
                for (; s + kStages <= U; s += kStages) {
#pragma unroll
                    for (int i = 0; i < kStages; ++i) {
                        if (!mbar_wait(&full[i], phase)) goto consumer_failed;
                        unit(i);
                    }
                    phase ^= 1u;
                }
#pragma unroll
                for (int i = 0; i < kStages - 1; ++i) {
                    if (s + i < U) {
                        if (!mbar_wait(&full[i], phase)) goto consumer_failed;
                        unit(i);
                    }
                }
            } else {
                for (; s + kStages <= ng; s += kStages) {
#pragma unroll
                    for (int i = 0; i < kStages; ++i) {
                        if (!mbar_wait(&full[i], phase)) goto consumer_failed;
                        const GroupData g = read_group(smem + i * kStageBytes, warp, lane);
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&empty[i]);   // stage copied to registers
                        if constexpr (FOLD)
                            group_mma_half_folded(acc, g, load_b(xrow + (s + i) * 64),
                                                  xs4[(s + i) * 4], zq, mask, mask_hi, magic);
                        else
                            group_mma(acc, g, load_b(xrow + (s + i) * 64), zq, mask, magic);
                    }
                    phase ^= 1u;
                }
#pragma unroll
                for (int i = 0; i < kStages - 1; ++i) {
                    if (s + i < ng) {
                        if (!mbar_wait(&full[i], phase)) goto consumer_failed;
                        const GroupData g = read_group(smem + i * kStageBytes, warp, lane);
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&empty[i]);
                        if constexpr (FOLD)
                            group_mma_half_folded(acc, g, load_b(xrow + (s + i) * 64),
                                                  xs4[(s + i) * 4], zq, mask, mask_hi, magic);
                        else
                            group_mma(acc, g, load_b(xrow + (s + i) * 64), zq, mask, magic);
                    }
                }
            }
        }
        if constexpr (FOLD && !PERSIST) {
            // undo the per-token scale of x (a power of two: exact)
            const int m0 = 2 * tq, m1 = m0 + 1;
            const float u0 = m0 < M ? token_scale(tok_max[m0], true) : 1.f;
            const float u1 = m1 < M ? token_scale(tok_max[m1], true) : 1.f;
            acc[0] *= u0;
            acc[1] *= u1;
            acc[2] *= u0;
            acc[3] *= u1;
        }
        goto consumer_done;
    consumer_failed:
        ok = false;
    consumer_done:
        if (!ok && lane == 0) atomicOr(err, 1u);
    }

    if constexpr (PERSIST) return;       // stored row block by row block
    wait_prerequisites();       // y may be read by the previous kernel in the stream
    const int t = b * kWarps + warp;
    if (S == 1) {
        if (warp < kWarps && ok) store_out<F32OUT>(yv, acc, t, lane, M, N, swiglu_I);
        return;
    }
    cluster_combine<F32OUT>(acc[0], acc[1], acc[2], acc[3], yv, smem + plan.red_off, t, S, split,
                            M, N, swiglu_I);
}

}  // namespace

bool gemv_shape(int K, int N, int num_sms, GemvShape *out) {
    const int NB = row_blocks(N);
    const int G = K / kGroup;
    const long long slots = 2LL * (num_sms > 0 ? num_sms : 1);
    const int fill = 2;          // start-up cost of a block, in groups
    // Cluster sizes 3, 5 and 7 measured slower than their neighbours on
    // GB300 (clusters of those sizes pack unevenly onto the SMs of a GPC).
    static const int kCandidates[] = {1, 2, 4, 6, 8};
    int best_s = 0;
    long long best_cost = 0;
    for (int S : kCandidates) {
        if (S > G || S > kMaxSplits) continue;
        if (smem_plan(K, S, W4_MAX_TOKENS, kStages).total > kBlockSmemBudget) continue;
        const long long ctas = (long long)NB * S;
        // A clustered grid counts as one wave only with 10% of the slots to
        // spare, as in plan_gemv (beyond that it runs uncapped and slower).
        const long long waves =
            S == 1 ? (ctas + slots - 1) / slots : (ctas * 11 + slots * 10 - 1) / (slots * 10);
        const long long cost = waves * ((G + S - 1) / S + fill);
        if (best_s == 0 || cost <= best_cost) {
            best_s = S;
            best_cost = cost;
        }
    }
    if (best_s == 0) return false;
    out->warps = kWarps;
    out->splits = best_s;
    out->stages = kStages;
    // Fold the zero point out of the inner product when a block streams at
    // least kFoldMinGroups groups: it saves the per-weight subtraction but
    // adds a prologue (the group sums of x) that short blocks cannot hide.
    out->fold = (G + best_s - 1) / best_s >= kFoldMinGroups;
    return true;
}

namespace {

struct DeviceSmem {
    int per_sm = 0, reserved = 0, optin = 0;
};

// Shared memory per SM, reserved per block and the opt-in maximum per block
// of device `dev`, read once.
const DeviceSmem &device_smem(int dev) {
    static DeviceSmem cache[64];
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    DeviceSmem &d = cache[dev];
    if (d.per_sm == 0) {
        cudaDeviceGetAttribute(&d.per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
        cudaDeviceGetAttribute(&d.reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
        cudaDeviceGetAttribute(&d.optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    }
    return d;
}

// Clusters of this launch configuration that can be resident at once, cached.
int active_clusters(const void *kern, cudaLaunchConfig_t cfg, int dev) {
    static std::mutex mu;
    static std::map<std::tuple<const void *, size_t, unsigned, int>, int> cache;
    const auto key = std::make_tuple(kern, cfg.dynamicSmemBytes, cfg.gridDim.y, dev);
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
    }
    std::lock_guard<std::mutex> lock(mu);
    cache[key] = n;
    return n;
}

// Blocks of `kern` with `smem` bytes of dynamic shared memory resident per
// SM, cached.
int resident_blocks(const void *kern, size_t smem, int dev) {
    static std::mutex mu;
    static std::map<std::tuple<const void *, size_t, int>, int> cache;
    const auto key = std::make_tuple(kern, smem, dev);
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kThreads, smem) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
    }
    cache[key] = n;
    return n;
}

}  // namespace

namespace {

using Kern = void (*)(const char *, const char *, const char *, const __nv_bfloat16 *, void *,
                      uint32_t *, int, int, int, int, int, int, uint32_t, uint32_t);

// [f32 out][variant][arithmetic][persistent]; variant 0: two blocks per SM,
// 6 stages; 1: three, 6; 2: three, 5; arithmetic 0: exact q - z, 1: folded,
// 2: folded with the wide x prologue
#define W4_GEMV_KERNELS(F, MB, ST)                                                        \
    {{gemv_kernel<F, MB, false, ST, false, false>, gemv_kernel<F, MB, false, ST, true, false>}, \
     {gemv_kernel<F, MB, true, ST, false, false>, gemv_kernel<F, MB, true, ST, true, false>},   \
     {gemv_kernel<F, MB, true, ST, false, true>, gemv_kernel<F, MB, true, ST, true, true>}}
const Kern kKernels[2][3][3][2] = {
    {W4_GEMV_KERNELS(false, 2, kStages), W4_GEMV_KERNELS(false, 3, kStages),
     W4_GEMV_KERNELS(false, 3, kStagesShort)},
    {W4_GEMV_KERNELS(true, 2, kStages), W4_GEMV_KERNELS(true, 3, kStages),
     W4_GEMV_KERNELS(true, 3, kStagesShort)}};
#undef W4_GEMV_KERNELS
const int kVariantStages[3] = {kStages, kStages, kStagesShort};

// Raise a kernel's dynamic shared memory limit to the device's opt-in
// maximum, once per (kernel, device).  The flag is atomic: host threads that
// race on a first call both set the attribute, which is idempotent.
cudaError_t prepare_kernel(int f32_out, int v, int arith, int pers, int dev, int optin) {
    static std::atomic<bool> done[2][3][3][2][64] = {};
    std::atomic<bool> &flag = done[f32_out][v][arith][pers][dev];
    if (flag.load(std::memory_order_acquire)) return cudaSuccess;
    const cudaError_t r = cudaFuncSetAttribute(kKernels[f32_out][v][arith][pers],
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
    if (r == cudaSuccess) flag.store(true, std::memory_order_release);
    return r;
}

}  // namespace

cudaError_t plan_gemv(bool f32_out, int M, int K, int N, const GemvShape &shape, int num_sms,
                      GemvLaunch *out) {
    const int S = shape.splits;
    const long long blocks = (long long)row_blocks(N) * S;
    const int sms = num_sms > 0 ? num_sms : 1;
    const int need = blocks <= sms ? 1 : blocks <= 2LL * sms ? 2 : 3;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    const DeviceSmem &ds = device_smem(dev);
    int arith = shape.fold ? 1 : 0;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)row_blocks(N), (unsigned)S, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cudaLaunchAttribute attr[1];
    if (S > 1) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1;
        attr[0].val.clusterDim.y = (unsigned)S;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }

    // Residency.  A grid of one wave runs as long as its most loaded SM, so
    // it should spread evenly: at most ceil(blocks / SMs) blocks per SM.
    // Programmatic dependent launch starts blocks early in whatever slots
    // the previous kernel leaves free; with room for three blocks per SM
    // they stack up unevenly, so a grid that needs at most two per SM asks
    // for enough shared memory that no more than that fit ("capped").  It
    // then also overlaps its start with the previous kernel's end.  Grids
    // that need three per SM launch without overlap (unless short); grids of
    // several waves always overlap.  A block whose own shared memory
    // already keeps a third one off the SM counts as capped as it stands.
    // Ring depth: three blocks per SM (more warps to hide the prologue and
    // memory latency) where x's slice leaves room for them, with a ring of
    // six stages or else five; otherwise two blocks with six.  (A ring of
    // twelve stages in half an SM measured slower at M = 1.)  The split S,
    // and so the arithmetic, is the same whichever runs.
    auto capped_smem = [&](const Kern kern, size_t total) -> size_t {
        // shared memory that caps the grid at `need` blocks per SM, or 0
        if (need >= 3 || ds.per_sm <= 0) return 0;
        const size_t pad = (size_t)(ds.per_sm / (need + 1) - ds.reserved + 16) / 16 * 16;
        const size_t want = pad > total ? pad : total;
        if (want > (size_t)ds.optin || want + (size_t)ds.reserved > (size_t)(ds.per_sm / need))
            return 0;
        cudaLaunchConfig_t probe = cfg;
        probe.dynamicSmemBytes = want;
        // With clusters, only where the grid stays one wave with 10% of the
        // cluster slots to spare: clusters are placed whole, within one GPC,
        // and a grid that only just fits measured slower capped.
        if (S > 1 &&
            (long long)active_clusters((const void *)kern, probe, dev) * S * 10 < blocks * 11)
            return 0;
        return want;
    };
    const int variant = smem_plan(K, S, M, kStages).total <= kBlockSmemBudget3        ? 1
                        : smem_plan(K, S, M, kStagesShort).total <= kBlockSmemBudget3 ? 2
                                                                                      : 0;
    if ((e = prepare_kernel(f32_out, variant, arith, 0, dev, ds.optin)) != cudaSuccess) return e;
    size_t smem_bytes = smem_plan(K, S, M, kVariantStages[variant]).total;
    bool capped = false;
    {
        const size_t c = capped_smem(kKernels[f32_out][variant][arith][0], smem_bytes);
        if (c > 0) {
            smem_bytes = c;
            capped = true;
        }
    }
    // A grid of several waves without clusters runs persistent from three
    // tokens on: one block per resident slot, each taking row blocks in
    // turn, so that the x prologue (which grows with M) and the ring's
    // start-up are paid once per slot rather than once per row block.  With
    // fewer tokens the prologue is short and the hardware's dynamic
    // assignment of row blocks to free slots measured faster.  The
    // arithmetic of a row block is the same either way.
    int pers = 0;
    if (S == 1 && M >= kPersistMinTokens) {
        if ((e = prepare_kernel(f32_out, variant, arith, 1, dev, ds.optin)) != cudaSuccess)
            return e;
        const int per_sm = resident_blocks((const void *)kKernels[f32_out][variant][arith][1],
                                           smem_bytes, dev);
        if (per_sm > 0 && blocks > (long long)per_sm * sms) {
            pers = 1;
            cfg.gridDim.x = (unsigned)(per_sm * sms);
        }
    }
    // The folded product's x prologue: from five tokens on, one-wave grids
    // spread it over (group, token) pairs (faster there by 2-11 % at M = 5-8);
    // with fewer tokens, and in persistent grids (which run it once per
    // slot), the token-by-token prologue measured faster.
    if (arith == 1 && !pers && M >= kWideMinTokens) {
        arith = 2;
        if ((e = prepare_kernel(f32_out, variant, arith, 0, dev, ds.optin)) != cudaSuccess)
            return e;
    }
    out->shape = shape;
    out->variant = variant;
    out->arith = arith;
    out->persistent = pers != 0;
    out->capped = capped;
    out->overlap = capped || (size_t)K * (size_t)N / 2 < kOverlapBelowBytes || blocks > 3LL * sms;
    out->grid = cfg.gridDim;
    out->smem_bytes = smem_bytes;
    out->stages = kVariantStages[variant];
    return cudaSuccess;
}

cudaError_t launch_gemv(const void *qweight, const void *scales, const void *zeros,
                        const uint16_t *x, void *y, bool f32_out, int M, int K, int N,
                        const GemvShape &shape, int swiglu_I, int num_sms,
                        cudaStream_t stream) {
    GemvLaunch L;
    cudaError_t e = plan_gemv(f32_out, M, K, N, shape, num_sms, &L);
    if (e != cudaSuccess) return e;
    const int S = shape.splits;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = L.grid;
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = L.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (S > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = 1;
        attr[na].val.clusterDim.y = (unsigned)S;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (L.overlap) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    const Kern kern = kKernels[f32_out][L.variant][L.arith][L.persistent ? 1 : 0];
    const char *q = static_cast<const char *>(qweight);
    // The kernel's one write outside y: the header's kernel-error word, set
    // only when a wait inside the kernel gives up.
    uint32_t *err = reinterpret_cast<uint32_t *>(const_cast<char *>(q) + kErrorOffset);
    return cudaLaunchKernelEx(&cfg, kern, q, static_cast<const char *>(scales),
                              static_cast<const char *>(zeros),
                              reinterpret_cast<const __nv_bfloat16 *>(x), y, err, M, K, N, S,
                              L.overlap ? kPreIssue : 0, swiglu_I, 0x000F000Fu,
                              shape.fold ? 0x64006400u : 0x43004300u);
}

}  // namespace w4
