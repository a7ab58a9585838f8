/*
 * w4.h -- C ABI of libw4: weight-only INT4 (group 128) matrix-vector product
 * y = W x on one NVIDIA GB300 (sm_103a).
 *
 * What is computed.  W is N x K.  Each weight is stored as a 4-bit unsigned
 * integer q in 0..15; every group of 128 consecutive weights of a row along K
 * has one fp16 scale s and one zero point z in 0..15, and the weight's value is
 * w = (q - z) * s.  Activations x are bfloat16, M = 1..8 token rows; the
 * product is y[m][n] = sum_k w[n][k] * x[m][k], accumulated in fp32.
 *   Sources (page title, section): group-wise INT4 weights with one fp16 scale
 *   per 128 weights of an output row -- "Building an LLM Inference Runtime: A
 *   Deep Dive into Qwen2.5-Coder-7B on NVIDIA H100", section "The Stack
 *   Architecture: A One-Page Overview"; a zero point per group applied as
 *   (q - z) * s -- "Custom AWQ Dequantization Kernel", section "Dead ends in
 *   profiling"; dequantisation fused into the matrix-vector kernel, no fp16 W
 *   materialised -- "CodeAlign-Runtime", section "Level 3 -- INT4 Quantization
 *   + Fused Kernel"; 1..8 rows (plain decode and a speculative-verify batch)
 *   with identical per-row results -- "qengine", section "How it works".
 *
 * Canonical layout (what callers hold; row-major, contiguous):
 *   qweight uint32 [N][K/8]: nibble j (bits 4j..4j+3) of word w is k = 8w + j
 *   scales  uint16 [N][K/128]: binary16 bit patterns
 *   zeros   uint8  [N][K/128]: values 0..15
 *   x       uint16 [M][K]: bfloat16 bit patterns
 *   y       uint16 [M][N] (bfloat16, round-to-nearest-even) or float [M][N]
 *
 * Conventions for every call:
 *   - Pointers named device are CUDA device pointers; the caller owns all
 *     memory.  The library never allocates device or pinned memory.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL is the legacy default
 *     stream) and is asynchronous unless stated otherwise.
 *   - Errors are returned, never aborted on.  Argument checks happen on the
 *     host before anything is enqueued; a failed launch returns W4_ERR_CUDA.
 *   - K must be a positive multiple of 128, N positive, 1 <= M <= 8.
 */
#ifndef W4_H
#define W4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
/* The same object as cudaStream_t. */
typedef struct CUstream_st *w4_stream_t;

typedef enum w4_status {
    W4_OK = 0,
    W4_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size, zero point > 15 */
    W4_ERR_UNSUPPORTED = 2,   /* M outside 1..8, or a call not allowed in stream capture */
    W4_ERR_LAYOUT = 3,        /* repacked buffer header does not match */
    W4_ERR_CUDA = 4,          /* a CUDA runtime call or kernel launch failed */
    W4_ERR_SCRATCH_LIMIT = 5  /* needs more than W4_STATIC_SCRATCH_BYTES of scratch */
} w4_status;

#define W4_GROUP_SIZE 128
#define W4_MAX_TOKENS 8
#define W4_LAYOUT_ID 1
#define W4_LAYOUT_ID_SWIGLU 2      /* gate/up-interleaved layout (w4_repack_swiglu) */
#define W4_LAYOUT_VERSION 4
#define W4_HEADER_BYTES 128
/* Size of the static device array behind w4_gemv_ws_static (4 MiB). */
#define W4_STATIC_SCRATCH_BYTES (4u * 1024u * 1024u)

/* Human-readable name of a status code (static string, never NULL). */
const char *w4_status_string(w4_status status);

/* Library version as major * 10000 + minor * 100 + patch. */
int w4_version(void);

/*
 * Sizes in bytes of the three buffers that w4_repack writes for an N x K
 * weight (the kernel layout): with NB = ceil(N / 128) row blocks and
 * G = K / 128 groups, qweight = W4_HEADER_BYTES + NB*G*8192, scales =
 * NB*G*256, zeros = NB*G*64.  The qweight buffer starts with a header
 * (layout id, version, K, N, error words).  Rows are padded to a multiple of
 * 128 with zero weights; the padding is never written back as output.
 * Errors: W4_ERR_INVALID_ARG for bad K/N or a NULL output pointer.
 */
w4_status w4_repacked_sizes(int K, int N, size_t *qweight_bytes,
                            size_t *scales_bytes, size_t *zeros_bytes);

/*
 * Offline, once per weight matrix: canonical layout -> kernel layout.
 * The offline packing step of "Building an LLM Inference Runtime ...",
 * sections "The Stack Architecture" and "Bug #3" (the runtime consumes one
 * fixed nibble interleave and refuses any other layout id).
 *
 *   qweight, scales, zeros : device, canonical layout (see top); qweight 16-byte
 *                            aligned, scales 2-byte aligned
 *   qweight_out, scales_out, zeros_out : device, sizes from w4_repacked_sizes,
 *                            each 16-byte aligned
 *
 * Validates every zero point on the device (must be <= 15) and therefore
 * synchronises `stream` before returning: not capturable into a CUDA graph
 * (returns W4_ERR_UNSUPPORTED if `stream` is capturing).
 * Errors: W4_ERR_INVALID_ARG (bad sizes/pointers, or a zero point > 15 -- the
 * outputs are then unspecified), W4_ERR_CUDA.
 */
w4_status w4_repack(const uint32_t *qweight, const uint16_t *scales,
                    const uint8_t *zeros, int K, int N, void *qweight_out,
                    void *scales_out, void *zeros_out, w4_stream_t stream);

/*
 * Host-side check of a repacked qweight buffer's header.  `header` is a host
 * copy of its first W4_HEADER_BYTES bytes.  Returns W4_OK when the magic,
 * layout id and version are this library's and K, N match; W4_ERR_LAYOUT
 * otherwise; W4_ERR_CUDA if a w4_gemv on this weight recorded that it gave up
 * waiting for its own copies (see w4_gemv); W4_ERR_INVALID_ARG for NULL.
 */
w4_status w4_check_header(const void *header, int K, int N);

/*
 * Weights to fp16, for checking: w_out[n][k] = fp16((q - z) * s), the exact
 * product rounded once to nearest-even.  Takes the canonical layout.
 * The "one thread per packed word, read once, unpack all eight" dequantiser of
 * "Custom AWQ Dequantization Kernel", section "Kernel versions" (v2).
 *
 *   qweight, scales, zeros : device, canonical; qweight 16-byte aligned
 *   w_out                  : device, uint16 [N][K] binary16 bits, 16-byte aligned
 * Errors: W4_ERR_INVALID_ARG, W4_ERR_CUDA.  Zero points > 15 are used as given.
 */
w4_status w4_dequant(const uint32_t *qweight, const uint16_t *scales,
                     const uint8_t *zeros, int K, int N, uint16_t *w_out,
                     w4_stream_t stream);

/*
 * The hot path: y = W x with W in the kernel layout written by w4_repack.
 * Dequantisation happens in registers; fp32 accumulation; deterministic (the
 * same inputs give bit-identical y on every call) and batch-invariant (row m
 * of y does not depend on M or on the other rows of x).  Graph-capturable:
 * no synchronisation, allocation or host read.
 * Fused dequantise-and-multiply GEMV of "CodeAlign-Runtime", section "Level 3",
 * and "qengine", section "How it works" (4-bit matrix-vector kernel, partial
 * sums added in a fixed order).
 *
 *   qweight, scales, zeros : device, the three buffers of w4_repack, each
 *                            16-byte aligned
 *   x                      : device, bfloat16 [M][K], 16-byte aligned
 *   y                      : device, bfloat16 [M][N], 2-byte aligned
 * The header is not read here (that would need a device read); check it once
 * with w4_check_header.  Every wait inside the kernel is bounded: a block that
 * gives up (about 2 s without progress -- never in normal operation) sets the
 * header's error word, which w4_check_header then reports, and leaves its
 * outputs unwritten.  So although qweight is passed as const, its buffer must
 * be writable device memory: the kernel may write that one 32-bit word of the
 * header (byte offset 28) and nothing else of it.  Weights, scales and zeros
 * must not be written by work still running on the device when w4_gemv is
 * enqueued.  The kernel writes no memory beyond y except that error word.
 * Errors: W4_ERR_INVALID_ARG, W4_ERR_UNSUPPORTED (M outside 1..8), W4_ERR_CUDA.
 */
w4_status w4_gemv(const void *qweight, const void *scales, const void *zeros,
                  const uint16_t *x, uint16_t *y, int M, int K, int N,
                  w4_stream_t stream);

/* Same as w4_gemv but writes the fp32 result before the bfloat16 cast
 * (y: device float [M][N], 4-byte aligned).  For checking. */
w4_status w4_gemv_f32(const void *qweight, const void *scales, const void *zeros,
                      const uint16_t *x, float *y, int M, int K, int N,
                      w4_stream_t stream);

/*
 * The product for any number of tokens M >= 1.  Up to 16 tokens it is w4_gemv
 * in passes of at most 8 tokens (one or two passes over the weight; row m is
 * bit-identical to w4_gemv on that token alone).  For more tokens the weight
 * is read once, in one pass on the tensor cores, where passes of 8 tokens
 * ("qengine", section "How the numbers were measured") would stream it once
 * per pass: a thread block owns a 128-row block of W and a tile of up to 128
 * tokens; per 128-k group it unpacks (q - z) exactly to bf16 into tensor
 * memory, multiplies it by the tile's x on the tensor cores with fp32
 * accumulation, and adds s times the group's sum into the token's fp32
 * result, group by group in order (the arithmetic of the GEMV's exact path).
 * There a token's result does not depend on M (> 16) or on which tokens share
 * its tile, and repeated calls give the same bits; its rows are not
 * bit-identical to w4_gemv's (different summation order inside a group), both
 * lying within the stated tolerances of the oracle.  Long K with few row
 * blocks is split over up to 8 blocks of a thread-block cluster, combined in
 * a fixed order.
 *   qweight, scales, zeros, y [M][N], stream : as for w4_gemv
 *   x [M][K]  : as for w4_gemv; for M > 16 read with tensor copies, so its
 *               address must be 16-byte aligned
 * The kernels may write the header's error word (byte offset 28), as w4_gemv.
 * For M > 16 every thread block takes all of its SM's tensor memory while it
 * runs: a kernel on another stream holding tensor memory on the same SM
 * delays it until that memory is freed.
 * Errors: W4_ERR_INVALID_ARG, W4_ERR_UNSUPPORTED (M < 1, or for M > 16:
 * M * K >= 2^40, more than 65535 tiles of 128 tokens, or a weight of 2^25 or
 * more 128 x 128 records), W4_ERR_CUDA; in passes, the first error stops the
 * rest.
 */
w4_status w4_gemm(const void *qweight, const void *scales, const void *zeros, const uint16_t *x,
                  uint16_t *y, int M, int K, int N, w4_stream_t stream);

/* w4_gemm writing the fp32 result before the bfloat16 cast (y: float [M][N]). */
w4_status w4_gemm_f32(const void *qweight, const void *scales, const void *zeros,
                      const uint16_t *x, float *y, int M, int K, int N, w4_stream_t stream);

/*
 * Workspace for w4_gemv_ws on the current device, in bytes (depends on K, N
 * and the SM count only).  Errors: W4_ERR_INVALID_ARG, W4_ERR_CUDA (no device).
 */
w4_status w4_gemv_workspace_bytes(int K, int N, size_t *bytes);

/*
 * The same product as w4_gemv, split evenly over one wave of thread blocks
 * (three per SM): every block streams an equal contiguous run of the weight's
 * 128-row x 128-k records, and the row blocks that fall between two blocks
 * are combined through `workspace` by the last block to finish its part, in a
 * fixed order (deterministic, no float atomics, no block ever waits for
 * another).  It needs no thread-block clusters and never launches more than
 * three blocks per SM, for callers that want that footprint; on the shapes
 * measured on GB300, w4_gemv is faster.  Same result for a token whatever M
 * is; bit-identical across calls.
 *
 *   qweight, scales, zeros, x, y : as for w4_gemv
 *   workspace       : device, 256-byte aligned, at least
 *                     w4_gemv_workspace_bytes(K, N) bytes, all zero before its
 *                     first use.  It starts with one 32-bit counter per
 *                     128-row block (padded to a multiple of 256 bytes), which
 *                     every completed call leaves at zero again; the rest holds
 *                     the partial sums of the last call.  So one workspace
 *                     serves any number of calls in a row, but calls that
 *                     share it must not overlap on the device; after a call
 *                     that reported a kernel error, zero it again.
 * Errors: W4_ERR_INVALID_ARG (also for a short or misaligned workspace),
 * W4_ERR_UNSUPPORTED (M outside 1..8), W4_ERR_CUDA.
 */
w4_status w4_gemv_ws(const void *qweight, const void *scales, const void *zeros,
                     const uint16_t *x, uint16_t *y, int M, int K, int N, void *workspace,
                     size_t workspace_bytes, w4_stream_t stream);

/* w4_gemv_ws writing the fp32 result before the bfloat16 cast (y: device
 * float [M][N], 4-byte aligned).  For checking. */
w4_status w4_gemv_ws_f32(const void *qweight, const void *scales, const void *zeros,
                         const uint16_t *x, float *y, int M, int K, int N, void *workspace,
                         size_t workspace_bytes, w4_stream_t stream);

/*
 * w4_gemv_ws without a caller workspace: the scratch lives in a static device
 * array of W4_STATIC_SCRATCH_BYTES inside the library, and this call allocates
 * nothing (no cudaMalloc, no cudaFree, no allocating library routine).  The
 * paper has no counterpart of this entry point; it is here for callers that
 * cannot allocate device memory where they call the GEMV -- code running
 * inside an allocator or memory-pool callback (an allocation there would
 * re-enter the allocator), a plug-in of a host program that has reserved all
 * device memory up front and hands out only the buffers it manages, or a
 * latency-bound path that must not take the device-wide synchronisation and
 * the failure mode of cudaMalloc.
 *
 *   qweight, scales, zeros, x, y, M, K, N, stream : as for w4_gemv
 *
 * The array costs W4_STATIC_SCRATCH_BYTES on every GPU that loads libw4,
 * held until the process exits.  The first call on a device (the current one)
 * looks up the array's device address; make that first call before any
 * stream capture.  Every call on a device uses the same array, which keeps
 * the last call's contents: each call clears the row-block counters it uses
 * (an asynchronous memset on `stream`) and overwrites the partial sums before
 * reading them, so consecutive calls are independent, but calls that overlap
 * on the GPU (other streams, other host threads) race and give wrong results.
 * A product needs w4_gemv_workspace_bytes(K, N) bytes of scratch; more than
 * W4_STATIC_SCRATCH_BYTES is refused with W4_ERR_SCRATCH_LIMIT before
 * anything else is checked or enqueued.  That need depends on the SM count:
 * with NB = ceil(N / 128) row blocks and W = NB * K / 128 records, it is
 * round_up(4 * NB, 256) bytes of counters plus 2 * min(W, 3 * SMs) * 4096
 * bytes of partial sums.  On a 152-SM GB300 the partial sums take at most
 * 3.56 MiB, which leaves room for about 114,000 row blocks (14.6 M output
 * rows); on a GPU with 171 or more SMs the partial sums alone exceed the
 * array for every product of at least 3 * SMs records.
 * Errors: W4_ERR_SCRATCH_LIMIT, W4_ERR_INVALID_ARG, W4_ERR_UNSUPPORTED (M
 * outside 1..8), W4_ERR_CUDA (no device, or the array could not be found).
 */
w4_status w4_gemv_ws_static(const void *qweight, const void *scales, const void *zeros,
                            const uint16_t *x, uint16_t *y, int M, int K, int N,
                            w4_stream_t stream);

/*
 * Gated MLP input projection with the SwiGLU activation fused into the
 * product ("qengine", section "How it works": gate and up projections
 * interleaved so that SwiGLU runs in registers).  The weight is the fused
 * [2I][K] matrix of the gate projection (rows 0..I-1) and the up projection
 * (rows I..2I-1), canonical layout as above; the result is
 *   y[m][j] = silu(g) * u,  g = sum_k Wgate[j][k] x[m][k],
 *   u = sum_k Wup[j][k] x[m][k],  silu(g) = g / (1 + exp(-g)),
 * with g and u accumulated exactly as by w4_gemv_f32 and the activation and
 * product in fp32.
 *
 * w4_repacked_sizes_swiglu: byte sizes of the three buffers of the
 *   interleaved layout for I outputs (16 * ceil(I / 8) kernel rows).
 * w4_repack_swiglu: as w4_repack, for the fused [2I][K] weight (qweight
 *   uint32 [2I][K/8], scales [2I][K/128], zeros [2I][K/128]); the header
 *   records layout W4_LAYOUT_ID_SWIGLU and N = I.  Synchronises; refuses
 *   stream capture (W4_ERR_UNSUPPORTED); zero points > 15 -> W4_ERR_INVALID_ARG.
 * w4_check_header_swiglu: as w4_check_header for that layout and I.
 * w4_gemv_swiglu: y bfloat16 [M][I] (round to nearest even); arguments as
 *   for w4_gemv with N replaced by I; the weight buffers must come from
 *   w4_repack_swiglu.  w4_gemv_swiglu_f32: the fp32 result.
 * Errors: W4_ERR_INVALID_ARG, W4_ERR_UNSUPPORTED (M outside 1..8),
 * W4_ERR_CUDA.
 */
w4_status w4_repacked_sizes_swiglu(int K, int I, size_t *qweight_bytes, size_t *scales_bytes,
                                   size_t *zeros_bytes);
w4_status w4_repack_swiglu(const uint32_t *qweight, const uint16_t *scales, const uint8_t *zeros,
                           int K, int I, void *qweight_out, void *scales_out, void *zeros_out,
                           w4_stream_t stream);
w4_status w4_check_header_swiglu(const void *header, int K, int I);
w4_status w4_gemv_swiglu(const void *qweight, const void *scales, const void *zeros,
                         const uint16_t *x, uint16_t *y, int M, int K, int I,
                         w4_stream_t stream);
w4_status w4_gemv_swiglu_f32(const void *qweight, const void *scales, const void *zeros,
                             const uint16_t *x, float *y, int M, int K, int I,
                             w4_stream_t stream);

/* Quantisation rules for w4_quantize. */
#define W4_QUANT_ASYMMETRIC 0
#define W4_QUANT_SYMMETRIC 1

/*
 * Quantise binary16 weights to the canonical layout, per row and group of
 * 128 consecutive weights along K, computing in fp32 from the exact binary16
 * values with every operation rounded to nearest (ties to even); the codes
 * are taken against the stored fp16 scale, so (q - z) * s is the value the
 * product uses:
 *   W4_QUANT_ASYMMETRIC: lo = min(0, min w), hi = max(0, max w),
 *     s = fp16((hi - lo) / 15), z = clamp(rint(-lo / s), 0, 15),
 *     q = clamp(rint(w / s) + z, 0, 15)  (round to nearest with a zero point
 *     per group: the storage format of this library);
 *   W4_QUANT_SYMMETRIC: s = fp16(max |w| / 7), z = 8,
 *     q = clamp(rint(w / s), -8, 7) + 8  (the pages' scheme: scale = absmax
 *     / 7, "Building an LLM Inference Runtime ...", section "The Stack
 *     Architecture: A One-Page Overview"; values in [-8, 7],
 *     "CodeAlign-Runtime", section "Level 3 -- INT4 Quantization + Fused
 *     Kernel"; stored with the fixed zero point 8).
 * A group whose scale rounds to 0 stores s = 0 and q = z.
 *
 *   w       : device, binary16 bit patterns [N][K], 16-byte aligned; finite
 *   mode    : W4_QUANT_ASYMMETRIC or W4_QUANT_SYMMETRIC
 *   qweight : device, uint32 [N][K/8] (canonical nibble order), 4-byte aligned
 *   scales  : device, binary16 [N][K/128], 2-byte aligned
 *   zeros   : device, uint8 [N][K/128]
 * Outputs are written completely; w4_repack then gives the kernel layout.
 * Errors: W4_ERR_INVALID_ARG (bad pointers, sizes or mode), W4_ERR_CUDA.
 */
w4_status w4_quantize(const uint16_t *w, int K, int N, int mode, uint32_t *qweight,
                      uint16_t *scales, uint8_t *zeros, w4_stream_t stream);

/*
 * The launch shape w4_gemv uses for an N x K weight on the current device:
 * 16-row tiles per thread block, the number of K splits (thread blocks of
 * one cluster that each reduce a slice of K and combine in a fixed order),
 * and whether the zero point is folded out of the inner product (1: fp16
 * operands 1024 + q and 1024 + 16 q with x scaled per token into fp16
 * range, the zero point removed once per group and output through the
 * group's half sums of x, chosen when a block streams at least 8 groups;
 * 0: the bf16 tensor-core operand is q - z, exactly).  Both are the same sum
 * up to fp32 rounding.  Depends on K and N only, never on M.  Outputs may be
 * NULL.
 * Errors: W4_ERR_INVALID_ARG, W4_ERR_CUDA (no device).
 */
w4_status w4_gemv_config(int K, int N, int *tiles_per_block, int *k_splits,
                         int *zero_point_folded);

/* How w4_gemv launches a product (filled by w4_gemv_plan). */
typedef struct w4_gemv_launch_info {
    int k_splits;            /* thread blocks per cluster, each reducing a slice of K */
    int zero_point_folded;   /* 1: fp16 operands, zero point folded out; 0: exact q - z */
    int grid_x, grid_y;      /* launch grid: row blocks (or persistent slots) x K splits */
    int persistent;          /* 1: each block takes row blocks in turn */
    int overlap;             /* 1: launched with programmatic dependent launch (starts
                                while the previous kernel in the stream finishes) */
    int capped;              /* 1: shared memory padded so that at most the needed
                                number of blocks share an SM */
    int ring_stages;         /* depth of the shared-memory weight ring */
    int wide_prologue;       /* 1: folded x prologue spread over (group, token) pairs */
    int blocks_per_sm_max;   /* blocks per SM the kernel instance is built for */
    size_t smem_bytes;       /* dynamic shared memory per block */
} w4_gemv_launch_info;

/*
 * Diagnostic with no counterpart in the pages: the launch w4_gemv makes for
 * M tokens of an N x K weight on the current device (split, arithmetic, grid,
 * residency, overlap), so that callers and tests can see which kernel path a
 * shape takes.  Computes the same plan w4_gemv computes before each launch;
 * launches nothing.
 *   info : host, written on success
 * Errors: W4_ERR_INVALID_ARG (bad K/N, NULL info), W4_ERR_UNSUPPORTED (M
 * outside 1..8, or no launch shape fits), W4_ERR_CUDA (no device).
 */
w4_status w4_gemv_plan(int M, int K, int N, w4_gemv_launch_info *info);

/*
 * Diagnostic with no counterpart in the pages: runs, in one thread of one
 * block, the bounded mbarrier wait the GEMV kernels use on a barrier that
 * nothing ever completes, and stores into *status (device, 4-byte aligned)
 * 1 if the wait gave up after its limit (about 2 s of clock cycles, the
 * expected outcome) or 0 if it wrongly returned success.  Shows on a real
 * GPU that a wait which can never finish ends, reports, and leaves the
 * context usable.  Asynchronous on `stream`; takes about 2 s on the GPU.
 * Errors: W4_ERR_INVALID_ARG (status NULL or misaligned), W4_ERR_CUDA.
 */
w4_status w4_selftest_bounded_wait(uint32_t *status, w4_stream_t stream);

/* Modes of w4_stream_read. */
#define W4_STREAM_READ_RING 0
#define W4_STREAM_READ_LD128 1

/*
 * Diagnostic: reads `bytes` of device memory once and folds them into one
 * word, to measure the read-only bandwidth a kernel gets on this GPU -- the
 * ceiling a memory-bound GEMV is judged against ("qengine", section
 * "Learnings": measure your own ceiling with a plain read benchmark; a copy
 * also writes, and the data sheet is a peak no kernel reaches).
 *   W4_STREAM_READ_RING : the GEMV's own method -- contiguous shares of the
 *     buffer moved in 8 KB cp.async.bulk records through a 12-stage
 *     shared-memory ring, two blocks per SM; `bytes` a multiple of 8192.
 *   W4_STREAM_READ_LD128: 16-byte streaming loads in a grid-stride loop, four
 *     blocks of 512 threads per SM; `bytes` a multiple of 16.
 *   src : device, 16-byte aligned
 *   out : device uint32 [2]; out[0] is xor-ed with the folded word, out[1]
 *         gets bit 0 if a bounded wait gave up (never in normal operation)
 * Asynchronous on `stream`; time it with events around the call.
 * Errors: W4_ERR_INVALID_ARG (pointers, alignment, size, mode), W4_ERR_CUDA.
 */
w4_status w4_stream_read(const void *src, size_t bytes, int mode, uint32_t *out,
                         w4_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* W4_H */
