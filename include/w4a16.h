/*
 * w4a16.h -- C ABI of the GB300 (sm_103a) W4A16 weight-only GEMM library,
 * libw4a16.so.
 *
 * The operation (page "Beating FP16 with 4-bit Weights: A Portable W4A16 GEMM
 * in Triton", sections "The design" and "Code"; GemLite README, usage section):
 *
 *     out[M,N] = x[M,K] . W[K,N],   x fp16, fp32 accumulation, out fp16,
 *     W[k,n]   = (q[k,n] - z[k/g,n]) * s[k/g,n]
 *
 * where q is an unsigned 4-bit code, g the group size (128 by default), and
 * s, z one fp16 scale and one fp16 zero per (group, column).
 *
 * Data layout (all row-major, all DEVICE memory owned by the caller):
 *   x       [M, K]    fp16 (binary16 bit patterns, uint16_t)
 *   packed  [K/8, N]  uint32: the code of row k sits at bits 4*(k%8) of word
 *                     (k/8, n) -- eight codes per word along K, LSB first
 *   scales  [K/g, N]  fp16
 *   zeros   [K/g, N]  fp16 holding an integer in [0, 15]
 *   out     [M, N]    fp16
 *
 * Conventions shared by every entry point:
 *   - All pointers are device pointers; nothing is allocated per call and no
 *     ownership is taken.  Calls are asynchronous on `stream` (0 = the legacy
 *     default stream) and return once the work is enqueued.
 *   - Arguments are validated on the host before anything is enqueued; a bad
 *     argument returns a non-zero status and enqueues nothing.  The message for
 *     the last non-OK status of the calling thread is w4a16_last_error().
 *   - Shapes: K % group == 0, group % 32 == 0 (group in [32, 1024]),
 *     N % 4 == 0, all of M, N, K >= 0 and below 2^31 elements per array.
 *     M == 0 (or N == 0) is a no-op that returns W4A16_OK.
 *   - Alignment: x, packed, scales, zeros and out must be 16-byte aligned
 *     (W4A16_ERR_MISALIGNED otherwise).
 *   - `out` is fully overwritten, never accumulated into, so repeated calls
 *     into a dirty buffer give the same bits.
 *   - For a fixed device, shape and configuration the result is bitwise
 *     reproducible run to run (all split-K reductions are in a fixed order).
 */
#ifndef W4A16_H_
#define W4A16_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define W4A16_API __attribute__((visibility("default")))
#else
#define W4A16_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum w4a16_status {
    W4A16_OK = 0,
    W4A16_ERR_INVALID_ARG = 1,   /* bad shape, group or null pointer */
    W4A16_ERR_UNSUPPORTED = 2,   /* valid request the library does not implement */
    W4A16_ERR_MISALIGNED = 3,    /* a pointer is not 16-byte aligned */
    W4A16_ERR_CUDA = 4,          /* a CUDA runtime call or kernel launch failed */
    W4A16_ERR_TIMEOUT = 5        /* a bounded device-side wait gave up (see
                                    w4a16_get_kernel_status) */
} w4a16_status;

/* Kernel family a GEMM call runs on. */
typedef enum w4a16_path {
    W4A16_PATH_AUTO = 0,     /* pick from the measured dispatch table */
    W4A16_PATH_DECODE = 1,   /* CUDA-core unpack + register-fed tensor-core MMA,
                                split-K across a thread-block cluster (M <= 16
                                per pass; larger M is processed in 16-row passes) */
    W4A16_PATH_PREFILL = 2   /* TMA-staged tiles, tcgen05 MMA, TMEM accumulator */
} w4a16_path;

/* flags */
#define W4A16_FLAG_PDL 0x1   /* launch with programmatic dependent launch: the
                                kernel streams its weights before waiting for the
                                previous kernel on the stream.  Only valid when
                                packed/scales/zeros are NOT written by the kernel
                                immediately before it on the same stream.  Decode
                                kernels only; the prefill kernels are compute-bound
                                and always launch in stream order. */
#define W4A16_FLAG_TEST_TIMEOUT 0x100  /* test aid (TMA decode kernel only): arm the
                                last pipeline stage without loading it, so its
                                bounded wait runs out (5 ms); the output is
                                undefined and w4a16_get_kernel_status reports
                                W4A16_ERR_TIMEOUT.  Never set in production. */

/* Decode kernel variants (w4a16_config.variant). */
#define W4A16_DECODE_AUTO 0
#define W4A16_DECODE_TMA 1        /* weights staged by TMA into a shared-memory ring */
#define W4A16_DECODE_REGISTERS 2  /* weights streamed by 128-bit loads into registers */
#define W4A16_DECODE_STREAM 3     /* persistent: at most one CTA per SM, each streams a
                                     contiguous run of (column tile, stage) units
                                     through a ring of bulk copies */
#define W4A16_DECODE_WARP 4       /* every warp streams its own run of 32-column x
                                     512-k units through a private TMA ring; no
                                     barrier between warps (M <= 4, N % 8 == 0,
                                     power-of-two groups 32..1024) */

/* Prefill kernel variants (w4a16_config.variant on the prefill path). */
#define W4A16_PREFILL_A_TMEM 1    /* dequantized W^T operand in tensor memory (default) */
#define W4A16_PREFILL_A_SMEM 2    /* dequantized W^T operand in shared memory */

/* Element type of x, scales, zeros and out (w4a16_config.dtype).  The codes
 * and their packing are the same for both. */
#define W4A16_DTYPE_F16 0   /* binary16 (default) */
#define W4A16_DTYPE_BF16 1  /* bfloat16: 1 sign, 8 exponent, 7 fraction bits.
                               The pages name bf16 as the other model dtype
                               (GemLite README, usage section; page "Beating
                               FP16 with 4-bit Weights", section "What's
                               next") but give no recipe; this library keeps
                               the fp16 recipe with bfloat16 wherever a value
                               is stored, and the kernels multiply x by the
                               dequantized weight bf16((q - z) * s), one
                               rounding of the exact product.  Decode path:
                               registers variant only (W4A16_DECODE_AUTO
                               selects it); prefill path: A in tensor memory
                               only.  Other combinations return
                               W4A16_ERR_UNSUPPORTED. */

/*
 * Launch configuration of one GEMM call.  Zero in any field means "choose
 * automatically"; w4a16_plan() returns the choice for a shape.
 */
typedef struct w4a16_config {
    int path;       /* w4a16_path */
    int split_k;    /* decode: CTAs of one cluster that split K (1..8);
                       prefill: the same for the one-ring kernel (1..8; its
                       CTAs' fp32 partials are summed in rank order by the
                       cluster's first CTA) */
    int warps_k;    /* decode, registers variant: warps per CTA that split K;
                       decode, TMA variant: consumer warps per CTA (4, 8 or 16;
                       4 lets three CTAs share an SM);
                       prefill: dequantizing warps (4, 8 or 16) */
    int warps_n;    /* decode: 32-column strips per CTA (TMA variant: 2 or 4) */
    int steps;      /* decode: K per warp in 32-row steps (registers variant) or
                       K per CTA in 256-row stages (TMA variant) */
    int tile_m;     /* prefill: rows of x per CTA tile (16..256, multiple of 16) */
    int flags;      /* W4A16_FLAG_* */
    int variant;    /* decode: W4A16_DECODE_*; prefill: W4A16_PREFILL_* */
    int ctas;       /* decode, stream variant: CTAs in the grid (0: one per SM) */
    int dtype;      /* W4A16_DTYPE_F16 (0) or W4A16_DTYPE_BF16 */
} w4a16_config;

/*
 * Group-wise asymmetric 4-bit quantization and packing of an fp16 weight.
 * (page "Beating FP16 with 4-bit Weights", section "The design": one scale and
 * one zero-point per group of rows, eight codes per int32 along K.)
 *
 * Per (group j, column n), over rows k in [j*g, (j+1)*g):
 *     s = fp16((max_k W - min_k W) / 15)     fp64 arithmetic, one rounding;
 *                                            s = 1.0 if that rounds to 0
 *     z = clamp(rint(-min / s), 0, 15)       rint = round half to even
 *     q = clamp(rint(W / s) + z, 0, 15)
 * using the rounded s throughout.  Bit-exact with the fp64 oracle.
 *   W       [K, N] fp16 device input
 *   packed  [K/8, N], scales [K/g, N], zeros [K/g, N] device outputs
 * Offline step: not on the timed path.
 */
W4A16_API w4a16_status w4a16_quantize_pack(const uint16_t *W, int K, int N, int group,
                                 uint32_t *packed, uint16_t *scales, uint16_t *zeros,
                                 cudaStream_t stream);

/*
 * Quantization modes of w4a16_quantize_pack_ex.
 *   W4A16_QUANT_ASYMMETRIC  the min/max recipe above (w4a16_quantize_pack).
 *   W4A16_QUANT_SYMMETRIC   signed codes stored with a +8 offset (page "Beating
 *       FP16 with 4-bit Weights", section "Code": its tests cover symmetric
 *       and asymmetric quantization; section "Things I got wrong along the
 *       way": the +8 zero-point of the symmetric packing).  Per (group j,
 *       column n):
 *           s = fp16(max_k |W| / 7)    fp64 arithmetic, one rounding;
 *                                      s = 1.0 if that rounds to 0
 *           z = 8
 *           q = clamp(rint(W / s) + 8, 0, 15)
 *       so the largest magnitude codes as +-7 and the same (q - z) * s
 *       dequantization, and every GEMM path, apply unchanged.
 * An unknown mode returns W4A16_ERR_INVALID_ARG (checked first).
 */
enum { W4A16_QUANT_ASYMMETRIC = 0, W4A16_QUANT_SYMMETRIC = 1 };
W4A16_API w4a16_status w4a16_quantize_pack_ex(const uint16_t *W, int K, int N, int group,
                                    int mode, uint32_t *packed, uint16_t *scales,
                                    uint16_t *zeros, cudaStream_t stream);

/*
 * Dequantize the packed weight back to fp16: W_out[k,n] = fp16((q - z) * s),
 * one rounding of the exact product.  Test aid (bit-exact with the oracle).
 */
W4A16_API w4a16_status w4a16_dequantize(const uint32_t *packed, const uint16_t *scales,
                              const uint16_t *zeros, uint16_t *W_out,
                              int K, int N, int group, cudaStream_t stream);

/*
 * bfloat16 counterparts of w4a16_quantize_pack and w4a16_dequantize (same
 * layouts; W, scales, zeros and W_out hold bfloat16 bit patterns):
 *     s = bf16((max - min) / 15)   fp64 arithmetic, one rounding; 1.0 if 0
 *     z = clamp(rint(-min / s), 0, 15), stored as a bfloat16 integer
 *     q = clamp(rint(W / s) + z, 0, 15)
 *     W_out[k,n] = bf16((q - z) * s), one rounding of the exact product.
 * Bit-exact with the oracle's bfloat16 variant.  Same argument checks and
 * error returns as the fp16 entries.
 */
W4A16_API w4a16_status w4a16_quantize_pack_bf16(const uint16_t *W, int K, int N, int group,
                                      uint32_t *packed, uint16_t *scales, uint16_t *zeros,
                                      cudaStream_t stream);
W4A16_API w4a16_status w4a16_dequantize_bf16(const uint32_t *packed, const uint16_t *scales,
                                   const uint16_t *zeros, uint16_t *W_out, int K, int N,
                                   int group, cudaStream_t stream);

/*
 * out[M,N] = x[M,K] . dequant(packed, scales, zeros), fp32 accumulation,
 * fp16 output (round to nearest even).  The weight is dequantized inside the
 * kernel and never materialized.  Automatic path selection.
 */
W4A16_API w4a16_status w4a16_gemm(const uint16_t *x, const uint32_t *packed,
                        const uint16_t *scales, const uint16_t *zeros, uint16_t *out,
                        int M, int N, int K, int group, cudaStream_t stream);

/* As w4a16_gemm, with an explicit (possibly partial) launch configuration;
 * cfg == NULL is the same as w4a16_gemm.  cfg->dtype = W4A16_DTYPE_BF16
 * makes x, scales, zeros and out bfloat16 (out rounded to nearest even).
 * Unsupported combinations return W4A16_ERR_UNSUPPORTED without enqueuing
 * anything. */
W4A16_API w4a16_status w4a16_gemm_ex(const uint16_t *x, const uint32_t *packed,
                           const uint16_t *scales, const uint16_t *zeros, uint16_t *out,
                           int M, int N, int K, int group, const w4a16_config *cfg,
                           cudaStream_t stream);

/*
 * The arguments of one w4a16_gemm_ex call in one block, for callers that
 * repeat the same call (a decode loop: same buffers, new contents): the
 * caller fills the block once and passes its address each time, which keeps
 * the per-call marshalling of a foreign-function binding to two arguments.
 * The pages have no counterpart (they call a Triton kernel from Python).
 * Same meaning, checks, errors and result as w4a16_gemm_ex; `cfg` may be
 * NULL (automatic).  The block and the configuration it points to are read
 * during the call only.
 */
typedef struct w4a16_gemm_args {
    const uint16_t *x;
    const uint32_t *packed;
    const uint16_t *scales;
    const uint16_t *zeros;
    uint16_t *out;
    int M, N, K, group;
    const w4a16_config *cfg;
} w4a16_gemm_args;
W4A16_API w4a16_status w4a16_gemm_call(const w4a16_gemm_args *args, cudaStream_t stream);

/*
 * Grouped GEMM: E independent products of one shape, out_e = x_e . W_e
 * (the experts of a mixture-of-experts layer, each with its own weights and
 * its own rows of x), in ONE kernel launch instead of E.  The pages measure
 * MoE-expert projections among the shapes where the method wins (page "Beating
 * FP16 with 4-bit Weights", section "Results") and name CUDA graphs and fewer
 * launches as the next step for launch overhead (page "Triton Kernel Matches
 * bitsandbytes", section "What's next"); this is the grouped entry that makes
 * 64 small expert GEMMs one weight stream.
 *   E          1 .. W4A16_MAX_EXPERTS
 *   x, packed, scales, zeros, out
 *              HOST arrays of E device pointers (the same layouts and
 *              alignment rules as w4a16_gemm for each expert); the arrays are
 *              read during the call and may be reused afterwards
 *   M, N, K, group  the shape shared by all experts
 *   cfg        NULL (automatic) or a decode-path configuration (registers
 *              or stream variant); the grouped kernels serve M <= 16, larger M
 *              runs the experts' GEMMs one launch after another on the same
 *              stream
 * Errors: W4A16_ERR_INVALID_ARG for E out of range or any NULL pointer,
 * W4A16_ERR_MISALIGNED as w4a16_gemm, W4A16_ERR_UNSUPPORTED for a
 * configuration with no kernel; nothing is enqueued on an error.
 */
#define W4A16_MAX_EXPERTS 64
W4A16_API w4a16_status w4a16_gemm_grouped(int E, const uint16_t *const *x,
                                const uint32_t *const *packed,
                                const uint16_t *const *scales,
                                const uint16_t *const *zeros, uint16_t *const *out,
                                int M, int N, int K, int group, const w4a16_config *cfg,
                                cudaStream_t stream);

/*
 * The pre-permuted ("repacked") weight layout.  Page "Beating FP16 with 4-bit
 * Weights", section "What's next", names permuting the packed weights offline
 * into the order the tensor-core MMA consumes them, with asynchronous copies,
 * as the way to the remaining speed; page "Triton Kernel Matches
 * bitsandbytes", section "Why Marlin Is Still Faster", credits the same
 * offline reordering.  The pages give no byte layout; this library's is:
 *
 *   requirements: K % 256 == 0, N % 32 == 0, and group (a multiple of 32)
 *   divides 256 or is a multiple of 256.  gps = 256/group if group < 256,
 *   else 1.
 *   The weight is cut into 32-column strips sn and 256-row blocks kb; block
 *   (sn, kb) starts at byte (sn * K/256 + kb) * B, B = 4096 + 128 * gps, and is:
 *     1024 uint32 words: word u8*128 + L*4 + c (u8 < 8, L < 32, c < 4) holds
 *       the codes of packed row 32kb + 4u8 + L%4 of column 32sn + 4(L/4) + c,
 *       nibble p holding the code of k = 8*row + 2(p%4) + p/4;
 *     then 16 bytes per (gi < gps, g < 8): the fp16 scales of columns
 *       32sn + 4g .. +3 of group row 256kb/group + gi, then their four zeros.
 *   So a 256-k stage of a strip is one contiguous block holding its scales and
 *   zeros, each lane of a consumer warp reads its MMA fragment with one
 *   128-bit load, and x enters the MMA without byte permutes.
 */

/* Bytes of the repacked form of a [K, N] weight; 0 if the shape or group is
 * not supported by the layout.  Host only. */
W4A16_API size_t w4a16_repacked_bytes(int K, int N, int group);

/*
 * natural (packed [K/8, N], scales, zeros [K/g, N]) -> repacked, on the GPU.
 *   repacked  device buffer of w4a16_repacked_bytes(K, N, group) bytes
 * packed and repacked 16-byte aligned, scales and zeros 8-byte aligned
 * (W4A16_ERR_MISALIGNED); an unsupported shape or group returns
 * W4A16_ERR_UNSUPPORTED.  Offline step: bit-exact with the oracle's map.
 */
W4A16_API w4a16_status w4a16_repack(const uint32_t *packed, const uint16_t *scales,
                          const uint16_t *zeros, int K, int N, int group, void *repacked,
                          cudaStream_t stream);

/*
 * out[M,N] = x[M,K] . W, with W given in the repacked form, reading one
 * contiguous block per strip and 256-k stage with one bulk copy.  Two kernels:
 *   W4A16_DECODE_WARP    M <= 8: every warp streams its own run of blocks
 *                        through a private ring (the design of the natural-
 *                        layout warp-stream kernel); at most 64 32-column
 *                        tiles per CTA (over all experts of a grouped call).
 *   W4A16_DECODE_STREAM  M up to 16 per launch; larger M runs ceil(M/16)
 *                        launches in stream order.
 * cfg NULL (or variant AUTO with warps_n and split_k 0) takes the warp kernel
 * where it serves the call and the call has at least four 256-k blocks per SM
 * (over all experts), else the stream kernel; a stream-variant
 * configuration (warps_n, split_k, ctas, flags) or the warp variant (ctas,
 * flags) may be requested, and a warp request it cannot serve returns
 * W4A16_ERR_UNSUPPORTED.  Same x / out layouts and alignment rules as
 * w4a16_gemm; `repacked` 16-byte aligned.  The result equals w4a16_gemm on the
 * natural weights within the GEMM tolerance (the MMAs see the same values;
 * only the summation order of the k-permutation differs).
 */
W4A16_API w4a16_status w4a16_gemm_repacked(const uint16_t *x, const void *repacked, uint16_t *out,
                                 int M, int N, int K, int group, const w4a16_config *cfg,
                                 cudaStream_t stream);

/* Grouped form of w4a16_gemm_repacked: E <= W4A16_MAX_EXPERTS experts of one
 * shape in one launch, M <= 16 (the warp kernel at M <= 8, as above); host
 * arrays of E device pointers as in w4a16_gemm_grouped. */
W4A16_API w4a16_status w4a16_gemm_grouped_repacked(int E, const uint16_t *const *x,
                                         const void *const *repacked, uint16_t *const *out,
                                         int M, int N, int K, int group,
                                         const w4a16_config *cfg, cudaStream_t stream);

/*
 * w4a16_gemm_noalloc: the decode GEMM for callers that must not allocate GPU
 * memory.  The pages have no counterpart to this entry point; it exists for
 * callers such as a runtime that may only use memory reserved at start-up, a
 * real-time loop where an allocation's unbounded latency is not allowed, or an
 * application whose memory is owned entirely by its own allocator.  w4a16_gemm
 * never allocates per call either, but the first stream-K call on a new stream
 * allocates that stream's scratch once; this entry point never does.
 *
 * It runs the stream decode kernel (W4A16_DECODE_STREAM) with stream-K shares
 * and the natural weight layout, and takes its scratch -- the arrival counters
 * and fp32 partial sums of output tiles shared by two CTAs -- from one array of
 * 4 MiB that the library keeps in device memory: 64 KiB of counters (one per
 * 32..128-column tile) and 4,128,768 bytes of partials (two tiles of M x 32..128
 * floats per CTA, one CTA per SM).  Every GPU that loads the library holds the
 * array until the process exits.  A shape that needs more than that returns
 * W4A16_ERR_UNSUPPORTED with the needed sizes in w4a16_last_error(); so do
 * M > 16, N % 8 != 0 and groups that are not powers of two.
 *
 * Arguments, layouts, alignment and result: as w4a16_gemm (x, packed, scales,
 * zeros, out device pointers; out fully overwritten).  The call allocates
 * nothing (no cudaMalloc or any allocating library routine); it enqueues a
 * clearing of the counters and the kernel on `stream`.
 * - The first call on a device looks up the array's device address on that
 *   device (once); make that first call before any stream capture begins.
 * - All calls share the one array and it keeps the last call's contents: calls
 *   whose work overlaps on the GPU (on different streams, or different threads
 *   without ordering) race on it and their results are undefined.  Order them,
 *   for example on one stream.
 */
W4A16_API w4a16_status w4a16_gemm_noalloc(const uint16_t *x, const uint32_t *packed,
                                const uint16_t *scales, const uint16_t *zeros, uint16_t *out,
                                int M, int N, int K, int group, cudaStream_t stream);

/*
 * Measurement aid, not part of the GEMM: reads `bytes` from `src` (device, 16-byte
 * aligned, a multiple of 16) into shared memory the way the decode kernels
 * stream their weights -- 16 KB bulk copies into a ring of shared-memory slots,
 * one CTA per SM, each taking a contiguous share -- with no arithmetic, and
 * writes one word per CTA to `sink` (device, at least one uint32 per SM).
 * flags: W4A16_FLAG_PDL launches it with programmatic dependent launch (the
 * copies start before the previous kernel ends; the store to `sink` waits for
 * it).  A chain of these calls over distinct buffers measures the per-launch
 * streaming ceiling a decode GEMM of the same size can reach.
 */
W4A16_API w4a16_status w4a16_stream_read(const void *src, size_t bytes, uint32_t *sink,
                               int flags, cudaStream_t stream);

/* Host-only: the launch configuration w4a16_gemm_ex would use for this shape
 * with `request` (may be NULL) filled in.  Touches no GPU.  Returns the same
 * validation status the GEMM would (pointer checks excepted). */
W4A16_API w4a16_status w4a16_plan(int M, int N, int K, int group, const w4a16_config *request,
                        w4a16_config *plan_out);

/* Reads and clears, in one atomic exchange on the device, the status word that
 * bounded waits inside the kernels set when they give up (W4A16_ERR_TIMEOUT).
 * The exchange is queued on `stream` after the work already there, and the
 * call returns once it has run.  W4A16_OK if no kernel reported a problem.
 * The word is one per device, shared by every stream: the status covers every
 * kernel of this library on the current device that finished before the
 * exchange ran, whichever stream it ran on; a kernel still running on another
 * stream reports at the next call.  A bounded wait's limit is counted from
 * after its kernel's wait for the previous kernel on the stream (programmatic
 * dependent launch), so a long-running predecessor never causes a timeout. */
W4A16_API w4a16_status w4a16_get_kernel_status(cudaStream_t stream);

/* Message for the last non-OK status returned to the calling thread
 * ("" if none).  The pointer stays valid until the thread's next call. */
W4A16_API const char *w4a16_last_error(void);

/* Library version as major*10000 + minor*100 + patch. */
W4A16_API int w4a16_version(void);

#ifdef __cplusplus
}
#endif

#endif /* W4A16_H_ */
