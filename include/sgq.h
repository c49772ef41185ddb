/*
 * sgq.h -- C ABI of the GB300 (sm_103a) W8A8 FP8 block-scaled linear layer.
 *
 * The layer has two steps, each one call:
 *
 *   1. sgq_quant_token_group: per-token-group activation quantisation,
 *      bf16 -> FP8 E4M3 codes plus one fp32 scale per group.
 *   2. sgq_fp8_block_gemm:   D = (Aq * As)(Wq * Ws)^T, fp32 accumulation,
 *      bf16 output, for the [1,128]/[128,128] and [1,32]/[32,32] recipes.
 *
 * plus sgq_quant_weight_block, the offline weight quantiser that produces the
 * block-scaled weights the GEMM consumes.
 *
 * Conventions shared by every call:
 *  - Every tensor argument is a DEVICE pointer to contiguous row-major data,
 *    owned by the caller (the library never frees or keeps it).  Pointers must
 *    be 16-byte aligned, else SGQ_ERR_MISALIGNED.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream).  The host call returns once the kernels are enqueued;
 *    errors found on the device are reported later by sgq_device_status.
 *  - Nothing aborts, asserts or falls back: every call returns an sgq_status.
 *    Arguments are checked on the host before anything is launched.
 *  - E4M3 is the OCP FP8 "E4M3FN" format (largest finite 448, no infinities).
 *    Scales are fp32.  A "UE8M0" scale is an fp32 value that is an exact
 *    power of two; the *_ue8m0 entry points below take or produce it as its
 *    8-bit biased exponent byte instead (2^(byte - 127); 255 is NaN).
 *  - The library allocates device memory only once per device, on first use
 *    of a GEMM shape that needs a split-K workspace (and a 4-byte status
 *    word).  That first use must not happen inside a CUDA stream capture;
 *    if it does, the call returns SGQ_ERR_UNSUPPORTED.
 *  - That split-K workspace (fp32 partial tiles and arrival counters) is one
 *    per device and shared by every GEMM call on it.  GEMMs that use split-K
 *    must therefore not overlap on the GPU: calls on one stream are safe;
 *    calls on different streams, or from several host threads, must be
 *    ordered (events, or one stream per device).  sgq_gemm_plan (and, for
 *    the power-of-two promise and UE8M0 bytes, sgq_gemm_plan_pow2) tells
 *    which shapes split K (out[2] > 1).
 */
#ifndef SGQ_H_
#define SGQ_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so the header needs no CUDA. */
typedef struct CUstream_st* sgq_stream_t;

typedef enum {
    SGQ_OK = 0,
    SGQ_ERR_INVALID_ARG = 1,   /* bad size, null pointer, unsupported value */
    SGQ_ERR_UNSUPPORTED = 2,   /* valid request this build cannot serve */
    SGQ_ERR_MISALIGNED = 3,    /* a pointer is not 16-byte aligned */
    SGQ_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
    SGQ_ERR_TIMEOUT = 5        /* a device-side wait ran out (reported by sgq_device_status) */
} sgq_status;

/* Flags for sgq_fp8_block_gemm_ex. */
#define SGQ_GEMM_DEFAULT 0u
/* Never use the block-scale MMA; apply every scale in the fp32 promotion
 * step.  Results stay within the same tolerance; meant for testing. */
#define SGQ_GEMM_FORCE_PROMOTE 1u
/* Wide tiles (M > 64) only: force two alternating MMA-issuing warps, or a
 * single one, instead of the launch plan's choice.  Both issue the same MMA
 * sequence, so the result is bit-identical either way; meant for testing.
 * Either flag also keeps 64 < M <= 1024 on the wide tiles where the plan
 * would take swap-AB tiles of 64 tokens. */
#define SGQ_GEMM_ISSUE_ALT 2u
#define SGQ_GEMM_ISSUE_SINGLE 4u
/* Testing only: the first CTA never loads the weight tile of its sixth K
 * stage, so its bounded waits run out, after about 1 ms instead of about 1 s.
 * The kernel then stops issuing work, lets its copies and tensor-core
 * operations land, frees its tensor memory and returns; sgq_device_status
 * reports SGQ_ERR_TIMEOUT and D is undefined.  The stream stays usable.
 * Needs a shape whose first CTA has at least six K stages. */
#define SGQ_GEMM_TEST_TIMEOUT 8u
/* The caller promises that every scale (As and Ws) is an exact power of two
 * (UE8M0), as the quantisers produce with ue8m0 = 1.  Shapes on the wide
 * tiles (M > 64, or the plan's choice for M <= 1024) with K a multiple of 128
 * and at least one tile of 256 activation rows x 224 weight rows per SM then
 * run on tiles of 256 activation rows x 224 (or 192, whichever fills the
 * grid's rounds better) weight rows with two accumulators, every scale
 * applied by the block-scaled MMA.  A scale that is
 * not a power of two makes sgq_device_status report SGQ_ERR_INVALID_ARG (D is
 * then undefined).  Results agree with the default path within the GEMM
 * tolerance. */
#define SGQ_GEMM_SCALES_POW2 16u

/*
 * Per-token-group quantisation.
 *
 * Defined by "Sgl project Sglang GEMM Interface", Description / Quantization
 * Routines (sgl_per_token_group_quant_8bit: group size, epsilon, clipping
 * range, UE8M0 scale format) and the "UE8M0 activation rounding" of sglang
 * PR #42604 "[SM90] Use native block32 DeepGEMM for DeepSeek-V4.1",
 * Modifications.  For row m and group j (columns j*group .. j*group+group-1):
 *
 *   amax    = max |x[m, k]| over the group
 *   s       = max(amax, 1e-10) / 448           (fp32, correctly rounded)
 *   if ue8m0: s = smallest power of two >= s
 *   xs[m,j] = s
 *   xq[m,k] = E4M3_RNE(clamp(x[m,k] / s, -448, 448))   (fp32 division)
 *
 * x:  bf16 [M, K].   xq: uint8 E4M3 codes [M, K].   xs: fp32 [M, K/group].
 * group in {32, 128}; K % group == 0; M >= 0 (M == 0 is a no-op); ue8m0 in
 * {0, 1}.  Inputs are finite (NaN/Inf in x give unspecified codes).
 */
sgq_status sgq_quant_token_group(const void* x, int64_t M, int64_t K, int group,
                                 int ue8m0, void* xq, float* xs, sgq_stream_t stream);

/*
 * Weight block quantisation (offline; produces the GEMM's Wq/Ws).
 *
 * One scale per [blk_n, blk_k] tile of W, stored [n_blocks, k_blocks]:
 * sglang PR #42604, Motivation ([32,32] and [128,128] weight blocks) and the
 * vLLM "scaled_mm" API page, XPUFp8BlockScaledMMKernel
 * (process_weights_after_loading: "[n_blocks, k_blocks]", one value per
 * block tile; ragged N keeps ceil(N/blk_n) rows).  The rule per tile is the
 * one of sgq_quant_token_group with amax taken over the whole tile (the last
 * N-tile uses only the rows that exist).
 *
 * w: bf16 [N, K].  wq: uint8 E4M3 [N, K].  ws: fp32 [ceil(N/blk_n), K/blk_k].
 * blk_n in {32, 128}, blk_k in {32, 128}, K % blk_k == 0, N >= 0.
 */
sgq_status sgq_quant_weight_block(const void* w, int64_t N, int64_t K, int blk_n,
                                  int blk_k, int ue8m0, void* wq, float* ws,
                                  sgq_stream_t stream);

/*
 * UE8M0 scale bytes.  A power-of-two scale 2^(e - 127) is held as the one
 * byte e (its biased exponent; 255 is NaN): the format of the block-scaled
 * MMA's scale factors, and of the scale buffers that sglang PR #42604
 * prepares (Modifications: "prepares block32 scale buffers", keeping "UE8M0
 * activation rounding").  Bytes carry the scales in a quarter of the fp32
 * bytes, and the GEMM reads them without conversion.
 *
 * sgq_quant_token_group_ue8m0: sgq_quant_token_group with ue8m0 = 1 (the
 * same codes, bit for bit), each group's scale written as its UE8M0 byte.
 * xe: uint8 [M, K/group], 16-byte aligned.
 *
 * sgq_scales_to_ue8m0: e[i] = UE8M0 byte of s[i], i < n, for fp32 scales
 * that are positive normal powers of two (the weight scales of
 * sgq_quant_weight_block with ue8m0 = 1, converted once at load time).  Any
 * other value gives 255 and sets the device status (sgq_device_status ->
 * SGQ_ERR_INVALID_ARG).
 */
sgq_status sgq_quant_token_group_ue8m0(const void* x, int64_t M, int64_t K, int group, void* xq,
                                       uint8_t* xe, sgq_stream_t stream);
sgq_status sgq_scales_to_ue8m0(const float* s, int64_t n, uint8_t* e, sgq_stream_t stream);

/*
 * Block-scaled FP8 GEMM, "NT" form.
 *
 * Defined by the vLLM "scaled_mm" API page, AiterInt8ScaledMMLinearKernel.
 * apply_weights docstring (output = mm(scale_a * a, scale_b * b) with
 * numpy-style broadcasting of the scales) in the layout of sglang PR #42604,
 * Modifications: fp8_gemm_nt((Aq, As), (Wq, Ws), D, recipe=(1, blk_n, blk_k)),
 * B given as [N, K]:
 *
 *   D[m,n] = bf16_RNE( sum_k  Aq[m,k] * As[m, k/blk_k]
 *                            * Wq[n,k] * Ws[n/blk_n, k/blk_k] )
 *
 * with fp32 accumulation (any order).  The activation group size equals blk_k.
 *
 * Aq: uint8 E4M3 [M, K].          As: fp32 [M, K/blk_k].
 * Wq: uint8 E4M3 [N, K].          Ws: fp32 [ceil(N/blk_n), K/blk_k].
 * D:  bf16 [M, N] (written, never read).
 * blk_n in {32, 128}; blk_k in {32, 128}; K % blk_k == 0; K > 0; N % 8 == 0
 * (16-byte D rows); N may be ragged with respect to blk_n; M >= 0 (M == 0 is
 * a no-op).  Scales must be finite and > 0.
 *
 * When every scale of a 128-wide K step is an exact power of two (UE8M0),
 * the GEMM applies it inside the tensor-core block-scale MMA; any other fp32
 * scale is applied in an fp32 promotion step.  Both give the same result up
 * to fp32 rounding.
 *
 * Launch overlap (programmatic dependent launch): the GEMM and
 * sgq_quant_token_group are launched so that each may start while the
 * previous kernel on the stream is still running, and each lets its own
 * successor start as soon as it has started.  sgq_quant_token_group touches
 * memory only after the previous kernel has finished.  The GEMM reads Aq/As,
 * and writes D, only after the previous kernel has finished, but it starts
 * reading Wq and Ws at once, possibly while earlier kernels of an unbroken
 * run of sgq kernels on the stream are still running.  So Wq/Ws must not be
 * written by any kernel on the stream after the last host synchronisation
 * (or non-kernel stream operation: copy, memset) that precedes the GEMM;
 * weights written once at load time meet this.
 */
sgq_status sgq_fp8_block_gemm(const void* Aq, const float* As, const void* Wq,
                              const float* Ws, void* D, int64_t M, int64_t N, int64_t K,
                              int blk_n, int blk_k, sgq_stream_t stream);

/* sgq_fp8_block_gemm with SGQ_GEMM_* flags. */
sgq_status sgq_fp8_block_gemm_ex(const void* Aq, const float* As, const void* Wq,
                                 const float* Ws, void* D, int64_t M, int64_t N, int64_t K,
                                 int blk_n, int blk_k, uint32_t flags, sgq_stream_t stream);

/*
 * sgq_fp8_block_gemm without any device allocation.  No counterpart in the
 * paper: this is a deployment variant of the GEMM above.
 *
 * Who needs it: callers that cannot let a library allocate device memory --
 * a serving engine that reserves nearly all of HBM for its own memory pool
 * up front (a later cudaMalloc fails or fragments that pool), or a host whose
 * allocator must account for every byte.  sgq_fp8_block_gemm allocates a
 * split-K workspace on first use; this entry point instead keeps that
 * scratch in a fixed device array that is part of the library image
 * (16 MiB of fp32 partial tiles plus 64 KiB of arrival counters), held by
 * every GPU that loads the library until the process exits.  It calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *
 * Same arguments as sgq_fp8_block_gemm (flags = SGQ_GEMM_DEFAULT) and the
 * same launch plan wherever that plan's split-K partials and counters fit the
 * fixed array; D is then bit-identical to sgq_fp8_block_gemm's.  Where they
 * would not fit, the plan takes fewer K splits (or, for 64 < M <= 1024, the
 * 128 x 256 tiles, which need no split-K), and D agrees with
 * sgq_fp8_block_gemm's within the GEMM tolerance (a different fp32 summation
 * order).  SGQ_ERR_UNSUPPORTED, before anything is launched, remains only for
 * a plan that still needs more scratch than the array holds.  Shapes that need
 * no split-K (large M, or few K blocks) never touch the array.
 *
 * The first call on each device looks up the array's device address (with
 * that device current); make that first call before any CUDA stream capture.
 * Every call shares the one array and it keeps the previous call's contents:
 * each call clears the arrival counters it uses (an asynchronous memset on
 * `stream`), and calls that overlap on the GPU -- on different streams, or
 * from several host threads -- race on the array and must be avoided.
 */
sgq_status sgq_fp8_block_gemm_noalloc(const void* Aq, const float* As, const void* Wq,
                                      const float* Ws, void* D, int64_t M, int64_t N, int64_t K,
                                      int blk_n, int blk_k, sgq_stream_t stream);

/*
 * sgq_fp8_block_gemm_ex with UE8M0 scale bytes: Ae uint8 [M, K/blk_k] and
 * We uint8 [ceil(N/blk_n), K/blk_k] in place of As and Ws (16-byte aligned;
 * byte e is the scale 2^(e - 127)).  D is bit-identical to
 * sgq_fp8_block_gemm_ex with the fp32 scales 2^(e - 127) and
 * SGQ_GEMM_SCALES_POW2 (which this call implies).  Flags: as for
 * sgq_fp8_block_gemm_ex, without SGQ_GEMM_TEST_TIMEOUT.  Where the
 * two-accumulator tiles take the shape they read the bytes directly; other
 * plans (e.g. decode sizes) first widen them to fp32 in a library buffer,
 * allocated on the first call that needs it (not inside a stream capture;
 * grown, with a device synchronisation, when a larger shape needs more).  A
 * byte of 255 is reported as SGQ_ERR_INVALID_ARG by sgq_device_status where
 * the bytes are read directly.
 */
sgq_status sgq_fp8_block_gemm_ue8m0(const void* Aq, const uint8_t* Ae, const void* Wq, const uint8_t* We,
                                    void* D, int64_t M, int64_t N, int64_t K, int blk_n, int blk_k,
                                    uint32_t flags, sgq_stream_t stream);

/*
 * Quantise-and-multiply: the whole W8A8 linear layer in one call.
 *
 *   D = sgq_fp8_block_gemm(quant(x), Wq, Ws)   with
 *   quant(x) = sgq_quant_token_group(x, group = blk_k, ue8m0)
 *
 * x: bf16 [M, K] (device).  Wq, Ws, D, M, N, K, blk_n, blk_k: as for
 * sgq_fp8_block_gemm.  xq (uint8 E4M3 [M, K]) and xs (fp32 [M, K/blk_k]):
 * both NULL or both given; when given they receive the quantised activations,
 * bit-identical to sgq_quant_token_group's.  The result D is bit-identical to
 * sgq_quant_token_group followed by sgq_fp8_block_gemm.
 *
 * No counterpart in the pages as one call; it fuses the two steps above.
 * With xq/xs given it runs the two kernels back to back, with xq/xs as
 * scratch (measured faster than the single kernel).  With xq/xs NULL, for
 * decode-sized M (<= 64) with K/blk_k a multiple of 4 and at least 8
 * (blk_k = 128) or 16 (blk_k = 32) -- every decode shape the pages use -- it
 * is ONE kernel: the GEMM's epilogue warps quantise each bf16 activation tile
 * into shared memory, so the codes never go through HBM and a launch
 * disappears; any other shape returns SGQ_ERR_UNSUPPORTED before launching.
 * Errors and the launch-overlap contract: as for sgq_fp8_block_gemm (x is
 * read only after the preceding kernel has finished).
 */
sgq_status sgq_fp8_block_linear(const void* x, int ue8m0, const void* Wq, const float* Ws,
                                void* D, int64_t M, int64_t N, int64_t K, int blk_n, int blk_k,
                                void* xq, float* xs, sgq_stream_t stream);

/*
 * V2 per-token-group quantisation: the same rule as sgq_quant_token_group,
 * with the V2 options of "Sgl project Sglang GEMM Interface", Quantization
 * Routines and Signature (fuse_silu_and_mul, masked_m).
 *
 * x: bf16 [E, T, W] row-major, W = 2H when fuse_silu_and_mul (each row is
 * [gate | up]) else W = H.  The value quantised is y = silu(gate) * up in fp32
 * with silu(g) = g / (1 + exp(-g)) (exp: Cody-Waite reduction and a degree-7
 * Taylor polynomial, so the result is reproducible bit for bit), or x itself.
 * xq: E4M3 [E, T, H]; xs: fp32 [E, T, H/group].  masked_m: int32 [E] on the
 * device, or NULL for all T rows: rows t >= masked_m[e] of expert e are not
 * read or written.  group in {32, 128}, H % group == 0, ue8m0 and
 * fuse_silu_and_mul in {0, 1}.  E or T == 0 is a no-op.
 */
sgq_status sgq_quant_token_group_v2(const void* x, int64_t E, int64_t T, int64_t H, int group,
                                    int ue8m0, int fuse_silu_and_mul, const int32_t* masked_m,
                                    void* xq, float* xs, sgq_stream_t stream);

/*
 * Per-token and per-tensor quantisation, and the per-tensor / per-channel
 * scaled GEMM: "Sgl project Sglang GEMM Interface", Quantization Routines and
 * Signature (sgl_per_token_quant_fp8, sgl_per_tensor_quant_fp8 with static or
 * dynamic scaling, fp8_scaled_mm with per-tensor or per-row scale_a,
 * per-tensor or per-column scale_b, optional bias).  The quantisation rule is
 * sgq_quant_token_group's with the group spanning a whole row (per token) or
 * the whole tensor (per tensor, dynamic); there is no UE8M0 option.
 *
 * sgq_quant_per_token: x bf16 [M, K] -> xq E4M3 [M, K], xs fp32 [M].
 *   K > 0, K % 16 == 0, M >= 0 (M == 0 is a no-op).
 * sgq_quant_per_tensor: x bf16 [n] (any shape, n elements) -> xq E4M3 [n].
 *   is_static = 0: xs[0] receives max(amax, 1e-10) / 448 over the tensor.
 *   is_static = 1: xs[0] is read as the scale.  n % 16 == 0.  Dynamic scaling
 *   keeps per-block maxima in a fixed device array of the library: calls that
 *   overlap on the GPU (other streams, other host threads) must be avoided.
 * sgq_fp8_scaled_mm: D[m, n] = bf16((sum_k Aq[m,k] Wq[n,k]) * sa[m] * sb[n]
 *   + bias[n]), fp32 accumulation, with sa of sa_n = 1 (per tensor) or M (per
 *   row) values, sb of sb_n = 1 or N (per column) values, bias bf16 [N] or
 *   NULL.  Aq [M, K] and Wq [N, K] E4M3 (B given as [N, K], like the block
 *   GEMM).  K % 32 == 0, N % 8 == 0; pointers 16-byte aligned.  Launch
 *   overlap and errors: as for sgq_fp8_block_gemm.
 */
sgq_status sgq_quant_per_token(const void* x, int64_t M, int64_t K, void* xq, float* xs,
                               sgq_stream_t stream);
sgq_status sgq_quant_per_tensor(const void* x, int64_t n, int is_static, void* xq, float* xs,
                                sgq_stream_t stream);
sgq_status sgq_fp8_scaled_mm(const void* Aq, const float* sa, int64_t sa_n, const void* Wq,
                             const float* sb, int64_t sb_n, const void* bias, void* D, int64_t M,
                             int64_t N, int64_t K, sgq_stream_t stream);

/* Human-readable name of a status code (static string, never NULL). */
const char* sgq_status_string(sgq_status s);

/*
 * Synchronises `stream`, then reads and clears the library's device status
 * word on the current device.  Returns SGQ_OK, SGQ_ERR_TIMEOUT (a bounded
 * device-side wait ran out; the kernel returned early and its outputs are
 * undefined), SGQ_ERR_INVALID_ARG (a GEMM called with SGQ_GEMM_SCALES_POW2
 * met a scale that is not a power of two; its D is undefined) or
 * SGQ_ERR_CUDA (the synchronisation itself failed).
 */
sgq_status sgq_device_status(sgq_stream_t stream);

/* Number of kernels this library has launched in this process. */
uint64_t sgq_launch_count(void);

/*
 * Bytes of device memory the library has allocated on the current device in
 * this process (the split-K workspace and its counters; 0 until the first GEMM
 * that needs them, and always 0 for a process that uses only the
 * allocation-free GEMM and the quantisers).  Host only; 0 without a device.
 */
uint64_t sgq_allocated_bytes(void);

/*
 * The launch plan sgq_fp8_block_gemm would use for this problem on a device
 * with `sm_count` SMs; host only (no device is touched), for tests and tools.
 * out (host, 8 entries, caller-owned): [0] 1 for swap-AB tiles (weights on the
 * MMA's 128-row side), [1] tile width BN (tokens for swap-AB, else columns),
 * [2] K splits, [3] work items (tiles x splits), [4] persistent grid before
 * the occupancy cap, [5] 1 for two alternating MMA issuers, [6] 1 for split-K
 * summed inside clusters of two, [7] 1 for CTA pairs.  SGQ_ERR_INVALID_ARG for
 * out == NULL, M, N or K < 1, blk_k not 32 or 128, or sm_count < 1.
 */
sgq_status sgq_gemm_plan(int64_t M, int64_t N, int64_t K, int blk_k, int sm_count, int32_t* out);

/*
 * The plan of the two-accumulator tiles that sgq_fp8_block_gemm_ex with
 * SGQ_GEMM_SCALES_POW2 (e8 = 0), or sgq_fp8_block_gemm_ue8m0 (e8 = 1), would
 * use on a device with `sm_count` SMs; host only (no device is touched), for
 * tests and tools.  The kernel computes the same D = (Aq * As)(Wq * Ws)^T as
 * sgq_fp8_block_gemm (sglang PR #42604, Modifications: fp8_gemm_nt with a
 * (1, blk_n, blk_k) recipe).  out (host, 8 entries, caller-owned):
 * [0] mode: 0 = these tiles are not used (sgq_gemm_plan's plan applies; byte
 * scales are widened to fp32 first), 1 = one CTA per 256-row tile, 2 = K split
 * over CTAs, 3 = CTA pairs on 512-row tiles; then, for modes 1-3: [1] tile
 * width in weight rows (192 or 224), [2] K splits, [3] work items (tiles x
 * splits), [4] grid in CTAs, [5] tiles, [6] K stages (of 128) per split,
 * [7] 0.  SGQ_ERR_INVALID_ARG for out == NULL, M, N or K < 1, blk_k not 32 or
 * 128, sm_count < 2, or e8 not 0 or 1.
 */
sgq_status sgq_gemm_plan_pow2(int64_t M, int64_t N, int64_t K, int blk_k, int sm_count, int e8, int32_t* out);

/* Library ABI version (major * 100 + minor). */
int sgq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SGQ_H_ */
