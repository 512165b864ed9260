/*
 * snip.h -- C ABI of the quantized linear layer for sub-byte mixed-precision
 * LLM training on GB300 (sm_103a).
 *
 * What it computes (page title, section):
 *  - "SNIP: An Adaptive Mixed Precision Framework for Subbyte Large Language
 *    Model Training", Figure 5: a linear layer whose forward GEMM Y = X W^T,
 *    dgrad dX = dY W and wgrad dW = dY^T X run in the layer's low precision,
 *    each operand quantized along that GEMM's own contraction dimension;
 *    Abstract / Figure 2: one format (FP8 or FP4) per layer, chosen by a plan;
 *    periodic statistics on activations, weights and gradients.
 *  - "FP4 all the way" (Chmiel, Fishman, Banner, Soudry), summary page,
 *    Outline: the FP4 format is NVFP4 -- blocks of 16 E2M1 values sharing one
 *    E4M3 scale -- with round-to-nearest in the forward pass and stochastic
 *    rounding in the backpropagation and update passes; quantized training
 *    loses efficiency once the gradient norm drops below about sqrt(3) times
 *    the quantization noise.
 *  - "Research on Mixed-Precision Training for LLMs", stochastic rounding
 *    paragraph: round up or down with probabilities that keep the expected
 *    value.
 *
 * Conventions for every entry point
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library
 *    allocates no device memory (except tensor memory inside its GEMM kernels,
 *    which is freed before each kernel exits), links no other GPU library and
 *    keeps no device state beyond the fixed scratch array of
 *    snip_tensor_scales_noalloc.  Host pointers are marked.
 *  - Tensors are dense row-major.  bf16 inputs are passed as `const void*` to
 *    2-byte IEEE bfloat16 values.  Device pointers must be 16-byte aligned
 *    (SNIP_ERR_ALIGN otherwise).
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream).  Argument errors are returned synchronously and launch
 *    nothing.  Errors found on the device (non-finite input, a kernel wait
 *    that timed out) are OR-ed into the status word of the caller's workspace
 *    and read with snip_workspace_status().  The quantizer and GEMM kernels
 *    are launched with programmatic dependent launch: the next kernel on the
 *    stream may be scheduled while one ends, but each waits for the work
 *    before it on the stream to finish before it reads or writes memory, so
 *    stream order holds as for ordinary launches.
 *  - Workspace: a caller-owned device buffer of at least the size returned by
 *    the matching *_workspace_size() call.  Its first SNIP_WS_HEADER_BYTES hold
 *    the sticky device status word; initialise them once with
 *    snip_workspace_init().  Calls that share a workspace must be ordered on
 *    one stream.
 *  - Sizes: a tensor dimension above 2^31 - 1, or a tensor (operand or GEMM
 *    output) of more than 2^40 elements, is SNIP_ERR_SHAPE (the kernels count
 *    tiles and segments in 32 bits and address TMA boxes with 32-bit
 *    coordinates).  Empty tensors are accepted wherever the entry point's
 *    text does not require a positive size: nothing is written to their
 *    outputs, and a tensor scale computed from no elements is 1.
 *  - Random bits for stochastic rounding come from Philox4x32-10 (Salmon et
 *    al., SC'11) keyed by `seed`; source element e (row-major index into the
 *    tensor being quantized, whatever the output orientation) uses 16 bits of
 *    the call with counter (e/8, stream_id): word (e/2) mod 4, low half for
 *    even e.  A result is therefore a pure function of (input, seed,
 *    stream_id).
 */
#ifndef SNIP_H
#define SNIP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SNIP_OK = 0,
    SNIP_ERR_INVALID_ARG = 1,       /* null pointer, bad enum, negative size    */
    SNIP_ERR_SHAPE = 2,             /* a dimension breaks the multiple-of-16 rule */
    SNIP_ERR_ALIGN = 3,             /* a device pointer is not 16-byte aligned  */
    SNIP_ERR_NONFINITE = 4,         /* (device) the input held an Inf or NaN     */
    SNIP_ERR_TIMEOUT = 5,           /* (device) a kernel wait gave up            */
    SNIP_ERR_CUDA = 6,              /* a CUDA runtime call failed                */
    SNIP_ERR_UNSUPPORTED_DEVICE = 7,/* the current device is not sm_103          */
    SNIP_ERR_WORKSPACE = 8          /* workspace missing or too small            */
} snip_status;

/* FP8_E4M3: one fp32 tensor scale.  NVFP4: 16 E2M1 values per E4M3 block
 * scale, plus an fp32 tensor scale ("FP4 all the way", Outline).  MXFP4: 32
 * E2M1 values per E8M0 power-of-two block scale, no tensor scale (OCP
 * Microscaling Formats v1.0; the block-size / scale-format alternative that
 * the FP4 study weighs NVFP4 against).  FP8_E5M2: one fp32 tensor scale
 * s = amax / 57344, for gradients; as a GEMM format it means A in E5M2 and B
 * in E4M3.  FP8_E5M2_GRAD is a layer format only (plans): E5M2 for dY and
 * dY^T, E4M3 for X, W, W^T and X^T.  NVFP4_B32 / _B64 / _B128: NVFP4's
 * elements, scales and tensor scale with 32, 64 or 128 values per E4M3
 * scale (the block-size axis of the FP4 study, "FP4 all the way", Outline);
 * they are stored in NVFP4's layouts with each scale repeated for every 16
 * elements it covers, so they are NVFP4 operands to the GEMM, which gives
 * exactly the longer blocks' product. */
typedef enum {
    SNIP_FMT_FP8_E4M3 = 0,
    SNIP_FMT_NVFP4 = 1,
    SNIP_FMT_MXFP4 = 2,
    SNIP_FMT_FP8_E5M2 = 3,
    SNIP_FMT_FP8_E5M2_GRAD = 4,
    SNIP_FMT_NVFP4_B32 = 5,
    SNIP_FMT_NVFP4_B64 = 6,
    SNIP_FMT_NVFP4_B128 = 7
} snip_format;
typedef enum { SNIP_RTN = 0, SNIP_SR = 1 } snip_round;

/* Orientation of a quantization of a rows x cols tensor.
 * ALONG_COLS: blocks run along the last dim; the output has rows x cols.
 * ALONG_ROWS: blocks run along the first dim; the output is the transpose,
 *             cols x rows (output row i = input column i). */
typedef enum { SNIP_BLOCKS_ALONG_COLS = 0, SNIP_BLOCKS_ALONG_ROWS = 1 } snip_orient;

/* Output layout of a quantization (OR x OC = output rows x contraction).
 * ROWMAJOR: NVFP4 codes OR x OC/2 bytes (element 2j in bits 0..3 of byte j,
 *           bit 3 of each code the sign), E4M3 scales OR x OC/16 bytes;
 *           MXFP4 codes the same, E8M0 scales OR x OC/32 bytes;
 *           FP8 (E4M3 or E5M2) codes OR x OC bytes.
 * MMA:      the GEMM operand layout.  Rows are padded to ORp = roundup(OR,256)
 *           and the contraction to OCp = roundup(OC,256) for NVFP4 (128 for
 *           FP8), padding filled with zero codes and zero scales.  Codes are
 *           row-major ORp x OCp/2 (NVFP4) or ORp x OCp (FP8).  NVFP4 scales
 *           are stored in 512-byte chunks, one per (128-row group rg, group of
 *           four 16-element blocks kc): chunk index rg*(OCp/64) + kc, and row
 *           r, block kb at byte (r%32)*16 + ((r/32)%4)*4 + kb%4 of its chunk.
 *           MXFP4 codes as NVFP4 (OCp = roundup(OC,256)); its E8M0 scales use
 *           the same chunk image with 32-element blocks: chunk index
 *           rg*(OCp/128) + kc, kc a group of four 32-element blocks. */
typedef enum { SNIP_LAYOUT_ROWMAJOR = 0, SNIP_LAYOUT_MMA = 1 } snip_layout;

/* Index of each quantization inside a qlinear call; the Philox stream id of
 * quantization `tag` of layer `l` is l*8 + tag. */
typedef enum {
    SNIP_TAG_X_FWD = 0,      /* X, blocks along K, forward            */
    SNIP_TAG_W_FWD = 1,      /* W, blocks along K, forward            */
    SNIP_TAG_DY_DGRAD = 2,   /* dY, blocks along N, dgrad             */
    SNIP_TAG_WT_DGRAD = 3,   /* W^T, blocks along N, dgrad            */
    SNIP_TAG_DYT_WGRAD = 4,  /* dY^T, blocks along T, wgrad           */
    SNIP_TAG_XT_WGRAD = 5    /* X^T, blocks along T, wgrad            */
} snip_tag;

#define SNIP_WS_HEADER_BYTES 256
#define SNIP_STATS_NVALS 8

/* Slots of the raw statistics vector written by snip_quant_stats. */
enum {
    SNIP_ST_SUM_X2 = 0,       /* ||A||^2                                              */
    SNIP_ST_NVFP4_ERR2 = 1,   /* ||Q_nvfp4(A) - A||^2 under the requested rounding     */
    SNIP_ST_FP8_ERR2 = 2,     /* ||Q_fp8(A) - A||^2 under the requested rounding       */
    SNIP_ST_NVFP4_SRVAR = 3,  /* sum (hi-|y|)(|y|-lo) q^2: expected SR error^2, NVFP4   */
    SNIP_ST_FP8_SRVAR = 4,    /* the same on the FP8 grid                               */
    SNIP_ST_AMAX = 5,         /* max |A|                                              */
    SNIP_ST_COUNT = 6         /* number of elements                                   */
};

typedef struct {
    double sum_x2, nvfp4_err2, fp8_err2, nvfp4_sr_var, fp8_sr_var, amax, count;
    double ratio_nvfp4;        /* ||A|| / ||Q_nvfp4(A) - A|| (+inf when the error is 0) */
    double ratio_fp8;
    int below_sqrt3_nvfp4;     /* ratio < sqrt(3): the "FP4 all the way" threshold      */
    int below_sqrt3_fp8;
} snip_stats;

typedef struct snip_plan snip_plan;

/* ---------------------------------------------------------------- misc */

/* Text of a status code (static storage). */
const char* snip_status_string(snip_status s);

/* ABI version (major*10000 + minor*100 + patch) of this header; snip_version()
 * returns the library's, which must match.  0.2.0: snip_requant gained the
 * column-block fields (NEXT-3), the longer-block NVFP4 formats,
 * snip_quantize_part and snip_wait_check.  0.3.0: snip_qlinear_fwd_multi;
 * snip_dw_noise needs only the small workspace (no K x N buffer). */
#define SNIP_ABI_VERSION 300
int snip_version(void);

/* SNIP_OK if the current CUDA device can run the kernels (compute capability
 * 10.3), else SNIP_ERR_UNSUPPORTED_DEVICE (or SNIP_ERR_CUDA). */
snip_status snip_device_check(void);

/* Self-check of the failure path shared by every pipeline wait in the GEMMs:
 * a one-CTA kernel waits on an mbarrier phase that nothing completes.  After
 * limit_ns (clamped to [1 us, 1 s]) the wait gives up, raises the timeout bit
 * of the workspace status word (snip_workspace_status then reports
 * SNIP_ERR_TIMEOUT) and sets the CTA's abort flag, on which a second waiting
 * thread with a 4x longer limit gives up too.  out (device, 3 uint32):
 * {1 if the first wait completed else 0, the same for the second wait, the
 * second thread's ns in its wait}.  No trap or fault: the context stays
 * usable.  ws: at least SNIP_WS_HEADER_BYTES. */
snip_status snip_wait_check(uint64_t limit_ns, uint32_t* out, void* ws, size_t ws_bytes, void* stream);

/* Zero the status word of a workspace (async on `stream`). */
snip_status snip_workspace_init(void* ws, size_t ws_bytes, void* stream);

/* Synchronize `stream`, read the workspace's device status word and return
 * it as a status code in *device_status: SNIP_OK, SNIP_ERR_NONFINITE or
 * SNIP_ERR_TIMEOUT (the first of those that any kernel raised since the last
 * snip_workspace_init).  *device_status is host memory. */
snip_status snip_workspace_status(const void* ws, void* stream, snip_status* device_status);

/* ---------------------------------------------------------------- a1: amax */

/* Workspace bytes for snip_amax / snip_quantize_* / snip_quant_stats. */
size_t snip_quantize_workspace_size(int64_t rows, int64_t cols);

/* amax_out[0] = max |x| over n bf16 elements (exact; the max of fp32 values
 * widened from bf16).  A non-finite element raises SNIP_ERR_NONFINITE in the
 * workspace status and writes NaN.  n may be 0 (result 0). */
snip_status snip_amax(const void* x, int64_t n, float* amax_out, void* ws, size_t ws_bytes, void* stream);

/* scales_out (device, 3 floats) = {amax, g, s}: amax = max |x| over n bf16
 * elements, g = amax / 2688 the NVFP4 tensor scale and s = amax / 448 the FP8
 * tensor scale (g = s = 1 when amax is 0), each a single fp32 division.
 * Pass scales_out + 1 as g_in of snip_quantize_nvfp4, scales_out + 2 as s_in of
 * snip_quantize_fp8, or scales_out as scales_in of snip_quant_stats, to reuse
 * one amax pass for several quantizations of the same tensor.  A non-finite
 * element raises SNIP_ERR_NONFINITE in the workspace status and writes NaN. */
snip_status snip_tensor_scales(const void* x, int64_t n, float* scales_out, void* ws, size_t ws_bytes,
                               void* stream);

/* The tensor scales of up to 8 tensors in one launch (as snip_tensor_scales
 * for each; one launch spreads its CTAs over the tensors in proportion to
 * their sizes).  xs[t] (device bf16, 16-byte aligned) holds ns[t] elements;
 * scales_out[t] (device, 3 floats) receives {amax, g, s}.  count in [1, 8]
 * (SNIP_ERR_INVALID_ARG otherwise).
 * ws as for snip_tensor_scales; its status word flags non-finite input. */
snip_status snip_tensor_scales_multi(int count, const void* const* xs, const int64_t* ns, float* const* scales_out,
                                     void* ws, size_t ws_bytes, void* stream);

/* Variant of snip_tensor_scales that needs no workspace and allocates nothing,
 * for callers that cannot allocate device memory at the point of the call:
 * code inside a framework whose caching allocator owns all device memory and
 * forbids raw cudaMalloc, or a path where an allocation (which may
 * synchronize the device) is not allowed.  It is an ordinary host-side CUDA
 * call: like every entry point here it must not be made from a host function
 * enqueued with cudaLaunchHostFunc, where CUDA forbids all CUDA calls.
 * The pages have no counterpart of this call; it exists for such callers.
 * x: device bf16, n elements, at most 2^30 (SNIP_ERR_SHAPE beyond that);
 * scales_out: device, 3 floats {amax, g, s} as for snip_tensor_scales; a
 * non-finite element makes them NaN (there is no status word to read).
 * The kernel's scratch is one fixed 64 KB device array shared by every call
 * on a device and kept until the process exits: calls that overlap on the GPU
 * (different streams without ordering) race on it and must not be issued.
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress), which may load the library's device code on that
 * device; make that first call outside any stream capture. */
snip_status snip_tensor_scales_noalloc(const void* x, int64_t n, float* scales_out, void* stream);

/* ---------------------------------------------------------------- a2/a3: NVFP4 */

/* NVFP4 quantization of a bf16 rows x cols tensor ("FP4 all the way",
 * Outline: 16 E2M1 values share one E4M3 scale), with a per-tensor fp32 scale
 * g above the block scales:
 *   g   = amax / 2688 (2688 = 6 * 448; g = 1 for an all-zero tensor), or *g_in;
 *   s_b = E4M3(amax_block / (6 g)), round to nearest even, saturating at 448;
 *   p   = decode(s_b) * g; y = |x| * (1/p) in fp32;
 *   code = sign(x) | E2M1(y): nearest with ties to the even code (rnd = RTN)
 *          or stochastic with 16 Philox bits (rnd = SR), y >= 6 -> 6; a zero
 *          element, or a block whose p is 0, encodes to magnitude 0.
 * x          device, rows x cols bf16.  The blocked dim (cols for ALONG_COLS,
 *            rows for ALONG_ROWS) must be a multiple of 16 (SNIP_ERR_SHAPE).
 * g_in       device float or NULL (NULL: compute from amax).
 * codes, scales   device outputs in `layout` (see snip_layout); sizes from
 *            snip_quantized_bytes().
 * g_out      device float: the g used.
 * block_sqerr  device float OR x OC/16 (row-major, in output orientation) or
 *            NULL: per-block sum of squared dequantization error.
 * A non-finite input raises SNIP_ERR_NONFINITE in the workspace status; the
 * outputs are then unspecified and *g_out is NaN. */
snip_status snip_quantize_nvfp4(const void* x, int64_t rows, int64_t cols, snip_orient orient,
                                snip_round rnd, uint64_t seed, uint64_t stream_id, const float* g_in,
                                snip_layout layout, uint8_t* codes, uint8_t* scales, float* g_out,
                                float* block_sqerr, void* ws, size_t ws_bytes, void* stream);

/* NVFP4 with `block` (16, 32, 64 or 128) elements per E4M3 scale: every step
 * as snip_quantize_nvfp4 with the block maximum taken over `block` elements
 * ("FP4 all the way", Outline: the block-size axis of the FP4 study).  The
 * outputs use NVFP4's layouts (sizes from snip_quantized_bytes with
 * SNIP_FMT_NVFP4), each scale written once per 16 elements it covers, so
 * they feed snip_gemm as NVFP4 operands.  The blocked dim must be a multiple
 * of `block` (SNIP_ERR_SHAPE); any other block is SNIP_ERR_INVALID_ARG.
 * block = 16 is snip_quantize_nvfp4 (without block errors). */
snip_status snip_quantize_nvfp4_block(const void* x, int64_t rows, int64_t cols, snip_orient orient,
                                      snip_round rnd, uint64_t seed, uint64_t stream_id, const float* g_in,
                                      int block, snip_layout layout, uint8_t* codes, uint8_t* scales,
                                      float* g_out, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------- a4: FP8 */

/* FP8 E4M3 quantization with one fp32 tensor scale s = amax / 448 (1 for an
 * all-zero tensor) or *s_in: code = sign(x) | E4M3(|x| * (1/s)), nearest-even
 * with saturation at 448 (RTN) or stochastic with 16 Philox bits (SR).
 * Orientation, layout and errors as for snip_quantize_nvfp4 (no blocks, so
 * no multiple-of-16 rule beyond the MMA layout's padding). */
snip_status snip_quantize_fp8(const void* x, int64_t rows, int64_t cols, snip_orient orient,
                              snip_round rnd, uint64_t seed, uint64_t stream_id, const float* s_in,
                              snip_layout layout, uint8_t* codes, float* s_out,
                              void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------- NEXT-2: MXFP4 */

/* MXFP4 quantization (OCP Microscaling Formats v1.0), a format variant of the
 * FP4 study ("FP4 all the way", Outline: block size and scale format): per
 * block of 32 along the blocked dim, the E8M0 scale code is
 * max(exponent field of the block's largest |x| as bf16 - 2, 0), i.e.
 * 2^(floor(log2 amax) - 2) clamped at 2^-127; elements y = |x| * 2^-(code-127)
 * are rounded to E2M1 exactly as for NVFP4 (RTN nearest-even saturating at 6,
 * or SR with the same Philox bits per source element); there is no tensor
 * scale.  codes/scales sized by snip_quantized_bytes(SNIP_FMT_MXFP4, ...).
 * The blocked dim (cols for ALONG_COLS, rows for ALONG_ROWS) must be a
 * multiple of 32 and cols a multiple of 16 (SNIP_ERR_SHAPE).  A non-finite
 * input raises SNIP_ERR_NONFINITE in the workspace status (outputs
 * unspecified).  ws as for snip_quantize_nvfp4. */
snip_status snip_quantize_mxfp4(const void* x, int64_t rows, int64_t cols, snip_orient orient,
                                snip_round rnd, uint64_t seed, uint64_t stream_id, snip_layout layout,
                                uint8_t* codes, uint8_t* scales, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------- NEXT-2: FP8 E5M2 gradients */

/* FP8 E5M2 quantization with one fp32 tensor scale s = amax / 57344 (1 for an
 * all-zero tensor): code = sign | E5M2(|x| * (1/s)), nearest-even saturating at
 * 57344 (RTN) or stochastic with 16 Philox bits (SR) -- the gradient format of
 * the FP8 variant (a NEXT-2 format alternative; the pages' FP8 is E4M3).
 * amax_in (device, nullable): the tensor's amax (scales_out[0] of
 * snip_tensor_scales); NULL computes it.  s_out (device) receives s.
 * Orientation, layout and errors as for snip_quantize_fp8. */
snip_status snip_quantize_e5m2(const void* x, int64_t rows, int64_t cols, snip_orient orient,
                               snip_round rnd, uint64_t seed, uint64_t stream_id, const float* amax_in,
                               snip_layout layout, uint8_t* codes, float* s_out,
                               void* ws, size_t ws_bytes, void* stream);

/* Quantization of a part of a larger tensor, for a layer split by tokens
 * across devices (SNIP, Figure 5: every operand of the layer quantized along
 * its contraction dim; a token shard of X or dY is a block of whole rows):
 * x holds rows x cols of a row-major tensor starting at its element
 * index_base = first row * cols.  index_base must be a multiple of cols and
 * of 16, and with ALONG_ROWS the first row a multiple of the format's block
 * length (16; 32 for MXFP4 and NVFP4_B32, 64, 128 for the longer NVFP4
 * blocks), else SNIP_ERR_SHAPE: a block never straddles two parts.  These
 * argument rules are checked before anything touches the device.  It is
 * quantized as fmt (an operand format) with the whole tensor's scales
 * scales_in (device, {amax, g, s} as snip_tensor_scales writes them for the
 * whole tensor, e.g. from a MAX all-reduce of the parts' amax), and every
 * element draws the random bits of its index in the whole tensor ("FP4 all
 * the way", Outline: SR; the bits of element e are those of R6), so the codes
 * equal the whole tensor's quantization's output rows (ALONG_COLS) or columns
 * (ALONG_ROWS, the part's rows a whole number of blocks).  raw_out (device,
 * nullable, ALONG_COLS only): SNIP's statistics of this part under those
 * scales, in the same pass; the parts' sums add up to the whole tensor's
 * (SNIP_ST_AMAX: take the maximum).  Other arguments and errors as for
 * snip_quantize_nvfp4 / snip_quantize_stats. */
snip_status snip_quantize_part(snip_format fmt, const void* x, int64_t rows, int64_t cols, snip_orient orient,
                               snip_round rnd, uint64_t seed, uint64_t stream_id, uint64_t index_base,
                               const float* scales_in, snip_layout layout, uint8_t* codes, uint8_t* scales,
                               double* raw_out, void* ws, size_t ws_bytes, void* stream);

/* Bytes of the code and scale buffers of a quantization whose output has
 * out_rows rows and contraction out_cols, in `layout`.  Host-only. */
snip_status snip_quantized_bytes(snip_format fmt, snip_layout layout, int64_t out_rows, int64_t out_cols,
                                 size_t* codes_bytes, size_t* scales_bytes);

/* ---------------------------------------------------------------- a5-a7: GEMM */

/* D[m, n] = ga * gb * sum_k A[m, k] B[n, k] for m < M, n < N, fp32 output with
 * row pitch ldd (elements).  A (M rows) and B (N rows) are quantized operands
 * in the MMA layout with contraction K; ga/gb are device floats (NVFP4: the
 * tensor scales g; FP8: the tensor scales s; MXFP4: unused, may be NULL;
 * FP8_E5M2: A is E5M2 with its scale s5, B is E4M3 with its scale s).
 * NVFP4 uses the tensor cores' block-scaled FP4 MMA with E4M3 block scales
 * (scale_vec::4X), MXFP4 the same MMA with E8M0 scales (scale_vec::2X), FP8
 * the E4M3 x E4M3 MMA.  NVFP4_B32/_B64/_B128 operands are NVFP4 operands
 * (their repeated scales give the longer blocks' product exactly).  Accumulation is fp32.  Needs K % 16 == 0 (MXFP4:
 * K % 32 == 0) and ldd % 4 == 0, else SNIP_ERR_SHAPE; ldd >= N, else SNIP_ERR_INVALID_ARG.  Only D[m, n] with
 * m < M, n < N is written (a row pitch's padding is left as it was); M == 0 or N == 0 writes nothing and
 * returns SNIP_OK.
 * ws: at least SNIP_WS_HEADER_BYTES (status word; a timed-out wait raises
 * SNIP_ERR_TIMEOUT there). */
snip_status snip_gemm(snip_format fmt, const uint8_t* a_codes, const uint8_t* a_scales, const float* ga,
                      const uint8_t* b_codes, const uint8_t* b_scales, const float* gb,
                      int64_t M, int64_t N, int64_t K, float* D, int64_t ldd,
                      void* ws, size_t ws_bytes, void* stream);

/* NEXT-3: the GEMM whose product is the next layer's operand -- typically the
 * dgrad product dX, the preceding layer's dY -- also writes that operand
 * quantized, in both orientations, so the bf16 round trip and two separate
 * quantization passes go away ("SNIP", Figure 5: each GEMM operand quantized
 * along its own contraction dim; the preceding layer's dgrad contracts over
 * this dX's columns, its wgrad over its rows).  The product D = ga*gb*A B^T
 * is rounded to bf16 and quantized to NVFP4 with the given tensor scale (the
 * pages say nothing about when its amax is known: the caller passes one,
 * e.g. the previous step's amax_out / 2688; values beyond 6 * 448 * g
 * saturate):
 *   rows    (codes, scales; rnd, stream_id): 16-element blocks along the rows
 *           of D (along N) -- the M x N operand, as snip_quantize_nvfp4 with
 *           SNIP_BLOCKS_ALONG_COLS on bf16(D);
 *   columns (codes_t, scales_t; rnd_t, stream_id_t): 16-element blocks down
 *           the columns of D (along M) -- the N x M operand D^T, as
 *           snip_quantize_nvfp4 with SNIP_BLOCKS_ALONG_ROWS on bf16(D).
 * Each orientation is nearest or stochastic; stochastic rounding takes the
 * bits of element index m*N + n of its own stream (the same bits the
 * quantizer draws for bf16(D)).  Either orientation may be omitted (NULL
 * codes), not both.  codes / scales (device, 16-byte aligned): the MMA layout
 * of the M x N (rows) or N x M (columns) NVFP4 operand, sized by
 * snip_quantized_bytes(SNIP_FMT_NVFP4, SNIP_LAYOUT_MMA, ...); padding is
 * written as zeros.  amax_out (device, nullable) receives max |bf16(D)| of
 * this product, for the next scale. */
typedef struct {
    const float* g_in;
    int rnd;               /* snip_round of the row blocks */
    uint64_t seed;         /* both orientations */
    uint64_t stream_id;    /* row blocks */
    uint8_t* codes;        /* row blocks: M x N operand (nullable) */
    uint8_t* scales;
    float* amax_out;
    int rnd_t;             /* snip_round of the column blocks */
    uint64_t stream_id_t;  /* column blocks */
    uint8_t* codes_t;      /* column blocks: N x M operand D^T (nullable) */
    uint8_t* scales_t;
} snip_requant;

/* snip_gemm plus the re-quantized product described above; D (fp32) may be
 * NULL when only the quantized operand is wanted.  N % 16 == 0, and M % 16 ==
 * 0 when the column blocks are written, else SNIP_ERR_SHAPE.  Errors as for
 * snip_gemm; SNIP_ERR_INVALID_ARG for a null rq or rq->g_in, no orientation,
 * an orientation without its scales, or a rounding outside snip_round. */
snip_status snip_gemm_requant(snip_format fmt, const uint8_t* a_codes, const uint8_t* a_scales, const float* ga,
                              const uint8_t* b_codes, const uint8_t* b_scales, const float* gb,
                              int64_t M, int64_t N, int64_t K, float* D, int64_t ldd, const snip_requant* rq,
                              void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------- plan */

/* A per-layer precision plan (SNIP, Abstract: one format per layer).  formats
 * (host, n_layers entries) are snip_format values: FP8_E4M3, NVFP4, MXFP4,
 * FP8_E5M2_GRAD or NVFP4_B32/_B64/_B128 (not FP8_E5M2, an operand format; a
 * longer-block layer needs T, K and N multiples of its block).  Every layer starts with
 * the rounding of "FP4 all the way": RTN for the forward quantizations (tags
 * X_FWD, W_FWD) and SR for the four backward ones.  *out is a host object
 * owned by the caller (snip_plan_destroy). */
snip_status snip_plan_create(int n_layers, const int* formats, uint64_t seed, snip_plan** out);
snip_status snip_plan_set_rounding(snip_plan* plan, int layer, snip_tag tag, snip_round rnd);
snip_status snip_plan_get(const snip_plan* plan, int layer, snip_format* fmt, uint64_t* seed);
void snip_plan_destroy(snip_plan* plan);

/* ---------------------------------------------------------------- qlinear */

/* Workspace bytes for snip_qlinear_fwd / snip_qlinear_bwd of this layer. */
size_t snip_qlinear_workspace_size(const snip_plan* plan, int layer, int64_t T, int64_t K, int64_t N);

/* Forward (SNIP Figure 5): Y = Q(X) Q(W)^T.  X device T x K bf16, W device
 * N x K bf16, Y device T x N fp32.  Both quantized along K in the layer's
 * format with the plan's rounding (default RTN), stream ids layer*8+{0,1}.
 * T, K, N multiples of 16 (32 for an MXFP4 layer).  stats_out (device, nullable, 2 x SNIP_STATS_NVALS
 * doubles): SNIP's statistics of X then of W (as snip_quant_stats with the
 * forward rounding), computed inside the forward quantization passes. */
snip_status snip_qlinear_fwd(const snip_plan* plan, int layer, const void* X, const void* W,
                             int64_t T, int64_t K, int64_t N, float* Y, double* stats_out,
                             void* ws, size_t ws_bytes, void* stream);

/* Forward of several layers that read one activation (SNIP, Figure 4: Q, K
 * and V read the same X, Gate and Up another): for i < count,
 * Y[i] = Q(X) Q(W[i])^T exactly as snip_qlinear_fwd(plan, layers[i], ...)
 * computes it, with X's tensor scales and statistics computed once and X's
 * quantization once per group of layers that quantize it alike (same
 * forward format, round-to-nearest X_FWD rounding: the stream id is then
 * irrelevant); a layer whose X_FWD rounding is stochastic quantizes X with
 * its own stream id.  count in [1, 8]; layers (host) distinct layer indices;
 * X device T x K bf16; W (host array) device N[i] x K bf16; N (host array);
 * Y (host array) device T x N[i] fp32.  stats_x (device, nullable,
 * SNIP_STATS_NVALS doubles): SNIP's statistics of X under the forward
 * rounding; stats_w (host array or NULL; entries device or NULL): those of
 * W[i].  ws: snip_qlinear_fwd_multi_workspace_size bytes.  Shape and
 * argument rules as snip_qlinear_fwd for every layer. */
size_t snip_qlinear_fwd_multi_workspace_size(const snip_plan* plan, int count, const int* layers, int64_t T,
                                             int64_t K, const int64_t* N);
snip_status snip_qlinear_fwd_multi(const snip_plan* plan, int count, const int* layers, const void* X,
                                   const void* const* W, int64_t T, int64_t K, const int64_t* N, float* const* Y,
                                   double* stats_x, double* const* stats_w, void* ws, size_t ws_bytes,
                                   void* stream);

/* Backward (SNIP Figure 5): dX = Q(dY) Q(W^T)^T (dY and W^T quantized along
 * N) and dW = Q(dY^T) Q(X^T)^T (both quantized along T), stochastic rounding
 * by default ("FP4 all the way", Outline), stream ids layer*8+{2,3,4,5}.
 * dY device T x N bf16, dX device T x K fp32, dW device N x K fp32.
 * stats_out (device, nullable, SNIP_STATS_NVALS doubles): SNIP's statistics of
 * dY under the dgrad rounding and stream (layer*8+2), computed inside dY's
 * dgrad quantization pass. */
snip_status snip_qlinear_bwd(const snip_plan* plan, int layer, const void* X, const void* W,
                             const void* dY, int64_t T, int64_t K, int64_t N, float* dX, float* dW,
                             double* stats_out, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------- NEXT-3: the backward chain */

/* SNIP, Figure 5 chains the linears: a layer's dX is the gradient dY of the
 * layer before it.  snip_qlinear_bwd_chain runs `layer`'s backward exactly
 * as snip_qlinear_bwd, except that its dgrad GEMM also writes its product,
 * rounded to bf16, as the preceding layer prev_layer's two gradient operands
 * (the re-quantizing epilogue of snip_gemm_requant): row blocks along K
 * (prev_layer's dgrad operand, its DY_DGRAD rounding and stream id
 * prev_layer*8+2) and column blocks along T (its wgrad operand dY^T,
 * DYT_WGRAD rounding, stream id prev_layer*8+4), NVFP4 in the MMA layout,
 * quantized with the given tensor scale g_prev (device float; a delayed
 * scale such as the previous step's amax_prev / 2688: the product's own
 * amax is known only after it is formed).  amax_prev (device float,
 * nullable) receives max |bf16(dX)|.  dX (fp32) may be NULL.
 * prev_layer's format must be NVFP4 (SNIP_ERR_INVALID_ARG otherwise).
 * Buffer sizes: snip_quantized_bytes(NVFP4, MMA, T, K) for prev_codes /
 * prev_scales, (NVFP4, MMA, K, T) for prev_codes_t / prev_scales_t.
 * The identity stands between the two layers: the pages place no function
 * between consecutive linears on this path. */
snip_status snip_qlinear_bwd_chain(const snip_plan* plan, int layer, int prev_layer, const void* X, const void* W,
                                   const void* dY, int64_t T, int64_t K, int64_t N, float* dX, float* dW,
                                   double* stats_out, const float* g_prev, uint8_t* prev_codes,
                                   uint8_t* prev_scales, uint8_t* prev_codes_t, uint8_t* prev_scales_t,
                                   float* amax_prev, void* ws, size_t ws_bytes, void* stream);

/* The backward of an NVFP4 layer whose gradient arrives already quantized
 * (snip_qlinear_bwd_chain's outputs): dX = Q(dY) Q(W^T)^T and
 * dW = Q(dY^T) Q(X^T)^T with Q(dY), Q(dY^T) given (dy_* and dyt_*, NVFP4,
 * MMA layout, tensor scale g_dy: device float) and W^T, X^T quantized as in
 * snip_qlinear_bwd.  The bf16 dY is never formed here, so this form has no
 * statistics of it.  The layer's format must be NVFP4; other arguments and
 * errors as snip_qlinear_bwd. */
snip_status snip_qlinear_bwd_q(const snip_plan* plan, int layer, const void* X, const void* W,
                               const uint8_t* dy_codes, const uint8_t* dy_scales, const uint8_t* dyt_codes,
                               const uint8_t* dyt_scales, const float* g_dy, int64_t T, int64_t K, int64_t N,
                               float* dX, float* dW, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------- a8: statistics */

/* SNIP's statistics pass over one bf16 rows x cols tensor (cols % 16 == 0),
 * blocks along cols, under the tensor's rounding rnd (seed, stream_id for SR):
 * raw_out (device, SNIP_STATS_NVALS doubles) receives the SNIP_ST_* sums;
 * block_err_nvfp4 / block_err_fp8 (device, rows x cols/16 floats, nullable)
 * receive per-block squared errors.  scales_in (device, nullable) holds the
 * tensor's {amax, g, s} from snip_tensor_scales; NULL computes them first.
 * Non-finite input raises SNIP_ERR_NONFINITE in the workspace status. */
snip_status snip_quant_stats(const void* a, int64_t rows, int64_t cols, snip_round rnd, uint64_t seed,
                             uint64_t stream_id, const float* scales_in, double* raw_out, float* block_err_nvfp4,
                             float* block_err_fp8, void* ws, size_t ws_bytes, void* stream);

/* One pass that both quantizes x with blocks along cols (as snip_quantize_*
 * with the given layout, rounding and stream) and computes SNIP's statistics
 * of x under that same rounding and random bits (as snip_quant_stats): the
 * tensor is read once.  fmt selects the codes written
 * (scales: the FP4 formats);
 * scales_in (device, nullable) = {amax, g, s} from snip_tensor_scales (NULL:
 * computed first); raw_out device SNIP_STATS_NVALS doubles.  Errors as for
 * snip_quantize_nvfp4 / snip_quant_stats. */
snip_status snip_quantize_stats(snip_format fmt, const void* x, int64_t rows, int64_t cols, snip_round rnd,
                                uint64_t seed, uint64_t stream_id, const float* scales_in, snip_layout layout,
                                uint8_t* codes, uint8_t* scales, double* raw_out, void* ws, size_t ws_bytes,
                                void* stream);

/* Host helper: derive ratios and sqrt(3) flags from a host copy of raw_out. */
snip_status snip_stats_finalize(const double* raw_host, snip_stats* out);

/* ---------------------------------------------------------------- NEXT-4: dW-level sqrt(3) check */

/* The weight-gradient form of the quantization-noise threshold of "FP4 all
 * the way" (Outline: quantized training loses efficiency once the gradient
 * norm falls below about sqrt(3) times the quantization noise): the
 * full-precision weight gradient dW = dY^T X of the bf16 tensors is compared
 * with a quantized one:
 * out2 (device, 2 doubles) = { ||dW||^2, ||dW_q - dW||^2 }.
 * One kernel: a bf16 tensor-core GEMM (fp32 accumulation in tensor memory)
 * whose epilogue reads dW_q beside each tile of dW and accumulates both
 * sums; dW is never written to memory.
 * X device T x K bf16, dY device T x N bf16, dW_q device N x K fp32 (dense,
 * e.g. snip_qlinear_bwd's dW).  T, K, N multiples of 16 and below 2^31
 * (SNIP_ERR_SHAPE).  ws: snip_dw_noise_workspace_size(K, N) bytes (partial
 * sums and the status word only).  Errors as for the other entry points. */
size_t snip_dw_noise_workspace_size(int64_t K, int64_t N);
snip_status snip_dw_noise(const void* X, const void* dY, int64_t T, int64_t K, int64_t N, const float* dW_q,
                          double* out2, void* ws, size_t ws_bytes, void* stream);
/* Host helper: ratio = sqrt(||dW||^2 / ||dW_q - dW||^2) (infinite for a zero
 * error) and below_sqrt3 = ratio < sqrt(3), from a host copy of out2.
 * SNIP_ERR_NONFINITE for a non-finite input sum. */
snip_status snip_dw_noise_finalize(const double* out2_host, double* ratio, int* below_sqrt3);

/* ---------------------------------------------------------------- plan selection (host) */

/* Per-layer cost of each format for SNIP's plan selection ("SNIP" (Pan et
 * al.), Abstract and Figure 2: statistics collected during training feed an
 * ILP over layer-wise precision).  The pages do not print the forward loss
 * divergence or backward weight divergence, so the cost of format f for a
 * layer is a proxy from the statistics pass: the relative squared
 * quantization error of its three operand tensors under their own rounding,
 * cost_f = sum over X, W, dY of ||Q_f(A) - A||^2 / ||A||^2 (a tensor with
 * ||A|| = 0 adds 0).
 * raw_host (host): n_layers x 3 x SNIP_STATS_NVALS doubles, the raw statistics
 * of X, W and dY of each layer in that order (as written by snip_qlinear_fwd's
 * and snip_qlinear_bwd's stats_out or by snip_quant_stats).
 * cost_fp8 / cost_nvfp4 (host, n_layers doubles) receive the costs.
 * Errors: SNIP_ERR_INVALID_ARG (null pointers, n_layers < 0),
 * SNIP_ERR_NONFINITE (a non-finite statistic).  No device work. */
snip_status snip_plan_costs(int n_layers, const double* raw_host, double* cost_fp8, double* cost_nvfp4);

/* SNIP's layer-wise format choice: among all FP8/NVFP4 assignments whose FP4
 * share of the GEMM FLOPs is at least fp4_fraction, the one with the least
 * total cost (sum of cost_nvfp4 over FP4 layers and cost_fp8 over the rest) --
 * the knapsack-like ILP of "SNIP" (Abstract; Figure 3 for the efficiency
 * measure), solved exactly by dynamic programming over the FP4 FLOPs in units
 * of their greatest common divisor.
 * flops (host, n_layers doubles): each layer's fwd+bwd GEMM FLOPs (6 T K N),
 * integral and <= 2^53.  The FP4 FLOPs required are ceil(fp4_fraction * U -
 * 1e-9) units of U in total (fp4_fraction in [0, 1]).  Ties go to FP8 for a
 * layer and to the smaller FP4 share for the set.
 * fmt_out (host, n_layers ints) receives snip_format values; fp4_fraction_out
 * and cost_out (host, nullable) the achieved FP4 FLOP share and total cost.
 * Errors: SNIP_ERR_INVALID_ARG (null pointers, a fraction outside [0, 1],
 * non-integral, negative or too large FLOPs, non-finite costs),
 * SNIP_ERR_SHAPE (the table n_layers x (U + 1) exceeds 2^28 cells).  The
 * pages' extension of the ILP to pipeline-parallel stages is not built. */
snip_status snip_plan_select(int n_layers, const double* flops, const double* cost_fp8, const double* cost_nvfp4,
                             double fp4_fraction, int* fmt_out, double* fp4_fraction_out, double* cost_out);

#ifdef __cplusplus
}
#endif

#endif /* SNIP_H */
