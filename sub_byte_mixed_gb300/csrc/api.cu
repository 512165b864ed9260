// api.cu -- the C ABI declared in include/snip.h: argument checks, workspace
// layout, the per-layer precision plan and the launch sequence of each call.
// Every compute step runs in the kernels of quant.cu, gemm.cu and dw_noise.cu
// (plan selection over the statistics is host code, plan_select.cu).
#include <cmath>
#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

#include "../../include/snip.h"
#include "snip_kernels.cuh"

using namespace snip;

namespace {

// ---------------------------------------------------------------- workspace header
// Byte offsets inside the SNIP_WS_HEADER_BYTES header and the small-scratch
// region that follows it.
constexpr size_t kOffStatus = 0;        // uint32 sticky status bits
constexpr size_t kOffAmaxCounter = 4;   // uint32, self-resetting
constexpr size_t kOffStatsCounter = 8;  // uint32, self-resetting
constexpr size_t kOffMultiCounters = 16; // kMaxMultiScales (8) x uint32, self-resetting
constexpr size_t kOffScaleSlots = 64;   // 8 slots x 4 floats {amax, NVFP4 g, FP8 s, -} (12 bytes used)
static_assert(kOffMultiCounters + 4 * kMaxMultiScales <= kOffScaleSlots, "multi-scale counters overlap the scale slots");
constexpr size_t kOffAmaxPartials = SNIP_WS_HEADER_BYTES;                            // kMaxPartials x uint32
constexpr size_t kOffStatsPartials = kOffAmaxPartials + 4 * kMaxPartials;            // kMaxPartials x 5 doubles
constexpr size_t kSmallWorkspace = kOffStatsPartials + 8 * 5 * kMaxPartials;         // 90368
constexpr size_t kSmallWorkspaceRounded = (kSmallWorkspace + 4095) / 4096 * 4096;   // 94208

constexpr uint64_t kTimeoutNs = 4000000000ull;   // a GEMM wait that takes 4 s is a fault

inline int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// Largest sizes the kernels index with 32-bit tile and segment counts and TMA coordinates: each dimension
// below 2^31, at most 2^40 elements a tensor (far beyond the device's memory).
inline bool too_large(int64_t rows, int64_t cols) {
  return rows > INT32_MAX || cols > INT32_MAX || rows * cols > ((int64_t)1 << 40);
}

template <typename T>
inline T* ws_at(void* ws, size_t off) { return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off); }

// Per-device facts, cached for device ordinals < 64.
struct DeviceInfo { int checked = 0; int ok = 0; int num_sms = 0; };
DeviceInfo g_dev[64];

snip_status current_device(int* num_sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SNIP_ERR_CUDA;
  if (dev < 0 || dev >= 64) return SNIP_ERR_UNSUPPORTED_DEVICE;
  DeviceInfo& d = g_dev[dev];
  if (!d.checked) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return SNIP_ERR_CUDA;
    d.ok = (major == 10 && minor == 3);
    d.num_sms = sms;
    d.checked = 1;
  }
  if (!d.ok) return SNIP_ERR_UNSUPPORTED_DEVICE;
  if (num_sms) *num_sms = d.num_sms;
  return SNIP_OK;
}

inline snip_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return SNIP_OK;
  fprintf(stderr, "snip: CUDA error %s\n", cudaGetErrorString(e));
  return SNIP_ERR_CUDA;
}

// Padded dims of the MMA operand layout.
inline int64_t mma_rows(int64_t r) { return round_up(r, 256); }
// NVFP4 and its longer-block variants (same layouts and GEMM; one scale per
// 16, 32, 64 or 128 elements)
inline bool is_nvfp4(int snip_fmt) {
  return snip_fmt == SNIP_FMT_NVFP4 || snip_fmt == SNIP_FMT_NVFP4_B32 || snip_fmt == SNIP_FMT_NVFP4_B64 ||
         snip_fmt == SNIP_FMT_NVFP4_B128;
}
inline bool is_fp4(int snip_fmt) { return is_nvfp4(snip_fmt) || snip_fmt == SNIP_FMT_MXFP4; }
// 16-element blocks sharing one scale
inline int nvfp4_group(int snip_fmt) {
  return snip_fmt == SNIP_FMT_NVFP4_B32 ? 2 : snip_fmt == SNIP_FMT_NVFP4_B64 ? 4 : snip_fmt == SNIP_FMT_NVFP4_B128 ? 8 : 1;
}
// operand formats (quantizer outputs, GEMM inputs); FP8_E5M2_GRAD is a layer format only
inline bool valid_operand_fmt(int f) { return f >= 0 && f <= 7 && f != SNIP_FMT_FP8_E5M2_GRAD; }
inline int64_t mma_cols(int snip_fmt, int64_t c) { return round_up(c, is_fp4(snip_fmt) ? 256 : 128); }
// quantizer kernel format ids: 0 FP8 E4M3, 1 NVFP4, 2 MXFP4, 3 FP8 E5M2
inline int kernel_fmt(int snip_fmt) {
  return is_nvfp4(snip_fmt) ? 1 : snip_fmt == SNIP_FMT_MXFP4 ? 2 : snip_fmt == SNIP_FMT_FP8_E5M2 ? 3 : 0;
}
// GEMM kernel format ids: 0 FP8 (A E4M3 or E5M2), 1 NVFP4, 2 MXFP4
inline int gemm_kernel_fmt(int snip_fmt) {
  return is_nvfp4(snip_fmt) ? 1 : snip_fmt == SNIP_FMT_MXFP4 ? 2 : 0;
}
// Which float of a tensor-scale slot {amax, g, s, s5} a quantization reads:
// NVFP4 g (MXFP4 only checks it for NaN), FP8 s, E5M2 the amax (the kernel
// derives s5 = amax / 57344 and writes it as g_out).
inline int scale_index(int snip_fmt) {
  return snip_fmt == SNIP_FMT_FP8_E4M3 ? 2 : snip_fmt == SNIP_FMT_FP8_E5M2 ? 0 : 1;
}
// ... and which one the GEMM epilogue multiplies by (null: none).
inline const float* gemm_scale(const float* slot, int snip_fmt) {
  return snip_fmt == SNIP_FMT_FP8_E4M3 ? slot + 2 : snip_fmt == SNIP_FMT_FP8_E5M2 ? slot + 3
         : snip_fmt == SNIP_FMT_MXFP4 ? nullptr : slot + 1;
}
// Operand formats of a layer format: a layer with E5M2 gradients quantizes
// dY and dY^T in E5M2 and everything else in E4M3.
inline int forward_fmt(int layer_fmt) { return layer_fmt == SNIP_FMT_FP8_E5M2_GRAD ? SNIP_FMT_FP8_E4M3 : layer_fmt; }
inline int gradient_fmt(int layer_fmt) { return layer_fmt == SNIP_FMT_FP8_E5M2_GRAD ? SNIP_FMT_FP8_E5M2 : layer_fmt; }
// elements per block along the blocked dim, and per stored scale byte
inline int64_t block_elems(int snip_fmt) { return snip_fmt == SNIP_FMT_MXFP4 ? 32 : 16 * nvfp4_group(snip_fmt); }
inline int64_t scale_elems(int snip_fmt) { return snip_fmt == SNIP_FMT_MXFP4 ? 32 : 16; }

struct OperandBytes { size_t codes, scales; };
OperandBytes operand_bytes(int fmt, int layout, int64_t orows, int64_t ocols) {
  int64_t r = orows, c = ocols;
  if (layout != SNIP_LAYOUT_ROWMAJOR) {
    r = mma_rows(orows);
    c = mma_cols(fmt, ocols);
  }
  if (is_fp4(fmt)) return {(size_t)(r * c / 2), (size_t)(r * c / scale_elems(fmt))};
  return {(size_t)(r * c), 0};
}

// ---------------------------------------------------------------- shared launch helpers
float* scale_slot(void* ws, int slot) { return ws_at<float>(ws, kOffScaleSlots + 16 * slot); }

// amax of a bf16 tensor and the two tensor scales derived from it -> out3
snip_status run_scales(const void* x, int64_t n, float* out3, void* ws, int num_sms, cudaStream_t st) {
  return cuda_status(launch_scales(static_cast<const uint16_t*>(x), n, ws_at<uint32_t>(ws, kOffAmaxPartials),
                                   ws_at<uint32_t>(ws, kOffAmaxCounter), out3, ws_at<uint32_t>(ws, kOffStatus),
                                   num_sms, st));
}

// Scales of `count` tensors in one launch (count <= kMaxMultiScales).
snip_status run_scales_multi(int count, const void* const* xs, const int64_t* ns, float* const* outs, void* ws,
                             int num_sms, cudaStream_t st) {
  ScalesMulti m = {};
  m.count = count;
  for (int t = 0; t < count; ++t) {
    m.x[t] = static_cast<const uint16_t*>(xs[t]);
    m.n[t] = ns[t];
    m.out3[t] = outs[t];
  }
  return cuda_status(launch_scales_multi(m, ws_at<uint32_t>(ws, kOffAmaxPartials), ws_at<uint32_t>(ws, kOffMultiCounters),
                                         ws_at<uint32_t>(ws, kOffStatus), num_sms, st));
}

// One quantization with the tensor scale `scale` (device float).
snip_status run_quantize(int fmt, const void* x, int64_t rows, int64_t cols, int orient, int rnd, uint64_t seed,
                         uint64_t stream_id, const float* scale, int layout, uint8_t* codes, uint8_t* scales,
                         float* g_out, float* block_err, int num_sms, cudaStream_t st, const float* scales3 = nullptr,
                         double* raw_out = nullptr, void* ws = nullptr, uint64_t index_base = 0) {
  QuantParams p = {};
  p.index_base = index_base;
  p.x = static_cast<const uint16_t*>(x);
  p.rows = rows;
  p.cols = cols;
  p.out_rows = orient == SNIP_BLOCKS_ALONG_COLS ? rows : cols;
  p.out_cols = orient == SNIP_BLOCKS_ALONG_COLS ? cols : rows;
  p.orp = layout == SNIP_LAYOUT_MMA ? mma_rows(p.out_rows) : p.out_rows;
  p.ocp = layout == SNIP_LAYOUT_MMA ? mma_cols(fmt, p.out_cols) : p.out_cols;
  p.seed = seed;
  p.stream_id = stream_id;
  p.rk = philox_round_keys(seed);
  p.scale = scale;
  p.codes = codes;
  p.scales = scales;
  p.g_out = g_out;
  p.block_err = block_err;
  p.group = nvfp4_group(fmt);
  if (raw_out) {   // statistics fused into this (row-block) quantization
    p.scales3 = scales3;
    p.partials = ws_at<double>(ws, kOffStatsPartials);
    p.counter = ws_at<uint32_t>(ws, kOffStatsCounter);
    p.raw_out = raw_out;
  }
  // an empty output still publishes its tensor scale: the one-CTA row kernel does that
  if (p.orp == 0 || p.ocp == 0) orient = SNIP_BLOCKS_ALONG_COLS;
  return cuda_status(launch_quant(kernel_fmt(fmt), p, orient, layout, rnd, block_err != nullptr, num_sms, st));
}

// Standalone quantization: tensor scales (unless given) then the quantizer.
snip_status run_quantize_api(int fmt, const void* x, int64_t rows, int64_t cols, int orient, int rnd, uint64_t seed,
                             uint64_t stream_id, const float* g_in, int layout, uint8_t* codes, uint8_t* scales,
                             float* g_out, float* block_err, void* ws, int num_sms, cudaStream_t st) {
  const float* scale = g_in;
  if (!scale) {
    float* slot = scale_slot(ws, 0);
    snip_status s = run_scales(x, rows * cols, slot, ws, num_sms, st);
    if (s != SNIP_OK) return s;
    scale = slot + scale_index(fmt);
  }
  return run_quantize(fmt, x, rows, cols, orient, rnd, seed, stream_id, scale, layout, codes, scales, g_out,
                      block_err, num_sms, st);
}

snip_status run_gemm(int fmt, const uint8_t* a_codes, const uint8_t* a_scales, const float* ga, const uint8_t* b_codes,
                     const uint8_t* b_scales, const float* gb, int64_t M, int64_t N, int64_t K, float* D, int64_t ldd,
                     void* ws, int num_sms, cudaStream_t st, const snip_requant* rq = nullptr) {
  GemmParams p;
  memset(&p, 0, sizeof p);
  p.a_scales = a_scales;
  p.b_scales = b_scales;
  p.ga = ga;
  p.gb = gb;
  p.D = D;
  p.M = M;
  p.N = N;
  p.ldd = ldd;
  p.kp = mma_cols(fmt, K);
  p.status = ws_at<uint32_t>(ws, kOffStatus);
  p.timeout_ns = kTimeoutNs;
  if (fmt == SNIP_FMT_MXFP4) p.ga = p.gb = nullptr;   // no tensor scales
  p.a_e5m2 = fmt == SNIP_FMT_FP8_E5M2;
  if (rq) {
    const int64_t orp = mma_rows(M), ocp = round_up(N, 256);
    p.rq_codes = rq->codes;
    p.rq_scales = rq->scales;
    p.rq_g = rq->g_in;
    p.rq_amax = reinterpret_cast<uint32_t*>(rq->amax_out);
    p.rq_ocp = ocp;
    p.rq_seed = rq->seed;
    p.rq_stream = rq->stream_id;
    p.rq_rnd = rq->rnd;
    // column blocks: the N x M transpose, rows padded to 256, contraction M to 256
    const int64_t orp_t = mma_rows(N), ocp_t = round_up(M, 256);
    p.rq_codes_t = rq->codes_t;
    p.rq_scales_t = rq->scales_t;
    p.rq_ocp_t = ocp_t;
    p.rq_stream_t = rq->stream_id_t;
    p.rq_rnd_t = rq->rnd_t;
    // the tiles write every padded row and column they cover; one-CTA tiles (128 rows) may
    // leave the last 128 rows of the 256-row padding of M, so those codes and all scales start at zero
    const int64_t covered = round_up(M, 128);
    cudaError_t e = cudaSuccess;
    if (rq->codes) {
      if (covered < orp)
        e = cudaMemsetAsync(rq->codes + covered * (ocp / 2), 0, (size_t)((orp - covered) * (ocp / 2)), st);
      if (e == cudaSuccess) e = cudaMemsetAsync(rq->scales, 0, (size_t)(orp * ocp / 16), st);
    }
    if (rq->codes_t) {   // there the uncovered rows of D are the last contraction columns of every row
      if (e == cudaSuccess && covered < ocp_t)
        e = cudaMemset2DAsync(rq->codes_t + covered / 2, (size_t)(ocp_t / 2), 0, (size_t)((ocp_t - covered) / 2),
                              (size_t)orp_t, st);
      if (e == cudaSuccess) e = cudaMemsetAsync(rq->scales_t, 0, (size_t)(orp_t * ocp_t / 16), st);
    }
    if (e == cudaSuccess && rq->amax_out) e = cudaMemsetAsync(rq->amax_out, 0, sizeof(float), st);
    if (e != cudaSuccess) return cuda_status(e);
  }
  return cuda_status(launch_gemm(gemm_kernel_fmt(fmt), a_codes, mma_rows(M), b_codes, mma_rows(N), p, num_sms, st));
}

bool valid_enum(int v, int n) { return v >= 0 && v < n; }

}  // namespace

// ---------------------------------------------------------------- plan object
struct snip_plan {
  std::vector<int> fmt;
  std::vector<int> rnd;   // 6 per layer, indexed by snip_tag
  uint64_t seed;
};

extern "C" {

const char* snip_status_string(snip_status s) {
  switch (s) {
    case SNIP_OK: return "ok";
    case SNIP_ERR_INVALID_ARG: return "invalid argument";
    case SNIP_ERR_SHAPE: return "shape not supported (dims must be multiples of 16; 32 along MXFP4 blocks)";
    case SNIP_ERR_ALIGN: return "device pointer not 16-byte aligned";
    case SNIP_ERR_NONFINITE: return "input holds a non-finite value";
    case SNIP_ERR_TIMEOUT: return "a kernel wait timed out";
    case SNIP_ERR_CUDA: return "CUDA runtime error";
    case SNIP_ERR_UNSUPPORTED_DEVICE: return "device is not compute capability 10.3 (sm_103)";
    case SNIP_ERR_WORKSPACE: return "workspace missing or too small";
  }
  return "unknown status";
}

int snip_version(void) { return SNIP_ABI_VERSION; }

snip_status snip_device_check(void) { return current_device(nullptr); }

snip_status snip_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  if (!ws || ws_bytes < SNIP_WS_HEADER_BYTES) return SNIP_ERR_WORKSPACE;
  return cuda_status(cudaMemsetAsync(ws, 0, SNIP_WS_HEADER_BYTES, static_cast<cudaStream_t>(stream)));
}

snip_status snip_workspace_status(const void* ws, void* stream, snip_status* device_status) {
  if (!ws || !device_status) return SNIP_ERR_INVALID_ARG;
  uint32_t word = 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(&word, ws, sizeof word, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_status(e);
  *device_status = (word & kDevNonFinite) ? SNIP_ERR_NONFINITE : (word & kDevTimeout) ? SNIP_ERR_TIMEOUT : SNIP_OK;
  return SNIP_OK;
}

size_t snip_quantize_workspace_size(int64_t rows, int64_t cols) {
  (void)rows;
  (void)cols;
  return kSmallWorkspaceRounded;
}

snip_status snip_amax(const void* x, int64_t n, float* amax_out, void* ws, size_t ws_bytes, void* stream) {
  int sms;
  snip_status s = current_device(&sms);
  if (s != SNIP_OK) return s;
  if ((!x && n > 0) || !amax_out || n < 0) return SNIP_ERR_INVALID_ARG;
  if (!ws || ws_bytes < kSmallWorkspace) return SNIP_ERR_WORKSPACE;
  if (!aligned16(x) || !aligned16(ws)) return SNIP_ERR_ALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  float* slot = scale_slot(ws, 0);
  if ((s = run_scales(x, n, slot, ws, sms, st)) != SNIP_OK) return s;
  return cuda_status(cudaMemcpyAsync(amax_out, slot, sizeof(float), cudaMemcpyDeviceToDevice, st));
}

snip_status snip_tensor_scales(const void* x, int64_t n, float* scales_out, void* ws, size_t ws_bytes, void* stream) {
  int sms;
  snip_status s = current_device(&sms);
  if (s != SNIP_OK) return s;
  if ((!x && n > 0) || !scales_out || n < 0) return SNIP_ERR_INVALID_ARG;
  if (!ws || ws_bytes < kSmallWorkspace) return SNIP_ERR_WORKSPACE;
  if (!aligned16(x) || !aligned16(ws)) return SNIP_ERR_ALIGN;
  return run_scales(x, n, scales_out, ws, sms, static_cast<cudaStream_t>(stream));
}

snip_status snip_tensor_scales_multi(int count, const void* const* xs, const int64_t* ns, float* const* scales_out,
                                     void* ws, size_t ws_bytes, void* stream) {
  int sms;
  snip_status s = current_device(&sms);
  if (s != SNIP_OK) return s;
  if (count < 1 || count > kMaxMultiScales || !xs || !ns || !scales_out) return SNIP_ERR_INVALID_ARG;
  for (int t = 0; t < count; ++t) {
    if (ns[t] < 0 || (!xs[t] && ns[t] > 0) || !scales_out[t]) return SNIP_ERR_INVALID_ARG;
    if (!aligned16(xs[t])) return SNIP_ERR_ALIGN;
  }
  if (!ws || ws_bytes < kSmallWorkspace) return SNIP_ERR_WORKSPACE;
  if (!aligned16(ws)) return SNIP_ERR_ALIGN;
  return run_scales_multi(count, xs, ns, scales_out, ws, sms, static_cast<cudaStream_t>(stream));
}

snip_status snip_wait_check(uint64_t limit_ns, uint32_t* out, void* ws, size_t ws_bytes, void* stream) {
  int sms;
  snip_status s = current_device(&sms);
  if (s != SNIP_OK) return s;
  if (!out) return SNIP_ERR_INVALID_ARG;
  if (!ws || ws_bytes < SNIP_WS_HEADER_BYTES) return SNIP_ERR_WORKSPACE;
  if (!aligned16(ws)) return SNIP_ERR_ALIGN;
  const uint64_t lim = limit_ns < 1000u ? 1000u : limit_ns > 1000000000u ? 1000000000u : limit_ns;
  return cuda_status(launch_wait_check(ws_at<uint32_t>(ws, kOffStatus), lim, out, static_cast<cudaStream_t>(stream)));
}

snip_status snip_quantized_bytes(snip_format fmt, snip_layout layout, int64_t out_rows, int64_t out_cols,
                                 size_t* codes_bytes, size_t* scales_bytes) {
  if (!valid_operand_fmt(fmt) || !valid_enum(layout, 2) || out_rows < 0 || out_cols < 0) return SNIP_ERR_INVALID_ARG;
  OperandBytes b = operand_bytes(fmt, layout, out_rows, out_cols);
  if (codes_bytes) *codes_bytes = b.codes;
  if (scales_bytes) *scales_bytes = b.scales;
  return SNIP_OK;
}

static snip_status check_quantize_args(int fmt, const void* x, int64_t rows, int64_t cols, int orient, int rnd,
                                       int layout, const void* codes, const void* scales, const void* g_out,
                                       const void* ws, size_t ws_bytes) {
  if (!valid_enum(orient, 2) || !valid_enum(rnd, 2) || !valid_enum(layout, 2)) return SNIP_ERR_INVALID_ARG;
  if (rows < 0 || cols < 0 || !g_out || !codes || (rows * cols > 0 && !x)) return SNIP_ERR_INVALID_ARG;
  if (is_fp4(fmt) && !scales) return SNIP_ERR_INVALID_ARG;
  const int64_t be = block_elems(fmt);   // the blocked dim is a whole number of blocks
  if (cols % 16 != 0 || (orient == SNIP_BLOCKS_ALONG_ROWS && rows % be != 0) ||
      (orient == SNIP_BLOCKS_ALONG_COLS && cols % be != 0) || too_large(rows, cols))
    return SNIP_ERR_SHAPE;
  if (!ws || ws_bytes < kSmallWorkspace) return SNIP_ERR_WORKSPACE;
  if (!aligned16(x) || !aligned16(codes) || !aligned16(ws) || (scales && !aligned16(scales))) return SNIP_ERR_ALIGN;
  return SNIP_OK;
}

snip_status snip_quantize_nvfp4(const void* x, int64_t rows, int64_t cols, snip_orient orient, snip_round rnd,
                                uint64_t seed, uint64_t stream_id, const float* g_in, snip_layout layout,
                                uint8_t* codes, uint8_t* scales, float* g_out, float* block_sqerr, void* ws,
                                size_t ws_bytes, void* stream) {
  int sms;
  snip_status s = current_device(&sms);
  if (s != SNIP_OK) return s;
  s = check_quantize_args(SNIP_FMT_NVFP4, x, rows, cols, orient, rnd, layout, codes, scales, g_out, ws, ws_bytes);
  if (s != SNIP_OK) return s;
  return run_quantize_api(SNIP_FMT_NVFP4, x, rows, cols, orient, rnd, seed, stream_id, g_in, layout, codes, scales,
                          g_out, block_sqerr, ws, sms, static_cast<cudaStream_t>(stream));
}

snip_status snip_quantize_nvfp4_block(const void* x, int64_t rows, int64_t cols, snip_orient orient, snip_round rnd,
                                      uint64_t seed, uint64_t stream_id, const float* g_in, int block,
                                      snip_layout layout, uint8_t* codes, uint8_t* scales, float* g_out, void* ws,
                                      size_t ws_bytes, void* stream) {
  int sms;
  snip_status s = current_device(&sms);
  if (s != SNIP_OK) return s;
  const int fmt = block == 16 ? SNIP_FMT_NVFP4 : block == 32 ? SNIP_FMT_NVFP4_B32 : block == 64 ? SNIP_FMT_NVFP4_B64
                  : block == 128 ? SNIP_FMT_NVFP4_B128 : -1;
  if (fmt < 0) return SNIP_ERR_INVALID_ARG;
  s = check_quantize_args(fmt, x, rows, cols, orient, rnd, layout, codes, scales, g_out, ws, ws_bytes);
  if (s != SNIP_OK) return s;
  return run_quantize_api(fmt, x, rows, cols, orient, rnd, seed, stream_id, g_in, layout, codes, scales, g_out,
                          nullptr, ws, sms, static_cast<cudaStream_t>(stream));
}

snip_status snip_quantize_fp8(const void* x, int64_t rows, int64_t cols, snip_orient orient, snip_round rnd,
                              uint64_t seed, uint64_t stream_id, const float* s_in, snip_layout layout,
                              uint8_t* codes, float* s_out, void* ws, size_t ws_bytes, void* stream) {
  int sms;
  snip_status s = current_device(&sms);
  if (s != SNIP_OK) return s;
  s = check_quantize_args(SNIP_FMT_FP8_E4M3, x, rows, cols, orient, rnd, layout, codes, nullptr, s_out, ws,
                          ws_bytes);
  if (s != SNIP_OK) return s;
  return run_quantize_api(SNIP_FMT_FP8_E4M3, x, rows, cols, orient, rnd, seed, stream_id, s_in, layout, codes,
                          nullptr, s_out, nullptr, ws, sms, static_cast<cudaStream_t>(stream));
}

snip_status snip_quantize_mxfp4(const void* x, int64_t rows, int64_t cols, snip_orient orient, snip_round rnd,
                                uint64_t seed, uint64_t stream_id, snip_layout layout, uint8_t* codes, uint8_t* scales,
                                void* ws, size_t ws_bytes, void* stream) {
  int sms;
  snip_status s = current_device(&sms);
  if (s != SNIP_OK) return s;
  float g_dummy;   // validation only: MXFP4 has no tensor scale to return
  s = check_quantize_args(SNIP_FMT_MXFP4, x, rows, cols, orient, rnd, layout, codes, scales, &g_dummy, ws, ws_bytes);
  if (s != SNIP_OK) return s;
  return run_quantize_api(SNIP_FMT_MXFP4, x, rows, cols, orient, rnd, seed, stream_id, nullptr, layout, codes, scales,
                          nullptr, nullptr, ws, sms, static_cast<cudaStream_t>(stream));
}

snip_status snip_quantize_e5m2(const void* x, int64_t rows, int64_t cols, snip_orient orient, snip_round rnd,
                               uint64_t seed, uint64_t stream_id, const float* amax_in, snip_layout layout,
                               uint8_t* codes, float* s_out, void* ws, size_t ws_bytes, void* stream) {
  int sms;
  snip_status s = current_device(&sms);
  if (s != SNIP_OK) return s;
  s = check_quantize_args(SNIP_FMT_FP8_E5M2, x, rows, cols, orient, rnd, layout, codes, nullptr, s_out, ws, ws_bytes);
  if (s != SNIP_OK) return s;
  return run_quantize_api(SNIP_FMT_FP8_E5M2, x, rows, cols, orient, rnd, seed, stream_id, amax_in, layout, codes,
                          nullptr, s_out, nullptr, ws, sms, static_cast<cudaStream_t>(stream));
}

snip_status snip_gemm(snip_format fmt, const uint8_t* a_codes, const uint8_t* a_scales, const float* ga,
                      const uint8_t* b_codes, const uint8_t* b_scales, const float* gb, int64_t M, int64_t N,
                      int64_t K, float* D, int64_t ldd, void* ws, size_t ws_bytes, void* stream) {
  int sms;
  snip_status s = current_device(&sms);
  if (s != SNIP_OK) return s;
  if (!valid_operand_fmt(fmt) || M < 0 || N < 0 || K < 0 || ldd < N) return SNIP_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return SNIP_OK;
  if (!a_codes || !b_codes || !D) return SNIP_ERR_INVALID_ARG;
  if (fmt != SNIP_FMT_MXFP4 && (!ga || !gb)) return SNIP_ERR_INVALID_ARG;
  if (is_fp4(fmt) && (!a_scales || !b_scales)) return SNIP_ERR_INVALID_ARG;
  if (fmt == SNIP_FMT_MXFP4 && K % 32 != 0) return SNIP_ERR_SHAPE;
  if (K % 16 != 0 || K == 0 || ldd % 4 != 0 || too_large(M, N) || too_large(M, K) || too_large(N, K))
    return SNIP_ERR_SHAPE;
  if (!ws || ws_bytes < SNIP_WS_HEADER_BYTES) return SNIP_ERR_WORKSPACE;
  if (!aligned16(a_codes) || !aligned16(b_codes) || !aligned16(D) || !aligned16(ws) ||
      (is_fp4(fmt) && (!aligned16(a_scales) || !aligned16(b_scales))))
    return SNIP_ERR_ALIGN;
  return run_gemm(fmt, a_codes, a_scales, ga, b_codes, b_scales, gb, M, N, K, D, ldd, ws, sms,
                  static_cast<cudaStream_t>(stream));
}

snip_status snip_gemm_requant(snip_format fmt, const uint8_t* a_codes, const uint8_t* a_scales, const float* ga,
                              const uint8_t* b_codes, const uint8_t* b_scales, const float* gb, int64_t M, int64_t N,
                              int64_t K, float* D, int64_t ldd, const snip_requant* rq, void* ws, size_t ws_bytes,
                              void* stream) {
  int sms;
  snip_status s = current_device(&sms);
  if (s != SNIP_OK) return s;
  if (!rq || !rq->g_in || (!rq->codes && !rq->codes_t) || (rq->codes && !rq->scales) ||
      (rq->codes_t && !rq->scales_t) || !valid_enum(rq->rnd, 2) || !valid_enum(rq->rnd_t, 2))
    return SNIP_ERR_INVALID_ARG;
  if (!valid_operand_fmt(fmt) || M < 0 || N < 0 || K < 0 || (D && ldd < N)) return SNIP_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return SNIP_OK;
  if (!a_codes || !b_codes) return SNIP_ERR_INVALID_ARG;
  if (fmt != SNIP_FMT_MXFP4 && (!ga || !gb)) return SNIP_ERR_INVALID_ARG;
  if (is_fp4(fmt) && (!a_scales || !b_scales)) return SNIP_ERR_INVALID_ARG;
  if (K % 16 != 0 || K == 0 || N % 16 != 0 || (rq->codes_t && M % 16 != 0) || (D && ldd % 4 != 0) ||
      (fmt == SNIP_FMT_MXFP4 && K % 32 != 0) || too_large(M, N) || too_large(M, K) || too_large(N, K))
    return SNIP_ERR_SHAPE;
  if (!ws || ws_bytes < SNIP_WS_HEADER_BYTES) return SNIP_ERR_WORKSPACE;
  if (!aligned16(a_codes) || !aligned16(b_codes) || (D && !aligned16(D)) || !aligned16(ws) ||
      !aligned16(rq->codes) || !aligned16(rq->scales) || !aligned16(rq->codes_t) || !aligned16(rq->scales_t) ||
      (is_fp4(fmt) && (!aligned16(a_scales) || !aligned16(b_scales))))
    return SNIP_ERR_ALIGN;
  return run_gemm(fmt, a_codes, a_scales, ga, b_codes, b_scales, gb, M, N, K, D, D ? ldd : N, ws, sms,
                  static_cast<cudaStream_t>(stream), rq);
}

// ---------------------------------------------------------------- plan
snip_status snip_plan_create(int n_layers, const int* formats, uint64_t seed, snip_plan** out) {
  if (n_layers <= 0 || !formats || !out) return SNIP_ERR_INVALID_ARG;
  for (int i = 0; i < n_layers; ++i)
    if (!valid_enum(formats[i], 8) || formats[i] == SNIP_FMT_FP8_E5M2) return SNIP_ERR_INVALID_ARG;
  snip_plan* p = new (std::nothrow) snip_plan;
  if (!p) return SNIP_ERR_INVALID_ARG;
  p->fmt.assign(formats, formats + n_layers);
  p->rnd.assign((size_t)n_layers * 6, SNIP_SR);
  for (int i = 0; i < n_layers; ++i) {
    p->rnd[(size_t)i * 6 + SNIP_TAG_X_FWD] = SNIP_RTN;
    p->rnd[(size_t)i * 6 + SNIP_TAG_W_FWD] = SNIP_RTN;
  }
  p->seed = seed;
  *out = p;
  return SNIP_OK;
}

snip_status snip_plan_set_rounding(snip_plan* plan, int layer, snip_tag tag, snip_round rnd) {
  if (!plan || layer < 0 || layer >= (int)plan->fmt.size() || !valid_enum(tag, 6) || !valid_enum(rnd, 2))
    return SNIP_ERR_INVALID_ARG;
  plan->rnd[(size_t)layer * 6 + tag] = rnd;
  return SNIP_OK;
}

snip_status snip_plan_get(const snip_plan* plan, int layer, snip_format* fmt, uint64_t* seed) {
  if (!plan || layer < 0 || layer >= (int)plan->fmt.size()) return SNIP_ERR_INVALID_ARG;
  if (fmt) *fmt = (snip_format)plan->fmt[layer];
  if (seed) *seed = plan->seed;
  return SNIP_OK;
}

void snip_plan_destroy(snip_plan* plan) { delete plan; }

// ---------------------------------------------------------------- qlinear
namespace {
struct QlOperand { size_t codes_off, scales_off; };
struct QlLayout {
  QlOperand op[4];
  size_t total;
};

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// fwd: op0 = X (T x K), op1 = W (N x K); bwd: op0 = dY (T x N), op1 = W^T
// (K x N), op2 = dY^T (N x T), op3 = X^T (K x T).  The two calls reuse the
// same region, so the workspace is sized for the larger of the two.
QlLayout ql_layout(int fmt, int64_t T, int64_t K, int64_t N, bool bwd) {
  QlLayout L;
  size_t off = kSmallWorkspaceRounded;
  const int64_t shapes_fwd[2][2] = {{T, K}, {N, K}};
  const int64_t shapes_bwd[4][2] = {{T, N}, {K, N}, {N, T}, {K, T}};
  const int n = bwd ? 4 : 2;
  for (int i = 0; i < n; ++i) {
    const int64_t* sh = bwd ? shapes_bwd[i] : shapes_fwd[i];
    OperandBytes b = operand_bytes(fmt, SNIP_LAYOUT_MMA, sh[0], sh[1]);
    L.op[i].codes_off = off;
    off = align_up(off + b.codes, 1024);
    L.op[i].scales_off = off;
    off = align_up(off + b.scales, 1024);
  }
  L.total = off;
  return L;
}

snip_status check_ql(const snip_plan* plan, int layer, int64_t T, int64_t K, int64_t N) {
  if (!plan || layer < 0 || layer >= (int)plan->fmt.size()) return SNIP_ERR_INVALID_ARG;
  if (T <= 0 || K <= 0 || N <= 0) return SNIP_ERR_INVALID_ARG;
  const int64_t be = block_elems(plan->fmt[layer]);   // every dim is blocked by one of the quantizations
  if (T % be || K % be || N % be || too_large(T, K) || too_large(T, N) || too_large(N, K)) return SNIP_ERR_SHAPE;
  return SNIP_OK;
}
}  // namespace

size_t snip_qlinear_workspace_size(const snip_plan* plan, int layer, int64_t T, int64_t K, int64_t N) {
  if (check_ql(plan, layer, T, K, N) != SNIP_OK) return 0;
  const int fmt = forward_fmt(plan->fmt[layer]);   // E5M2 operands have E4M3's size
  size_t a = ql_layout(fmt, T, K, N, false).total, b = ql_layout(fmt, T, K, N, true).total;
  return a > b ? a : b;
}

snip_status snip_qlinear_fwd(const snip_plan* plan, int layer, const void* X, const void* W, int64_t T, int64_t K,
                             int64_t N, float* Y, double* stats_out, void* ws, size_t ws_bytes, void* stream) {
  int sms;
  snip_status s = current_device(&sms);
  if (s != SNIP_OK) return s;
  if ((s = check_ql(plan, layer, T, K, N)) != SNIP_OK) return s;
  if (!X || !W || !Y) return SNIP_ERR_INVALID_ARG;
  if (!ws || ws_bytes < snip_qlinear_workspace_size(plan, layer, T, K, N)) return SNIP_ERR_WORKSPACE;
  if (!aligned16(X) || !aligned16(W) || !aligned16(Y) || !aligned16(ws)) return SNIP_ERR_ALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int qf = forward_fmt(plan->fmt[layer]);   // format of X and W
  const int* rnd = &plan->rnd[(size_t)layer * 6];
  const uint64_t sid = (uint64_t)layer * 8;
  QlLayout L = ql_layout(qf, T, K, N, false);
  uint8_t* b = static_cast<uint8_t*>(ws);
  float* sx = scale_slot(ws, 0);
  float* sw = scale_slot(ws, 1);
  {
    const void* xs[2] = {X, W};
    const int64_t ns[2] = {T * K, N * K};
    float* outs[2] = {sx, sw};
    if ((s = run_scales_multi(2, xs, ns, outs, ws, sms, st)) != SNIP_OK) return s;
  }
  if ((s = run_quantize(qf, X, T, K, SNIP_BLOCKS_ALONG_COLS, rnd[SNIP_TAG_X_FWD], plan->seed, sid + SNIP_TAG_X_FWD,
                        sx + scale_index(qf), SNIP_LAYOUT_MMA, b + L.op[0].codes_off, b + L.op[0].scales_off, nullptr,
                        nullptr, sms, st, sx, stats_out, ws)) != SNIP_OK)
    return s;
  if ((s = run_quantize(qf, W, N, K, SNIP_BLOCKS_ALONG_COLS, rnd[SNIP_TAG_W_FWD], plan->seed, sid + SNIP_TAG_W_FWD,
                        sw + scale_index(qf), SNIP_LAYOUT_MMA, b + L.op[1].codes_off, b + L.op[1].scales_off, nullptr,
                        nullptr, sms, st, sw, stats_out ? stats_out + SNIP_STATS_NVALS : nullptr, ws)) != SNIP_OK)
    return s;
  return run_gemm(qf, b + L.op[0].codes_off, b + L.op[0].scales_off, gemm_scale(sx, qf), b + L.op[1].codes_off,
                  b + L.op[1].scales_off, gemm_scale(sw, qf), T, N, K, Y, N, ws, sms, st);
}

namespace {
constexpr int kMaxMulti = 8;
// Groups of the layers of a multi-layer forward that share one quantization of X: same forward
// format and round-to-nearest X_FWD rounding; a stochastic X_FWD rounding is the layer's own group.
// group[i] = index of layer i's group; first[g] = its first member; returns the number of groups.
int fwd_groups(const snip_plan* plan, int count, const int* layers, int* group, int* first) {
  int ng = 0;
  for (int i = 0; i < count; ++i) {
    const int l = layers[i], f = forward_fmt(plan->fmt[l]);
    const bool rtn = plan->rnd[(size_t)l * 6 + SNIP_TAG_X_FWD] == SNIP_RTN;
    group[i] = -1;
    for (int g = 0; rtn && g < ng; ++g) {
      const int l0 = layers[first[g]];
      if (forward_fmt(plan->fmt[l0]) == f && plan->rnd[(size_t)l0 * 6 + SNIP_TAG_X_FWD] == SNIP_RTN) group[i] = g;
    }
    if (group[i] < 0) { first[ng] = i; group[i] = ng++; }
  }
  return ng;
}
struct MultiLayout {
  size_t x_codes[kMaxMulti], x_scales[kMaxMulti], w_codes, w_scales, total;
};
MultiLayout multi_layout(const snip_plan* plan, int count, const int* layers, int64_t T, int64_t K, const int64_t* N,
                         const int* first, int ng) {
  MultiLayout L;
  size_t off = kSmallWorkspaceRounded;
  for (int g = 0; g < ng; ++g) {
    OperandBytes b = operand_bytes(forward_fmt(plan->fmt[layers[first[g]]]), SNIP_LAYOUT_MMA, T, K);
    L.x_codes[g] = off;
    off = align_up(off + b.codes, 1024);
    L.x_scales[g] = off;
    off = align_up(off + b.scales, 1024);
  }
  size_t wc = 0, wsz = 0;
  for (int i = 0; i < count; ++i) {
    OperandBytes b = operand_bytes(forward_fmt(plan->fmt[layers[i]]), SNIP_LAYOUT_MMA, N[i], K);
    wc = b.codes > wc ? b.codes : wc;
    wsz = b.scales > wsz ? b.scales : wsz;
  }
  L.w_codes = off;
  off = align_up(off + wc, 1024);
  L.w_scales = off;
  off = align_up(off + wsz, 1024);
  L.total = off;
  return L;
}
snip_status check_multi(const snip_plan* plan, int count, const int* layers, int64_t T, int64_t K, const int64_t* N) {
  if (!plan || count < 1 || count > kMaxMulti || !layers || !N) return SNIP_ERR_INVALID_ARG;
  for (int i = 0; i < count; ++i) {
    for (int j = 0; j < i; ++j)
      if (layers[j] == layers[i]) return SNIP_ERR_INVALID_ARG;
    snip_status s = check_ql(plan, layers[i], T, K, N[i]);
    if (s != SNIP_OK) return s;
  }
  return SNIP_OK;
}
}  // namespace

size_t snip_qlinear_fwd_multi_workspace_size(const snip_plan* plan, int count, const int* layers, int64_t T,
                                             int64_t K, const int64_t* N) {
  if (check_multi(plan, count, layers, T, K, N) != SNIP_OK) return 0;
  int group[kMaxMulti], first[kMaxMulti];
  const int ng = fwd_groups(plan, count, layers, group, first);
  return multi_layout(plan, count, layers, T, K, N, first, ng).total;
}

snip_status snip_qlinear_fwd_multi(const snip_plan* plan, int count, const int* layers, const void* X,
                                   const void* const* W, int64_t T, int64_t K, const int64_t* N, float* const* Y,
                                   double* stats_x, double* const* stats_w, void* ws, size_t ws_bytes,
                                   void* stream) {
  int sms;
  snip_status s = current_device(&sms);
  if (s != SNIP_OK) return s;
  if ((s = check_multi(plan, count, layers, T, K, N)) != SNIP_OK) return s;
  if (!X || !W || !Y) return SNIP_ERR_INVALID_ARG;
  for (int i = 0; i < count; ++i)
    if (!W[i] || !Y[i]) return SNIP_ERR_INVALID_ARG;
  if (!ws || ws_bytes < snip_qlinear_fwd_multi_workspace_size(plan, count, layers, T, K, N))
    return SNIP_ERR_WORKSPACE;
  if (!aligned16(X) || !aligned16(ws)) return SNIP_ERR_ALIGN;
  for (int i = 0; i < count; ++i)
    if (!aligned16(W[i]) || !aligned16(Y[i])) return SNIP_ERR_ALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int group[kMaxMulti], first[kMaxMulti];
  const int ng = fwd_groups(plan, count, layers, group, first);
  const MultiLayout L = multi_layout(plan, count, layers, T, K, N, first, ng);
  uint8_t* b = static_cast<uint8_t*>(ws);
  float* sx = scale_slot(ws, 0);
  float* sw = scale_slot(ws, 1);
  if ((s = run_scales(X, T * K, sx, ws, sms, st)) != SNIP_OK) return s;
  // X once per group; its statistics with the first quantization
  for (int g = 0; g < ng; ++g) {
    const int l = layers[first[g]], qf = forward_fmt(plan->fmt[l]);
    if ((s = run_quantize(qf, X, T, K, SNIP_BLOCKS_ALONG_COLS, plan->rnd[(size_t)l * 6 + SNIP_TAG_X_FWD], plan->seed,
                          (uint64_t)l * 8 + SNIP_TAG_X_FWD, sx + scale_index(qf), SNIP_LAYOUT_MMA, b + L.x_codes[g],
                          b + L.x_scales[g], nullptr, nullptr, sms, st, sx, g == 0 ? stats_x : nullptr, ws)) != SNIP_OK)
      return s;
  }
  // each weight: scales, quantization (+ statistics), GEMM; in stream order, so one W region serves all
  for (int i = 0; i < count; ++i) {
    const int l = layers[i], qf = forward_fmt(plan->fmt[l]), g = group[i];
    if ((s = run_scales(W[i], N[i] * K, sw, ws, sms, st)) != SNIP_OK) return s;
    if ((s = run_quantize(qf, W[i], N[i], K, SNIP_BLOCKS_ALONG_COLS, plan->rnd[(size_t)l * 6 + SNIP_TAG_W_FWD],
                          plan->seed, (uint64_t)l * 8 + SNIP_TAG_W_FWD, sw + scale_index(qf), SNIP_LAYOUT_MMA,
                          b + L.w_codes, b + L.w_scales, nullptr, nullptr, sms, st, sw,
                          stats_w ? stats_w[i] : nullptr, ws)) != SNIP_OK)
      return s;
    if ((s = run_gemm(qf, b + L.x_codes[g], b + L.x_scales[g], gemm_scale(sx, qf), b + L.w_codes, b + L.w_scales,
                      gemm_scale(sw, qf), T, N[i], K, Y[i], N[i], ws, sms, st)) != SNIP_OK)
      return s;
  }
  return SNIP_OK;
}

namespace {
// The backward of one layer (snip_qlinear_bwd); with rq, its dgrad GEMM also writes the preceding
// layer's gradient operands (snip_qlinear_bwd_chain) and dX may be NULL.  Arguments checked by the
// callers.
snip_status run_qlinear_bwd(const snip_plan* plan, int layer, const void* X, const void* W, const void* dY,
                            int64_t T, int64_t K, int64_t N, float* dX, float* dW, double* stats_out, void* ws,
                            int sms, cudaStream_t st, const snip_requant* rq) {
  snip_status s;
  const int qg = gradient_fmt(plan->fmt[layer]);   // format of dY and dY^T (the GEMMs' A operands)
  const int qf = forward_fmt(plan->fmt[layer]);    // format of W^T and X^T
  const int* rnd = &plan->rnd[(size_t)layer * 6];
  const uint64_t sid = (uint64_t)layer * 8;
  QlLayout L = ql_layout(qf, T, K, N, true);
  uint8_t* b = static_cast<uint8_t*>(ws);
  float* sx = scale_slot(ws, 0);
  float* sw = scale_slot(ws, 1);
  float* sd = scale_slot(ws, 2);
  float* sd_out = qg == SNIP_FMT_FP8_E5M2 ? sd + 3 : nullptr;   // E5M2: the quantizer publishes s5 here
  {
    const void* xs[3] = {dY, W, X};
    const int64_t ns[3] = {T * N, N * K, T * K};
    float* outs[3] = {sd, sw, sx};
    if ((s = run_scales_multi(3, xs, ns, outs, ws, sms, st)) != SNIP_OK) return s;
  }
  // dgrad: dX = Q(dY) Q(W^T)^T, contraction N
  if ((s = run_quantize(qg, dY, T, N, SNIP_BLOCKS_ALONG_COLS, rnd[SNIP_TAG_DY_DGRAD], plan->seed,
                        sid + SNIP_TAG_DY_DGRAD, sd + scale_index(qg), SNIP_LAYOUT_MMA, b + L.op[0].codes_off,
                        b + L.op[0].scales_off, sd_out, nullptr, sms, st, sd, stats_out, ws)) != SNIP_OK)
    return s;
  if ((s = run_quantize(qf, W, N, K, SNIP_BLOCKS_ALONG_ROWS, rnd[SNIP_TAG_WT_DGRAD], plan->seed,
                        sid + SNIP_TAG_WT_DGRAD, sw + scale_index(qf), SNIP_LAYOUT_MMA, b + L.op[1].codes_off,
                        b + L.op[1].scales_off, nullptr, nullptr, sms, st)) != SNIP_OK)
    return s;
  if ((s = run_gemm(qg, b + L.op[0].codes_off, b + L.op[0].scales_off, gemm_scale(sd, qg), b + L.op[1].codes_off,
                    b + L.op[1].scales_off, gemm_scale(sw, qf), T, K, N, dX, K, ws, sms, st, rq)) != SNIP_OK)
    return s;
  // wgrad: dW = Q(dY^T) Q(X^T)^T, contraction T
  if ((s = run_quantize(qg, dY, T, N, SNIP_BLOCKS_ALONG_ROWS, rnd[SNIP_TAG_DYT_WGRAD], plan->seed,
                        sid + SNIP_TAG_DYT_WGRAD, sd + scale_index(qg), SNIP_LAYOUT_MMA, b + L.op[2].codes_off,
                        b + L.op[2].scales_off, sd_out, nullptr, sms, st)) != SNIP_OK)
    return s;
  if ((s = run_quantize(qf, X, T, K, SNIP_BLOCKS_ALONG_ROWS, rnd[SNIP_TAG_XT_WGRAD], plan->seed,
                        sid + SNIP_TAG_XT_WGRAD, sx + scale_index(qf), SNIP_LAYOUT_MMA, b + L.op[3].codes_off,
                        b + L.op[3].scales_off, nullptr, nullptr, sms, st)) != SNIP_OK)
    return s;
  return run_gemm(qg, b + L.op[2].codes_off, b + L.op[2].scales_off, gemm_scale(sd, qg), b + L.op[3].codes_off,
                  b + L.op[3].scales_off, gemm_scale(sx, qf), N, K, T, dW, K, ws, sms, st);
}
}  // namespace

snip_status snip_qlinear_bwd(const snip_plan* plan, int layer, const void* X, const void* W, const void* dY,
                             int64_t T, int64_t K, int64_t N, float* dX, float* dW, double* stats_out, void* ws,
                             size_t ws_bytes, void* stream) {
  int sms;
  snip_status s = current_device(&sms);
  if (s != SNIP_OK) return s;
  if ((s = check_ql(plan, layer, T, K, N)) != SNIP_OK) return s;
  if (!X || !W || !dY || !dX || !dW) return SNIP_ERR_INVALID_ARG;
  if (!ws || ws_bytes < snip_qlinear_workspace_size(plan, layer, T, K, N)) return SNIP_ERR_WORKSPACE;
  if (!aligned16(X) || !aligned16(W) || !aligned16(dY) || !aligned16(dX) || !aligned16(dW) || !aligned16(ws))
    return SNIP_ERR_ALIGN;
  return run_qlinear_bwd(plan, layer, X, W, dY, T, K, N, dX, dW, stats_out, ws, sms,
                         static_cast<cudaStream_t>(stream), nullptr);
}

// ---------------------------------------------------------------- NEXT-3: the backward chain
snip_status snip_qlinear_bwd_chain(const snip_plan* plan, int layer, int prev_layer, const void* X, const void* W,
                                   const void* dY, int64_t T, int64_t K, int64_t N, float* dX, float* dW,
                                   double* stats_out, const float* g_prev, uint8_t* prev_codes,
                                   uint8_t* prev_scales, uint8_t* prev_codes_t, uint8_t* prev_scales_t,
                                   float* amax_prev, void* ws, size_t ws_bytes, void* stream) {
  int sms;
  snip_status s = current_device(&sms);
  if (s != SNIP_OK) return s;
  if ((s = check_ql(plan, layer, T, K, N)) != SNIP_OK) return s;
  if (prev_layer < 0 || prev_layer >= (int)plan->fmt.size()) return SNIP_ERR_INVALID_ARG;
  // the preceding layer's gradient operands are what the re-quantizing epilogue writes: NVFP4
  if (gradient_fmt(plan->fmt[prev_layer]) != SNIP_FMT_NVFP4) return SNIP_ERR_INVALID_ARG;
  if (!X || !W || !dY || !dW || !g_prev || !prev_codes || !prev_scales || !prev_codes_t || !prev_scales_t)
    return SNIP_ERR_INVALID_ARG;
  if (!ws || ws_bytes < snip_qlinear_workspace_size(plan, layer, T, K, N)) return SNIP_ERR_WORKSPACE;
  if (!aligned16(X) || !aligned16(W) || !aligned16(dY) || (dX && !aligned16(dX)) || !aligned16(dW) ||
      !aligned16(ws) || !aligned16(prev_codes) || !aligned16(prev_scales) || !aligned16(prev_codes_t) ||
      !aligned16(prev_scales_t))
    return SNIP_ERR_ALIGN;
  // the dgrad product dX (T x K) is the preceding layer's dY, written as that layer's two NVFP4
  // operands (row blocks along K for its dgrad, column blocks along T for its wgrad) with the given
  // tensor scale and that layer's roundings and stream ids
  const int* prnd = &plan->rnd[(size_t)prev_layer * 6];
  const uint64_t psid = (uint64_t)prev_layer * 8;
  snip_requant rq;
  rq.g_in = g_prev;
  rq.rnd = prnd[SNIP_TAG_DY_DGRAD];
  rq.seed = plan->seed;
  rq.stream_id = psid + SNIP_TAG_DY_DGRAD;
  rq.codes = prev_codes;
  rq.scales = prev_scales;
  rq.amax_out = amax_prev;
  rq.rnd_t = prnd[SNIP_TAG_DYT_WGRAD];
  rq.stream_id_t = psid + SNIP_TAG_DYT_WGRAD;
  rq.codes_t = prev_codes_t;
  rq.scales_t = prev_scales_t;
  return run_qlinear_bwd(plan, layer, X, W, dY, T, K, N, dX, dW, stats_out, ws, sms,
                         static_cast<cudaStream_t>(stream), &rq);
}

snip_status snip_qlinear_bwd_q(const snip_plan* plan, int layer, const void* X, const void* W,
                               const uint8_t* dy_codes, const uint8_t* dy_scales, const uint8_t* dyt_codes,
                               const uint8_t* dyt_scales, const float* g_dy, int64_t T, int64_t K, int64_t N,
                               float* dX, float* dW, void* ws, size_t ws_bytes, void* stream) {
  int sms;
  snip_status s = current_device(&sms);
  if (s != SNIP_OK) return s;
  if ((s = check_ql(plan, layer, T, K, N)) != SNIP_OK) return s;
  if (plan->fmt[layer] != SNIP_FMT_NVFP4) return SNIP_ERR_INVALID_ARG;
  if (!X || !W || !dy_codes || !dy_scales || !dyt_codes || !dyt_scales || !g_dy || !dX || !dW)
    return SNIP_ERR_INVALID_ARG;
  if (!ws || ws_bytes < snip_qlinear_workspace_size(plan, layer, T, K, N)) return SNIP_ERR_WORKSPACE;
  if (!aligned16(X) || !aligned16(W) || !aligned16(dy_codes) || !aligned16(dy_scales) || !aligned16(dyt_codes) ||
      !aligned16(dyt_scales) || !aligned16(dX) || !aligned16(dW) || !aligned16(ws))
    return SNIP_ERR_ALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int q = SNIP_FMT_NVFP4;
  const int* rnd = &plan->rnd[(size_t)layer * 6];
  const uint64_t sid = (uint64_t)layer * 8;
  QlLayout L = ql_layout(q, T, K, N, true);
  uint8_t* b = static_cast<uint8_t*>(ws);
  float* sx = scale_slot(ws, 0);
  float* sw = scale_slot(ws, 1);
  {
    const void* xs[2] = {W, X};
    const int64_t ns[2] = {N * K, T * K};
    float* outs[2] = {sw, sx};
    if ((s = run_scales_multi(2, xs, ns, outs, ws, sms, st)) != SNIP_OK) return s;
  }
  if ((s = run_quantize(q, W, N, K, SNIP_BLOCKS_ALONG_ROWS, rnd[SNIP_TAG_WT_DGRAD], plan->seed,
                        sid + SNIP_TAG_WT_DGRAD, sw + scale_index(q), SNIP_LAYOUT_MMA, b + L.op[1].codes_off,
                        b + L.op[1].scales_off, nullptr, nullptr, sms, st)) != SNIP_OK)
    return s;
  if ((s = run_gemm(q, dy_codes, dy_scales, g_dy, b + L.op[1].codes_off, b + L.op[1].scales_off,
                    gemm_scale(sw, q), T, K, N, dX, K, ws, sms, st)) != SNIP_OK)
    return s;
  if ((s = run_quantize(q, X, T, K, SNIP_BLOCKS_ALONG_ROWS, rnd[SNIP_TAG_XT_WGRAD], plan->seed,
                        sid + SNIP_TAG_XT_WGRAD, sx + scale_index(q), SNIP_LAYOUT_MMA, b + L.op[3].codes_off,
                        b + L.op[3].scales_off, nullptr, nullptr, sms, st)) != SNIP_OK)
    return s;
  return run_gemm(q, dyt_codes, dyt_scales, g_dy, b + L.op[3].codes_off, b + L.op[3].scales_off,
                  gemm_scale(sx, q), N, K, T, dW, K, ws, sms, st);
}

// ---------------------------------------------------------------- statistics
snip_status snip_quant_stats(const void* a, int64_t rows, int64_t cols, snip_round rnd, uint64_t seed,
                             uint64_t stream_id, const float* scales_in, double* raw_out, float* block_err_nvfp4,
                             float* block_err_fp8, void* ws, size_t ws_bytes, void* stream) {
  int sms;
  snip_status s = current_device(&sms);
  if (s != SNIP_OK) return s;
  if (!valid_enum(rnd, 2) || rows < 0 || cols < 0 || !raw_out || (rows * cols > 0 && !a)) return SNIP_ERR_INVALID_ARG;
  if (cols % 16 != 0 || too_large(rows, cols)) return SNIP_ERR_SHAPE;
  if (!ws || ws_bytes < kSmallWorkspace) return SNIP_ERR_WORKSPACE;
  if (!aligned16(a) || !aligned16(ws)) return SNIP_ERR_ALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const float* sc = scales_in;
  if (!sc) {
    float* slot = scale_slot(ws, 3);
    if ((s = run_scales(a, rows * cols, slot, ws, sms, st)) != SNIP_OK) return s;
    sc = slot;
  }
  StatsParams p = {};
  p.x = static_cast<const uint16_t*>(a);
  p.rows = rows;
  p.cols = cols;
  p.seed = seed;
  p.stream_id = stream_id;
  p.rk = philox_round_keys(seed);
  p.scales3 = sc;
  p.partials = ws_at<double>(ws, kOffStatsPartials);
  p.counter = ws_at<uint32_t>(ws, kOffStatsCounter);
  p.raw_out = raw_out;
  p.block_err4 = block_err_nvfp4;
  p.block_err8 = block_err_fp8;
  return cuda_status(launch_stats(p, rnd, sms, st));
}

snip_status snip_quantize_stats(snip_format fmt, const void* x, int64_t rows, int64_t cols, snip_round rnd,
                                uint64_t seed, uint64_t stream_id, const float* scales_in, snip_layout layout,
                                uint8_t* codes, uint8_t* scales, double* raw_out, void* ws, size_t ws_bytes,
                                void* stream) {
  int sms;
  snip_status s = current_device(&sms);
  if (s != SNIP_OK) return s;
  if (!valid_operand_fmt(fmt) || !raw_out) return SNIP_ERR_INVALID_ARG;
  float g_dummy;   // validation only: g_out is not written by this entry point
  s = check_quantize_args(fmt, x, rows, cols, SNIP_BLOCKS_ALONG_COLS, rnd, layout, codes,
                          is_fp4(fmt) ? scales : nullptr, &g_dummy, ws, ws_bytes);
  if (s != SNIP_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const float* sc = scales_in;
  if (!sc) {
    float* slot = scale_slot(ws, 3);
    if ((s = run_scales(x, rows * cols, slot, ws, sms, st)) != SNIP_OK) return s;
    sc = slot;
  }
  return run_quantize(fmt, x, rows, cols, SNIP_BLOCKS_ALONG_COLS, rnd, seed, stream_id, sc + scale_index(fmt), layout,
                      codes, scales, nullptr, nullptr, sms, st, sc, raw_out, ws);
}

snip_status snip_quantize_part(snip_format fmt, const void* x, int64_t rows, int64_t cols, snip_orient orient,
                               snip_round rnd, uint64_t seed, uint64_t stream_id, uint64_t index_base,
                               const float* scales_in, snip_layout layout, uint8_t* codes, uint8_t* scales,
                               double* raw_out, void* ws, size_t ws_bytes, void* stream) {
  // argument rules first (they need no device): the part starts on a whole row of the tensor, and
  // with blocks along the rows (the tokens) on a whole block of rows, so no block straddles parts
  if (!valid_operand_fmt(fmt) || !scales_in || (raw_out && orient != SNIP_BLOCKS_ALONG_COLS) || cols <= 0 ||
      (orient != SNIP_BLOCKS_ALONG_COLS && orient != SNIP_BLOCKS_ALONG_ROWS))
    return SNIP_ERR_INVALID_ARG;
  if (index_base % 16 != 0 || index_base % (uint64_t)cols != 0) return SNIP_ERR_SHAPE;
  if (orient == SNIP_BLOCKS_ALONG_ROWS && (index_base / (uint64_t)cols) % (uint64_t)block_elems(fmt) != 0)
    return SNIP_ERR_SHAPE;
  int sms;
  snip_status s = current_device(&sms);
  if (s != SNIP_OK) return s;
  float g_dummy;   // validation only: the scales come in, none is written
  s = check_quantize_args(fmt, x, rows, cols, orient, rnd, layout, codes, is_fp4(fmt) ? scales : nullptr, &g_dummy,
                          ws, ws_bytes);
  if (s != SNIP_OK) return s;
  return run_quantize(fmt, x, rows, cols, orient, rnd, seed, stream_id, scales_in + scale_index(fmt), layout, codes,
                      is_fp4(fmt) ? scales : nullptr, nullptr, nullptr, sms, static_cast<cudaStream_t>(stream),
                      raw_out ? scales_in : nullptr, raw_out, ws, index_base);
}

// ---------------------------------------------------------------- NEXT-4: dW-level sqrt(3) check
size_t snip_dw_noise_workspace_size(int64_t K, int64_t N) {
  if (K < 0 || N < 0) return 0;
  return kSmallWorkspaceRounded;   // partial sums and the status word: dW itself is never stored
}

snip_status snip_dw_noise(const void* X, const void* dY, int64_t T, int64_t K, int64_t N, const float* dW_q,
                          double* out2, void* ws, size_t ws_bytes, void* stream) {
  int sms;
  snip_status s = current_device(&sms);
  if (s != SNIP_OK) return s;
  if (!X || !dY || !dW_q || !out2 || T <= 0 || K <= 0 || N <= 0) return SNIP_ERR_INVALID_ARG;
  if (T % 16 || K % 16 || N % 16) return SNIP_ERR_SHAPE;
  if (too_large(T, K) || too_large(T, N) || too_large(N, K)) return SNIP_ERR_SHAPE;
  if (!ws || ws_bytes < snip_dw_noise_workspace_size(K, N)) return SNIP_ERR_WORKSPACE;
  if (!aligned16(X) || !aligned16(dY) || !aligned16(dW_q) || !aligned16(ws)) return SNIP_ERR_ALIGN;
  return cuda_status(launch_dw_noise_gemm(X, dY, T, K, N, dW_q, ws_at<double>(ws, kOffStatsPartials),
                                          ws_at<uint32_t>(ws, kOffStatsCounter), out2,
                                          ws_at<uint32_t>(ws, kOffStatus), kTimeoutNs, sms,
                                          static_cast<cudaStream_t>(stream)));
}

snip_status snip_dw_noise_finalize(const double* out2_host, double* ratio, int* below_sqrt3) {
  if (!out2_host || !ratio || !below_sqrt3) return SNIP_ERR_INVALID_ARG;
  if (!std::isfinite(out2_host[0]) || !std::isfinite(out2_host[1])) return SNIP_ERR_NONFINITE;
  *ratio = out2_host[1] == 0.0 ? HUGE_VAL : std::sqrt(out2_host[0] / out2_host[1]);
  *below_sqrt3 = *ratio < 1.7320508075688772;
  return SNIP_OK;
}

snip_status snip_stats_finalize(const double* raw, snip_stats* out) {
  if (!raw || !out) return SNIP_ERR_INVALID_ARG;
  out->sum_x2 = raw[SNIP_ST_SUM_X2];
  out->nvfp4_err2 = raw[SNIP_ST_NVFP4_ERR2];
  out->fp8_err2 = raw[SNIP_ST_FP8_ERR2];
  out->nvfp4_sr_var = raw[SNIP_ST_NVFP4_SRVAR];
  out->fp8_sr_var = raw[SNIP_ST_FP8_SRVAR];
  out->amax = raw[SNIP_ST_AMAX];
  out->count = raw[SNIP_ST_COUNT];
  const double inf = __builtin_huge_val();
  out->ratio_nvfp4 = out->nvfp4_err2 == 0.0 ? inf : __builtin_sqrt(out->sum_x2 / out->nvfp4_err2);
  out->ratio_fp8 = out->fp8_err2 == 0.0 ? inf : __builtin_sqrt(out->sum_x2 / out->fp8_err2);
  out->below_sqrt3_nvfp4 = out->ratio_nvfp4 < 1.7320508075688772;
  out->below_sqrt3_fp8 = out->ratio_fp8 < 1.7320508075688772;
  return SNIP_OK;
}

}  // extern "C"
