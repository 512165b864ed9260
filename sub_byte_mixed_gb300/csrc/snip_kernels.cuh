// snip_kernels.cuh -- parameter blocks, block-level reductions and launcher
// declarations shared by the kernels (quant.cu, gemm.cu) and the C ABI
// (api.cu).  Internal to the library.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "snip_device.cuh"

namespace snip {

// One quantization launch (NVFP4 or FP8, either orientation, either layout).
struct QuantParams {
  const uint16_t* x;        // source bf16 rows x cols
  int64_t rows, cols;
  int64_t out_rows, out_cols;   // output orientation (out_cols = the blocked/contraction dim)
  int64_t orp, ocp;             // padded output dims (== out_rows/out_cols for the row-major layout)
  uint64_t seed, stream_id;
  PhiloxKey rk;                 // round keys of seed (philox_round_keys)
  const float* scale;           // device fp32 tensor scale to use (NVFP4 g or FP8 s)
  uint8_t* codes;
  uint8_t* scales;              // NVFP4 only
  float* g_out;                 // nullable: receives *scale
  float* block_err;             // NVFP4 only, nullable
  int group;                    // NVFP4: 16-element blocks sharing one scale (0 or 1: NVFP4;
                                // 2, 4, 8: 32-, 64-, 128-element blocks)
  uint64_t index_base;          // x is a part of a larger tensor starting at this element (a
                                // multiple of 16): random bits follow the whole tensor's indices
  // statistics fused into a row-block quantization (raw_out non-null)
  const float* scales3;         // {amax, NVFP4 g, FP8 s}
  double* partials;
  uint32_t* counter;
  double* raw_out;
};

struct StatsParams {
  const uint16_t* x;
  int64_t rows, cols;
  uint64_t seed, stream_id;
  PhiloxKey rk;                 // round keys of seed
  const float* scales3;         // {amax, NVFP4 g, FP8 s}
  double* partials;             // 5 doubles per CTA
  uint32_t* counter;
  double* raw_out;              // SNIP_STATS_NVALS doubles
  float* block_err4;
  float* block_err8;
};

struct GemmParams {
  const uint8_t* a_scales;
  const uint8_t* b_scales;
  const float* ga;
  const float* gb;
  float* D;
  int64_t M, N, ldd;
  int64_t kp;                   // padded contraction (elements)
  int num_k_stages;             // kp / elements-per-stage
  int num_m_tiles, num_n_tiles;
  int v8;                       // D rows allow 32-byte stores
  int a_e5m2;                   // FP8 only: A is E5M2 (B stays E4M3)
  // NVFP4 re-quantization of the output for the next GEMM (null rq_codes: no row blocks)
  uint8_t* rq_codes;            // MMA layout, rows padded to 256, N padded to rq_ocp
  uint8_t* rq_scales;
  const float* rq_g;            // tensor scale to quantize with (given, e.g. delayed)
  uint32_t* rq_amax;            // max |bf16(output)| as float bits (atomicMax; zeroed by the host)
  int64_t rq_ocp;
  uint64_t rq_seed, rq_stream;
  int rq_rnd;
  // column blocks of the same bf16 output: rows of its transpose (null rq_codes_t: off)
  uint8_t* rq_codes_t;          // MMA layout, N padded to 256 rows, M padded to rq_ocp_t
  uint8_t* rq_scales_t;
  int64_t rq_ocp_t;
  uint64_t rq_stream_t;
  int rq_rnd_t;
  uint32_t* status;
  uint64_t timeout_ns;
};

// ------------------------------------------------------------------ block reductions
__device__ __forceinline__ uint32_t mag_max4(uint4 a) {
  return __vmaxu2(__vmaxu2(a.x & 0x7fff7fffu, a.y & 0x7fff7fffu), __vmaxu2(a.z & 0x7fff7fffu, a.w & 0x7fff7fffu));
}

// Max over the CTA (blockDim.x a multiple of 32, <= 1024); result valid in
// every thread.
__device__ __forceinline__ uint32_t block_max_u32(uint32_t v) {
  __shared__ uint32_t red[32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31, nw = blockDim.x >> 5;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  v = l < nw ? red[l] : 0u;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Sum of N floats over the CTA; result valid in thread 0.  (The fp64 pipe of
// this GPU is a small fraction of its fp32 rate: sums within a CTA stay fp32.)
template <int N>
__device__ __forceinline__ void block_sum_f32(float (&v)[N]) {
  __shared__ float red32[32][N];
#pragma unroll
  for (int k = 0; k < N; ++k)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v[k] += __shfl_xor_sync(0xffffffffu, v[k], o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31, nw = blockDim.x >> 5;
  __syncthreads();
  if (l == 0)
#pragma unroll
    for (int k = 0; k < N; ++k) red32[w][k] = v[k];
  __syncthreads();
  if (w == 0) {
#pragma unroll
    for (int k = 0; k < N; ++k) {
      v[k] = l < nw ? red32[l][k] : 0.0f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v[k] += __shfl_xor_sync(0xffffffffu, v[k], o);
    }
  }
}

// Sum of N doubles over the CTA; result valid in thread 0.
template <int N>
__device__ __forceinline__ void block_sum_f64(double (&v)[N]) {
  __shared__ double red[32][N];
#pragma unroll
  for (int k = 0; k < N; ++k)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v[k] += __shfl_xor_sync(0xffffffffu, v[k], o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31, nw = blockDim.x >> 5;
  __syncthreads();
  if (l == 0)
#pragma unroll
    for (int k = 0; k < N; ++k) red[w][k] = v[k];
  __syncthreads();
  if (w == 0) {
#pragma unroll
    for (int k = 0; k < N; ++k) {
      v[k] = l < nw ? red[l][k] : 0.0;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v[k] += __shfl_xor_sync(0xffffffffu, v[k], o);
    }
  }
}

// ------------------------------------------------------------------ launchers
cudaError_t launch_scales(const uint16_t* x, int64_t n, uint32_t* partials, uint32_t* counter, float* out3,
                          uint32_t* status, int num_sms, cudaStream_t st);
// Up to kMaxMultiScales tensors' scales in one launch (cta0 filled by the launcher).
constexpr int kMaxMultiScales = 8;
struct ScalesMulti {
  const uint16_t* x[kMaxMultiScales];
  int64_t n[kMaxMultiScales];
  float* out3[kMaxMultiScales];
  int cta0[kMaxMultiScales + 1];
  int count;
};
cudaError_t launch_scales_multi(ScalesMulti m, uint32_t* partials, uint32_t* counters, uint32_t* status,
                                int num_sms, cudaStream_t st);
cudaError_t launch_quant(int fmt, const QuantParams& p, int orient, int layout, int rnd, bool err, int num_sms,
                         cudaStream_t st);
cudaError_t launch_stats(const StatsParams& p, int rnd, int num_sms, cudaStream_t st);
// {||dW||^2, ||dW_q - dW||^2} into out2 (device) with dW = dY^T X from the bf16 tensors X (T x K) and
// dY (T x N), dW_q N x K fp32: a bf16 tensor-core GEMM with the two sums in its epilogue (dw_noise.cu).
cudaError_t launch_dw_noise_gemm(const void* X, const void* dY, int64_t T, int64_t K, int64_t N, const float* dwq,
                                 double* partials, uint32_t* counter, double* out2, uint32_t* status,
                                 uint64_t timeout_ns, int num_sms, cudaStream_t st);

// GEMM: D = ga*gb*A B^T on MMA-layout operands.  fmt 1 = NVFP4, 2 = MXFP4 (ga, gb
// null: no tensor scales), 0 = FP8 (p.a_e5m2: A in E5M2, B in E4M3).
// a_codes / b_codes are passed to the launcher, which builds the TMA tensor
// maps.
cudaError_t launch_gemm(int fmt, const uint8_t* a_codes, int64_t a_rows_padded, const uint8_t* b_codes,
                        int64_t b_rows_padded, const GemmParams& p, int num_sms, cudaStream_t st);

// The driver's cuTensorMapEncodeTiled (looked up once through the runtime), or null if unavailable.
// Defined in gemm.cu, used by every kernel launcher that builds TMA tensor maps.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn tensor_map_encoder();

// Raise a kernel's dynamic shared-memory limit to `bytes` on the current device, once per kernel and
// device (the attribute is per device; thread-safe).  Defined in quant.cu.
cudaError_t ensure_max_dynamic_smem(const void* fn, int bytes);

// Launch with programmatic stream serialization (the kernel starts with pdl_enter) and, for cluster > 1,
// thread-block clusters of that many CTAs along x.
template <class... K, class... A>
cudaError_t launch_pdl(void (*kernel)(K...), unsigned grid, unsigned block, unsigned smem, unsigned cluster,
                       cudaStream_t st, A... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(block, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = cluster > 1 ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Self-check of the bounded wait (waitcheck.cu): out = {completed 0, completed 1, ns}.
cudaError_t launch_wait_check(uint32_t* status, uint64_t limit_ns, uint32_t* out, cudaStream_t st);

// Upper bound on the number of amax / stats partial slots any launch uses.
constexpr int kMaxPartials = 2048;

__device__ __forceinline__ U4 make_zero_u4() { return U4{0u, 0u, 0u, 0u}; }

}  // namespace snip
