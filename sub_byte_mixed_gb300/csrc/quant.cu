// quant.cu -- HBM-bound kernels of the quantized linear layer: tensor scales
// (a1: amax, NVFP4 g, FP8 s), NVFP4 quantization with blocks along columns
// (a2) or rows (a3), FP8 E4M3 quantization (a4) and SNIP's statistics pass
// (a8).
//
// Sources: "FP4 all the way" (Chmiel et al.), summary page, Outline (NVFP4 =
// 16 E2M1 values sharing an E4M3 scale; RTN forward, SR backward; the
// sqrt(3)-times-noise threshold); "SNIP", Abstract and Figure 2 (statistics of
// activations, weights and gradients); "SNIP", Figure 5 (each GEMM operand
// quantized along its own contraction dim).
//
// Design: every kernel streams its input once with 16-byte loads.  One thread
// owns one 16-element block (32 source bytes), so the block's scale is
// computed once and no shuffles are needed; a warp covers 32 consecutive
// blocks of a row.  The transposed (column-block) kernels stage a 128 x 64
// tile in shared memory so that loads and stores both stay coalesced.
// Rounding to nearest and stochastic rounding both run as fp32 additions on
// the FMA pipe (grid_rn2 / grid_sr2, snip_device.cuh) with one Philox4x32-10
// call per 8 source elements; codes come from the hardware E2M1/E4M3/E5M2
// conversions of the exact grid values.
#include <algorithm>
#include <mutex>
#include <utility>
#include <vector>

#include "snip_kernels.cuh"
#include "snip_quant.cuh"

namespace snip {


// ------------------------------------------------------------------ a1: tensor scales
// Magnitudes are compared as bf16 bit patterns (sign cleared): for finite
// values the integer order is the float order, and any pattern >= 0x7f80 is
// an infinity or NaN.  Each CTA publishes its max; the last CTA to finish
// reduces them and writes out3 = {amax, g = amax/2688, s = amax/448} (g = s = 1
// for an all-zero tensor; all NaN and the status bit for non-finite input).
// The work of one CTA among nblk on one tensor (local CTA index lb).
__device__ __forceinline__ void scales_body(const uint16_t* __restrict__ x, int64_t n, uint32_t lb, uint32_t nblk,
                                            uint32_t* __restrict__ partials, uint32_t* __restrict__ counter,
                                            float* __restrict__ out3, uint32_t* __restrict__ status) {
  uint32_t m2 = 0;
  const int64_t nvec = n >> 3;
  const uint4* xv = reinterpret_cast<const uint4*>(x);
  const int64_t stride = (int64_t)nblk * blockDim.x;
  int64_t i = (int64_t)lb * blockDim.x + threadIdx.x;
  // eight independent 16-byte loads in flight per thread (128 B), then four
  for (; i + 7 * stride < nvec; i += 8 * stride) {
    uint4 r[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) r[k] = __ldg(xv + i + k * stride);
#pragma unroll
    for (int k = 0; k < 8; ++k) m2 = __vmaxu2(m2, mag_max4(r[k]));
  }
  for (; i + 3 * stride < nvec; i += 4 * stride) {
    const uint4 a = __ldg(xv + i), b = __ldg(xv + i + stride), c = __ldg(xv + i + 2 * stride),
                d = __ldg(xv + i + 3 * stride);
    m2 = __vmaxu2(m2, __vmaxu2(__vmaxu2(mag_max4(a), mag_max4(b)), __vmaxu2(mag_max4(c), mag_max4(d))));
  }
  for (; i < nvec; i += stride) m2 = __vmaxu2(m2, mag_max4(__ldg(xv + i)));
  if (lb == 0 && threadIdx.x < (n & 7)) m2 = __vmaxu2(m2, (uint32_t)(x[(nvec << 3) + threadIdx.x] & 0x7fffu));
  uint32_t m = max(m2 & 0xffffu, m2 >> 16);
  m = block_max_u32(m);
  __shared__ bool s_last;
  if (threadIdx.x == 0) {
    partials[lb] = m;
    if (m >= 0x7f80u) atomicOr(status, kDevNonFinite);
    __threadfence();
    s_last = atomicAdd(counter, 1u) == nblk - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  uint32_t mm = 0;
  for (uint32_t j = threadIdx.x; j < nblk; j += blockDim.x) mm = max(mm, ((volatile uint32_t*)partials)[j]);
  mm = block_max_u32(mm);
  if (threadIdx.x == 0) {
    if (mm >= 0x7f80u) {
      const float nan = __int_as_float(0x7fc00000);
      out3[0] = nan; out3[1] = nan; out3[2] = nan;
    } else {
      const float a = bf16_bits_to_float(mm);
      out3[0] = a;
      out3[1] = a == 0.0f ? 1.0f : __fdiv_rn(a, 2688.0f);   // 6 * 448: largest E2M1 x largest E4M3
      out3[2] = a == 0.0f ? 1.0f : __fdiv_rn(a, 448.0f);
    }
    *counter = 0;  // ready for the next reduction on this workspace
  }
}

__global__ void __launch_bounds__(256, 4) scales_kernel(const uint16_t* __restrict__ x, int64_t n,
                                                        uint32_t* __restrict__ partials,
                                                        uint32_t* __restrict__ counter, float* __restrict__ out3,
                                                        uint32_t* __restrict__ status) {
  pdl_enter();
  scales_body(x, n, blockIdx.x, gridDim.x, partials, counter, out3, status);
}

// Several tensors in one launch: tensor t owns CTAs [cta0[t], cta0[t+1]), its
// partial slots at the same indices and its own completion counter.
__global__ void __launch_bounds__(256, 4) scales_multi_kernel(ScalesMulti m, uint32_t* __restrict__ partials,
                                                              uint32_t* __restrict__ counters,
                                                              uint32_t* __restrict__ status) {
  pdl_enter();
  // this CTA's tensor, picked with constant indices (a run-time index into the parameter block would
  // copy it to local memory)
  const uint16_t* x = m.x[0];
  int64_t n = m.n[0];
  float* out3 = m.out3[0];
  int t = 0, c0 = 0, c1 = m.cta0[1];
#pragma unroll
  for (int k = 1; k < kMaxMultiScales; ++k)
    if (k < m.count && (int)blockIdx.x >= m.cta0[k]) {
      t = k; x = m.x[k]; n = m.n[k]; out3 = m.out3[k]; c0 = m.cta0[k]; c1 = m.cta0[k + 1];
    }
  scales_body(x, n, blockIdx.x - (uint32_t)c0, (uint32_t)(c1 - c0), partials + c0, counters + t, out3, status);
}

// Squared dequantization error of an encoded block (x_hat = value(code) * p).
__device__ __forceinline__ float nvfp4_block_err(const float (&v)[16], const uint2& c, float p) {
  float e = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t byte = ((i < 4 ? c.x : c.y) >> (8 * (i & 3))) & 0xffu;
    const float2 q = e2m1x2_decode(byte);
    const float d0 = __fsub_rn(__fmul_rn(q.x, p), v[2 * i]);
    const float d1 = __fsub_rn(__fmul_rn(q.y, p), v[2 * i + 1]);
    e = __fadd_rn(e, __fadd_rn(__fmul_rn(d0, d0), __fmul_rn(d1, d1)));
  }
  return e;
}

// Encode 16 signed values to E4M3 (E5 false) or E5M2 (E5 true) with the
// tensor scale's inverse.
template <int RND, bool E5 = false, class Bits = PackedBits>
__device__ __forceinline__ uint4 fp8_encode16(const float (&v)[16], float inv, Bits bits) {
  constexpr uint32_t kMaxCode = E5 ? 0x7bu : 0x7eu;
  uint32_t w[4] = {0u, 0u, 0u, 0u};
  if (!(inv < kInf)) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t sign = (__float_as_uint(v[i]) >> 24) & 0x80u;
      w[i >> 2] |= (sign | (v[i] == 0.0f ? 0u : kMaxCode)) << (8 * (i & 3));
    }
  } else if (RND == 0) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      w[j] = fp8x4_rn_sat<E5>(__fmul_rn(v[4 * j], inv), __fmul_rn(v[4 * j + 1], inv), __fmul_rn(v[4 * j + 2], inv),
                              __fmul_rn(v[4 * j + 3], inv));
  } else {
    // stochastic rounding on the FMA pipe (grid_sr2), the code converted from the exact grid value.
    // y is not clamped to the grid's top: past it (the tensor scale's rounding) the grid value is the
    // top or more and the saturating conversion gives the top either way.
    constexpr float kC = E5 ? 2097152.0f : 1048576.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float a[4];
#pragma unroll
      for (int k = 0; k < 4; k += 2) {
        const int i = 4 * j + k;
        const float2 y = __fmul2_rn(make_float2(fabsf(v[i]), fabsf(v[i + 1])), make_float2(inv, inv));
        const float2 H = E5 ? make_float2(e5m2_step_x4(y.x), e5m2_step_x4(y.y))
                            : make_float2(e4m3_step_x8(y.x), e4m3_step_x8(y.y));
        const float2 g = E5 ? sr_g2<18>(bits.f23(i), bits.f23(i + 1)) : sr_g2<19>(bits.f23(i), bits.f23(i + 1));
        const float2 q = grid_sr2(y, H, g, kC);
        a[k] = copysignf(q.x, v[i]);
        a[k + 1] = copysignf(q.y, v[i + 1]);
      }
      w[j] = fp8x4_rn_sat<E5>(a[0], a[1], a[2], a[3]);
    }
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// E5M2 tensor scale from the tensor's amax: amax / 57344 (1 for zero; NaN stays NaN).
__device__ __forceinline__ float e5m2_tensor_scale(float amax) {
  return amax == 0.0f ? 1.0f : __fdiv_rn(amax, 57344.0f);
}

// ------------------------------------------------------------------ a8: statistics
// One pass: ||A||^2, the squared errors of NVFP4 and FP8 quantization under
// the tensor's rounding, and the expected SR squared error on both grids,
// sum (hi-|y|)(|y|-lo) q^2.  With c the signed distance from |y| (clamped to
// the grid's top, where the product is 0) to a neighbouring grid value and
// h = hi - lo, that product is |c| (h - |c|) for either neighbour: the
// rounding of the pass (nearest, or the stochastic pick) supplies the
// neighbour.  It is summed in units of the scale and multiplied by p^2 (s^2)
// per block.  The sums
// need no bit exactness, so they use fused multiply-adds; per-thread sums are
// fp32 (a few hundred elements), per-CTA and final sums fp64.

// Statistics of one 16-element block: squares of the values, the squared
// errors of NVFP4 (block scale bs) and FP8 (tensor scale s8) quantization
// under rounding RND, and the expected SR variance on both grids.
// CF = 1 / 0 also returns the block's NVFP4 / FP8 codes (packed as by
// nvfp4_encode16 / fp8_encode16) from the same roundings, except where that
// format's scale is special (bs.special, special8): there the caller
// encodes.  CF = -1: statistics only.
// Element pairs go through Blackwell's packed fp32 operations (__fmul2_rn,
// __ffma2_rn, __fadd2_rz: per lane the IEEE result of the scalar operation),
// and each candidate's rounding is the FMA-pipe form (grid_rn2 / grid_sr2),
// which gives the grid value q of the code the rule picks; the code is then
// the hardware conversion of that exact value.  With y clamped to the grid's
// top (yc; the FP8 candidate needs no clamp, see there) and c = q - yc, the
// expected SR variance (hi - y)(y - lo) is |c| (h - |c|) whichever neighbour
// q is, summed as 1/2 sum |c| H - sum c^2 (H = twice the E2M1 step; eight
// times the E4M3 step with 1/8).
// The running sums of one thread over its blocks.  Only the NVFP4 variance is
// scaled per block (by its p^2); everything else accumulates across blocks
// (the FP8 variance in units of the tensor scale s8, multiplied at the end).
struct StatsAcc {
  float2 x2, e4, e8, S8;
  float T8, v4;
  __device__ __forceinline__ void init() {
    x2 = e4 = e8 = S8 = make_float2(0.f, 0.f);
    T8 = v4 = 0.f;
  }
  // the five sums: ||A||^2, NVFP4 err^2, FP8 err^2, NVFP4 and FP8 expected SR variance
  __device__ __forceinline__ void finish(float s8, bool special8, float (&out)[5]) const {
    out[0] = x2.x + x2.y;
    out[1] = e4.x + e4.y;
    out[2] = e8.x + e8.y;
    out[3] = v4;
    out[4] = special8 ? 0.0f : fmaf(0.125f, T8, -(S8.x + S8.y)) * (s8 * s8);
  }
};
// BE: also return the block's two squared errors (per-block error outputs).
// GEN: the general form, which handles a special NVFP4 block scale or FP8 tensor scale; without it
// both are taken as ordinary, and the unrolled body has no branch (stats_block16 picks the form).
template <int CF, int RND, bool BE, bool GEN>
__device__ __forceinline__ void stats_block16_form(const float (&v)[16], const BlockScale& bs, const uint32_t (&u)[8],
                                                   float s8, float inv8, bool special8, uint4& codes, StatsAcc& acc,
                                                   float* be4, float* be8) {
  float2 S4 = make_float2(0.f, 0.f), b4 = S4, b8 = S4;
  float T4 = 0.f;
  uint32_t cw[4] = {0u, 0u, 0u, 0u};
  float qa[8];   // signed grid values of the CF format awaiting conversion (one word's worth)
  const float2 inv2 = make_float2(bs.inv, bs.inv), np2 = make_float2(-bs.p, -bs.p);
  const float2 i8 = make_float2(inv8, inv8), ns8 = make_float2(-s8, -s8), m1 = make_float2(-1.0f, -1.0f);
  float2& E4 = BE ? b4 : acc.e4;
  float2& E8 = BE ? b8 : acc.e8;
#pragma unroll
  for (int i = 0; i < 16; i += 2) {
    const float2 va = make_float2(fabsf(v[i]), fabsf(v[i + 1]));
    acc.x2 = __ffma2_rn(va, va, acc.x2);
    float2 g17 = va, g19 = va;   // random fractions of the pair (stochastic rounding)
    if (RND) {
      const float f0 = sr_f23<false>(u[i >> 1]), f1 = sr_f23<true>(u[i >> 1]);
      g17 = sr_g2<17>(f0, f1);
      g19 = sr_g2<19>(f0, f1);
    }
    // ---------------- NVFP4
    if (GEN && bs.special) {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const float q = (bs.p == 0.0f || v[i + k] == 0.0f) ? 0.0f : copysignf(6.0f, v[i + k]);
        const float d = fmaf(q, bs.p, -v[i + k]);
        E4.x = fmaf(d, d, E4.x);
      }
    } else {
      const float2 y = __fmul2_rn(va, inv2);
      const float2 yc = make_float2(fminf(y.x, 6.0f), fminf(y.y, 6.0f));
      const float2 H = make_float2(e2m1_step_x2(yc.x), e2m1_step_x2(yc.y));
      const float2 q = RND ? grid_sr2(yc, H, g17, 4194304.0f) : grid_rn2(yc, H, 4194304.0f);
      if (CF == 1) {
        qa[i & 7] = copysignf(q.x, v[i]);
        qa[(i & 7) + 1] = copysignf(q.y, v[i + 1]);
        if ((i & 7) == 6) cw[i >> 3] = e2m1x8_rn(qa);
      }
      const float2 d = __ffma2_rn(q, np2, va);            // |x| - |x_hat|
      E4 = __ffma2_rn(d, d, E4);
      const float2 c = __ffma2_rn(yc, m1, q);
      S4 = __ffma2_rn(c, c, S4);
      T4 = fmaf(fabsf(c.x), H.x, T4);
      T4 = fmaf(fabsf(c.y), H.y, T4);
    }
    // ---------------- FP8
    if (GEN && special8) {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const float q = v[i + k] == 0.0f ? 0.0f : copysignf(448.0f, v[i + k]);
        const float d = fmaf(q, s8, -v[i + k]);
        E8.x = fmaf(d, d, E8.x);
      }
    } else {
      // y is not clamped to 448: under the tensor scale only an element equal to the tensor's amax
      // can pass 448 (any other bf16 value is smaller by a factor of at most 1 - 2^-8), and only by the
      // roundings of amax / 448, its inverse and the product (under 2^-21 relative); its grid value
      // is 448 either way, so codes and error sums are those of the clamped form, and its SR-variance
      // term moves by under 2^-21 * 448 * H
      const float2 yc = __fmul2_rn(va, i8);
      const float2 H = make_float2(e4m3_step_x8(yc.x), e4m3_step_x8(yc.y));
      const float2 q = RND ? grid_sr2(yc, H, g19, 1048576.0f) : grid_rn2(yc, H, 1048576.0f);
      if (CF == 0) {
        qa[i & 3] = copysignf(q.x, v[i]);
        qa[(i & 3) + 1] = copysignf(q.y, v[i + 1]);
        if ((i & 3) == 2) cw[i >> 2] = fp8x4_rn_sat(qa[0], qa[1], qa[2], qa[3]);
      }
      const float2 d = __ffma2_rn(q, ns8, va);
      E8 = __ffma2_rn(d, d, E8);
      const float2 c = __ffma2_rn(yc, m1, q);
      acc.S8 = __ffma2_rn(c, c, acc.S8);
      acc.T8 = fmaf(fabsf(c.x), H.x, acc.T8);
      acc.T8 = fmaf(fabsf(c.y), H.y, acc.T8);
    }
  }
  // the NVFP4 variance was summed in units of this block's scale
  if (!(GEN && bs.special)) acc.v4 = fmaf(fmaf(0.5f, T4, -(S4.x + S4.y)), bs.p * bs.p, acc.v4);
  if (BE) {
    *be4 = b4.x + b4.y;
    *be8 = b8.x + b8.y;
    acc.e4.x += *be4;
    acc.e8.x += *be8;
  }
  codes = make_uint4(cw[0], cw[1], cw[2], cw[3]);
}
template <int CF, int RND, bool BE = false>
__device__ __forceinline__ void stats_block16(const float (&v)[16], const BlockScale& bs, const uint32_t (&u)[8],
                                              float s8, float inv8, bool special8, uint4& codes, StatsAcc& acc,
                                              float* be4 = nullptr, float* be8 = nullptr) {
  if (bs.special || special8)
    stats_block16_form<CF, RND, BE, true>(v, bs, u, s8, inv8, special8, codes, acc, be4, be8);
  else
    stats_block16_form<CF, RND, BE, false>(v, bs, u, s8, inv8, special8, codes, acc, be4, be8);
}

// CTA reduction of the five fp32 per-thread sums into fp64, then the last CTA
// to finish adds all CTAs' partials and writes the raw statistics vector.
__device__ __forceinline__ void stats_finish(const float (&sums)[5], double* partials, uint32_t* counter,
                                             double* raw_out, float amax, int64_t count) {
  // within the CTA in fp32 (256 partial sums: a few ulps), across CTAs in fp64
  float acc[5] = {sums[0], sums[1], sums[2], sums[3], sums[4]};
  block_sum_f32<5>(acc);
  __shared__ bool s_last;
  if (threadIdx.x == 0) {
    for (int k = 0; k < 5; ++k) partials[(int64_t)blockIdx.x * 5 + k] = (double)acc[k];
    __threadfence();
    s_last = atomicAdd(counter, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // the last CTA: warp k adds quantity k of every CTA's partials
  double tot[5] = {0, 0, 0, 0, 0};
  const uint32_t w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __shared__ double s_tot[5];
  if (w < 5) {
    double t = 0.0;
    for (uint32_t j = l; j < gridDim.x; j += 32) t += ((volatile double*)partials)[(int64_t)j * 5 + w];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if (l == 0) s_tot[w] = t;
  }
  __syncthreads();
  if (threadIdx.x == 0)
    for (int k = 0; k < 5; ++k) tot[k] = s_tot[k];
  if (threadIdx.x == 0) {
    for (int k = 0; k < 5; ++k) raw_out[k] = tot[k];
    raw_out[5] = (double)amax;
    raw_out[6] = (double)count;
    raw_out[7] = 0.0;
    *counter = 0;
  }
}

__device__ __forceinline__ void stats_nan(double* raw_out) {
  if (blockIdx.x == 0 && threadIdx.x == 0)
    for (int k = 0; k < 8; ++k) raw_out[k] = __longlong_as_double(0x7ff8000000000000ll);
}

// ------------------------------------------------------------------ a2 / a4: blocks along columns
// One thread per 16-element block; a warp covers 32 consecutive blocks of one
// output row.  Rows and blocks past the source tensor (MMA padding) encode as
// zeros.
// STATS: also accumulate SNIP's statistics of the tensor (both formats, this
// call's rounding and random bits) from the same read; needs p.scales3.
// FMT: 0 FP8, 1 NVFP4, 2 MXFP4 (lanes 2i and 2i+1 hold the two halves of one
// 32-element block and share its scale through a shuffle; with STATS each lane
// also takes the statistics of its 16 elements under the candidate formats).
// LONG (with STATS, NVFP4 only): codes with p.group-block scales beside the
// 16-element statistics -- its own instantiation, so the statistics kernels of
// the other formats keep their registers.  Without STATS p.group is read at run
// time.
template <int FMT, int LAYOUT, int RND, bool ERR, bool STATS, bool LONG = false>
__global__ void __launch_bounds__(256, STATS ? 3 : 4) quant_rows_kernel(QuantParams p) {
  pdl_enter();
  static_assert(!LONG || (FMT == 1 && STATS), "LONG: NVFP4 with fused statistics");
  static_assert(FMT < 2 || !ERR, "MXFP4 / E5M2 quantization has no block errors");
  // FMT 3 (E5M2): p.scale is the amax; MXFP4: read only for the non-finite check
  const float g = FMT == 3 ? e5m2_tensor_scale(*p.scale) : *p.scale;
  if (blockIdx.x == 0 && threadIdx.x == 0 && p.g_out) *p.g_out = (FMT == 2 && !isnan(g)) ? 1.0f : g;
  if (isnan(g)) {
    if (STATS) stats_nan(p.raw_out);
    return;
  }
  // the two tensor scales (the one not used by this format feeds the statistics)
  const float g4 = STATS ? p.scales3[1] : g, s8 = STATS ? p.scales3[2] : g;
  const float six_g = __fmul_rn(6.0f, g4);
  // p and 1/p of every NVFP4 block-scale code under g4
  constexpr bool TAB = FMT == 1 || STATS;
  __shared__ float2 s_tab[TAB ? kScaleCodes : 1];
  if (TAB) {
    fill_scale_table(s_tab, g4);
    __syncthreads();
  }
  const float inv8 = __frcp_rn(s8);
  const bool special8 = !(inv8 < kInf);
  // E5M2 codes beside the statistics: the E5M2 tensor scale's inverse (without statistics, inv8)
  const float inv5 = FMT == 3 && STATS ? __frcp_rn(g) : inv8;
  const uint32_t bpr = (uint32_t)(p.ocp >> 4);   // blocks per output row (padded)
  const uint32_t spr = (bpr + 31) >> 5;          // 32-block segments per row
  const uint32_t total = (uint32_t)p.orp * spr;
  const uint32_t lane = threadIdx.x & 31;
  const uint32_t wstride = gridDim.x * (blockDim.x >> 5);
  StatsAcc acc;
  acc.init();
  // segment -> (row, segment in row), stepped without a division per iteration
  const uint32_t seg0 = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const uint32_t wq = wstride / spr, wr = wstride - wq * spr;
  uint32_t nr = seg0 / spr, nsr = seg0 - nr * spr;
  // software pipeline: the next segment's 32 bytes are requested before this one is encoded
  uint4 na = make_uint4(0u, 0u, 0u, 0u), nb = na;
  auto fetch = [&](uint32_t rr, uint32_t ss) {
    const uint32_t kk = ss * 32 + lane;
    na = make_uint4(0u, 0u, 0u, 0u);
    nb = na;
    if (rr < p.out_rows && (int64_t)kk * 16 < p.out_cols) {
      const uint4* src = reinterpret_cast<const uint4*>(p.x + (int64_t)rr * p.cols + (int64_t)kk * 16);
      na = __ldg(src);
      nb = __ldg(src + 1);
    }
  };
  if (seg0 < total) fetch(nr, nsr);
  for (uint32_t seg = seg0; seg < total; seg += wstride) {
    const uint32_t r = nr, sr = nsr;
    const uint4 a = na, b = nb;
    nr += wq;
    nsr += wr;
    if (nsr >= spr) { nsr -= spr; ++nr; }
    if (seg + wstride < total) fetch(nr, nsr);
    const uint32_t kb = sr * 32 + lane;
    // MXFP4 lanes, and NVFP4 lanes of longer blocks, leave after the shuffles that share block maxima
    const bool longer = FMT == 1 && (STATS ? LONG : p.group > 1);
    if (FMT != 2 && kb >= bpr && !longer) continue;
    const bool real = r < p.out_rows && (int64_t)kb * 16 < p.out_cols;
    const int64_t e0 = (int64_t)r * p.cols + (int64_t)kb * 16;
    float v[16];
    unpack16(a, b, v);
    uint32_t u[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    if (RND == 1 && real) sr_bits16_rk(e0 + (int64_t)p.index_base, p.stream_id, p.rk, u);
    // bs: the 16-element NVFP4 scale (codes, and the statistics' NVFP4 candidate); bw: the scale
    // the codes are written with -- bs, or with longer blocks the scale of p.group 16-element blocks
    BlockScale bs, bw;
    if (FMT == 2) {
      const uint32_t m16 = amax16_bits(a, b);
      const uint32_t m = max(m16, __shfl_xor_sync(0xffffffffu, m16, 1));
      if (kb >= bpr) continue;
      bw = mxfp4_block_scale(m);
      // the statistics' NVFP4 candidate has its own 16-element scale; the codes use the E8M0 one
      bs = STATS ? nvfp4_block_scale_tab(m16, six_g, s_tab) : bw;
    }
    if (longer) {
      // one scale for p.group consecutive 16-element blocks: lanes 2^k apart share their maxima
      const uint32_t m16 = amax16_bits(a, b);
      uint32_t m = m16;
      for (int o = 1; o < p.group; o <<= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (kb >= bpr) continue;
      bw = nvfp4_block_scale_tab(m, six_g, s_tab);
      bs = STATS ? nvfp4_block_scale_tab(m16, six_g, s_tab) : bw;
    } else if (FMT == 1 || STATS) {
      bs = nvfp4_block_scale_tab(amax16_bits(a, b), six_g, s_tab);
    }
    if (!longer && FMT != 2) bw = bs;
    uint4 c = make_uint4(0u, 0u, 0u, 0u);   // FP8: 16 codes; FP4: .x, .y
    if (STATS && (longer || FMT >= 2)) {
      // statistics of the two candidate formats (16-element NVFP4, E4M3); codes with the scale of
      // the longer NVFP4 block, of the MXFP4 block, or E5M2's tensor scale
      if (real) {
        stats_block16<-1, RND>(v, bs, u, s8, inv8, special8, c, acc);
        if (FMT == 3) {
          c = fp8_encode16<RND, true>(v, inv5, PackedBits{u});
        } else {
          const uint2 e = nvfp4_encode16<RND>(v, bw, PackedBits{u});
          c.x = e.x;
          c.y = e.y;
        }
      }
    } else if (STATS) {
      // the codes come out of the statistics' own conversions
      if (real) {
        stats_block16<FMT, RND>(v, bs, u, s8, inv8, special8, c, acc);
        if (FMT == 1 && bs.special) {
          const uint2 e = nvfp4_encode16<RND>(v, bs, PackedBits{u});
          c.x = e.x;
          c.y = e.y;
        }
        if (FMT == 0 && special8) c = fp8_encode16<RND>(v, inv8, PackedBits{u});
      }
    } else if (FMT == 1 || FMT == 2) {
      const uint2 e = nvfp4_encode16<RND>(v, bw, PackedBits{u});
      c.x = e.x;
      c.y = e.y;
    } else {
      c = fp8_encode16<RND, FMT == 3>(v, inv8, PackedBits{u});
    }
    if (FMT == 2) {   // the even lane of a pair writes the block's scale
      const uint2 c2 = make_uint2(c.x, c.y);
      if (LAYOUT == 0) {
        if (!real) continue;
        *reinterpret_cast<uint2*>(p.codes + (int64_t)r * (p.out_cols >> 1) + (int64_t)kb * 8) = c2;
        if (!(kb & 1)) p.scales[(int64_t)r * (p.out_cols >> 5) + (kb >> 1)] = (uint8_t)bw.s;
      } else {
        *reinterpret_cast<uint2*>(p.codes + (int64_t)r * (p.ocp >> 1) + (int64_t)kb * 8) = c2;
        if (!(kb & 1)) p.scales[mma_scale_offset_mx(r, kb >> 1, p.ocp)] = (uint8_t)bw.s;
      }
    } else if (FMT == 1) {
      const uint2 c2 = make_uint2(c.x, c.y);
      if (LAYOUT == 0) {
        if (!real) continue;
        *reinterpret_cast<uint2*>(p.codes + (int64_t)r * (p.out_cols >> 1) + (int64_t)kb * 8) = c2;
        p.scales[(int64_t)r * (p.out_cols >> 4) + kb] = (uint8_t)bw.s;
      } else {
        *reinterpret_cast<uint2*>(p.codes + (int64_t)r * (p.ocp >> 1) + (int64_t)kb * 8) = c2;
        p.scales[mma_scale_offset(r, kb, p.ocp)] = (uint8_t)bw.s;
      }
      if (ERR && real && p.block_err) p.block_err[(int64_t)r * (p.out_cols >> 4) + kb] = nvfp4_block_err(v, c2, bw.p);
    } else {
      const int64_t pitch = LAYOUT == 0 ? p.out_cols : p.ocp;
      if (LAYOUT == 0 && !real) continue;
      *reinterpret_cast<uint4*>(p.codes + (int64_t)r * pitch + (int64_t)kb * 16) = c;
    }
  }
  if (STATS) {
    float sums[5];
    acc.finish(s8, special8, sums);
    stats_finish(sums, p.partials, p.counter, p.raw_out, p.scales3[0], p.rows * p.cols);
  }
}

// ------------------------------------------------------------------ a3 / a4: blocks along rows (transposed output)
// Tile: TR source rows (TR/16 blocks of the output contraction) x 64 source
// columns (64 output rows), 2 TR threads.  Thread (column pair cp, block b)
// encodes the two blocks of source columns 2cp and 2cp+1, rows 16b..16b+15.
// TR = 64 (128 threads, ~22 KB of shared memory) fits on an SM beside a GEMM
// CTA, so the column quantizations run next to the GEMMs; TR = 128 serves the
// 128-element NVFP4 blocks, which need all 128 rows of the tile.
constexpr int kTC = 64;
constexpr int kXW = kTC / 2 + 4;   // words per staged source row (pairs of bf16), padded

// FMT: 0 FP8, 1 NVFP4, 2 MXFP4 (a 32-row block is split over threads b and
// b^1, which exchange their half maxima through shared memory).
template <int FMT, int LAYOUT, int RND, bool ERR, int TR>
__global__ void __launch_bounds__(2 * TR) quant_cols_kernel(QuantParams p) {
  pdl_enter();
  static_assert(FMT < 2 || !ERR, "MXFP4 / E5M2 quantization has no block errors");
  static_assert(TR == 64 || TR == 128, "tile rows");
  constexpr bool FP4 = FMT == 1 || FMT == 2;
  constexpr int NT = 2 * TR;                      // threads
  constexpr int NB = TR / 16;                     // 16-row blocks per tile
  constexpr int OB = FP4 ? TR / 2 : TR;           // output bytes per row of the tile
  constexpr int OW = OB / 4 + 1;                  // staged output row, words (odd: fewer conflicts)
  __shared__ __align__(16) uint32_t xs[TR][kXW];
  __shared__ __align__(16) uint32_t rs[RND ? TR : 1][RND ? kXW : 4];
  __shared__ uint32_t oc[kTC][OW];
  __shared__ uint8_t os[FP4 ? kTC : 1][NB];
  __shared__ uint32_t amx[FP4 ? NB : 1][FP4 ? 32 : 1][2];
  __shared__ float oe[ERR ? kTC : 1][NB];
  // FMT 3 (E5M2): p.scale is the amax; MXFP4: read only for the non-finite check
  const float g = FMT == 3 ? e5m2_tensor_scale(*p.scale) : *p.scale;
  if (blockIdx.x == 0 && threadIdx.x == 0 && p.g_out)
    *p.g_out = (FMT == 2 && !isnan(g)) ? 1.0f : g;
  if (isnan(g)) return;
  const float six_g = __fmul_rn(6.0f, g);
  const float inv8 = __frcp_rn(g);
  __shared__ float2 s_tab[FMT == 1 ? kScaleCodes : 1];
  if (FMT == 1) fill_scale_table(s_tab, g);   // ordered before its reads by the staging barrier below
  // a one-dimensional grid (a second dimension would cap the output rows at 65535 tiles): tile
  // (bx, by), bx along the output contraction fastest
  const uint32_t gx = (uint32_t)((p.ocp + TR - 1) / TR);
  const uint32_t by = blockIdx.x / gx, bx = blockIdx.x - by * gx;
  const int64_t r0 = (int64_t)bx * TR;    // source row = output contraction index
  const int64_t c0 = (int64_t)by * kTC;   // source col = output row
  const int t = threadIdx.x;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int row = (t >> 3) + (TR / 4) * j, ch = t & 7;   // NT / 8 rows per pass
    const int64_t gr = r0 + row, gc = c0 + ch * 8;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    const bool in = gr < p.rows && gc < p.cols;
    if (in) v = __ldg(reinterpret_cast<const uint4*>(p.x + gr * p.cols + gc));
    *reinterpret_cast<uint4*>(&xs[row][ch * 4]) = v;
    if (RND == 1) {
      U4 w = make_zero_u4();
      if (in) w = sr_words_rk(((uint64_t)(gr * p.cols + gc) + p.index_base) >> 3, p.stream_id, p.rk);
      *reinterpret_cast<uint4*>(&rs[row][ch * 4]) = make_uint4(w.x, w.y, w.z, w.w);
    }
  }
  __syncthreads();
  {
    const int cp = t & 31, b = t >> 5;
    float v0[16], v1[16];
    uint32_t m01 = 0;   // the two columns' maxima of |bf16| bits, as the word's two 16-bit halves
    // random words of rows b*16..b*16+15: column 2cp's bits in the low half, 2cp+1's in the high half
    uint32_t rw[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t w = xs[b * 16 + i][cp];
      v0[i] = __uint_as_float(w << 16);
      v1[i] = __uint_as_float(w & 0xffff0000u);
      m01 = __vmaxu2(m01, w & 0x7fff7fffu);
      rw[i] = RND == 1 ? rs[b * 16 + i][cp] : 0u;
    }
    uint32_t m0 = m01 & 0xffffu, m1 = m01 >> 16;
    const WordHalfBits<false> u0{rw};
    const WordHalfBits<true> u1{rw};
    if (FMT == 2) {
      amx[b][cp][0] = m0;
      amx[b][cp][1] = m1;
      __syncthreads();
      m0 = max(m0, amx[b ^ 1][cp][0]);
      m1 = max(m1, amx[b ^ 1][cp][1]);
      const BlockScale s0 = mxfp4_block_scale(m0), s1 = mxfp4_block_scale(m1);
      const uint2 e0 = nvfp4_encode16<RND>(v0, s0, u0), e1 = nvfp4_encode16<RND>(v1, s1, u1);
      oc[2 * cp][2 * b] = e0.x; oc[2 * cp][2 * b + 1] = e0.y;
      oc[2 * cp + 1][2 * b] = e1.x; oc[2 * cp + 1][2 * b + 1] = e1.y;
      if (!(b & 1)) {
        os[2 * cp][b >> 1] = (uint8_t)s0.s;
        os[2 * cp + 1][b >> 1] = (uint8_t)s1.s;
      }
    } else if (FMT == 1) {
      if (p.group > 1) {   // longer blocks: the maxima of the tile's p.group-block groups (uniform branch)
        amx[b][cp][0] = m0;
        amx[b][cp][1] = m1;
        __syncthreads();
        const int b0 = b & ~(p.group - 1);
        for (int j = 0; j < p.group; ++j) {
          m0 = max(m0, amx[b0 + j][cp][0]);
          m1 = max(m1, amx[b0 + j][cp][1]);
        }
      }
      const BlockScale s0 = nvfp4_block_scale_tab(m0, six_g, s_tab), s1 = nvfp4_block_scale_tab(m1, six_g, s_tab);
      const uint2 e0 = nvfp4_encode16<RND>(v0, s0, u0), e1 = nvfp4_encode16<RND>(v1, s1, u1);
      oc[2 * cp][2 * b] = e0.x; oc[2 * cp][2 * b + 1] = e0.y;
      oc[2 * cp + 1][2 * b] = e1.x; oc[2 * cp + 1][2 * b + 1] = e1.y;
      os[2 * cp][b] = (uint8_t)s0.s;
      os[2 * cp + 1][b] = (uint8_t)s1.s;
      if (ERR) {
        oe[2 * cp][b] = nvfp4_block_err(v0, e0, s0.p);
        oe[2 * cp + 1][b] = nvfp4_block_err(v1, e1, s1.p);
      }
    } else {
      const uint4 e0 = fp8_encode16<RND, FMT == 3>(v0, inv8, u0), e1 = fp8_encode16<RND, FMT == 3>(v1, inv8, u1);
      oc[2 * cp][4 * b] = e0.x; oc[2 * cp][4 * b + 1] = e0.y; oc[2 * cp][4 * b + 2] = e0.z; oc[2 * cp][4 * b + 3] = e0.w;
      oc[2 * cp + 1][4 * b] = e1.x; oc[2 * cp + 1][4 * b + 1] = e1.y;
      oc[2 * cp + 1][4 * b + 2] = e1.z; oc[2 * cp + 1][4 * b + 3] = e1.w;
    }
  }
  __syncthreads();
  // codes: output rows c0.., contraction r0..r0+127 (OB bytes per row)
  constexpr int BPB = FP4 ? 8 : 16;   // bytes per 16-element block
  if (LAYOUT == 0) {
    // row pitch of the row-major layout is only block-aligned: one store per block
    for (int idx = t; idx < kTC * NB; idx += NT) {
      const int row = idx / NB, b = idx % NB;
      const int64_t orow = c0 + row;
      if (orow >= p.out_rows || r0 + 16 * b >= p.out_cols) continue;
      uint8_t* dst = p.codes + orow * (p.out_cols * BPB / 16) + (r0 + 16 * b) * BPB / 16;
      if (FP4) *reinterpret_cast<uint2*>(dst) = make_uint2(oc[row][2 * b], oc[row][2 * b + 1]);
      else *reinterpret_cast<uint4*>(dst) = make_uint4(oc[row][4 * b], oc[row][4 * b + 1], oc[row][4 * b + 2],
                                                       oc[row][4 * b + 3]);
    }
  } else {
    constexpr int CH = OB / 16;              // 16-byte chunks per tile row
    for (int idx = t; idx < kTC * CH; idx += NT) {
      const int row = idx / CH, ch = idx % CH;
      const int64_t orow = c0 + row;
      if (orow >= p.orp) continue;
      *reinterpret_cast<uint4*>(p.codes + orow * (p.ocp * BPB / 16) + r0 * BPB / 16 + ch * 16) =
          make_uint4(oc[row][4 * ch], oc[row][4 * ch + 1], oc[row][4 * ch + 2], oc[row][4 * ch + 3]);
    }
  }
  if (FMT == 2 && t < kTC) {
    // NB/2 E8M0 bytes per output row: the tile's TR contraction elements
    const int64_t orow = c0 + t;
    const int64_t kb0 = r0 >> 5;
    if (LAYOUT == 0) {
      if (orow < p.out_rows)
        for (int b = 0; b < NB / 2 && (kb0 + b) * 32 < p.out_cols; ++b)
          p.scales[orow * (p.out_cols >> 5) + kb0 + b] = os[t][b];
    } else if (orow < p.orp) {
      if constexpr (NB == 8) {
        const uint32_t v = (uint32_t)os[t][0] | ((uint32_t)os[t][1] << 8) | ((uint32_t)os[t][2] << 16) |
                           ((uint32_t)os[t][3] << 24);
        *reinterpret_cast<uint32_t*>(p.scales + mma_scale_offset_mx(orow, kb0, p.ocp)) = v;
      } else {   // two blocks: a byte pair at an even byte of the chunk word
        const uint16_t v = (uint16_t)(os[t][0] | (os[t][1] << 8));
        *reinterpret_cast<uint16_t*>(p.scales + mma_scale_offset_mx(orow, kb0, p.ocp)) = v;
      }
    }
  }
  if (FMT == 1 && t < kTC) {
    const int64_t orow = c0 + t;
    const int64_t kb0 = r0 >> 4;
    if (LAYOUT == 0) {
      if (orow < p.out_rows)
        for (int b = 0; b < NB && (kb0 + b) * 16 < p.out_cols; ++b)
          p.scales[orow * (p.out_cols >> 4) + kb0 + b] = os[t][b];
    } else if (orow < p.orp) {
#pragma unroll
      for (int h = 0; h < NB / 4; ++h) {
        const uint32_t v = (uint32_t)os[t][4 * h] | ((uint32_t)os[t][4 * h + 1] << 8) |
                           ((uint32_t)os[t][4 * h + 2] << 16) | ((uint32_t)os[t][4 * h + 3] << 24);
        *reinterpret_cast<uint32_t*>(p.scales + mma_scale_offset(orow, kb0 + 4 * h, p.ocp)) = v;
      }
    }
    if (ERR && p.block_err && orow < p.out_rows)
      for (int b = 0; b < NB && (kb0 + b) * 16 < p.out_cols; ++b)
        p.block_err[orow * (p.out_cols >> 4) + kb0 + b] = oe[t][b];
  }
}

// ------------------------------------------------------------------ a8: statistics kernel
template <int RND, bool BLK>
__global__ void __launch_bounds__(256) stats_kernel(StatsParams p) {
  pdl_enter();
  const float amax = p.scales3[0], g = p.scales3[1], s8 = p.scales3[2];
  if (isnan(amax)) {
    stats_nan(p.raw_out);
    return;
  }
  const float six_g = __fmul_rn(6.0f, g);
  const float inv8 = __frcp_rn(s8);
  const bool special8 = !(inv8 < kInf);
  __shared__ float2 s_tab[kScaleCodes];
  fill_scale_table(s_tab, g);
  __syncthreads();
  const uint32_t bpr = (uint32_t)(p.cols >> 4);
  const uint32_t spr = (bpr + 31) >> 5;
  const uint32_t total = (uint32_t)p.rows * spr;
  const uint32_t lane = threadIdx.x & 31;
  const uint32_t wstride = gridDim.x * (blockDim.x >> 5);
  StatsAcc acc;
  acc.init();
  // segment -> (row, segment in row), stepped without a division per iteration
  const uint32_t seg0 = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const uint32_t wq = wstride / spr, wr = wstride - wq * spr;
  uint32_t nr = seg0 / spr, nsr = seg0 - nr * spr;
  // software pipeline: the next segment's 32 bytes are requested before this one is evaluated
  uint4 na = make_uint4(0u, 0u, 0u, 0u), nb = na;
  auto fetch = [&](uint32_t rr, uint32_t ss) {
    const uint32_t kk = ss * 32 + lane;
    if (kk < bpr) {
      const uint4* src = reinterpret_cast<const uint4*>(p.x + (int64_t)rr * p.cols + (int64_t)kk * 16);
      na = __ldg(src);
      nb = __ldg(src + 1);
    }
  };
  if (seg0 < total) fetch(nr, nsr);
  for (uint32_t seg = seg0; seg < total; seg += wstride) {
    const uint32_t r = nr, sr = nsr;
    const uint4 a = na, b = nb;
    nr += wq;
    nsr += wr;
    if (nsr >= spr) { nsr -= spr; ++nr; }
    if (seg + wstride < total) fetch(nr, nsr);
    const uint32_t kb = sr * 32 + lane;
    if (kb >= bpr) continue;
    const int64_t e0 = (int64_t)r * p.cols + (int64_t)kb * 16;
    float v[16];
    unpack16(a, b, v);
    uint32_t u[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    if (RND == 1) sr_bits16_rk(e0, p.stream_id, p.rk, u);
    const BlockScale bs = nvfp4_block_scale_tab(amax16_bits(a, b), six_g, s_tab);
    uint4 unused;
    float be4 = 0.f, be8 = 0.f;
    stats_block16<-1, RND, BLK>(v, bs, u, s8, inv8, special8, unused, acc, &be4, &be8);
    if (BLK) {
      const int64_t bi = (int64_t)r * bpr + kb;
      if (p.block_err4) p.block_err4[bi] = be4;
      if (p.block_err8) p.block_err8[bi] = be8;
    }
  }
  float sums[5];
  acc.finish(s8, special8, sums);
  stats_finish(sums, p.partials, p.counter, p.raw_out, amax, p.rows * p.cols);
}

// ------------------------------------------------------------------ host-side launchers
// CTAs of 256 threads one SM holds at once for a kernel (occupancy query, cached per kernel and device).
static int resident_ctas(const void* fn) {
  static std::mutex mu;
  static std::vector<std::pair<std::pair<const void*, int>, int>> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  for (const auto& e : cache)
    if (e.first.first == fn && e.first.second == dev) return e.second;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, 256, 0) != cudaSuccess || n < 1) n = 1;
  cache.emplace_back(std::make_pair(fn, dev), n);
  return n;
}

cudaError_t ensure_max_dynamic_smem(const void* fn, int bytes) {
  static std::mutex mu;
  static std::vector<std::pair<const void*, int>> done;   // (kernel, device) pairs already raised
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  for (const auto& d : done)
    if (d.first == fn && d.second == dev) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.emplace_back(fn, dev);
  return e;
}

// A grid-stride kernel: as many CTAs as the work asks for, but no more than two waves of resident
// CTAs, and no more than max_ctas (the partial-result slots).  Every CTA has the same share of the
// work.  Alone on the GPU the two waves run one after the other at the speed of one; beside another
// kernel that holds part of every SM (a GEMM's CTA) only some CTAs are resident at a time, and
// shares half the size let the CTAs that start late finish sooner (measured on the 7B step: one wave
// 2337, two 2361, four 2327 TFLOP/s).
template <class P>
static void launch_persistent(void (*kernel)(P), int64_t want, int max_ctas, int num_sms, cudaStream_t st,
                              const P& p) {
  int64_t g = want < 1 ? 1 : want;
  const int64_t wave = (int64_t)resident_ctas(reinterpret_cast<const void*>(kernel)) * num_sms;
  if (g > 2 * wave) g = 2 * wave;
  if (g > max_ctas) g = max_ctas;
  launch_pdl(kernel, (unsigned)g, 256u, 0u, 1u, st, p);
}

static int fill_grid(int64_t work_items, int per_cta, int max_ctas) {
  int64_t g = (work_items + per_cta - 1) / per_cta;
  if (g < 1) g = 1;
  if (g > max_ctas) g = max_ctas;
  return (int)g;
}

cudaError_t launch_scales_multi(ScalesMulti m, uint32_t* partials, uint32_t* counters, uint32_t* status,
                                int num_sms, cudaStream_t st) {
  // CTAs in proportion to each tensor's size, at least one each, within the partial slots
  int64_t total = 0;
  for (int t = 0; t < m.count; ++t) total += m.n[t];
  // rounding each tensor's share up adds at most one CTA a tensor: stay within the partial slots
  const int64_t want = fill_grid(total >> 3, 256 * 4, std::min(4 * num_sms, kMaxPartials - kMaxMultiScales));
  int c = 0;
  for (int t = 0; t < m.count; ++t) {
    m.cta0[t] = c;
    int64_t k = total > 0 ? (want * m.n[t] + total - 1) / total : 1;
    const int64_t need = ((m.n[t] >> 3) + 1023) / 1024;   // no more CTAs than 4 loads per thread need
    if (k > need) k = need;
    if (k < 1) k = 1;
    c += (int)k;
  }
  m.cta0[m.count] = c;
  return launch_pdl(scales_multi_kernel, (unsigned)c, 256u, 0u, 1u, st, m, partials, counters, status);
}

cudaError_t launch_scales(const uint16_t* x, int64_t n, uint32_t* partials, uint32_t* counter, float* out3,
                          uint32_t* status, int num_sms, cudaStream_t st) {
  const int grid = fill_grid(n >> 3, 256 * 4, std::min(4 * num_sms, kMaxPartials));
  return launch_pdl(scales_kernel, (unsigned)grid, 256u, 0u, 1u, st, x, n, partials, counter, out3, status);
}

// a row-block quantization (persistent: want CTAs at most, cap partial slots)
#define SNIP_ROWS(...) launch_persistent(quant_rows_kernel<__VA_ARGS__>, want, cap, num_sms, st, p)

template <int FMT, int LY, int RN, bool ER, int TR>
static void launch_cols(const QuantParams& p, cudaStream_t st) {
  const int64_t tiles = ((p.ocp + TR - 1) / TR) * ((p.orp + kTC - 1) / kTC);   // checked < 2^31 by the API
  launch_pdl(quant_cols_kernel<FMT, LY, RN, ER, TR>, (unsigned)tiles, (unsigned)(2 * TR), 0u, 1u, st, p);
}

template <int FMT>
static void launch_quant_fmt(const QuantParams& p, int orient, int layout, int rnd, bool err, int num_sms,
                             cudaStream_t st) {
  if (orient == 0) {
    const int64_t segs = p.orp * (((p.ocp >> 4) + 31) >> 5);
    const bool stats = p.raw_out != nullptr;
    // one warp per 32-block segment at a time; with statistics, one partial slot per CTA
    const int64_t want = (segs + 7) / 8;
    const int cap = stats ? kMaxPartials : 16 * num_sms;
    if constexpr (FMT == 1) {
      if (stats && p.group > 1) {   // longer NVFP4 blocks with fused statistics (no block errors)
        if (layout == 0) {
          if (rnd == 0) SNIP_ROWS(1, 0, 0, false, true, true);
          else SNIP_ROWS(1, 0, 1, false, true, true);
        } else {
          if (rnd == 0) SNIP_ROWS(1, 1, 0, false, true, true);
          else SNIP_ROWS(1, 1, 1, false, true, true);
        }
        return;
      }
    }
#define SNIP_L(LY, RN, ER, SS) SNIP_ROWS(FMT, LY, RN, ER, SS)
#define SNIP_LS(LY, RN, ER) do { if (stats) SNIP_L(LY, RN, ER, true); else SNIP_L(LY, RN, ER, false); } while (0)
    if (layout == 0) {
      if (rnd == 0) { if (err) SNIP_LS(0, 0, true); else SNIP_LS(0, 0, false); }
      else { if (err) SNIP_LS(0, 1, true); else SNIP_LS(0, 1, false); }
    } else {
      if (rnd == 0) { if (err) SNIP_LS(1, 0, true); else SNIP_LS(1, 0, false); }
      else { if (err) SNIP_LS(1, 1, true); else SNIP_LS(1, 1, false); }
    }
#undef SNIP_LS
#undef SNIP_L
  } else {
    // source rows tile the output contraction, source cols the output rows; 64-row tiles, except
    // for blocks of 128 rows
    if constexpr (FMT == 1) {
      if (p.group >= 8) {
#define SNIP_L(LY, RN, ER) launch_cols<FMT, LY, RN, ER, 128>(p, st)
        if (layout == 0) {
          if (rnd == 0) { if (err) SNIP_L(0, 0, true); else SNIP_L(0, 0, false); }
          else { if (err) SNIP_L(0, 1, true); else SNIP_L(0, 1, false); }
        } else {
          if (rnd == 0) { if (err) SNIP_L(1, 0, true); else SNIP_L(1, 0, false); }
          else { if (err) SNIP_L(1, 1, true); else SNIP_L(1, 1, false); }
        }
#undef SNIP_L
        return;
      }
    }
#define SNIP_L(LY, RN, ER) launch_cols<FMT, LY, RN, ER, 64>(p, st)
    if (layout == 0) {
      if (rnd == 0) { if (err) SNIP_L(0, 0, true); else SNIP_L(0, 0, false); }
      else { if (err) SNIP_L(0, 1, true); else SNIP_L(0, 1, false); }
    } else {
      if (rnd == 0) { if (err) SNIP_L(1, 0, true); else SNIP_L(1, 0, false); }
      else { if (err) SNIP_L(1, 1, true); else SNIP_L(1, 1, false); }
    }
#undef SNIP_L
  }
}

// MXFP4: no block errors; row blocks with or without fused statistics.
static void launch_quant_mx(const QuantParams& p, int orient, int layout, int rnd, int num_sms, cudaStream_t st) {
  if (orient == 0) {
    const int64_t segs = p.orp * (((p.ocp >> 4) + 31) >> 5);
    const bool stats = p.raw_out != nullptr;
    const int64_t want = (segs + 7) / 8;
    const int cap = stats ? kMaxPartials : 16 * num_sms;
    if (stats) {
      if (layout == 0) {
        if (rnd == 0) SNIP_ROWS(2, 0, 0, false, true);
        else SNIP_ROWS(2, 0, 1, false, true);
      } else {
        if (rnd == 0) SNIP_ROWS(2, 1, 0, false, true);
        else SNIP_ROWS(2, 1, 1, false, true);
      }
    } else if (layout == 0) {
      if (rnd == 0) SNIP_ROWS(2, 0, 0, false, false);
      else SNIP_ROWS(2, 0, 1, false, false);
    } else {
      if (rnd == 0) SNIP_ROWS(2, 1, 0, false, false);
      else SNIP_ROWS(2, 1, 1, false, false);
    }
  } else {
    if (layout == 0) {
      if (rnd == 0) launch_cols<2, 0, 0, false, 64>(p, st);
      else launch_cols<2, 0, 1, false, 64>(p, st);
    } else {
      if (rnd == 0) launch_cols<2, 1, 0, false, 64>(p, st);
      else launch_cols<2, 1, 1, false, 64>(p, st);
    }
  }
}

// E5M2: no block errors either.
static void launch_quant_e5(const QuantParams& p, int orient, int layout, int rnd, int num_sms, cudaStream_t st) {
  if (orient == 0) {
    const int64_t segs = p.orp * (((p.ocp >> 4) + 31) >> 5);
    const bool stats = p.raw_out != nullptr;
    const int64_t want = (segs + 7) / 8;
    const int cap = stats ? kMaxPartials : 16 * num_sms;
    if (stats) {
      if (layout == 0) {
        if (rnd == 0) SNIP_ROWS(3, 0, 0, false, true);
        else SNIP_ROWS(3, 0, 1, false, true);
      } else {
        if (rnd == 0) SNIP_ROWS(3, 1, 0, false, true);
        else SNIP_ROWS(3, 1, 1, false, true);
      }
    } else if (layout == 0) {
      if (rnd == 0) SNIP_ROWS(3, 0, 0, false, false);
      else SNIP_ROWS(3, 0, 1, false, false);
    } else {
      if (rnd == 0) SNIP_ROWS(3, 1, 0, false, false);
      else SNIP_ROWS(3, 1, 1, false, false);
    }
  } else {
    if (layout == 0) {
      if (rnd == 0) launch_cols<3, 0, 0, false, 64>(p, st);
      else launch_cols<3, 0, 1, false, 64>(p, st);
    } else {
      if (rnd == 0) launch_cols<3, 1, 0, false, 64>(p, st);
      else launch_cols<3, 1, 1, false, 64>(p, st);
    }
  }
}

cudaError_t launch_quant(int fmt, const QuantParams& p, int orient, int layout, int rnd, bool err, int num_sms,
                         cudaStream_t st) {
  if (fmt == 3) launch_quant_e5(p, orient, layout, rnd, num_sms, st);
  else if (fmt == 2) launch_quant_mx(p, orient, layout, rnd, num_sms, st);
  else if (fmt == 1) launch_quant_fmt<1>(p, orient, layout, rnd, err, num_sms, st);
  else launch_quant_fmt<0>(p, orient, layout, rnd, false, num_sms, st);
  return cudaGetLastError();
}

cudaError_t launch_stats(const StatsParams& p, int rnd, int num_sms, cudaStream_t st) {
  const int64_t segs = p.rows * (((p.cols >> 4) + 31) >> 5);
  const int64_t want = (segs + 31) / 32;   // four segments per warp at least
  const bool blk = p.block_err4 || p.block_err8;
#define SNIP_ST(RN, BK) launch_persistent(stats_kernel<RN, BK>, want, kMaxPartials, num_sms, st, p)
  if (rnd == 0) { if (blk) SNIP_ST(0, true); else SNIP_ST(0, false); }
  else { if (blk) SNIP_ST(1, true); else SNIP_ST(1, false); }
#undef SNIP_ST
  return cudaGetLastError();
}

}  // namespace snip
