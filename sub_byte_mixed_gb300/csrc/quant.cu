// quant.cu -- HBM-bound kernels of the quantized linear layer: tensor amax
// (a1), NVFP4 quantization with blocks along columns (a2) or rows (a3), FP8
// E4M3 quantization (a4) and SNIP's statistics pass (a8).
//
// Sources: "FP4 all the way" (Chmiel et al.), summary page, Outline (NVFP4 =
// 16 E2M1 values sharing an E4M3 scale; RTN forward, SR backward; the
// sqrt(3)-times-noise threshold); "SNIP", Abstract and Figure 2 (statistics of
// activations, weights and gradients); "SNIP", Figure 5 (each GEMM operand
// quantized along its own contraction dim).
//
// Design: every kernel streams its input once with 16-byte coalesced loads;
// one thread owns 8 consecutive source elements (one Philox call supplies
// their 8 x 16 random bits) and a lane pair owns one 16-element block, whose
// amax is exchanged with one shuffle.  The transposed (column-block) kernels
// stage a 128 x 64 tile in shared memory so that loads and stores both stay
// coalesced.  The tensor scale comes from a two-stage amax reduction whose
// last CTA publishes one word, so quantizer CTAs read a single value.
#include "snip_kernels.cuh"

namespace snip {

// ------------------------------------------------------------------ amax
// Magnitudes are compared as bf16 bit patterns (sign cleared): for finite
// values the integer order is the float order, and any pattern >= 0x7f80 is
// an infinity or NaN.
__global__ void __launch_bounds__(256) amax_kernel(const uint16_t* __restrict__ x, int64_t n,
                                                   uint32_t* __restrict__ partials,
                                                   uint32_t* __restrict__ counter,
                                                   uint32_t* __restrict__ result_bits,
                                                   float* __restrict__ result_float,
                                                   uint32_t* __restrict__ status) {
  uint32_t m2 = 0;  // two 16-bit lanes of magnitudes (sign bits cleared before the max)
  const int64_t nvec = n >> 3;
  const uint4* xv = reinterpret_cast<const uint4*>(x);
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < nvec; i += 4 * stride) {
    const uint4 a = __ldg(xv + i), b = __ldg(xv + i + stride), c = __ldg(xv + i + 2 * stride),
                d = __ldg(xv + i + 3 * stride);
    m2 = __vmaxu2(m2, __vmaxu2(__vmaxu2(mag_max4(a), mag_max4(b)), __vmaxu2(mag_max4(c), mag_max4(d))));
  }
  for (; i < nvec; i += stride) m2 = __vmaxu2(m2, mag_max4(__ldg(xv + i)));
  // tail (n % 8 elements)
  if (blockIdx.x == 0 && threadIdx.x < (n & 7)) m2 = __vmaxu2(m2, (uint32_t)(x[(nvec << 3) + threadIdx.x] & 0x7fffu));
  uint32_t m = max(m2 & 0xffffu, m2 >> 16);
  m = block_max_u32(m);
  __shared__ bool s_last;
  if (threadIdx.x == 0) {
    partials[blockIdx.x] = m;
    if (m >= 0x7f80u) atomicOr(status, kDevNonFinite);
    __threadfence();
    uint32_t done = atomicAdd(counter, 1u);
    s_last = (done == gridDim.x - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  uint32_t mm = 0;
  for (uint32_t j = threadIdx.x; j < gridDim.x; j += blockDim.x) mm = max(mm, ((volatile uint32_t*)partials)[j]);
  mm = block_max_u32(mm);
  if (threadIdx.x == 0) {
    *result_bits = mm;
    if (result_float) *result_float = mm >= 0x7f80u ? __int_as_float(0x7fc00000) : bf16_bits_to_float(mm);
    *counter = 0;  // ready for the next reduction on this workspace
  }
}

// Tensor scale of an NVFP4 tensor (amax / (6*448), 1 for an all-zero tensor)
// or of an FP8 tensor (amax / 448); NaN when the amax word flags non-finite.
__device__ __forceinline__ float tensor_scale_from_bits(uint32_t mbits, float divisor) {
  if (mbits >= 0x7f80u) return __int_as_float(0x7fc00000);
  float m = bf16_bits_to_float(mbits);
  return m == 0.0f ? 1.0f : __fdiv_rn(m, divisor);
}

__device__ __forceinline__ float load_scale(const QuantParams& p, float divisor) {
  return p.g_in ? *p.g_in : tensor_scale_from_bits(*p.amax_bits, divisor);
}

// Byte offset of the E4M3 scale of (row r, block kb) in the MMA layout.
__device__ __forceinline__ int64_t mma_scale_offset(int64_t r, int64_t kb, int64_t ocp) {
  int64_t chunk = (r >> 7) * (ocp >> 6) + (kb >> 2);
  return chunk * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (kb & 3);
}

// ------------------------------------------------------------------ NVFP4 block encode
// Encodes 8 elements (bf16 bits in w[0..3], element i in half i of w[i/2])
// that are one half of a 16-element block whose partner half sits in the
// lane with index ^1.  Returns the 8 packed codes; *scale gets the block's
// E4M3 code, *err (if ERR) this half's squared dequantization error.
template <int RND, bool ERR>
__device__ __forceinline__ uint32_t nvfp4_encode_half(const uint32_t (&w)[4], float g, float six_g,
                                                      const U4& rbits, uint32_t* scale, float* err) {
  uint32_t m2 = __vmaxu2(__vmaxu2(w[0] & 0x7fff7fffu, w[1] & 0x7fff7fffu),
                         __vmaxu2(w[2] & 0x7fff7fffu, w[3] & 0x7fff7fffu));
  uint32_t mh = max(m2 & 0xffffu, m2 >> 16);
  mh = max(mh, __shfl_xor_sync(0xffffffffu, mh, 1));
  const float ab = bf16_bits_to_float(mh);
  const uint32_t s = e4m3_rn_sat(__fdiv_rn(ab, six_g));
  const float p = __fmul_rn(e4m3_decode_pos(s), g);
  const float inv = __frcp_rn(p);
  uint32_t packed = 0;
  float e = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t h = (i & 1) ? (w[i >> 1] >> 16) : (w[i >> 1] & 0xffffu);
    const float ax = bf16_bits_to_float(h & 0x7fffu);
    const float y = __fmul_rn(ax, inv);
    uint32_t mag;
    if (RND == 0) mag = e2m1_rn(y);
    else mag = e2m1_sr(y, sr_half(rbits, i));
    if (p == 0.0f || ax == 0.0f) mag = 0u;
    packed |= (((h >> 12) & 8u) | mag) << (4 * i);
    if (ERR) {
      const float d = __fsub_rn(__fmul_rn(e2m1_value(mag), p), ax);
      e = __fadd_rn(e, __fmul_rn(d, d));
    }
  }
  *scale = s;
  if (ERR) *err = e;
  return packed;
}

// ------------------------------------------------------------------ a2: NVFP4, blocks along columns
template <int LAYOUT, int RND, bool ERR>
__global__ void __launch_bounds__(256) quant_nvfp4_rows_kernel(QuantParams p) {
  const float g = load_scale(p, 2688.0f);
  if (isnan(g)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) *p.g_out = g;
    return;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) *p.g_out = g;
  const float six_g = __fmul_rn(6.0f, g);
  const int64_t hb_row = p.ocp >> 3;                  // half-blocks per output row
  const int64_t total = p.orp * hb_row;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t base = (int64_t)blockIdx.x * blockDim.x; base < total; base += stride) {
    const int64_t hb = base + threadIdx.x;
    const int64_t r = hb / hb_row, c8 = hb - r * hb_row;
    const bool valid = hb < total && r < p.out_rows && (c8 << 3) < p.out_cols;
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    if (valid) {
      uint4 v = __ldg(reinterpret_cast<const uint4*>(p.x + r * p.cols + (c8 << 3)));
      w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    }
    U4 rb{0u, 0u, 0u, 0u};
    if (RND == 1 && valid) rb = sr_words((uint64_t)((r * p.cols + (c8 << 3)) >> 3), p.seed, p.stream_id);
    uint32_t scale;
    float err = 0.0f;
    const uint32_t packed = nvfp4_encode_half<RND, ERR>(w, g, six_g, rb, &scale, &err);
    if (ERR) err = __fadd_rn(err, __shfl_xor_sync(0xffffffffu, err, 1));
    if (hb >= total) continue;
    if (LAYOUT == 0) {
      if (!valid) continue;
      *reinterpret_cast<uint32_t*>(p.codes + r * (p.out_cols >> 1) + (c8 << 2)) = packed;
      if ((c8 & 1) == 0) {
        p.scales[r * (p.out_cols >> 4) + (c8 >> 1)] = (uint8_t)scale;
        if (ERR && p.block_err) p.block_err[r * (p.out_cols >> 4) + (c8 >> 1)] = err;
      }
    } else {
      *reinterpret_cast<uint32_t*>(p.codes + r * (p.ocp >> 1) + (c8 << 2)) = packed;
      if ((c8 & 1) == 0) {
        p.scales[mma_scale_offset(r, c8 >> 1, p.ocp)] = (uint8_t)scale;
        if (ERR && p.block_err && valid) p.block_err[r * (p.out_cols >> 4) + (c8 >> 1)] = err;
      }
    }
  }
}

// ------------------------------------------------------------------ a3: NVFP4, blocks along rows (transposed output)
// Tile: 128 source rows (8 blocks of the output contraction) x 64 source
// columns (64 output rows).
constexpr int kTR = 128, kTC = 64, kXP = kTC + 8;  // bf16 pitch (halfwords)

template <int LAYOUT, int RND, bool ERR>
__global__ void __launch_bounds__(256) quant_nvfp4_cols_kernel(QuantParams p) {
  __shared__ __align__(16) uint16_t xs[kTR][kXP];
  __shared__ __align__(16) uint16_t rs[RND ? kTR : 1][RND ? kTC : 8];
  __shared__ __align__(16) uint8_t oc[kTC][kTR / 2 + 16];
  __shared__ uint8_t os[kTC][8];
  __shared__ float oe[ERR ? kTC : 1][8];
  const float g = load_scale(p, 2688.0f);
  if (isnan(g)) {
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *p.g_out = g;
    return;
  }
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *p.g_out = g;
  const float six_g = __fmul_rn(6.0f, g);
  const int64_t r0 = (int64_t)blockIdx.x * kTR;   // source row = output contraction index
  const int64_t c0 = (int64_t)blockIdx.y * kTC;   // source col = output row
  const int t = threadIdx.x;
  // load 128 x 64 bf16 (zero outside the source tensor) and the random bits
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int row = (t >> 3) + 32 * j, ch = t & 7;
    const int64_t gr = r0 + row, gc = c0 + ch * 8;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (gr < p.rows && gc < p.cols) v = __ldg(reinterpret_cast<const uint4*>(p.x + gr * p.cols + gc));
    *reinterpret_cast<uint4*>(&xs[row][ch * 8]) = v;
    if (RND == 1) {
      U4 w = sr_words((uint64_t)((gr * p.cols + gc) >> 3), p.seed, p.stream_id);
      *reinterpret_cast<uint4*>(&rs[row][ch * 8]) = make_uint4(w.x, w.y, w.z, w.w);
    }
  }
  __syncthreads();
  // encode: thread -> (output row c, block b); a warp covers 32 consecutive c
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int c = t & 63, b = (t >> 6) + 4 * j;
    uint32_t mh = 0;
    uint32_t hv[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      hv[i] = xs[b * 16 + i][c];
      mh = max(mh, hv[i] & 0x7fffu);
    }
    const float ab = bf16_bits_to_float(mh);
    const uint32_t s = e4m3_rn_sat(__fdiv_rn(ab, six_g));
    const float pq = __fmul_rn(e4m3_decode_pos(s), g);
    const float inv = __frcp_rn(pq);
    uint32_t lo = 0, hi = 0;
    float e = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float ax = bf16_bits_to_float(hv[i] & 0x7fffu);
      const float y = __fmul_rn(ax, inv);
      uint32_t mag;
      if (RND == 0) mag = e2m1_rn(y);
      else mag = e2m1_sr(y, rs[b * 16 + i][c]);
      if (pq == 0.0f || ax == 0.0f) mag = 0u;
      const uint32_t code = ((hv[i] >> 12) & 8u) | mag;
      if (i < 8) lo |= code << (4 * i);
      else hi |= code << (4 * (i - 8));
      if (ERR) {
        const float d = __fsub_rn(__fmul_rn(e2m1_value(mag), pq), ax);
        e = __fadd_rn(e, __fmul_rn(d, d));
      }
    }
    *reinterpret_cast<uint2*>(&oc[c][b * 8]) = make_uint2(lo, hi);
    os[c][b] = (uint8_t)s;
    if (ERR) oe[c][b] = e;
  }
  __syncthreads();
  // store codes: 64 output rows x 64 bytes
  if (LAYOUT == 0) {
    // row pitch out_cols/2 is only a multiple of 8 bytes: one 8-byte store per block
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int idx = t + 256 * j, row = idx >> 3, b = idx & 7;
      const int64_t orow = c0 + row;
      if (orow < p.out_rows && r0 + 16 * b < p.out_cols)
        *reinterpret_cast<uint2*>(p.codes + orow * (p.out_cols >> 1) + (r0 >> 1) + 8 * b) =
            *reinterpret_cast<const uint2*>(&oc[row][8 * b]);
    }
  } else {
    const int row = t >> 2, ch = t & 3;
    const int64_t orow = c0 + row;
    if (orow < p.orp)
      *reinterpret_cast<uint4*>(p.codes + orow * (p.ocp >> 1) + (r0 >> 1) + ch * 16) =
          *reinterpret_cast<const uint4*>(&oc[row][ch * 16]);
  }
  if (t < kTC) {
    const int64_t orow = c0 + t;
    const int64_t kb0 = r0 >> 4;
    if (LAYOUT == 0) {
      if (orow < p.out_rows) {
        for (int b = 0; b < 8 && (kb0 + b) * 16 < p.out_cols; ++b) {
          p.scales[orow * (p.out_cols >> 4) + kb0 + b] = os[t][b];
          if (ERR && p.block_err) p.block_err[orow * (p.out_cols >> 4) + kb0 + b] = oe[t][b];
        }
      }
    } else if (orow < p.orp) {
      for (int h = 0; h < 2; ++h) {
        if ((kb0 + 4 * h) * 16 >= p.ocp) break;
        const uint32_t v = (uint32_t)os[t][4 * h] | ((uint32_t)os[t][4 * h + 1] << 8) |
                           ((uint32_t)os[t][4 * h + 2] << 16) | ((uint32_t)os[t][4 * h + 3] << 24);
        *reinterpret_cast<uint32_t*>(p.scales + mma_scale_offset(orow, kb0 + 4 * h, p.ocp)) = v;
      }
      if (ERR && p.block_err && orow < p.out_rows)
        for (int b = 0; b < 8 && (kb0 + b) * 16 < p.out_cols; ++b)
          p.block_err[orow * (p.out_cols >> 4) + kb0 + b] = oe[t][b];
    }
  }
}

// ------------------------------------------------------------------ a4: FP8 E4M3 with a tensor scale
template <int RND>
__device__ __forceinline__ uint32_t fp8_encode(uint32_t h, float inv, uint32_t u16) {
  const float ax = bf16_bits_to_float(h & 0x7fffu);
  uint32_t mag;
  if (RND == 0) mag = e4m3_rn_sat(__fmul_rn(ax, inv));
  else mag = e4m3_sr(__fmul_rn(ax, inv), u16);
  if (ax == 0.0f) mag = 0u;
  return ((h >> 8) & 0x80u) | mag;
}

template <int LAYOUT, int RND>
__global__ void __launch_bounds__(256) quant_fp8_rows_kernel(QuantParams p) {
  const float s = load_scale(p, 448.0f);
  if (blockIdx.x == 0 && threadIdx.x == 0) *p.g_out = s;
  if (isnan(s)) return;
  const float inv = __frcp_rn(s);
  const int64_t hb_row = p.ocp >> 3;
  const int64_t total = p.orp * hb_row;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t hb = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; hb < total; hb += stride) {
    const int64_t r = hb / hb_row, c8 = hb - r * hb_row;
    const bool valid = r < p.out_rows && (c8 << 3) < p.out_cols;
    if (LAYOUT == 0 && !valid) continue;
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    if (valid) {
      uint4 v = __ldg(reinterpret_cast<const uint4*>(p.x + r * p.cols + (c8 << 3)));
      w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    }
    U4 rb{0u, 0u, 0u, 0u};
    if (RND == 1 && valid) rb = sr_words((uint64_t)((r * p.cols + (c8 << 3)) >> 3), p.seed, p.stream_id);
    uint32_t o[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t h = (i & 1) ? (w[i >> 1] >> 16) : (w[i >> 1] & 0xffffu);
      o[i >> 2] |= fp8_encode<RND>(h, inv, RND ? sr_half(rb, i) : 0u) << (8 * (i & 3));
    }
    const int64_t pitch = LAYOUT == 0 ? p.out_cols : p.ocp;
    *reinterpret_cast<uint2*>(p.codes + r * pitch + (c8 << 3)) = make_uint2(o[0], o[1]);
  }
}

template <int LAYOUT, int RND>
__global__ void __launch_bounds__(256) quant_fp8_cols_kernel(QuantParams p) {
  __shared__ __align__(16) uint16_t xs[kTR][kXP];
  __shared__ __align__(16) uint16_t rs[RND ? kTR : 1][RND ? kTC : 8];
  __shared__ __align__(16) uint8_t oc[kTC][kTR + 16];
  const float s = load_scale(p, 448.0f);
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *p.g_out = s;
  if (isnan(s)) return;
  const float inv = __frcp_rn(s);
  const int64_t r0 = (int64_t)blockIdx.x * kTR, c0 = (int64_t)blockIdx.y * kTC;
  const int t = threadIdx.x;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int row = (t >> 3) + 32 * j, ch = t & 7;
    const int64_t gr = r0 + row, gc = c0 + ch * 8;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (gr < p.rows && gc < p.cols) v = __ldg(reinterpret_cast<const uint4*>(p.x + gr * p.cols + gc));
    *reinterpret_cast<uint4*>(&xs[row][ch * 8]) = v;
    if (RND == 1) {
      U4 w = sr_words((uint64_t)((gr * p.cols + gc) >> 3), p.seed, p.stream_id);
      *reinterpret_cast<uint4*>(&rs[row][ch * 8]) = make_uint4(w.x, w.y, w.z, w.w);
    }
  }
  __syncthreads();
  // thread -> (output row c, 16 consecutive contraction elements b*16..b*16+15)
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int c = t & 63, b = (t >> 6) + 4 * j;
    uint32_t o[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t h = xs[b * 16 + i][c];
      o[i >> 2] |= fp8_encode<RND>(h, inv, RND ? (uint32_t)rs[b * 16 + i][c] : 0u) << (8 * (i & 3));
    }
    *reinterpret_cast<uint4*>(&oc[c][b * 16]) = make_uint4(o[0], o[1], o[2], o[3]);
  }
  __syncthreads();
  // store: 64 output rows x 128 bytes
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int row = (t >> 3) + 32 * j, ch = t & 7;
    const int64_t orow = c0 + row;
    const uint4 v = *reinterpret_cast<const uint4*>(&oc[row][ch * 16]);
    if (LAYOUT == 0) {
      if (orow < p.out_rows && r0 + ch * 16 < p.out_cols)
        *reinterpret_cast<uint4*>(p.codes + orow * p.out_cols + r0 + ch * 16) = v;
    } else if (orow < p.orp && r0 + ch * 16 < p.ocp) {
      *reinterpret_cast<uint4*>(p.codes + orow * p.ocp + r0 + ch * 16) = v;
    }
  }
}

// ------------------------------------------------------------------ a8: statistics
// One pass over the tensor: ||A||^2, the squared errors of NVFP4 and FP8
// quantization under the tensor's rounding, and the expected SR squared
// error sum (hi-|y|)(|y|-lo) q^2 on both grids.  Per-thread sums are fp32
// (each covers a few hundred elements), per-CTA and final sums fp64.
template <int RND, bool BLK>
__global__ void __launch_bounds__(256) stats_kernel(StatsParams p) {
  const uint32_t mbits = *p.amax_bits;
  if (mbits >= 0x7f80u) {
    if (blockIdx.x == 0 && threadIdx.x == 0)
      for (int k = 0; k < 8; ++k) p.raw_out[k] = __longlong_as_double(0x7ff8000000000000ll);
    return;
  }
  const float g = tensor_scale_from_bits(mbits, 2688.0f);
  const float s8 = tensor_scale_from_bits(mbits, 448.0f);
  const float inv8 = __frcp_rn(s8);
  const float six_g = __fmul_rn(6.0f, g);
  const int64_t hb_row = p.cols >> 3;
  const int64_t total = p.rows * hb_row;
  const int64_t total_w = (total + 31) & ~(int64_t)31;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  float sx2 = 0.f, e4 = 0.f, e8 = 0.f, v4 = 0.f, v8 = 0.f;
  for (int64_t hb = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; hb - (threadIdx.x & 31) < total_w;
       hb += stride) {
    const bool valid = hb < total;
    const int64_t r = valid ? hb / hb_row : 0, c8 = valid ? hb - r * hb_row : 0;
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    U4 rb{0u, 0u, 0u, 0u};
    if (valid) {
      uint4 v = __ldg(reinterpret_cast<const uint4*>(p.x + r * p.cols + (c8 << 3)));
      w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
      if (RND == 1) rb = sr_words((uint64_t)((r * p.cols + (c8 << 3)) >> 3), p.seed, p.stream_id);
    }
    uint32_t m2 = __vmaxu2(__vmaxu2(w[0] & 0x7fff7fffu, w[1] & 0x7fff7fffu),
                           __vmaxu2(w[2] & 0x7fff7fffu, w[3] & 0x7fff7fffu));
    uint32_t mh = max(m2 & 0xffffu, m2 >> 16);
    mh = max(mh, __shfl_xor_sync(0xffffffffu, mh, 1));
    const uint32_t sb = e4m3_rn_sat(__fdiv_rn(bf16_bits_to_float(mh), six_g));
    const float pq = __fmul_rn(e4m3_decode_pos(sb), g);
    const float inv = __frcp_rn(pq);
    const float pq2 = __fmul_rn(pq, pq), s82 = __fmul_rn(s8, s8);
    float be4 = 0.f, be8 = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t h = (i & 1) ? (w[i >> 1] >> 16) : (w[i >> 1] & 0xffffu);
      const float ax = bf16_bits_to_float(h & 0x7fffu);
      const uint32_t u = RND ? sr_half(rb, i) : 0u;
      sx2 = __fadd_rn(sx2, __fmul_rn(ax, ax));
      // NVFP4
      const float y = __fmul_rn(ax, inv);
      uint32_t mag = RND ? e2m1_sr(y, u) : e2m1_rn(y);
      const bool z4 = (pq == 0.0f || ax == 0.0f);
      if (z4) mag = 0u;
      const float d4 = __fsub_rn(__fmul_rn(e2m1_value(mag), pq), ax);
      be4 = __fadd_rn(be4, __fmul_rn(d4, d4));
      if (!z4 && y < 6.0f) {
        const uint32_t lo = (uint32_t)(y >= 0.5f) + (uint32_t)(y >= 1.0f) + (uint32_t)(y >= 1.5f) +
                            (uint32_t)(y >= 2.0f) + (uint32_t)(y >= 3.0f) + (uint32_t)(y >= 4.0f);
        const float vl = e2m1_value(lo), vh = e2m1_value(lo + 1u);
        v4 = __fadd_rn(v4, __fmul_rn(__fmul_rn(__fsub_rn(vh, y), __fsub_rn(y, vl)), pq2));
      }
      // FP8
      const float y8 = __fmul_rn(ax, inv8);
      uint32_t c8c = RND ? e4m3_sr(y8, u) : e4m3_rn_sat(y8);
      if (ax == 0.0f) c8c = 0u;
      const float d8 = __fsub_rn(__fmul_rn(e4m3_decode_pos(c8c), s8), ax);
      be8 = __fadd_rn(be8, __fmul_rn(d8, d8));
      if (ax != 0.0f && y8 < 448.0f) {
        const uint32_t lo8 = e4m3_sr(y8, 0xffffu);   // threshold never met: truncation code
        const float vl = e4m3_decode_pos(lo8), vh = e4m3_decode_pos(lo8 + 1u);
        v8 = __fadd_rn(v8, __fmul_rn(__fmul_rn(__fsub_rn(vh, y8), __fsub_rn(y8, vl)), s82));
      }
    }
    e4 = __fadd_rn(e4, be4);
    e8 = __fadd_rn(e8, be8);
    if (BLK) {
      const float b4 = __fadd_rn(be4, __shfl_xor_sync(0xffffffffu, be4, 1));
      const float b8 = __fadd_rn(be8, __shfl_xor_sync(0xffffffffu, be8, 1));
      if (valid && (c8 & 1) == 0) {
        const int64_t bi = r * (p.cols >> 4) + (c8 >> 1);
        if (p.block_err4) p.block_err4[bi] = b4;
        if (p.block_err8) p.block_err8[bi] = b8;
      }
    }
  }
  double acc[5] = {(double)sx2, (double)e4, (double)e8, (double)v4, (double)v8};
  block_sum_f64<5>(acc);
  __shared__ bool s_last;
  if (threadIdx.x == 0) {
    for (int k = 0; k < 5; ++k) p.partials[(int64_t)blockIdx.x * 5 + k] = acc[k];
    __threadfence();
    s_last = atomicAdd(p.counter, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  double tot[5] = {0, 0, 0, 0, 0};
  for (uint32_t j = threadIdx.x; j < gridDim.x; j += blockDim.x)
    for (int k = 0; k < 5; ++k) tot[k] += ((volatile double*)p.partials)[(int64_t)j * 5 + k];
  block_sum_f64<5>(tot);
  if (threadIdx.x == 0) {
    for (int k = 0; k < 5; ++k) p.raw_out[k] = tot[k];
    p.raw_out[5] = (double)bf16_bits_to_float(mbits);
    p.raw_out[6] = (double)(p.rows * p.cols);
    p.raw_out[7] = 0.0;
    *p.counter = 0;
  }
}

// ------------------------------------------------------------------ host-side launchers
static int fill_grid(int64_t work_items, int per_cta, int max_ctas) {
  int64_t g = (work_items + per_cta - 1) / per_cta;
  if (g < 1) g = 1;
  if (g > max_ctas) g = max_ctas;
  return (int)g;
}

cudaError_t launch_amax(const uint16_t* x, int64_t n, uint32_t* partials, uint32_t* counter, uint32_t* result_bits,
                        float* result_float, uint32_t* status, int num_sms, cudaStream_t st) {
  int grid = fill_grid(n >> 3, 256 * 4, 2 * num_sms);
  amax_kernel<<<grid, 256, 0, st>>>(x, n, partials, counter, result_bits, result_float, status);
  return cudaGetLastError();
}

cudaError_t launch_quant_nvfp4(const QuantParams& p, int orient, int layout, int rnd, bool err, int num_sms,
                               cudaStream_t st) {
  if (orient == 0) {
    int grid = fill_grid(p.orp * (p.ocp >> 3), 256, 8 * num_sms);
#define SNIP_L(LY, RN, ER) quant_nvfp4_rows_kernel<LY, RN, ER><<<grid, 256, 0, st>>>(p)
    if (layout == 0) {
      if (rnd == 0) { if (err) SNIP_L(0, 0, true); else SNIP_L(0, 0, false); }
      else { if (err) SNIP_L(0, 1, true); else SNIP_L(0, 1, false); }
    } else {
      if (rnd == 0) { if (err) SNIP_L(1, 0, true); else SNIP_L(1, 0, false); }
      else { if (err) SNIP_L(1, 1, true); else SNIP_L(1, 1, false); }
    }
#undef SNIP_L
  } else {
    // source rows tile the output contraction, source cols the output rows
    dim3 grid((unsigned)((p.ocp + kTR - 1) / kTR), (unsigned)((p.orp + kTC - 1) / kTC));
#define SNIP_L(LY, RN, ER) quant_nvfp4_cols_kernel<LY, RN, ER><<<grid, 256, 0, st>>>(p)
    if (layout == 0) {
      if (rnd == 0) { if (err) SNIP_L(0, 0, true); else SNIP_L(0, 0, false); }
      else { if (err) SNIP_L(0, 1, true); else SNIP_L(0, 1, false); }
    } else {
      if (rnd == 0) { if (err) SNIP_L(1, 0, true); else SNIP_L(1, 0, false); }
      else { if (err) SNIP_L(1, 1, true); else SNIP_L(1, 1, false); }
    }
#undef SNIP_L
  }
  return cudaGetLastError();
}

cudaError_t launch_quant_fp8(const QuantParams& p, int orient, int layout, int rnd, int num_sms, cudaStream_t st) {
  if (orient == 0) {
    int grid = fill_grid(p.orp * (p.ocp >> 3), 256, 8 * num_sms);
    if (layout == 0) { if (rnd == 0) quant_fp8_rows_kernel<0, 0><<<grid, 256, 0, st>>>(p); else quant_fp8_rows_kernel<0, 1><<<grid, 256, 0, st>>>(p); }
    else { if (rnd == 0) quant_fp8_rows_kernel<1, 0><<<grid, 256, 0, st>>>(p); else quant_fp8_rows_kernel<1, 1><<<grid, 256, 0, st>>>(p); }
  } else {
    dim3 grid((unsigned)((p.ocp + kTR - 1) / kTR), (unsigned)((p.orp + kTC - 1) / kTC));
    if (layout == 0) { if (rnd == 0) quant_fp8_cols_kernel<0, 0><<<grid, 256, 0, st>>>(p); else quant_fp8_cols_kernel<0, 1><<<grid, 256, 0, st>>>(p); }
    else { if (rnd == 0) quant_fp8_cols_kernel<1, 0><<<grid, 256, 0, st>>>(p); else quant_fp8_cols_kernel<1, 1><<<grid, 256, 0, st>>>(p); }
  }
  return cudaGetLastError();
}

cudaError_t launch_stats(const StatsParams& p, int rnd, int num_sms, cudaStream_t st) {
  int grid = fill_grid(p.rows * (p.cols >> 3), 256 * 4, 2 * num_sms);
  const bool blk = p.block_err4 || p.block_err8;
  if (rnd == 0) { if (blk) stats_kernel<0, true><<<grid, 256, 0, st>>>(p); else stats_kernel<0, false><<<grid, 256, 0, st>>>(p); }
  else { if (blk) stats_kernel<1, true><<<grid, 256, 0, st>>>(p); else stats_kernel<1, false><<<grid, 256, 0, st>>>(p); }
  return cudaGetLastError();
}

}  // namespace snip
