// snip_quant.cuh -- the NVFP4 / MXFP4 block helpers shared by the quantizers
// (quant.cu) and the GEMM epilogue that re-quantizes dX (gemm.cu): block
// scales, random bits, the element encoder and the MMA scale layout.
// Internal to the library.
#pragma once
#include <cstdint>

#include "snip_device.cuh"
#include "snip_kernels.cuh"

namespace snip {

constexpr float kInf = __builtin_huge_valf();

// Byte offset of the E4M3 scale of (row r, block kb) in the MMA layout.
__device__ __forceinline__ int64_t mma_scale_offset(int64_t r, int64_t kb, int64_t ocp) {
  const int64_t chunk = (r >> 7) * (ocp >> 6) + (kb >> 2);
  return chunk * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (kb & 3);
}
// MXFP4: the same chunk image with one E8M0 byte per 32-element block, so a
// chunk covers 128 contraction elements (two MMAs of 64).
__device__ __forceinline__ int64_t mma_scale_offset_mx(int64_t r, int64_t kb32, int64_t ocp) {
  const int64_t chunk = (r >> 7) * (ocp >> 7) + (kb32 >> 2);
  return chunk * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (kb32 & 3);
}


// ------------------------------------------------------------------ per-block helpers
// 16 bf16 values (two uint4) -> signed floats.
__device__ __forceinline__ void unpack16(const uint4& a, const uint4& b, float (&v)[16]) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
__device__ __forceinline__ uint32_t amax16_bits(const uint4& a, const uint4& b) {
  const uint32_t m2 = __vmaxu2(mag_max4(a), mag_max4(b));
  return max(m2 & 0xffffu, m2 >> 16);
}

// Block scale of NVFP4: s_b = E4M3(amax_b / (6 g)) (nearest even, saturating),
// p = decode(s_b) * g, inv = 1 / p.  `special` marks p == 0 or 1/p overflow,
// where codes are decided without the product (zero -> 0, else 6).
struct BlockScale {
  uint32_t s;
  float p, inv;
  bool special;
};
__device__ __forceinline__ BlockScale nvfp4_block_scale(uint32_t amax_bits, float g, float six_g) {
  BlockScale r;
  r.s = e4m3_rn_sat(__fdiv_rn(bf16_bits_to_float(amax_bits), six_g));
  r.p = __fmul_rn(e4m3_decode_pos(r.s), g);
  r.inv = __frcp_rn(r.p);
  r.special = !(r.inv < kInf);
  return r;
}

// The same scale with p and 1/p read from a table of all E4M3 scale codes
// (fill_scale_table): the division and the E4M3 rounding stay per block.
constexpr int kScaleCodes = 128;
__device__ __forceinline__ void fill_scale_table(float2* tab, float g) {
  for (int c = threadIdx.x; c < kScaleCodes; c += blockDim.x) {
    const float pc = __fmul_rn(e4m3_decode_pos((uint32_t)c), g);
    tab[c] = make_float2(pc, __frcp_rn(pc));
  }
}
__device__ __forceinline__ BlockScale nvfp4_block_scale_tab(uint32_t amax_bits, float six_g, const float2* tab) {
  BlockScale r;
  r.s = e4m3_rn_sat(__fdiv_rn(bf16_bits_to_float(amax_bits), six_g));
  const float2 t = tab[r.s];
  r.p = t.x;
  r.inv = t.y;
  r.special = !(r.inv < kInf);
  return r;
}

// MXFP4 block scale (OCP Microscaling v1.0) from the 32-block's largest
// magnitude as a bf16 bit pattern: E8M0 code = max(exponent field - 2, 0),
// i.e. 2^(floor(log2 amax) - 2) clamped at 2^-127 (subnormal or zero amax);
// inv = 2^-(code - 127), a normal power of two.  Encoding then runs the
// NVFP4 element path with this inverse.
__device__ __forceinline__ BlockScale mxfp4_block_scale(uint32_t amax_bits) {
  BlockScale r;
  const int32_t e = (int32_t)(amax_bits >> 7) - 2;
  r.s = (uint32_t)max(e, 0);
  r.inv = __uint_as_float((254u - r.s) << 23);
  r.p = 0.0f;   // unused: MXFP4 never takes the special path
  r.special = false;
  return r;
}

// The 16 random halves of source elements e0 .. e0+15 (e0 % 8 == 0).
__device__ __forceinline__ void sr_bits16(int64_t e0, uint64_t seed, uint64_t sid, uint32_t (&u)[8]) {
  const U4 w0 = sr_words((uint64_t)e0 >> 3, seed, sid);
  const U4 w1 = sr_words(((uint64_t)e0 >> 3) + 1, seed, sid);
  u[0] = w0.x; u[1] = w0.y; u[2] = w0.z; u[3] = w0.w;
  u[4] = w1.x; u[5] = w1.y; u[6] = w1.z; u[7] = w1.w;
}
__device__ __forceinline__ void sr_bits16_rk(int64_t e0, uint64_t sid, const PhiloxKey& rk, uint32_t (&u)[8]) {
  const U4 w0 = sr_words_rk((uint64_t)e0 >> 3, sid, rk);
  const U4 w1 = sr_words_rk(((uint64_t)e0 >> 3) + 1, sid, rk);
  u[0] = w0.x; u[1] = w0.y; u[2] = w0.z; u[3] = w0.w;
  u[4] = w1.x; u[5] = w1.y; u[6] = w1.z; u[7] = w1.w;
}
// Sources of the 16 random bits of element i of a block, for the encoders:
// packed two per word (element i in half i%2 of word i/2) ...
// Each also gives f23(i) = 2^23 + u16 as a float (sr_f23), for the FMA-pipe rounding.
struct PackedBits {
  const uint32_t* u;
  __device__ __forceinline__ uint32_t operator()(int i) const { return (i & 1) ? (u[i >> 1] >> 16) : (u[i >> 1] & 0xffffu); }
  __device__ __forceinline__ float f23(int i) const { return (i & 1) ? sr_f23<true>(u[i >> 1]) : sr_f23<false>(u[i >> 1]); }
};
// ... or one word per element, shared by two source columns: the even column's
// bits in the low half (HI false), the odd column's in the high half.
template <bool HI>
struct WordHalfBits {
  const uint32_t* r;
  __device__ __forceinline__ uint32_t operator()(int i) const { return HI ? (r[i] >> 16) : (r[i] & 0xffffu); }
  __device__ __forceinline__ float f23(int i) const { return sr_f23<HI>(r[i]); }
};

// Encode one NVFP4 block of 16 signed values into two words of packed codes
// (element 2j in the low nibble of byte j).  RND: 0 nearest, 1 stochastic.
template <int RND, class Bits = PackedBits>
__device__ __forceinline__ uint2 nvfp4_encode16(const float (&v)[16], const BlockScale& bs, Bits bits) {
  uint32_t w[2] = {0u, 0u};
  if (bs.special) {
    // p == 0: every magnitude 0; 1/p overflowed: non-zero elements saturate to 6
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t sign = (__float_as_uint(v[i]) >> 28) & 8u;
      const uint32_t mag = (bs.p == 0.0f || v[i] == 0.0f) ? 0u : 7u;
      w[i >> 3] |= (sign | mag) << (4 * (i & 7));
    }
  } else if (RND == 0) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float a[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) a[k] = __fmul_rn(v[8 * h + k], bs.inv);
      w[h] = e2m1x8_rn(a);
    }
  } else {
    // stochastic rounding on the FMA pipe (grid_sr2), the code converted from the exact grid value.
    // y is not clamped to the grid's top: above 6 (a block scale rounded down) the grid value is
    // 6 or more and the saturating conversion gives 6 either way.
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float a[8];
#pragma unroll
      for (int k = 0; k < 8; k += 2) {
        const int i = 8 * h + k;
        const float2 y = __fmul2_rn(make_float2(fabsf(v[i]), fabsf(v[i + 1])), make_float2(bs.inv, bs.inv));
        const float2 H = make_float2(e2m1_step_x2(y.x), e2m1_step_x2(y.y));
        const float2 q = grid_sr2(y, H, sr_g2<17>(bits.f23(i), bits.f23(i + 1)), 4194304.0f);
        a[k] = copysignf(q.x, v[i]);
        a[k + 1] = copysignf(q.y, v[i + 1]);
      }
      w[h] = e2m1x8_rn(a);
    }
  }
  return make_uint2(w[0], w[1]);
}


}  // namespace snip
