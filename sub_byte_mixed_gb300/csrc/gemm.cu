// gemm.cu -- the three GEMMs of the quantized linear layer (SNIP, Figure 5:
// forward Y = X W^T, dgrad dX = dY W, wgrad dW = dY^T X).  All three are "TN"
// products D = ga*gb * A B^T of two operands quantized along the contraction
// dim (K-major), so one kernel serves them.
//
// NVFP4 operands ("FP4 all the way" (Chmiel et al.), summary page, Outline:
// 16 E2M1 values share one E4M3 scale) run on the block-scaled FP4 tensor-core
// MMA (tcgen05.mma kind::mxf4nvf4, scale_vec::4X: one E4M3 scale per 16
// elements of each operand row); FP8 E4M3 operands on kind::f8f6f4.  The fp32
// tensor scales multiply the fp32 accumulator in the epilogue.
//
// Structure (one CTA per SM, persistent over output tiles, 14 warps):
//   warp 0      TMA producer: 128B-swizzled code tiles via cp.async.bulk.tensor,
//               block-scale chunks via cp.async.bulk, into a STAGES-deep ring;
//   warp 1      allocates tensor memory and issues tcgen05.mma (accumulator in
//               TMEM) from one thread;
//   warps 2-5   NVFP4 only: stage each ring slot's block scales into tensor
//               memory through registers (ld.shared + tcgen05.st), one warp per
//               32-lane quadrant, writing the 32-lane x 4-column image that a
//               32x128b.warpx4 copy would make.  tcgen05.cp from the MMA thread
//               costs ~60 tensor-pipe cycles per copy, serialised with the
//               MMAs; the register path runs beside them;
//   warps 6-13  epilogue: each warp drains 32 accumulator rows x BN/2 columns
//               from TMEM into registers (two rounds), hands the accumulator
//               back to the MMA warp, then scales by ga*gb and stores fp32
//               rows while the next tile's MMAs run.  The CTA-pair kernel's
//               single-accumulator instantiations store through shared memory
//               with TMA instead (32 x 16 fp32 boxes, two buffers per warp).
// Every wait is bounded (globaltimer); on expiry the CTA raises the timeout
// bit of the status word, lets all roles fall through, drains in-flight
// tensor-core work and frees its tensor memory before returning.
#include <cuda.h>
#include <cuda_bf16.h>

#include <cstring>

#include "snip_kernels.cuh"
#include "snip_quant.cuh"

namespace snip {

// Shared memory per CTA (227 KB), and the transposed re-quantization's
// staging: per epilogue warp 32 rows x 9 pairs {two bf16 values, their two
// random halves} (8 used, one pad: conflict-free row writes and column reads).
constexpr int kMaxSmem = 232448;
constexpr int kRqStageWords = 32 * 9;

template <int FMT, int BN, bool RQ = false>
struct GemmCfg {
  static constexpr int BM = 128;
  static constexpr int KB = 128;  // contraction bytes per stage and row (256 FP4 / 128 FP8 elements)
  static constexpr int A_BYTES = BM * KB;
  static constexpr int B_BYTES = BN * KB;
  // block-scale chunks of 512 B per 128 rows and stage: NVFP4 4 (16-element
  // blocks, 4 per MMA), MXFP4 2 (32-element blocks, 4 per chunk word = 2 MMAs)
  static constexpr int CH = FMT == 2 ? 2 : 4;
  static constexpr int SFA_BYTES = FMT ? CH * 512 : 0;
  static constexpr int SFB_BYTES = FMT ? (BN / 128) * CH * 512 : 0;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
  static constexpr int RQ_BYTES = RQ ? 8 * kRqStageWords * 8 : 0;   // 8 epilogue warps
  // four stages; a re-quantizing instantiation gives one up where its staging would not fit
  static constexpr int STAGES = 4 * STAGE_BYTES + 2048 + RQ_BYTES <= kMaxSmem ? 4 : 3;
  static constexpr int ACC_STAGES = (FMT && BN == 256) ? 1 : 2;
  // tensor-memory columns of one stage's scale factors: per MMA (K=64), A
  // takes 4 columns (128 rows / 32 lanes) and B takes BN/32
  static constexpr int SFA_COLS = 4 * CH;
  static constexpr int SF_COLS = FMT ? SFA_COLS + CH * (BN / 32) : 0;
  static constexpr int SF_TMEM_BASE = ACC_STAGES * BN;
  static constexpr int TMEM_COLS = 512;
  static_assert(SF_TMEM_BASE + STAGES * SF_COLS <= TMEM_COLS, "tensor memory budget");
  static_assert(STAGE_BYTES % 1024 == 0, "stages must keep 1024-byte alignment for the 128B swizzle");
  static constexpr int NUM_BARS = 3 * STAGES + 2 * ACC_STAGES + 1;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 1024 + RQ_BYTES;
  static_assert(SMEM_BYTES <= kMaxSmem, "shared memory budget");
  static constexpr int SF_WARPS = 4;               // scale staging, one per TMEM lane quadrant
  static constexpr int EPI_WARP0 = 2 + SF_WARPS;
  static constexpr int EPI_WARPS = 8;
  static constexpr int EPI_COLS = BN / 2;          // accumulator columns drained by one epilogue warp
  static constexpr int EPI_ROUND = RQ ? 32 : 64;   // columns per drain round (register budget)
  static constexpr int THREADS = 32 * (EPI_WARP0 + EPI_WARPS);
  // Instruction descriptor.  Block-scaled FP4: A/B type E2M1 (1) in bits 7-9
  // and 10-12, K-major, N>>3 in bits 17-22, scale type in bit 23 (UE4M3 0 for
  // NVFP4, UE8M0 1 for MXFP4), M>>4 in bits 24-28; MXFP4's scale-factor IDs
  // (bits 4-5 for B, 29-30 for A) are set per MMA.  FP8: D type f32 (1) in
  // bits 4-5, A/B type E4M3 (0) in bits 7-9 and 10-12 (A may be E5M2, 1, per GEMM).
  static constexpr uint32_t IDESC =
      FMT ? ((1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((FMT == 2 ? 1u : 0u) << 23) |
             ((uint32_t)(BM >> 4) << 24))
          : ((1u << 4) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24));
};

// NEXT-3: NVFP4 re-quantization of 32 output columns of one row.  The values
// alpha * acc are rounded to bf16 (the output's storage type), then quantized
// with the given tensor scale in 16-element row blocks -- nearest, or
// stochastic with the bits of each element's index in the row-major M x N
// output -- and written in the MMA operand layout.  Returns the largest
// magnitude as a bf16 bit pattern.
template <int RND>
__device__ __forceinline__ uint32_t requant32(const uint32_t (&r)[32], float alpha, int64_t row, int64_t col,
                                              const GemmParams& p, float g, float six_g) {
  uint32_t am = 0;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float v[16];
    uint32_t mb = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t bits = __bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(alpha, __uint_as_float(r[16 * h + i]))));
      v[i] = __uint_as_float(bits << 16);
      mb = max(mb, bits & 0x7fffu);
    }
    const BlockScale bs = nvfp4_block_scale(mb, g, six_g);
    const int64_t c = col + 16 * h;
    uint32_t u[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    if (RND) sr_bits16(row * p.N + c, p.rq_seed, p.rq_stream, u);
    *reinterpret_cast<uint2*>(p.rq_codes + row * (p.rq_ocp >> 1) + (c >> 1)) = nvfp4_encode16<RND>(v, bs, PackedBits{u});
    p.rq_scales[mma_scale_offset(row, c >> 4, p.rq_ocp)] = (uint8_t)bs.s;
    am = max(am, mb);
  }
  return am;
}

// The largest magnitude of a warp's re-quantized values, published once per warp.
__device__ __forceinline__ void requant_publish_amax(uint32_t am, uint32_t* out) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) am = max(am, __shfl_xor_sync(0xffffffffu, am, o));
  if ((threadIdx.x & 31) == 0) atomicMax(out, am << 16);   // bf16 pattern -> fp32 bits: order kept
}

// Random half of a block's element i, read from the staging (row i of the
// lane's block, the half chosen by the lane's column parity).
struct StagedBits {
  const uint2* s;   // the lane's first staged pair
  uint32_t sh;
  __device__ __forceinline__ uint32_t operator()(int i) const { return (s[i * 9].y >> sh) & 0xffffu; }
  __device__ __forceinline__ float f23(int i) const {   // 2^23 + the 16 bits, as a float (sh is 0 or 16)
    return __uint_as_float(__byte_perm(s[i * 9].y, 0x4B000000u, 0x7610u + (sh >> 3) * 0x11u));
  }
};

// NEXT-3, transposed: NVFP4 blocks of 16 consecutive rows m of one column n
// (the operand D^T, contraction M) for 32 output columns of the warp's 32
// rows m0..m0+31; `row` is this lane's row, `col` the first column.  The warp
// swaps rows and columns through its shared-memory staging in halves of 16
// columns: lane l then holds column l%16, rows 16*(l/16)..+15 -- one block,
// with the random bits the column quantizer draws for element m*N + n.
// Returns the largest magnitude as a bf16 bit pattern.
template <int RND>
__device__ __forceinline__ uint32_t requant32_t(const uint32_t (&r)[32], float alpha, int64_t row, int64_t m0,
                                                int64_t col, const GemmParams& p, float g, float six_g, uint2* stg) {
  const int lane = threadIdx.x & 31, cc = lane & 15, h = lane >> 4;
  const uint32_t sh = 16u * (uint32_t)(cc & 1);
  uint32_t am = 0;
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    uint32_t u[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    if (RND) sr_bits16(row * p.N + col + 16 * s, p.rq_seed, p.rq_stream_t, u);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(alpha, __uint_as_float(r[16 * s + 2 * k]))));
      const uint32_t hi =
          __bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(alpha, __uint_as_float(r[16 * s + 2 * k + 1]))));
      am = max(am, max(lo & 0x7fffu, hi & 0x7fffu));
      stg[lane * 9 + k] = make_uint2(lo | (hi << 16), u[k]);
    }
    __syncwarp();
    const uint2* mine = stg + 16 * h * 9 + (cc >> 1);
    float v[16];
    uint32_t mb = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t x = (mine[i * 9].x >> sh) & 0xffffu;
      v[i] = __uint_as_float(x << 16);
      mb = max(mb, x & 0x7fffu);
    }
    const BlockScale bs = nvfp4_block_scale(mb, g, six_g);
    const int64_t n = col + 16 * s + cc, m = m0 + 16 * h;
    *reinterpret_cast<uint2*>(p.rq_codes_t + n * (p.rq_ocp_t >> 1) + (m >> 1)) =
        nvfp4_encode16<RND>(v, bs, StagedBits{mine, sh});
    p.rq_scales_t[mma_scale_offset(n, m >> 4, p.rq_ocp_t)] = (uint8_t)bs.s;
    __syncwarp();   // every lane has read this half before the next one is staged
  }
  return am;
}

// RQ: the epilogue also re-quantizes the product (snip_gemm_requant); a
// separate instantiation, so the plain GEMM keeps its registers.
template <int FMT, int BN, bool RQ = false>
__global__ void __launch_bounds__(448, 1)
    gemm_tn_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, GemmParams p) {
  // the set-up below touches no memory that earlier work on the stream writes: it overlaps that
  // work's end, and the wait comes before the first operand load, scale read or store
  pdl_launch_dependents();
  using C = GemmCfg<FMT, BN, RQ>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
  const uint32_t bar0 = smem_u32(bars);
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
  auto tfull = [&](int a) { return bar0 + 8u * (2 * C::STAGES + a); };
  auto tempty = [&](int a) { return bar0 + 8u * (2 * C::STAGES + C::ACC_STAGES + a); };
  const uint32_t drain = bar0 + 8u * (2 * C::STAGES + 2 * C::ACC_STAGES);
  auto sfready = [&](int s) { return bar0 + 8u * (2 * C::STAGES + 2 * C::ACC_STAGES + 1 + s); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) { mbar_init(full(s), 1); mbar_init(empty(s), 1); }
    for (int a = 0; a < C::ACC_STAGES; ++a) { mbar_init(tfull(a), 1); mbar_init(tempty(a), C::EPI_WARPS); }
    mbar_init(drain, 1);
    for (int st = 0; st < C::STAGES; ++st) mbar_init(sfready(st), C::SF_WARPS);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) { prefetch_tmap(&tmA); prefetch_tmap(&tmB); }
  if (warp == 1) { tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_wait();
  const uint32_t tmem = *tmem_slot;
  const int num_tiles = p.num_m_tiles * p.num_n_tiles;
  const int64_t sf_chunks_per_group = p.kp >> (FMT == 2 ? 7 : 6);   // 512-byte scale chunks per 128-row group

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
        const int mt = tile % p.num_m_tiles, nt = tile / p.num_m_tiles;
        for (int kb = 0; kb < p.num_k_stages; ++kb) {
          if (!mbar_wait_bounded(empty(stage), phase ^ 1u, abort_flag, p.status, p.timeout_ns)) { ok = false; break; }
          uint8_t* sA = smem + stage * C::STAGE_BYTES;
          uint8_t* sB = sA + C::A_BYTES;
          mbar_arrive_expect_tx(full(stage), C::STAGE_BYTES);
          tma_load_2d(smem_u32(sA), &tmA, kb * C::KB, mt * C::BM, full(stage));
          tma_load_2d(smem_u32(sB), &tmB, kb * C::KB, nt * BN, full(stage));
          if (FMT) {
            uint8_t* sSFA = sB + C::B_BYTES;
            uint8_t* sSFB = sSFA + C::SFA_BYTES;
            bulk_load(smem_u32(sSFA), p.a_scales + ((int64_t)mt * sf_chunks_per_group + kb * C::CH) * 512,
                      C::SFA_BYTES, full(stage));
#pragma unroll
            for (int nb = 0; nb < BN / 128; ++nb)
              bulk_load(smem_u32(sSFB + nb * C::SFA_BYTES),
                        p.b_scales + ((int64_t)(nt * (BN / 128) + nb) * sf_chunks_per_group + kb * C::CH) * 512,
                        C::SFA_BYTES, full(stage));
          }
          if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok || *abort_flag) {
        // aborted (here or by another role of this CTA): let copies already in flight land before
        // the CTA leaves (bounded)
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 2000000ull) {}
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
        if (!mbar_wait_bounded(tempty(acc), acc_phase ^ 1u, abort_flag, p.status, p.timeout_ns)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem + acc * BN;
        for (int kb = 0; kb < p.num_k_stages; ++kb) {
          // NVFP4: the scale-staging warps signal once the slot's data and scales are in place
          if (!mbar_wait_bounded(FMT ? sfready(stage) : full(stage), phase, abort_flag, p.status, p.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sA = smem_u32(smem + stage * C::STAGE_BYTES);
          const uint32_t sB = sA + C::A_BYTES;
          const uint32_t sf = tmem + C::SF_TMEM_BASE + stage * C::SF_COLS;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint64_t adesc = smem_desc(sA + 32 * k, 16, 1024, 2);
            const uint64_t bdesc = smem_desc(sB + 32 * k, 16, 1024, 2);
            const uint32_t accum = (kb | k) != 0 ? 1u : 0u;
            if (FMT == 1) tc_mma_nvf4(d_tmem, adesc, bdesc, C::IDESC, sf + 4 * k, sf + C::SFA_COLS + k * (BN / 32), accum);
            else if (FMT == 2)   // chunk word k/2, byte pair 2*(k%2) as the scale-factor ID of A and B
              tc_mma_mxf4(d_tmem, adesc, bdesc, C::IDESC | ((2u * (k & 1)) << 4) | ((2u * (k & 1)) << 29),
                          sf + 4 * (k >> 1), sf + C::SFA_COLS + (k >> 1) * (BN / 32), accum);
            else tc_mma_f8(d_tmem, adesc, bdesc, C::IDESC | ((uint32_t)p.a_e5m2 << 7), accum);   // A type E5M2 = 1
          }
          tc_commit(empty(stage));
          if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tc_commit(tfull(acc));
        if (++acc == C::ACC_STAGES) { acc = 0; acc_phase ^= 1u; }
      }
      // all tensor-core work issued by this thread completes before TMEM is freed
      tc_commit(drain);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(drain, 0) && globaltimer_ns() - t0 < p.timeout_ns) {}
    }
  } else if (warp < C::EPI_WARP0) {
    // ---------------------------------------------------------- scale staging (block-scaled formats)
    if constexpr (FMT >= 1) {
      const int q = warp & 3;   // TMEM lane quadrant this warp may access
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
        for (int kb = 0; kb < p.num_k_stages; ++kb) {
          // the slot's previous scales were consumed: the producer refilled it only after its MMAs completed
          if (!mbar_wait_bounded(full(stage), phase, abort_flag, p.status, p.timeout_ns)) { ok = false; break; }
          const uint8_t* sSFA = smem + stage * C::STAGE_BYTES + C::A_BYTES + C::B_BYTES;
          const uint8_t* sSFB = sSFA + C::SFA_BYTES;
          uint32_t v[C::SF_COLS];
          // lane l of every quadrant holds row l of each 512-byte chunk: columns 4k..4k+3 of the
          // A scales of MMA k, then per MMA k the BN/128 chunks of the B scales
#pragma unroll
          for (int k = 0; k < C::CH; ++k) {
            const uint4 t = *reinterpret_cast<const uint4*>(sSFA + 512 * k + 16 * lane);
            v[4 * k] = t.x; v[4 * k + 1] = t.y; v[4 * k + 2] = t.z; v[4 * k + 3] = t.w;
          }
#pragma unroll
          for (int k = 0; k < C::CH; ++k)
#pragma unroll
            for (int nb = 0; nb < BN / 128; ++nb) {
              const uint4 t = *reinterpret_cast<const uint4*>(sSFB + C::SFA_BYTES * nb + 512 * k + 16 * lane);
              const int o = C::SFA_COLS + k * (BN / 32) + 4 * nb;
              v[o] = t.x; v[o + 1] = t.y; v[o + 2] = t.z; v[o + 3] = t.w;
            }
          const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + C::SF_TMEM_BASE + stage * C::SF_COLS;
#pragma unroll
          for (int c = 0; c < C::SF_COLS / 16; ++c) tmem_st_32x32b_x16(taddr + 16 * c, v + 16 * c);
          if constexpr (C::SF_COLS % 16 != 0)
            tmem_st_32x32b_x8(taddr + C::SF_COLS / 16 * 16, v + C::SF_COLS / 16 * 16);
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(sfready(stage));
          if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
        }
      }
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int q = warp & 3;                          // TMEM lane quadrant this warp may access
    const int half = (warp - C::EPI_WARP0) >> 2;     // which BN/2 columns it drains
    const float alpha = p.ga ? __fmul_rn(*p.ga, *p.gb) : 1.0f;   // MXFP4 has no tensor scales
    const float rq_g = RQ ? *p.rq_g : 1.0f, rq_six_g = __fmul_rn(6.0f, rq_g);
    uint32_t rq_am = 0;
    uint2* rq_stg = reinterpret_cast<uint2*>(smem + C::STAGES * C::STAGE_BYTES + 1024) +
                    (warp - C::EPI_WARP0) * kRqStageWords;
    uint32_t acc = 0, acc_phase = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      const int mt = tile % p.num_m_tiles, nt = tile / p.num_m_tiles;
      if (!mbar_wait_bounded(tfull(acc), acc_phase, abort_flag, p.status, p.timeout_ns)) break;
      tc_fence_after();
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + acc * BN + half * C::EPI_COLS;
      const int64_t row = (int64_t)mt * C::BM + q * 32 + lane;
      float* drow = p.D ? p.D + row * p.ldd : nullptr;
      const int64_t col0 = (int64_t)nt * BN + half * C::EPI_COLS;
#pragma unroll 1
      for (int rd = 0; rd < C::EPI_COLS / C::EPI_ROUND; ++rd) {
        uint32_t r[C::EPI_ROUND / 32][32];
#pragma unroll
        for (int c = 0; c < C::EPI_ROUND / 32; ++c) tmem_ld_32x32b_x32(taddr + rd * C::EPI_ROUND + c * 32, r[c]);
        tmem_ld_wait();
        if (rd == C::EPI_COLS / C::EPI_ROUND - 1) {   // accumulator fully read: hand it back
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(tempty(acc));
        }
        if (RQ) {   // the next GEMM's operand, written for the padded rows too (zeros)
#pragma unroll
          for (int c = 0; c < C::EPI_ROUND / 32; ++c) {
            const int64_t col = col0 + rd * C::EPI_ROUND + c * 32;
            if (p.rq_codes)
              rq_am = max(rq_am, p.rq_rnd ? requant32<1>(r[c], alpha, row, col, p, rq_g, rq_six_g)
                                          : requant32<0>(r[c], alpha, row, col, p, rq_g, rq_six_g));
            if (p.rq_codes_t)
              rq_am = max(rq_am, p.rq_rnd_t ? requant32_t<1>(r[c], alpha, row, row - lane, col, p, rq_g, rq_six_g, rq_stg)
                                            : requant32_t<0>(r[c], alpha, row, row - lane, col, p, rq_g, rq_six_g, rq_stg));
          }
        }
        if (p.D && row < p.M) {
          // 32-byte (or 16-byte when D is only 16-byte aligned) streaming stores: whole L2 sectors
          // per thread, without evicting the operands
#pragma unroll
          for (int c = 0; c < C::EPI_ROUND / 32; ++c)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int64_t col = col0 + rd * C::EPI_ROUND + c * 32 + 8 * j;
              const uint32_t* rr = &r[c][8 * j];
              if (p.v8 && col + 8 <= p.N) {
                st_global_cs_v8(drow + col, __fmul_rn(alpha, __uint_as_float(rr[0])),
                                __fmul_rn(alpha, __uint_as_float(rr[1])), __fmul_rn(alpha, __uint_as_float(rr[2])),
                                __fmul_rn(alpha, __uint_as_float(rr[3])), __fmul_rn(alpha, __uint_as_float(rr[4])),
                                __fmul_rn(alpha, __uint_as_float(rr[5])), __fmul_rn(alpha, __uint_as_float(rr[6])),
                                __fmul_rn(alpha, __uint_as_float(rr[7])));
              } else {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                  const int64_t c4 = col + 4 * h;
                  if (c4 + 4 <= p.N) {
                    st_global_cs_v4(drow + c4, __fmul_rn(alpha, __uint_as_float(rr[4 * h])),
                                    __fmul_rn(alpha, __uint_as_float(rr[4 * h + 1])),
                                    __fmul_rn(alpha, __uint_as_float(rr[4 * h + 2])),
                                    __fmul_rn(alpha, __uint_as_float(rr[4 * h + 3])));
                  } else {   // the row's last 1-3 columns: nothing past N is written
                    for (int e = 0; e < 4 && c4 + e < p.N; ++e)
                      drow[c4 + e] = __fmul_rn(alpha, __uint_as_float(rr[4 * h + e]));
                  }
                }
              }
            }
        }
      }
      if (++acc == C::ACC_STAGES) { acc = 0; acc_phase ^= 1u; }
    }
    if (RQ && p.rq_amax) requant_publish_amax(rq_am, p.rq_amax);
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ 2-CTA variant
// A cluster of two CTAs on neighbouring SMs computes one 256 x 256 tile with
// tcgen05.mma.cta_group::2: CTA r holds rows 128r..128r+127 of the pair's A
// tile and of its B tile, and accumulates its 128 rows x 256 columns in its
// own tensor memory.  Per SM that halves the B bytes per FLOP, which is what
// limits the one-CTA kernel (shared-memory fill).  The leader (rank 0) issues
// the MMAs and multicasts its commits to both CTAs; both CTAs' A/B loads
// complete on the leader's full barrier; block scales land on a local barrier
// and each CTA's four staging warps write them into its own tensor memory,
// then arrive on the leader's sf_ready barrier.  Each CTA's tensor memory must
// hold the scales of all 256 B rows (each CTA's tensor core multiplies its A
// rows by the whole B tile); holding only its own 128 gives wrong products.
// The library routes every GEMM with at least one full wave of 256 x 256
// tiles here (both formats); smaller ones run on the one-CTA kernel.
// NS: 256-column MMA sub-tiles per pair tile.  NS = 2 (FP8 only, which keeps no
// scale factors in tensor memory) makes 256 x 512 tiles: two MMAs per k-step
// share the A tile, so a CTA receives 48 KB per stage for twice the FLOPs of
// a 32 KB stage (25% less shared-memory fill per FLOP), with its two 256-column
// accumulators filling tensor memory (one accumulator stage).
template <int FMT, bool RQ = false, int NS = 1>
struct Gemm2Cfg {
  static_assert(NS == 1 || (NS == 2 && FMT == 0 && !RQ), "256 x 512 pair tiles: FP8 without re-quantization");
  static constexpr int MMA_N = 256;
  static constexpr int BM = 128, BN = MMA_N * NS, BNC = 128, KB = 128;
  static constexpr int A_BYTES = BM * KB, B_BYTES = NS * BNC * KB;
  static constexpr int CH = FMT == 2 ? 2 : 4;      // 512-byte scale chunks per 128 rows and stage
  static constexpr int SFA_BYTES = FMT ? CH * 512 : 0;
  static constexpr int SFB_BYTES = FMT ? 2 * CH * 512 : 0;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
  static constexpr int RQ_BYTES = RQ ? 8 * kRqStageWords * 8 : 0;
  static constexpr int ACC_STAGES = (FMT || NS == 2) ? 1 : 2;
  // With one accumulator stage (and no re-quantization) D leaves through TMA stores: each epilogue warp
  // stages 32 x 16 fp32 boxes (2 KB, 64-byte swizzle) in STG_BUFS shared-memory buffers.  With two
  // (FP8), whose epilogue already overlaps the next tile's MMAs, stores from registers measured
  // 3-5% faster.
  static constexpr bool TMA_D = !RQ && ACC_STAGES == 1;
  static constexpr int STG_BUFS = 2;
  static constexpr int STG_BYTES = TMA_D ? 8 * STG_BUFS * 2048 : 0;
  // NVFP4 five stages (tensor memory holds five stages of scales), else six, or fewer to fit
  static constexpr int BASE_STAGES = FMT == 1 ? 5 : 6;
  static constexpr int FIT_STAGES = (kMaxSmem - 2048 - RQ_BYTES - STG_BYTES) / STAGE_BYTES;
  static constexpr int STAGES = BASE_STAGES < FIT_STAGES ? BASE_STAGES : FIT_STAGES;
  static constexpr int SFA_COLS = 4 * CH;
  static constexpr int SFB_COLS_K = 8;                    // scale columns of B per chunk (256 rows)
  static constexpr int SF_COLS = FMT ? SFA_COLS + CH * SFB_COLS_K : 0;
  static constexpr int SF_TMEM_BASE = ACC_STAGES * BN;
  static constexpr int TMEM_COLS = 512;
  static_assert(SF_TMEM_BASE + STAGES * SF_COLS <= TMEM_COLS, "tensor memory budget");
  static_assert(STAGE_BYTES % 1024 == 0, "1024-byte aligned stages");
  static constexpr int NUM_BARS = 4 * STAGES + 2 * ACC_STAGES + 1;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 1024 + RQ_BYTES + STG_BYTES;
  static_assert(SMEM_BYTES <= kMaxSmem, "shared memory budget");
  static constexpr int SF_WARPS = 4, EPI_WARP0 = 6, EPI_WARPS = 8, EPI_COLS = BN / 2, EPI_ROUND = RQ ? 32 : 64;
  static constexpr int THREADS = 32 * (EPI_WARP0 + EPI_WARPS);
  static constexpr uint32_t IDESC =
      FMT ? ((1u << 7) | (1u << 10) | ((uint32_t)(MMA_N >> 3) << 17) | ((FMT == 2 ? 1u : 0u) << 23) |
             ((uint32_t)(256 >> 4) << 24))
          : ((1u << 4) | ((uint32_t)(MMA_N >> 3) << 17) | ((uint32_t)(256 >> 4) << 24));
};

// 448 threads; 96 registers a thread without re-quantization, so that a 256-thread quantizer CTA of
// up to 80 registers fits beside the GEMM CTA on its SM when the two streams overlap.
template <int FMT, bool RQ = false, int NS = 1>
__global__ void __maxnreg__(RQ ? 128 : 96)
    gemm_tn_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmSFA, const __grid_constant__ CUtensorMap tmSFB,
                        const __grid_constant__ CUtensorMap tmD, GemmParams p) {
  // the set-up below touches no memory that earlier work on the stream writes: it overlaps that
  // work's end, and the wait comes before the first operand load, scale read or store
  pdl_launch_dependents();
  using C = Gemm2Cfg<FMT, RQ, NS>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
  const uint32_t bar0 = smem_u32(bars);
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
  auto sffull = [&](int s) { return bar0 + 8u * (2 * C::STAGES + s); };
  auto sfready = [&](int s) { return bar0 + 8u * (3 * C::STAGES + s); };
  auto tfull = [&](int a) { return bar0 + 8u * (4 * C::STAGES + a); };
  auto tempty = [&](int a) { return bar0 + 8u * (4 * C::STAGES + C::ACC_STAGES + a); };
  const uint32_t drain = bar0 + 8u * (4 * C::STAGES + 2 * C::ACC_STAGES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
      mbar_init(sffull(s), 1);
      mbar_init(sfready(s), 2 * C::SF_WARPS);
    }
    for (int a = 0; a < C::ACC_STAGES; ++a) { mbar_init(tfull(a), 1); mbar_init(tempty(a), 2 * C::EPI_WARPS); }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) { prefetch_tmap(&tmA); prefetch_tmap(&tmB); }
  if (warp == 1) { tmem_alloc_pair(smem_u32(tmem_slot), C::TMEM_COLS); tmem_relinquish_pair(); }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // both CTAs' barriers and tensor memory exist before any cross-CTA traffic
  tc_fence_after();
  pdl_wait();
  const uint32_t tmem = *tmem_slot;
  const int num_pairs = gridDim.x >> 1, pair = blockIdx.x >> 1;
  const int num_tiles = p.num_m_tiles * p.num_n_tiles;   // 256 x 256 tiles
  const int64_t groups_k = p.kp >> 8;                     // 2 KB scale slabs per 128-row group

  if (warp == 0) {
    // ---------------------------------------------------------- producer (both CTAs)
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int tile = pair; ok && tile < num_tiles; tile += num_pairs) {
        const int mt = tile % p.num_m_tiles, nt = tile / p.num_m_tiles;
        for (int kb = 0; kb < p.num_k_stages; ++kb) {
          if (!mbar_wait_bounded(empty(stage), phase ^ 1u, abort_flag, p.status, p.timeout_ns)) { ok = false; break; }
          uint8_t* sA = smem + stage * C::STAGE_BYTES;
          uint8_t* sB = sA + C::A_BYTES;
          if (FMT) {
            uint8_t* sSFA = sB + C::B_BYTES;
            uint8_t* sSFB = sSFA + C::SFA_BYTES;
            mbar_arrive_expect_tx(sffull(stage), C::SFA_BYTES + C::SFB_BYTES);
            const int64_t ga = 2 * mt + rank;
            constexpr int R = C::SFA_BYTES / 256;   // 256-byte rows of one 128-row group's stage scales
            tma_load_2d(smem_u32(sSFA), &tmSFA, 0, (int32_t)(R * (ga * groups_k + kb)), sffull(stage));
            // both CTAs need the scales of all 256 B rows: each loads its own 128 rows' half and
            // multicasts it to the pair (the peer's half lands here on this CTA's barrier)
            tma_load_2d_mc(smem_u32(sSFB + C::SFA_BYTES * rank), &tmSFB, 0,
                           (int32_t)(R * ((2 * nt + rank) * groups_k + kb)), sffull(stage), (uint16_t)0x3);
          }
          if (rank == 0) mbar_arrive_expect_tx(full(stage), 2 * (C::A_BYTES + C::B_BYTES));
          const uint32_t leader_full = mapa_shared(full(stage), 0);
          tma_load_2d_pair(smem_u32(sA), &tmA, kb * C::KB, (2 * mt + rank) * C::BM, leader_full);
#pragma unroll
          for (int h = 0; h < NS; ++h)   // this CTA's 128 rows of each 256-row B sub-tile
            tma_load_2d_pair(smem_u32(sB + h * C::BNC * C::KB), &tmB, kb * C::KB, (2 * (NS * nt + h) + rank) * C::BNC,
                             leader_full);
          if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok || *abort_flag) {   // aborted here or by another role: let copies in flight land (bounded)
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 2000000ull) {}
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer (leader only)
    if (lane == 0 && rank == 0) {
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      // descriptors of stage 0's A and B tiles: a stage or a k-step only moves the 14-bit start address
      // (16-byte units; shared memory ends below 256 KB, so the field never carries into the next)
      const uint64_t adesc0 = smem_desc(smem_u32(smem), 16, 1024, 2);
      const uint64_t bdesc0 = smem_desc(smem_u32(smem) + C::A_BYTES, 16, 1024, 2);
      for (int tile = pair; ok && tile < num_tiles; tile += num_pairs) {
        if (!mbar_wait_bounded(tempty(acc), acc_phase ^ 1u, abort_flag, p.status, p.timeout_ns)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem + acc * C::BN;
        for (int kb = 0; kb < p.num_k_stages; ++kb) {
          if (!mbar_wait_bounded(full(stage), phase, abort_flag, p.status, p.timeout_ns)) { ok = false; break; }
          if (FMT && !mbar_wait_bounded(sfready(stage), phase, abort_flag, p.status, p.timeout_ns)) { ok = false; break; }
          tc_fence_after();
          const uint64_t soff = (uint64_t)((stage * (uint32_t)C::STAGE_BYTES) >> 4);
          const uint64_t ad = adesc0 + soff, bd = bdesc0 + soff;
          const uint32_t sf = tmem + C::SF_TMEM_BASE + stage * C::SF_COLS;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint64_t adesc = ad + (uint64_t)(2 * k);   // 32 bytes: the next 64 FP4 / 32 FP8 elements
            const uint32_t accum = (kb | k) != 0 ? 1u : 0u;
#pragma unroll
            for (int h = 0; h < NS; ++h) {   // sub-tile h accumulates in columns [256 h, 256 h + 256)
              const uint64_t bdesc = bd + (uint64_t)(((h * C::BNC * C::KB) >> 4) + 2 * k);
              if (FMT == 1)
                tc_mma_nvf4_pair(d_tmem, adesc, bdesc, C::IDESC, sf + 4 * k, sf + C::SFA_COLS + k * C::SFB_COLS_K,
                                 accum);
              else if (FMT == 2)
                tc_mma_mxf4_pair(d_tmem, adesc, bdesc, C::IDESC | ((2u * (k & 1)) << 4) | ((2u * (k & 1)) << 29),
                                 sf + 4 * (k >> 1), sf + C::SFA_COLS + (k >> 1) * C::SFB_COLS_K, accum);
              else tc_mma_f8_pair(d_tmem + h * C::MMA_N, adesc, bdesc, C::IDESC | ((uint32_t)p.a_e5m2 << 7), accum);
            }
          }
          tc_commit_pair_mc(empty(stage), 0x3);
          if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tc_commit_pair_mc(tfull(acc), 0x3);
        if (++acc == C::ACC_STAGES) { acc = 0; acc_phase ^= 1u; }
      }
      tc_commit_pair_mc(drain, 0x1);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(drain, 0) && globaltimer_ns() - t0 < p.timeout_ns) {}
    }
  } else if (warp < C::EPI_WARP0) {
    // ---------------------------------------------------------- scale staging (both CTAs, block-scaled formats)
    if constexpr (FMT >= 1) {
      const int q = warp & 3;
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int tile = pair; ok && tile < num_tiles; tile += num_pairs) {
        for (int kb = 0; kb < p.num_k_stages; ++kb) {
          if (!mbar_wait_bounded(sffull(stage), phase, abort_flag, p.status, p.timeout_ns)) { ok = false; break; }
          const uint8_t* sSFA = smem + stage * C::STAGE_BYTES + C::A_BYTES + C::B_BYTES;
          const uint8_t* sSFB = sSFA + C::SFA_BYTES;
          uint32_t v[C::SF_COLS];
#pragma unroll
          for (int k = 0; k < C::CH; ++k) {
            const uint4 t = *reinterpret_cast<const uint4*>(sSFA + 512 * k + 16 * lane);
            v[4 * k] = t.x; v[4 * k + 1] = t.y; v[4 * k + 2] = t.z; v[4 * k + 3] = t.w;
          }
#pragma unroll
          for (int k = 0; k < C::CH; ++k)
#pragma unroll
            for (int nb = 0; nb < C::SFB_COLS_K / 4; ++nb) {
              const uint4 t = *reinterpret_cast<const uint4*>(sSFB + C::SFA_BYTES * nb + 512 * k + 16 * lane);
              const int o = C::SFA_COLS + k * C::SFB_COLS_K + 4 * nb;
              v[o] = t.x; v[o + 1] = t.y; v[o + 2] = t.z; v[o + 3] = t.w;
            }
          const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + C::SF_TMEM_BASE + stage * C::SF_COLS;
#pragma unroll
          for (int c = 0; c < C::SF_COLS / 16; ++c) tmem_st_32x32b_x16(taddr + 16 * c, v + 16 * c);
          if constexpr (C::SF_COLS % 16 != 0)
            tmem_st_32x32b_x8(taddr + C::SF_COLS / 16 * 16, v + C::SF_COLS / 16 * 16);
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_remote(mapa_shared(sfready(stage), 0));
          if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
        }
      }
    }
  } else {
    // ---------------------------------------------------------- epilogue (both CTAs)
    const int q = warp & 3;
    const int half = (warp - C::EPI_WARP0) >> 2;
    const float alpha = p.ga ? __fmul_rn(*p.ga, *p.gb) : 1.0f;   // MXFP4 has no tensor scales
    const float rq_g = RQ ? *p.rq_g : 1.0f, rq_six_g = __fmul_rn(6.0f, rq_g);
    uint32_t rq_am = 0;
    uint2* rq_stg = reinterpret_cast<uint2*>(smem + C::STAGES * C::STAGE_BYTES + 1024) +
                    (warp - C::EPI_WARP0) * kRqStageWords;
    // TMA-store staging of this warp: STG_BUFS 2 KB buffers, each a 32-row x 16-column box with row i
    // (its lane i's row) at 64 i and 16-byte chunk j of the row at position j ^ ((i >> 1) & 3) (the
    // 64-byte swizzle; buffers 2048-byte aligned).  A box is staged while earlier ones are being stored.
    const uint32_t stg = smem_u32(smem + C::STAGES * C::STAGE_BYTES + 1024 + C::RQ_BYTES) +
                         (uint32_t)(warp - C::EPI_WARP0) * (uint32_t)(C::STG_BUFS * 2048);
    uint32_t nbox = 0;   // boxes this warp has stored: picks the buffer
    uint32_t acc = 0, acc_phase = 0;
    for (int tile = pair; tile < num_tiles; tile += num_pairs) {
      const int mt = tile % p.num_m_tiles, nt = tile / p.num_m_tiles;
      if (!mbar_wait_bounded(tfull(acc), acc_phase, abort_flag, p.status, p.timeout_ns)) break;
      tc_fence_after();
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + acc * C::BN + half * C::EPI_COLS;
      const int64_t row0 = (int64_t)(2 * mt + rank) * C::BM + q * 32;   // the warp's first row
      const int64_t row = row0 + lane;
      float* drow = p.D ? p.D + row * p.ldd : nullptr;
      const int64_t col0 = (int64_t)nt * C::BN + half * C::EPI_COLS;
#pragma unroll 1
      for (int rd = 0; rd < C::EPI_COLS / C::EPI_ROUND; ++rd) {
        uint32_t r[C::EPI_ROUND / 32][32];
#pragma unroll
        for (int c = 0; c < C::EPI_ROUND / 32; ++c) tmem_ld_32x32b_x32(taddr + rd * C::EPI_ROUND + c * 32, r[c]);
        tmem_ld_wait();
        if (rd == C::EPI_COLS / C::EPI_ROUND - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_remote(mapa_shared(tempty(acc), 0));
        }
        if (RQ) {
#pragma unroll
          for (int c = 0; c < C::EPI_ROUND / 32; ++c) {
            const int64_t col = col0 + rd * C::EPI_ROUND + c * 32;
            if (p.rq_codes)
              rq_am = max(rq_am, p.rq_rnd ? requant32<1>(r[c], alpha, row, col, p, rq_g, rq_six_g)
                                          : requant32<0>(r[c], alpha, row, col, p, rq_g, rq_six_g));
            if (p.rq_codes_t)
              rq_am = max(rq_am, p.rq_rnd_t ? requant32_t<1>(r[c], alpha, row, row - lane, col, p, rq_g, rq_six_g, rq_stg)
                                            : requant32_t<0>(r[c], alpha, row, row - lane, col, p, rq_g, rq_six_g, rq_stg));
          }
        }
        if constexpr (C::TMA_D) {
#pragma unroll
          for (int c = 0; c < C::EPI_ROUND / 32; ++c)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int64_t col = col0 + rd * C::EPI_ROUND + c * 32 + 16 * h;
              if (row0 < p.M && col < p.N) {   // (warp-uniform) a box wholly past D is skipped
                const uint32_t buf = stg + 2048u * (nbox % (uint32_t)C::STG_BUFS);
                if (lane == 0) bulk_wait_read<C::STG_BUFS - 1>();   // this buffer's previous box has left it
                __syncwarp();
#pragma unroll
                for (int k = 0; k < 4; ++k)
                  st_shared_v4(buf + 64u * lane + 16u * (uint32_t)(k ^ ((lane >> 1) & 3)),
                               __fmul_rn(alpha, __uint_as_float(r[c][16 * h + 4 * k])),
                               __fmul_rn(alpha, __uint_as_float(r[c][16 * h + 4 * k + 1])),
                               __fmul_rn(alpha, __uint_as_float(r[c][16 * h + 4 * k + 2])),
                               __fmul_rn(alpha, __uint_as_float(r[c][16 * h + 4 * k + 3])));
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {   // elements past M or N are not written
                  tma_store_2d(&tmD, buf, (int32_t)col, (int32_t)row0);
                  bulk_commit();
                }
                ++nbox;
              }
            }
        } else if (p.D && row < p.M) {   // the re-quantizing kernels: D optional, stored from registers
#pragma unroll
          for (int c = 0; c < C::EPI_ROUND / 32; ++c)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int64_t col = col0 + rd * C::EPI_ROUND + c * 32 + 8 * j;
              const uint32_t* rr = &r[c][8 * j];
              if (p.v8 && col + 8 <= p.N) {
                st_global_cs_v8(drow + col, __fmul_rn(alpha, __uint_as_float(rr[0])),
                                __fmul_rn(alpha, __uint_as_float(rr[1])), __fmul_rn(alpha, __uint_as_float(rr[2])),
                                __fmul_rn(alpha, __uint_as_float(rr[3])), __fmul_rn(alpha, __uint_as_float(rr[4])),
                                __fmul_rn(alpha, __uint_as_float(rr[5])), __fmul_rn(alpha, __uint_as_float(rr[6])),
                                __fmul_rn(alpha, __uint_as_float(rr[7])));
              } else {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                  const int64_t c4 = col + 4 * h;
                  if (c4 + 4 <= p.N) {
                    st_global_cs_v4(drow + c4, __fmul_rn(alpha, __uint_as_float(rr[4 * h])),
                                    __fmul_rn(alpha, __uint_as_float(rr[4 * h + 1])),
                                    __fmul_rn(alpha, __uint_as_float(rr[4 * h + 2])),
                                    __fmul_rn(alpha, __uint_as_float(rr[4 * h + 3])));
                  } else {   // the row's last 1-3 columns: nothing past N is written
                    for (int e = 0; e < 4 && c4 + e < p.N; ++e)
                      drow[c4 + e] = __fmul_rn(alpha, __uint_as_float(rr[4 * h + e]));
                  }
                }
              }
            }
        }
      }
      if (++acc == C::ACC_STAGES) { acc = 0; acc_phase ^= 1u; }
    }
    if (RQ && p.rq_amax) requant_publish_amax(rq_am, p.rq_amax);
    if (C::TMA_D && lane == 0) bulk_wait0();   // every box written before the CTA leaves
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // the peer's epilogue and the leader's MMAs are done with both tensor memories
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, C::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host side
EncodeTiledFn tensor_map_encoder() {
  static const EncodeTiledFn fn = [] {   // looked up once (thread-safe initialisation)
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(ptr);
    return (EncodeTiledFn) nullptr;
  }();
  return fn;
}

// 2-D byte tensor rows x row_bytes, loaded in boxes of box_rows x 128 bytes
// with the 128-byte swizzle the MMA descriptors expect.
static bool make_code_map(CUtensorMap* m, const uint8_t* base, int64_t rows, int64_t row_bytes, int box_rows) {
  EncodeTiledFn fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  cuuint32_t box[2] = {128u, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int FMT, int BN, bool RQ>
static cudaError_t launch_gemm_cfg(const uint8_t* a_codes, int64_t a_rows, const uint8_t* b_codes, int64_t b_rows,
                                   GemmParams p, int num_sms, cudaStream_t st) {
  using C = GemmCfg<FMT, BN, RQ>;
  cudaError_t e = ensure_max_dynamic_smem(reinterpret_cast<const void*>(gemm_tn_kernel<FMT, BN, RQ>), C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int64_t row_bytes = FMT ? p.kp / 2 : p.kp;
  CUtensorMap ta, tb;
  if (!make_code_map(&ta, a_codes, a_rows, row_bytes, C::BM) || !make_code_map(&tb, b_codes, b_rows, row_bytes, BN))
    return cudaErrorInvalidValue;
  p.num_k_stages = (int)(row_bytes / C::KB);
  p.v8 = (reinterpret_cast<uintptr_t>(p.D) % 32 == 0) && (p.ldd % 8 == 0);
  p.num_m_tiles = (int)((p.M + C::BM - 1) / C::BM);
  p.num_n_tiles = (int)((p.N + BN - 1) / BN);
  const int tiles = p.num_m_tiles * p.num_n_tiles;
  const int grid = tiles < num_sms ? tiles : num_sms;
  return launch_pdl(gemm_tn_kernel<FMT, BN, RQ>, (unsigned)grid, (unsigned)C::THREADS, (unsigned)C::SMEM_BYTES, 1u,
                    st, ta, tb, p);
}

// 2-D byte view of an MMA-layout scale buffer: rows of 256 bytes, loaded
// box_rows rows (one 128-row group's scales for 256 contraction elements:
// 2 KB for NVFP4, 1 KB for MXFP4) at a time.
static bool make_scale_map(CUtensorMap* m, const uint8_t* base, int64_t bytes, int box_rows) {
  EncodeTiledFn fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[2] = {256u, (cuuint64_t)(bytes / 256)};
  cuuint64_t strides[1] = {256u};
  cuuint32_t box[2] = {256u, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// D (M x N fp32, row stride ldd) for TMA stores of 32-row x 16-column boxes with the 64-byte swizzle;
// false when D's base or row stride is not 16-byte aligned.
static bool make_out_map(CUtensorMap* m, float* D, int64_t M, int64_t N, int64_t ldd) {
  EncodeTiledFn fn = tensor_map_encoder();
  if (!fn || !D || reinterpret_cast<uintptr_t>(D) % 16 != 0 || ldd % 4 != 0) return false;
  cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)M};
  cuuint64_t strides[1] = {(cuuint64_t)ldd * 4u};
  cuuint32_t box[2] = {16u, 32u};
  cuuint32_t estr[2] = {1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, D, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

template <int FMT, bool RQ, int NS = 1>
static cudaError_t launch_gemm_pair(const uint8_t* a_codes, int64_t a_rows, const uint8_t* b_codes, int64_t b_rows,
                                    GemmParams p, int num_sms, cudaStream_t st) {
  using C = Gemm2Cfg<FMT, RQ, NS>;
  CUtensorMap td;
  memset(&td, 0, sizeof td);
  // a D whose base or row stride does not suit TMA stores goes to the one-CTA kernel
  if (C::TMA_D && !make_out_map(&td, p.D, p.M, p.N, p.ldd))
    return launch_gemm_cfg<FMT, 256, RQ>(a_codes, a_rows, b_codes, b_rows, p, num_sms, st);
  cudaError_t e = ensure_max_dynamic_smem(reinterpret_cast<const void*>(gemm_tn_pair_kernel<FMT, RQ, NS>),
                                          C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int64_t row_bytes = FMT ? p.kp / 2 : p.kp;
  CUtensorMap ta, tb, tsa, tsb;
  memset(&tsa, 0, sizeof tsa);
  memset(&tsb, 0, sizeof tsb);
  if (!make_code_map(&ta, a_codes, a_rows, row_bytes, C::BM) || !make_code_map(&tb, b_codes, b_rows, row_bytes, C::BNC))
    return cudaErrorInvalidValue;
  const int64_t sf_div = FMT == 2 ? 32 : 16;   // elements per scale byte
  if (FMT && (!make_scale_map(&tsa, p.a_scales, a_rows * p.kp / sf_div, C::SFA_BYTES / 256) ||
              !make_scale_map(&tsb, p.b_scales, b_rows * p.kp / sf_div, C::SFA_BYTES / 256)))
    return cudaErrorInvalidValue;
  p.num_k_stages = (int)(row_bytes / C::KB);
  p.v8 = (reinterpret_cast<uintptr_t>(p.D) % 32 == 0) && (p.ldd % 8 == 0);
  p.num_m_tiles = (int)((p.M + 255) / 256);
  p.num_n_tiles = (int)((p.N + C::BN - 1) / C::BN);
  const int tiles = p.num_m_tiles * p.num_n_tiles;
  const int pairs = tiles < num_sms / 2 ? tiles : num_sms / 2;
  return launch_pdl(gemm_tn_pair_kernel<FMT, RQ, NS>, (unsigned)(2 * pairs), (unsigned)C::THREADS,
                    (unsigned)C::SMEM_BYTES, 2u, st, ta, tb, tsa, tsb, td, p);
}

// FP8 on 256 x 512 pair tiles for long contractions (measured on GB300: the
// 16384 x 8192 x 28672 GEMM 21% faster, 8192 x 4096 x 4096 25% and
// 8192 x 4096 x 11008 13% slower: the single accumulator stage exposes the
// 512-column drain once per tile, which short contractions cannot hide),
// where N's 256-row blocks pair up (so no TMA box starts past the padded B
// rows) and their coarser waves over the SM pairs cost less than the ~20%
// the wider tile saves.
static bool fp8_wide_tiles(const GemmParams& p, int num_sms) {
  const int64_t mt = (p.M + 255) / 256, nb = (p.N + 255) / 256, P = num_sms / 2;
  if (p.kp < 16384 || nb % 2 != 0 || P <= 0) return false;
  const int64_t t1 = mt * nb, t2 = t1 / 2;
  if (t2 < P) return false;
  const double e1 = (double)t1 / (double)((t1 + P - 1) / P * P), e2 = (double)t2 / (double)((t2 + P - 1) / P * P);
  return e2 * 1.2 > e1;
}

// Measured on GB300 at the Llama-7B shapes, the CTA pair beats the one-CTA
// kernel by about 11% (NVFP4) and 2-15% (FP8).  GEMMs too small to give
// every SM pair a 256 x 256 tile run on the one-CTA kernel's 128 x 256
// tiles instead, which spreads them over twice as many SMs.
template <bool RQ>
static cudaError_t launch_gemm_rq(int fmt, bool pair, const uint8_t* a_codes, int64_t a_rows_padded,
                                  const uint8_t* b_codes, int64_t b_rows_padded, const GemmParams& p, int num_sms,
                                  cudaStream_t st) {
  if (fmt == 1)
    return pair ? launch_gemm_pair<1, RQ>(a_codes, a_rows_padded, b_codes, b_rows_padded, p, num_sms, st)
                : launch_gemm_cfg<1, 256, RQ>(a_codes, a_rows_padded, b_codes, b_rows_padded, p, num_sms, st);
  if (fmt == 2)
    return pair ? launch_gemm_pair<2, RQ>(a_codes, a_rows_padded, b_codes, b_rows_padded, p, num_sms, st)
                : launch_gemm_cfg<2, 256, RQ>(a_codes, a_rows_padded, b_codes, b_rows_padded, p, num_sms, st);
  if constexpr (!RQ)
    if (pair && fp8_wide_tiles(p, num_sms))
      return launch_gemm_pair<0, false, 2>(a_codes, a_rows_padded, b_codes, b_rows_padded, p, num_sms, st);
  return pair ? launch_gemm_pair<0, RQ>(a_codes, a_rows_padded, b_codes, b_rows_padded, p, num_sms, st)
              : launch_gemm_cfg<0, 256, RQ>(a_codes, a_rows_padded, b_codes, b_rows_padded, p, num_sms, st);
}

cudaError_t launch_gemm(int fmt, const uint8_t* a_codes, int64_t a_rows_padded, const uint8_t* b_codes,
                        int64_t b_rows_padded, const GemmParams& p, int num_sms, cudaStream_t st) {
  const int64_t pair_tiles = ((p.M + 255) / 256) * ((p.N + 255) / 256);
  const bool pair = pair_tiles >= num_sms / 2;
  if (p.rq_codes || p.rq_codes_t) return launch_gemm_rq<true>(fmt, pair, a_codes, a_rows_padded, b_codes, b_rows_padded, p, num_sms, st);
  return launch_gemm_rq<false>(fmt, pair, a_codes, a_rows_padded, b_codes, b_rows_padded, p, num_sms, st);
}

}  // namespace snip

