// dw_noise.cu -- the weight-gradient form of the sqrt(3) check ("FP4 all the
// way" (Chmiel et al.), summary page, Outline: quantized training stops paying
// off once the gradient's norm falls below about sqrt(3) times the
// quantization noise).  With dW = dY^T X from the unquantized bf16 tensors and
// dW_q the layer's quantized weight gradient, one kernel computes
//   ||dW||^2 and ||dW_q - dW||^2
// without writing dW anywhere: a bf16 GEMM on the tensor cores
// (tcgen05.mma kind::f16, fp32 accumulator in tensor memory) whose epilogue
// reads dW_q beside each accumulator tile and reduces both sums.
//
// Operands: the contraction runs over the tokens T, which index the rows of
// both dY (T x N) and X (T x K).  Both are therefore MN-major operands of
// dW = A B^T with A = dY^T (N x T) and B = X^T (K x T): a TMA box of 64
// consecutive columns (128 bytes) x 64 token rows, 128-byte swizzled, is one
// column of 8-row swizzle atoms.  An A tile (128 rows of dW) is two boxes, a B
// tile (256 columns of dW) four, 8 KB apart: the descriptors' leading byte
// offset (between 64-element chunks along M or N) is 8 KB and the stride byte
// offset (between 8-token groups) 1 KB; an MMA consumes 16 tokens, 2 KB.
//
// Structure (one CTA per SM, persistent over 128 x 256 tiles of dW, 10 warps):
//   warp 0      TMA producer into a 4-stage ring (48 KB per stage);
//   warp 1      allocates tensor memory (two 256-column accumulators) and
//               issues the MMAs from one thread;
//   warps 2-9   epilogue: each warp reads 32 accumulator rows x 128 columns
//               with tcgen05.ld, 32 columns at a time, beside the same dW_q
//               entries from global memory, and accumulates both sums (fp32
//               per thread); the CTA's sums go to fp64 partials, which the
//               last CTA adds up.
// Every wait is bounded (globaltimer): on expiry the CTA raises the timeout
// bit of the status word, every role falls through, the MMA thread waits
// (bounded) for its tensor-core work and the tensor memory is freed.
#include <cuda.h>

#include "snip_kernels.cuh"

namespace snip {

namespace {

struct DwCfg {
  static constexpr int BM = 128, BN = 256, BK = 64;           // tile of dW (rows n, columns k), tokens per stage
  static constexpr int BOX = 64;                               // columns per TMA box (128 bytes of bf16)
  static constexpr int A_BYTES = BM * BK * 2, B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;        // 48 KB
  static constexpr int STAGES = 4;
  static constexpr int ACC_STAGES = 2;
  static constexpr int TMEM_COLS = 512;
  static constexpr int NUM_BARS = 2 * STAGES + 2 * ACC_STAGES + 1;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 1024;
  static constexpr int EPI_WARP0 = 2, EPI_WARPS = 8;
  static constexpr int THREADS = 32 * (EPI_WARP0 + EPI_WARPS);
  static constexpr int BOX_BYTES = BOX * BK * 2;               // 8 KB: leading byte offset of both operands
  // Instruction descriptor, kind::f16: D f32 (bits 4-5 = 1), A and B bf16 (bits 7-9, 10-12 = 1), A and B
  // MN-major (bits 15, 16), N >> 3 in bits 17-22, M >> 4 in bits 24-28.
  static constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) | (1u << 16) |
                                    ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
  static_assert(ACC_STAGES * BN <= TMEM_COLS, "tensor memory budget");
};

__device__ __forceinline__ void tc_mma_f16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(accum)
      : "memory");
}

struct DwParams {
  const float* dwq;          // N x K fp32, row-major (the quantized weight gradient)
  int64_t N, K;
  int num_k_stages, num_m_tiles, num_n_tiles;
  double* partials;          // 2 per CTA
  uint32_t* counter;         // self-resetting
  double* out2;              // {||dW||^2, ||dW_q - dW||^2}
  uint32_t* status;
  uint64_t timeout_ns;
};

__global__ void __launch_bounds__(DwCfg::THREADS, 1)
    dw_noise_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                         DwParams p) {
  using C = DwCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
  const uint32_t bar0 = smem_u32(bars);
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
  auto tfull = [&](int a) { return bar0 + 8u * (2 * C::STAGES + a); };
  auto tempty = [&](int a) { return bar0 + 8u * (2 * C::STAGES + C::ACC_STAGES + a); };
  const uint32_t drain = bar0 + 8u * (2 * C::STAGES + 2 * C::ACC_STAGES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) { mbar_init(full(s), 1); mbar_init(empty(s), 1); }
    for (int a = 0; a < C::ACC_STAGES; ++a) { mbar_init(tfull(a), 1); mbar_init(tempty(a), C::EPI_WARPS); }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) { prefetch_tmap(&tmA); prefetch_tmap(&tmB); }
  if (warp == 1) { tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int num_tiles = p.num_m_tiles * p.num_n_tiles;
  float s_ref = 0.0f, s_err = 0.0f;   // this thread's sums (epilogue warps)

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
        const int mt = tile % p.num_m_tiles, nt = tile / p.num_m_tiles;
        for (int kb = 0; kb < p.num_k_stages; ++kb) {
          if (!mbar_wait_bounded(empty(stage), phase ^ 1u, abort_flag, p.status, p.timeout_ns)) { ok = false; break; }
          const uint32_t sA = smem_u32(smem + stage * C::STAGE_BYTES);
          const uint32_t sB = sA + C::A_BYTES;
          mbar_arrive_expect_tx(full(stage), C::STAGE_BYTES);
          // boxes of 64 columns x 64 tokens; out-of-range columns or tokens arrive as zeros
#pragma unroll
          for (int b = 0; b < C::BM / C::BOX; ++b)
            tma_load_2d(sA + b * C::BOX_BYTES, &tmA, mt * C::BM + b * C::BOX, kb * C::BK, full(stage));
#pragma unroll
          for (int b = 0; b < C::BN / C::BOX; ++b)
            tma_load_2d(sB + b * C::BOX_BYTES, &tmB, nt * C::BN + b * C::BOX, kb * C::BK, full(stage));
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
        const uint32_t d_tmem = tmem + acc * C::BN;
        for (int kb = 0; kb < p.num_k_stages; ++kb) {
          if (!mbar_wait_bounded(full(stage), phase, abort_flag, p.status, p.timeout_ns)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sA = smem_u32(smem + stage * C::STAGE_BYTES);
          const uint32_t sB = sA + C::A_BYTES;
#pragma unroll
          for (int k = 0; k < C::BK / 16; ++k) {
            // MN-major, 128-byte swizzle: leading byte offset 8 KB (next 64 columns), stride byte
            // offset 1 KB (next 8 tokens); 16 tokens per MMA
            const uint64_t adesc = smem_desc(sA + 2048 * k, C::BOX_BYTES, 1024, 2);
            const uint64_t bdesc = smem_desc(sB + 2048 * k, C::BOX_BYTES, 1024, 2);
            tc_mma_f16(d_tmem, adesc, bdesc, C::IDESC, (kb | k) != 0 ? 1u : 0u);
          }
          tc_commit(empty(stage));
          if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tc_commit(tfull(acc));
        if (++acc == C::ACC_STAGES) { acc = 0; acc_phase ^= 1u; }
      }
      // all tensor-core work issued by this thread completes before the tensor memory is freed
      tc_commit(drain);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(drain, 0) && globaltimer_ns() - t0 < p.timeout_ns) {}
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int q = warp & 3;                         // tensor-memory lane quadrant this warp may read
    const int half = (warp - C::EPI_WARP0) >> 2;    // which 128 of the tile's 256 columns
    uint32_t acc = 0, acc_phase = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      const int mt = tile % p.num_m_tiles, nt = tile / p.num_m_tiles;
      if (!mbar_wait_bounded(tfull(acc), acc_phase, abort_flag, p.status, p.timeout_ns)) break;
      tc_fence_after();
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + acc * C::BN + half * (C::BN / 2);
      const int64_t row = (int64_t)mt * C::BM + q * 32 + lane;
      const int64_t col0 = (int64_t)nt * C::BN + half * (C::BN / 2);
      const float* qrow = p.dwq + row * p.K;
      const bool row_in = row < p.N;
#pragma unroll 1
      for (int c = 0; c < (C::BN / 2) / 32; ++c) {
        const int64_t col = col0 + 32 * c;
        // this thread's 32 dW_q entries (128 contiguous bytes), requested before the accumulator
        float4 w[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          w[j] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (row_in && col + 4 * j < p.K) w[j] = __ldcs(reinterpret_cast<const float4*>(qrow + col + 4 * j));
        }
        uint32_t r[32];
        tmem_ld_32x32b_x32(taddr + 32 * c, r);
        tmem_ld_wait();
        if (c == (C::BN / 2) / 32 - 1) {   // accumulator fully read: hand it back
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(tempty(acc));
        }
        // rows and columns past dW are zero in the accumulator and read as zero from dW_q
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float a0 = __uint_as_float(r[4 * j]), a1 = __uint_as_float(r[4 * j + 1]);
          const float a2 = __uint_as_float(r[4 * j + 2]), a3 = __uint_as_float(r[4 * j + 3]);
          s_ref = fmaf(a0, a0, fmaf(a1, a1, fmaf(a2, a2, fmaf(a3, a3, s_ref))));
          const float d0 = w[j].x - a0, d1 = w[j].y - a1, d2 = w[j].z - a2, d3 = w[j].w - a3;
          s_err = fmaf(d0, d0, fmaf(d1, d1, fmaf(d2, d2, fmaf(d3, d3, s_err))));
        }
      }
      if (++acc == C::ACC_STAGES) { acc = 0; acc_phase ^= 1u; }
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
  // the CTA's sums (fp32 within the CTA), fp64 across CTAs; the last CTA writes out2
  float acc2[2] = {s_ref, s_err};
  block_sum_f32<2>(acc2);
  __shared__ bool s_last;
  if (threadIdx.x == 0) {
    p.partials[2 * blockIdx.x] = (double)acc2[0];
    p.partials[2 * blockIdx.x + 1] = (double)acc2[1];
    __threadfence();
    s_last = atomicAdd(p.counter, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  __shared__ double s_tot[2];
  if (warp < 2) {
    double t = 0.0;
    for (uint32_t j = lane; j < gridDim.x; j += 32) t += ((volatile double*)p.partials)[2 * j + warp];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if (lane == 0) s_tot[warp] = t;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    p.out2[0] = s_tot[0];
    p.out2[1] = s_tot[1];
    *p.counter = 0;
  }
}

// A row-major bf16 tensor rows x cols, loaded in boxes of 64 columns x 64 rows with the 128-byte swizzle.
bool make_bf16_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols) {
  EncodeTiledFn fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2u};
  cuuint32_t box[2] = {(cuuint32_t)DwCfg::BOX, (cuuint32_t)DwCfg::BK};
  cuuint32_t estr[2] = {1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_dw_noise_gemm(const void* X, const void* dY, int64_t T, int64_t K, int64_t N, const float* dwq,
                                 double* partials, uint32_t* counter, double* out2, uint32_t* status,
                                 uint64_t timeout_ns, int num_sms, cudaStream_t st) {
  using C = DwCfg;
  cudaError_t e = ensure_max_dynamic_smem(reinterpret_cast<const void*>(dw_noise_gemm_kernel), C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  CUtensorMap ta, tb;
  if (!make_bf16_map(&ta, dY, T, N) || !make_bf16_map(&tb, X, T, K)) return cudaErrorInvalidValue;
  DwParams p;
  p.dwq = dwq;
  p.N = N;
  p.K = K;
  p.num_k_stages = (int)((T + C::BK - 1) / C::BK);
  p.num_m_tiles = (int)((N + C::BM - 1) / C::BM);
  p.num_n_tiles = (int)((K + C::BN - 1) / C::BN);
  p.partials = partials;
  p.counter = counter;
  p.out2 = out2;
  p.status = status;
  p.timeout_ns = timeout_ns;
  const int tiles = p.num_m_tiles * p.num_n_tiles;
  const int grid = tiles < num_sms ? tiles : num_sms;
  dw_noise_gemm_kernel<<<grid, C::THREADS, C::SMEM_BYTES, st>>>(ta, tb, p);
  return cudaGetLastError();
}

}  // namespace snip
