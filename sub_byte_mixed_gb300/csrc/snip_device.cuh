// snip_device.cuh -- device primitives of the quantized linear layer:
// element formats and rounding rules, Philox4x32-10, and thin inline-PTX
// wrappers for mbarrier / TMA / tcgen05 on sm_103a.
//
// Format rules ("FP4 all the way" (Chmiel et al.), summary page, Outline):
// NVFP4 is 16 E2M1 elements sharing one E4M3 scale; round-to-nearest forward,
// stochastic rounding backward.  Stochastic rounding keeps the expected value
// ("Research on Mixed-Precision Training for LLMs", stochastic rounding
// paragraph).  Every fp32 step is a single IEEE round-to-nearest operation
// (explicit __f*_rn intrinsics, no contraction), so results are bit-exact
// functions of the input.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace snip {

// Programmatic dependent launch (the kernels of this library are launched with programmatic stream
// serialization): every kernel first lets the next kernel on its stream be scheduled, then waits
// until the work it follows on the stream has finished and its writes are visible, before it touches
// memory; so stream order holds as with ordinary launches, and only the next launch's scheduling
// overlaps this one's end.  Without the launch attribute both are no-ops.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_enter() {
  pdl_launch_dependents();
  pdl_wait();
}

// Status bits OR-ed into the workspace status word by kernels.
constexpr uint32_t kDevNonFinite = 1u;
constexpr uint32_t kDevTimeout = 2u;

// ------------------------------------------------------------------ bf16
__device__ __forceinline__ float bf16_bits_to_float(uint32_t h) { return __uint_as_float(h << 16); }

// ------------------------------------------------------------------ E4M3
// Round-to-nearest-even conversion of t >= 0 to E4M3 with saturation at 448
// (hardware cvt with .satfinite).  Both halves get t, the low byte is used.
__device__ __forceinline__ uint32_t e4m3_rn_sat(float t) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(t), "f"(t));
  return r & 0xffu;
}
// Four signed values -> one word of E4M3 (E5 false) or E5M2 codes, value k in
// byte k, nearest even, saturating (E5M2: 1 sign, 5 exponent bits with bias 15,
// 2 mantissa bits; largest finite 57344, code 0x7b).
template <bool E5 = false>
__device__ __forceinline__ uint32_t fp8x4_rn_sat(float a0, float a1, float a2, float a3) {
  uint32_t r;
  if (E5)
    asm("{\n\t.reg .b16 h0, h1;\n\t"
        "cvt.rn.satfinite.e5m2x2.f32 h0, %2, %1;\n\t"
        "cvt.rn.satfinite.e5m2x2.f32 h1, %4, %3;\n\t"
        "mov.b32 %0, {h0, h1};\n\t}"
        : "=r"(r) : "f"(a0), "f"(a1), "f"(a2), "f"(a3));
  else
    asm("{\n\t.reg .b16 h0, h1;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 h0, %2, %1;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 h1, %4, %3;\n\t"
        "mov.b32 %0, {h0, h1};\n\t}"
        : "=r"(r) : "f"(a0), "f"(a1), "f"(a2), "f"(a3));
  return r;
}

// Value of a non-negative E4M3 code (0..0x7e): 2^(e-7)(1+m/8), or m 2^-9.
__device__ __forceinline__ float e4m3_decode_pos(uint32_t c) {
  uint32_t e = (c >> 3) & 15u, m = c & 7u;
  return e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : __fmul_rn((float)m, 0.001953125f);
}

// ------------------------------------------------------------------ E2M1
// Eight signed values -> one word of E2M1 codes, value k in nibble k: round to
// nearest even, saturating at +-6 (hardware cvt, two values a byte, the first
// in the low nibble), the four bytes joined by one vector move.
__device__ __forceinline__ uint32_t e2m1x8_rn(const float (&a)[8]) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(a[0]), "f"(a[1]), "f"(a[2]), "f"(a[3]), "f"(a[4]), "f"(a[5]), "f"(a[6]), "f"(a[7]));
  return r;
}
// Two E2M1 codes (one byte, low nibble first) -> their values.
__device__ __forceinline__ float2 e2m1x2_decode(uint32_t byte) {
  uint32_t h2;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(h2) : "r"(byte));
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(h);
}


// ------------------------------------------------------------------ grid rounding on the FMA pipe
// The E2M1, E4M3 and E5M2 grids have a power-of-two step h at every y >= 0
// (E2M1: 0.5 below 2, 1 below 4, 2 up to 6; E4M3: 2^(e-3), and 2^-9 below
// 2^-6; E5M2: 2^(e-2), and 2^-16 below 2^-14).  With C = 2^23 h, y + C
// rounded to fp32 is C plus a multiple of h, so for y clamped to the grid's
// top (6, 448, 57344):
//  - nearest, ties to even: q = (y + C) - C.  The even multiple of h is the
//    value whose code has a 0 last bit, the even code of the rule.
//  - stochastic with 16 random bits u and n = 65535 - u:
//    q = RZ(RZ(y + h n / 2^16) + C) - C.  y + h n / 2^16 reaches the upper
//    neighbour hi = lo + h exactly when y - lo >= h (u + 1) / 2^16, i.e. when
//    u < floor(frac 2^16): the 16-bit rule.  Rounding toward zero never moves
//    a sum across a grid value (grid values are fp32 numbers), so the
//    comparison is exact.
// Both return the grid value itself (as fp32), and they run on the FMA pipe,
// where integer carry forms of the same rules would use the slower ALU pipe.
// H is a fixed multiple of h per grid (the *_step_x* helpers) and
// k = 2^23 h / H.  A pass that needs only the code may leave y unclamped: past
// the top, h is the step of y's own binade and q a multiple of it no smaller
// than the top, which the saturating conversion maps to the top code.
__device__ __forceinline__ float2 grid_rn2(float2 yc, float2 H, float k) {
  const float2 C = __fmul2_rn(H, make_float2(k, k));
  return __ffma2_rn(C, make_float2(-1.0f, -1.0f), __fadd2_rn(yc, C));   // exact: the sum is C plus a multiple of h
}
// g = h n / 2^16 / H (sr_g2)
__device__ __forceinline__ float2 grid_sr2(float2 yc, float2 H, float2 g, float k) {
  const float2 t = __fadd2_rz(yc, __fmul2_rn(H, g));                     // H g = h n / 2^16, exact
  const float2 C = __fmul2_rn(H, make_float2(k, k));
  return __ffma2_rn(C, make_float2(-1.0f, -1.0f), __fadd2_rz(t, C));
}
// The float 2^23 + u of a 16-bit value u (its bits: 0x4B000000 | u): the low
// (HI false) or high half of a random word, with one byte permutation.
template <bool HI>
__device__ __forceinline__ float sr_f23(uint32_t word) {
  return __uint_as_float(__byte_perm(word, 0x4B000000u, HI ? 0x7632u : 0x7610u));
}
// n / 2^S with n = 65535 - u for a pair of sr_f23 values: (2^23 + 65535 - f) / 2^S, exact.
template <int S>
__device__ __forceinline__ float2 sr_g2(float f0, float f1) {
  constexpr float kNeg = -1.0f / (float)(1u << S);
  constexpr float kAdd = 8454143.0f / (float)(1u << S);   // (2^23 + 65535) / 2^S
  return __ffma2_rn(make_float2(f0, f1), make_float2(kNeg, kNeg), make_float2(kAdd, kAdd));
}
// Twice, eight and four times the E2M1, E4M3 and E5M2 step at y >= 0 (the
// exponent of y as a power of two, at least the grid's bottom binade).
__device__ __forceinline__ float e2m1_step_x2(float y) {
  return fmaxf(__uint_as_float(__float_as_uint(y) & 0x7f800000u), 1.0f);
}
__device__ __forceinline__ float e4m3_step_x8(float y) {
  return fmaxf(__uint_as_float(__float_as_uint(y) & 0x7f800000u), 0.015625f);
}
__device__ __forceinline__ float e5m2_step_x4(float y) {
  return fmaxf(__uint_as_float(__float_as_uint(y) & 0x7f800000u), 6.103515625e-05f);
}

// ------------------------------------------------------------------ Philox4x32-10
// Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3"
// (SC'11): ten rounds of two 32x32->64-bit products on a 4-word counter, the
// 2-word key bumped by the Weyl constants between rounds.
struct U4 { uint32_t x, y, z, w; };
// The 64-bit product of two words as its low and high words, one wide multiply.
__device__ __forceinline__ void mul_wide_u32(uint32_t a, uint32_t b, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b64 t;\n\tmul.wide.u32 t, %2, %3;\n\tmov.b64 {%0, %1}, t;\n\t}" : "=r"(lo), "=r"(hi) : "r"(a), "r"(b));
}

__device__ __forceinline__ U4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                            uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) { k0 += 0x9E3779B9u; k1 += 0xBB67AE85u; }
    uint32_t lo0, hi0, lo1, hi1;
    mul_wide_u32(0xD2511F53u, c0, lo0, hi0);
    mul_wide_u32(0xCD9E8D57u, c2, lo1, hi1);
    const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
  }
  return U4{c0, c1, c2, c3};
}

// The round keys of one seed: round r uses (k[r], k[10 + r]), the seed's two
// words plus r Weyl steps.  Computed once on the host and passed in a kernel's
// parameters, the rounds read them as constants and spend no instruction on
// the key schedule.
struct PhiloxKey { uint32_t k[20]; };
__host__ __device__ inline PhiloxKey philox_round_keys(uint64_t seed) {
  PhiloxKey r;
  uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32);
  for (int i = 0; i < 10; ++i) {
    r.k[i] = k0;
    r.k[10 + i] = k1;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return r;
}
__device__ __forceinline__ U4 philox4x32_10_rk(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, const PhiloxKey& rk) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    uint32_t lo0, hi0, lo1, hi1;
    mul_wide_u32(0xD2511F53u, c0, lo0, hi0);
    mul_wide_u32(0xCD9E8D57u, c2, lo1, hi1);
    const uint32_t n0 = hi1 ^ c1 ^ rk.k[r], n2 = hi0 ^ c3 ^ rk.k[10 + r];
    c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
  }
  return U4{c0, c1, c2, c3};
}
// sr_words with the seed's round keys
__device__ __forceinline__ U4 sr_words_rk(uint64_t group, uint64_t stream_id, const PhiloxKey& rk) {
  return philox4x32_10_rk((uint32_t)group, (uint32_t)(group >> 32), (uint32_t)stream_id, (uint32_t)(stream_id >> 32),
                          rk);
}

// The 4 random words covering source elements 8*group .. 8*group+7: element
// 8*group + i takes word i/2, low half for even i.
__device__ __forceinline__ U4 sr_words(uint64_t group, uint64_t seed, uint64_t stream_id) {
  return philox4x32_10((uint32_t)group, (uint32_t)(group >> 32), (uint32_t)stream_id,
                       (uint32_t)(stream_id >> 32), (uint32_t)seed, (uint32_t)(seed >> 32));
}

// ------------------------------------------------------------------ misc
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait: spins until the phase with `parity` completes, the shared
// abort flag is raised by another role, or `limit_ns` elapse (then raises the
// abort flag and the timeout bit of the status word).  Returns true when the
// phase completed.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                  uint32_t* status, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0u) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        *abort_flag = 1;
        if (status) atomicOr(status, kDevTimeout);
        return false;
      }
    }
  }
}

// ------------------------------------------------------------------ clusters
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// shared::cluster address of the same shared variable in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t mapa_shared(uint32_t local_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_addr), "r"(rank));
  return r;
}
// Arrive on a barrier of another CTA of the cluster.  The release is at CTA
// scope: what the arrive publishes is tensor-memory traffic (ordered by
// tcgen05.wait + tcgen05.fence::before_thread_sync on this side and
// tcgen05.fence::after_thread_sync on the waiting side), not generic memory.
// A cluster-scope release here costs about a microsecond per arrive, which
// made a per-stage handshake the bottleneck of the CTA-pair GEMM.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cta.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ------------------------------------------------------------------ TMA / bulk copies
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int32_t c0, int32_t c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"(tmap), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}
// TMA load into this CTA's shared memory whose completion is counted on an
// mbarrier of either CTA of the pair (shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const void* tmap, int32_t c0, int32_t c1,
                                                 uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(dst),
      "l"(tmap), "r"(c0), "r"(c1), "r"(bar_cluster)
      : "memory");
}
// TMA load multicast to the CTAs of `mask` in the cluster: each receives the box at the same shared-memory
// offset and its completion on its own mbarrier at the same offset.
__device__ __forceinline__ void tma_load_2d_mc(uint32_t dst, const void* tmap, int32_t c0, int32_t c1, uint32_t bar,
                                               uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster "
      "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(tmap), "r"(c0), "r"(c1), "r"(bar), "h"(mask)
      : "memory");
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
// TMA store of one box from this CTA's shared memory to global memory; the issuing thread tracks its
// completion as a bulk async-group (commit, then wait for the source to be read or the write done).
// Elements of the box outside the tensor are not written.
__device__ __forceinline__ void tma_store_2d(const void* tmap, uint32_t src, int32_t c0, int32_t c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];"
               ::"l"(tmap), "r"(src), "r"(c0), "r"(c1)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most N of this thread's bulk async-groups still read their shared-memory source.
template <int N>
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory"); }
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Orders this thread's generic-proxy shared-memory writes before later async-proxy (TMA) reads.
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void st_shared_v4(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// ------------------------------------------------------------------ tcgen05
// Pair forms: issued by one warp of each CTA of the pair (alloc, relinquish,
// dealloc) or by one thread of the leader CTA for both (mma, commit).
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// arrive on the mbarrier at the same shared offset in every CTA of `mask`
__device__ __forceinline__ void tc_commit_pair_mc(uint32_t bar_local, uint16_t mask) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
               ::"r"(bar_local), "h"(mask)
               : "memory");
}
__device__ __forceinline__ void tc_mma_nvf4_pair(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                                 uint32_t sfb, uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
      ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accum)
      : "memory");
}
__device__ __forceinline__ void tc_mma_mxf4_pair(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                                 uint32_t sfb, uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
      ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accum)
      : "memory");
}
__device__ __forceinline__ void tc_mma_f8_pair(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(accum)
      : "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void tc_mma_nvf4(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                            uint32_t sfb, uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
      ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accum)
      : "memory");
}
__device__ __forceinline__ void tc_mma_mxf4(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                            uint32_t sfb, uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
      ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accum)
      : "memory");
}
__device__ __forceinline__ void tc_mma_f8(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(accum)
      : "memory");
}
// 32 lanes x 32 consecutive 32-bit columns -> 32 registers per thread.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// 16 registers per thread -> 32 lanes x 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};"
      ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st_32x32b_x8(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
      ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
      : "memory");
}
// 32-byte store of 8 floats with the streaming (evict-first) cache hint; ptr 32-byte aligned.
__device__ __forceinline__ void st_global_cs_v8(float* ptr, float a0, float a1, float a2, float a3, float a4, float a5,
                                                float a6, float a7) {
  asm volatile("st.global.cs.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(ptr), "f"(a0), "f"(a1), "f"(a2),
               "f"(a3), "f"(a4), "f"(a5), "f"(a6), "f"(a7)
               : "memory");
}
__device__ __forceinline__ void st_global_cs_v4(float* ptr, float a0, float a1, float a2, float a3) {
  asm volatile("st.global.cs.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(ptr), "f"(a0), "f"(a1), "f"(a2), "f"(a3) : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor (tcgen05): start address, leading and
// stride byte offsets (16-byte units), version 1, layout type in bits 61..63
// (0 = no swizzle, 2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes,
                                              uint32_t layout) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3fffu);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3fffu) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3fffu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)(layout & 7u) << 61;
  return d;
}

}  // namespace snip
