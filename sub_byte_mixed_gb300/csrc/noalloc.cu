// noalloc.cu -- snip_tensor_scales_noalloc: the tensor-scales computation
// (amax, NVFP4 g, FP8 s) for callers that cannot hand the library a device
// workspace because they cannot allocate device memory at that point: code
// inside a framework whose caching allocator owns all device memory and
// forbids raw cudaMalloc, or a path where an allocation, which may
// synchronize the device, is not allowed.  The call itself makes ordinary
// CUDA runtime calls (a memset and a launch), so it cannot run inside a host
// function enqueued with cudaLaunchHostFunc.
//
// The kernel's scratch (one partial maximum per CTA, the completion counter
// and a status word) lives in one file-scope device array of fixed size that
// every GPU loading the library keeps until the process exits.
#include <cstdio>

#include "../../include/snip.h"
#include "snip_kernels.cuh"

namespace snip {

// scales_kernel is defined in quant.cu.
__global__ void scales_kernel(const uint16_t* __restrict__ x, int64_t n, uint32_t* __restrict__ partials,
                              uint32_t* __restrict__ counter, float* __restrict__ out3, uint32_t* __restrict__ status);

namespace {

constexpr int64_t kElemsPerSlot = 65536;                        // one CTA (and one partial) per 64 Ki elements
constexpr int kSlots = 16384;                                   // 64 KB of partial maxima
constexpr int64_t kMaxElems = kElemsPerSlot * kSlots;           // 2^30 elements
constexpr int kScratchWords = kSlots + 64;                      // partials, then counter and status

static __device__ __align__(256) uint32_t g_scales_scratch[kScratchWords];

// Host-side device address of g_scales_scratch, looked up once per device.
// The symbol's name in host code is only a stand-in, never a device address.
uint32_t* g_scratch_ptr[64] = {nullptr};

}  // namespace
}  // namespace snip

extern "C" snip_status snip_tensor_scales_noalloc(const void* x, int64_t n, float* scales_out, void* stream) {
  using namespace snip;
  if ((!x && n > 0) || !scales_out || n < 0) return SNIP_ERR_INVALID_ARG;
  if (n > kMaxElems) {
    fprintf(stderr, "snip_tensor_scales_noalloc: %lld elements exceed the fixed scratch (at most %lld)\n",
            (long long)n, (long long)kMaxElems);
    return SNIP_ERR_SHAPE;
  }
  if ((reinterpret_cast<uintptr_t>(x) & 15u) != 0) return SNIP_ERR_ALIGN;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SNIP_ERR_CUDA;
  if (dev < 0 || dev >= 64) return SNIP_ERR_UNSUPPORTED_DEVICE;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return SNIP_ERR_CUDA;
  if (major != 10 || minor != 3) return SNIP_ERR_UNSUPPORTED_DEVICE;
  if (!g_scratch_ptr[dev]) {
    // set-up on this device's first call (device current): the lookup may load the module on this
    // device, so this first call belongs outside stream capture
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_scales_scratch);
    if (e != cudaSuccess || !p) {
      fprintf(stderr, "snip_tensor_scales_noalloc: cudaGetSymbolAddress failed: %s\n", cudaGetErrorString(e));
      return SNIP_ERR_CUDA;
    }
    g_scratch_ptr[dev] = static_cast<uint32_t*>(p);
  }
  uint32_t* scratch = g_scratch_ptr[dev];
  uint32_t* counter = scratch + kSlots;
  uint32_t* status = scratch + kSlots + 1;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the counter must start at zero; the last call may have left anything there
  cudaError_t e = cudaMemsetAsync(counter, 0, 2 * sizeof(uint32_t), st);
  if (e != cudaSuccess) return SNIP_ERR_CUDA;
  int64_t grid = (n + kElemsPerSlot - 1) / kElemsPerSlot;
  if (grid < 1) grid = 1;
  scales_kernel<<<(unsigned)grid, 256, 0, st>>>(static_cast<const uint16_t*>(x), n, scratch, counter, scales_out,
                                               status);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    fprintf(stderr, "snip_tensor_scales_noalloc: launch failed: %s\n", cudaGetErrorString(e));
    return SNIP_ERR_CUDA;
  }
  return SNIP_OK;
}
