// Device helpers shared by the kernels of the MHLA library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "mhla.h"

namespace mhla {

// The opt-in dynamic shared memory size of a kernel, set on each device the
// first time the kernel is launched there (cudaFuncSetAttribute is per device;
// the first call of a process may run on any device and from any host thread).
class SmemOptIn {
 public:
  cudaError_t ensure(const void* fn, int bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(mu_);
    if (dev < 64 && ((done_ >> dev) & 1ull)) return cudaSuccess;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && dev < 64) done_ |= 1ull << dev;
    return e;
  }

 private:
  std::mutex mu_;
  unsigned long long done_ = 0;  // a bit per device
};

// phi(x) = ELU(x) + 1: x + 1 for x > 0, exp(x) otherwise
// ("Linear Attention notes" §二, first kernel choice).
__device__ __forceinline__ float phi(float x) { return x > 0.f ? x + 1.f : expf(x); }

// The feature maps of "Linear Attention notes" §二: 0 = ELU + 1, 1 = ReLU, 2 = exp.
__device__ __forceinline__ float phi_k(float x, int kind) {
  return kind == 0 ? phi(x) : kind == 1 ? fmaxf(x, 0.f) : expf(x);
}

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Status word at the start of every workspace: bit 0 = a bounded wait gave up.
struct WorkspaceHeader {
  unsigned int status;
  unsigned int pad[63];  // keeps what follows 256-byte aligned
};

// Every workspace starts with the header and a fixed counter region used by
// the persistent kernels (ticket, finished, two per-head counters for up to
// kMaxCounterHeads heads).  The kernels leave these counters at zero when
// they exit and no kernel writes data into the region, so a workspace that
// was zero-filled once stays valid for any later call, shape or path.
constexpr int kMaxCounterHeads = 65536;
constexpr size_t kCounterOffset = sizeof(WorkspaceHeader);
constexpr size_t kWorkspacePrefix =
    ((sizeof(WorkspaceHeader) + (2 + 2 * (size_t)kMaxCounterHeads) * sizeof(unsigned)) + 255) &
    ~size_t(255);

}  // namespace mhla
