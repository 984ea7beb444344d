// mhla_forward_noalloc: the non-causal MHLA forward for callers that cannot
// allocate device memory.
//
// Some callers have no way to obtain device memory for a workspace: code
// running where the allocator is forbidden or unavailable (a plugin inside a
// host framework that owns a fixed memory pool, a real-time loop that must
// not allocate after start-up, a caller from a runtime with no CUDA allocator
// binding).  For them this entry point takes its scratch from a fixed
// file-scope device array instead of a caller-provided workspace.  It runs
// the same summary / mixing / output kernels as the SIMT path of mhla_forward.
#include <cmath>
#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace mhla {
namespace {

constexpr size_t kScratchBytes = MHLA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// One copy per GPU that loads this library, held until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Device addresses of g_noalloc_scratch, looked up once per device.  In host
// code the symbol itself is only a host-side stand-in for the array and must
// never be passed to a kernel.
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlap(const void* a, size_t an, const void* b, size_t bn) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return an != 0 && bn != 0 && x < y + bn && y < x + an;
}

mhla_status scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MHLA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MHLA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return MHLA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return MHLA_OK;
}

}  // namespace
}  // namespace mhla

using namespace mhla;

extern "C" mhla_status mhla_forward_noalloc(const void* q, const void* k, const void* v,
                                            const float* mixing, void* y, float* den_out, int B,
                                            int H, int N, int d, int block_size, mhla_dtype dt,
                                            float eps, void* stream) {
  if (B < 0 || H < 0 || N < 0) return MHLA_ERR_INVALID_ARG;
  if (!(d == 16 || d == 32 || d == 64 || d == 128)) return MHLA_ERR_INVALID_ARG;
  if (dt != MHLA_F32 && dt != MHLA_BF16) return MHLA_ERR_INVALID_ARG;
  if (!std::isfinite(eps) || eps < 0.f) return MHLA_ERR_INVALID_ARG;
  if (block_size <= 0 || (N > 0 && N % block_size != 0)) return MHLA_ERR_INVALID_ARG;
  if ((size_t)B * H * N == 0) return MHLA_OK;
  if (!q || !k || !v || !mixing || !y) return MHLA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(mixing) || !aligned16(y) ||
      (den_out && !aligned16(den_out)))
    return MHLA_ERR_INVALID_ARG;
  const size_t tb = (size_t)B * H * N * d * (dt == MHLA_F32 ? 4 : 2);
  if (overlap(y, tb, q, tb) || overlap(y, tb, k, tb) || overlap(y, tb, v, tb))
    return MHLA_ERR_INVALID_ARG;
  if (den_out) {
    const size_t db = (size_t)B * H * N * sizeof(float);
    if (overlap(den_out, db, q, tb) || overlap(den_out, db, k, tb) ||
        overlap(den_out, db, v, tb) || overlap(den_out, db, y, tb))
      return MHLA_ERR_INVALID_ARG;
  }
  const MhlaShape s{B, H, N, d, block_size};
  if (simt_mhla_workspace(s) > kScratchBytes) return MHLA_ERR_UNSUPPORTED;  // scratch too small
  void* scratch = nullptr;
  const mhla_status st = scratch_for_current_device(&scratch);
  if (st != MHLA_OK) return st;
  // Every intermediate in the scratch is fully written before it is read, so
  // nothing needs clearing between calls.
  const cudaError_t err = simt_mhla_launch(s, dt, q, k, v, mixing, y, den_out, eps, MIX_FULL,
                                           scratch, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? MHLA_OK : MHLA_ERR_CUDA;
}
