// Causal MHLA inference, one token at a time ("MHLA: Restoring Expressivity of
// Linear Attention via Token-Level Multi-Head", App. C, causal inference).
//
// The summaries of finished blocks are frozen; the running summary S_i, z_i of
// the current block i takes each token (S_i += phi(k) v^T, z_i += phi(k)), and
// the token reads the mixture
//   num = phi(q) (sum_{b<i} m_ib S_b + m_ii S_i),
//   den = phi(q) . (sum_{b<i} m_ib z_b + m_ii z_i) + eps,   out = num / den,
// the chunk form of the causal MHLA forward evaluated at one token.
//
// One CTA per (batch, head) unit walks the call's tokens in order (their rows
// arrive through a cp.async ring several tokens ahead; phi of token n + 1 is
// taken while token n is computed).  Its
// threads hold the unit's running summary S_i and the mixed state
// R = P_i + m_ii S_i, P_i = sum_{b<i} m_ib S_b, in registers (thread (g, e)
// owns column e of rows g, g + G, ...); P_i is formed from the frozen
// summaries in memory when block i starts, so a token costs three d^2 FMAs
// (S_i, R, and the output) whatever i is.  A finished block's summary is
// written back to its slot.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace mhla {
namespace {

template <int D> struct StreamGeom {
  static constexpr int NT = D == 128 ? 512 : 256;  // threads
  static constexpr int G = NT / D;                 // row groups
  static constexpr int RPT = D / G;                // rows per thread
};

constexpr int kPipe = 8;  // tokens in flight in the cp.async ring

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const unsigned sa = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(sa), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

template <typename T, int D>
__global__ void __launch_bounds__(StreamGeom<D>::NT)
causal_stream_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                     const float* __restrict__ mixing, float* __restrict__ S, float* __restrict__ z,
                     T* __restrict__ out, float* __restrict__ den_out, int t0, int T_steps, int units, int H,
                     int block, int M, float eps) {
  using G_ = StreamGeom<D>;
  constexpr int G = G_::G, RPT = G_::RPT;
  constexpr int RC = D * (int)sizeof(T) / 16;  // 16-byte chunks of a q, k or v row
  __shared__ __align__(16) T ring[kPipe][3][D];
  __shared__ float sq[2][D], sk[2][D], sv[2][D];  // phi(q), phi(k), v of a token, by parity
  __shared__ float red[G][D];
  __shared__ float sden[(D + 31) / 32];  // per-warp sums of the denominator terms
  if (T_steps <= 0) return;
  const int u = blockIdx.x, tid = threadIdx.x;
  const int e = tid % D, g = tid / D;
  const float* mh = mixing + (size_t)(u % H) * M * M;
  float* Su = S + (size_t)u * M * D * D;
  float* zu = z + (size_t)u * M * D;
  const size_t tstride = (size_t)units * D;  // elements from one token of the unit to the next

  // token n's q, k, v rows into ring stage n % kPipe (past the last token: the last again, into
  // a stage no later token uses); one commit group per token
  auto issue = [&](int n) {
    const int nn = n < T_steps ? n : T_steps - 1;
    if (tid < 3 * RC) {
      const int w = tid / RC, c = tid - w * RC;
      const T* src = (w == 0 ? q : w == 1 ? k : v) + (size_t)nn * tstride + (size_t)u * D;
      cp_async16(reinterpret_cast<char*>(ring[n % kPipe][w]) + c * 16, reinterpret_cast<const char*>(src) + c * 16);
    }
    cp_async_commit();
  };
  // phi of token n from its ring stage into the parity-n buffers (threads tid < D)
  auto prep = [&](int n) {
    if (tid < D) {
      const T* rs = ring[n % kPipe][0];
      sq[n & 1][tid] = phi(to_f(rs[tid]));
      sk[n & 1][tid] = phi(to_f(rs[D + tid]));
      sv[n & 1][tid] = to_f(rs[2 * D + tid]);
    }
  };

  for (int n = 0; n < kPipe; ++n) issue(n);
  cp_async_wait<kPipe - 2>();  // tokens 0 and 1
  __syncthreads();
  prep(0);

  float sc[RPT], r[RPT];  // S_i and R = P_i + m_ii S_i at rows g + G j, column e
  float zc = 0.f, zeta = 0.f, mii = 0.f;  // threads tid < D: z_i and sum_{b<i} m_ib z_b of row tid
  int cur = -1;                           // the block the registers hold
  for (int n = 0; n < T_steps; ++n) {
    const int t = t0 + n, bi = t / block;
    if (bi != cur) {
      // block bi starts (or the call starts inside it): its running summary (zero at its
      // first token, else the slot's), and P_bi from the frozen summaries
      const bool fresh = t % block == 0;
      mii = mh[(size_t)bi * M + bi];
      float p[RPT];
#pragma unroll
      for (int j = 0; j < RPT; ++j) p[j] = 0.f;
      float pz = 0.f;
      for (int b = 0; b < bi; ++b) {  // the RPT loads of a block are independent
        const float w = mh[(size_t)bi * M + b];
        const float* sb = Su + (size_t)b * D * D + e;
#pragma unroll
        for (int j = 0; j < RPT; ++j) p[j] = fmaf(w, sb[(size_t)(g + G * j) * D], p[j]);
        if (tid < D) pz = fmaf(w, zu[(size_t)b * D + tid], pz);
      }
#pragma unroll
      for (int j = 0; j < RPT; ++j) {
        sc[j] = fresh ? 0.f : Su[((size_t)bi * D + g + G * j) * D + e];
        r[j] = fmaf(mii, sc[j], p[j]);
      }
      if (tid < D) {
        zeta = pz;
        zc = fresh ? 0.f : zu[(size_t)bi * D + tid];
      }
      cur = bi;
    }
    cp_async_wait<kPipe - 2>();  // token n + 1 copied (this thread's chunks)
    __syncthreads();             // token n's phi and token n + 1's rows visible; token n - 1 done
    if (n + 1 < T_steps) prep(n + 1);
    issue(n + kPipe);            // into token n's stage, read by prep(n) before this barrier
    const float* pq = sq[n & 1];
    const float* pk = sk[n & 1];
    const float ve = sv[n & 1][e];
    float part = 0.f;
#pragma unroll
    for (int j = 0; j < RPT; ++j) {
      const int c = g + G * j;
      const float kc = pk[c];
      sc[j] = fmaf(kc, ve, sc[j]);
      r[j] = fmaf(mii * kc, ve, r[j]);
      part = fmaf(pq[c], r[j], part);
    }
    red[g][e] = part;
    if (tid < ((D + 31) & ~31)) {  // the warps holding z rows: warp sums of phi(q)_c (zeta_c + m_ii z_c)
      float dp = 0.f;
      if (tid < D) {
        zc += pk[tid];
        dp = pq[tid] * fmaf(mii, zc, zeta);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) dp += __shfl_xor_sync(0xffffffffu, dp, o);
      if ((tid & 31) == 0) sden[tid >> 5] = dp;
    }
    __syncthreads();
    if (tid < D) {
      float den = 0.f;
#pragma unroll
      for (int w = 0; w < (D + 31) / 32; ++w) den += sden[w];
      den += eps;
      float num = 0.f;
#pragma unroll
      for (int gg = 0; gg < G; ++gg) num += red[gg][tid];
      const size_t row = (size_t)n * tstride + (size_t)u * D;
      out[row + tid] = from_f<T>(num / den);
      if (den_out != nullptr && tid == 0) den_out[(size_t)n * units + u] = den;
    }
    if (t % block == block - 1 || n == T_steps - 1) {
      // the block is finished (frozen from now on) or the call ends inside it: its slot
#pragma unroll
      for (int j = 0; j < RPT; ++j) Su[((size_t)bi * D + g + G * j) * D + e] = sc[j];
      if (tid < D) zu[(size_t)bi * D + tid] = zc;
      __syncthreads();  // the next block's P reads this slot
    }
  }
  cp_async_wait<0>();
}

template <typename T, int D>
cudaError_t stream_t(const void* q, const void* k, const void* v, const float* mixing, float* S, float* z,
                     void* out, float* den_out, int t0, int T_steps, int units, int H, int block, int M, float eps,
                     cudaStream_t st) {
  causal_stream_kernel<T, D><<<units, StreamGeom<D>::NT, 0, st>>>(
      static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v), mixing, S, z,
      static_cast<T*>(out), den_out, t0, T_steps, units, H, block, M, eps);
  note_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t causal_stream_launch(int t0, int T_steps, int units, int H, int d, int block, int M, mhla_dtype dt,
                                 const void* q, const void* k, const void* v, const float* mixing, float* S,
                                 float* z, void* out, float* den_out, float eps, cudaStream_t st) {
#define MHLA_STREAM_CASE(DV)                                                                              \
  case DV:                                                                                               \
    return dt == MHLA_F32 ? stream_t<float, DV>(q, k, v, mixing, S, z, out, den_out, t0, T_steps, units, H, \
                                                block, M, eps, st)                                          \
                          : stream_t<__nv_bfloat16, DV>(q, k, v, mixing, S, z, out, den_out, t0, T_steps,   \
                                                        units, H, block, M, eps, st);
  switch (d) {
    MHLA_STREAM_CASE(16)
    MHLA_STREAM_CASE(32)
    MHLA_STREAM_CASE(64)
    MHLA_STREAM_CASE(128)
    default: return cudaErrorInvalidValue;
  }
#undef MHLA_STREAM_CASE
}

}  // namespace mhla
