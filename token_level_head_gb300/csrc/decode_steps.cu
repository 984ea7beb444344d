// Fused multi-step recurrent decode ("Linear Attention notes" §四 recurrence,
// §七 RetNet decay, §八 fixed-size state).
//
// T consecutive steps for every (batch, head) unit in one launch.  A warp owns
// one unit (or, for d = 128, a 32-column slab of it: four warps per unit) and
// keeps its columns of the fp32 state S in registers for all T steps, so the
// state is read from and written to memory once per call instead of once per
// step.  Per step the warp
//   - takes the step's q, k (all d) and v (its columns) from a per-warp shared
//     memory ring that cp.async fills kPipe - 1 steps ahead;
//   - computes phi(q), phi(k) (each lane d/32 rows) into a per-warp buffer and
//     updates its rows of z; the denominator phi(q).z + eps is a warp sum;
//     this "prep" of step t + 1 runs in iteration t, beside step t's update;
//   - for its columns e and every row c: S[c][e] = gamma S[c][e] + phi(k)_c v_e,
//     out_e += phi(q)_c S[c][e]  (phi values read as broadcast float4 loads),
//     two rows per packed fp32x2 FMA (rows 2p and 2p+1 share a register pair);
//   - writes out_e / den and the denominator.
// 2 d^2 FMAs per unit and step (plus d^2 multiplies with decay), issued as d^2
// packed instructions.  With 128 state registers per lane (d = 64) a warp's
// step is latency-bound (shared-memory broadcasts, the warp sum, the
// exponentials); three warps per scheduler hide part of it.

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace mhla {
namespace {

constexpr int kDecodeWarps = 4;  // warps per CTA for d < 128 (d = 128: one unit per CTA)
constexpr int kPipe = 8;         // ring stages: steps in flight ahead of the one computed

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

template <typename T> __device__ __forceinline__ void store_cols(T* p, const float* x, int n);
template <>
__device__ __forceinline__ void store_cols<float>(float* p, const float* x, int n) {
  if (n == 2) *reinterpret_cast<float2*>(p) = make_float2(x[0], x[1]);
  else p[0] = x[0];
}
template <>
__device__ __forceinline__ void store_cols<__nv_bfloat16>(__nv_bfloat16* p, const float* x, int n) {
  if (n == 2) *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(x[0], x[1]);
  else p[0] = __float2bfloat16_rn(x[0]);
}

// Geometry of one warp's task for head dimension D.
template <int D>
struct DecodeGeom {
  static constexpr int CPL = D == 64 ? 2 : 1;              // state columns per lane
  static constexpr int LA = D < 32 ? D : 32;                // lanes that own columns
  static constexpr int VC = LA * CPL;                       // columns per warp (slab width)
  static constexpr int SLABS = D / VC;                      // warps per unit
  static constexpr int R = (D + 31) / 32;                   // phi / z rows per lane
  static constexpr int WARPS = SLABS > 1 ? SLABS : kDecodeWarps;
  static_assert(VC * SLABS == D, "slabs must tile the columns");
  static_assert(SLABS == 1 || WARPS == SLABS, "a CTA holds exactly one multi-slab unit");
};

template <typename T, int D, bool DECAY>
__global__ void __launch_bounds__(DecodeGeom<D>::WARPS * 32, 12 / DecodeGeom<D>::WARPS)
decode_steps_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                    float* __restrict__ S, float* __restrict__ z, T* __restrict__ out,
                    float* __restrict__ den_out, int T_steps, int units, float eps, float gamma) {
  using G = DecodeGeom<D>;
  constexpr int CPL = G::CPL, LA = G::LA, VC = G::VC, SLABS = G::SLABS, R = G::R, WARPS = G::WARPS;
  constexpr int QC = D * (int)sizeof(T) / 16;   // 16-byte chunks of a q or k row
  constexpr int VCH = VC * (int)sizeof(T) / 16; // 16-byte chunks of the slab's v columns
  constexpr int NCH = 2 * QC + VCH;             // chunks copied per step
  constexpr int NI = (NCH + 31) / 32;           // copy rounds per lane
  constexpr int STAGE = 2 * D + VC;             // elements of one ring stage: q, k, v slab
  static_assert(QC >= 1 && VCH >= 1, "rows must be whole 16-byte chunks");
  static_assert((kPipe & (kPipe - 1)) == 0, "ring depth a power of two");

  __shared__ __align__(16) T ring[WARPS][kPipe][STAGE];
  __shared__ __align__(16) float phq[WARPS][2][D];
  __shared__ __align__(16) float phk[WARPS][2][D];

  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const long long task = (long long)blockIdx.x * WARPS + wid;
  if (T_steps <= 0 || task >= (long long)units * SLABS) return;  // no block-wide barrier follows when SLABS == 1
  const int u = (int)(task / SLABS), slab = (int)(task % SLABS);
  const int col0 = slab * VC + lane * CPL;     // first state column of this lane
  const bool owns = LA == 32 || lane < LA;     // compile-time true unless d = 16

  // ---- the unit's state: S columns in registers as row pairs sp[p][j] = (S[2p][e], S[2p+1][e]),
  // e = col0 + j (packed fp32x2 FMAs then update two rows per instruction); z rows (every
  // slab keeps all of z)
  float2 sp[D / 2][CPL];
  float zr[R];
  float* Su = S + (size_t)u * D * D;
  float* zu = z + (size_t)u * D;
#pragma unroll
  for (int p = 0; p < D / 2; ++p)
#pragma unroll
    for (int j = 0; j < CPL; ++j)
      sp[p][j] = owns ? make_float2(Su[(size_t)(2 * p) * D + col0 + j], Su[(size_t)(2 * p + 1) * D + col0 + j])
                      : make_float2(0.f, 0.f);
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const int c = lane + 32 * i;
    zr[i] = c < D ? zu[c] : 0.f;
  }
  if constexpr (SLABS > 1) __syncthreads();  // every slab has read z before slab 0 may write it

  // ---- this lane's copy chunks: source address at step 0 and ring offset; a step adds `stride`
  const size_t stride = (size_t)units * D * sizeof(T);
  const char* src[NI];
  uint32_t dst_off[NI];
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const int c = lane + 32 * i;
    const size_t row = (size_t)u * D;
    const T* base = c < QC ? q + row : c < 2 * QC ? k + row : v + row + slab * VC;
    const int cc = c < QC ? c : c < 2 * QC ? c - QC : c - 2 * QC;
    src[i] = reinterpret_cast<const char*>(base) + cc * 16;
    dst_off[i] = (uint32_t)(c * 16);
  }
  char* ring_w = reinterpret_cast<char*>(ring[wid][0]);
  // Copies step tt into its ring stage; past the last step it copies the last step again (a
  // stage no later step uses), so that the issue needs no branch.
  auto issue = [&](int tt) {
    const int ts = tt < T_steps ? tt : T_steps - 1;
    char* dst = ring_w + (tt & (kPipe - 1)) * (STAGE * (int)sizeof(T));
#pragma unroll
    for (int i = 0; i < NI; ++i)
      if (lane + 32 * i < NCH) cp_async16(dst + dst_off[i], src[i] + (size_t)ts * stride);
    cp_async_commit();  // one group per step, so the wait count stays fixed
  };
#pragma unroll
  for (int tt = 0; tt < kPipe - 1; ++tt) issue(tt);

  T* out_p = out + (size_t)u * D + col0;
  const size_t out_stride = (size_t)units * D;
  // Step t's phi values, z update and denominator ("prep") do not depend on the state
  // update of step t - 1, so iteration t preps step t + 1 while it updates the state for
  // step t: the exponentials and the warp sum overlap the FMAs.  phi buffers alternate.
  // Prep of step tt: phi(q), phi(k) into the phi buffer of its parity, the z update and the
  // denominator phi(q).z + eps (a warp sum).  It does not depend on the state update of step
  // tt - 1, and it runs unconditionally (past the last step on stale ring data, with `live`
  // false so that z keeps its value), so that the compiler can interleave it with that update.
  auto prep = [&](int tt, bool live, float (&vv)[CPL], float& den) {
    const T* rq = ring[wid][tt & (kPipe - 1)];
    const T* rk = rq + D;
    const T* rv = rq + 2 * D;
    float* pq = phq[wid][tt & 1];
    float* pk = phk[wid][tt & 1];
    float part = 0.f;
#pragma unroll
    for (int i = 0; i < R; ++i) {
      const int c = lane + 32 * i;
      if (c < D) {
        const float fq = tc::phi_f(to_f(rq[c])), fk = tc::phi_f(to_f(rk[c]));
        pq[c] = fq;
        pk[c] = fk;
        const float zn = DECAY ? fmaf(zr[i], gamma, fk) : zr[i] + fk;
        zr[i] = live ? zn : zr[i];
        part = fmaf(fq, zn, part);
      }
    }
#pragma unroll
    for (int j = 0; j < CPL; ++j) vv[j] = owns ? to_f(rv[lane * CPL + j]) : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    den = part + eps;
  };

  float vv_next[CPL], den_next = 1.f;
  if (T_steps > 0) {
    cp_async_wait<kPipe - 2>();  // step 0 copied (this lane's chunks)
    __syncwarp();                // and every lane's
    prep(0, true, vv_next, den_next);
  }
  const float2 g2 = make_float2(gamma, gamma);
  for (int t = 0; t < T_steps; ++t) {
    float2 v2[CPL];
#pragma unroll
    for (int j = 0; j < CPL; ++j) v2[j] = make_float2(vv_next[j], vv_next[j]);
    const float den = den_next;
    issue(t + kPipe - 1);        // into the stage of step t - 1, whose prep ended two iterations ago
    cp_async_wait<kPipe - 2>();  // step t + 1 copied (this lane's chunks)
    __syncwarp();                // every lane's copies and phi writes of step t visible; step t - 1's
                                 // reads of the other phi buffer done
    prep(t + 1, t + 1 < T_steps, vv_next, den_next);

    // S_t = gamma S_{t-1} + phi(k) v^T, then out = phi(q) S_t / den
    const float* pq = phq[wid][t & 1];
    const float* pk = phk[wid][t & 1];
    float2 acc[CPL][2];  // two independent row-pair accumulation chains per column
#pragma unroll
    for (int j = 0; j < CPL; ++j) acc[j][0] = acc[j][1] = make_float2(0.f, 0.f);
    if (owns) {
#pragma unroll
      for (int c4 = 0; c4 < D; c4 += 4) {
        const float4 k4 = *reinterpret_cast<const float4*>(pk + c4);
        const float4 q4 = *reinterpret_cast<const float4*>(pq + c4);
        const float2 kp[2] = {make_float2(k4.x, k4.y), make_float2(k4.z, k4.w)};
        const float2 qp[2] = {make_float2(q4.x, q4.y), make_float2(q4.z, q4.w)};
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int j = 0; j < CPL; ++j) {
            float2& sc = sp[c4 / 2 + h][j];
            sc = DECAY ? __ffma2_rn(g2, sc, __fmul2_rn(kp[h], v2[j])) : __ffma2_rn(kp[h], v2[j], sc);
          }
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int j = 0; j < CPL; ++j) acc[j][h] = __ffma2_rn(qp[h], sp[c4 / 2 + h][j], acc[j][h]);
      }
      float o[CPL];
#pragma unroll
      for (int j = 0; j < CPL; ++j) {
        o[j] = __fdividef((acc[j][0].x + acc[j][0].y) + (acc[j][1].x + acc[j][1].y), den);
      }
      store_cols<T>(out_p + (size_t)t * out_stride, o, CPL);
    }
    if (den_out != nullptr && slab == 0 && lane == 0) den_out[(size_t)t * units + u] = den;
  }
  cp_async_wait<0>();

  // ---- state back
  if (owns) {
#pragma unroll
    for (int p = 0; p < D / 2; ++p) {
      float lo[CPL], hi[CPL];
#pragma unroll
      for (int j = 0; j < CPL; ++j) {
        lo[j] = sp[p][j].x;
        hi[j] = sp[p][j].y;
      }
      store_cols<float>(Su + (size_t)(2 * p) * D + col0, lo, CPL);
      store_cols<float>(Su + (size_t)(2 * p + 1) * D + col0, hi, CPL);
    }
  }
  if (slab == 0) {
#pragma unroll
    for (int i = 0; i < R; ++i) {
      const int c = lane + 32 * i;
      if (c < D) zu[c] = zr[i];
    }
  }
}

template <typename T, int D>
cudaError_t decode_steps_t(int T_steps, int units, const void* q, const void* k, const void* v, float* S,
                           float* z, void* out, float* den_out, float eps, float gamma, cudaStream_t st) {
  using G = DecodeGeom<D>;
  const long long tasks = (long long)units * G::SLABS;
  const long long blocks = (tasks + G::WARPS - 1) / G::WARPS;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  const auto* tq = static_cast<const T*>(q);
  const auto* tk = static_cast<const T*>(k);
  const auto* tv = static_cast<const T*>(v);
  auto* to = static_cast<T*>(out);
  if (gamma == 1.f)
    decode_steps_kernel<T, D, false><<<(unsigned)blocks, G::WARPS * 32, 0, st>>>(
        tq, tk, tv, S, z, to, den_out, T_steps, units, eps, gamma);
  else
    decode_steps_kernel<T, D, true><<<(unsigned)blocks, G::WARPS * 32, 0, st>>>(
        tq, tk, tv, S, z, to, den_out, T_steps, units, eps, gamma);
  note_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t decode_steps_launch(int T_steps, int units, int d, mhla_dtype dt, const void* q, const void* k,
                                const void* v, float* S, float* z, void* out, float* den_out, float eps,
                                float gamma, cudaStream_t st) {
#define MHLA_DECODE_CASE(DV)                                                                          \
  case DV:                                                                                           \
    return dt == MHLA_F32 ? decode_steps_t<float, DV>(T_steps, units, q, k, v, S, z, out, den_out,   \
                                                      eps, gamma, st)                                 \
                          : decode_steps_t<__nv_bfloat16, DV>(T_steps, units, q, k, v, S, z, out,     \
                                                              den_out, eps, gamma, st);
  switch (d) {
    MHLA_DECODE_CASE(16)
    MHLA_DECODE_CASE(32)
    MHLA_DECODE_CASE(64)
    MHLA_DECODE_CASE(128)
    default: return cudaErrorInvalidValue;
  }
#undef MHLA_DECODE_CASE
}

}  // namespace mhla
