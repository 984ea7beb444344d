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
// d = 128: one CTA per (batch, head) unit walks the call's tokens in order (their rows
// arrive through a cp.async ring several tokens ahead; phi of token n + 1 is
// taken while token n is computed).  Its
// threads hold the unit's running summary S_i and the mixed state
// R = P_i + m_ii S_i, P_i = sum_{b<i} m_ib S_b, in registers (thread (g, e)
// owns column e of rows g, g + G, ...); P_i is formed from the frozen
// summaries in memory when block i starts, so a token costs three d^2 FMAs
// (S_i, R, and the output) whatever i is.  A finished block's summary is
// written back to its slot.
//
// d <= 64: a warp per (unit, 32-column slab) instead (below), with the same registers
// per column and no barrier wider than the warp.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace mhla {
namespace {

template <int D> struct StreamGeom {
  static constexpr int NT = D == 128 ? 512 : 256;  // threads
  static constexpr int G = NT / D;                 // row groups
  static constexpr int RPT = D / G;                // rows per thread
};

constexpr int kPipe = 8;      // tokens in flight in the cp.async ring
constexpr int kMixGroup = 8;  // premix: blocks accumulated per pass over the frozen slots
constexpr int kMixRows = 8;   // premix: rows of a lane's column per accumulator

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

// ------------------------------------------------------------------------------------------
// d <= 64: a warp per (unit, 32-column slab).  Lane e holds column e of both the running summary
// S_i and the mixed state R = P_i + m_ii S_i, as row pairs (packed fp32x2 FMAs update two rows
// at once), so a warp needs nothing from any other warp: each slab warp also keeps the whole z
// (rows lane + 32 j) and its own denominator.  The step's rows come through a per-warp cp.async
// ring; phi of token n + 1 is taken while token n is computed (within a block).  At call start
// the frozen part of the mixed state of every block starting inside the call is premixed into that
// block's slot, so each frozen slot is read once per call.
template <int D> struct WarpGeom {
  static constexpr int LA = D < 32 ? D : 32;   // lanes holding a column
  static constexpr int SL = D / LA;            // slab warps per unit
  static constexpr int RZ = (D + 31) / 32;     // z rows per lane
  static constexpr int WARPS = 4;              // warps per CTA
};

template <typename T, int D>
__global__ void __launch_bounds__(WarpGeom<D>::WARPS * 32, 12 / WarpGeom<D>::WARPS)
causal_stream_warp_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                          const float* __restrict__ mixing, float* __restrict__ S, float* __restrict__ z,
                          T* __restrict__ out, float* __restrict__ den_out, int t0, int T_steps, int units, int H,
                          int block, int M, float eps) {
  using G = WarpGeom<D>;
  constexpr int LA = G::LA, SL = G::SL, RZ = G::RZ, WARPS = G::WARPS;
  constexpr int QC = D * (int)sizeof(T) / 16;   // 16-byte chunks of a q or k row
  constexpr int VCH = LA * (int)sizeof(T) / 16; // 16-byte chunks of the slab's v columns
  constexpr int NCH = 2 * QC + VCH;
  constexpr int NI = (NCH + 31) / 32;
  constexpr int STAGE = 2 * D + LA;
  static_assert(QC >= 1 && VCH >= 1 && D % 4 == 0, "whole 16-byte chunks");
  static_assert(D % kMixRows == 0, "premix row chunks");

  __shared__ __align__(16) T ring[WARPS][kPipe][STAGE];
  __shared__ __align__(16) float phq[WARPS][2][D];
  __shared__ __align__(16) float phk[WARPS][2][D];

  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const long long task = (long long)blockIdx.x * WARPS + wid;
  if (T_steps <= 0 || task >= (long long)units * SL) return;  // no block-wide barrier in this kernel
  const int u = (int)(task / SL), slab = (int)(task % SL);
  const int e = slab * LA + lane;             // this lane's column
  const bool owns = LA == 32 || lane < LA;
  const int ec = owns ? e : 0;                // a valid column for the idle lanes' dummy loads
  const float* mh = mixing + (size_t)(u % H) * M * M;
  float* Su = S + (size_t)u * M * D * D;
  float* zu = z + (size_t)u * M * D;

  // ---- ring of the call's tokens: token n at stage n % kPipe (past the end: the last token again)
  const size_t tstride = (size_t)units * D * sizeof(T);
  const char* src[NI];
  uint32_t dst_off[NI];
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const int c = lane + 32 * i;
    const size_t row = (size_t)u * D;
    const T* base = c < QC ? q + row : c < 2 * QC ? k + row : v + row + slab * LA;
    const int cc = c < QC ? c : c < 2 * QC ? c - QC : c - 2 * QC;
    src[i] = reinterpret_cast<const char*>(base) + cc * 16;
    dst_off[i] = (uint32_t)(c * 16);
  }
  char* ring_w = reinterpret_cast<char*>(ring[wid][0]);
  auto issue = [&](int n) {
    const int nn = n < T_steps ? n : T_steps - 1;
    char* dst = ring_w + (n % kPipe) * (STAGE * (int)sizeof(T));
#pragma unroll
    for (int i = 0; i < NI; ++i)
      if (lane + 32 * i < NCH) cp_async16(dst + dst_off[i], src[i] + (size_t)nn * tstride);
    cp_async_commit();
  };

  float2 rp[D / 2], sp[D / 2];  // R and S_i of column e, rows (2p, 2p + 1)
  float zr[RZ], zc[RZ];          // rows lane + 32 j: zeta_i + m_ii z_i, and z_i
  float mii = 0.f;
  int cur = -1;

  // phi of token n, its v and the denominator with this block's weights
  auto prep = [&](int n, float& vv, float& den) {
    const T* rq = ring[wid][n % kPipe];
    const T* rk = rq + D;
    const T* rv = rq + 2 * D;
    float part = 0.f;
#pragma unroll
    for (int j = 0; j < RZ; ++j) {
      const int c = lane + 32 * j;
      if (c < D) {
        const float fq = tc::phi_f(to_f(rq[c])), fk = tc::phi_f(to_f(rk[c]));
        phq[wid][n & 1][c] = fq;
        phk[wid][n & 1][c] = fk;
        zc[j] += fk;
        zr[j] = fmaf(mii, fk, zr[j]);
        part = fmaf(fq, zr[j], part);
      }
    }
    vv = owns ? to_f(rv[lane]) : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    den = part + eps;
  };

  for (int n = 0; n < kPipe - 1; ++n) issue(n);
  cp_async_wait<kPipe - 2>();  // token 0
  __syncwarp();

  // ---- the frozen part of the mixed state of every block that starts inside the call,
  // sum_{b<F} m_ib S_b over the F slots frozen before it, into that block's own slot (free until
  // the block ends): each frozen slot is read once per call instead of once per block start.
  // A lane reads and writes only its own column, so no other lane is involved.
  const int F = t0 / block;
  const int first_fresh = t0 % block == 0 ? F : F + 1;
  const int last_blk = (t0 + T_steps - 1) / block;
  const bool premix = F > 0 && first_fresh <= last_blk;
  if (premix) {
    for (int i0 = first_fresh; i0 <= last_blk; i0 += kMixGroup) {
      const int ni = min(kMixGroup, last_blk + 1 - i0);
      const float* wrow = mh + (size_t)i0 * M;
      for (int r0 = 0; r0 < D; r0 += kMixRows) {
        float acc[kMixGroup][kMixRows];
#pragma unroll
        for (int ii = 0; ii < kMixGroup; ++ii)
#pragma unroll
          for (int rr = 0; rr < kMixRows; ++rr) acc[ii][rr] = 0.f;
#pragma unroll 2
        for (int b = 0; b < F; ++b) {
          const float* sb = Su + ((size_t)b * D + r0) * D + ec;
          float val[kMixRows];
#pragma unroll
          for (int rr = 0; rr < kMixRows; ++rr) val[rr] = __ldcg(sb + (size_t)rr * D);
#pragma unroll
          for (int ii = 0; ii < kMixGroup; ++ii) {
            const float w = ii < ni ? __ldg(wrow + (size_t)ii * M + b) : 0.f;
#pragma unroll
            for (int rr = 0; rr < kMixRows; ++rr) acc[ii][rr] = fmaf(w, val[rr], acc[ii][rr]);
          }
        }
        if (owns) {
#pragma unroll
          for (int ii = 0; ii < kMixGroup; ++ii)
            if (ii < ni) {
#pragma unroll
              for (int rr = 0; rr < kMixRows; ++rr) Su[((size_t)(i0 + ii) * D + r0 + rr) * D + e] = acc[ii][rr];
            }
        }
      }
#pragma unroll
      for (int j = 0; j < RZ; ++j) {
        const int c = lane + 32 * j;
        if (c < D) {
          float az[kMixGroup];
#pragma unroll
          for (int ii = 0; ii < kMixGroup; ++ii) az[ii] = 0.f;
          for (int b = 0; b < F; ++b) {
            const float zb = __ldcg(zu + (size_t)b * D + c);
#pragma unroll
            for (int ii = 0; ii < kMixGroup; ++ii)
              az[ii] = fmaf(ii < ni ? __ldg(wrow + (size_t)ii * M + b) : 0.f, zb, az[ii]);
          }
          // every slab warp writes the same values (each reads back only what it wrote)
#pragma unroll
          for (int ii = 0; ii < kMixGroup; ++ii)
            if (ii < ni) zu[(size_t)(i0 + ii) * D + c] = az[ii];
        }
      }
    }
  }

  bool have = false;  // token n's prep done (in the previous iteration)
  float vv = 0.f, den = 1.f;
  for (int n = 0; n < T_steps; ++n) {
    const int t = t0 + n, bi = t / block;
    if (bi != cur) {
      // block bi starts (or the call starts inside it): S_i from its slot (zero at its first
      // token), R = sum_{b<i} m_ib S_b + m_ii S_i, z likewise.  A block that starts inside the
      // call finds the frozen part of its sum in its slot when the call premixed it, and adds
      // the blocks finished during the call; otherwise every earlier slot is mixed here.
      const bool fresh = t % block == 0;
      const bool pre = fresh && premix;
      mii = __ldg(mh + (size_t)bi * M + bi);
#pragma unroll
      for (int pp = 0; pp < D / 2; ++pp) {
        const float2 slot = (fresh && !pre) ? make_float2(0.f, 0.f)
                                            : make_float2(Su[((size_t)bi * D + 2 * pp) * D + ec],
                                                          Su[((size_t)bi * D + 2 * pp + 1) * D + ec]);
        sp[pp] = fresh ? make_float2(0.f, 0.f) : slot;
        rp[pp] = pre ? slot : make_float2(mii * slot.x, mii * slot.y);
      }
#pragma unroll
      for (int j = 0; j < RZ; ++j) {
        const int c = lane + 32 * j;
        const float zs = ((fresh && !pre) || c >= D) ? 0.f : zu[(size_t)bi * D + c];
        zc[j] = fresh ? 0.f : zs;
        zr[j] = pre ? zs : mii * zs;
      }
      for (int b = pre ? F : 0; b < bi; ++b) {
        const float w = __ldg(mh + (size_t)bi * M + b);
        const float* sb = Su + (size_t)b * D * D + ec;
#pragma unroll
        for (int pp = 0; pp < D / 2; ++pp) {
          rp[pp].x = fmaf(w, __ldcg(sb + (size_t)(2 * pp) * D), rp[pp].x);
          rp[pp].y = fmaf(w, __ldcg(sb + (size_t)(2 * pp + 1) * D), rp[pp].y);
        }
#pragma unroll
        for (int j = 0; j < RZ; ++j) {
          const int c = lane + 32 * j;
          if (c < D) zr[j] = fmaf(w, __ldcg(zu + (size_t)b * D + c), zr[j]);
        }
      }
      cur = bi;
      have = false;
    }
    if (!have) prep(n, vv, den);  // its rows have landed (the previous wait) and are visible
    const float v0 = vv, d0 = den;
    issue(n + kPipe - 1);          // into token n - 1's stage (read before the last barrier)
    cp_async_wait<kPipe - 2>();    // token n + 1 copied (this lane's chunks)
    __syncwarp();                  // every lane's copies and phi writes visible; token n - 1's reads done
    have = n + 1 < T_steps && (t + 1) / block == bi;
    if (have) prep(n + 1, vv, den);

    const float* pq = phq[wid][n & 1];
    const float* pk = phk[wid][n & 1];
    const float mv = mii * v0;
    const float2 v2 = make_float2(v0, v0), mv2 = make_float2(mv, mv);
    float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int c4 = 0; c4 < D; c4 += 4) {
      const float4 k4 = *reinterpret_cast<const float4*>(pk + c4);
      const float4 q4 = *reinterpret_cast<const float4*>(pq + c4);
      const float2 ka = make_float2(k4.x, k4.y), kb = make_float2(k4.z, k4.w);
      sp[c4 / 2] = __ffma2_rn(ka, v2, sp[c4 / 2]);
      sp[c4 / 2 + 1] = __ffma2_rn(kb, v2, sp[c4 / 2 + 1]);
      rp[c4 / 2] = __ffma2_rn(ka, mv2, rp[c4 / 2]);
      rp[c4 / 2 + 1] = __ffma2_rn(kb, mv2, rp[c4 / 2 + 1]);
      acc0 = __ffma2_rn(make_float2(q4.x, q4.y), rp[c4 / 2], acc0);
      acc1 = __ffma2_rn(make_float2(q4.z, q4.w), rp[c4 / 2 + 1], acc1);
    }
    const size_t row = (size_t)n * units + u;
    if (owns) out[row * D + e] = from_f<T>(__fdividef((acc0.x + acc0.y) + (acc1.x + acc1.y), d0));
    if (den_out != nullptr && slab == 0 && lane == 0) den_out[row] = d0;
    if (t % block == block - 1 || n == T_steps - 1) {
      // the block is finished (frozen from now on) or the call ends inside it: its slot (every
      // slab writes the same z, so that each reads back only values it wrote)
      if (owns) {
#pragma unroll
        for (int pp = 0; pp < D / 2; ++pp) {
          Su[((size_t)bi * D + 2 * pp) * D + e] = sp[pp].x;
          Su[((size_t)bi * D + 2 * pp + 1) * D + e] = sp[pp].y;
        }
      }
#pragma unroll
      for (int j = 0; j < RZ; ++j) {
        const int c = lane + 32 * j;
        if (c < D) zu[(size_t)bi * D + c] = zc[j];
      }
    }
  }
  cp_async_wait<0>();
}

template <typename T, int D>
cudaError_t stream_t(const void* q, const void* k, const void* v, const float* mixing, float* S, float* z,
                     void* out, float* den_out, int t0, int T_steps, int units, int H, int block, int M, float eps,
                     cudaStream_t st) {
  if constexpr (D <= 64) {
    using G = WarpGeom<D>;
    const long long blocks = ((long long)units * G::SL + G::WARPS - 1) / G::WARPS;
    causal_stream_warp_kernel<T, D><<<(unsigned)blocks, G::WARPS * 32, 0, st>>>(
        static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v), mixing, S, z,
        static_cast<T*>(out), den_out, t0, T_steps, units, H, block, M, eps);
  } else {
    causal_stream_kernel<T, D><<<units, StreamGeom<D>::NT, 0, st>>>(
        static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v), mixing, S, z,
        static_cast<T*>(out), den_out, t0, T_steps, units, H, block, M, eps);
  }
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
