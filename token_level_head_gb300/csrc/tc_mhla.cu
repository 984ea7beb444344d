// bf16 MHLA forward on the sm_103a tensor cores: one persistent kernel per call.
//
// "MHLA: Restoring Expressivity of Linear Attention via Token-Level
// Multi-Head" §4.1 computes, per (batch, head):
//   S_b = sum_{t in b} phi(K_t) V_t^T,  z_b = sum_{t in b} phi(K_t)       (local KV summaries)
//   S~_i = sum_b m_ib S_b,  z~_i = sum_b m_ib z_b                          (multi-head mixing)
//   Y_t = phi(Q_t) S~_i / (phi(Q_t) . z~_i + eps)                           (output)
// with phi = ELU + 1 and eps from "Linear Attention notes" §四/§五.
//
// Work is split into units handed out by a global ticket counter:
//   SUM (head, 128-token chunk): TMA K, V tiles -> phi(K) in smem -> one
//       tcgen05.mma chain D = V^T phi(K) (M = N = 64, K = 128) gives the
//       chunk's S^T partial in TMEM; z partial by a CUDA-core reduction.
//       fp32 partials to L2, one contiguous 128-byte row per thread.
//   MIX (head, slice of the 64*64+64 summary entries): sums the partials of
//       each block and mixes them for every query block; writes S~ (bf16, in
//       the K-major layout the output MMA reads) and z~ (fp32).  Four entries
//       per thread (float4), G threads per 4-entry vector chosen on the host.
//       The MIX units of head h are placed in the ticket order a few heads
//       after its SUM units, so they run while other CTAs keep streaming.
//   OUT (head, 128-token tile): TMA Q tile -> phi(Q) in smem and the fp32
//       denominator phi(Q) . z~ on CUDA cores -> tcgen05.mma (M = 128,
//       N = 64, K = 64) against S~ -> divide in registers -> bf16 -> TMA store.
// A unit only ever waits (bounded) on units with smaller tickets, which are
// held by running CTAs, so there is no deadlock whatever the residency.
// Each CTA prefetches the next unit's TMA inputs as soon as its tensor-core
// work has consumed the current ones.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace mhla {
namespace {

using namespace tc;

constexpr int kThreads = 256;
constexpr int kTile = 128;                   // tokens per SUM / OUT unit
constexpr int kD = 64;                       // head dimension of this kernel
constexpr int kTileBytes = kTile * kD * 2;   // 16 KB bf16 tile
constexpr int kSTileBytes = kD * kD * 2;     // 8 KB bf16 S~ tile
constexpr int kEnt = kD * kD + kD;           // summary entries: S^T (e*64 + c), then z
constexpr int kCtasPerSm = 3;
constexpr uint32_t kTmemCols = 64;
constexpr uint32_t kSpinBudget = 1u << 24;
constexpr int kMixBytes = 16384;             // MIX staging: at most 1024 float4

enum { UNIT_SUM = 0, UNIT_MIX = 1, UNIT_OUT = 2 };

struct Params {
  CUtensorMap tm_q, tm_k, tm_v, tm_y;  // [heads*N rows][64] bf16, box 64 x 128
  CUtensorMap tm_s;                    // S~ [heads*M*64 rows][64] bf16, box 64 x 64
  const float* mixing;                 // [H][M][M]
  float* s_part;                       // [heads][C][64 e][64 c]
  float* z_part;                       // [heads][C][64]
  __nv_bfloat16* s_mix;                // [heads][M][64 e][64 c]
  float* z_mix;                        // [heads][M][64]
  float* den_out;                      // [heads][N] or null
  unsigned* ctr;                       // ticket, finished, sum_done[heads], mix_done[heads]
  unsigned* status;
  int heads, H, N, M, C, cpb;          // C = chunks per head, cpb = chunks per block
  int L, I, T1, total;                 // lag (heads), MIX items per head, tickets before OUT, all
  int G, nvec, split;                  // MIX: threads per vector, vectors per item, threads per block (G >= M)
  float eps;
  int mode;                            // MixMode
};

struct Small {
  float zt[kD];              // z~ of the current OUT tile (bulk-copied; 16-byte aligned)
  float den_half[2][kTile];
  float zred[8][kD];
  uint64_t bar_in, bar_s, bar_mma;
  uint32_t tbase;
  int next;
  int flag;
  int s_ticket;              // OUT ticket whose S~ / z~ loads are already in flight on bar_s
  int s_inflight;            // 1 while a bar_s load has been issued and not yet waited for
};

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ bool wait_geq(const unsigned* p, unsigned target) {
  for (uint32_t it = 0; it < kSpinBudget; ++it) {
    if (ld_acquire(p) >= target) return true;
    __nanosleep(it < 16 ? 32 : 256);
  }
  return false;
}

// Every thread waits (bounded) and the CTA agrees on the outcome, so a time-out
// can never leave some threads at a barrier the others skipped.
__device__ __forceinline__ bool cta_wait(uint64_t* bar, uint32_t parity) {
  return __syncthreads_and(mbar_wait(bar, parity) ? 1 : 0) != 0;
}

__device__ __forceinline__ float phi_fast(float x) { return x > 0.f ? x + 1.f : __expf(x); }

struct Unit {
  int kind, h, idx;
};

// Ticket order: rounds r = 0 .. heads+L-1, round r = [SUM units of head r]
// [MIX items of head r-L], then every OUT unit head by head.  A MIX item of
// head h only waits for SUM units of head h and an OUT unit only for MIX
// items of its head: always smaller tickets.
__device__ __forceinline__ Unit decode(const Params& p, int t) {
  Unit u;
  if (t >= p.T1) {
    const int o = t - p.T1;
    u.kind = UNIT_OUT;
    u.h = o / p.C;
    u.idx = o - u.h * p.C;
    return u;
  }
  const int head_sum = p.L * p.C;
  if (t < head_sum) {
    u.kind = UNIT_SUM;
    u.h = t / p.C;
    u.idx = t - u.h * p.C;
    return u;
  }
  const int t2 = t - head_sum;
  const int mid = (p.heads - p.L) * (p.C + p.I);
  if (t2 < mid) {
    const int r = t2 / (p.C + p.I), off = t2 - r * (p.C + p.I);
    if (off < p.C) {
      u.kind = UNIT_SUM;
      u.h = p.L + r;
      u.idx = off;
    } else {
      u.kind = UNIT_MIX;
      u.h = r;
      u.idx = off - p.C;
    }
    return u;
  }
  const int t3 = t2 - mid;
  u.kind = UNIT_MIX;
  u.h = p.heads - p.L + t3 / p.I;
  u.idx = t3 - (u.h - (p.heads - p.L)) * p.I;
  return u;
}

// Thread 0: S~ tile and z~ of OUT ticket t (its head's mixing is complete).
__device__ __forceinline__ void issue_mix_loads(const Params& p, int t, uint8_t* regC, Small* sh) {
  const Unit u = decode(p, t);
  const int blk = (u.idx * kTile) / (p.N / p.M);
  const size_t sidx = (size_t)u.h * p.M + blk;
  fence_proxy_async_global();
  mbar_arrive_expect_tx(&sh->bar_s, kSTileBytes + kD * 4);
  tma_load_2d(regC, &p.tm_s, 0, (int)(sidx * kD), &sh->bar_s);
  bulk_load_1d(sh->zt, p.z_mix + sidx * kD, kD * 4, &sh->bar_s);
  sh->s_ticket = t;
  sh->s_inflight = 1;
}

// Thread 0: issues the TMA loads a unit needs at its start (none for MIX);
// for an OUT unit also its S~ / z~ if that head's mixing is already done.
__device__ __forceinline__ void issue_inputs(const Params& p, int t, uint8_t* regA, uint8_t* regB,
                                             uint8_t* regC, Small* sh) {
  const Unit u = decode(p, t);
  const int row = u.h * p.N + u.idx * kTile;
  if (u.kind == UNIT_SUM) {
    mbar_arrive_expect_tx(&sh->bar_in, 2 * kTileBytes);
    tma_load_2d(regA, &p.tm_k, 0, row, &sh->bar_in);
    tma_load_2d(regB, &p.tm_v, 0, row, &sh->bar_in);
  } else if (u.kind == UNIT_OUT) {
    mbar_arrive_expect_tx(&sh->bar_in, kTileBytes);
    tma_load_2d(regA, &p.tm_q, 0, row, &sh->bar_in);
    if (ld_acquire(&p.ctr[2 + p.heads + u.h]) >= (unsigned)p.I) issue_mix_loads(p, t, regC, sh);
  }
}

__device__ __forceinline__ bool has_inputs(const Params& p, int t) {
  return t < p.total && decode(p, t).kind != UNIT_MIX;
}

__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ float4 f4add(float4 a, float4 b) {
  return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}

// One MIX item of head h: summary entries [item*4*nvec, +4*nvec) (S^T entries
// e*64 + c first, then the 64 z entries) for every query block i:
//   T_b = sum of the chunk partials of block b,   out_i = sum_b w_ib T_b
// with w_ib = m_ib (MIX_FULL), m_ib for b < i (MIX_STRICT_LOWER) or 1 for
// b < i (MIX_PREFIX).  Thread (g, v): vector v = 4 consecutive entries,
// g = one of the G threads sharing it.
__device__ void mix_item(const Params& p, int h, int item, float4* sT, Small* sh) {
  if (threadIdx.x == 0) sh->flag = wait_geq(&p.ctr[2 + h], (unsigned)p.C) ? 1 : 0;
  __syncthreads();
  if (!sh->flag) {
    if (threadIdx.x == 0) atomicOr(p.status, 1u);
    return;
  }
  const int nvec = p.nvec, G = p.G, M = p.M, cpb = p.cpb, split = p.split;
  const int g = threadIdx.x / nvec, v = threadIdx.x - g * nvec;
  const int ent = (item * nvec + v) * 4;
  const bool live = ent < kEnt;
  const size_t chunk0 = (size_t)h * p.C;
  const float* base = ent < kD * kD ? p.s_part + (chunk0 << 12) + ent : p.z_part + chunk0 * kD + (ent - kD * kD);
  const size_t cstride = ent < kD * kD ? (size_t)kD * kD : (size_t)kD;   // floats between chunks
  if (live) {  // phase 1: block sums (split == 0) or partial block sums (split > 0)
    if (split == 0) {
      for (int b = g; b < M; b += G) {
        const float4* src = reinterpret_cast<const float4*>(base + (size_t)b * cpb * cstride);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
        for (int c = 0; c < cpb; ++c) acc = f4add(acc, __ldcg(src + c * (cstride / 4)));
        sT[b * nvec + v] = acc;
      }
    } else {
      const int b = g / split, sub = g - b * split, per = cpb / split;
      const float4* src = reinterpret_cast<const float4*>(base + ((size_t)b * cpb + (size_t)sub * per) * cstride);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
      for (int c = 0; c < per; ++c) acc = f4add(acc, __ldcg(src + c * (cstride / 4)));
      sT[g * nvec + v] = acc;
    }
  }
  __syncthreads();
  if (live) {  // phase 2: mix
    const float* mh = p.mixing + (size_t)(h % p.H) * M * M;
    for (int i = g; i < M; i += G) {
      const int bend = p.mode == MIX_FULL ? M : i;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
      for (int b = 0; b < bend; ++b) {
        float4 tb;
        if (split == 0) {
          tb = sT[b * nvec + v];
        } else {
          tb = sT[(b * split) * nvec + v];
          for (int s2 = 1; s2 < split; ++s2) tb = f4add(tb, sT[(b * split + s2) * nvec + v]);
        }
        const float w = p.mode == MIX_PREFIX ? 1.f : __ldg(mh + (size_t)i * M + b);
        acc.x = fmaf(w, tb.x, acc.x);
        acc.y = fmaf(w, tb.y, acc.y);
        acc.z = fmaf(w, tb.z, acc.z);
        acc.w = fmaf(w, tb.w, acc.w);
      }
      if (ent < kD * kD) {
        uint2 packed;
        __nv_bfloat162* h2 = reinterpret_cast<__nv_bfloat162*>(&packed);
        h2[0] = __floats2bfloat162_rn(acc.x, acc.y);
        h2[1] = __floats2bfloat162_rn(acc.z, acc.w);
        *reinterpret_cast<uint2*>(p.s_mix + (((size_t)h * M + i) << 12) + ent) = packed;
      } else {
        *reinterpret_cast<float4*>(p.z_mix + ((size_t)h * M + i) * kD + (ent - kD * kD)) = acc;
      }
    }
  }
  fence_proxy_async_global();  // S~ is read later through TMA (async proxy)
  __syncthreads();
  if (threadIdx.x == 0) red_release_add(&p.ctr[2 + p.heads + h], 1u);
}

__global__ void __launch_bounds__(kThreads, kCtasPerSm) mhla_tc_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* regA = sm;                                   // K or Q tile
  uint8_t* regB = sm + kTileBytes;                      // V tile or Y staging
  uint8_t* regC = sm + 2 * kTileBytes;                  // S~ tile
  float4* sT = reinterpret_cast<float4*>(sm + 2 * kTileBytes + kSTileBytes);   // MIX staging
  Small* sh = reinterpret_cast<Small*>(sm + 2 * kTileBytes + kSTileBytes + kMixBytes);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    sh->s_ticket = -1;
    sh->s_inflight = 0;
    mbar_init(&sh->bar_in, 1);
    mbar_init(&sh->bar_s, 1);
    mbar_init(&sh->bar_mma, 1);
    fence_mbar_init();
    prefetch_tmap(&p.tm_q);
    prefetch_tmap(&p.tm_k);
    prefetch_tmap(&p.tm_v);
    prefetch_tmap(&p.tm_y);
    prefetch_tmap(&p.tm_s);
  }
  if (warp == 0) {
    tmem_alloc(&sh->tbase, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh->tbase;

  uint32_t ph_in = 0, ph_s = 0, ph_mma = 0;
  bool pend_in = false, pend_s = false;  // TMA loads issued and not yet waited for
  bool abort = false;

  if (tid == 0) {
    const int t0 = (int)atomicAdd(&p.ctr[0], 1u);
    sh->next = t0;
    if (t0 < p.total) issue_inputs(p, t0, regA, regB, regC, sh);
  }
  __syncthreads();
  int t = sh->next;
  pend_in = has_inputs(p, t);

  // SUM: D = V^T phi(K) = S^T (A = V^T, B = phi(K): both MN-major views of the token-major tiles)
  const uint32_t idesc_sum = idesc_bf16_f32(64, 64, 1, 1);
  // OUT: D = phi(Q) S~ (A = phi(Q), B = S~ stored e rows x c cols: both K-major)
  const uint32_t idesc_out = idesc_bf16_f32(128, 64, 0, 0);

  while (t < p.total && !abort) {
    const Unit u = decode(p, t);
    // the next ticket is taken now; its loads are issued once this unit's inputs are consumed
    unsigned nt_reg = 0;
    if (tid == 0) nt_reg = atomicAdd(&p.ctr[0], 1u);
    if (u.kind == UNIT_SUM) {
      // ---------------------------------------------------------------- SUM
      if (!cta_wait(&sh->bar_in, ph_in)) { abort = true; break; }
      ph_in ^= 1;
      pend_in = false;
      {  // phi(K) in place (bf16) and the fp32 z partial of this chunk
        const int j = tid & 7;
        float zacc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) zacc[e] = 0.f;
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          const int r = (tid >> 3) + 32 * s;
          uint4* ptr = reinterpret_cast<uint4*>(regA + swz128(r, j * 8));
          uint4 raw = *ptr;
          __nv_bfloat162* h2 = reinterpret_cast<__nv_bfloat162*>(&raw);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(h2[e]);
            const float a = phi_fast(f.x), b = phi_fast(f.y);
            zacc[2 * e] += a;
            zacc[2 * e + 1] += b;
            h2[e] = __floats2bfloat162_rn(a, b);
          }
          *ptr = raw;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          float v = zacc[e];
          v += __shfl_xor_sync(0xffffffffu, v, 8);
          v += __shfl_xor_sync(0xffffffffu, v, 16);
          if (lane < 8) sh->zred[warp][lane * 8 + e] = v;
        }
      }
      fence_proxy_async_smem();
      __syncthreads();
      if (tid < kD) {
        float z = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) z += sh->zred[w][tid];
        p.z_part[((size_t)u.h * p.C + u.idx) * kD + tid] = z;
      }
      if (tid == 0) {
        tc_fence_after();
        const uint32_t k0 = smem_u32(regA), v0 = smem_u32(regB);
#pragma unroll
        for (int k = 0; k < kTile / 16; ++k)
          mma_bf16(tmem, smem_desc(v0 + k * 2048, 8192, 1024), smem_desc(k0 + k * 2048, 8192, 1024),
                   idesc_sum, k > 0);
        mma_commit(&sh->bar_mma);
      }
      if (!cta_wait(&sh->bar_mma, ph_mma)) { abort = true; break; }
      ph_mma ^= 1;
      tc_fence_after();
      if (tid == 0) {  // K, V consumed: issue the next unit's loads
        sh->next = (int)nt_reg;
        if ((int)nt_reg < p.total) issue_inputs(p, (int)nt_reg, regA, regB, regC, sh);
      }
      {  // epilogue: D row e (M = 64: TMEM lane 32*(e/16) + e%16) = S^T[e][0..63]
        const int q = warp & 3, half = warp >> 2;
        float v[32];
        const uint32_t ta = tmem + ((uint32_t)(32 * q) << 16) + half * 32;
        tmem_ld16(ta, v);
        tmem_ld16(ta + 16, v + 16);
        tmem_ld_wait();
        if (lane < 16) {
          const int e = 16 * q + lane;
          float4* dst = reinterpret_cast<float4*>(p.s_part + (((size_t)u.h * p.C + u.idx) << 12) + e * kD + half * 32);
#pragma unroll
          for (int j4 = 0; j4 < 8; ++j4) dst[j4] = make_float4(v[4 * j4], v[4 * j4 + 1], v[4 * j4 + 2], v[4 * j4 + 3]);
        }
      }
      tc_fence_before();
      __syncthreads();
      if (tid == 0) red_release_add(&p.ctr[2 + u.h], 1u);  // publish this chunk's partial
      t = sh->next;
      pend_in = has_inputs(p, t);
    } else if (u.kind == UNIT_MIX) {
      // ---------------------------------------------------------------- MIX
      if (tid == 0) {
        sh->next = (int)nt_reg;
        if ((int)nt_reg < p.total) issue_inputs(p, (int)nt_reg, regA, regB, regC, sh);
      }
      __syncthreads();
      t = sh->next;
      pend_in = has_inputs(p, t);
      mix_item(p, u.h, u.idx, sT, sh);
    } else {
      // ---------------------------------------------------------------- OUT
      if (tid == 0 && sh->s_ticket != t) {
        const int ok = wait_geq(&p.ctr[2 + p.heads + u.h], (unsigned)p.I) ? 1 : 0;
        sh->flag = ok;
        if (ok) issue_mix_loads(p, t, regC, sh);
        else atomicOr(p.status, 1u);
      } else if (tid == 0) {
        sh->flag = 1;
      }
      __syncthreads();
      if (!sh->flag) { abort = true; break; }
      pend_s = true;
      if (!cta_wait(&sh->bar_in, ph_in)) { abort = true; break; }
      ph_in ^= 1;
      pend_in = false;
      if (!cta_wait(&sh->bar_s, ph_s)) { abort = true; break; }  // S~ tile and z~ have landed
      ph_s ^= 1;
      pend_s = false;
      if (tid == 0) sh->s_inflight = 0;
      const int q = warp & 3, half = warp >> 2, r = 32 * q + lane;
      {  // phi(Q) in place; partial denominator over this thread's 32 columns
        float dpart = 0.f;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int jc = half * 4 + jj;
          uint4* ptr = reinterpret_cast<uint4*>(regA + swz128(r, jc * 8));
          uint4 raw = *ptr;
          __nv_bfloat162* h2 = reinterpret_cast<__nv_bfloat162*>(&raw);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(h2[e]);
            const float a = phi_fast(f.x), b = phi_fast(f.y);
            dpart = fmaf(a, sh->zt[jc * 8 + 2 * e], dpart);
            dpart = fmaf(b, sh->zt[jc * 8 + 2 * e + 1], dpart);
            h2[e] = __floats2bfloat162_rn(a, b);
          }
          *ptr = raw;
        }
        sh->den_half[half][r] = dpart;
      }
      fence_proxy_async_smem();
      __syncthreads();
      if (tid == 0) {
        tc_fence_after();
        const uint32_t a0 = smem_u32(regA), b0 = smem_u32(regC);
#pragma unroll
        for (int k = 0; k < kD / 16; ++k)
          mma_bf16(tmem, smem_desc(a0 + 32 * k, 16, 1024), smem_desc(b0 + 32 * k, 16, 1024), idesc_out,
                   k > 0);
        mma_commit(&sh->bar_mma);
      }
      if (!cta_wait(&sh->bar_mma, ph_mma)) { abort = true; break; }
      ph_mma ^= 1;
      tc_fence_after();
      const float den = sh->den_half[0][r] + sh->den_half[1][r] + p.eps;
      if (tid == 0) {  // Q and S~ consumed: prefetch; then make sure the last Y store has left regB
        sh->next = (int)nt_reg;
        if ((int)nt_reg < p.total) issue_inputs(p, (int)nt_reg, regA, regB, regC, sh);
        tma_store_wait_read0();
      }
      __syncthreads();
      {  // epilogue: row r, columns half*32 .. +32
        float v[32];
        const uint32_t ta = tmem + ((uint32_t)(32 * q) << 16) + half * 32;
        tmem_ld16(ta, v);
        tmem_ld16(ta + 16, v + 16);
        tmem_ld_wait();
        const float inv = 1.f / den;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          uint4 raw;
          __nv_bfloat162* h2 = reinterpret_cast<__nv_bfloat162*>(&raw);
#pragma unroll
          for (int e = 0; e < 4; ++e) h2[e] = __floats2bfloat162_rn(v[jj * 8 + 2 * e] * inv, v[jj * 8 + 2 * e + 1] * inv);
          *reinterpret_cast<uint4*>(regB + swz128(r, (half * 4 + jj) * 8)) = raw;
        }
        if (half == 0 && p.den_out != nullptr) p.den_out[(size_t)u.h * p.N + u.idx * kTile + r] = den;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();
      if (tid == 0) {
        tma_store_2d(&p.tm_y, regB, 0, u.h * p.N + u.idx * kTile);
        tma_store_commit();
      }
      t = sh->next;
      pend_in = has_inputs(p, t);
    }
  }

  // ------------------------------------------------------------------ drain
  if (tid == 0) {
    if (abort) atomicOr(p.status, 1u);
    if (pend_in) mbar_wait(&sh->bar_in, ph_in);
    if (pend_s || sh->s_inflight) mbar_wait(&sh->bar_s, ph_s);
    tma_store_wait_all0();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
  if (tid == 0) {
    __threadfence();
    const unsigned f = atomicAdd(&p.ctr[1], 1u);
    if (f == gridDim.x - 1) {  // last CTA: every other CTA is done with the counters; reset them
      p.ctr[0] = 0;
      for (int i = 0; i < 2 * p.heads; ++i) p.ctr[2 + i] = 0;
      __threadfence();
      p.ctr[1] = 0;
    }
  }
}

// ------------------------------------------------------------------- host
PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  cuuint32_t box[2] = {(cuuint32_t)kD, box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct TcPlan {
  int C, M, cpb;
  size_t off_ctr, off_spart, off_zpart, off_smix, off_zmix, total;
};

inline size_t a256(size_t x) { return (x + 255) & ~size_t(255); }

TcPlan tc_plan(const MhlaShape& s) {
  TcPlan p;
  p.C = s.N / kTile;
  p.M = s.M();
  p.cpb = s.block / kTile;
  const size_t heads = (size_t)s.heads();
  p.off_ctr = kCounterOffset;
  size_t off = kWorkspacePrefix;
  p.off_spart = off; off = a256(off + heads * p.C * (size_t)kD * kD * sizeof(float));
  p.off_zpart = off; off = a256(off + heads * p.C * (size_t)kD * sizeof(float));
  p.off_smix = off;  off = a256(off + heads * p.M * (size_t)kD * kD * 2);
  p.off_zmix = off;  off = a256(off + heads * p.M * (size_t)kD * sizeof(float));
  p.total = off;
  return p;
}

// MIX work split: G threads share each 4-entry vector (G * nvec = 256).
// Constraints: per-thread chunk loads <= 32 (latency), block sums fit the
// 16 KB staging (M <= 4 G when G < M), and when G >= M the G/M threads of a
// block split its chunks evenly.  Among valid G, minimise the estimated total
// MIX time: items per head x (fixed cost + load latency + mixing work).
bool choose_mix_split(int M, int cpb, int* G_out, int* split_out) {
  long best = -1;
  for (int G = 1; G <= kThreads; G *= 2) {
    const int nvec = kThreads / G;
    int split = 0, loads = 0, work = 0;
    if (G < M) {
      if (M > 4 * G) continue;
      loads = ((M + G - 1) / G) * cpb;
      work = ((M + G - 1) / G) * M;
    } else {
      if (G % M != 0 || cpb % (G / M) != 0) continue;
      split = G / M;
      loads = cpb / split;
      work = M * split;
    }
    if (loads > 32) continue;
    const long items = (kEnt + 4 * nvec - 1) / (4 * nvec);
    const long cost = items * (400 + 50 * (long)loads + work);
    if (best < 0 || cost < best) {
      best = cost;
      *G_out = G;
      *split_out = split;
    }
  }
  return best >= 0;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

}  // namespace

bool tc_mhla_supported(const MhlaShape& s, mhla_dtype dt, MixMode mode) {
  if (dt != MHLA_BF16 || s.d != kD || mode != MIX_FULL) return false;
  if (s.block % kTile != 0 || s.N % kTile != 0) return false;
  if ((long long)s.heads() * s.N >= (1ll << 31)) return false;
  if (s.heads() > kMaxCounterHeads) return false;
  if (s.M() > 64) return false;
  int G = 0, split = 0;
  return choose_mix_split(s.M(), s.block / kTile, &G, &split);
}

size_t tc_mhla_workspace(const MhlaShape& s) { return tc_plan(s).total; }

cudaError_t tc_mhla_launch(const MhlaShape& s, const void* q, const void* k, const void* v,
                           const float* mixing, void* y, float* den_out, float eps, MixMode mode,
                           void* ws, cudaStream_t st) {
  const TcPlan pl = tc_plan(s);
  char* w = static_cast<char*>(ws);
  Params p;
  const uint64_t rows = (uint64_t)s.heads() * s.N;
  if (!make_map(&p.tm_q, q, rows, kTile) || !make_map(&p.tm_k, k, rows, kTile) ||
      !make_map(&p.tm_v, v, rows, kTile) || !make_map(&p.tm_y, y, rows, kTile) ||
      !make_map(&p.tm_s, w + pl.off_smix, (uint64_t)s.heads() * pl.M * kD, kD))
    return cudaErrorInvalidValue;
  p.mixing = mixing;
  p.s_part = reinterpret_cast<float*>(w + pl.off_spart);
  p.z_part = reinterpret_cast<float*>(w + pl.off_zpart);
  p.s_mix = reinterpret_cast<__nv_bfloat16*>(w + pl.off_smix);
  p.z_mix = reinterpret_cast<float*>(w + pl.off_zmix);
  p.den_out = den_out;
  p.ctr = reinterpret_cast<unsigned*>(w + pl.off_ctr);
  p.status = &reinterpret_cast<WorkspaceHeader*>(w)->status;
  p.heads = s.heads();
  p.H = s.H;
  p.N = s.N;
  p.M = pl.M;
  p.C = pl.C;
  p.cpb = pl.cpb;
  if (!choose_mix_split(p.M, p.cpb, &p.G, &p.split)) return cudaErrorInvalidValue;
  p.nvec = kThreads / p.G;
  p.I = (kEnt + 4 * p.nvec - 1) / (4 * p.nvec);
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const int grid_cap = sms * kCtasPerSm;
  // MIX items of head h go L heads after its SUM units: about two grids of tickets later
  int L = (2 * grid_cap + p.C + p.I - 1) / (p.C + p.I) + 1;
  p.L = L < p.heads ? L : p.heads;
  p.T1 = p.heads * (p.C + p.I);
  p.total = p.T1 + p.heads * p.C;
  p.eps = eps;
  p.mode = (int)mode;
  const int grid = p.total < grid_cap ? p.total : grid_cap;
  const size_t smem = 1024 + 2 * kTileBytes + kSTileBytes + kMixBytes + sizeof(Small);
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(mhla_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         227 * 1024);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  mhla_tc_kernel<<<grid, kThreads, smem, st>>>(p);
  note_launch();
  return cudaGetLastError();
}

}  // namespace mhla
