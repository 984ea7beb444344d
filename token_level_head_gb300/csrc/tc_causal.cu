// Causal linear attention (bf16, d = 64) on the sm_103a tensor cores.
//
// "MHLA: Restoring Expressivity of Linear Attention via Token-Level
// Multi-Head" App. C cuts each head's sequence into chunks of C tokens:
//   Y_t = [phi(q_t) P_c + sum_{s in c, s <= t} (phi(q_t) . phi(k_s)) v_s]
//       / [phi(q_t) . zeta_c + sum_{s in c, s <= t} phi(q_t) . phi(k_s) + eps]
// with the exclusive prefixes P_c = sum_{c' < c} phi(K_c')^T V_c' and
// zeta_c = sum_{c' < c} sum_{s in c'} phi(k_s).  The lower triangle includes
// the diagonal, as in the recurrence of "Linear Attention notes" §四 (token t
// enters the state before it is read).  The result does not depend on C; this
// kernel uses C = 128.
//
// The chunks of all heads (head-major) are cut into G contiguous segments, one
// per CTA.  A segment that starts inside a head needs that head's prefix up to
// its first chunk, so there are two launches:
//   causal_agg_kernel   each CTA sums phi(K)^T V (tensor cores, fp32 in TMEM)
//                       and phi(K) (fp32) over the last head piece of its
//                       segment, unless the head ends with the segment
//   causal_out_kernel   each CTA starts from its predecessors' aggregates in
//                       its first head and walks its chunks in order; P is
//                       carried in TMEM, zeta in shared memory
// Roles of causal_out_kernel (16 warps, one CTA per SM):
//   warp 0      TMA producer: the Q, K, V tiles of each chunk (3-stage ring)
//   warps 8-15  phi in place on the Q and K tiles (16 rows a warp), the fp32
//               inclusive prefix of phi(K) inside the chunk and from it the
//               denominator phi(q_t) . (zeta_c + sum_{s <= t} phi(k_s)) + eps
//   warp 1      MMA issuer: P += phi(K)^T V (carried in TMEM, M 128 with a
//               ones tile as A rows 0-63, so P lands in lanes 64-127);
//               scores = phi(Q) phi(K)^T (M 128, N 128); Y~ = phi(Q) P_c;
//               then Y~ += mask(scores) V once the masked scores are back
//   warps 2-3   P -> bf16 tile of the next chunk's P_c
//   warps 4-7   epilogue, one TMEM lane quadrant each: scores -> lower-
//               triangle mask -> bf16 A tile (written over the stage's Q and
//               K tiles, which are dead by then); Y = Y~ / den in bf16
//               through a TMA store
// All waits are bounded: on time-out the kernel sets the status word and
// winds down.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace mhla {
namespace {

using namespace tc;

constexpr int kThreads = 512;
constexpr int kTile = 128;                   // tokens per chunk
constexpr int kD = 64;                       // head dimension
constexpr int kTileBytes = kTile * kD * 2;   // 16 KB bf16 tile
constexpr int kPTile = kD * kD * 2;          // 8 KB bf16 P_c^T tile
constexpr int kWarpProd = 0, kWarpMma = 1, kWarpP = 2, kWarpEpi = 4, kWarpPhi = 8;
constexpr int kPhiWarps = 8;
constexpr int kBarPhi = 1;                   // named barrier of the phi warps
constexpr uint64_t kWaitLimitNs = 500000000ull;
constexpr int kMaxCtas = 256;                // aggregates in the workspace

// causal_out_kernel: TMEM columns of the running P (rows 64-127), the two
// score accumulators and the two Y~.
constexpr uint32_t kOutCols = 512, kColP = 0, kColSc = 128, kColNum = 384;
constexpr int kNSB = 3;                      // stages: Q, K, V
constexpr int kStageB = 3 * kTileBytes;
constexpr int kOffOnesB = 0;                 // 16 KB of bf16 ones: A rows 0..63 of the P MMA
constexpr int kOffStages = kTileBytes;       // the ring (above the ones tile: the MMA's LBO is positive)
constexpr int kOffP = kOffStages + kNSB * kStageB;  // 2 P_c^T tiles
constexpr int kOffY = kOffP + 2 * kPTile;    // Y staging, 4 warps x 2 x 4 KB
constexpr int kNDen = 4;                     // denominator slots
constexpr int kOffDen = kOffY + 4 * 8192;    // [kNDen][128] fp32
constexpr int kOffWs = kOffDen + kNDen * kTile * 4;  // [2][8 warps][64] fp32 column sums of phi(K)
constexpr int kOffZ = kOffWs + 2 * kPhiWarps * kD * 4;  // [2][64] fp32 zeta_c
constexpr int kOffSmallB = kOffZ + 2 * kD * 4;

// causal_agg_kernel: a K, V ring and the warps' phi(K) column sums.
constexpr uint32_t kAggCols = 128;           // two accumulators, one per MMA issuer
constexpr int kNSA = 6;
constexpr int kStageA = 2 * kTileBytes;
constexpr int kOffZA = kNSA * kStageA;       // [8 warps][64] fp32
constexpr int kOffSmallA = kOffZA + kPhiWarps * kD * 4;

struct OSmall {
  uint64_t full[kNSB], ready[kNSB], empty[kNSB];
  uint64_t p_full, ptile_full[2], sc_full[2], sc_empty[2], scores_full[2], num_full[2], num_empty[2];
  uint64_t den_free[kNDen];
  uint64_t fin;
  uint32_t tbase;
  int abort;
  int prod_q;
};

struct ASmall {
  uint64_t full[kNSA], ready[kNSA], empty[kNSA];
  uint64_t done, fin;
  uint32_t tbase;
  int abort;
  int prod_q;
};

constexpr size_t kOutSmem = 1024 + kOffSmallB + sizeof(OSmall);
constexpr size_t kAggSmem = 1024 + kOffSmallA + sizeof(ASmall);
static_assert(kOutSmem <= 232448 && kAggSmem <= 232448, "shared memory budget");

struct CParams {
  CUtensorMap tm_q, tm_k, tm_v;  // [T * 128 rows][64] bf16, box 64 x 128, 128-byte swizzle
  CUtensorMap tm_y;              // same tensor shape, box 64 x 32
  float* agg_s;                  // [G][64 e][64 c]: sum of V[t][e] phi(K)[t][c] over the last head piece
  float* agg_z;                  // [G][64]: sum of phi(K)[t][c] over the same tokens
  float* den_out;                // [T * 128] or null
  unsigned* status;
  // causal MHLA (mixing, chunk = block): the mixed prefixes P_i^T (bf16 tiles in the output
  // MMA's B layout) and zeta_i (fp32) of every (head, block), and the mixing matrix for m_ii
  const uint8_t* smix;
  const float* zmix;
  const float* mixing;
  int mix, H;                    // mix: 1 for causal MHLA; H: heads of the mixing matrix
  int T, CH, G;                  // chunks in all, chunks per head, CTAs
  int normalise;                 // 0: Y is the numerator alone (den_out still the denominator)
  float eps;
};

// m_ii of chunk c (causal MHLA: chunk = block, CH blocks a head).
__device__ __forceinline__ float self_weight(const CParams& p, int c) {
  const int hd = c / p.CH, b = c - hd * p.CH;
  return __ldg(p.mixing + ((size_t)(hd % p.H) * p.CH + b) * p.CH + b);
}

// First chunk of segment j (j = G gives T).
__device__ __forceinline__ int seg_lo(const CParams& p, int j) { return (int)(((long long)j * p.T) / p.G); }

__device__ __forceinline__ int ab_get(int* ab) { return *reinterpret_cast<volatile int*>(ab); }
__device__ __forceinline__ void ab_set(int* ab) { *reinterpret_cast<volatile int*>(ab) = 1; }

// Bounded mbarrier phase wait (polls, then suspended waits with a short
// limit); false after kWaitLimitNs (the CTA then aborts) or once another role
// has aborted.
__device__ __noinline__ bool cwait_slow(uint64_t* bar, uint32_t parity, int* ab) {
  for (int i = 0; i < 16; ++i)
    if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait_ns(bar, parity, 128)) return true;
    if (ab_get(ab)) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) break;
  }
  ab_set(ab);
  return false;
}

// A phase that has already completed costs one test and no call.
__device__ __forceinline__ bool cwait(uint64_t* bar, uint32_t parity, int* ab) {
  return mbar_test(bar, parity) || cwait_slow(bar, parity, ab);
}

// Short wait (10 ms at most), only while winding down after an abort.
__device__ __noinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait_ns(bar, parity, 1000))
    if (globaltimer_ns() - t0 > 10000000ull) return;
}

// The 16 rows 16 w .. 16 w + 15 of a 128-byte-swizzled bf16 tile with 64
// columns: lane (r0 = lane / 8, j = lane % 8) takes the logical 16-byte piece
// j (columns 8 j .. 8 j + 7) of the consecutive rows 16 w + 4 r0 + i, i = 0..3
// (four whole rows per access).  Replaces them by phi in bf16 and returns phi
// in fp32.
__device__ __forceinline__ void phi_rows(uint8_t* tile, int w, int lane, float (&f)[4][8]) {
  const int r0 = lane >> 3, j = lane & 7;
  uint4* ptr[4];
  uint4 x[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = 16 * w + 4 * r0 + i;
    ptr[i] = reinterpret_cast<uint4*>(tile + t * 128 + ((j ^ (t & 7)) << 4));
    x[i] = *ptr[i];
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t wd[4] = {x[i].x, x[i].y, x[i].z, x[i].w};
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      f[i][2 * m] = phi_f(__uint_as_float(wd[m] << 16));
      f[i][2 * m + 1] = phi_f(__uint_as_float(wd[m] & 0xffff0000u));
      wd[m] = pack_bf16(f[i][2 * m], f[i][2 * m + 1]);
    }
    *ptr[i] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
  }
}

// 16-byte piece j of row `row` of a 128-byte-swizzled tile (1024-byte aligned).
__device__ __forceinline__ uint4* swz_piece(uint8_t* tile, int row, int j) {
  return reinterpret_cast<uint4*>(tile + row * 128 + ((j ^ (row & 7)) << 4));
}

__device__ __forceinline__ uint4 pack8(const float* v) {
  return make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]), pack_bf16(v[6], v[7]));
}

// ================================================================ aggregates
__global__ void __launch_bounds__(kThreads, 1) causal_agg_kernel(const __grid_constant__ CParams p) {
  const int lo = seg_lo(p, blockIdx.x), hi = seg_lo(p, blockIdx.x + 1);
  if (hi % p.CH == 0) return;  // the head ends with the segment: no successor needs it
  const int pa = max(lo, ((hi - 1) / p.CH) * p.CH), n = hi - pa;
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  ASmall* sh = reinterpret_cast<ASmall*>(sm + kOffSmallA);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < kNSA; ++s) {
      mbar_init(&sh->full[s], 1);
      mbar_init(&sh->ready[s], kPhiWarps);
      mbar_init(&sh->empty[s], 1);
    }
    mbar_init(&sh->done, 2);
    mbar_init(&sh->fin, 2);
    sh->abort = 0;
    sh->prod_q = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(&sh->tbase, kAggCols);
    tmem_relinquish();
  }
  if (warp == kWarpProd && lane == 0) {
    prefetch_tmap(&p.tm_k);
    prefetch_tmap(&p.tm_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh->tbase;
  int* ab = &sh->abort;

  if (warp == kWarpProd) {
    if (lane == 0) {
      const uint64_t once = policy_evict_first();
      int i = 0;
      for (; i < n; ++i) {
        const int s = i % kNSA;
        if (i >= kNSA && !cwait(&sh->empty[s], ((i / kNSA) - 1) & 1, ab)) break;
        uint8_t* st = sm + s * kStageA;
        const int row = (pa + i) * kTile;
        mbar_arrive_expect_tx(&sh->full[s], kStageA);
        tma_load_2d_hint(st, &p.tm_k, 0, row, &sh->full[s], once);
        tma_load_2d_hint(st + kTileBytes, &p.tm_v, 0, row, &sh->full[s], once);
      }
      sh->prod_q = i;
    }
    __syncwarp();
  } else if (warp == kWarpMma || warp == kWarpMma + 1) {
    // two MMA issuers (one thread alone spends about a chunk's streaming time
    // on its waits and MMAs): issuer r takes chunks i with i % 2 = r into
    // accumulator r (TMEM columns 64 r ..)
    if (lane == 0) {
      const int r = warp - kWarpMma;
      // D[e][c] += sum_t V[t][e] phi(K)[t][c]: A = V (MN-major, M 64), B = phi(K) (MN-major)
      const uint32_t idesc = idesc_bf16_f32(64, 64, 1, 1);
      bool ok = true;
      for (int i = r; i < n && ok; i += 2) {
        const int s = i % kNSA;
        ok = cwait(&sh->ready[s], (i / kNSA) & 1, ab);
        if (!ok) break;
        tc_fence_after();
        const uint32_t st = smem_u32(sm + s * kStageA);
        const uint64_t da = smem_desc(st + kTileBytes, kTileBytes, 1024), db = smem_desc(st, 8192, 1024);
#pragma unroll
        for (int k = 0; k < kTile / 16; ++k)
          mma_bf16(tmem + 64 * r, da + k * (2048 >> 4), db + k * (2048 >> 4), idesc, i > r || k > 0);
        mma_commit(&sh->empty[s]);
      }
      if (ok) mma_commit(&sh->done);
      mma_commit(&sh->fin);
    }
    __syncwarp();
  } else if (warp >= kWarpPhi) {
    // phi(K) in place; fp32 column sums of phi(K) over the warp's rows
    const int w = warp - kWarpPhi, r0 = lane >> 3, j = lane & 7;
    float zs[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    bool ok = true;
    for (int i = 0; i < n; ++i) {
      const int s = i % kNSA;
      ok = __all_sync(0xffffffffu, cwait(&sh->full[s], (i / kNSA) & 1, ab));
      if (!ok) break;
      float f[4][8];
      phi_rows(sm + s * kStageA, w, lane, f);
#pragma unroll
      for (int x = 0; x < 8; ++x) zs[x] += (f[0][x] + f[1][x]) + (f[2][x] + f[3][x]);
      fence_proxy_async_smem();  // phi tile -> tensor core reads
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->ready[s]);
    }
    float* zw = reinterpret_cast<float*>(sm + kOffZA);
#pragma unroll
    for (int x = 0; x < 8; ++x) {
      zs[x] += __shfl_xor_sync(0xffffffffu, zs[x], 8);
      zs[x] += __shfl_xor_sync(0xffffffffu, zs[x], 16);
    }
    if (r0 == 0) {
#pragma unroll
      for (int x = 0; x < 8; ++x) zw[w * kD + 8 * j + x] = zs[x];
    }
    if (group_and(kBarPhi, kPhiWarps * 32, ok && !ab_get(ab)) && w == 0) {
      for (int c = lane; c < kD; c += 32) {
        float z = 0.f;
#pragma unroll
        for (int ww = 0; ww < kPhiWarps; ++ww) z += zw[ww * kD + c];
        p.agg_z[(size_t)blockIdx.x * kD + c] = z;
      }
    }
  } else if (warp >= kWarpEpi) {
    const int qd = warp - kWarpEpi;
    if (cwait(&sh->done, 0, ab)) {
      tc_fence_after();
      const uint32_t ta = tmem + ((uint32_t)(qd * 32) << 16);
      const bool two = n > 1;  // the second accumulator holds the odd chunks
      float4* dst = reinterpret_cast<float4*>(p.agg_s + ((size_t)blockIdx.x * kD + 16 * qd + lane) * kD);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float v[32], v2[32];
        tmem_ld16(ta + 32 * h, v);
        tmem_ld16(ta + 32 * h + 16, v + 16);
        if (two) {
          tmem_ld16(ta + 64 + 32 * h, v2);
          tmem_ld16(ta + 64 + 32 * h + 16, v2 + 16);
        }
        tmem_ld_wait();
        if (two) {
#pragma unroll
          for (int x = 0; x < 32; ++x) v[x] += v2[x];
        }
        if (lane < 16) {
#pragma unroll
          for (int c = 0; c < 8; ++c)
            dst[8 * h + c] = make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
        }
      }
    }
  }
  __syncthreads();
  if (tid == 0 && ab_get(ab)) {
    const int nq = sh->prod_q;
    for (int q = nq > kNSA ? nq - kNSA : 0; q < nq; ++q) drain_wait(&sh->full[q % kNSA], (q / kNSA) & 1);
    drain_wait(&sh->fin, 0);
    atomicOr(p.status, 1u);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tmem, kAggCols);
}

// ================================================================ output
__device__ __noinline__ int out_producer(const CParams& p, uint8_t* sm, OSmall* sh, int lo, int n) {
  const uint64_t once = policy_evict_first();
  int i = 0;
  for (; i < n; ++i) {
    const int s = i % kNSB;
    if (i >= kNSB && !cwait(&sh->empty[s], ((i / kNSB) - 1) & 1, &sh->abort)) break;
    uint8_t* st = sm + kOffStages + s * kStageB;
    const int row = (lo + i) * kTile;
    mbar_arrive_expect_tx(&sh->full[s], kStageB);
    tma_load_2d_hint(st, &p.tm_q, 0, row, &sh->full[s], once);
    tma_load_2d_hint(st + kTileBytes, &p.tm_k, 0, row, &sh->full[s], once);
    tma_load_2d_hint(st + 2 * kTileBytes, &p.tm_v, 0, row, &sh->full[s], once);
  }
  return i;
}

// phi warp w: phi(K), its in-chunk inclusive prefix, zeta, phi(Q) and den.
__device__ __noinline__ void out_phi(const CParams& p, uint8_t* sm, OSmall* sh, int w, int lane, int lo, int n) {
  float* den = reinterpret_cast<float*>(sm + kOffDen);
  float* wsum = reinterpret_cast<float*>(sm + kOffWs);
  float* zb = reinterpret_cast<float*>(sm + kOffZ);
  int* ab = &sh->abort;
  const int r0 = lane >> 3, j = lane & 7;
  if (w == 0 && r0 == 0 && !p.mix) {
    // zeta of the first chunk: the predecessors' phi(K) sums in this head
    float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    const int h0 = lo - lo % p.CH;
    if (lo != h0)
      for (int jj = (int)blockIdx.x - 1; jj >= 0 && seg_lo(p, jj + 1) > h0; --jj)
#pragma unroll
        for (int x = 0; x < 8; ++x) z[x] += __ldcg(p.agg_z + (size_t)jj * kD + 8 * j + x);
#pragma unroll
    for (int x = 0; x < 8; ++x) zb[8 * j + x] = z[x];
  }
  for (int i = 0; i < n; ++i) {
    const int s = i % kNSB, a = i & 1, c = lo + i;
    bool ok = cwait(&sh->full[s], (i / kNSB) & 1, ab);
    // den slot i % kNDen is free once the epilogue of chunk i - kNDen has read it
    const int dslot = i % kNDen;
    if (ok && i >= kNDen) ok = cwait(&sh->den_free[dslot], ((i / kNDen) - 1) & 1, ab);
    ok = __all_sync(0xffffffffu, ok);
    uint8_t* st = sm + kOffStages + s * kStageB;
    float kf[4][8], run[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (ok) {
      phi_rows(st + kTileBytes, w, lane, kf);
      // inclusive prefix over the rows 16 w + 4 r0 + i: over i inside the lane,
      // over r0 by shuffles of the lane totals (lanes 8 apart)
#pragma unroll
      for (int x = 0; x < 8; ++x) {
#pragma unroll
        for (int i4 = 1; i4 < 4; ++i4) kf[i4][x] += kf[i4 - 1][x];
        const float tl = kf[3][x];  // this lane's four rows
        float v = tl;
        float u = __shfl_up_sync(0xffffffffu, v, 8);
        if (r0 >= 1) v += u;
        u = __shfl_up_sync(0xffffffffu, v, 16);
        if (r0 >= 2) v += u;
        run[x] = __shfl_sync(0xffffffffu, v, 24 + j);  // the warp's total
        const float ex = v - tl;                       // rows of the lanes before
#pragma unroll
        for (int i4 = 0; i4 < 4; ++i4) kf[i4][x] += ex;
      }
      if (r0 == 0) {
        float4* ws4 = reinterpret_cast<float4*>(wsum + (a * kPhiWarps + w) * kD + 8 * j);
        ws4[0] = make_float4(run[0], run[1], run[2], run[3]);
        ws4[1] = make_float4(run[4], run[5], run[6], run[7]);
      }
    }
    if (!group_and(kBarPhi, kPhiWarps * 32, ok && !ab_get(ab))) return;
    // zeta_c plus the rows of the warps before this one (all warps' totals are
    // read at once, 16-byte loads; warp 0 also forms zeta of the next chunk)
    float off[8], tot[8], zeta[8];
    float mii = 1.f;
    if (p.mix) {
      // causal MHLA: zeta_i = sum_{b<i} m_ib z_b from the MIX pass; the in-chunk terms
      // are weighted by m_ii
      const float4* z4 = reinterpret_cast<const float4*>(p.zmix + (size_t)c * kD + 8 * j);
      const float4 z0 = __ldcg(z4), z1 = __ldcg(z4 + 1);
      zeta[0] = z0.x; zeta[1] = z0.y; zeta[2] = z0.z; zeta[3] = z0.w;
      zeta[4] = z1.x; zeta[5] = z1.y; zeta[6] = z1.z; zeta[7] = z1.w;
      mii = self_weight(p, c);
#pragma unroll
      for (int x = 0; x < 8; ++x) off[x] = 0.f;
    } else {
      const float4* z4 = reinterpret_cast<const float4*>(zb + a * kD + 8 * j);
      const float4 z0 = z4[0], z1 = z4[1];
      off[0] = z0.x; off[1] = z0.y; off[2] = z0.z; off[3] = z0.w;
      off[4] = z1.x; off[5] = z1.y; off[6] = z1.z; off[7] = z1.w;
#pragma unroll
      for (int x = 0; x < 8; ++x) zeta[x] = 0.f;
    }
#pragma unroll
    for (int x = 0; x < 8; ++x) tot[x] = off[x];
#pragma unroll
    for (int ww = 0; ww < kPhiWarps; ++ww) {
      const float4* w4 = reinterpret_cast<const float4*>(wsum + (a * kPhiWarps + ww) * kD + 8 * j);
      const float4 u0 = w4[0], u1 = w4[1];
      const float u[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
      for (int x = 0; x < 8; ++x) {
        tot[x] += u[x];
        if (ww < w) off[x] += u[x];
      }
    }
    if (w == 0 && r0 == 0 && i + 1 < n && !p.mix) {
      // zeta of the next chunk (zero when it starts a new head)
      const bool fresh = (c + 1) % p.CH == 0;
      float4* zn = reinterpret_cast<float4*>(zb + (a ^ 1) * kD + 8 * j);
      zn[0] = fresh ? make_float4(0.f, 0.f, 0.f, 0.f) : make_float4(tot[0], tot[1], tot[2], tot[3]);
      zn[1] = fresh ? make_float4(0.f, 0.f, 0.f, 0.f) : make_float4(tot[4], tot[5], tot[6], tot[7]);
    }
    float qf[4][8];
    phi_rows(st, w, lane, qf);
#pragma unroll
    for (int i4 = 0; i4 < 4; ++i4) {
      float d = 0.f;
#pragma unroll
      for (int x = 0; x < 8; ++x) d = fmaf(qf[i4][x], fmaf(mii, off[x] + kf[i4][x], zeta[x]), d);
      d += __shfl_xor_sync(0xffffffffu, d, 1);
      d += __shfl_xor_sync(0xffffffffu, d, 2);
      d += __shfl_xor_sync(0xffffffffu, d, 4);
      if (j == 0) den[dslot * kTile + 16 * w + 4 * r0 + i4] = d + p.eps;
    }
    fence_proxy_async_smem();  // phi tiles -> tensor core reads
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh->ready[s]);
  }
}

// The second half of chunk i's MMAs, once its masked scores are in place:
// Y~ += mask(scores) V; frees the stage.
__device__ void out_finish(uint8_t* sm, OSmall* sh, uint32_t tmem, int i) {
  const int a = i & 1, s = i % kNSB;
  const uint32_t st = smem_u32(sm + kOffStages + s * kStageB);
  // A = masked scores, K-major: s 0..63 over the K tile, s 64..127 over the Q
  // tile; B = V (N = e, K = s: MN-major)
  const uint64_t d0 = smem_desc(st + kTileBytes, 16, 1024), d1 = smem_desc(st, 16, 1024);
  const uint64_t dv = smem_desc(st + 2 * kTileBytes, 8192, 1024);
  const uint32_t idesc = idesc_bf16_f32(128, 64, 0, 1);
#pragma unroll
  for (int k = 0; k < kTile / 16; ++k)
    mma_bf16(tmem + kColNum + 64 * a, k < 4 ? d0 + k * (32 >> 4) : d1 + (k - 4) * (32 >> 4), dv + k * (2048 >> 4),
             idesc, true);
  mma_commit(&sh->empty[s]);
  mma_commit(&sh->num_full[a]);
}

// The first MMAs of chunk i: P += phi(K)^T V, scores, Y~ = phi(Q) P_c.
__device__ void out_start(const CParams& p, uint8_t* sm, OSmall* sh, uint32_t tmem, int lo, int i) {
  const int a = i & 1, s = i % kNSB, c = lo + i;
  const uint32_t ones = smem_u32(sm + kOffOnesB);
  const uint32_t st = smem_u32(sm + kOffStages + s * kStageB);
  const uint32_t q0 = st, k0 = st + kTileBytes, v0 = st + 2 * kTileBytes;
  if (!p.mix) {
    // D = [1 ; V^T] phi(K) (M 128, MN-major A: the ones tile, then V, v0 - ones
    // bytes apart): rows 64 + e hold P^T[e][c] += sum_t V[t][e] phi(K)[t][c];
    // a chunk that starts a head starts from zero
    const uint64_t da = smem_desc(ones, v0 - ones, 1024), db = smem_desc(k0, 8192, 1024);
    const uint32_t idesc = idesc_bf16_f32(128, 64, 1, 1);
    const bool cont = c % p.CH != 0;
#pragma unroll
    for (int k = 0; k < kTile / 16; ++k)
      mma_bf16(tmem + kColP, da + k * (2048 >> 4), db + k * (2048 >> 4), idesc, cont || k > 0);
    mma_commit(&sh->p_full);
  }
  {
    const uint64_t da = smem_desc(q0, 16, 1024), db = smem_desc(k0, 16, 1024);
    const uint32_t idesc = idesc_bf16_f32(128, 128, 0, 0);
#pragma unroll
    for (int k = 0; k < kD / 16; ++k)
      mma_bf16(tmem + kColSc + 128 * a, da + k * (32 >> 4), db + k * (32 >> 4), idesc, k > 0);
  }
  {
    const uint64_t da = smem_desc(q0, 16, 1024), db = smem_desc(smem_u32(sm + kOffP) + a * kPTile, 16, 1024);
    const uint32_t idesc = idesc_bf16_f32(128, 64, 0, 0);
#pragma unroll
    for (int k = 0; k < kD / 16; ++k)
      mma_bf16(tmem + kColNum + 64 * a, da + k * (32 >> 4), db + k * (32 >> 4), idesc, k > 0);
  }
  mma_commit(&sh->sc_full[a]);
}

// MMA issuer: polls the two kinds of work it can do, finishing a chunk whose
// masked scores are back first (that frees a stage), else starting the next
// chunk once its phi tiles, its P_c tile and its accumulators are ready.
__device__ __noinline__ void out_mma(const CParams& p, uint8_t* sm, OSmall* sh, uint32_t tmem, int lo, int n) {
  int* ab = &sh->abort;
  int i = 0, f = 0;  // next chunk to start, next chunk to finish
  uint64_t t0 = globaltimer_ns();
  while (f < n) {
    if (f < i && mbar_test(&sh->scores_full[f & 1], (f >> 1) & 1)) {
      tc_fence_after();
      out_finish(sm, sh, tmem, f++);
      t0 = globaltimer_ns();
      continue;
    }
    if (i < n && mbar_test(&sh->ready[i % kNSB], (i / kNSB) & 1) &&
        mbar_test(&sh->ptile_full[i & 1], (i >> 1) & 1) &&
        (i < 2 || (mbar_test(&sh->sc_empty[i & 1], ((i >> 1) - 1) & 1) &&
                   mbar_test(&sh->num_empty[i & 1], ((i >> 1) - 1) & 1)))) {
      tc_fence_after();
      out_start(p, sm, sh, tmem, lo, i++);
      t0 = globaltimer_ns();
      continue;
    }
    if (ab_get(ab)) break;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      ab_set(ab);
      break;
    }
    __nanosleep(32);
  }
  mma_commit(&sh->fin);
}

// Y rows of chunk i for epilogue warp qd.
__device__ bool out_store(const CParams& p, uint8_t* sm, OSmall* sh, uint32_t tmem, int qd, int lane, int lo, int i,
                          int& nst) {
  const int a = i & 1;
  if (!cwait(&sh->num_full[a], (i >> 1) & 1, &sh->abort)) return false;
  tc_fence_after();
  const float* den = reinterpret_cast<const float*>(sm + kOffDen);
  uint8_t* yb = sm + kOffY + qd * 8192 + (nst & 1) * 4096;  // two buffers a warp
  float v[64];
  const uint32_t ta = tmem + kColNum + 64 * a + ((uint32_t)(qd * 32) << 16);
#pragma unroll
  for (int g = 0; g < 4; ++g) tmem_ld16(ta + 16 * g, v + 16 * g);
  tmem_ld_wait();
  const int t = qd * 32 + lane;
  const float dn = den[(i % kNDen) * kTile + t];
  tc_fence_before();
  __syncwarp();
  if (lane == 0) {
    mbar_arrive(&sh->num_empty[a]);
    mbar_arrive(&sh->den_free[i % kNDen]);
  }
  const size_t row = (size_t)(lo + i) * kTile + t;
  if (p.den_out != nullptr) p.den_out[row] = dn;
  const float r = p.normalise ? 1.f / dn : 1.f;
#pragma unroll
  for (int x = 0; x < 64; ++x) v[x] *= r;
  if (lane == 0 && nst >= 1) tma_store_wait_read1();  // the store of two chunks ago has read yb
  __syncwarp();
#pragma unroll
  for (int jj = 0; jj < 8; ++jj) *swz_piece(yb, lane, jj) = pack8(v + 8 * jj);
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d_hint(&p.tm_y, yb, 0, (lo + i) * kTile + qd * 32, policy_evict_first());
    tma_store_commit();
  }
  ++nst;
  return true;
}

// Warps 2-3 carry P: TMEM lanes 64 + e hold P^T row e (warp 2 rows 0..31,
// warp 3 rows 32..63).  They seed P with the predecessors' aggregates and,
// after each chunk's P MMA, write the bf16 P_c^T tile of the next chunk.
__device__ __noinline__ void out_pchain(const CParams& p, uint8_t* sm, OSmall* sh, uint32_t tmem, int wq, int lane, int lo, int n) {
  int* ab = &sh->abort;
  uint8_t* ptile = sm + kOffP;
  const uint32_t lq = (uint32_t)(64 + 32 * wq) << 16;
  const int e = 32 * wq + lane;
  if (p.mix) {
    // causal MHLA: the P tile of chunk i is the MIX pass's P_i^T tile, copied as it is (the
    // same swizzled image); tile i % 2 was last read by the MMAs of chunk i - 2
    for (int i = 0; i < n; ++i) {
      const int a = i & 1;
      if (i >= 2 && !cwait(&sh->sc_full[a], ((i - 2) >> 1) & 1, ab)) return;
      const uint4* src = reinterpret_cast<const uint4*>(p.smix + (size_t)(lo + i) * kPTile) + 8 * e;
      uint4* dst = reinterpret_cast<uint4*>(ptile + a * kPTile) + 8 * e;
      uint4 u[8];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) u[jj] = __ldcg(src + jj);
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) dst[jj] = u[jj];
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->ptile_full[a]);
    }
    return;
  }
  {
    float v[64];
#pragma unroll
    for (int x = 0; x < 64; ++x) v[x] = 0.f;
    const int h0 = lo - lo % p.CH;
    if (lo != h0) {
      for (int jj = (int)blockIdx.x - 1; jj >= 0 && seg_lo(p, jj + 1) > h0; --jj) {
        const float4* src = reinterpret_cast<const float4*>(p.agg_s + ((size_t)jj * kD + e) * kD);
#pragma unroll
        for (int c4 = 0; c4 < 16; ++c4) {
          const float4 u = __ldcg(src + c4);
          v[4 * c4] += u.x;
          v[4 * c4 + 1] += u.y;
          v[4 * c4 + 2] += u.z;
          v[4 * c4 + 3] += u.w;
        }
      }
#pragma unroll
      for (int g = 0; g < 4; ++g) tmem_st16(tmem + kColP + lq + 16 * g, v + 16 * g);
      tmem_st_wait();
    }
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) *swz_piece(ptile, e, jj) = pack8(v + 8 * jj);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh->ptile_full[0]);
  }
  for (int i = 0; i + 1 < n; ++i) {
    if (!cwait(&sh->p_full, i & 1, ab)) return;
    tc_fence_after();
    float v[64];
#pragma unroll
    for (int g = 0; g < 4; ++g) tmem_ld16(tmem + kColP + lq + 16 * g, v + 16 * g);
    tmem_ld_wait();
    tc_fence_before();
    // the tile of chunk i + 1 was last read by the MMAs of chunk i - 1, which
    // completed before this chunk's P MMA did
    uint8_t* dst = ptile + ((i + 1) & 1) * kPTile;
    const bool fresh = (lo + i + 1) % p.CH == 0;  // chunk i + 1 starts a head
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) *swz_piece(dst, e, jj) = fresh ? make_uint4(0, 0, 0, 0) : pack8(v + 8 * jj);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh->ptile_full[(i + 1) & 1]);
  }
}

// Epilogue warp qd (TMEM lanes 32 qd ..): the Y rows of chunk i - 1, then the
// masked scores of chunk i.
__device__ __noinline__ void out_epi(const CParams& p, uint8_t* sm, OSmall* sh, uint32_t tmem, int qd, int lane, int lo, int n) {
  int* ab = &sh->abort;
  const uint32_t lq = (uint32_t)(qd * 32) << 16;
  int nst = 0;
  for (int i = 0; i < n; ++i) {
    const int a = i & 1;
    // Y of chunk i - 1 first: its accumulator is what chunk i + 1 starts on
    if (i >= 1 && !out_store(p, sm, sh, tmem, qd, lane, lo, i - 1, nst)) return;
    // scores -> mask s <= t -> bf16 A tiles over the stage's K (s < 64) and Q tiles
    if (!cwait(&sh->sc_full[a], (i >> 1) & 1, ab)) return;
    tc_fence_after();
    uint8_t* st = sm + kOffStages + (i % kNSB) * kStageB;
    const int t = 32 * qd + lane;
    const float mii = p.mix ? self_weight(p, lo + i) : 1.f;  // causal MHLA: the in-chunk scores times m_ii
    // 32 columns s0 = 32 qr at a time: below this quadrant's rows they are kept
    // whole, beyond them they are zero, on the diagonal (qr = qd) masked
    for (int qr = 0; qr < 4; ++qr) {
      uint8_t* tile = qr < 2 ? st + kTileBytes : st;
      const int j0 = 4 * (qr & 1);
      if (qr > qd) {
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) *swz_piece(tile, t, j0 + jj) = make_uint4(0, 0, 0, 0);
        continue;
      }
      float v[32];
      tmem_ld16(tmem + kColSc + 128 * a + lq + 32 * qr, v);
      tmem_ld16(tmem + kColSc + 128 * a + lq + 32 * qr + 16, v + 16);
      tmem_ld_wait();
      if (qr == qd) {
#pragma unroll
        for (int x = 0; x < 32; ++x)
          if (x > lane) v[x] = 0.f;
      }
#pragma unroll
      for (int x = 0; x < 32; ++x) v[x] *= mii;
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) *swz_piece(tile, t, j0 + jj) = pack8(v + 8 * jj);
    }
    tc_fence_before();
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(&sh->sc_empty[a]);
      mbar_arrive(&sh->scores_full[a]);
    }
  }
  if (n >= 1) out_store(p, sm, sh, tmem, qd, lane, lo, n - 1, nst);
}

__global__ void __launch_bounds__(kThreads, 1) causal_out_kernel(const __grid_constant__ CParams p) {
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  OSmall* sh = reinterpret_cast<OSmall*>(sm + kOffSmallB);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int lo = seg_lo(p, blockIdx.x), n = seg_lo(p, blockIdx.x + 1) - lo;
  if (tid == 0) {
    for (int s = 0; s < kNSB; ++s) {
      mbar_init(&sh->full[s], 1);
      mbar_init(&sh->ready[s], kPhiWarps);
      mbar_init(&sh->empty[s], 1);
    }
    mbar_init(&sh->p_full, 1);
    mbar_init(&sh->fin, 1);
    for (int a = 0; a < 2; ++a) {
      mbar_init(&sh->ptile_full[a], 2);
      mbar_init(&sh->sc_full[a], 1);
      mbar_init(&sh->sc_empty[a], 4);
      mbar_init(&sh->scores_full[a], 4);
      mbar_init(&sh->num_full[a], 1);
      mbar_init(&sh->num_empty[a], 4);
    }
    for (int d = 0; d < kNDen; ++d) mbar_init(&sh->den_free[d], 4);
    sh->abort = 0;
    sh->prod_q = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(&sh->tbase, kOutCols);
    tmem_relinquish();
  }
  if (warp == kWarpProd && lane == 0) {
    prefetch_tmap(&p.tm_q);
    prefetch_tmap(&p.tm_k);
    prefetch_tmap(&p.tm_v);
    prefetch_tmap(&p.tm_y);
  }
  for (int i = tid; i < kTileBytes / 16; i += kThreads)
    reinterpret_cast<uint4*>(sm + kOffOnesB)[i] = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh->tbase;

  if (warp == kWarpProd) {
    if (lane == 0) sh->prod_q = out_producer(p, sm, sh, lo, n);
    __syncwarp();
  } else if (warp == kWarpMma) {
    if (lane == 0) out_mma(p, sm, sh, tmem, lo, n);
    __syncwarp();
  } else if (warp >= kWarpPhi) {
    out_phi(p, sm, sh, warp - kWarpPhi, lane, lo, n);
  } else if (warp >= kWarpEpi) {
    out_epi(p, sm, sh, tmem, warp - kWarpEpi, lane, lo, n);
    if (lane == 0) tma_store_wait_all0();
  } else if (warp >= kWarpP) {
    out_pchain(p, sm, sh, tmem, warp - kWarpP, lane, lo, n);
  }
  __syncthreads();
  if (tid == 0 && ab_get(&sh->abort)) {
    const int nq = sh->prod_q;
    for (int q = nq > kNSB ? nq - kNSB : 0; q < nq; ++q) drain_wait(&sh->full[q % kNSB], (q / kNSB) & 1);
    drain_wait(&sh->fin, 0);
    atomicOr(p.status, 1u);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tmem, kOutCols);
}

// ================================================================ host
PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// [rows][64] bf16, box 64 x box_rows, 128-byte swizzle.
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

inline size_t a256(size_t x) { return (x + 255) & ~size_t(255); }
// Workspace: the header and counter prefix, then agg_s and agg_z of up to
// min(T, kMaxCtas) CTAs.
int max_ctas(const MhlaShape& s) { return (int)std::min<long long>((long long)s.heads() * (s.N / kTile), kMaxCtas); }
size_t off_agg_z(const MhlaShape& s) { return kWorkspacePrefix + a256((size_t)max_ctas(s) * kD * kD * sizeof(float)); }

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

}  // namespace

bool tc_causal_supported(const MhlaShape& s, mhla_dtype dt, MixMode mode) {
  if (!s.plain_phi()) return false;  // ELU + 1 without decay only
  if (dt != MHLA_BF16 || s.d != kD || mode != MIX_PREFIX) return false;
  if (s.N % kTile != 0) return false;
  return (long long)s.heads() * s.N < (1ll << 31);
}

size_t tc_causal_workspace(const MhlaShape& s) { return off_agg_z(s) + a256((size_t)max_ctas(s) * kD * sizeof(float)); }

cudaError_t tc_causal_launch(const MhlaShape& s, const void* q, const void* k, const void* v, void* y,
                             float* den_out, float eps, void* ws, cudaStream_t st) {
  char* w = static_cast<char*>(ws);
  CParams p;
  const uint64_t rows = (uint64_t)s.heads() * s.N;
  if (!make_map(&p.tm_q, q, rows, kTile) || !make_map(&p.tm_k, k, rows, kTile) || !make_map(&p.tm_v, v, rows, kTile) ||
      !make_map(&p.tm_y, y, rows, 32))
    return cudaErrorInvalidValue;
  p.agg_s = reinterpret_cast<float*>(w + kWorkspacePrefix);
  p.agg_z = reinterpret_cast<float*>(w + off_agg_z(s));
  p.den_out = den_out;
  p.status = &reinterpret_cast<WorkspaceHeader*>(w)->status;
  p.T = s.heads() * (s.N / kTile);
  p.CH = s.N / kTile;
  p.eps = eps;
  p.normalise = s.normalise ? 1 : 0;
  p.smix = nullptr;
  p.zmix = nullptr;
  p.mixing = nullptr;
  p.mix = 0;
  p.H = s.H;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  p.G = std::min(max_ctas(s), sms);
  static SmemOptIn opt_out, opt_agg;
  cudaError_t e = opt_out.ensure((const void*)causal_out_kernel, (int)kOutSmem);
  if (e == cudaSuccess) e = opt_agg.ensure((const void*)causal_agg_kernel, (int)kAggSmem);
  if (e != cudaSuccess) return e;
  if (p.CH > 1) {  // with one chunk per head no segment starts inside a head
    causal_agg_kernel<<<p.G, kThreads, kAggSmem, st>>>(p);
    note_launch();
  }
  causal_out_kernel<<<p.G, kThreads, kOutSmem, st>>>(p);
  note_launch();
  return cudaGetLastError();
}

// Causal MHLA with a mixing matrix, chunk = block = 128 tokens ("MHLA" paper §4.2 / App. C chunk
// form): the tcgen05 MHLA kernel's SUM and MIX passes with the weights m_ib for b < i give P_i
// and zeta_i of every (head, block); the output kernel reads them instead of carrying a prefix
// and weights its in-chunk terms by m_ii.
bool tc_causal_mhla_supported(const MhlaShape& s, mhla_dtype dt, MixMode mode) {
  if (!s.plain_phi() || s.grid() || mode != MIX_STRICT_LOWER) return false;
  if (dt != MHLA_BF16 || s.d != kD || s.block != kTile || s.N % kTile != 0) return false;
  if ((long long)s.heads() * s.N >= (1ll << 31)) return false;
  return tc_mhla_prefix_supported(s, dt);
}

size_t tc_causal_mhla_workspace(const MhlaShape& s) { return tc_mhla_workspace(s); }

cudaError_t tc_causal_mhla_launch(const MhlaShape& s, const void* q, const void* k, const void* v,
                                  const float* mixing, void* y, float* den_out, float eps, void* ws,
                                  cudaStream_t st) {
  cudaError_t e = tc_mhla_prefix_launch(s, k, v, mixing, ws, st);
  if (e != cudaSuccess) return e;
  char* w = static_cast<char*>(ws);
  CParams p;
  const uint64_t rows = (uint64_t)s.heads() * s.N;
  if (!make_map(&p.tm_q, q, rows, kTile) || !make_map(&p.tm_k, k, rows, kTile) || !make_map(&p.tm_v, v, rows, kTile) ||
      !make_map(&p.tm_y, y, rows, 32))
    return cudaErrorInvalidValue;
  p.agg_s = nullptr;
  p.agg_z = nullptr;
  p.den_out = den_out;
  p.status = &reinterpret_cast<WorkspaceHeader*>(w)->status;
  p.T = s.heads() * (s.N / kTile);
  p.CH = s.N / kTile;
  p.eps = eps;
  p.normalise = s.normalise ? 1 : 0;
  tc_mhla_mixed_summaries(s, ws, &p.smix, &p.zmix);
  p.mixing = mixing;
  p.mix = 1;
  p.H = s.H;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  p.G = std::min(max_ctas(s), sms);
  static SmemOptIn opt_out;
  e = opt_out.ensure((const void*)causal_out_kernel, (int)kOutSmem);
  if (e != cudaSuccess) return e;
  causal_out_kernel<<<p.G, kThreads, kOutSmem, st>>>(p);
  note_launch();
  return cudaGetLastError();
}

}  // namespace mhla
