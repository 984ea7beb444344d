// RALA (rank-augmented linear attention) forward on the sm_103a tensor cores:
// bf16, d = 32, Cx = 64, H <= 2, N a multiple of 64.
//
// "Breaking the Low-Rank Dilemma of Linear Attention", key design 1: per
// (batch, head) the query mean Q_g = (1/N) sum_t Q_t (raw queries) weighs the
// keys, l_j = Q_g . phi(K_j), alpha = softmax_j(l), and
//   B = sum_j alpha_j phi(K_j)^T V_j                (d x d)
// key design 2: G = X W (shared by the heads of a batch) and
//   Y_t = G_t * (phi(Q_t) B)                        (elementwise)
//
// d = 32 rows are 64 bytes; the kernels view every [N][32] head slice as
// [N / 2][64] token pairs, so each row is one 128-byte swizzle row:
//  - sum_r Vpair_r^T (w phi(K))pair_r is a 64 x 64 matrix whose two diagonal
//    32 x 32 blocks are the even- and odd-token halves of B^T; their sum is B^T
//  - phi(Q)pair times blockdiag(B, B) gives the outputs of both tokens of a
//    pair side by side, which is the pair layout of Y
//  - Xpair (two 64-wide halves) times blockdiag(W, W) gives G in pair layout.
// Three launches:
//   rala_qsum_kernel   fp32 partial sums of Q over 8 slices of each (b, h)
//   rala_b_kernel      one CTA per (b, h): logits of all its keys and their
//                      maximum (pass A), then weights exp(l - max), the
//                      weighted phi(K) and B^T on the tensor cores (pass B)
//   rala_out_kernel    persistent: per tile of 128 pairs of a batch, G and
//                      phi(Q_h) B_h on the tensor cores, Y_h = G * (phi(Q_h) B_h)
// All waits are bounded: on time-out the kernels set the status word and
// wind down.
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
constexpr int kD = 32;                        // head dimension
constexpr int kCx = 64;                       // channels of X
constexpr int kRows = 128;                    // pair rows per tile (256 tokens)
constexpr int kTileBytes = kRows * 128;       // 16 KB
constexpr int kSlices = 8;                    // Q partial sums per (b, h)
constexpr int kMaxN = 8192;                   // logits kept in shared memory
constexpr int kWarpProd = 0, kWarpMma = 1, kWarpAux = 2, kWarpEpi = 4, kWarpPhi = 8;
constexpr int kPhiWarps = 8;
constexpr int kBarPhi = 1;
constexpr int kBarAux = 3;                    // named barrier of warps 2-3 (output kernel)
constexpr uint64_t kWaitLimitNs = 500000000ull;

struct RParams {
  CUtensorMap tm_q, tm_k, tm_v, tm_y;  // [U * N / 2][64] bf16, box 64 x 128 (y: 64 x 32), 128-byte swizzle
  CUtensorMap tm_x;                    // [B * N / 2][128] bf16, box 64 x 128
  const __nv_bfloat16* w;              // [64 k][32 e]
  float* qpart;                        // [U][kSlices][32]
  float* bt;                           // [U][32 e][32 c]: B^T, normalised
  unsigned* status;
  int B, H, N, NP;                     // NP = N / 2 pair rows per head
  int TPB, tiles;                      // output tiles per batch, in all
};

__device__ __forceinline__ int ab_get(int* ab) { return *reinterpret_cast<volatile int*>(ab); }
__device__ __forceinline__ void ab_set(int* ab) { *reinterpret_cast<volatile int*>(ab) = 1; }

// Bounded mbarrier phase wait; false after kWaitLimitNs (the CTA aborts) or
// once another role has aborted.
__device__ __noinline__ bool rwait(uint64_t* bar, uint32_t parity, int* ab) {
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

__device__ __noinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait_ns(bar, parity, 1000))
    if (globaltimer_ns() - t0 > 10000000ull) return;
}

// Rows 16 w + r0 + 4 i (r0 = lane / 8, i = 0..3) of a 128-byte-swizzled tile,
// logical 16-byte piece j = lane % 8 of each.
__device__ __forceinline__ uint4* piece_ptr(uint8_t* tile, int row, int j) {
  return reinterpret_cast<uint4*>(tile + row * 128 + ((j ^ (row & 7)) << 4));
}

__device__ __forceinline__ void unpack8(uint4 x, float* f) {
  const uint32_t wd[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    f[2 * m] = __uint_as_float(wd[m] << 16);
    f[2 * m + 1] = __uint_as_float(wd[m] & 0xffff0000u);
  }
}

__device__ __forceinline__ uint4 pack8(const float* v) {
  return make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]), pack_bf16(v[6], v[7]));
}

// ================================================================ Q sums
// Slice s of (b, h) = pair rows [s NP / 8, (s + 1) NP / 8); thread piece p of
// a row holds columns 8 (p % 4) .. of token 2 r + p / 4.
__global__ void __launch_bounds__(256) rala_qsum_kernel(const __nv_bfloat16* __restrict__ q, float* __restrict__ qpart,
                                                       int NP) {
  __shared__ float red[32][33];
  const int u = blockIdx.y, s = blockIdx.x;
  const int r0 = (int)((long long)s * NP / kSlices), r1 = (int)((long long)(s + 1) * NP / kSlices);
  const int p = threadIdx.x & 7, rr = threadIdx.x >> 3;  // 32 rows at a time
  const uint4* src = reinterpret_cast<const uint4*>(q) + ((size_t)u * NP) * 8;
  // the output kernel reads Q again: keep it in L2 (evict-last) across the B^T kernel
  const uint64_t keep = policy_evict_last();
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int r = r0 + rr; r < r1; r += 4 * 32) {  // four 16-byte loads in flight
    uint4 u[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      u[k] = r + 32 * k < r1 ? ld_global_hint(src + (size_t)(r + 32 * k) * 8 + p, keep) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float f[8];
      unpack8(u[k], f);
#pragma unroll
      for (int x = 0; x < 8; ++x) acc[x] += f[x];
    }
  }
  // lanes p and p ^ 4 hold the same columns (the two tokens of a pair)
#pragma unroll
  for (int x = 0; x < 8; ++x) acc[x] += __shfl_xor_sync(0xffffffffu, acc[x], 4);
  if (p < 4)
#pragma unroll
    for (int x = 0; x < 8; ++x) red[rr][8 * p + x] = acc[x];
  __syncthreads();
  if (threadIdx.x < 32) {
    float t = 0.f;
    for (int i = 0; i < 32; ++i) t += red[i][threadIdx.x];
    qpart[((size_t)u * kSlices + s) * kD + threadIdx.x] = t;
  }
}

// ================================================================ B^T
constexpr int kNSR = 5;                         // K (+ V) stages
constexpr int kStageR = 2 * kTileBytes;
constexpr int kOffLogit = kNSR * kStageR;       // [kMaxN] fp32
constexpr int kOffQg = kOffLogit + kMaxN * 4;   // [32] fp32
constexpr int kOffRed = kOffQg + kD * 4;        // [2][8] fp32: warp maxima, warp weight sums
constexpr int kOffTbl = kOffRed + 2 * kPhiWarps * 4;  // [32][33] fp32
constexpr int kOffSmallR = kOffTbl + kD * 33 * 4;

struct BSmall {
  uint64_t full[kNSR], ready[kNSR], empty[kNSR];
  uint64_t done, sums, fin;
  uint32_t tbase;
  int abort;
  int prod_q;
};
constexpr size_t kBSmem = 1024 + kOffSmallR + sizeof(BSmall);
static_assert(kBSmem <= 232448, "shared memory budget");

__device__ __forceinline__ float exp2_hw(float x) {
  float e;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(x));
  return e;
}

// One CTA per (b, h) = unit u.  Items 0 .. T-1 are the K tiles of pass A,
// items T .. 2T-1 the K and V tiles of pass B (T tiles of 128 pair rows).
__global__ void __launch_bounds__(kThreads, 1) rala_b_kernel(const __grid_constant__ RParams p) {
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  BSmall* sh = reinterpret_cast<BSmall*>(sm + kOffSmallR);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int u = blockIdx.x;
  const int T = (p.NP + kRows - 1) / kRows;
  if (tid == 0) {
    for (int s = 0; s < kNSR; ++s) {
      mbar_init(&sh->full[s], 1);
      mbar_init(&sh->ready[s], kPhiWarps);
      mbar_init(&sh->empty[s], 1);
    }
    mbar_init(&sh->done, 1);
    mbar_init(&sh->sums, kPhiWarps);
    mbar_init(&sh->fin, 1);
    sh->abort = 0;
    sh->prod_q = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(&sh->tbase, 64);
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
      for (; i < 2 * T; ++i) {
        const int s = i % kNSR, k = i < T ? i : i - T;
        if (i >= kNSR && !rwait(&sh->empty[s], ((i / kNSR) - 1) & 1, ab)) break;
        uint8_t* st = sm + s * kStageR;
        const int row = u * p.NP + k * kRows;
        if (i < T) {
          // pass A: the K tile stays in L2 for pass B
          mbar_arrive_expect_tx(&sh->full[s], kTileBytes);
          tma_load_2d(st, &p.tm_k, 0, row, &sh->full[s]);
        } else {
          mbar_arrive_expect_tx(&sh->full[s], 2 * kTileBytes);
          tma_load_2d_hint(st, &p.tm_k, 0, row, &sh->full[s], once);
          tma_load_2d_hint(st + kTileBytes, &p.tm_v, 0, row, &sh->full[s], once);
        }
      }
      sh->prod_q = i;
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    if (lane == 0) {
      // D[m][n] += sum_r Vpair[r][m] (w phi(K))pair[r][n]: A = V (MN-major,
      // M 64), B = weighted phi(K) (MN-major, N 64), K = 128 pair rows
      const uint32_t idesc = idesc_bf16_f32(64, 64, 1, 1);
      bool ok = true;
      for (int i = 0; i < 2 * T && ok; ++i) {
        const int s = i % kNSR;
        ok = rwait(&sh->ready[s], (i / kNSR) & 1, ab);
        if (!ok) break;
        tc_fence_after();
        if (i >= T) {
          const uint32_t st = smem_u32(sm + s * kStageR);
          const uint64_t da = smem_desc(st + kTileBytes, kTileBytes, 1024), db = smem_desc(st, 8192, 1024);
#pragma unroll
          for (int k = 0; k < kRows / 16; ++k)
            mma_bf16(tmem, da + k * (2048 >> 4), db + k * (2048 >> 4), idesc, i > T || k > 0);
        }
        mma_commit(&sh->empty[s]);
      }
      if (ok) mma_commit(&sh->done);
      mma_commit(&sh->fin);
    }
    __syncwarp();
  } else if (warp >= kWarpPhi) {
    const int w = warp - kWarpPhi, r0 = lane >> 3, j = lane & 7;
    float* logit = reinterpret_cast<float*>(sm + kOffLogit);
    float* qg = reinterpret_cast<float*>(sm + kOffQg);
    float* red = reinterpret_cast<float*>(sm + kOffRed);
    if (w == 0) {
      float t = 0.f;
      for (int s = 0; s < kSlices; ++s) t += __ldcg(p.qpart + ((size_t)u * kSlices + s) * kD + lane);
      qg[lane] = t / (float)p.N;  // Q_g: the mean of the raw queries
    }
    named_bar(kBarPhi, kPhiWarps * 32);
    float qv[8];
#pragma unroll
    for (int x = 0; x < 8; ++x) qv[x] = qg[8 * (j & 3) + x];
    float lmax = -INFINITY, wsum = 0.f, m = 0.f;
    bool ok = true;
    // after a failed wait a warp keeps walking the items without waiting or
    // working, so that all of them meet at the barrier before pass B
    for (int i = 0; i < 2 * T; ++i) {
      const int s = i % kNSR, k = i < T ? i : i - T;
      if (ok) ok = __all_sync(0xffffffffu, rwait(&sh->full[s], (i / kNSR) & 1, ab));
      if (i == T) {
        // every logit is in: the maximum over the unit
        float mm = lmax;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mm = fmaxf(mm, __shfl_xor_sync(0xffffffffu, mm, o));
        if (lane == 0) red[w] = mm;
        ok = group_and(kBarPhi, kPhiWarps * 32, ok && !ab_get(ab));
        m = red[0];
#pragma unroll
        for (int ww = 1; ww < kPhiWarps; ++ww) m = fmaxf(m, red[ww]);
      }
      if (!ok) continue;
      uint8_t* st = sm + s * kStageR;
#pragma unroll
      for (int i4 = 0; i4 < 4; ++i4) {
        const int row = 16 * w + r0 + 4 * i4;
        const int tok = 2 * (k * kRows + row) + (j >> 2);  // token of this piece
        uint4* pp = piece_ptr(st, row, j);
        float f[8];
        unpack8(*pp, f);
#pragma unroll
        for (int x = 0; x < 8; ++x) f[x] = phi_f(f[x]);
        if (i < T) {
          float l = 0.f;
#pragma unroll
          for (int x = 0; x < 8; ++x) l = fmaf(f[x], qv[x], l);
          l += __shfl_xor_sync(0xffffffffu, l, 1);
          l += __shfl_xor_sync(0xffffffffu, l, 2);
          if (tok < p.N) {
            lmax = fmaxf(lmax, l);
            if ((j & 3) == 0) logit[tok] = l;
          }
        } else {
          const float wt = tok < p.N ? exp2_hw((logit[tok] - m) * 1.4426950408889634f) : 0.f;
          if ((j & 3) == 0) wsum += wt;
#pragma unroll
          for (int x = 0; x < 8; ++x) f[x] *= wt;
          *pp = pack8(f);
        }
      }
      if (i >= T) fence_proxy_async_smem();  // weighted phi(K) -> tensor core reads
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->ready[s]);
    }
    if (ok) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
      if (lane == 0) {
        red[kPhiWarps + w] = wsum;
        mbar_arrive(&sh->sums);
      }
    }
  } else if (warp >= kWarpEpi) {
    // B^T[e][c] = D[e][c] + D[32 + e][32 + c], divided by the sum of the weights
    const int qd = warp - kWarpEpi, mrow = 16 * qd + lane;  // lanes 0..15: D row (M 64 layout)
    float* tbl = reinterpret_cast<float*>(sm + kOffTbl);
    const float* red = reinterpret_cast<const float*>(sm + kOffRed);
    const bool ok = rwait(&sh->done, 0, ab) && rwait(&sh->sums, 0, ab);
    float v[32];
    if (ok) {
      tc_fence_after();
      const uint32_t ta = tmem + ((uint32_t)(qd * 32) << 16) + (qd < 2 ? 0 : 32);
      tmem_ld16(ta, v);
      tmem_ld16(ta + 16, v + 16);
      tmem_ld_wait();
      if (qd < 2 && lane < 16)
#pragma unroll
        for (int c = 0; c < kD; ++c) tbl[mrow * 33 + c] = v[c];
    }
    named_bar(kBarPhi + 1, 128);
    if (ok && qd >= 2 && lane < 16)
#pragma unroll
      for (int c = 0; c < kD; ++c) tbl[(mrow - 32) * 33 + c] += v[c];
    named_bar(kBarPhi + 1, 128);
    if (ok) {
      float S = 0.f;
#pragma unroll
      for (int ww = 0; ww < kPhiWarps; ++ww) S += red[kPhiWarps + ww];
      const float rs = 1.f / S;
      const int t = tid - kWarpEpi * 32;
      for (int idx = t; idx < kD * kD; idx += 128)
        p.bt[(size_t)u * kD * kD + idx] = tbl[(idx / kD) * 33 + idx % kD] * rs;
    }
  }
  __syncthreads();
  if (tid == 0 && ab_get(ab)) {
    const int nq = sh->prod_q;
    for (int q = nq > kNSR ? nq - kNSR : 0; q < nq; ++q) drain_wait(&sh->full[q % kNSR], (q / kNSR) & 1);
    drain_wait(&sh->fin, 0);
    atomicOr(p.status, 1u);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tmem, 64);
}

// ================================================================ output
// Stage of one tile (128 pair rows of batch b): X even / odd halves, the H
// phi(Q_h) tiles and the H blockdiag(B_h, B_h) operand tiles.
constexpr int kNSO = 2;
constexpr int kOffXo = kTileBytes, kOffQ = 2 * kTileBytes, kOffBd = 4 * kTileBytes;
constexpr int kBdBytes = 64 * 128;                   // 8 KB
constexpr int kStageO = kOffBd + 2 * kBdBytes;       // 80 KB
constexpr int kOffW = kNSO * kStageO;                // W0, W1 operand tiles
constexpr int kOffYO = kOffW + 2 * kBdBytes;         // Y staging, 4 warps x 4 KB
constexpr int kOffSmallO = kOffYO + 4 * 4096;
constexpr uint32_t kOutColsR = 512;                  // slot a: G at 192 a, Y_h at 192 a + 64 (1 + h)

struct OSmallR {
  uint64_t full[kNSO], ready[kNSO], empty[kNSO];
  uint64_t acc_full[2], acc_empty[2], fin;
  uint32_t tbase;
  int abort;
  int prod_q;
};
constexpr size_t kOSmem = 1024 + kOffSmallO + sizeof(OSmallR);
static_assert(kOSmem <= 232448, "shared memory budget");

__global__ void __launch_bounds__(kThreads, 1) rala_out_kernel(const __grid_constant__ RParams p) {
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  OSmallR* sh = reinterpret_cast<OSmallR*>(sm + kOffSmallO);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g0 = (int)((long long)blockIdx.x * p.tiles / gridDim.x);
  const int n = (int)((long long)(blockIdx.x + 1) * p.tiles / gridDim.x) - g0;
  if (tid == 0) {
    for (int s = 0; s < kNSO; ++s) {
      mbar_init(&sh->full[s], 1);
      mbar_init(&sh->ready[s], kPhiWarps + 2);
      mbar_init(&sh->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&sh->acc_full[a], 1);
      mbar_init(&sh->acc_empty[a], 4);
    }
    mbar_init(&sh->fin, 1);
    sh->abort = 0;
    sh->prod_q = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(&sh->tbase, kOutColsR);
    tmem_relinquish();
  }
  if (warp == kWarpProd && lane == 0) {
    prefetch_tmap(&p.tm_q);
    prefetch_tmap(&p.tm_x);
    prefetch_tmap(&p.tm_y);
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
        const int s = i % kNSO, g = g0 + i, b = g / p.TPB, k = g % p.TPB;
        if (i >= kNSO && !rwait(&sh->empty[s], ((i / kNSO) - 1) & 1, ab)) break;
        uint8_t* st = sm + s * kStageO;
        mbar_arrive_expect_tx(&sh->full[s], (2 + p.H) * kTileBytes);
        const int xrow = b * p.NP + k * kRows;
        tma_load_2d_hint(st, &p.tm_x, 0, xrow, &sh->full[s], once);
        tma_load_2d_hint(st + kOffXo, &p.tm_x, 64, xrow, &sh->full[s], once);
        for (int h = 0; h < p.H; ++h)
          tma_load_2d_hint(st + kOffQ + h * kTileBytes, &p.tm_q, 0, (b * p.H + h) * p.NP + k * kRows, &sh->full[s],
                           once);
      }
      sh->prod_q = i;
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    if (lane == 0) {
      // G = Xe W0^T + Xo W1^T and Y_h = phi(Q_h) Bd_h^T: M 128 pair rows, N 64, K-major operands
      const uint32_t idesc = idesc_bf16_f32(128, 64, 0, 0);
      const uint32_t w0 = smem_u32(sm + kOffW), w1 = w0 + kBdBytes;
      bool ok = true;
      for (int i = 0; i < n && ok; ++i) {
        const int s = i % kNSO, a = i & 1;
        ok = rwait(&sh->ready[s], (i / kNSO) & 1, ab) && (i < 2 || rwait(&sh->acc_empty[a], ((i >> 1) - 1) & 1, ab));
        if (!ok) break;
        tc_fence_after();
        const uint32_t st = smem_u32(sm + s * kStageO);
        const uint32_t dg = tmem + 192 * a;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16(dg, smem_desc(st, 16, 1024) + kk * 2, smem_desc(w0, 16, 1024) + kk * 2, idesc, kk > 0);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16(dg, smem_desc(st + kOffXo, 16, 1024) + kk * 2, smem_desc(w1, 16, 1024) + kk * 2, idesc, true);
        for (int h = 0; h < p.H; ++h) {
          const uint64_t da = smem_desc(st + kOffQ + h * kTileBytes, 16, 1024);
          const uint64_t db = smem_desc(st + kOffBd + h * kBdBytes, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) mma_bf16(dg + 64 * (1 + h), da + kk * 2, db + kk * 2, idesc, kk > 0);
        }
        mma_commit(&sh->empty[s]);
        mma_commit(&sh->acc_full[a]);
      }
      mma_commit(&sh->fin);
    }
    __syncwarp();
  } else if (warp >= kWarpPhi) {
    // phi in place on the Q_h tiles
    const int w = warp - kWarpPhi, r0 = lane >> 3, j = lane & 7;
    for (int i = 0; i < n; ++i) {
      const int s = i % kNSO;
      if (!__all_sync(0xffffffffu, rwait(&sh->full[s], (i / kNSO) & 1, ab))) break;
      uint8_t* st = sm + s * kStageO;
      for (int h = 0; h < p.H; ++h) {
        uint4* pp[4];
        uint4 x[4];
#pragma unroll
        for (int i4 = 0; i4 < 4; ++i4) {
          pp[i4] = piece_ptr(st + kOffQ + h * kTileBytes, 16 * w + r0 + 4 * i4, j);
          x[i4] = *pp[i4];
        }
#pragma unroll
        for (int i4 = 0; i4 < 4; ++i4) {
          x[i4].x = pack_bf16(phi_f(__uint_as_float(x[i4].x << 16)), phi_f(__uint_as_float(x[i4].x & 0xffff0000u)));
          x[i4].y = pack_bf16(phi_f(__uint_as_float(x[i4].y << 16)), phi_f(__uint_as_float(x[i4].y & 0xffff0000u)));
          x[i4].z = pack_bf16(phi_f(__uint_as_float(x[i4].z << 16)), phi_f(__uint_as_float(x[i4].z & 0xffff0000u)));
          x[i4].w = pack_bf16(phi_f(__uint_as_float(x[i4].w << 16)), phi_f(__uint_as_float(x[i4].w & 0xffff0000u)));
          *pp[i4] = x[i4];
        }
      }
      fence_proxy_async_smem();  // phi tiles -> tensor core reads
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->ready[s]);
    }
  } else if (warp >= kWarpEpi) {
    const int qd = warp - kWarpEpi;
    uint8_t* yb = sm + kOffYO + qd * 4096;
    const uint64_t once = policy_evict_first();
    const uint32_t lq = (uint32_t)(qd * 32) << 16;
    int nst = 0;
    for (int i = 0; i < n; ++i) {
      const int a = i & 1, g = g0 + i, b = g / p.TPB, k = g % p.TPB;
      if (!rwait(&sh->acc_full[a], (i >> 1) & 1, ab)) break;
      tc_fence_after();
      const bool valid = k * kRows + 32 * qd < p.NP;  // this warp's 32 pair rows exist
      for (int h = 0; h < p.H; ++h) {
        if (lane == 0 && nst >= 1) tma_store_wait_read0();  // the previous store has read yb
        __syncwarp();
#pragma unroll
        for (int hc = 0; hc < 2; ++hc) {
          float gv[32], yv[32];
          const uint32_t ta = tmem + lq + 192 * a + 32 * hc;
          tmem_ld16(ta, gv);
          tmem_ld16(ta + 16, gv + 16);
          tmem_ld16(ta + 64 * (1 + h), yv);
          tmem_ld16(ta + 64 * (1 + h) + 16, yv + 16);
          tmem_ld_wait();
#pragma unroll
          for (int x = 0; x < 32; ++x) yv[x] *= gv[x];
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) *piece_ptr(yb, lane, 4 * hc + jj) = pack8(yv + 8 * jj);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && valid) {
          tma_store_2d_hint(&p.tm_y, yb, 0, (b * p.H + h) * p.NP + k * kRows + 32 * qd, once);
          tma_store_commit();
        }
        nst += valid ? 1 : 0;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->acc_empty[a]);
    }
    if (lane == 0) tma_store_wait_all0();
  } else {
    // warps 2-3: the W operand tiles once, then the blockdiag(B_h, B_h) tiles of each stage
    const int t = tid - kWarpAux * 32;  // operand row n = 0..63
    {
      // W [64 k][32 e] (4 KB) through the Y staging area (free until the first
      // tile's MMAs, which wait for these tiles) with 16-byte loads, then
      // W0[n][k] = W[k][n] (n < 32), W1[n][k] = W[k][n - 32] (n >= 32), zero elsewhere
      __nv_bfloat16* wst = reinterpret_cast<__nv_bfloat16*>(sm + kOffYO);
      for (int i = t; i < kCx * kD / 8; i += 64)
        reinterpret_cast<uint4*>(wst)[i] = __ldg(reinterpret_cast<const uint4*>(p.w) + i);
      named_bar(kBarAux, 64);
      uint8_t* wt = sm + kOffW + (t < 32 ? 0 : kBdBytes);
      uint8_t* wz = sm + kOffW + (t < 32 ? kBdBytes : 0);
      for (int jj = 0; jj < 8; ++jj) {
        float v[8];
#pragma unroll
        for (int x = 0; x < 8; ++x) v[x] = __bfloat162float(wst[(8 * jj + x) * kD + (t & 31)]);
        *piece_ptr(wt, t, jj) = pack8(v);
        *piece_ptr(wz, t, jj) = make_uint4(0, 0, 0, 0);
      }
    }
    // row t % 32 of B_h^T for the current batch, kept in registers (a CTA's
    // tiles are consecutive, so the batch rarely changes)
    float bv[2][kD];
    int cur_b = -1;
    for (int i = 0; i < n; ++i) {
      const int s = i % kNSO, g = g0 + i, b = g / p.TPB;
      if (b != cur_b) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (h >= p.H) break;
          const float4* src = reinterpret_cast<const float4*>(p.bt + ((size_t)(b * p.H + h) * kD + (t & 31)) * kD);
#pragma unroll
          for (int c4 = 0; c4 < kD / 4; ++c4) {
            const float4 u = __ldcg(src + c4);
            bv[h][4 * c4] = u.x;
            bv[h][4 * c4 + 1] = u.y;
            bv[h][4 * c4 + 2] = u.z;
            bv[h][4 * c4 + 3] = u.w;
          }
        }
        cur_b = b;
      }
      if (i >= kNSO && !rwait(&sh->empty[s], ((i / kNSO) - 1) & 1, ab)) break;
      uint8_t* st = sm + s * kStageO;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (h >= p.H) break;
        // Bd[n][k] = B^T[n % 32][k % 32] when n and k are in the same half
        uint8_t* bd = st + kOffBd + h * kBdBytes;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          *piece_ptr(bd, t, (t < 32 ? 0 : 4) + jj) = pack8(&bv[h][8 * jj]);
          *piece_ptr(bd, t, (t < 32 ? 4 : 0) + jj) = make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->ready[s]);
    }
  }
  __syncthreads();
  if (tid == 0 && ab_get(ab)) {
    const int nq = sh->prod_q;
    for (int q = nq > kNSO ? nq - kNSO : 0; q < nq; ++q) drain_wait(&sh->full[q % kNSO], (q / kNSO) & 1);
    drain_wait(&sh->fin, 0);
    atomicOr(p.status, 1u);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tmem, kOutColsR);
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

// [rows][inner] bf16, box 64 x box_rows, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows, uint64_t inner) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)inner * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline size_t a256(size_t x) { return (x + 255) & ~size_t(255); }

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

}  // namespace

bool tc_rala_supported(int B, int H, int N, int d, int cx, mhla_dtype dt) {
  if (dt != MHLA_BF16 || d != kD || cx != kCx || H < 1 || H > 2) return false;
  if (N <= 0 || N % 64 != 0 || N > kMaxN) return false;
  return (long long)B * H * N < (1ll << 31);
}

size_t tc_rala_workspace(int B, int H, int N) {
  (void)N;
  const size_t U = (size_t)B * H;
  return kWorkspacePrefix + a256(U * kSlices * kD * sizeof(float)) + a256(U * kD * kD * sizeof(float));
}

cudaError_t tc_rala_launch(int B, int H, int N, const void* q, const void* k, const void* v, const void* x,
                           const void* w, void* y, void* ws, cudaStream_t st) {
  char* wsp = static_cast<char*>(ws);
  RParams p;
  const int U = B * H, NP = N / 2;
  const uint64_t rows = (uint64_t)U * NP;
  if (!make_map(&p.tm_q, q, rows, kRows, 64) || !make_map(&p.tm_k, k, rows, kRows, 64) ||
      !make_map(&p.tm_v, v, rows, kRows, 64) || !make_map(&p.tm_y, y, rows, 32, 64) ||
      !make_map(&p.tm_x, x, (uint64_t)B * NP, kRows, 2 * kCx))
    return cudaErrorInvalidValue;
  p.w = static_cast<const __nv_bfloat16*>(w);
  p.qpart = reinterpret_cast<float*>(wsp + kWorkspacePrefix);
  p.bt = reinterpret_cast<float*>(wsp + kWorkspacePrefix + a256((size_t)U * kSlices * kD * sizeof(float)));
  p.status = &reinterpret_cast<WorkspaceHeader*>(wsp)->status;
  p.B = B;
  p.H = H;
  p.N = N;
  p.NP = NP;
  p.TPB = (NP + kRows - 1) / kRows;
  p.tiles = B * p.TPB;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  static SmemOptIn opt_b, opt_out;
  cudaError_t e = opt_b.ensure((const void*)rala_b_kernel, (int)kBSmem);
  if (e == cudaSuccess) e = opt_out.ensure((const void*)rala_out_kernel, (int)kOSmem);
  if (e != cudaSuccess) return e;
  rala_qsum_kernel<<<dim3(kSlices, U), 256, 0, st>>>(static_cast<const __nv_bfloat16*>(q), p.qpart, NP);
  rala_b_kernel<<<U, kThreads, kBSmem, st>>>(p);
  rala_out_kernel<<<std::min(p.tiles, sms), kThreads, kOSmem, st>>>(p);
  note_launch(3);
  return cudaGetLastError();
}

}  // namespace mhla
