// The token passes of the MHLA backward on the sm_103a tensor cores (bf16, d = 64, blocks of
// whole 128-token chunks).  The products of the backward of "MHLA: Restoring Expressivity of
// Linear Attention via Token-Level Multi-Head" §4.1 (the chain rule through its block form) are
// dense 64-wide contractions:
//   query pass, per chunk of block i, with S~_i = z~_i mu_i^T + S'_i (mu_i = S~_i^T z~_i / |z~_i|^2:
//       phi is near 1, so the rows of S~ are near multiples of one vector and the two terms of
//       dphi(q) below nearly cancel; the rank-one part is carried in fp32, only the small S' is
//       rounded to bf16 for the tensor cores):
//       num = (den - eps) mu + phi(Q) S';  den = phi(Q) . z~_i + eps (fp32);  dnum = dY / den,
//       dden = -(dY . num) / den^2;  dphi(Q) = dnum S'^T + (mu . dnum + dden) z~_i;
//       dq = phi'(q) dphi(q);
//       [dS~_i^T ; dz~_i] += [dnum^T ; dden] phi(Q)   (one M = 128 MMA: a tile of dden repeated
//       along the rows gives dz~ in the lower half, as the forward's summary takes z from a tile
//       of ones)
//   key pass, per chunk of block b:    dv = phi(K) dS_b;  dphi(K) = V dS_b^T;
//       dk = phi'(k) (dphi(k) + dz_b)
// with phi'(x) = min(1, phi(x)).  S'_i and dS_b arrive as bf16 tiles in both orientations (K-major
// B operands, 128-byte swizzle), written by the centring and mixing kernels.
//
// The block summaries S_b, z_b come from a third pass of the same shape ([V^T ; 1] phi(K), as the
// forward's summary pass).  One CTA per (unit, block), 6 warps: warp 0 TMA producer (the block's d x d tiles, then each
// chunk's two 128 x 64 tiles), warp 1 MMA issuer (one thread), warps 2-5 epilogue (TMEM lane
// quadrant = warp % 4, one token row a thread: phi in place, the fp32 denominator, the dnum and
// dden tiles, the gradients).  Every hand-over is an mbarrier; every wait is bounded (on time-out
// the CTA stops, sets the status word and drains what it has in flight).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace mhla {
namespace {

using namespace tc;

constexpr int kT = 128;                 // tokens per chunk
constexpr int kD = 64;                  // head dimension
constexpr int kTile = kT * kD * 2;      // 16 KB bf16 chunk tile
constexpr int kSTile = kD * kD * 2;     // 8 KB bf16 d x d tile
constexpr int kX = kD * kD + kD;        // floats of a slot (S then z)
constexpr int kThreads = 192;
constexpr int kWarpProd = 0, kWarpMma = 1, kWarpEpi = 2, kEpiWarps = 4;
constexpr uint64_t kWaitNs = 500000000ull;  // 0.5 s: a wait's default limit

// query pass: Q (phi in place), dY (dnum is written over it, row by row), dden repeated (right
// after dnum: the LBO of the stacked A operand), S'^T, S', z~ then mu (fp32).  65 KB and 128 TMEM
// columns: three CTAs an SM, so three chunk chains in flight (a chunk is a serial chain of phi,
// MMA, dnum/dden, MMAs, dq; the chains in flight set the pass's rate).
constexpr int kQ_Q = 0, kQ_Y = kTile, kQ_R = 2 * kTile, kQ_ST = 3 * kTile, kQ_SN = kQ_ST + kSTile,
              kQ_Z = kQ_SN + kSTile, kQ_BAR = kQ_Z + 512;
constexpr uint32_t kQCols = 128;        // phi(Q) S', then dnum S'^T, in [0, 64); [dS~^T ; dz~] [64, 128)
// key pass: K (phi in place), V, dS^T, dS, dz
constexpr int kK_K = 0, kK_V = kTile, kK_ST = 2 * kTile, kK_SN = kK_ST + kSTile, kK_Z = kK_SN + kSTile,
              kK_BAR = kK_Z + 256;
constexpr uint32_t kKCols = 128;        // dv [0, 64), dphi(K) [64, 128)

struct Bars {
  uint64_t full;   // the chunk's tiles landed (tx)
  uint64_t sfull;  // the block's d x d tiles and z landed (tx)
  uint64_t phi;    // phi written (4 epilogue warps)
  uint64_t acc1;   // query: num ready; key: dv, dphi(K) ready (MMA commit)
  uint64_t mid;    // query: dnum and dden tiles written (4 epilogue warps)
  uint64_t acc2;   // query: dphi(Q) and the dS~ accumulation done (MMA commit)
  uint64_t free_;  // the chunk's tiles may be overwritten (4 epilogue warps)
  uint64_t fin;    // every MMA of the CTA has completed (MMA commit)
  unsigned long long wait_ns;  // a wait's limit
  uint32_t tbase;
  int abort;
  int issued;      // chunks whose loads the producer issued
};

constexpr size_t kQSmem = 1024 + kQ_BAR + sizeof(Bars);
constexpr size_t kKSmem = 1024 + kK_BAR + sizeof(Bars);
static_assert(kQSmem <= 232448 / 3, "three query CTAs per SM (their TMEM columns fit too)");
static_assert(kQ_R - kQ_Y == kTile, "the stacked A operand: dden right after dnum");
static_assert(kKSmem <= 232448 / 4, "four key CTAs per SM");

struct BParams {
  CUtensorMap tm_a, tm_b;   // query: Q, dY; key: K, V ([U*N rows][64] bf16, box 64 x 128, 128-byte swizzle)
  const uint8_t* tiles_t;   // [U*M] x 8 KB: rows e, columns c (S'^T resp. dS^T)
  const uint8_t* tiles_n;   // [U*M] x 8 KB: rows c, columns e (S' resp. dS)
  const float* mu;          // query: [U*M][64] fp32
  const float* zslots;      // [U*M][kX] fp32: z~ resp. dz at kD*kD
  __nv_bfloat16* g0;        // query: dq; key: dk  ([U*N][64])
  __nv_bfloat16* g1;        // key: dv
  float* out_slots;         // query: dS~ [c][e] and dz~ per slot
  unsigned* status;
  unsigned long long wait_ns;  // the limit of every wait (the default, or a diagnostic's shorter one)
  int N, L, M;
  float eps;
};

__device__ __forceinline__ bool ab_get(const int* ab) { return *reinterpret_cast<const volatile int*>(ab) != 0; }

__device__ __noinline__ bool bwait_slow(uint64_t* bar, uint32_t parity, int* ab, unsigned long long limit) {
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait_ns(bar, parity, 256)) return true;
    if (ab_get(ab)) return false;
    if (globaltimer_ns() - t0 > limit) break;
  }
  *reinterpret_cast<volatile int*>(ab) = 1;
  return false;
}
// ab: the CTA's abort flag; limit: the wait's limit in ns
__device__ __forceinline__ bool bwait(uint64_t* bar, uint32_t parity, int* ab, unsigned long long limit) {
  return mbar_test(bar, parity) || bwait_slow(bar, parity, ab, limit);
}
// Short wait (10 ms at most), only while winding down after an abort.
__device__ __noinline__ void drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait_ns(bar, parity, 1000))
    if (globaltimer_ns() - t0 > 10000000ull) return;
}

// 16-byte piece j (columns 8 j .. 8 j + 7) of row r of a 128-byte-swizzled [rows][64] bf16 tile.
__device__ __forceinline__ uint4* piece(uint8_t* tile, int r, int j) {
  return reinterpret_cast<uint4*>(tile + r * 128 + ((j ^ (r & 7)) << 4));
}
__device__ __forceinline__ void unpack8(uint4 u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    f[2 * m] = __uint_as_float(w[m] << 16);
    f[2 * m + 1] = __uint_as_float(w[m] & 0xffff0000u);
  }
}
__device__ __forceinline__ uint4 pack8(const float* v) {
  return make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]), pack_bf16(v[6], v[7]));
}

// phi in place (bf16) on row r of a chunk tile, and phi - bf16(phi) at the same place of `lo` when
// given; returns phi(row) . z + eps (fp32 phi) when z is given
__device__ __forceinline__ float phi_row(uint8_t* tile, int r, const float* z, float eps, uint8_t* lo = nullptr) {
  float den = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint4* p = piece(tile, r, j);
    float f[8];
    unpack8(*p, f);
#pragma unroll
    for (int x = 0; x < 8; ++x) {
      f[x] = phi_f(f[x]);
      if (z) den = fmaf(f[x], z[8 * j + x], den);
    }
    const uint4 hi = pack8(f);
    *p = hi;
    if (lo) {
      float h[8];
      unpack8(hi, h);
#pragma unroll
      for (int x = 0; x < 8; ++x) h[x] = f[x] - h[x];
      *piece(lo, r, j) = pack8(h);
    }
  }
  return den + eps;
}

// Common prologue: barriers, TMEM, tensor-map prefetch.
__device__ __forceinline__ void setup(Bars* b, uint32_t cols, const BParams& p, int warp, int lane) {
  if (threadIdx.x == 0) {
    mbar_init(&b->full, 1);
    mbar_init(&b->sfull, 1);
    mbar_init(&b->phi, kEpiWarps);
    mbar_init(&b->acc1, 1);
    mbar_init(&b->mid, kEpiWarps);
    mbar_init(&b->acc2, 1);
    mbar_init(&b->free_, kEpiWarps);
    mbar_init(&b->fin, 1);
    b->abort = 0;
    b->issued = 0;
    b->wait_ns = p.wait_ns;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(&b->tbase, cols);
    tmem_relinquish();
  }
  if (warp == kWarpProd && lane == 0) {
    prefetch_tmap(&p.tm_a);
    prefetch_tmap(&p.tm_b);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
}

// Producer: the block's two d x d tiles, z and (query) mu once, then the chunks' two tiles.
__device__ __forceinline__ void produce(const BParams& p, uint8_t* sm, Bars* b, int st_off, int sn_off, int z_off,
                                        int a_off, int b_off, size_t slot, int row0, int nch) {
  int* ab = &b->abort;
  mbar_arrive_expect_tx(&b->sfull, 2 * kSTile + kD * 4 + (p.mu ? kD * 4 : 0));
  bulk_load_1d(sm + st_off, p.tiles_t + slot * kSTile, kSTile, &b->sfull);
  bulk_load_1d(sm + sn_off, p.tiles_n + slot * kSTile, kSTile, &b->sfull);
  if (p.mu) bulk_load_1d(sm + z_off + kD * 4, p.mu + slot * kD, kD * 4, &b->sfull);
  bulk_load_1d(sm + z_off, p.zslots + slot * kX + kD * kD, kD * 4, &b->sfull);
  int j = 0;
  for (; j < nch; ++j) {
    if (j > 0 && !bwait(&b->free_, (j - 1) & 1, ab, b->wait_ns)) break;
    mbar_arrive_expect_tx(&b->full, 2 * kTile);
    tma_load_2d(sm + a_off, &p.tm_a, 0, row0 + j * kT, &b->full);
    tma_load_2d(sm + b_off, &p.tm_b, 0, row0 + j * kT, &b->full);
  }
  b->issued = j;
}

// Wind-down: after an abort wait (briefly) for the loads and MMAs in flight; then free TMEM.
__device__ __forceinline__ void finish(const BParams& p, Bars* b, uint32_t tmem, uint32_t cols, int warp) {
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) {
    drain(&b->fin, 0);
    if (ab_get(&b->abort)) {
      drain(&b->sfull, 0);
      if (b->issued > 0) drain(&b->full, (b->issued - 1) & 1);
      atomicOr(p.status, 1u);
    }
  }
  __syncthreads();
  if (warp == kWarpMma) tmem_dealloc(tmem, cols);
}

// ================================================================ query pass
__global__ void __launch_bounds__(kThreads, 3) tc_bwd_query_kernel(const __grid_constant__ BParams p) {
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  Bars* b = reinterpret_cast<Bars*>(sm + kQ_BAR);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int u = blockIdx.x / p.M, i = blockIdx.x % p.M, nch = p.L / kT;
  const size_t slot = (size_t)u * p.M + i;
  const int row0 = u * p.N + i * p.L;
  setup(b, kQCols, p, warp, lane);
  const uint32_t tmem = b->tbase;
  int* ab = &b->abort;

  if (warp == kWarpProd) {
    if (lane == 0) produce(p, sm, b, kQ_ST, kQ_SN, kQ_Z, kQ_Q, kQ_Y, slot, row0, nch);
    __syncwarp();
  } else if (warp == kWarpMma) {
    if (lane == 0) {
      const uint32_t q = smem_u32(sm + kQ_Q), n = smem_u32(sm + kQ_Y), r = smem_u32(sm + kQ_R);
      const uint32_t id_k = idesc_bf16_f32(128, 64, 0, 0), id_mn = idesc_bf16_f32(128, 64, 1, 1);
      const uint64_t a1 = smem_desc(q, 16, 1024), b1 = smem_desc(smem_u32(sm + kQ_ST), 16, 1024);
      const uint64_t a2 = smem_desc(n, 16, 1024), b2 = smem_desc(smem_u32(sm + kQ_SN), 16, 1024);
      const uint64_t a3 = smem_desc(n, r - n, 1024), b3 = smem_desc(q, 8192, 1024);
      if (bwait(&b->sfull, 0, ab, b->wait_ns)) {
        for (int j = 0; j < nch; ++j) {
          if (!bwait(&b->phi, j & 1, ab, b->wait_ns)) break;
          tc_fence_after();
          // phi(Q) S'[t][e] = sum_c phi(Q)[t][c] S'[c][e]: A = phi(Q) (K-major), B = S'^T tile (K-major)
#pragma unroll
          for (int k = 0; k < kD / 16; ++k) mma_bf16(tmem, a1 + k * 2, b1 + k * 2, id_k, k > 0);
          mma_commit(&b->acc1);
          if (!bwait(&b->mid, j & 1, ab, b->wait_ns)) break;
          tc_fence_after();
          // dnum S'^T[t][c] = sum_e dnum[t][e] S'[c][e]: A = dnum (K-major, over dY), B = S' tile
          // (K-major); into the columns of phi(Q) S', which the epilogue read before releasing dnum
#pragma unroll
          for (int k = 0; k < kD / 16; ++k) mma_bf16(tmem, a2 + k * 2, b2 + k * 2, id_k, k > 0);
          // [dS~^T ; dz~][m][c] += sum_t [dnum^T ; dden][m][t] phi(Q)[t][c]: A MN-major (the dnum
          // tile, then the dden tile r - n bytes on), B = phi(Q) (MN-major)
#pragma unroll
          for (int k = 0; k < kT / 16; ++k)
            mma_bf16(tmem + 64, a3 + k * (2048 >> 4), b3 + k * (2048 >> 4), id_mn, j > 0 || k > 0);
          mma_commit(&b->acc2);
        }
      }
      mma_commit(&b->fin);
    }
    __syncwarp();
  } else {
    const int qd = warp & 3, t = qd * 32 + lane;
    const uint32_t trow = tmem + ((uint32_t)(qd * 32) << 16);
    const float* z = reinterpret_cast<const float*>(sm + kQ_Z);
    uint8_t* qt = sm + kQ_Q;
    bool ok = bwait(&b->sfull, 0, ab, b->wait_ns);
    for (int j = 0; ok && j < nch; ++j) {
      ok = __all_sync(0xffffffffu, bwait(&b->full, j & 1, ab, b->wait_ns));
      if (!ok) break;
      const float den = phi_row(qt, t, z, p.eps);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&b->phi);
      ok = __all_sync(0xffffffffu, bwait(&b->acc1, j & 1, ab, b->wait_ns));
      if (!ok) break;
      tc_fence_after();
      // num = (den - eps) mu + phi(Q) S';  dnum = dY / den (bf16 tile), mu . dnum (fp32),
      // dden = -(dY . num) / den^2 (a tile of it repeated)
      const float inv = 1.f / den, dz0 = den - p.eps;
      const float* mu = z + kD;
      float s = 0.f, mdn = 0.f;
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        float nm[16], dy[16];
        tmem_ld16(trow + 16 * g, nm);
        unpack8(*piece(sm + kQ_Y, t, 2 * g), dy);
        unpack8(*piece(sm + kQ_Y, t, 2 * g + 1), dy + 8);
        tmem_ld_wait();
#pragma unroll
        for (int x = 0; x < 16; ++x) {
          s = fmaf(dy[x], fmaf(dz0, mu[16 * g + x], nm[x]), s);
          dy[x] *= inv;
          mdn = fmaf(mu[16 * g + x], dy[x], mdn);
        }
        *piece(sm + kQ_Y, t, 2 * g) = pack8(dy);  // dnum over the row's dY
        *piece(sm + kQ_Y, t, 2 * g + 1) = pack8(dy + 8);
      }
      const float dd = -s * inv * inv;
      const uint32_t ddw = pack_bf16(dd, dd);
      const uint4 rep = make_uint4(ddw, ddw, ddw, ddw);
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) *piece(sm + kQ_R, t, jj) = rep;
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&b->mid);
      ok = __all_sync(0xffffffffu, bwait(&b->acc2, j & 1, ab, b->wait_ns));
      if (!ok) break;
      tc_fence_after();
      // dq = min(1, phi(q)) (dnum S'^T + (mu . dnum + dden) z~)
      const float zc = mdn + dd;
      uint4* dst = reinterpret_cast<uint4*>(p.g0 + (size_t)(row0 + j * kT + t) * kD);
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        float gq[16], qf[16];
        tmem_ld16(trow + 16 * g, gq);
        unpack8(*piece(qt, t, 2 * g), qf);
        unpack8(*piece(qt, t, 2 * g + 1), qf + 8);
        tmem_ld_wait();
#pragma unroll
        for (int x = 0; x < 16; ++x) qf[x] = fminf(1.f, qf[x]) * fmaf(zc, z[16 * g + x], gq[x]);
        dst[2 * g] = pack8(qf);
        dst[2 * g + 1] = pack8(qf + 8);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&b->free_);
    }
    if (ok && !ab_get(ab)) {
      // lanes 0-63: dS~^T[e][c] -> the slot's dS~[c][e]; lane 64: dz~[c]
      // (tcgen05.ld is warp-collective: whole warps load, then the owning lanes store)
      float* out = p.out_slots + slot * kX;
      if (qd < 3) {
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          float v[16];
          tmem_ld16(trow + 64 + 16 * g, v);
          tmem_ld_wait();
          if (qd < 2) {
#pragma unroll
            for (int x = 0; x < 16; ++x) out[(16 * g + x) * kD + t] = v[x];
          } else if (lane == 0) {
#pragma unroll
            for (int x = 0; x < 16; ++x) out[kD * kD + 16 * g + x] = v[x];
          }
        }
      }
    }
  }
  finish(p, b, tmem, kQCols, warp);
}

// ================================================================ key pass
__global__ void __launch_bounds__(kThreads, 4) tc_bwd_key_kernel(const __grid_constant__ BParams p) {
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  Bars* b = reinterpret_cast<Bars*>(sm + kK_BAR);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int u = blockIdx.x / p.M, bb = blockIdx.x % p.M, nch = p.L / kT;
  const size_t slot = (size_t)u * p.M + bb;
  const int row0 = u * p.N + bb * p.L;
  setup(b, kKCols, p, warp, lane);
  const uint32_t tmem = b->tbase;
  int* ab = &b->abort;

  if (warp == kWarpProd) {
    if (lane == 0) produce(p, sm, b, kK_ST, kK_SN, kK_Z, kK_K, kK_V, slot, row0, nch);
    __syncwarp();
  } else if (warp == kWarpMma) {
    if (lane == 0) {
      const uint32_t id_k = idesc_bf16_f32(128, 64, 0, 0);
      const uint64_t ak = smem_desc(smem_u32(sm + kK_K), 16, 1024), av = smem_desc(smem_u32(sm + kK_V), 16, 1024);
      const uint64_t bt = smem_desc(smem_u32(sm + kK_ST), 16, 1024), bn = smem_desc(smem_u32(sm + kK_SN), 16, 1024);
      if (bwait(&b->sfull, 0, ab, b->wait_ns)) {
        for (int j = 0; j < nch; ++j) {
          if (!bwait(&b->phi, j & 1, ab, b->wait_ns)) break;
          tc_fence_after();
          // dv[t][e] = sum_c phi(K)[t][c] dS[c][e]: B = dS^T tile;  dphi(K)[t][c] = sum_e V[t][e] dS[c][e]: B = dS tile
#pragma unroll
          for (int k = 0; k < kD / 16; ++k) mma_bf16(tmem, ak + k * 2, bt + k * 2, id_k, k > 0);
#pragma unroll
          for (int k = 0; k < kD / 16; ++k) mma_bf16(tmem + 64, av + k * 2, bn + k * 2, id_k, k > 0);
          mma_commit(&b->acc1);
        }
      }
      mma_commit(&b->fin);
    }
    __syncwarp();
  } else {
    const int qd = warp & 3, t = qd * 32 + lane;
    const uint32_t trow = tmem + ((uint32_t)(qd * 32) << 16);
    const float* z = reinterpret_cast<const float*>(sm + kK_Z);
    uint8_t* kt = sm + kK_K;
    bool ok = bwait(&b->sfull, 0, ab, b->wait_ns);
    for (int j = 0; ok && j < nch; ++j) {
      ok = __all_sync(0xffffffffu, bwait(&b->full, j & 1, ab, b->wait_ns));
      if (!ok) break;
      phi_row(kt, t, nullptr, 0.f);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&b->phi);
      ok = __all_sync(0xffffffffu, bwait(&b->acc1, j & 1, ab, b->wait_ns));
      if (!ok) break;
      tc_fence_after();
      const size_t row = (size_t)(row0 + j * kT + t) * kD;
      uint4* dv = reinterpret_cast<uint4*>(p.g1 + row);
      uint4* dk = reinterpret_cast<uint4*>(p.g0 + row);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {  // 32 columns at a time: four loads in flight, one wait
        float gv[32], gk[32];
        tmem_ld16(trow + 32 * hh, gv);
        tmem_ld16(trow + 32 * hh + 16, gv + 16);
        tmem_ld16(trow + 64 + 32 * hh, gk);
        tmem_ld16(trow + 64 + 32 * hh + 16, gk + 16);
        tmem_ld_wait();
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          const int gg = 2 * hh + g;
          float kf[16];
          unpack8(*piece(kt, t, 2 * gg), kf);
          unpack8(*piece(kt, t, 2 * gg + 1), kf + 8);
#pragma unroll
          for (int x = 0; x < 16; ++x) kf[x] = fminf(1.f, kf[x]) * (gk[16 * g + x] + z[16 * gg + x]);
          dv[2 * gg] = pack8(gv + 16 * g);
          dv[2 * gg + 1] = pack8(gv + 16 * g + 8);
          dk[2 * gg] = pack8(kf);
          dk[2 * gg + 1] = pack8(kf + 8);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&b->free_);
    }
  }
  finish(p, b, tmem, kKCols, warp);
}

// ================================================================ summaries
// S_b^T and z_b in one M = 128 accumulator, as the forward's summary pass:
// D[m][c] += sum_t [V^T ; 1][m][t] phi(K)[t][c] (A: the V tile, then a tile of ones, 16 KB on;
// B = phi(K); both MN-major), with phi(K) as its bf16 high part plus its bf16 low part (two
// products; V and the ones are exact in bf16), so S and z are those of fp32 phi: dq depends on
// the small part of S~ that is not a multiple of z~, where bf16 phi(K) alone would cost ~1.5%.
constexpr int kS_K = 0, kS_V = kTile, kS_ONE = 2 * kTile, kS_LO = 3 * kTile, kS_BAR = 4 * kTile;
constexpr uint32_t kSCols = 64;
constexpr size_t kSSmem = 1024 + kS_BAR + sizeof(Bars);
static_assert(kSSmem <= 232448 / 3, "three summary CTAs per SM");

__global__ void __launch_bounds__(kThreads, 3) tc_bwd_summary_kernel(const __grid_constant__ BParams p) {
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  Bars* b = reinterpret_cast<Bars*>(sm + kS_BAR);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int u = blockIdx.x / p.M, bb = blockIdx.x % p.M, nch = p.L / kT;
  const size_t slot = (size_t)u * p.M + bb;
  const int row0 = u * p.N + bb * p.L;
  setup(b, kSCols, p, warp, lane);
  const uint32_t tmem = b->tbase;
  int* ab = &b->abort;

  if (warp == kWarpProd) {
    if (lane == 0) {
      int j = 0;
      for (; j < nch; ++j) {
        if (j > 0 && !bwait(&b->acc1, (j - 1) & 1, ab, b->wait_ns)) break;  // chunk j - 1's MMAs have read the tiles
        mbar_arrive_expect_tx(&b->full, 2 * kTile);
        tma_load_2d(sm + kS_K, &p.tm_a, 0, row0 + j * kT, &b->full);
        tma_load_2d(sm + kS_V, &p.tm_b, 0, row0 + j * kT, &b->full);
      }
      b->issued = j;
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    if (lane == 0) {
      const uint32_t v = smem_u32(sm + kS_V), one = smem_u32(sm + kS_ONE);
      const uint64_t da = smem_desc(v, one - v, 1024), db = smem_desc(smem_u32(sm + kS_K), 8192, 1024);
      const uint64_t dbl = smem_desc(smem_u32(sm + kS_LO), 8192, 1024);
      const uint32_t id = idesc_bf16_f32(128, 64, 1, 1);
      for (int j = 0; j < nch; ++j) {
        if (!bwait(&b->phi, j & 1, ab, b->wait_ns)) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < kT / 16; ++k) mma_bf16(tmem, da + k * (2048 >> 4), db + k * (2048 >> 4), id, j > 0 || k > 0);
#pragma unroll
        for (int k = 0; k < kT / 16; ++k) mma_bf16(tmem, da + k * (2048 >> 4), dbl + k * (2048 >> 4), id, true);
        mma_commit(&b->acc1);
      }
      mma_commit(&b->fin);
    }
    __syncwarp();
  } else {
    const int qd = warp & 3, t = qd * 32 + lane;
    const uint32_t trow = tmem + ((uint32_t)(qd * 32) << 16);
    const uint32_t one2 = pack_bf16(1.f, 1.f);
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) *piece(sm + kS_ONE, t, jj) = make_uint4(one2, one2, one2, one2);
    bool ok = true;
    for (int j = 0; ok && j < nch; ++j) {
      ok = __all_sync(0xffffffffu, bwait(&b->full, j & 1, ab, b->wait_ns));
      if (!ok) break;
      phi_row(sm + kS_K, t, nullptr, 0.f, sm + kS_LO);
      fence_proxy_async_smem();  // phi (and, the first time, the ones tile) -> tensor core reads
      __syncwarp();
      if (lane == 0) mbar_arrive(&b->phi);
    }
    if (ok) ok = __all_sync(0xffffffffu, bwait(&b->acc1, (nch - 1) & 1, ab, b->wait_ns));
    if (ok && !ab_get(ab)) {
      tc_fence_after();
      // lanes 0-63: S^T[e][c] -> the slot's S[c][e]; lane 64: z[c]  (whole warps load)
      float* out = p.out_slots + slot * kX;
      if (qd < 3) {
        float v[64];
#pragma unroll
        for (int g = 0; g < 4; ++g) tmem_ld16(trow + 16 * g, v + 16 * g);
        tmem_ld_wait();
        if (qd < 2) {
#pragma unroll
          for (int x = 0; x < 64; ++x) out[x * kD + t] = v[x];
        } else if (lane == 0) {
#pragma unroll
          for (int x = 0; x < 64; ++x) out[kD * kD + x] = v[x];
        }
      }
    }
  }
  finish(p, b, tmem, kSCols, warp);
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

// [rows][64] bf16, box 64 x 128, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  cuuint32_t box[2] = {(cuuint32_t)kD, (cuuint32_t)kT};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

unsigned long long g_wait_ns = kWaitNs;

}  // namespace

void tc_backward_set_wait_limit(unsigned long long ns) { g_wait_ns = ns == 0 ? kWaitNs : ns; }

bool tc_backward_supported(int B, int H, int N, int d, int block, mhla_dtype dt) {
  if (dt != MHLA_BF16 || d != kD || block <= 0 || block % kT != 0 || N % block != 0) return false;
  return (long long)B * H * N < (1ll << 31);
}

cudaError_t tc_backward_query_launch(int units, int N, int block, const void* q, const void* dy,
                                     const uint8_t* tiles_t, const uint8_t* tiles_n, const float* mu,
                                     const float* mixed, void* dq, float* dmixed, float eps, unsigned* status,
                                     cudaStream_t st) {
  BParams p;
  const uint64_t rows = (uint64_t)units * N;
  if (!make_map(&p.tm_a, q, rows) || !make_map(&p.tm_b, dy, rows)) return cudaErrorInvalidValue;
  p.tiles_t = tiles_t;
  p.tiles_n = tiles_n;
  p.mu = mu;
  p.zslots = mixed;
  p.g0 = static_cast<__nv_bfloat16*>(dq);
  p.g1 = nullptr;
  p.out_slots = dmixed;
  p.status = status;
  p.wait_ns = g_wait_ns;
  p.N = N;
  p.L = block;
  p.M = N / block;
  p.eps = eps;
  static SmemOptIn opt;
  cudaError_t e = opt.ensure((const void*)tc_bwd_query_kernel, (int)kQSmem);
  if (e != cudaSuccess) return e;
  tc_bwd_query_kernel<<<(unsigned)((size_t)units * p.M), kThreads, kQSmem, st>>>(p);
  note_launch();
  return cudaGetLastError();
}

cudaError_t tc_backward_summary_launch(int units, int N, int block, const void* k, const void* v, float* slots,
                                       unsigned* status, cudaStream_t st) {
  BParams p;
  const uint64_t rows = (uint64_t)units * N;
  if (!make_map(&p.tm_a, k, rows) || !make_map(&p.tm_b, v, rows)) return cudaErrorInvalidValue;
  p.tiles_t = nullptr;
  p.tiles_n = nullptr;
  p.mu = nullptr;
  p.zslots = nullptr;
  p.g0 = nullptr;
  p.g1 = nullptr;
  p.out_slots = slots;
  p.status = status;
  p.wait_ns = g_wait_ns;
  p.N = N;
  p.L = block;
  p.M = N / block;
  p.eps = 0.f;
  static SmemOptIn opt;
  cudaError_t e = opt.ensure((const void*)tc_bwd_summary_kernel, (int)kSSmem);
  if (e != cudaSuccess) return e;
  tc_bwd_summary_kernel<<<(unsigned)((size_t)units * p.M), kThreads, kSSmem, st>>>(p);
  note_launch();
  return cudaGetLastError();
}

cudaError_t tc_backward_key_launch(int units, int N, int block, const void* k, const void* v,
                                   const uint8_t* tiles_t, const uint8_t* tiles_n, const float* dslots, void* dk,
                                   void* dv, unsigned* status, cudaStream_t st) {
  BParams p;
  const uint64_t rows = (uint64_t)units * N;
  if (!make_map(&p.tm_a, k, rows) || !make_map(&p.tm_b, v, rows)) return cudaErrorInvalidValue;
  p.tiles_t = tiles_t;
  p.tiles_n = tiles_n;
  p.mu = nullptr;
  p.zslots = dslots;
  p.g0 = static_cast<__nv_bfloat16*>(dk);
  p.g1 = static_cast<__nv_bfloat16*>(dv);
  p.out_slots = nullptr;
  p.status = status;
  p.wait_ns = g_wait_ns;
  p.N = N;
  p.L = block;
  p.M = N / block;
  p.eps = 0.f;
  static SmemOptIn opt;
  cudaError_t e = opt.ensure((const void*)tc_bwd_key_kernel, (int)kKSmem);
  if (e != cudaSuccess) return e;
  tc_bwd_key_kernel<<<(unsigned)((size_t)units * p.M), kThreads, kKSmem, st>>>(p);
  note_launch();
  return cudaGetLastError();
}

}  // namespace mhla
