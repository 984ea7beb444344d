// bf16 MHLA forward on the sm_103a tensor cores: one persistent kernel per call.
//
// "MHLA: Restoring Expressivity of Linear Attention via Token-Level
// Multi-Head" §4.1 computes, per (batch, head):
//   S_b = sum_{t in b} phi(K_t) V_t^T,  z_b = sum_{t in b} phi(K_t)       (local KV summaries)
//   S~_i = sum_b m_ib S_b,  z~_i = sum_b m_ib z_b                          (multi-head mixing)
//   Y_t = phi(Q_t) S~_i / (phi(Q_t) . z~_i + eps)                           (output)
// with phi = ELU + 1 and eps from "Linear Attention notes" §四/§五.
//
// One CTA per SM (cooperative launch), 16 warps, a SUM pass, a MIX phase and
// an OUT pass; every hand-over inside a CTA is an mbarrier ring:
//   warp 0      TMA producer: the CTA's SUM chunks (K and V tiles), then its
//               OUT chunks (Q tile at once; S~ tile and z~ of the chunk's block
//               once every CTA has finished the MIX phase)
//   warps 8-15  phi: phi in place on each K / Q tile, 16 rows a warp; for an
//               OUT chunk also the fp32 denominator phi(Q_t) . z~ + eps
//   warp 1      MMA issuer (one thread): SUM  D = [V^T ; 1] phi(K)  (M 128,
//               N 64, K 128): rows 0-63 are the chunk's S^T, rows 64-127 its z;
//               OUT  D = phi(Q) S~  (M 128, N 64, K 64); four TMEM accumulators
//   warps 4-7   epilogue, one TMEM lane quadrant each: SUM -> the chunk's
//               partial (S^T bf16, z fp32) to global; OUT -> Y = D / den in
//               bf16, TMA store of the warp's 32 rows
//   warps 2-15  MIX phase, between the passes, behind a grid barrier on all
//               SUM partials: each CTA takes a range of summary rows (64 rows
//               of S^T and the z row per head), sums the chunk partials of each
//               block and mixes the block sums for every query block; writes
//               S~^T (bf16, the K-major layout the OUT MMA reads) and z~ (fp32),
//               then arrives at a second grid barrier
// Chunks go to CTAs with stride gridDim.x.  The producer keeps loading Q tiles
// during the MIX phase, so HBM stays busy across it.  The grid barriers need
// every CTA resident (one per SM, cooperative launch).  All waits are bounded:
// on time-out the kernel sets the status word and winds down.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace mhla {
namespace {

using namespace tc;

constexpr int kThreads = 512;
constexpr int kTile = 128;                  // tokens per chunk
constexpr int kD = 64;                      // head dimension of this kernel
constexpr int kTileBytes = kTile * kD * 2;  // 16 KB bf16 tile
constexpr int kStageBytes = 2 * kTileBytes; // SUM: K, V.  OUT: Q, S~^T (8 KB), z~ (256 B)
constexpr int kSTile = kD * kD * 2;         // 8 KB S~^T tile
constexpr int kNA = 4;                      // TMEM accumulators, 64 columns each
constexpr uint32_t kTmemCols = 512;         // SUM / OUT use the first kNA x 64 columns, MIX all
constexpr int kMixRows = kD + 1;            // MIX rows per head: 64 of S^T, then z
constexpr uint64_t kWaitLimitNs = 500000000ull;  // a wait gives up after 0.5 s (the default)

constexpr int kWarpProd = 0, kWarpMma = 1, kWarpMix = 2, kWarpEpi = 4, kWarpPhi = 8;
constexpr int kMixThreads = (16 - kWarpMix) * 32;  // warps 2-15 run the MIX phase
constexpr int kPhiWarps = 8;
constexpr int kBarMix = 1;                  // named barrier of the MIX phase (0 is __syncthreads)
constexpr int kBarZ = 2;                    // named barrier of warps 2-3 (z rows)

constexpr int kMaxNS = 5;
// The OUT pass re-cuts the input ring into kNSO slots of kOutStage bytes:
// Q tile (16 KB), S~^T tile (8 KB) and z~ (256 B).
constexpr int kOutStage = 25 * 1024;
constexpr int kNSO = 6;

struct Small {
  uint64_t full[kMaxNS], ready[kMaxNS], empty[kMaxNS];
  uint64_t fullO[kNSO], readyO[kNSO], emptyO[kNSO];  // the OUT pass's ring
  uint64_t acc_full[kNA], acc_empty[kNA];
  uint64_t mixf[2], mixe[2];  // MIX accumulators: TMEM columns [256 j, 256 j + 256)
  uint64_t mixs[kMaxNS];      // transposed MIX: the MMAs of MIX stage j have completed
  uint64_t wready;            // transposed MIX: the weight tiles are in place
  uint64_t fin;               // both MMA issuers' last commits
  uint32_t tbase;
  int abort;
  int last;
  int prod_q, prod_qo, mma_q;
};

// Dynamic shared memory, from a 1024-byte aligned base: input ring, ones
// tile, Y staging (4 warps x 4 KB; during the MIX phase, with the 16 KB after
// it, the transposed mixing matrix of up to MAXM blocks), den per accumulator
// and the barriers.
template <int MAXM>
struct Layout {
  static constexpr int kMaxM = MAXM;
  static constexpr int NS = 5;                            // stages of the input ring
  static constexpr int kOffOnes = NS * kStageBytes;       // 16 KB of bf16 ones (A rows 64..127 of SUM)
  static constexpr int kOffY = kOffOnes + kTileBytes;     // Y staging / mixing matrix
  static constexpr int kOffDen = kOffY + 32768;           // kNA x 128 fp32
  static constexpr int kOffSmall = kOffDen + kNA * kTile * 4;
  static constexpr size_t kBytes = 1024 + kOffSmall + sizeof(Small);
  static_assert(MAXM * MAXM * 4 <= 32768, "mixing matrix staging");
  static_assert(kNSO * kOutStage <= NS * kStageBytes, "OUT ring inside the input ring");
  static_assert(kBytes <= 232448, "shared memory budget");
};

struct Params {
  CUtensorMap tm_q, tm_k, tm_v;  // [heads*N rows][64] bf16, box 64 x 128, 128-byte swizzle
  CUtensorMap tm_y;              // same tensor shape, box 64 x 32
                                 // (2-D blocks: (64, gw, heads*gh) boxes of 128 / 32 tokens of a tile)
  CUtensorMap tm_p;              // chunk partials [heads*C rows][4096] bf16, box 64 x C (tensor-core MIX)
  CUtensorMap tm_ps;             // chunk partials [heads*C*64 rows][64] bf16, box 64 x 32 (SUM stores)
  CUtensorMap tm_pp;             // chunk partials as (c 64, x heads*C, e 64), box 64 x C x 2 (transposed MIX)
  const float* mixing;           // [H][M][M], m[h][i][b]
  __nv_bfloat16* ps;             // chunk partial S^T: [heads * C][64 e][64 c]
  float* pz;                     // chunk partial z: [heads * C][64]
  uint8_t* smix;                 // S~^T tiles: [heads * M] x 8 KB, K-major, 128-byte swizzle
  float* zmix;                   // z~: [heads * M][64]
  float* den_out;                // [heads * N] or null
  unsigned* ctr;                 // [1] finished CTAs, [2] SUM barrier, [3] MIX barrier
  unsigned* status;
  int heads, H, N, M, C, cpb, TS;  // C = chunks per head, cpb = chunks per block, TS = heads * C
  int tc_mix;                    // 1: S^T rows mixed on the tensor cores (C % 16 == 0, C <= 64 or C % 64 == 0)
  int XS;                        // tensor-core MIX units: heads * 64 (0 without tc_mix)
  int mix_t;                     // 1: transposed tensor-core MIX (C <= 64; see the MIX stages)
  int mix_n;                     // transposed MIX: N of its MMAs, M rounded up to 16
  int zx;                        // 1: the CTAs with a z row take no MIX units (C > 64, heads <= grid / 4)
  int grid2d;                    // 1: 2-D blocks (tokens on a gw-wide grid, blocks th x tw tiles)
  int normalise;                 // 0: Y is the numerator alone (den_out still the denominator)
  int strict;                    // 1: weights m_ib for b < i only (causal MHLA's mixed prefix)
  int mix_only;                  // 1: SUM and MIX only (S~, z~ left in the workspace), no OUT pass
  int gw, gh, tw, th, bpr;       // grid width / height, tile width / height, tiles per grid row
  unsigned long long wait_ns;    // limit of the producer's waits for the mixed summaries (kWaitLimitNs
                                 // unless a diagnostic shortened it)
  float eps;
};

// 2-D blocks: grid position (x = column, y = head * gh + row) of the token at offset `off`
// of chunk g, a chunk being 128 consecutive tokens of its block in the tile's row-major order.
struct GridPos {
  int x, y;
};
__device__ __forceinline__ GridPos grid_pos(const Params& p, int g, int off) {
  const int hd = g / p.C, gi = g - hd * p.C;
  const int b = gi / p.cpb;
  const int lo = (gi - b * p.cpb) * kTile + off;
  const int lr = lo / p.tw, lc = lo - lr * p.tw;
  const int br = b / p.bpr, bc = b - br * p.bpr;
  return {bc * p.tw + lc, hd * p.gh + br * p.th + lr};
}

// Q / K / V tile of chunk g: 128 rows of 64 (contiguous blocks: rows g * 128 ..; 2-D blocks:
// a box of whole tile rows, or 128 tokens of one tile row), the same 128-byte-swizzled image.
__device__ __forceinline__ void load_chunk(void* dst, const CUtensorMap* m, const Params& p, int g, uint64_t* bar,
                                           uint64_t pol) {
  if (p.grid2d) {
    const GridPos t = grid_pos(p, g, 0);
    tma_load_3d_hint(dst, m, 0, t.x, t.y, bar, pol);
  } else {
    tma_load_2d_hint(dst, m, 0, g * kTile, bar, pol);
  }
}

// Token index (head * N + t) of row `row` of chunk g.
__device__ __forceinline__ size_t chunk_token(const Params& p, int g, int row) {
  if (!p.grid2d) return (size_t)g * kTile + row;
  const GridPos t = grid_pos(p, g, row);
  return (size_t)t.y * p.gw + t.x;
}

// ------------------------------------------------------------------ waits
__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}


__device__ __forceinline__ int aborted(Small* sh) { return *reinterpret_cast<volatile int*>(&sh->abort); }
__device__ __forceinline__ void set_abort(Small* sh) { *reinterpret_cast<volatile int*>(&sh->abort) = 1; }

// mbarrier phase wait.  The waiting thread sleeps in the barrier unit (it
// issues nothing while suspended); false once the wait limit has passed (and
// then the CTA aborts) or as soon as another role has aborted.
__device__ __noinline__ bool bwait_slow(uint64_t* bar, uint32_t parity, Small* sh) {
  // A few polls, then suspended waits with a short limit: a waiter is not
  // always woken when the phase completes, so the limit bounds the delay,
  // and suspension keeps waiting warps off the issue slots and the barrier
  // unit.
  for (int i = 0; i < 16; ++i)
    if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait_ns(bar, parity, 128)) return true;
    if (aborted(sh)) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) break;
  }
  set_abort(sh);
  return false;
}

// A phase that has already completed costs one test and no call.
__device__ __forceinline__ bool bwait(uint64_t* bar, uint32_t parity, Small* sh) {
  return mbar_test(bar, parity) || bwait_slow(bar, parity, sh);
}

// Short wait (10 ms at most) used only while winding down after an abort.
__device__ __noinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait_ns(bar, parity, 1000))
    if (globaltimer_ns() - t0 > 10000000ull) return;
}

// Global counter wait (acquire): false after the wait limit or on abort.
__device__ __noinline__ bool gwait(const unsigned* p, unsigned target, Small* sh) {
  if (ld_acquire(p) >= target) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    __nanosleep(32);
    if (ld_acquire(p) >= target) return true;
    if (aborted(sh)) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) break;
  }
  set_abort(sh);
  return false;
}

// ------------------------------------------------------------------ phi
__device__ __forceinline__ uint32_t phi2(uint32_t w) {
  return pack_bf16(phi_f(__uint_as_float(w << 16)), phi_f(__uint_as_float(w & 0xffff0000u)));
}

// phi of 8 bf16 values in place; returns sum_j phi(x_j) z[j] in fp32.
__device__ __forceinline__ float phi8_dot(uint4& x, const float* z) {
  uint32_t w[4] = {x.x, x.y, x.z, x.w};
  float a = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float lo = phi_f(__uint_as_float(w[j] << 16));
    const float hi = phi_f(__uint_as_float(w[j] & 0xffff0000u));
    a = fmaf(lo, z[2 * j], a);
    a = fmaf(hi, z[2 * j + 1], a);
    w[j] = pack_bf16(lo, hi);
  }
  x = make_uint4(w[0], w[1], w[2], w[3]);
  return a;
}

// ------------------------------------------------------------------ stores
// MIX results go out through the load/store units: a warp stages rows of 128
// bytes in shared memory, then writes them as coalesced 16-byte pieces, four
// whole rows per instruction.  Staged row r holds its piece c at
// r * 128 + c * 16; global row r starts at dst + r * stride.
__device__ __forceinline__ void st_global_v4(void* p, uint4 v) {
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void warp_store_rows(const uint8_t* yb, uint8_t* dst, int nrows, size_t stride, int lane) {
  __syncwarp();
  for (int piece = lane; piece < nrows * 8; piece += 32) {
    const int r = piece >> 3, c = piece & 7;
    st_global_v4(dst + r * stride + c * 16, *reinterpret_cast<const uint4*>(yb + r * 128 + c * 16));
  }
  __syncwarp();
}

// ------------------------------------------------------------------ MIX stages
// The tensor-core MIX units of a CTA are the contiguous range [u0, u1) of the
// heads x 64 (head, row e of S^T) pairs.  A ring stage carries n <=
// mix_per_stage(C) consecutive units of one head: their chunk-partial boxes
// (C slots x 64 entries, C x 128 bytes each) from offset 0 (TMA) and the
// head's 128-row weight tile (row i: m[i][x / cpb] over the C slots x) at
// 16 KB, which the phi warps write from the mixing matrix.
// MMA: D (128 x 64 n) = W (128 x C) . [boxes] (C x 64 n), fp32 in TMEM.
// With M <= 32 the weight rows are repeated in every 32-row quarter, so each
// TMEM lane quadrant holds all M query blocks and epilogue warp k reads unit
// k's 64 columns from its own quadrant; otherwise rows 0..M-1 hold them once
// and each unit is its own N = 64 MMA chain.
constexpr int kMixWOff = 16384;
// With C > 64 partials a head's units go through the MMAs in K chunks of 64
// partials (one stage each, accumulating in TMEM).
__host__ __device__ __forceinline__ int mix_kslots(int C) { return C < kD ? C : kD; }
__host__ __device__ __forceinline__ int mix_nkc(int C) { return C / mix_kslots(C); }
__device__ __forceinline__ int mix_per_stage(int C) { return min(4, kMixWOff / (mix_kslots(C) * kD * 2)); }
__host__ __device__ __forceinline__ bool mix_rep(int M) { return M <= 32; }
// With zx set (C > 64 and few heads; only kernels with M > 32) the CTAs that
// mix a z row (heads rows over the grid, see mix_rows_all) take no units: the
// z rows then run beside the units instead of after them.  CTA b is then unit
// CTA b - (z rows before b).  The kernels with M <= 32 keep the plain split
// (their code stays as compact as before).
template <class L>
__device__ __forceinline__ int mix_ubound(const Params& p, int k) {
  if constexpr (L::kMaxM > 32) {
    if (p.zx) {
      const long long b = blockIdx.x, G = gridDim.x;
      if ((b + 1) * p.heads / G > b * p.heads / G) return 0;  // a z-row CTA: no units
      return (int)((b - b * p.heads / G + k) * p.XS / (G - p.heads));
    }
  }
  return (int)(((long long)blockIdx.x + k) * p.XS / gridDim.x);
}
template <class L>
__device__ __forceinline__ int mix_u0(const Params& p) { return mix_ubound<L>(p, 0); }
template <class L>
__device__ __forceinline__ int mix_u1(const Params& p) { return mix_ubound<L>(p, 1); }
// SUM chunks of this CTA (the OUT pass's accumulators follow theirs)
__device__ __forceinline__ int sum_chunks(const Params& p) {
  return (int)blockIdx.x < p.TS ? (p.TS - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
}
// units in the stage that starts at unit u
__device__ __forceinline__ int mix_stage_units(const Params& p, int u, int u1) {
  return min(min(mix_per_stage(p.C), u1 - u), (u / kD + 1) * kD - u);
}

// Transposed MIX (C <= 64).  The MMA computes D^T = P^T W^T: A = the
// chunk-partial boxes of a PAIR of units of one head (MN-major, M 128: unit k's
// 64 entries c are rows 64 k + c), B = the head's weight tile (K-major, row i =
// query block, column x = m[i][x / cpb]; N = M rounded up to 16), K = C.  TMEM
// lane 64 k + c, column i then holds S~_i^T[e_k][c].  A pair needs only N TMEM
// columns, so every pair of the CTA gets its own accumulator and no MMA waits
// for an epilogue; 128 / C pairs share a ring stage, and the weight tiles of
// the CTA's heads sit in the Y staging area (which the MIX phase does not use).
__device__ __forceinline__ int mix_pair_units(int u, int u1) { return min(2, min(u1 - u, (u / kD + 1) * kD - u)); }
__device__ __forceinline__ int mix_t_pps(const Params& p) { return 128 / p.C; }

// ------------------------------------------------------------------ roles
// Producer (one thread).  Returns the number of stages it filled.  The OUT
// stages' Q tiles are loaded as soon as a stage is free; their S~ / z~ loads
// wait for the MIX phase of every CTA (grid barrier 2).
template <class L>
__device__ bool mix_ready(const Params& p, bool& ready) {
  if (!ready && ld_acquire(&p.ctr[3]) >= gridDim.x) {
    fence_proxy_async_global();  // S~ / z~ were written by generic stores of other CTAs
    ready = true;
  }
  return ready;
}

__device__ void issue_mix_loads(const Params& p, uint8_t* sm, Small* sh, int qo, int g) {
  const int s = qo % kNSO;
  uint8_t* st = sm + s * kOutStage;
  const size_t blk = (size_t)(g / p.C) * p.M + (g % p.C) / p.cpb;
  bulk_load_1d(st + kTileBytes, p.smix + blk * kSTile, kSTile, &sh->fullO[s]);
  bulk_load_1d(st + kTileBytes + kSTile, p.zmix + blk * kD, kD * 4, &sh->fullO[s]);
}

template <class L>
__device__ int producer(const Params& p, uint8_t* sm, Small* sh) {
  constexpr int kNS = L::NS;
  const uint64_t once = policy_evict_first();  // Q, K, V are read once
  int q = 0;
  for (int g = blockIdx.x; g < p.TS; g += gridDim.x, ++q) {
    const int s = q % kNS;
    if (q >= kNS && !bwait(&sh->empty[s], ((q / kNS) - 1) & 1, sh)) return q;
    uint8_t* st = sm + s * kStageBytes;
    mbar_arrive_expect_tx(&sh->full[s], kStageBytes);
    load_chunk(st, &p.tm_k, p, g, &sh->full[s], once);
    load_chunk(st + kTileBytes, &p.tm_v, p, g, &sh->full[s], once);
  }
  // MIX units (head h, row e of S^T): the chunk partials' row e, once every CTA
  // has stored its partials (grid barrier 1); the phi warps add the weights
  const int u1 = mix_u1<L>(p);
  if (p.mix_t && mix_u0<L>(p) < u1) {
    if (!gwait(&p.ctr[2], gridDim.x, sh)) return q;
    fence_proxy_async_global();  // the partials were written by other CTAs' bulk stores
    const int pps = mix_t_pps(p), box = p.C * kD * 2;
    for (int u = mix_u0<L>(p); u < u1; ++q) {
      const int s = q % kNS;
      if (q >= kNS && !bwait(&sh->empty[s], ((q / kNS) - 1) & 1, sh)) return q;
      int np = 0;
      for (int uu = u; np < pps && uu < u1; ++np) uu += mix_pair_units(uu, u1);
      uint8_t* st = sm + s * kStageBytes;
      // one box per pair: rows e, e + 1 of its head's partials (past e = 63 the
      // box reads zeros; past the CTA's range, rows it does not use)
      mbar_arrive_expect_tx(&sh->full[s], np * 2 * box);
      for (int k = 0; k < pps && u < u1; ++k) {
        tma_load_3d(st + 2 * k * box, &p.tm_pp, 0, (u / kD) * p.C, u % kD, &sh->full[s]);
        u += mix_pair_units(u, u1);
      }
    }
  } else if (p.tc_mix && mix_u0<L>(p) < u1) {
    if (!gwait(&p.ctr[2], gridDim.x, sh)) return q;
    fence_proxy_async_global();  // the partials were written by other CTAs' bulk stores
    const int ks = mix_kslots(p.C), nkc = mix_nkc(p.C);
    for (int u = mix_u0<L>(p); u < u1;) {
      const int n = mix_stage_units(p, u, u1), h = u / kD;
      for (int kc = 0; kc < nkc; ++kc, ++q) {
        const int s = q % kNS;
        if (q >= kNS && !bwait(&sh->empty[s], ((q / kNS) - 1) & 1, sh)) return q;
        uint8_t* st = sm + s * kStageBytes;
        mbar_arrive_expect_tx(&sh->full[s], n * ks * kD * 2);
        for (int k = 0; k < n; ++k)
          tma_load_2d(st + k * ks * kD * 2, &p.tm_p, (u % kD + k) * kD, h * p.C + kc * ks, &sh->full[s]);
      }
      u += n;
    }
  }
  if (p.mix_only) return q;
  // OUT pass, on the OUT ring over the same memory: every SUM / MIX stage must
  // have been consumed first.  qm = first OUT stage without its S~ / z~ loads.
  for (int qq = q > kNS ? q - kNS : 0; qq < q; ++qq)
    if (!bwait(&sh->empty[qq % kNS], (qq / kNS) & 1, sh)) return q;
  int qo = 0, qm = 0;
  int gm = blockIdx.x;  // chunk of stage qm
  bool ready = false;
  for (int g = blockIdx.x; g < p.TS; g += gridDim.x, ++qo) {
    const int s = qo % kNSO;
    if (qo >= kNSO) {
      // wait for the slot; until the MIX phase is done, keep checking for it,
      // since the stages ahead cannot drain without their S~ / z~
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait_ns(&sh->emptyO[s], ((qo / kNSO) - 1) & 1, 500)) {
        if (!ready && mix_ready<L>(p, ready)) {
          for (; qm < qo; ++qm, gm += gridDim.x) issue_mix_loads(p, sm, sh, qm, gm);
        }
        if (aborted(sh)) break;
        if (globaltimer_ns() - t0 > p.wait_ns) {
          set_abort(sh);
          break;
        }
      }
      if (aborted(sh)) break;
    }
    uint8_t* st = sm + s * kOutStage;
    mbar_arrive_expect_tx(&sh->fullO[s], kTileBytes + kSTile + kD * 4);
    load_chunk(st, &p.tm_q, p, g, &sh->fullO[s], once);
    sh->prod_qo = qo + 1;
    if (mix_ready<L>(p, ready)) {
      for (; qm <= qo; ++qm, gm += gridDim.x) issue_mix_loads(p, sm, sh, qm, gm);
    }
  }
  // every OUT stage still needs its S~ / z~ before the consumers can finish
  const uint64_t t0 = globaltimer_ns();
  while (qm < qo && !aborted(sh)) {
    if (mix_ready<L>(p, ready)) {
      for (; qm < qo; ++qm, gm += gridDim.x) issue_mix_loads(p, sm, sh, qm, gm);
      break;
    }
    if (globaltimer_ns() - t0 > p.wait_ns) {
      set_abort(sh);
      break;
    }
    __nanosleep(200);
  }
  return q;
}

// phi warp w (0..7): rows 16w .. 16w+15 of every tile of one pass (0 SUM,
// 1 OUT); qs counts ring stages, qa accumulators (units), over all passes.
template <class L>
__device__ void phi_pass(const Params& p, uint8_t* sm, Small* sh, int w, int lane, int pass, int& qs, int& qa) {
  constexpr int kNS = L::NS;
  float* den = reinterpret_cast<float*>(sm + L::kOffDen);
  // 16-byte piece w*128 + lane + 32i of a tile holds row 16w + (lane>>3) + 4i;
  // physical piece lane&7 is logical piece (lane&7) ^ (row&7) (128-byte swizzle)
  const int r0 = lane >> 3;
  const int g0 = (lane & 7) ^ r0, g1 = (lane & 7) ^ (r0 + 4);
  // SUM stages come from the input ring (counter qs), OUT stages from the OUT ring
  int qo = 0;
  for (int g = blockIdx.x; g < p.TS; g += gridDim.x, ++qa) {
    const int s = pass == 0 ? qs % kNS : qo % kNSO;
    uint64_t* full = pass == 0 ? &sh->full[s] : &sh->fullO[s];
    uint64_t* ready = pass == 0 ? &sh->ready[s] : &sh->readyO[s];
    if (!bwait(full, pass == 0 ? (qs / kNS) & 1 : (qo / kNSO) & 1, sh)) return;
    if (pass == 0) ++qs;
    else ++qo;
    uint8_t* st = sm + (pass == 0 ? s * kStageBytes : s * kOutStage);
    uint4* t4 = reinterpret_cast<uint4*>(st) + w * 128 + lane;
    uint4 x[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] = t4[32 * i];
    if (pass == 0) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        x[i].x = phi2(x[i].x);
        x[i].y = phi2(x[i].y);
        x[i].z = phi2(x[i].z);
        x[i].w = phi2(x[i].w);
        t4[32 * i] = x[i];
      }
    } else {
      const int a = qa % kNA;
      // den[a] is free once the epilogue of the unit kNA earlier has read it
      if (qa >= kNA && !bwait(&sh->acc_empty[a], ((qa / kNA) - 1) & 1, sh)) return;
      const float4* zt = reinterpret_cast<const float4*>(st + kTileBytes + kSTile);
      float z0[8], z1[8];
      {
        const float4 u0 = zt[2 * g0], u1 = zt[2 * g0 + 1], v0 = zt[2 * g1], v1 = zt[2 * g1 + 1];
        z0[0] = u0.x; z0[1] = u0.y; z0[2] = u0.z; z0[3] = u0.w;
        z0[4] = u1.x; z0[5] = u1.y; z0[6] = u1.z; z0[7] = u1.w;
        z1[0] = v0.x; z1[1] = v0.y; z1[2] = v0.z; z1[3] = v0.w;
        z1[4] = v1.x; z1[5] = v1.y; z1[6] = v1.z; z1[7] = v1.w;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float dsum = phi8_dot(x[i], (i & 1) ? z1 : z0);
        t4[32 * i] = x[i];
        dsum += __shfl_xor_sync(0xffffffffu, dsum, 1);
        dsum += __shfl_xor_sync(0xffffffffu, dsum, 2);
        dsum += __shfl_xor_sync(0xffffffffu, dsum, 4);
        if ((lane & 7) == 0) den[a * kTile + w * 16 + r0 + 4 * i] = dsum + p.eps;
      }
    }
    fence_proxy_async_smem();  // phi tile -> tensor core reads
    __syncwarp();
    if (lane == 0) mbar_arrive(ready);
  }
}

// MIX weight tile of head hh, the A operand of the MIX MMAs (M 128 rows, K = C
// chunk partials): row r, column x is m[hh][i][x / cpb] with i = r % 32 (M <= 32:
// the query blocks repeated in the four TMEM lane quadrants) or i = r, for
// i < M and x < C, zero elsewhere.  Thread t (of 256) holds the bf16 piece
// (columns 8 (t % 8) ..) of rows t / 8 + 32 kk in v[kk] (v[0] for all kk when
// M <= 32).
__device__ __forceinline__ void mix_weight_values(const Params& p, int hh, int kc, int t, uint4 (&v)[4]) {
  const float* m = p.mixing + (size_t)hh * p.M * p.M;
  const int ks = mix_kslots(p.C), x0 = 8 * (t & 7);  // columns x0 .. x0 + 7: partials kc ks + x
  // block of each of the 8 partials (one division, then a running offset)
  int bc[8];
  {
    const int xg = kc * ks + x0;
    int b = xg / p.cpb, r = xg - b * p.cpb;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      bc[c] = b;
      if (++r == p.cpb) {
        r = 0;
        ++b;
      }
    }
  }
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    const int i = (t >> 3) + 32 * kk;
    float w[8];
#pragma unroll
    for (int c = 0; c < 8; ++c)
      w[c] = (i < p.M && x0 + c < ks && !(p.strict && bc[c] >= i)) ? __ldg(m + i * p.M + bc[c]) : 0.f;
    v[kk] = make_uint4(pack_bf16(w[0], w[1]), pack_bf16(w[2], w[3]), pack_bf16(w[4], w[5]), pack_bf16(w[6], w[7]));
    if (mix_rep(p.M)) break;
  }
}

// One MIX group (n units from unit u, TMEM columns 256 half ..) for the warp
// on TMEM lane quadrant qd: with M <= 32 the warp takes unit qd from its own
// quadrant, else rows 32 qd .. of every unit.  S~^T rows go out through the
// warp's staging buffer yb (whole rows, M <= 32) or straight to the tiles.
__device__ __forceinline__ void mix_group_rows(const Params& p, uint32_t tmem, int qd, int lane, int u, int n, int half,
                                               uint8_t* yb) {
  const bool rep4 = mix_rep(p.M);
  const int h = u / kD;
  const int i = rep4 ? lane : 32 * qd + lane;  // query block of this thread's row
  for (int k = 0; k < n; ++k) {
    if (rep4 ? k != qd : 32 * qd >= p.M) continue;
    float v[64];
    const uint32_t ta = tmem + (uint32_t)(256 * half + 64 * k) + ((uint32_t)(qd * 32) << 16);
    tmem_ld16(ta, v);
    tmem_ld16(ta + 16, v + 16);
    tmem_ld16(ta + 32, v + 32);
    tmem_ld16(ta + 48, v + 48);
    tmem_ld_wait();
    const int e = u % kD + k;
    if (rep4 && yb != nullptr) {
      // row e of the M tiles S~_i^T: lane i's 128-byte row (pieces already in
      // the tile's swizzled order) into this warp's staging, then out
      if (i < p.M) {
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(yb + i * 128 + (swz128(e, 8 * c) & 127)) =
              make_uint4(pack_bf16(v[8 * c], v[8 * c + 1]), pack_bf16(v[8 * c + 2], v[8 * c + 3]),
                         pack_bf16(v[8 * c + 4], v[8 * c + 5]), pack_bf16(v[8 * c + 6], v[8 * c + 7]));
      }
      warp_store_rows(yb, p.smix + (size_t)h * p.M * kSTile + e * 128, p.M, kSTile, lane);
    } else if (i < p.M) {
      uint8_t* dst = p.smix + ((size_t)h * p.M + i) * kSTile;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(dst + swz128(e, 8 * c)) =
            make_uint4(pack_bf16(v[8 * c], v[8 * c + 1]), pack_bf16(v[8 * c + 2], v[8 * c + 3]),
                       pack_bf16(v[8 * c + 4], v[8 * c + 5]), pack_bf16(v[8 * c + 6], v[8 * c + 7]));
    }
  }
}

// phi warps during the MIX stages: the weight tile of the stage's head, next
// to the chunk-partial boxes the producer loaded; warps 8-11 (TMEM lane
// quadrants 0-3) also take the rows of the odd MIX groups out of TMEM, after
// writing the next group's weights.
// An odd MIX group j (TMEM columns 256..511) for phi warp qd = 0..3.
__device__ __forceinline__ bool mix_odd_group(const Params& p, Small* sh, uint32_t tmem, int qd, int lane, int j, int u,
                                              int n) {
  if (!bwait(&sh->mixf[1], (j >> 1) & 1, sh)) return false;
  tc_fence_after();
  mix_group_rows(p, tmem, qd, lane, u, n, 1, nullptr);
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(&sh->mixe[1]);
  return true;
}

template <class L>
__device__ void phi_mix(const Params& p, uint8_t* sm, Small* sh, uint32_t tmem, int w, int lane, int& qs) {
  constexpr int kNS = L::NS;
  const int t = w * 32 + lane;  // rows t / 8 + 32 kk, piece t % 8 of the tile
  const int u1 = mix_u1<L>(p);
  const int nkc = mix_nkc(p.C);
  // kernels with M > 32 (long K chunks of partials) load the next stage's
  // mixing values one stage ahead; the others just before the stage
  constexpr bool kAhead = L::kMaxM > 32;
  uint4 wv[4];
  int wh = -1;  // (head, K chunk) of the values in wv
  if (kAhead && mix_u0<L>(p) < u1) {
    wh = ((mix_u0<L>(p) / kD) % p.H) * nkc;
    mix_weight_values(p, wh / nkc, 0, t, wv);
  }
  int j = 0, up = 0, np = 0;  // group index; the previous group's units
  for (int u = mix_u0<L>(p); u < u1; ++j) {
    const int n = mix_stage_units(p, u, u1), hh = (u / kD) % p.H;
    for (int kc = 0; kc < nkc; ++kc, ++qs) {
      if (!kAhead && hh * nkc + kc != wh) {  // the mixing values of a head (chunk) are loaded once
        mix_weight_values(p, hh, kc, t, wv);
        wh = hh * nkc + kc;
      }
      const int s = qs % kNS;
      if (!bwait(&sh->full[s], (qs / kNS) & 1, sh)) return;
      uint8_t* wtile = sm + s * kStageBytes + kMixWOff;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const int r = (t >> 3) + 32 * kk;
        *reinterpret_cast<uint4*>(wtile + r * 128 + (((t & 7) ^ (r & 7)) << 4)) = mix_rep(p.M) ? wv[0] : wv[kk];
      }
      fence_proxy_async_smem();  // weight tile -> tensor core reads
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->ready[s]);
      // the next stage's values (its head, its K chunk): their loads run while
      // this stage's MMAs do and while the next stage's boxes arrive
      int nh = hh, nk = kc + 1;
      if (nk == nkc) {
        nk = 0;
        nh = u + n < u1 ? ((u + n) / kD) % p.H : -1;
      }
      if (kAhead && nh >= 0 && nh * nkc + nk != wh) {
        mix_weight_values(p, nh, nk, t, wv);
        wh = nh * nkc + nk;
      }
    }
    if (w < 4 && j >= 1 && ((j - 1) & 1) && !mix_odd_group(p, sh, tmem, w, lane, j - 1, up, np)) return;
    up = u;
    np = n;
    u += n;
  }
  if (w < 4 && j >= 1 && ((j - 1) & 1)) mix_odd_group(p, sh, tmem, w, lane, j - 1, up, np);
}

// Transposed MIX, phi warps: the weight tiles of the heads of the CTA's units
// (head h0 + l at l N 128 bytes of the Y staging area; row i, piece pc holds
// m[h][i][x / cpb] for x = 8 pc .. 8 pc + 7, zero past M or C).  Thread t
// holds pieces t + 256 k (at most four: the tiles fit 16 KB); the values are
// read before grid barrier 1 and written once the staging area is free.
template <class L>
__device__ __forceinline__ void mix_t_weights_load(const Params& p, int w, int lane, uint4 (&pk)[4]) {
  const int u0 = mix_u0<L>(p), u1 = mix_u1<L>(p), N = p.mix_n;
  const int h0 = u0 / kD, nh = u0 < u1 ? (u1 - 1) / kD - h0 + 1 : 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int idx = w * 32 + lane + k * kPhiWarps * 32;
    if (idx >= nh * N * 8) break;
    const int pc = idx & 7, r = idx >> 3, i = r % N, l = r / N;
    const float* m = p.mixing + ((size_t)((h0 + l) % p.H) * p.M + i) * p.M;
    float v[8];
    int b = (8 * pc) / p.cpb, rr = 8 * pc - b * p.cpb;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      v[c] = (i < p.M && 8 * pc + c < p.C && !(p.strict && b >= i)) ? __ldg(m + b) : 0.f;
      if (++rr == p.cpb) {
        rr = 0;
        ++b;
      }
    }
    pk[k] = make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]), pack_bf16(v[6], v[7]));
  }
}

template <class L>
__device__ void mix_t_weights_store(const Params& p, uint8_t* sm, Small* sh, int w, int lane, const uint4 (&pk)[4]) {
  const int u0 = mix_u0<L>(p), u1 = mix_u1<L>(p), N = p.mix_n;
  const int h0 = u0 / kD, nh = u0 < u1 ? (u1 - 1) / kD - h0 + 1 : 0;
  uint8_t* wt = sm + L::kOffY;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int idx = w * 32 + lane + k * kPhiWarps * 32;
    if (idx >= nh * N * 8) break;
    const int pc = idx & 7, r = idx >> 3, i = r % N;
    *reinterpret_cast<uint4*>(wt + r * 128 + ((pc ^ (i & 7)) << 4)) = pk[k];
  }
  fence_proxy_async_smem();  // weight tiles -> tensor core reads
  __syncwarp();
  if (lane == 0) mbar_arrive(&sh->wready);
}

// Transposed MIX, warps 4-15 in three groups of four: group g takes the pairs
// j = g mod 3, and the warp on TMEM lane quadrant qd reads unit qd / 2 of the
// pair, entries c = 32 (qd % 2) + lane: S~_i^T[e][c] for the M query blocks i,
// in bf16, straight into the S~^T tiles.
template <class L>
__device__ bool mix_t_epi(const Params& p, Small* sh, uint32_t tmem, int g, int qd, int lane) {
  constexpr int MAXM = L::kMaxM;
  const int u1 = mix_u1<L>(p), pps = mix_t_pps(p), N = p.mix_n;
  const int kq = qd >> 1, c = 32 * (qd & 1) + lane;
  int j = 0;
  for (int u = mix_u0<L>(p); u < u1; ++j) {
    const int n = mix_pair_units(u, u1);
    if (j % 3 == g) {
      if (!bwait(&sh->mixs[j / pps], 0, sh)) return false;
      tc_fence_after();
      float v[MAXM];
      const uint32_t ta = tmem + (uint32_t)(j * N) + ((uint32_t)(qd * 32) << 16);
#pragma unroll
      for (int cc = 0; cc < MAXM / 16; ++cc)
        if (16 * cc < N) tmem_ld16(ta + 16 * cc, v + 16 * cc);
      tmem_ld_wait();
      if (kq < n) {
        const int uu = u + kq;
        uint8_t* dst = p.smix + (size_t)(uu / kD) * p.M * kSTile + swz128(uu % kD, c);
#pragma unroll
        for (int i = 0; i < MAXM; ++i)
          if (i < p.M) *reinterpret_cast<__nv_bfloat16*>(dst + (size_t)i * kSTile) = __float2bfloat16_rn(v[i]);
      }
    }
    u += n;
  }
  tc_fence_before();
  return true;
}

// MMA issuer (one thread).  Returns the number of chunks it issued.
template <class L>
__device__ int mma_issuer(const Params& p, uint8_t* sm, Small* sh, uint32_t tmem, int role, int pass_lo, int pass_hi) {
  constexpr int kNS = L::NS;
  const uint32_t ones = smem_u32(sm + L::kOffOnes);
  // SUM: A = V tile (MN-major) with the ones tile as M rows 64..127, B = phi(K)
  // (MN-major).  OUT: A = phi(Q) (K-major), B = S~^T (K-major).
  // MIX: A = weight tile (K-major, M 128), B = chunk-partial boxes (MN-major).
  const uint32_t idesc_sum = idesc_bf16_f32(128, 64, 1, 1);
  const uint32_t idesc_out = idesc_bf16_f32(128, 64, 0, 0);
  const uint32_t idesc_mix = idesc_bf16_f32(128, 64, 0, 1);
  // role 0 issues the even chunks of the SUM and OUT passes and every MIX
  // stage, role 1 the odd chunks (a single thread spends about as long on one
  // chunk's waits, MMAs and commits as the chunk takes to stream in)
  int qs = 0, qa = pass_lo == 2 ? sum_chunks(p) : 0;
  for (int pass = pass_lo; pass <= pass_hi; ++pass) {
    if (pass == 1 && p.mix_t) {
      if (role != 0 || mix_u0<L>(p) >= mix_u1<L>(p)) continue;
      if (!bwait(&sh->wready, 0, sh)) return qa;
      tc_fence_after();
      const int u1 = mix_u1<L>(p), pps = mix_t_pps(p), box = p.C * kD * 2, h0 = mix_u0<L>(p) / kD;
      const uint32_t idesc = idesc_bf16_f32(128, p.mix_n, 1, 0);
      const uint32_t wt = smem_u32(sm + L::kOffY);
      int j = 0;
      for (int u = mix_u0<L>(p), sg = 0; u < u1; ++sg, ++qs) {
        const int s = qs % kNS;
        if (!bwait(&sh->full[s], (qs / kNS) & 1, sh)) return qa;
        tc_fence_after();
        const uint32_t st = smem_u32(sm + s * kStageBytes);
        for (int k = 0; k < pps && u < u1; ++k, ++j) {
          // A: the pair's two boxes, one 64-entry atom each (box bytes apart);
          // B: the weight tile of the pair's head
          const uint64_t da = smem_desc(st + 2 * k * box, box, 1024);
          const uint64_t db = smem_desc(wt + (uint32_t)((u / kD - h0) * p.mix_n * 128), 16, 1024);
          for (int kk = 0; kk < p.C / 16; ++kk)
            mma_bf16(tmem + (uint32_t)(j * p.mix_n), da + kk * (2048 >> 4), db + kk * (32 >> 4), idesc, kk > 0);
          u += mix_pair_units(u, u1);
        }
        mma_commit(&sh->mixs[sg]);
        mma_commit(&sh->empty[s]);  // the stage is free once these MMAs have read it
      }
      continue;
    }
    if (pass == 1) {
      if (role != 0) continue;
      // MIX stages: TMEM columns [256 (j % 2), +256) for MIX stage j
      const int u1 = mix_u1<L>(p);
      const bool rep4 = mix_rep(p.M);
      int j = 0;
      const int ks = mix_kslots(p.C), nkc = mix_nkc(p.C);
      for (int u = mix_u0<L>(p); u < u1; ++j) {
        const int n = mix_stage_units(p, u, u1), half = j & 1;
        if (j >= 2 && !bwait(&sh->mixe[half], ((j >> 1) - 1) & 1, sh)) return qa;
        const uint32_t dst = tmem + (uint32_t)(256 * half);
        for (int kc = 0; kc < nkc; ++kc, ++qs) {
          const int s = qs % kNS;
          if (!bwait(&sh->ready[s], (qs / kNS) & 1, sh)) return qa;
          tc_fence_after();
          const uint32_t st = smem_u32(sm + s * kStageBytes);
          const uint64_t da = smem_desc(st + kMixWOff, 16, 1024);
          if (rep4) {
            // one chain, N = 64 n: the boxes are the N units, ks x 128 bytes apart
            const uint64_t db = smem_desc(st, ks * kD * 2, 1024);
            const uint32_t idesc = idesc_bf16_f32(128, 64 * n, 0, 1);
            for (int kk = 0; kk < ks / 16; ++kk)
              mma_bf16(dst, da + kk * (32 >> 4), db + kk * (2048 >> 4), idesc, kk > 0 || kc > 0);
          } else {
            for (int k = 0; k < n; ++k) {
              const uint64_t db = smem_desc(st + k * ks * kD * 2, 8192, 1024);
              for (int kk = 0; kk < ks / 16; ++kk)
                mma_bf16(dst + 64 * k, da + kk * (32 >> 4), db + kk * (2048 >> 4), idesc_mix, kk > 0 || kc > 0);
            }
          }
          if (kc == nkc - 1) mma_commit(&sh->mixf[half]);
          mma_commit(&sh->empty[s]);  // the stage is free once these MMAs have read it
        }
        u += n;
      }
      continue;
    }
    int qo = 0;  // OUT stages run on the OUT ring
    for (int g = blockIdx.x; g < p.TS; g += gridDim.x, ++qa) {
      const int s = pass == 0 ? qs % kNS : qo % kNSO, a = qa % kNA;
      uint64_t* ready = pass == 0 ? &sh->ready[s] : &sh->readyO[s];
      uint64_t* empty = pass == 0 ? &sh->empty[s] : &sh->emptyO[s];
      const uint32_t parity = pass == 0 ? (qs / kNS) & 1 : (qo / kNSO) & 1;
      if (pass == 0) ++qs;
      else ++qo;
      if ((qa & 1) != role) continue;
      if (qa >= kNA && !bwait(&sh->acc_empty[a], ((qa / kNA) - 1) & 1, sh)) return qa;
      if (!bwait(ready, parity, sh)) return qa;
      tc_fence_after();
      const uint32_t st = smem_u32(sm + (pass == 0 ? s * kStageBytes : s * kOutStage));
      const uint32_t dst = tmem + (uint32_t)(a * 64);
      // descriptors built once per stage; a K step only moves the start
      // address field (bytes >> 4 in the low bits)
      if (pass == 0) {
        const uint32_t v0 = st + kTileBytes;
        const uint64_t da = smem_desc(v0, ones - v0, 1024), db = smem_desc(st, 8192, 1024);
#pragma unroll
        for (int k = 0; k < kTile / 16; ++k) mma_bf16(dst, da + k * (2048 >> 4), db + k * (2048 >> 4), idesc_sum, k > 0);
      } else {
        const uint64_t da = smem_desc(st, 16, 1024), db = smem_desc(st + kTileBytes, 16, 1024);
#pragma unroll
        for (int k = 0; k < kD / 16; ++k) mma_bf16(dst, da + k * (32 >> 4), db + k * (32 >> 4), idesc_out, k > 0);
      }
      mma_commit(empty);             // the stage is free once these MMAs have read it
      mma_commit(&sh->acc_full[a]);  // and the accumulator is ready
    }
  }
  return qa;
}

// Epilogue warp for TMEM lane quadrant qd, one pass (0 SUM, 1 OUT); q counts
// the chunks across both passes, nst the Y stores.
template <class L>
__device__ void epi_pass(const Params& p, uint8_t* sm, Small* sh, uint32_t tmem, int qd, int lane, int pass, int& q,
                         int& nst) {
  const float* den = reinterpret_cast<const float*>(sm + L::kOffDen);
  uint8_t* yb = sm + L::kOffY + qd * 4096;
  const uint64_t once = policy_evict_first();  // Y is written once
  if (pass == 2) {
    // MIX groups (see the MMA issuer): the even ones (TMEM columns 0..255);
    // phi warps 8-11 take the odd ones
    const int u1 = mix_u1<L>(p);
    int j = 0;
    for (int u = mix_u0<L>(p); u < u1; ++j) {
      const int n = mix_stage_units(p, u, u1), half = j & 1;
      if (half) {
        u += n;
        continue;
      }
      if (!bwait(&sh->mixf[half], (j >> 1) & 1, sh)) return;
      tc_fence_after();
      mix_group_rows(p, tmem, qd, lane, u, n, half, yb);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->mixe[half]);
      u += n;
    }
    return;
  }
  {
    for (int g = blockIdx.x; g < p.TS; g += gridDim.x, ++q) {
      const int a = q % kNA;
      if (!bwait(&sh->acc_full[a], (q / kNA) & 1, sh)) return;
      tc_fence_after();
      const uint32_t ta = tmem + (uint32_t)(a * 64) + ((uint32_t)(qd * 32) << 16);
      float v[64];
      if (pass == 0) {
        if (qd < 3) {
          tmem_ld16(ta, v);
          tmem_ld16(ta + 16, v + 16);
          tmem_ld16(ta + 32, v + 32);
          tmem_ld16(ta + 48, v + 48);
          tmem_ld_wait();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->acc_empty[a]);
        // the chunk's partial goes out through this warp's staging buffer and
        // a bulk store: rows 32 qd .. 32 qd + 31 of S^T (qd 0, 1; bf16, 128-byte
        // swizzle for the tensor map), or z (qd 2: rows 64.. all hold it)
        if (qd < 3) {
          // two staging buffers per warp, as in the OUT pass
          uint8_t* yo = sm + L::kOffY + qd * 8192 + (nst & 1) * 4096;
          if (lane == 0 && nst >= 1) tma_store_wait_read1();  // the store of two chunks ago has read yo
          __syncwarp();
          if (qd < 2) {
#pragma unroll
            for (int c = 0; c < 8; ++c)
              *reinterpret_cast<uint4*>(yo + swz128(lane, 8 * c)) =
                  make_uint4(pack_bf16(v[8 * c], v[8 * c + 1]), pack_bf16(v[8 * c + 2], v[8 * c + 3]),
                             pack_bf16(v[8 * c + 4], v[8 * c + 5]), pack_bf16(v[8 * c + 6], v[8 * c + 7]));
          } else if (lane == 0) {
#pragma unroll
            for (int c = 0; c < 16; ++c)
              reinterpret_cast<float4*>(yo)[c] = make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (qd < 2) tma_store_2d(&p.tm_ps, yo, 0, g * kD + qd * 32);
            else bulk_store_1d(p.pz + (size_t)g * kD, yo, kD * 4);
            tma_store_commit();
          }
          ++nst;
        }
      } else {
        tmem_ld16(ta, v);
        tmem_ld16(ta + 16, v + 16);
        tmem_ld16(ta + 32, v + 32);
        tmem_ld16(ta + 48, v + 48);
        tmem_ld_wait();
        const int row = qd * 32 + lane;
        const float dn = den[a * kTile + row];
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->acc_empty[a]);
        if (p.den_out != nullptr) p.den_out[chunk_token(p, g, row)] = dn;
        const float r = p.normalise ? 1.f / dn : 1.f;
        // Y staging: two 4 KB buffers per warp (the whole 32 KB area is free
        // after the MIX phase); the store of two chunks ago has read this one
        uint8_t* yo = sm + L::kOffY + qd * 8192 + (nst & 1) * 4096;
        if (lane == 0 && nst >= 1) tma_store_wait_read1();
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(yo + swz128(lane, 8 * c)) =
              make_uint4(pack_bf16(v[8 * c] * r, v[8 * c + 1] * r), pack_bf16(v[8 * c + 2] * r, v[8 * c + 3] * r),
                         pack_bf16(v[8 * c + 4] * r, v[8 * c + 5] * r), pack_bf16(v[8 * c + 6] * r, v[8 * c + 7] * r));
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (p.grid2d) {
            const GridPos t = grid_pos(p, g, qd * 32);
            tma_store_3d_hint(&p.tm_y, yo, 0, t.x, t.y, once);
          } else {
            tma_store_2d_hint(&p.tm_y, yo, 0, g * kTile + qd * 32, once);
          }
          tma_store_commit();
        }
        ++nst;
      }
    }
  }
}

// SIMT mixing of one summary row for entry c: sums the chunk partials of each
// block (loads straight from L2) and mixes the block sums with the staged
// weights wt[b * MAXM + i] = m[i][b]; e = 0..63 is row e of S^T, e = 64 is z.
template <int MAXM>
__device__ void mix_row_simt(const Params& p, const float* wt, int h, int e, int c) {
  constexpr int kBatch = MAXM <= 32 ? 32 : 16;  // slot values loaded at once
  const size_t part0 = (size_t)h * p.C;         // first chunk partial of head h
  float acc[MAXM];
#pragma unroll
  for (int i = 0; i < MAXM; ++i) acc[i] = 0.f;
  float T = 0.f;
  int xin = 0, b = 0;
  for (int x0 = 0; x0 < p.C; x0 += kBatch) {
    const int n = min(kBatch, p.C - x0);
    float val[kBatch];
    if (e < kD) {
      const unsigned short* src = reinterpret_cast<const unsigned short*>(p.ps) + (part0 + x0) * (kD * kD) + e * kD + c;
#pragma unroll
      for (int k = 0; k < kBatch; ++k)
        val[k] = k < n ? __uint_as_float((uint32_t)__ldcg(src + (size_t)k * (kD * kD)) << 16) : 0.f;
    } else {
      const float* src = p.pz + (part0 + x0) * kD + c;
#pragma unroll
      for (int k = 0; k < kBatch; ++k) val[k] = k < n ? __ldcg(src + (size_t)k * kD) : 0.f;
    }
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      if (k >= n) break;
      T += val[k];
      if (++xin == p.cpb) {
        const float4* w4 = reinterpret_cast<const float4*>(wt + b * MAXM);
#pragma unroll
        for (int i = 0; i < MAXM / 4; ++i) {
          const float4 m4 = w4[i];
          acc[4 * i] = fmaf(m4.x, T, acc[4 * i]);
          acc[4 * i + 1] = fmaf(m4.y, T, acc[4 * i + 1]);
          acc[4 * i + 2] = fmaf(m4.z, T, acc[4 * i + 2]);
          acc[4 * i + 3] = fmaf(m4.w, T, acc[4 * i + 3]);
        }
        T = 0.f;
        xin = 0;
        ++b;
      }
    }
  }
  if (e < kD) {
#pragma unroll
    for (int i = 0; i < MAXM; ++i)
      if (i < p.M)
        *reinterpret_cast<__nv_bfloat16*>(p.smix + ((size_t)h * p.M + i) * kSTile + swz128(e, c)) =
            __float2bfloat16_rn(acc[i]);
  } else {
#pragma unroll
    for (int i = 0; i < MAXM; ++i)
      if (i < p.M) p.zmix[((size_t)h * p.M + i) * kD + c] = acc[i];
  }
}

// z row (e = 64) with a compile-time block length CPB and all C <= 32 chunk
// partials in registers: block sums first, then independent FMA chains.
template <int MAXM, int CPB>
__device__ void mix_z_row_fast(const Params& p, const float* wt, int h, int c) {
  constexpr int NB = 32 / CPB;
  const float* src = p.pz + (size_t)h * p.C * kD + c;
  float val[32];
#pragma unroll
  for (int k = 0; k < 32; ++k) val[k] = k < p.C ? __ldcg(src + (size_t)k * kD) : 0.f;
  float tb[NB];
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    float t = val[b * CPB];
#pragma unroll
    for (int k = 1; k < CPB; ++k) t += val[b * CPB + k];
    tb[b] = t;
  }
  float acc[MAXM];
#pragma unroll
  for (int i = 0; i < MAXM; ++i) acc[i] = 0.f;
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    if (b >= p.M) break;
    const float4* w4 = reinterpret_cast<const float4*>(wt + b * MAXM);
#pragma unroll
    for (int i = 0; i < MAXM / 4; ++i) {
      const float4 m4 = w4[i];
      acc[4 * i] = fmaf(m4.x, tb[b], acc[4 * i]);
      acc[4 * i + 1] = fmaf(m4.y, tb[b], acc[4 * i + 1]);
      acc[4 * i + 2] = fmaf(m4.z, tb[b], acc[4 * i + 2]);
      acc[4 * i + 3] = fmaf(m4.w, tb[b], acc[4 * i + 3]);
    }
  }
#pragma unroll
  for (int i = 0; i < MAXM; ++i)
    if (i < p.M) p.zmix[((size_t)h * p.M + i) * kD + c] = acc[i];
}

// Stages the transposed mixing matrix of head hh (zero-padded to MAXM) for
// the n threads of named barrier `bar`.
template <int MAXM>
__device__ void stage_weights(const Params& p, float* wt, int hh, int t, int n, int bar) {
  named_bar(bar, n);
  const float* mw = p.mixing + (size_t)hh * p.M * p.M;
  for (int j0 = 0; j0 < MAXM * MAXM; j0 += 16 * n) {  // 16 independent loads per thread in flight
    float v[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const int j = j0 + k * n + t;
      const int b = j / MAXM, i = j % MAXM;
      v[k] = (j < MAXM * MAXM && b < p.M && i < p.M && !(p.strict && b >= i)) ? __ldcg(mw + i * p.M + b) : 0.f;
    }
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const int j = j0 + k * n + t;
      if (j < MAXM * MAXM) wt[j] = v[k];
    }
  }
  named_bar(bar, n);
}

// Start of the MIX phase for warps 2-15 (448 threads): grid barrier 1, on
// every CTA's SUM partials (and MIX weights).  False after an abort.
__device__ bool mix_begin(const Params& p, Small* sh, int t) {
  named_bar(kBarMix, kMixThreads);
  bool ok = true;
  if (t == 0) {
    red_release_add(&p.ctr[2], 1u);
    ok = gwait(&p.ctr[2], gridDim.x, sh);
  }
  return group_and(kBarMix, kMixThreads, ok && !aborted(sh));
}

// End of the MIX phase: this CTA's share of S~ / z~ is stored; arrive at grid
// barrier 2, which the producers wait on before loading S~ / z~.
__device__ void mix_end(const Params& p, int t) {
  named_bar(kBarMix, kMixThreads);
  if (t == 0) red_release_add(&p.ctr[3], 1u);
}

// Sum of chunk partials x0 .. x1-1 of head h, row e (e < 64: row e of S^T in
// bf16, e = 64: z in fp32), entry c; up to 16 loads in flight.
__device__ __forceinline__ float sum_partials(const Params& p, int h, int e, int c, int x0, int x1) {
  float T = 0.f;
  for (int xb = x0; xb < x1; xb += 16) {
    const int n = min(16, x1 - xb);
    float val[16];
    if (e < kD) {
      const unsigned short* src =
          reinterpret_cast<const unsigned short*>(p.ps) + ((size_t)h * p.C + xb) * (kD * kD) + e * kD + c;
#pragma unroll
      for (int k = 0; k < 16; ++k)
        val[k] = k < n ? __uint_as_float((uint32_t)__ldcg(src + (size_t)k * (kD * kD)) << 16) : 0.f;
    } else {
      const float* src = p.pz + ((size_t)h * p.C + xb) * kD + c;
#pragma unroll
      for (int k = 0; k < 16; ++k) val[k] = k < n ? __ldcg(src + (size_t)k * kD) : 0.f;
    }
#pragma unroll
    for (int k = 0; k < 16; ++k) T += val[k];
  }
  return T;
}

// SIMT MIX of all summary rows (when the tensor-core MIX does not apply), by
// warps 2-15 (448 threads = 7 groups of 64, thread c of a group on entry c):
// the CTA takes rows [blockIdx.x R / G, (blockIdx.x + 1) R / G) of the R =
// heads x 65 rows, one row at a time.  The mixing is linear, so a row's chunk
// partials are cut into units - whole blocks (M >= 7) or equal slices of one
// block (M < 7) - and each group sums the partials of its units and adds
// m[i][b] x (unit sum) into its accumulator for every query block i; the 7
// accumulators are then added in shared memory, kRound query blocks at a time.
template <int MAXM>
__device__ void mix_rows_all(const Params& p, uint8_t* sm, int t, bool zonly) {
  using L = Layout<MAXM>;
  constexpr int kGroups = kMixThreads / kD;  // 7
  constexpr int kRound = 8;
  static_assert(MAXM * MAXM * 4 + kGroups * kRound * kD * 4 <= 32768, "MIX staging");
  float* wt = reinterpret_cast<float*>(sm + L::kOffY);                       // [b][i] = m[i][b]
  float* red = reinterpret_cast<float*>(sm + L::kOffY + MAXM * MAXM * 4);    // [g][kRound][64]
  const unsigned G = gridDim.x;
  const int rows_per_head = zonly ? 1 : kMixRows;  // zonly: the z rows alone
  const int R = p.heads * rows_per_head;
  const int r0 = (int)((long long)blockIdx.x * R / G), r1 = (int)((long long)(blockIdx.x + 1) * R / G);
  const int g = t / kD, c = t % kD;
  const int S = p.M >= kGroups ? 1 : (kGroups + p.M - 1) / p.M;  // slices per block
  const int units = p.M * S;
  int cur_hh = -1;
  for (int row = r0; row < r1; ++row) {
    const int h = row / rows_per_head, e = zonly ? kD : row % kMixRows;
    if (h % p.H != cur_hh) {
      cur_hh = h % p.H;
      stage_weights<MAXM>(p, wt, cur_hh, t, kMixThreads, kBarMix);
    }
    float acc[MAXM];
#pragma unroll
    for (int i = 0; i < MAXM; ++i) acc[i] = 0.f;
    for (int un = g; un < units; un += kGroups) {
      const int b = un / S, sl = un % S;
      const int x0 = b * p.cpb + (sl * p.cpb) / S, x1 = b * p.cpb + ((sl + 1) * p.cpb) / S;
      const float T = sum_partials(p, h, e, c, x0, x1);
      const float4* w4 = reinterpret_cast<const float4*>(wt + b * MAXM);
#pragma unroll
      for (int i = 0; i < MAXM / 4; ++i) {
        const float4 m4 = w4[i];
        acc[4 * i] = fmaf(m4.x, T, acc[4 * i]);
        acc[4 * i + 1] = fmaf(m4.y, T, acc[4 * i + 1]);
        acc[4 * i + 2] = fmaf(m4.z, T, acc[4 * i + 2]);
        acc[4 * i + 3] = fmaf(m4.w, T, acc[4 * i + 3]);
      }
    }
#pragma unroll
    for (int i0 = 0; i0 < MAXM; i0 += kRound) {
      if (i0 >= p.M) break;
#pragma unroll
      for (int ii = 0; ii < kRound; ++ii) red[(g * kRound + ii) * kD + c] = acc[i0 + ii];
      named_bar(kBarMix, kMixThreads);
      for (int idx = t; idx < kRound * kD; idx += kMixThreads) {
        const int ii = idx / kD, i = i0 + ii, cc = idx % kD;
        if (i < p.M) {
          float v = 0.f;
#pragma unroll
          for (int gg = 0; gg < kGroups; ++gg) v += red[(gg * kRound + ii) * kD + cc];
          if (e < kD)
            *reinterpret_cast<__nv_bfloat16*>(p.smix + ((size_t)h * p.M + i) * kSTile + swz128(e, cc)) =
                __float2bfloat16_rn(v);
          else
            p.zmix[((size_t)h * p.M + i) * kD + cc] = v;
        }
      }
      named_bar(kBarMix, kMixThreads);
    }
  }
}

// z rows of the heads h = blockIdx.x + k G, by warps 2-3 (64 threads), while
// the other warps run the tensor-core MIX units.
template <int MAXM>
__device__ void mix_z_rows(const Params& p, uint8_t* sm, int c) {
  using L = Layout<MAXM>;
  float* wt = reinterpret_cast<float*>(sm + L::kOffY + 16384);  // the epilogue warps stage in the lower half
  int cur_hh = -1;
  for (int h = blockIdx.x; h < p.heads; h += gridDim.x) {
    if (h % p.H != cur_hh) {
      cur_hh = h % p.H;
      stage_weights<MAXM>(p, wt, cur_hh, c, 64, kBarZ);
    }
    // (with M > 32 there are more than 32 chunks, so the fast rows never apply)
    if constexpr (MAXM <= 32) {
      if (p.C <= 32 && p.cpb == 2) { mix_z_row_fast<MAXM, 2>(p, wt, h, c); continue; }
      if (p.C <= 32 && p.cpb == 1) { mix_z_row_fast<MAXM, 1>(p, wt, h, c); continue; }
      if (p.C <= 32 && p.cpb == 4) { mix_z_row_fast<MAXM, 4>(p, wt, h, c); continue; }
    }
    mix_row_simt<MAXM>(p, wt, h, kD, c);
  }
}

template <int MAXM>
__global__ void __launch_bounds__(kThreads, 1) mhla_tc_kernel(const __grid_constant__ Params p) {
  using L = Layout<MAXM>;
  constexpr int kNS = L::NS;
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  Small* sh = reinterpret_cast<Small*>(sm + L::kOffSmall);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < kNS; ++s) {
      mbar_init(&sh->full[s], 1);
      mbar_init(&sh->ready[s], kPhiWarps);
      mbar_init(&sh->empty[s], 1);
    }
    for (int s = 0; s < kNSO; ++s) {
      mbar_init(&sh->fullO[s], 1);
      mbar_init(&sh->readyO[s], kPhiWarps);
      mbar_init(&sh->emptyO[s], 1);
    }
    for (int a = 0; a < kNA; ++a) {
      mbar_init(&sh->acc_full[a], 1);
      mbar_init(&sh->acc_empty[a], 4);
    }
    for (int hf = 0; hf < 2; ++hf) {
      mbar_init(&sh->mixf[hf], 1);
      mbar_init(&sh->mixe[hf], 4);
    }
    sh->abort = 0;
    sh->prod_q = 0;
    sh->prod_qo = 0;
    sh->mma_q = 0;
    mbar_init(&sh->fin, 2);
    for (int j = 0; j < kMaxNS; ++j) mbar_init(&sh->mixs[j], 1);
    mbar_init(&sh->wready, kPhiWarps);
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(&sh->tbase, kTmemCols);
    tmem_relinquish();
  }
  if (warp == kWarpProd && lane == 0) {
    prefetch_tmap(&p.tm_q);
    prefetch_tmap(&p.tm_k);
    prefetch_tmap(&p.tm_v);
    prefetch_tmap(&p.tm_y);
    if (p.mix_t) prefetch_tmap(&p.tm_pp);
    else if (p.tc_mix) prefetch_tmap(&p.tm_p);
  }
  for (int i = tid; i < kTileBytes / 16; i += kThreads)
    reinterpret_cast<uint4*>(sm + L::kOffOnes)[i] = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh->tbase;

  if (warp == kWarpProd) {
    if (lane == 0) sh->prod_q = producer<L>(p, sm, sh);
    __syncwarp();
  } else if (warp == kWarpMma) {
    if (lane == 0) {
      mma_issuer<L>(p, sm, sh, tmem, 0, 0, p.mix_only ? 1 : 2);
      mma_commit(&sh->fin);  // arrives once this thread's MMAs have all completed
    }
    __syncwarp();
  } else {
    // warps 2-15: SUM pass (phi and epilogue warps), MIX phase (all), OUT pass
    const int t = tid - kWarpMix * 32;
    int q = 0, qs = 0, nst = 0;
    if (warp == kWarpMix) {  // the second MMA issuer: odd SUM chunks
      if (lane == 0) mma_issuer<L>(p, sm, sh, tmem, 1, 0, 0);
      __syncwarp();
    }
    if (warp >= kWarpPhi) phi_pass<L>(p, sm, sh, warp - kWarpPhi, lane, 0, qs, q);
    else if (warp >= kWarpEpi) {
      epi_pass<L>(p, sm, sh, tmem, warp - kWarpEpi, lane, 0, q, nst);
      // the SUM partials are read after grid barrier 1, some through TMA
      if (lane == 0) tma_store_wait_all0();
      fence_proxy_async_global();
    }
    uint4 wpk[4];
    if (p.mix_t && warp >= kWarpPhi) mix_t_weights_load<L>(p, warp - kWarpPhi, lane, wpk);
    if (mix_begin(p, sh, t)) {
      if (p.mix_t) {
        if (warp >= kWarpPhi) mix_t_weights_store<L>(p, sm, sh, warp - kWarpPhi, lane, wpk);
        if (warp >= kWarpEpi) mix_t_epi<L>(p, sh, tmem, (warp - kWarpEpi) >> 2, warp & 3, lane);
        else mix_z_rows<MAXM>(p, sm, t);
      } else if (p.tc_mix) {
        if (warp >= kWarpPhi) phi_mix<L>(p, sm, sh, tmem, warp - kWarpPhi, lane, qs);
        else if (warp >= kWarpEpi) {
          epi_pass<L>(p, sm, sh, tmem, warp - kWarpEpi, lane, 2, q, nst);
        }
        else if (p.C <= kD) mix_z_rows<MAXM>(p, sm, t);
        // with more than 64 partials the z rows take warps 2-15 after the units
        if (p.C > kD) mix_rows_all<MAXM>(p, sm, t, true);
      } else {
        mix_rows_all<MAXM>(p, sm, t, false);
      }
      mix_end(p, t);
      if (p.mix_only) {
      } else if (warp >= kWarpPhi) {
        phi_pass<L>(p, sm, sh, warp - kWarpPhi, lane, 1, qs, q);
      } else if (warp >= kWarpEpi) {
        epi_pass<L>(p, sm, sh, tmem, warp - kWarpEpi, lane, 1, q, nst);
      } else if (warp == kWarpMix && lane == 0) {
        mma_issuer<L>(p, sm, sh, tmem, 1, 2, 2);  // odd OUT chunks
      }
    }
    if (warp == kWarpMix && lane == 0) mma_commit(&sh->fin);
    __syncwarp();
    if (warp >= kWarpEpi && warp < kWarpPhi && lane == 0) tma_store_wait_all0();
  }
  __syncthreads();

  // Wind down.  On the normal path every wait below is already satisfied; after
  // an abort they let TMA loads and MMAs still in flight finish first.
  if (tid == 0 && aborted(sh)) {
    const int nq = sh->prod_q;
    for (int q = nq > kNS ? nq - kNS : 0; q < nq; ++q) drain_wait(&sh->full[q % kNS], (q / kNS) & 1);
    const int no = sh->prod_qo;
    for (int q = no > kNSO ? no - kNSO : 0; q < no; ++q) drain_wait(&sh->fullO[q % kNSO], (q / kNSO) & 1);
    drain_wait(&sh->fin, 0);  // every MMA issued has completed
    atomicOr(p.status, 1u);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tmem, kTmemCols);

  // The last CTA out leaves the counters at zero for the next call.
  if (tid == 0) {
    __threadfence();
    sh->last = atomicAdd(&p.ctr[1], 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (sh->last && tid == 0) {
    __threadfence();
    p.ctr[2] = 0;
    p.ctr[3] = 0;
    p.ctr[1] = 0;
  }
}

// ------------------------------------------------------------------- host
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
bool make_map_2d(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows, uint64_t inner = kD) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)inner * 2};
  cuuint32_t box[2] = {(cuuint32_t)kD, box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Q / K / V / Y of 2-D blocks: (64, gw, rows = heads * gh) bf16, box 64 x bw x bh, 128-byte swizzle.
bool make_map_grid(CUtensorMap* m, const void* base, uint64_t gw, uint64_t rows, uint32_t bw, uint32_t bh) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)gw, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)gw * kD * 2};
  cuuint32_t box[3] = {(cuuint32_t)kD, bw, bh};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The chunk partials [heads * C][64 e][64 c] bf16 as a 3-D tensor (c, x =
// head * C + chunk, e), box 64 x C x 2: the two units of a transposed-MIX pair,
// each a C x 128-byte box with the 128-byte swizzle.
bool make_map_pairs(CUtensorMap* m, const void* base, int heads, int C) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)heads * C, (cuuint64_t)kD};
  cuuint64_t strides[2] = {(cuuint64_t)kD * kD * 2, (cuuint64_t)kD * 2};
  cuuint32_t box[3] = {(cuuint32_t)kD, (cuuint32_t)C, 2};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct TcPlan {
  int C, M, cpb;
  bool tc_mix;  // S^T rows mixed on the tensor cores
  size_t off_ps, off_pz, off_smix, off_zmix, total;
};

inline size_t a256(size_t x) { return (x + 255) & ~size_t(255); }

TcPlan tc_plan(const MhlaShape& s) {
  TcPlan p;
  p.C = s.N / kTile;
  p.M = s.M();
  p.cpb = s.block / kTile;
  const size_t heads = (size_t)s.heads();
  size_t off = kWorkspacePrefix;
  p.off_ps = off;   off = a256(off + heads * p.C * (size_t)kD * kD * 2);
  p.off_pz = off;   off = a256(off + heads * p.C * (size_t)kD * sizeof(float));
  p.off_smix = off; off = a256(off + heads * p.M * (size_t)kSTile);
  p.off_zmix = off; off = a256(off + heads * p.M * (size_t)kD * sizeof(float));
  p.tc_mix = p.C % 16 == 0 && (p.C <= kD || p.C % kD == 0);
  p.total = off;
  return p;
}

// Whether the transposed MIX applies with this grid: C <= 64, and every CTA's
// pairs fit the TMEM columns, its weight tiles the 16 KB below the z weights,
// and its MIX stages the input ring once.
bool mix_t_fits(const TcPlan& pl, int heads, int grid) {
  if (!pl.tc_mix || pl.C > kD || grid <= 0) return false;
  const int N = (pl.M + 15) / 16 * 16;
  const long long upc = ((long long)heads * kD + grid - 1) / grid;  // units of a CTA, at most
  const long long hs = (upc - 1) / kD + 2;                          // heads they can touch
  const long long pairs = (upc + 1) / 2 + hs;                       // a head boundary splits a pair
  const long long pps = 128 / pl.C;
  return hs * N * 128 <= 16384 && pairs * N <= (long long)kTmemCols && (pairs + pps - 1) / pps <= kMaxNS;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

template <int MAXM>
cudaError_t launch_t(const Params& p, int grid, cudaStream_t st) {
  static SmemOptIn opt_in;
  if (cudaError_t e = opt_in.ensure((const void*)mhla_tc_kernel<MAXM>, (int)Layout<MAXM>::kBytes); e != cudaSuccess)
    return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Layout<MAXM>::kBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mhla_tc_kernel<MAXM>, p);
}

}  // namespace

bool tc_mhla_supported(const MhlaShape& s, mhla_dtype dt, MixMode mode) {
  if (!s.plain_phi()) return false;  // ELU + 1 without decay only
  if (dt != MHLA_BF16 || s.d != kD || mode != MIX_FULL) return false;
  if (s.block % kTile != 0 || s.N % kTile != 0) return false;
  // 2-D blocks: a 128-token chunk is whole tile rows (tw divides 128) or part of one
  // (128 divides tw); so is a 32-token piece of Y (tw divides 32, or 32 divides tw)
  if (s.grid() && !(kTile % s.tw == 0 || s.tw % kTile == 0)) return false;
  if ((long long)s.heads() * s.N >= (1ll << 31)) return false;
  if (s.heads() > kMaxCounterHeads) return false;
  return s.M() <= 64;
}

size_t tc_mhla_workspace(const MhlaShape& s) { return tc_plan(s).total; }

namespace {
unsigned long long g_wait_ns = kWaitLimitNs;

cudaError_t tc_mhla_run(const MhlaShape& s, const void* q, const void* k, const void* v, const float* mixing,
                        void* y, float* den_out, float eps, bool strict, bool mix_only, void* ws, cudaStream_t st) {
  const TcPlan pl = tc_plan(s);
  char* w = static_cast<char*>(ws);
  Params p;
  const uint64_t rows = (uint64_t)s.heads() * s.N;
  if (s.grid()) {
    const uint64_t grows = (uint64_t)s.heads() * s.gh;
    const uint32_t bw = s.tw < kTile ? s.tw : kTile, yw = s.tw < 32 ? s.tw : 32;
    if (!make_map_grid(&p.tm_q, q, s.gw, grows, bw, kTile / bw) ||
        !make_map_grid(&p.tm_k, k, s.gw, grows, bw, kTile / bw) ||
        !make_map_grid(&p.tm_v, v, s.gw, grows, bw, kTile / bw) ||
        !make_map_grid(&p.tm_y, y, s.gw, grows, yw, 32 / yw))
      return cudaErrorInvalidValue;
  } else if (!make_map_2d(&p.tm_q, q, rows, kTile) || !make_map_2d(&p.tm_k, k, rows, kTile) ||
             !make_map_2d(&p.tm_v, v, rows, kTile) || !make_map_2d(&p.tm_y, y, rows, 32)) {
    return cudaErrorInvalidValue;
  }
  p.grid2d = s.grid() ? 1 : 0;
  p.gw = s.gw;
  p.gh = s.gh;
  p.tw = s.grid() ? s.tw : 1;
  p.th = s.th;
  p.bpr = s.grid() ? s.gw / s.tw : 1;
  if (!make_map_2d(&p.tm_ps, w + pl.off_ps, (uint64_t)s.heads() * pl.C * kD, 32)) return cudaErrorInvalidValue;
  if (pl.tc_mix && !make_map_2d(&p.tm_p, w + pl.off_ps, (uint64_t)s.heads() * pl.C, mix_kslots(pl.C), (uint64_t)kD * kD))
    return cudaErrorInvalidValue;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const int grid = s.heads() * pl.C < sms ? s.heads() * pl.C : sms;
  p.mix_t = mix_t_fits(pl, s.heads(), grid) && make_map_pairs(&p.tm_pp, w + pl.off_ps, s.heads(), pl.C) ? 1 : 0;
  p.mix_n = (pl.M + 15) / 16 * 16;
  p.zx = pl.tc_mix && pl.C > kD && 4 * s.heads() <= grid ? 1 : 0;
  p.mixing = mixing;
  p.ps = reinterpret_cast<__nv_bfloat16*>(w + pl.off_ps);
  p.pz = reinterpret_cast<float*>(w + pl.off_pz);
  p.smix = reinterpret_cast<uint8_t*>(w + pl.off_smix);
  p.zmix = reinterpret_cast<float*>(w + pl.off_zmix);
  p.den_out = den_out;
  p.ctr = reinterpret_cast<unsigned*>(w + kCounterOffset);
  p.status = &reinterpret_cast<WorkspaceHeader*>(w)->status;
  p.heads = s.heads();
  p.H = s.H;
  p.N = s.N;
  p.M = pl.M;
  p.C = pl.C;
  p.cpb = pl.cpb;
  p.TS = s.heads() * pl.C;
  p.tc_mix = pl.tc_mix ? 1 : 0;
  p.XS = pl.tc_mix ? s.heads() * kD : 0;
  p.eps = eps;
  p.normalise = s.normalise ? 1 : 0;
  p.strict = strict ? 1 : 0;
  p.mix_only = mix_only ? 1 : 0;
  p.wait_ns = g_wait_ns;
  cudaError_t e;
  if (p.M <= 16)
    e = launch_t<16>(p, grid, st);
  else if (p.M <= 32)
    e = launch_t<32>(p, grid, st);
  else
    e = launch_t<64>(p, grid, st);
  note_launch();
  return e;
}
}  // namespace

void tc_mhla_set_wait_limit(unsigned long long ns) { g_wait_ns = ns == 0 ? kWaitLimitNs : ns; }

cudaError_t tc_mhla_launch(const MhlaShape& s, const void* q, const void* k, const void* v,
                           const float* mixing, void* y, float* den_out, float eps, MixMode mode,
                           void* ws, cudaStream_t st) {
  (void)mode;
  return tc_mhla_run(s, q, k, v, mixing, y, den_out, eps, false, false, ws, st);
}

bool tc_mhla_prefix_supported(const MhlaShape& s, mhla_dtype dt) {
  MhlaShape f = s;
  f.gh = f.gw = f.th = f.tw = 0;
  return !s.grid() && tc_mhla_supported(f, dt, MIX_FULL);
}

cudaError_t tc_mhla_prefix_launch(const MhlaShape& s, const void* k, const void* v, const float* mixing, void* ws,
                                  cudaStream_t st) {
  // Q and Y are not touched in this mode: their tensor maps take K's and V's addresses
  return tc_mhla_run(s, k, k, v, mixing, const_cast<void*>(v), nullptr, 0.f, true, true, ws, st);
}

void tc_mhla_mixed_summaries(const MhlaShape& s, void* ws, const uint8_t** smix, const float** zmix) {
  const TcPlan pl = tc_plan(s);
  char* w = static_cast<char*>(ws);
  *smix = reinterpret_cast<const uint8_t*>(w + pl.off_smix);
  *zmix = reinterpret_cast<const float*>(w + pl.off_zmix);
}

}  // namespace mhla
