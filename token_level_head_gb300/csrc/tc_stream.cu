// bf16 MHLA forward on the sm_103a tensor cores as one ordered stream of work
// items (no grid-wide barrier).
//
// "MHLA: Restoring Expressivity of Linear Attention via Token-Level
// Multi-Head" §4.1 computes, per (batch, head) — a "head" below:
//   S_b = sum_{t in b} phi(K_t) V_t^T,  z_b = sum_{t in b} phi(K_t)       (local KV summaries)
//   S~_i = sum_b m_ib S_b,  z~_i = sum_b m_ib z_b                          (multi-head mixing)
//   Y_t = phi(Q_t) S~_i / (phi(Q_t) . z~_i + eps)                           (output)
// with phi = ELU + 1 and eps from "Linear Attention notes" §四/§五.
//
// Only the head's own summaries feed its output, so the work is cut into items
// with per-head dependencies instead of passes separated by grid barriers:
//   SUM(h, j)  chunk j (128 tokens) of head h: the partial P_hj = sum over the
//              chunk of phi(K_t) V_t^T (stored transposed, bf16) and its z
//              partial (fp32), both to the workspace (they stay in L2)
//   MIX(h, r)  rows [2 T r, 2 T r + 2 T) of S~_i^T for every query block i of
//              head h, from the C chunk partials, on the tensor cores (the
//              weight of partial j for query block i is m_{i, block(j)}); and
//              z~_i in fp32 for the query blocks [r M / I, (r + 1) M / I)
//   OUT(h, j)  Y of chunk j: phi(Q) S~_i on the tensor cores, the fp32
//              denominator beside it
// MIX(h, .) waits for every SUM(h, .), OUT(h, .) for every MIX(h, .), through
// two per-head counters in the workspace (fence and count / acquire).
//
// Order.  The items form one list of steps: step t holds SUM(t), then
// MIX(t - Dx), then OUT(t - Do) (each where the head exists).  CTA b takes list
// positions b, b + G, b + 2 G, ... and runs them in order, so every item
// depends only on items earlier in the list (no deadlock), and the lags Dx, Do
// (chosen on the host) put a head's MIX items and then its OUT items far
// enough behind its SUM items that the counters are normally complete by the
// time a CTA reaches them: HBM keeps streaming K, V of later heads and Q, Y of
// earlier ones, with no phase in which it idles.
//
// Roles of the 19 warps of a CTA (one CTA per SM, cooperative launch so that
// every CTA is resident while others wait on it):
//   warps 0-15  four worker warpgroups; warpgroup g carries the CTA's items
//               k = g, g + 4, ... through every step, one at a time:
//                 phi  thread r owns tile row r (TMEM lane r): SUM phi(K)
//                      in place in shared memory; OUT phi(Q) in fp32, the
//                      denominator phi(Q_r) . z~ + eps in a register, phi(Q)
//                      as bf16 into the group's TMEM A buffer; MIX the weight
//                      tile
//                 MMA  one thread, into the group's TMEM accumulator:
//                      SUM  D = [V^T ; 1] phi(K)  (M 128, N 64, K 128): rows
//                           0-63 the chunk's S^T, rows 64-127 its z
//                      MIX  D = P^T W^T per 128-entry tile (M 128, N = M
//                           rounded up to 16, K = C): lane x, column i = S~_i^T
//                           entry x
//                      OUT  D = phi(Q) S~  (M 128, N 64, K 64; A from TMEM)
//                 out  warp w reads TMEM lanes 32 w ..: partial rows, S~^T
//                      entries and Y = D / den go out with plain stores
//               so no hand-over between warps sits inside an item, and the
//               four groups overlap each other's steps
//   warp 16     producer (one thread): K and V tiles (SUM), the chunk-partial
//               box of a MIX item (one 4-D TMA, zero-filled past C), the Q
//               tile and then — once the head's MIX items are done — the
//               S~^T tile and z~ of an OUT item, into a ring of NS stages
//   warp 17     publisher (one thread): once a worker group reports an item's
//               stores issued, one fence for each batch of ready items, then
//               the per-head counts (no worker waits on a fence)
//   warp 18     z~ of the CTA's MIX items in fp32 from the z partials (it
//               waits only on the head's SUM counts, off the pipeline)
// All waits are bounded; on time-out the CTA raises the call's abort flag,
// winds down (in-flight copies and MMAs first) and latches the status word.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>

#include "common.cuh"
#include "internal.h"
#include "stream_sched.h"
#include "tc_common.cuh"

namespace mhla {
namespace {

using namespace tc;
using namespace sched;

constexpr int kThreads = 608;                // 19 warps
constexpr int kTile = 128;                   // tokens per chunk
constexpr int kD = 64;                       // head dimension
constexpr int kTileBytes = kTile * kD * 2;   // 16 KB bf16 tile
constexpr int kBox = 2 * kTileBytes;         // K + V, a MIX box, or Q + S~^T + z~
constexpr int kSTile = kD * kD * 2;          // S~^T tile: 8 KB
constexpr uint32_t kTmemCols = 512;          // per group: accumulator 64 columns at 64 g, OUT A 32 at 256 + 32 g
constexpr int kMaxStages = 8;
constexpr int kCachedItems = 256;            // list items of a CTA looked up once, at the start
constexpr int kLog = 32;                     // posted items remembered for the other roles
constexpr int kSmemLimit = 232448;           // opt-in shared memory per block
constexpr int kGroups = 4;                   // worker warpgroups (warps 0-15)
constexpr int kWarpProd = 16, kWarpPub = 17, kWarpZ = 18;
constexpr int kPub = 8;                      // items the epilogue may run ahead of the publisher
constexpr unsigned long long kDefaultWaitNs = 500000000ull;  // 0.5 s

// ------------------------------------------------------------------ layout
struct Small {
  uint64_t full[kMaxStages], empty[kMaxStages];
  uint64_t acc_full[kGroups];          // a group's MMAs have completed
  uint64_t pub[kPub], pub_free[kPub];  // workers -> publisher: an item's stores are issued
  uint64_t fin;
  uint32_t tbase;
  int abort;
  int last;
  int issued;     // items whose loads the producer has posted
  int zdone;      // posted items the z warp has gone through
  int half_open;  // an OUT item's Q load is posted, its arrival not yet
  uint32_t items[kCachedItems];  // this CTA's first list items, packed (kind 2 | head 22 | j 8 bits)
  uint32_t log[kLog];            // the item posted as the k-th ring use, at k % kLog
};

struct Params {
  CUtensorMap tm_q, tm_k, tm_v;  // [heads*N rows][64] bf16, box 64 x 128, 128-byte swizzle
  CUtensorMap tm_pb;             // the same memory as (c 64, j C, e 64, h heads), box 64 x cpad x 2T x 1
  const float* mixing;           // [H][M][M]
  __nv_bfloat16* y;              // [heads*N][64]
  __nv_bfloat16* ps;             // chunk partials S^T: [heads*C][64 e][64 c] bf16
  float* pz;                     // chunk partial z: [heads*C][64] fp32
  uint8_t* smix;                 // S~^T tiles: [heads*M] x 8 KB, K-major, 128-byte swizzle
  float* zmix;                   // z~: [heads*M][64] fp32
  float* den_out;                // [heads*N] or null
  unsigned* ctr;                 // [0] abort flag of the call, [1] CTAs finished
  unsigned* sum_done;            // [heads]: one count per SUM item
  unsigned* mix_done;            // [heads]: two counts per MIX item (S~^T rows, z~)
  unsigned* status;
  unsigned long long wait_ns;    // limit of every wait
  int heads, H, N, M, C, cpb, cpad, T, I, nmix;
  int E, Dx, Do;
  int NS, stage, off_w, off_ones, off_small;
  int normalise;                 // 0: Y is the numerator alone (den_out still the denominator)
  float eps;
};

// ------------------------------------------------------------------ waits
__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned ld_relaxed(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ int aborted(Small* sh) { return *reinterpret_cast<volatile int*>(&sh->abort); }
__device__ __forceinline__ void set_abort(Small* sh) { *reinterpret_cast<volatile int*>(&sh->abort) = 1; }

// mbarrier phase wait: a few polls, then suspended waits; false once the
// limit has passed (the CTA then aborts) or another role has aborted.
__device__ __noinline__ bool bwait_slow(uint64_t* bar, uint32_t parity, Small* sh, unsigned long long limit) {
  for (int i = 0; i < 16; ++i)
    if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait_ns(bar, parity, 128)) return true;
    if (aborted(sh)) return false;
    if (globaltimer_ns() - t0 > limit) break;
  }
  set_abort(sh);
  return false;
}
__device__ __forceinline__ bool bwait(uint64_t* bar, uint32_t parity, Small* sh, const Params& p) {
  return mbar_test(bar, parity) || bwait_slow(bar, parity, sh, p.wait_ns);
}

// Wait (acquire) for a per-head counter of another CTA; gives up after the
// limit, when this CTA aborts, or when another CTA has raised the abort flag.
__device__ __noinline__ bool gwait(const unsigned* c, unsigned target, Small* sh, const Params& p) {
  if (ld_acquire(c) >= target) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    __nanosleep(64);
    if (ld_relaxed(c) >= target) {
      (void)ld_acquire(c);  // polls without ordering, one acquire once the count is there
      return true;
    }
    if (aborted(sh) || ld_relaxed(p.ctr) != 0) break;
    if (globaltimer_ns() - t0 > p.wait_ns) break;
  }
  set_abort(sh);
  return false;
}

// Short wait (10 ms at most) used only while winding down after an abort.
__device__ __noinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait_ns(bar, parity, 1000))
    if (globaltimer_ns() - t0 > 10000000ull) return;
}

// ------------------------------------------------------------------ phi
// phi of two packed bf16 values (fp32 arithmetic), packed back to bf16.
__device__ __forceinline__ uint32_t phi2(uint32_t w) {
  return pack_bf16(phi_f(__uint_as_float(w << 16)), phi_f(__uint_as_float(w & 0xffff0000u)));
}

// 16 bf16 (8 packed words) to global memory in one 32-byte store.
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t* w) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]),
               "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

// Position in a ring of n slots: slot and phase parity of use number k,
// advanced one use at a time (no division in the loops).
struct Ring {
  int slot = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void next(int n) {
    if (++slot == n) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

__device__ __noinline__ Item item_lookup(const Sched& sc, int k) {
  return item_at(sc, (int)blockIdx.x + k * (int)gridDim.x);
}
__device__ __forceinline__ uint32_t pack_item(const Item& it) {
  return (uint32_t)it.kind << 30 | (uint32_t)it.h << 8 | (uint32_t)it.j;
}
__device__ __forceinline__ Item unpack_item(uint32_t v) {
  return {(int)(v >> 30), (int)((v >> 8) & 0x3FFFFFu), (int)(v & 0xFFu)};
}
// The item posted as this CTA's k-th ring use.
__device__ __forceinline__ Item posted_item(const Small* sh, int k) {
  return unpack_item(*reinterpret_cast<const volatile uint32_t*>(&sh->log[k % kLog]));
}
// This CTA's k-th list item: from the table built at the start, or looked up.
__device__ __forceinline__ Item my_item(const Small* sh, const Sched& sc, int k) {
  if (k < kCachedItems) return unpack_item(sh->items[k]);
  return item_lookup(sc, k);
}

// ------------------------------------------------------------------ producer
// The producer posts this CTA's items into the ring in list order.  An OUT
// item's Q tile is requested at once; its S~^T tile and z~ once the head's MIX
// items are counted.  A MIX item waits for its head's SUM counts.
__device__ void producer(const Params& p, const Sched& sc, uint8_t* sm, Small* sh, int nloc) {
  const uint64_t once = policy_evict_first();  // Q, K, V are read once
  volatile int* issued = &sh->issued;
  volatile int* zdone = &sh->zdone;
  Ring r;
  for (int k = 0; k < nloc; ++k, r.next(p.NS)) {
    const int s = r.slot;
    if (k >= p.NS && !bwait(&sh->empty[s], r.phase ^ 1u, sh, p)) return;
    // the z warp must have read the log entry this post reuses
    for (uint64_t t0 = globaltimer_ns(); k >= kLog && *zdone <= k - kLog;) {
      if (aborted(sh) || globaltimer_ns() - t0 > p.wait_ns) {
        set_abort(sh);
        return;
      }
      __nanosleep(128);
    }
    const Item it = my_item(sh, sc, k);
    sh->log[k % kLog] = pack_item(it);
    uint8_t* st = sm + s * p.stage;
    uint64_t* fb = &sh->full[s];
    const int row = it.h * p.N + it.j * kTile;
    if (it.kind == kSum) {
      mbar_arrive_expect_tx(fb, kBox);
      tma_load_2d_hint(st, &p.tm_k, 0, row, fb, once);
      tma_load_2d_hint(st + kTileBytes, &p.tm_v, 0, row, fb, once);
      *issued = k + 1;
    } else if (it.kind == kMix) {
      if (!gwait(p.sum_done + it.h, (unsigned)p.C, sh, p)) return;
      fence_proxy_async_global();  // the partials were written by other CTAs
      mbar_arrive_expect_tx(fb, (uint32_t)(p.T * 2 * p.cpad * 128));
      tma_load_4d(st, &p.tm_pb, 0, 0, it.j * 2 * p.T, it.h, fb);
      *issued = k + 1;
    } else {
      mbar_expect_tx(fb, kTileBytes);  // the Q tile, before the arrival below
      tma_load_2d_hint(st, &p.tm_q, 0, row, fb, once);
      sh->half_open = 1;
      *issued = k + 1;
      if (!gwait(p.mix_done + it.h, 2u * p.I, sh, p)) return;
      fence_proxy_async_global();  // S~ / z~ were written by other CTAs
      const size_t blk = (size_t)it.h * p.M + it.j / p.cpb;
      mbar_arrive_expect_tx(fb, kSTile + kD * 4);
      sh->half_open = 0;
      bulk_load_1d(st + kTileBytes, p.smix + blk * kSTile, kSTile, fb);
      bulk_load_1d(st + kTileBytes + kSTile, p.zmix + blk * kD, kD * 4, fb);
    }
  }
}

// ------------------------------------------------------------------ workers
// MIX weight tile of head h, the B operand of the MIX MMAs (K-major, nmix rows
// of 128 bytes, 128-byte swizzle): row i, column j = m[h][i][j / cpb] for
// i < M and j < C, zero elsewhere.  Thread t of a group writes pieces t, t + 128, ...
__device__ __forceinline__ void write_weights(const Params& p, int h, uint8_t* wt, int t) {
  const float* m = p.mixing + (size_t)(h % p.H) * p.M * p.M;
  for (int piece = t; piece < p.nmix * 8; piece += 128) {
    const int i = piece >> 3, c16 = piece & 7;
    float w[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int j = 8 * c16 + e;
      w[e] = (i < p.M && j < p.C) ? __ldg(m + i * p.M + j / p.cpb) : 0.f;
    }
    *reinterpret_cast<uint4*>(wt + i * 128 + ((c16 ^ (i & 7)) << 4)) =
        make_uint4(pack_bf16(w[0], w[1]), pack_bf16(w[2], w[3]), pack_bf16(w[4], w[5]), pack_bf16(w[6], w[7]));
  }
}

// MIX item of head h, tiles t < T, for the warp on lane quadrant qd: entry
// 32 qd + lane of tile t is S~^T[e][c], e = e0 + 2t + qd / 2, c = 32 (qd % 2) +
// lane, column i of the tile = query block i.  Neighbouring lanes pair up so
// that each stores two adjacent entries (4 bytes) of one tile.
__device__ __forceinline__ void mix_out(const Params& p, uint32_t ta, int h, int e0, int qd, int lane) {
  const int c = 32 * (qd & 1) + lane;
  const bool odd = lane & 1;
  uint8_t* base = p.smix + (size_t)h * p.M * kSTile;
  for (int t = 0; t < p.T; ++t) {
    const int e = e0 + 2 * t + (qd >> 1);
    for (int q = 0; q < p.nmix / 16; ++q) {
      float v[16];
      tmem_ld16(ta + (uint32_t)(t * p.nmix + 16 * q), v);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 16; i += 2) {
        // even lane: (c, c + 1) of block i; odd lane: (c - 1, c) of block i + 1
        const float other = __shfl_xor_sync(0xffffffffu, odd ? v[i] : v[i + 1], 1);
        const int blk = 16 * q + (odd ? i + 1 : i);
        if (blk < p.M) {
          const uint32_t pk = odd ? pack_bf16(other, v[i + 1]) : pack_bf16(v[i], other);
          *reinterpret_cast<uint32_t*>(base + (size_t)blk * kSTile + swz128(e, c & ~1)) = pk;
        }
      }
    }
  }
}

// One item's MMAs, issued by the group's leader into accumulator `acc`.
__device__ __forceinline__ void issue_mmas(const Params& p, const Item& it, uint32_t st, uint32_t ones, uint32_t acc,
                                           uint32_t abuf) {
  if (it.kind == kSum) {
    // A = V tile (MN-major) with the ones tile as M rows 64..127, B = phi(K) (MN-major)
    const uint32_t v0 = st + kTileBytes;
    const uint64_t da = smem_desc(v0, ones - v0, 1024), db = smem_desc(st, 8192, 1024);
    const uint32_t idesc = idesc_bf16_f32(128, 64, 1, 1);
#pragma unroll
    for (int kk = 0; kk < kTile / 16; ++kk) mma_bf16(acc, da + kk * (2048 >> 4), db + kk * (2048 >> 4), idesc, kk > 0);
  } else if (it.kind == kOut) {
    // A = phi(Q) in TMEM (K = 64: 32 columns, 8 a step), B = S~^T (K-major)
    const uint64_t db = smem_desc(st + kTileBytes, 16, 1024);
    const uint32_t idesc = idesc_bf16_f32(128, 64, 0, 0);
#pragma unroll
    for (int kk = 0; kk < kD / 16; ++kk) mma_bf16_ts(acc, abuf + 8 * kk, db + kk * (32 >> 4), idesc, kk > 0);
  } else {
    // per tile t: A = box rows e = 2t, 2t + 1 (MN-major, the two 64-entry M
    // groups ebytes apart), B = the weight tile (K-major), K = cpad
    const uint32_t ebytes = (uint32_t)p.cpad * 128;
    const uint64_t db = smem_desc(st + p.off_w, 16, 1024);
    const uint32_t idesc = idesc_bf16_f32(128, p.nmix, 1, 0);
    for (int t = 0; t < p.T; ++t) {
      const uint64_t da = smem_desc(st + 2 * t * ebytes, ebytes, 1024);
      for (int kk = 0; kk < p.cpad / 16; ++kk)
        mma_bf16(acc + t * p.nmix, da + kk * (2048 >> 4), db + kk * (32 >> 4), idesc, kk > 0);
    }
  }
}

// Worker warpgroup g (warps 4 g .. 4 g + 3): warp qd = warp % 4 owns TMEM lane
// quadrant qd, thread (qd, lane) tile row r = 32 qd + lane.  Items k = g,
// g + kGroups, ... of this CTA, each through phi, MMA and output before the
// next; the group's threads meet once an item (named barrier g + 1, which also
// makes an abort uniform).
__device__ void worker(const Params& p, const Sched& sc, uint8_t* sm, Small* sh, uint32_t tmem, int g, int qd,
                       int lane, int nloc) {
  const int r = 32 * qd + lane;
  const uint32_t lane_off = (uint32_t)(32 * qd) << 16;
  const uint32_t acc = tmem + (uint32_t)(64 * g);          // accumulator, 64 columns
  const uint32_t abuf = tmem + (uint32_t)(256 + 32 * g);   // OUT A operand, 32 columns
  const uint32_t ones = smem_u32(sm + p.off_ones);
  const int bar = 1 + g;
  int s = g % p.NS;  // ring slot and phase of item k
  uint32_t ph = (uint32_t)((g / p.NS) & 1), aph = 0;
  bool mma_pending = false;  // an issued MMA whose completion this group has not seen
  for (int k = g; k < nloc; k += kGroups) {
    uint8_t* st = sm + s * p.stage;
    float dn = 0.f;
    bool ok = bwait(&sh->full[s], ph, sh, p);
    const Item it = ok ? posted_item(sh, k) : Item{kSum, 0, 0};
    if (it.kind == kMix) {
      // the weight area is free: the producer posted this stage after its
      // previous item's MMAs completed
      if (ok) {
        write_weights(p, it.h, st + p.off_w, r);
        fence_proxy_async_smem();  // weight tile -> tensor core reads
      }
    } else {
      uint4* row = reinterpret_cast<uint4*>(st + r * 128);
      if (ok && it.kind == kSum) {
        // phi(K) in place (elementwise: the swizzled order does not matter)
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 x = row[c];
          row[c] = make_uint4(phi2(x.x), phi2(x.y), phi2(x.z), phi2(x.w));
        }
        fence_proxy_async_smem();  // phi tile -> tensor core reads
      } else if (ok) {
        // phi(Q) row r: logical piece c of the row sits at piece c ^ (r & 7)
        // (128-byte swizzle); fp32 phi for the denominator, bf16 to TMEM
        const float4* zt = reinterpret_cast<const float4*>(st + kTileBytes + kSTile);
        uint32_t pk[32];
        float d = 0.f;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 x = row[c ^ (r & 7)];
          const float4 za = zt[2 * c], zb = zt[2 * c + 1];
          const uint32_t w[4] = {x.x, x.y, x.z, x.w};
          const float zz[8] = {za.x, za.y, za.z, za.w, zb.x, zb.y, zb.z, zb.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float lo = phi_f(__uint_as_float(w[j] << 16));
            const float hi = phi_f(__uint_as_float(w[j] & 0xffff0000u));
            d = fmaf(lo, zz[2 * j], d);
            d = fmaf(hi, zz[2 * j + 1], d);
            pk[4 * c + j] = pack_bf16(lo, hi);
          }
        }
        dn = d + p.eps;
        tmem_st32(abuf + lane_off, pk);
        tmem_st_wait();
      }
    }
    tc_fence_before();
    if (!group_and(bar, 128, ok && !aborted(sh))) break;
    if (r == 0) {
      tc_fence_after();
      issue_mmas(p, it, smem_u32(st), ones, acc, abuf);
      mma_commit(&sh->empty[s]);        // the stage is free once these MMAs have read it
      mma_commit(&sh->acc_full[g]);     // and the accumulator is ready
    }
    mma_pending = true;
    ok = bwait(&sh->acc_full[g], aph, sh, p);
    if (ok) {
      mma_pending = false;
      aph ^= 1u;
      tc_fence_after();
      const uint32_t ta = acc + lane_off;
      if (it.kind == kMix) {
        mix_out(p, ta, it.h, it.j * 2 * p.T, qd, lane);
      } else if (it.kind == kOut || qd < 3) {
        // two halves of 32 columns: Y row r = D / den (bf16), or the chunk's
        // partial S^T row e = r (qd 0, 1; bf16), or its z (qd 2: TMEM rows
        // 64.. all hold it; lane 0 writes it, fp32)
        const float rd = it.kind == kOut && p.normalise ? 1.f / dn : 1.f;
        const size_t g_chunk = (size_t)it.h * p.C + it.j;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float v[32];
          tmem_ld16(ta + 32 * half, v);
          tmem_ld16(ta + 32 * half + 16, v + 16);
          tmem_ld_wait();
          if (it.kind == kSum && qd == 2) {
            if (lane == 0) {
              float4* zo = reinterpret_cast<float4*>(p.pz + g_chunk * kD + 32 * half);
#pragma unroll
              for (int c = 0; c < 8; ++c) zo[c] = make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
            }
          } else {
            __nv_bfloat16* dst = it.kind == kOut ? p.y + ((size_t)it.h * p.N + (size_t)it.j * kTile + r) * kD + 32 * half
                                                 : p.ps + (g_chunk * kD + r) * kD + 32 * half;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              uint32_t w[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) w[i] = pack_bf16(v[16 * c + 2 * i] * rd, v[16 * c + 2 * i + 1] * rd);
              st_global_v8(dst + 16 * c, w);
            }
          }
        }
        if (it.kind == kOut && p.den_out != nullptr) p.den_out[(size_t)it.h * p.N + (size_t)it.j * kTile + r] = dn;
      }
      // report the item's stores to the publisher (one arrival per warp)
      __syncwarp();
      if (lane == 0) {
        const int e = k % kPub;
        if (k < kPub || bwait(&sh->pub_free[e], ((k / kPub) - 1) & 1, sh, p)) mbar_arrive(&sh->pub[e]);
      }
    }
    s += kGroups;
    while (s >= p.NS) {
      s -= p.NS;
      ph ^= 1u;
    }
  }
  // after an abort: MMAs this group issued must finish before TMEM is freed
  if (mma_pending && r == 0) drain_wait(&sh->acc_full[g], aph);
}
// ------------------------------------------------------------------ publisher
// Warp 2, one thread: takes the epilogue's arrivals item by item and makes
// the stores behind them visible to the other CTAs — one fence for every
// batch of items that are ready together — then counts them: one per SUM
// item on the head's sum_done, one per MIX item on its mix_done.  It waits
// only for this CTA's epilogue, never for another CTA.
__device__ void publisher(const Params& p, const Sched& sc, Small* sh, int nloc) {
  int hs[kPub], ks[kPub];  // heads and kinds waiting for the fence
  int n = 0;
  for (int k = 0; k < nloc; ++k) {
    const int e = k % kPub;
    if (n > 0 && !mbar_test(&sh->pub[e], (k / kPub) & 1)) {
      __threadfence();
      for (int i = 0; i < n; ++i) atomicAdd((ks[i] == kSum ? p.sum_done : p.mix_done) + hs[i], 1u);
      n = 0;
    }
    if (!bwait(&sh->pub[e], (k / kPub) & 1, sh, p)) return;
    const Item it = posted_item(sh, k);
    mbar_arrive(&sh->pub_free[e]);
    if (it.kind != kOut) {
      hs[n] = it.h;
      ks[n] = it.kind;
      ++n;
    }
    if (n == kPub) {
      __threadfence();
      for (int i = 0; i < n; ++i) atomicAdd((ks[i] == kSum ? p.sum_done : p.mix_done) + hs[i], 1u);
      n = 0;
    }
  }
  if (n > 0) {
    __threadfence();
    for (int i = 0; i < n; ++i) atomicAdd((ks[i] == kSum ? p.sum_done : p.mix_done) + hs[i], 1u);
  }
}

// ------------------------------------------------------------------ z warp
// Warp 3: z~ of the MIX items of this CTA, fp32, straight from the z
// partials in L2: z~_i[c] = sum_j m_{i, j / cpb} z_j[c] for the item's query
// blocks [r M / I, (r + 1) M / I) (at most two: I >= M T / 32 >= M / 2).
// Lane l takes columns l and l + 32, reading each column once for both
// blocks, 32 partials in flight at a time.  The warps wait only for the head's SUM counts, never for this CTA's
// pipeline.
__device__ void z_role(const Params& p, Small* sh, int lane, int nloc) {
  volatile int* zdone = &sh->zdone;
  for (int k = 0; k < nloc; ++k) {
    for (uint64_t t0 = globaltimer_ns(); *reinterpret_cast<volatile int*>(&sh->issued) <= k;) {
      if (aborted(sh)) return;
      if (globaltimer_ns() - t0 > p.wait_ns) {
        set_abort(sh);
        return;
      }
      __nanosleep(256);
    }
    const Item it = posted_item(sh, k);
    __syncwarp();
    if (lane == 0) *zdone = k + 1;
    if (it.kind != kMix) continue;
    const int i0 = it.j * p.M / p.I, i1 = (it.j + 1) * p.M / p.I;
    if (i1 > i0) {
      if (!gwait(p.sum_done + it.h, (unsigned)p.C, sh, p)) return;
      const float* m0 = p.mixing + ((size_t)(it.h % p.H) * p.M + i0) * p.M;
      const float* m1 = i1 - i0 > 1 ? m0 + p.M : m0;
      for (int c = lane; c < kD; c += 32) {
        const float* zc = p.pz + (size_t)it.h * p.C * kD + c;
        float acc0 = 0.f, acc1 = 0.f;
        for (int j0 = 0; j0 < p.C; j0 += 32) {
          float zv[32];
#pragma unroll
          for (int u = 0; u < 32; ++u) zv[u] = j0 + u < p.C ? __ldcg(zc + (size_t)(j0 + u) * kD) : 0.f;
#pragma unroll
          for (int u = 0; u < 32; ++u) {
            const int b = (j0 + u) / p.cpb;
            if (j0 + u < p.C) {
              acc0 = fmaf(__ldg(m0 + b), zv[u], acc0);
              acc1 = fmaf(__ldg(m1 + b), zv[u], acc1);
            }
          }
        }
        float* zo = p.zmix + ((size_t)it.h * p.M + i0) * kD + c;
        zo[0] = acc0;
        if (i1 - i0 > 1) zo[kD] = acc1;
      }
      __threadfence();  // this thread's z~ stores before the count
    }
    __syncwarp();
    if (lane == 0) atomicAdd(p.mix_done + it.h, 1u);
  }
}

// ------------------------------------------------------------------ kernel
__global__ void __launch_bounds__(kThreads, 1) mhla_stream_kernel(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Small* sh = reinterpret_cast<Small*>(sm + p.off_small);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const Sched sc{p.heads, p.C, p.I, p.Dx, p.Do};
  const int nloc = (int)blockIdx.x < p.E ? (p.E - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;

  if (tid == 0) {
    for (int s = 0; s < p.NS; ++s) {
      mbar_init(&sh->full[s], 1);
      mbar_init(&sh->empty[s], 1);
    }
    for (int g = 0; g < kGroups; ++g) mbar_init(&sh->acc_full[g], 1);
    for (int e = 0; e < kPub; ++e) {
      mbar_init(&sh->pub[e], 4);
      mbar_init(&sh->pub_free[e], 1);
    }
    sh->abort = 0;
    sh->issued = 0;
    sh->zdone = 0;
    sh->half_open = 0;
    fence_mbar_init();
  }
  if (warp == kWarpProd) {
    tmem_alloc(&sh->tbase, kTmemCols);
    tmem_relinquish();
    if (lane == 0) {
      prefetch_tmap(&p.tm_q);
      prefetch_tmap(&p.tm_k);
      prefetch_tmap(&p.tm_v);
      prefetch_tmap(&p.tm_pb);
    }
  }
  for (int i = tid; i < kTileBytes / 16; i += kThreads)
    reinterpret_cast<uint4*>(sm + p.off_ones)[i] = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
  for (int k = tid; k < nloc && k < kCachedItems; k += kThreads) sh->items[k] = pack_item(item_lookup(sc, k));
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh->tbase;

  if (warp < 4 * kGroups) {
    worker(p, sc, sm, sh, tmem, warp >> 2, warp & 3, lane, nloc);
  } else if (warp == kWarpProd) {
    if (lane == 0) producer(p, sc, sm, sh, nloc);
    __syncwarp();
  } else if (warp == kWarpPub) {
    if (lane == 0) publisher(p, sc, sh, nloc);
    __syncwarp();
  } else if (warp == kWarpZ) {
    z_role(p, sh, lane, nloc);
  }
  tc_fence_before();
  __syncthreads();

  // Wind down.  On the normal path every wait below is already satisfied;
  // after an abort they let the TMA loads and MMAs still in flight finish.
  if (tid == 0) {
    if (aborted(sh)) {
      atomicExch(p.ctr, 1u);  // the other CTAs stop waiting for this one
      const int n = sh->issued;
      if (sh->half_open) mbar_arrive(&sh->full[(n - 1) % p.NS]);  // its Q tile is all that is in flight
      for (int k = n > p.NS ? n - p.NS : 0; k < n; ++k) drain_wait(&sh->full[k % p.NS], (k / p.NS) & 1);
      atomicOr(p.status, 1u);
    }
  }
  tc_fence_after();
  if (warp == kWarpProd) tmem_dealloc(tmem, kTmemCols);

  // The last CTA out leaves the counters at zero for the next call.
  if (tid == 0) {
    __threadfence();
    sh->last = atomicAdd(&p.ctr[1], 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (sh->last) {
    __threadfence();
    for (int h = tid; h < p.heads; h += kThreads) {
      p.sum_done[h] = 0;
      p.mix_done[h] = 0;
    }
    if (tid == 0) {
      p.ctr[0] = 0;
      p.ctr[1] = 0;
    }
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

// [rows][64] bf16, box 64 x box_rows, 128-byte swizzle.
bool map_rows(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows) {
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

// The chunk partials [heads][C][64 e][64 c] bf16 as the 4-D tensor (c, j, e, h):
// a box (64, cpad, 2T, 1) lands as 2T rows e of cpad x 128 bytes (rows j past
// C read as zero), the MN-major layout of the MIX MMAs' A operand.
bool map_partial_boxes(CUtensorMap* m, const void* base, int heads, int C, int cpad, int T) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)C, (cuuint64_t)kD, (cuuint64_t)heads};
  cuuint64_t strides[3] = {(cuuint64_t)kD * kD * 2, (cuuint64_t)kD * 2, (cuuint64_t)C * kD * kD * 2};
  cuuint32_t box[4] = {(cuuint32_t)kD, (cuuint32_t)cpad, (cuuint32_t)(2 * T), 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline size_t a256(size_t x) { return (x + 255) & ~size_t(255); }

struct Plan {
  int C, M, cpb, cpad, nmix, T, I;
  size_t off_ps, off_pz, off_smix, off_zmix, total;
};

Plan make_plan(const MhlaShape& s) {
  Plan p;
  p.C = s.N / kTile;
  p.M = s.M();
  p.cpb = s.block / kTile;
  p.cpad = (p.C + 15) / 16 * 16;
  p.nmix = (p.M + 15) / 16 * 16;
  p.T = std::min(64 / p.nmix, 128 / p.cpad);  // tiles per MIX item: TMEM columns, box bytes
  p.I = kD / (2 * p.T);
  const size_t heads = (size_t)s.heads();
  size_t off = kWorkspacePrefix;
  p.off_ps = off;   off = a256(off + heads * p.C * (size_t)kD * kD * 2);
  p.off_pz = off;   off = a256(off + heads * p.C * (size_t)kD * sizeof(float));
  p.off_smix = off; off = a256(off + heads * p.M * (size_t)kSTile);
  p.off_zmix = off; off = a256(off + heads * p.M * (size_t)kD * sizeof(float));
  p.total = off;
  return p;
}

// choose_lags, once per (heads, C, I, grid)
std::pair<int, int> cached_lags(int heads, int C, int I, int grid) {
  static std::mutex mu;
  static std::map<std::tuple<int, int, int, int>, std::pair<int, int>> cache;
  const auto key = std::make_tuple(heads, C, I, grid);
  std::lock_guard<std::mutex> lk(mu);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  const auto r = choose_lags(heads, C, I, 6 * grid);
  if (cache.size() < 4096) cache[key] = r;
  return r;
}

unsigned long long g_wait_ns = kDefaultWaitNs;

}  // namespace

void tc_stream_set_wait_limit(unsigned long long ns) { g_wait_ns = ns == 0 ? kDefaultWaitNs : ns; }

// Taken where the three-pass kernel (tc_mhla.cu) has no tensor-core MIX: C =
// N / 128 chunk partials not a multiple of 16 (at most 64).  Measured on the
// B x H x 1024-token shapes: 16-17 us against 24-26 us; for C a multiple of 16
// the three-pass kernel is faster (DiT-like B8 H6 N4096: 32 us against 57 us,
// L2-warm) and keeps those shapes.
bool tc_stream_supported(const MhlaShape& s, mhla_dtype dt, MixMode mode) {
  if (!s.plain_phi()) return false;  // ELU + 1 without decay only
  if (s.grid()) return false;  // contiguous blocks only
  if (dt != MHLA_BF16 || s.d != kD || mode != MIX_FULL) return false;
  if (s.block % kTile != 0 || s.N % kTile != 0 || s.N / kTile > 64 || (s.N / kTile) % 16 == 0) return false;
  if (s.heads() > kMaxCounterHeads || (long long)s.heads() * s.N >= (1ll << 31)) return false;
  const Plan pl = make_plan(s);
  return (long long)s.heads() * (2 * pl.C + pl.I) < (1ll << 30);
}

size_t tc_stream_workspace(const MhlaShape& s) { return make_plan(s).total; }

cudaError_t tc_stream_launch(const MhlaShape& s, const void* q, const void* k, const void* v, const float* mixing,
                             void* y, float* den_out, float eps, void* ws, cudaStream_t st) {
  const Plan pl = make_plan(s);
  char* w = static_cast<char*>(ws);
  Params p;
  const uint64_t rows = (uint64_t)s.heads() * s.N;
  if (!map_rows(&p.tm_q, q, rows, kTile) || !map_rows(&p.tm_k, k, rows, kTile) || !map_rows(&p.tm_v, v, rows, kTile) ||
      !map_partial_boxes(&p.tm_pb, w + pl.off_ps, s.heads(), pl.C, pl.cpad, pl.T))
    return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  p.heads = s.heads();
  p.H = s.H;
  p.N = s.N;
  p.M = pl.M;
  p.C = pl.C;
  p.cpb = pl.cpb;
  p.cpad = pl.cpad;
  p.T = pl.T;
  p.I = pl.I;
  p.nmix = pl.nmix;
  const int grid_max = sms;
  const int e_all = n_items(Sched{p.heads, p.C, p.I, 0, p.heads});
  const int grid = std::max(1, std::min(grid_max, e_all));
  const auto lags = cached_lags(p.heads, p.C, p.I, grid);
  p.Dx = lags.first;
  p.Do = lags.second;
  p.E = n_items(Sched{p.heads, p.C, p.I, p.Dx, p.Do});
  // shared memory: ring stages (32 KB box + the MIX weight tile), ones tile, barriers
  p.stage = kBox + (pl.nmix * 128 + 1023) / 1024 * 1024;
  p.off_w = kBox;
  const int fixed = 1024 + kTileBytes + (int)sizeof(Small);
  p.NS = std::min(kMaxStages, (kSmemLimit - fixed) / p.stage);
  if (p.NS < 2) return cudaErrorInvalidValue;
  p.off_ones = p.NS * p.stage;
  p.off_small = p.off_ones + kTileBytes;
  const int smem = 1024 + p.off_small + (int)sizeof(Small);
  p.mixing = mixing;
  p.y = static_cast<__nv_bfloat16*>(y);
  p.ps = reinterpret_cast<__nv_bfloat16*>(w + pl.off_ps);
  p.pz = reinterpret_cast<float*>(w + pl.off_pz);
  p.smix = reinterpret_cast<uint8_t*>(w + pl.off_smix);
  p.zmix = reinterpret_cast<float*>(w + pl.off_zmix);
  p.den_out = den_out;
  unsigned* ctr = reinterpret_cast<unsigned*>(w + kCounterOffset);
  p.ctr = ctr;
  p.sum_done = ctr + 2;
  p.mix_done = ctr + 2 + kMaxCounterHeads;
  p.status = &reinterpret_cast<WorkspaceHeader*>(w)->status;
  p.wait_ns = g_wait_ns;
  p.eps = eps;
  p.normalise = s.normalise ? 1 : 0;

  static SmemOptIn opt_in;
  if ((e = opt_in.ensure((const void*)mhla_stream_kernel, kSmemLimit)) != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, mhla_stream_kernel, p);
  note_launch();
  return e;
}

}  // namespace mhla
