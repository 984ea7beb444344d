// Backward of the non-causal MHLA block form: dQ, dK, dV and dM from dY.
//
// "MHLA: Restoring Expressivity of Linear Attention via Token-Level Multi-Head"
// §4.2 learns the mixing coefficients end to end; §4.1 defines the forward
//   S_b = sum_{j in b} phi(k_j) v_j^T,  z_b = sum_{j in b} phi(k_j),
//   S~_i = sum_b m_ib S_b,  z~_i = sum_b m_ib z_b,
//   Y_t = phi(q_t)^T S~_i / (phi(q_t) . z~_i + eps)        (t in block i),
// and the chain rule through those steps in reverse gives
//   dnum_t = dY_t / den_t,  dden_t = -(dY_t . Y_t) / den_t,
//   dS~_i = sum_{t in i} phi(q_t) dnum_t^T,  dz~_i = sum_{t in i} phi(q_t) dden_t,
//   dphi(q_t) = S~_i dnum_t + dden_t z~_i,
//   dS_b = sum_i m_ib dS~_i,  dz_b = sum_i m_ib dz~_i,
//   dm_ib = sum over the samples of <dS~_i, S_b> + dz~_i . z_b,
//   dphi(k_j) = dS_b v_j + dz_b,  dv_j = dS_b^T phi(k_j),
//   dq = phi'(q) dphi(q),  dk = phi'(k) dphi(k),  phi'(x) = min(1, phi(x)).
//
// SIMT path, seven launches, everything in fp32 (bf16 inputs and gradients are
// converted at the loads and stores):
//   bwd_summary  (unit, block)   S_b, z_b                      from K, V
//   bwd_mix      (unit, columns) S~, z~  = M  applied to the slots
//   bwd_query    (unit, block)   dQ, dS~_i, dz~_i              from Q, dY, S~_i, z~_i
//   bwd_mix      (unit, columns) dS, dz  = M^T applied to the dS~ slots
//   bwd_dm       (head, range)   partial sums of dM over a range of the head's slot entries
//   bwd_dm_sum   (head)          dM = the partials summed in a fixed order (deterministic)
//   bwd_key      (unit, block)   dK, dV                        from K, V, dS_b, dz_b
// bf16 with d = 64 and blocks of whole 128-token chunks: the summary, query and
// key passes run on the tensor cores (tc_backward.cu), fed by bwd_tiles (the
// bf16 operand tiles of S~ - z~ mu^T and of dS); mixing and dM stay here.
// A slot is the d^2 + d floats (S then z) of one (unit, block).  The token
// passes walk a block in chunks of TC tokens staged in shared memory, both
// token-major ([t][c]) and feature-major ([c][t]), so that every product
// reads float4 / float2 vectors: a chunk product out[t][n] = sum_k X[k][t] W[k][n]
// gives a thread TT tokens x 4 columns, a d x d reduction sum_t A[t][c] B[t][e]
// gives it an R x R tile (R = d / 16).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace mhla {
namespace {

constexpr int kBT = 256;     // threads of every backward kernel
constexpr int kMaxMixM = 64; // blocks per sequence the mixing kernels stage
constexpr int kDmK = 64;     // slot entries per stage of the dM kernel
constexpr int kDmRange = 128; // slot entries of one sample per dM CTA (many short CTAs hide the load latency)

template <int D>
struct BwdGeom {
  static constexpr int TC = D == 128 ? 32 : 64;  // tokens per chunk
  static constexpr int NQ = D / 4;               // column quads of a chunk product
  static constexpr int TT = TC * D / 4 / kBT;    // tokens per thread in a chunk product
  static constexpr int TG = TC / TT;             // token groups
  static constexpr int R = D / 16;               // d x d reductions: R x R per thread
  static constexpr int LD = D + 4;               // row of a token-major tile / a d x d tile (floats)
  static constexpr int LT = TC + 4;              // row of a feature-major tile
  static constexpr int TPT = kBT / TC;           // threads per token in the denominator sums
  static constexpr int X = D * D + D;            // floats of a slot
  static constexpr int NL = TC * D / 4 / kBT;    // quads of a chunk staged per thread
  static_assert(TG * NQ == kBT && TT >= 1 && (TT & (TT - 1)) == 0, "chunk product layout");
  static_assert(16 * R == D, "reduction layout");
  static_assert(NL >= 1 && TC % 16 == 0, "chunk staging layout");
};

// CTAs per SM each token pass is compiled for (its register budget): d = 128 tiles and fp32
// prefetch registers need more per thread; the query pass's 105 KB tiles allow two CTAs anyway.
template <typename T, int D>
struct BwdOcc {
  static constexpr int SUMMARY = D == 128 ? 1 : 3;
  static constexpr int QUERY = D == 128 ? 1 : 2;
  static constexpr int KEY = D == 128 ? 1 : (sizeof(T) == 4 ? 2 : 3);
};

// Four consecutive elements as stored (8 bytes of bf16, 16 bytes of fp32), and their fp32 values.
template <typename T> struct Quad;
template <> struct Quad<float> { float4 v; };
template <> struct Quad<__nv_bfloat16> { uint2 v; };

__device__ __forceinline__ Quad<float> ldq(const float* p) { return {*reinterpret_cast<const float4*>(p)}; }
__device__ __forceinline__ Quad<__nv_bfloat16> ldq(const __nv_bfloat16* p) {
  return {*reinterpret_cast<const uint2*>(p)};
}
__device__ __forceinline__ float4 to_f4(const Quad<float>& q) { return q.v; }
__device__ __forceinline__ float4 to_f4(const Quad<__nv_bfloat16>& q) {
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&q.v.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&q.v.y));
  return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ void stq(float* p, float4 x) { *reinterpret_cast<float4*>(p) = x; }
__device__ __forceinline__ void stq(__nv_bfloat16* p, float4 x) {
  __nv_bfloat162 a = __floats2bfloat162_rn(x.x, x.y), b = __floats2bfloat162_rn(x.z, x.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = u;
}

// n consecutive floats of shared memory (n = 1, 2, 4 or 8; 8 as two float4)
template <int N>
__device__ __forceinline__ void lds(float (&r)[N], const float* p) {
  if constexpr (N == 1) {
    r[0] = p[0];
  } else if constexpr (N == 2) {
    const float2 a = *reinterpret_cast<const float2*>(p);
    r[0] = a.x; r[1] = a.y;
  } else {
#pragma unroll
    for (int i = 0; i < N; i += 4) {
      const float4 a = *reinterpret_cast<const float4*>(p + i);
      r[i] = a.x; r[i + 1] = a.y; r[i + 2] = a.z; r[i + 3] = a.w;
    }
  }
}

struct PhiOp { __device__ float operator()(float x) const { return phi(x); } };
struct IdOp { __device__ float operator()(float x) const { return x; } };

// A chunk of TC tokens of a [L][D] block held in registers between its global loads and its
// shared-memory stores, so that the next chunk's loads are in flight while this one is computed.
// Quad j of a thread: a warp covers 8 tokens x 4 column quads (full 32-byte sectors per token of
// bf16, two-way bank conflicts at most in the feature-major stores).
template <typename T, int D>
struct ChunkRegs {
  using G = BwdGeom<D>;
  Quad<T> q[G::NL];

  __device__ __forceinline__ static void where(int j, int& t, int& c) {
    const int qi = threadIdx.x + kBT * j, lane = qi % 32, w = qi / 32;
    constexpr int TB = G::TC / 8;
    t = (w % TB) * 8 + lane % 8;
    c = ((w / TB) * 4 + lane / 8) * 4;
  }
  // rows at and past `valid` are not read (their addresses are clamped to the last real row)
  __device__ __forceinline__ void load(const T* __restrict__ src, int valid) {
#pragma unroll
    for (int j = 0; j < G::NL; ++j) {
      int t, c;
      where(j, t, c);
      q[j] = ldq(src + (size_t)min(t, valid - 1) * D + c);
    }
  }
  // token-major tok[t][c] and / or feature-major fea[c][t], through f; rows past `valid` are zero
  template <typename F>
  __device__ __forceinline__ void store(int valid, float* tok, float* fea, F f) const {
#pragma unroll
    for (int j = 0; j < G::NL; ++j) {
      int t, c;
      where(j, t, c);
      float4 x = to_f4(q[j]);
      if (t < valid) {
        x = make_float4(f(x.x), f(x.y), f(x.z), f(x.w));
      } else {
        x = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      if (tok) *reinterpret_cast<float4*>(tok + t * G::LD + c) = x;
      if (fea) {
        fea[(c + 0) * G::LT + t] = x.x;
        fea[(c + 1) * G::LT + t] = x.y;
        fea[(c + 2) * G::LT + t] = x.z;
        fea[(c + 3) * G::LT + t] = x.w;
      }
    }
  }
};

// out[t][n] (+)= sum_{k < D} X[k][t] W[k][n]: this thread's TT tokens x 4 columns.  The next k's
// operands are loaded before this k's FMAs; with two or more tokens the FMAs are packed fp32x2
// (two tokens against one column value).
template <int D>
__device__ __forceinline__ void chunk_product(float (&acc)[BwdGeom<D>::TT][4], const float* Xf, const float* W,
                                              int t0, int n0) {
  using G = BwdGeom<D>;
  float xn[G::TT];
  lds<G::TT>(xn, Xf + t0);
  float4 wn = *reinterpret_cast<const float4*>(W + n0);
#pragma unroll 4
  for (int k = 0; k < D; ++k) {
    float x[G::TT];
#pragma unroll
    for (int i = 0; i < G::TT; ++i) x[i] = xn[i];
    const float4 w = wn;
    if (k + 1 < D) {
      lds<G::TT>(xn, Xf + (k + 1) * G::LT + t0);
      wn = *reinterpret_cast<const float4*>(W + (k + 1) * G::LD + n0);
    }
    if constexpr (G::TT >= 2) {
#pragma unroll
      for (int i = 0; i < G::TT; i += 2) {
        const float2 xx = make_float2(x[i], x[i + 1]);
        float2 a0 = make_float2(acc[i][0], acc[i + 1][0]), a1 = make_float2(acc[i][1], acc[i + 1][1]);
        float2 a2 = make_float2(acc[i][2], acc[i + 1][2]), a3 = make_float2(acc[i][3], acc[i + 1][3]);
        a0 = __ffma2_rn(xx, make_float2(w.x, w.x), a0);
        a1 = __ffma2_rn(xx, make_float2(w.y, w.y), a1);
        a2 = __ffma2_rn(xx, make_float2(w.z, w.z), a2);
        a3 = __ffma2_rn(xx, make_float2(w.w, w.w), a3);
        acc[i][0] = a0.x; acc[i + 1][0] = a0.y; acc[i][1] = a1.x; acc[i + 1][1] = a1.y;
        acc[i][2] = a2.x; acc[i + 1][2] = a2.y; acc[i][3] = a3.x; acc[i + 1][3] = a3.y;
      }
    } else {
      acc[0][0] = fmaf(x[0], w.x, acc[0][0]);
      acc[0][1] = fmaf(x[0], w.y, acc[0][1]);
      acc[0][2] = fmaf(x[0], w.z, acc[0][2]);
      acc[0][3] = fmaf(x[0], w.w, acc[0][3]);
    }
  }
}

// acc[c][e] += sum_{t < TC} A[t][c0 + c] B[t][e0 + e]  (token-major tiles); the next token's
// operands are loaded before this token's FMAs, packed fp32x2 over pairs of e when R >= 2
template <int D>
__device__ __forceinline__ void reduce_tokens(float (&acc)[BwdGeom<D>::R][BwdGeom<D>::R], const float* A,
                                              const float* B, int c0, int e0) {
  using G = BwdGeom<D>;
  float an[G::R], bn[G::R];
  lds<G::R>(an, A + c0);
  lds<G::R>(bn, B + e0);
#pragma unroll 4
  for (int t = 0; t < G::TC; ++t) {
    float a[G::R], b[G::R];
#pragma unroll
    for (int i = 0; i < G::R; ++i) { a[i] = an[i]; b[i] = bn[i]; }
    if (t + 1 < G::TC) {
      lds<G::R>(an, A + (t + 1) * G::LD + c0);
      lds<G::R>(bn, B + (t + 1) * G::LD + e0);
    }
    if constexpr (G::R >= 2) {
#pragma unroll
      for (int i = 0; i < G::R; ++i)
#pragma unroll
        for (int j = 0; j < G::R; j += 2) {
          float2 c = make_float2(acc[i][j], acc[i][j + 1]);
          c = __ffma2_rn(make_float2(a[i], a[i]), make_float2(b[j], b[j + 1]), c);
          acc[i][j] = c.x;
          acc[i][j + 1] = c.y;
        }
    } else {
      acc[0][0] = fmaf(a[0], b[0], acc[0][0]);
    }
  }
}

// acc[c] += sum over this thread's tokens t = re, re + 16, ... of A[t][c0 + c] w(t); the sixteen
// threads sharing c0 (lanes 16 r .. 16 r + 15 of a warp) together cover the chunk
template <int D, typename W>
__device__ __forceinline__ void reduce_rows(float (&acc)[BwdGeom<D>::R], const float* A, int c0, int re, W w) {
  using G = BwdGeom<D>;
#pragma unroll
  for (int t = re; t < G::TC; t += 16) {
    float a[G::R];
    lds<G::R>(a, A + t * G::LD + c0);
    const float wt = w(t);
#pragma unroll
    for (int i = 0; i < G::R; ++i) acc[i] = fmaf(a[i], wt, acc[i]);
  }
}
template <int R>
__device__ __forceinline__ void sum16(float (&acc)[R]) {
#pragma unroll
  for (int i = 0; i < R; ++i)
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], o);
}

// ------------------------------------------------------------------ S_b, z_b
template <typename T, int D>
__global__ void __launch_bounds__(kBT, BwdOcc<T, D>::SUMMARY) bwd_summary_kernel(const T* __restrict__ k, const T* __restrict__ v,
                                                             float* __restrict__ slots, int N, int L, int M) {
  using G = BwdGeom<D>;
  extern __shared__ __align__(16) float sm[];
  float* Kt = sm;                 // [TC][LD] phi(K)
  float* Vt = Kt + G::TC * G::LD; // [TC][LD] V
  const int u = blockIdx.x / M, b = blockIdx.x % M;
  const size_t base = ((size_t)u * N + (size_t)b * L) * D;
  const int rc = threadIdx.x / 16, re = threadIdx.x % 16, c0 = rc * G::R, e0 = re * G::R;
  float acc[G::R][G::R] = {};
  float zacc[G::R] = {};
  ChunkRegs<T, D> rk, rv;
  rk.load(k + base, min(G::TC, L));
  rv.load(v + base, min(G::TC, L));
  for (int t0 = 0; t0 < L; t0 += G::TC) {
    const int valid = min(G::TC, L - t0);
    __syncthreads();  // the previous chunk is no longer read
    rk.store(valid, Kt, nullptr, PhiOp{});
    rv.store(valid, Vt, nullptr, IdOp{});
    __syncthreads();
    if (t0 + G::TC < L) {  // the next chunk's loads fly while this one is summed
      const int nv = min(G::TC, L - t0 - G::TC);
      rk.load(k + base + (size_t)(t0 + G::TC) * D, nv);
      rv.load(v + base + (size_t)(t0 + G::TC) * D, nv);
    }
    reduce_tokens<D>(acc, Kt, Vt, c0, e0);
    reduce_rows<D>(zacc, Kt, c0, re, [](int) { return 1.f; });
  }
  sum16<G::R>(zacc);
  float* slot = slots + ((size_t)u * M + b) * G::X;
#pragma unroll
  for (int i = 0; i < G::R; ++i)
#pragma unroll
    for (int j = 0; j < G::R; ++j) slot[(c0 + i) * D + e0 + j] = acc[i][j];
  if (re == 0)
#pragma unroll
    for (int i = 0; i < G::R; ++i) slot[D * D + c0 + i] = zacc[i];
}

// ------------------------------------------------- out_i = sum_b w_ib in_b over the slots
// w_ib = m[h][i][b] (transpose = 0) or m[h][b][i] (transpose = 1); a thread takes one entry x of
// every slot of one unit (a CTA kBT consecutive entries) and all M outputs, 16 at a time.
__device__ __forceinline__ size_t swz64(int row, int col) {  // byte of (row, col) in a [64][64] bf16 tile
  return (size_t)row * 128 + ((((col >> 3) ^ (row & 7)) << 4) | ((col & 7) << 1));
}
__global__ void __launch_bounds__(kBT) bwd_mix_kernel(const float* __restrict__ in, const float* __restrict__ mixing,
                                                      float* __restrict__ out, int H, int M, int X, int transpose) {
  __shared__ float sw[kMaxMixM * kMaxMixM];
  const int cols = (X + kBT - 1) / kBT;
  const int u = blockIdx.x / cols, x = (blockIdx.x % cols) * kBT + threadIdx.x;
  const float* mh = mixing + (size_t)(u % H) * M * M;
  const int xc = min(x, X - 1);  // threads past the slot load a valid entry and store nothing
  const float* ib = in + (size_t)u * M * X + xc;
  float* ob = out + (size_t)u * M * X + x;
  float pre[16];  // the first 16 inputs, in flight while the weights are staged
#pragma unroll
  for (int j = 0; j < 16; ++j) pre[j] = ib[(size_t)min(j, M - 1) * X];
  for (int e = threadIdx.x; e < M * M; e += kBT) {
    const int i = e / M, b = e % M;
    sw[i * M + b] = transpose ? mh[(size_t)b * M + i] : mh[(size_t)i * M + b];
  }
  __syncthreads();
  if (x >= X) return;
  for (int i0 = 0; i0 < M; i0 += 16) {
    float acc[16];
#pragma unroll
    for (int ii = 0; ii < 16; ++ii) acc[ii] = 0.f;
    for (int b0 = 0; b0 < M; b0 += 16) {  // sixteen independent loads in flight, then their FMAs
      float val[16];
#pragma unroll
      for (int j = 0; j < 16; ++j)
        val[j] = b0 + j < M ? (b0 == 0 ? pre[j] : ib[(size_t)min(b0 + j, M - 1) * X]) : 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j)
#pragma unroll
        for (int ii = 0; ii < 16; ++ii) {
          const float w = (i0 + ii < M && b0 + j < M) ? sw[(i0 + ii) * M + b0 + j] : 0.f;
          acc[ii] = fmaf(w, val[j], acc[ii]);
        }
    }
#pragma unroll
    for (int ii = 0; ii < 16; ++ii)
      if (i0 + ii < M) ob[(size_t)(i0 + ii) * X] = acc[ii];
  }
}

// ------------------------------------------------- bf16 tiles of the slots (d = 64)
// The two 8 KB 128-byte-swizzled bf16 tiles of each slot's d x d matrix A (rows e / columns c and
// rows c / columns e), the tensor-core passes' B operands, built in shared memory and written
// with 16-byte stores.  With mu: A = S~_i - z~_i mu_i^T, mu_i = S~_i^T z~_i / |z~_i|^2 (the
// least-squares rank-one part, zero when z~_i = 0; written in fp32): phi is near 1, so S~'s rows
// are near multiples of one vector; the remainder is small and its bf16 rounding costs little,
// while the rank-one part stays in fp32.  A CTA per slot.
__global__ void __launch_bounds__(kBT) bwd_tiles_kernel(const float* __restrict__ slots, float* __restrict__ mu,
                                                        uint8_t* __restrict__ tiles_t, uint8_t* __restrict__ tiles_n) {
  constexpr int D = 64, X = D * D + D;
  __shared__ __align__(16) uint8_t st[8192], sn[8192];
  __shared__ __align__(16) float sl[X];  // the slot, staged with all of a thread's loads in flight
  __shared__ float zz[D], smu[D], part[4][D], z2p[4];
  const size_t slot = blockIdx.x;
  const int tid = threadIdx.x;
  {
    const float4* g = reinterpret_cast<const float4*>(slots + slot * X);  // X * 4 bytes: 16-byte aligned slots
    float4 v[(X / 4 + kBT - 1) / kBT];
#pragma unroll
    for (int j = 0; j < (X / 4 + kBT - 1) / kBT; ++j) {
      const int q = tid + j * kBT;
      v[j] = q < X / 4 ? g[q] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int j = 0; j < (X / 4 + kBT - 1) / kBT; ++j) {
      const int q = tid + j * kBT;
      if (q < X / 4) reinterpret_cast<float4*>(sl)[q] = v[j];
    }
    __syncthreads();
  }
  if (mu != nullptr) {
    if (tid < D) zz[tid] = sl[D * D + tid];
    __syncthreads();
    const int e = tid & 63, pc = tid >> 6;  // 4 threads an e, 16 c's each
    float a = 0.f, z2 = 0.f;
#pragma unroll
    for (int c = 16 * pc; c < 16 * pc + 16; ++c) {
      a = fmaf(zz[c], sl[c * D + e], a);
      z2 = fmaf(zz[c], zz[c], z2);
    }
    part[pc][e] = a;
    if (e == 0) z2p[pc] = z2;
    __syncthreads();
    if (tid < D) {
      const float zt = (z2p[0] + z2p[1]) + (z2p[2] + z2p[3]);
      const float m = zt > 0.f ? ((part[0][tid] + part[1][tid]) + (part[2][tid] + part[3][tid])) / zt : 0.f;
      smu[tid] = m;
      mu[slot * D + tid] = m;
    }
    __syncthreads();
  }
  for (int x = tid; x < D * D; x += kBT) {
    const int c = x >> 6, e = x & 63;
    const __nv_bfloat16 v = __float2bfloat16_rn(mu != nullptr ? sl[x] - zz[c] * smu[e] : sl[x]);
    *reinterpret_cast<__nv_bfloat16*>(st + swz64(e, c)) = v;
    *reinterpret_cast<__nv_bfloat16*>(sn + swz64(c, e)) = v;
  }
  __syncthreads();
  uint4* gt = reinterpret_cast<uint4*>(tiles_t + slot * 8192);
  uint4* gn = reinterpret_cast<uint4*>(tiles_n + slot * 8192);
  for (int i = tid; i < 512; i += kBT) {
    gt[i] = reinterpret_cast<const uint4*>(st)[i];
    gn[i] = reinterpret_cast<const uint4*>(sn)[i];
  }
}

// ------------------------------------------------------------------ query pass
template <typename T, int D>
__global__ void __launch_bounds__(kBT, BwdOcc<T, D>::QUERY) bwd_query_kernel(const T* __restrict__ q, const T* __restrict__ dy,
                                                           const float* __restrict__ mixed,
                                                           float* __restrict__ dmixed, T* __restrict__ dq, int N,
                                                           int L, int M, float eps) {
  using G = BwdGeom<D>;
  extern __shared__ __align__(16) float sm[];
  float* St = sm;                    // [D][LD]  S~_i (row c, column e)
  float* Stt = St + D * G::LD;       // [D][LD]  S~_i^T (row e, column c)
  float* zt = Stt + D * G::LD;       // [D]      z~_i
  float* Qk = zt + D;                // [TC][LD] phi(Q), token-major
  float* Qf = Qk + G::TC * G::LD;    // [D][LT]  phi(Q), feature-major
  float* Nk = Qf + D * G::LT;        // [TC][LD] dnum, token-major
  float* Nf = Nk + G::TC * G::LD;    // [D][LT]  dnum, feature-major
  float* den = Nf + D * G::LT;       // [TC]
  float* dd = den + G::TC;           // [TC]     dden
  const int u = blockIdx.x / M, i = blockIdx.x % M;
  const size_t base = ((size_t)u * N + (size_t)i * L) * D;
  const int tg = threadIdx.x / G::NQ, nq = threadIdx.x % G::NQ;  // chunk products
  const int tp0 = tg * G::TT, n0 = nq * 4;
  const int rc = threadIdx.x / 16, re = threadIdx.x % 16, c0 = rc * G::R, e0 = re * G::R;  // dS~

  // first chunk's loads, then S~_i, z~_i into shared memory while they fly
  ChunkRegs<T, D> rq;
  Quad<T> ry[G::TT];  // this thread's dY quads of the chunk
  auto load_chunk = [&](int t0) {
    const int valid = min(G::TC, L - t0);
    rq.load(q + base + (size_t)t0 * D, valid);
#pragma unroll
    for (int a = 0; a < G::TT; ++a)
      ry[a] = ldq(dy + base + (size_t)(t0 + min(tp0 + a, valid - 1)) * D + n0);
  };
  load_chunk(0);
  const float* slot = mixed + ((size_t)u * M + i) * G::X;
  for (int e = threadIdx.x; e < D * D; e += kBT) {
    const int c = e / D, n = e % D;
    const float s = slot[e];
    St[c * G::LD + n] = s;
    Stt[n * G::LD + c] = s;
  }
  for (int c = threadIdx.x; c < D; c += kBT) zt[c] = slot[D * D + c];

  float ds[G::R][G::R] = {};
  float dz[G::R] = {};
  for (int t0 = 0; t0 < L; t0 += G::TC) {
    const int valid = min(G::TC, L - t0);
    __syncthreads();  // the previous chunk's tiles are no longer read
    rq.store(valid, Qk, Qf, PhiOp{});
    float g[G::TT][4];
#pragma unroll
    for (int a = 0; a < G::TT; ++a) {
      const float4 x = to_f4(ry[a]);
      const bool ok = tp0 + a < valid;
      g[a][0] = ok ? x.x : 0.f; g[a][1] = ok ? x.y : 0.f; g[a][2] = ok ? x.z : 0.f; g[a][3] = ok ? x.w : 0.f;
    }
    __syncthreads();
    if (t0 + G::TC < L) load_chunk(t0 + G::TC);  // in flight during this chunk
    {  // den[t] = phi(q_t) . z~ + eps, G::TPT threads a token
      const int t = threadIdx.x / G::TPT, part = threadIdx.x % G::TPT;
      float s = 0.f;
      for (int c = part; c < D; c += G::TPT) s = fmaf(Qk[t * G::LD + c], zt[c], s);
#pragma unroll
      for (int o = G::TPT / 2; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (part == 0) den[t] = s + eps;
    }
    float num[G::TT][4] = {};
    chunk_product<D>(num, Qf, St, tp0, n0);
    __syncthreads();  // den
    // dnum = dY / den, dden = -(dY . num) / den^2 (dY . Y = dY . num / den)
    float part[G::TT];
#pragma unroll
    for (int a = 0; a < G::TT; ++a) {
      part[a] = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) part[a] = fmaf(g[a][j], num[a][j], part[a]);
    }
#pragma unroll
    for (int a = 0; a < G::TT; ++a) {
#pragma unroll
      for (int o = G::NQ / 2; o > 0; o >>= 1) part[a] += __shfl_xor_sync(0xffffffffu, part[a], o);
      const int t = tp0 + a;
      const float inv = t < valid ? 1.f / den[t] : 0.f;  // rows past the block: no contribution
      if (nq == 0) dd[t] = -part[a] * inv * inv;
      const float4 dn = make_float4(g[a][0] * inv, g[a][1] * inv, g[a][2] * inv, g[a][3] * inv);
      *reinterpret_cast<float4*>(Nk + t * G::LD + n0) = dn;
      Nf[(n0 + 0) * G::LT + t] = dn.x;
      Nf[(n0 + 1) * G::LT + t] = dn.y;
      Nf[(n0 + 2) * G::LT + t] = dn.z;
      Nf[(n0 + 3) * G::LT + t] = dn.w;
    }
    __syncthreads();
    // dphi(q) = S~ dnum + dden z~ (as dnum^T S~^T); dq = phi'(q) dphi(q), phi' = min(1, phi)
    float dqf[G::TT][4] = {};
    chunk_product<D>(dqf, Nf, Stt, tp0, n0);
    const float4 z4 = *reinterpret_cast<const float4*>(zt + n0);
#pragma unroll
    for (int a = 0; a < G::TT; ++a) {
      const int t = tp0 + a;
      if (t < valid) {
        const float4 qf = *reinterpret_cast<const float4*>(Qk + t * G::LD + n0);
        const float w = dd[t];
        stq(dq + base + (size_t)(t0 + t) * D + n0,
            make_float4(fminf(1.f, qf.x) * fmaf(w, z4.x, dqf[a][0]), fminf(1.f, qf.y) * fmaf(w, z4.y, dqf[a][1]),
                        fminf(1.f, qf.z) * fmaf(w, z4.z, dqf[a][2]), fminf(1.f, qf.w) * fmaf(w, z4.w, dqf[a][3])));
      }
    }
    // dS~ += phi(Q)^T dnum, dz~ += phi(Q)^T dden
    reduce_tokens<D>(ds, Qk, Nk, c0, e0);
    reduce_rows<D>(dz, Qk, c0, re, [&](int t) { return dd[t]; });
  }
  sum16<G::R>(dz);
  float* out = dmixed + ((size_t)u * M + i) * G::X;
#pragma unroll
  for (int a = 0; a < G::R; ++a)
#pragma unroll
    for (int b = 0; b < G::R; ++b) out[(c0 + a) * D + e0 + b] = ds[a][b];
  if (re == 0)
#pragma unroll
    for (int a = 0; a < G::R; ++a) out[D * D + c0 + a] = dz[a];
}

// ------------------------------------------------------------------ dM partials
// part[h][smp][p][i][b] = sum over the entries x of range p of sample smp's slots of head h of
// dS~[u][i][x] * S[u][b][x]; a thread owns outputs (i, b) = (ti + 16 r, tb + 16 c), r, c < RI,
// RI = ceil(M / 16).
template <int RI>
__global__ void __launch_bounds__(kBT) bwd_dm_kernel(const float* __restrict__ dmixed, const float* __restrict__ slots,
                                                     float* __restrict__ part, int B, int H, int M, int X, int XP) {
  __shared__ float sa[kDmK][kMaxMixM + 1];  // [entry][block]; odd rows: conflict-free stores and loads
  __shared__ float sb[kDmK][kMaxMixM + 1];
  const int p = blockIdx.x % XP, smp = (blockIdx.x / XP) % B, h = blockIdx.x / (XP * B);
  const size_t u = (size_t)smp * H + h;
  const int x_begin = p * kDmRange, x_end = min(X, x_begin + kDmRange);
  const int ti = threadIdx.x / 16, tb = threadIdx.x % 16;
  const float* A = dmixed + u * M * X;
  const float* S = slots + u * M * X;
  float acc[RI][RI] = {};
  for (int xs = x_begin; xs < x_end; xs += kDmK) {
    __syncthreads();
#pragma unroll 8
    for (int e = threadIdx.x; e < kMaxMixM * kDmK; e += kBT) {  // constant trip count: loads in flight
      const int r = e / kDmK, kk = e % kDmK, x = xs + kk;
      if (r >= M) break;  // rows grow with e
      const bool ok = x < x_end;
      const size_t at = (size_t)r * X + min(x, x_end - 1);  // past the range: not read
      sa[kk][r] = ok ? A[at] : 0.f;
      sb[kk][r] = ok ? S[at] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kDmK; ++kk) {
      float a[RI], s[RI];
#pragma unroll
      for (int r = 0; r < RI; ++r) {
        a[r] = sa[kk][ti + 16 * r];  // rows at and past M are never staged: their stale values
        s[r] = sb[kk][tb + 16 * r];  // reach only outputs (i or b >= M) that are not written
      }
#pragma unroll
      for (int r = 0; r < RI; ++r)
#pragma unroll
        for (int c = 0; c < RI; ++c) acc[r][c] = fmaf(a[r], s[c], acc[r][c]);
    }
  }
  float* out = part + (((size_t)h * B + smp) * XP + p) * M * M;
#pragma unroll
  for (int r = 0; r < RI; ++r)
#pragma unroll
    for (int c = 0; c < RI; ++c) {
      const int i = ti + 16 * r, b = tb + 16 * c;
      if (i < M && b < M) out[i * M + b] = acc[r][c];
    }
}

// dM[h] = the head's B * XP partials summed in a fixed order: a warp per output, lane l taking
// partials l, l + 32, ..., then a fixed shuffle tree
__global__ void __launch_bounds__(kBT) bwd_dm_sum_kernel(const float* __restrict__ part, float* __restrict__ dm,
                                                         int H, int M, int P) {
  const int e = blockIdx.x * (kBT / 32) + threadIdx.x / 32, lane = threadIdx.x % 32;
  if (e >= H * M * M) return;  // whole warps leave together
  const int h = e / (M * M), ib = e % (M * M);
  const float* src = part + (size_t)h * P * M * M + ib;
  float s = 0.f;
#pragma unroll 4
  for (int p = lane; p < P; p += 32) s += src[(size_t)p * M * M];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) dm[e] = s;
}

// ------------------------------------------------------------------ key pass
template <typename T, int D>
__global__ void __launch_bounds__(kBT, BwdOcc<T, D>::KEY) bwd_key_kernel(const T* __restrict__ k, const T* __restrict__ v,
                                                         const float* __restrict__ dslots, T* __restrict__ dk,
                                                         T* __restrict__ dv, int N, int L, int M) {
  using G = BwdGeom<D>;
  extern __shared__ __align__(16) float sm[];
  float* dS = sm;                 // [D][LD] dS_b (row c, column e)
  float* dSt = dS + D * G::LD;    // [D][LD] dS_b^T (row e, column c)
  float* dzb = dSt + D * G::LD;   // [D]
  float* Kf = dzb + D;            // [D][LT] phi(K), feature-major
  float* Vf = Kf + D * G::LT;     // [D][LT] V, feature-major
  const int u = blockIdx.x / M, b = blockIdx.x % M;
  const size_t base = ((size_t)u * N + (size_t)b * L) * D;
  ChunkRegs<T, D> rk, rv;
  rk.load(k + base, min(G::TC, L));
  rv.load(v + base, min(G::TC, L));
  const float* slot = dslots + ((size_t)u * M + b) * G::X;
  for (int e = threadIdx.x; e < D * D; e += kBT) {
    const int c = e / D, n = e % D;
    const float s = slot[e];
    dS[c * G::LD + n] = s;
    dSt[n * G::LD + c] = s;
  }
  for (int c = threadIdx.x; c < D; c += kBT) dzb[c] = slot[D * D + c];
  const int tg = threadIdx.x / G::NQ, nq = threadIdx.x % G::NQ;
  const int tp0 = tg * G::TT, n0 = nq * 4;
  for (int t0 = 0; t0 < L; t0 += G::TC) {
    const int valid = min(G::TC, L - t0);
    __syncthreads();
    rk.store(valid, nullptr, Kf, PhiOp{});
    rv.store(valid, nullptr, Vf, IdOp{});
    __syncthreads();
    if (t0 + G::TC < L) {
      const int nv = min(G::TC, L - t0 - G::TC);
      rk.load(k + base + (size_t)(t0 + G::TC) * D, nv);
      rv.load(v + base + (size_t)(t0 + G::TC) * D, nv);
    }
    float gv[G::TT][4] = {}, gk[G::TT][4] = {};
    chunk_product<D>(gv, Kf, dS, tp0, n0);   // dv_t = dS^T phi(k_t):  sum_c phi(k)[c][t] dS[c][e]
    chunk_product<D>(gk, Vf, dSt, tp0, n0);  // dphi(k_t) = dS v_t:    sum_e v[e][t] dS^T[e][c]
    const float4 z4 = *reinterpret_cast<const float4*>(dzb + n0);
#pragma unroll
    for (int a = 0; a < G::TT; ++a) {
      const int t = tp0 + a;
      if (t < valid) {
        const size_t row = base + (size_t)(t0 + t) * D + n0;
        stq(dv + row, make_float4(gv[a][0], gv[a][1], gv[a][2], gv[a][3]));
        stq(dk + row, make_float4(fminf(1.f, Kf[(n0 + 0) * G::LT + t]) * (gk[a][0] + z4.x),
                                  fminf(1.f, Kf[(n0 + 1) * G::LT + t]) * (gk[a][1] + z4.y),
                                  fminf(1.f, Kf[(n0 + 2) * G::LT + t]) * (gk[a][2] + z4.z),
                                  fminf(1.f, Kf[(n0 + 3) * G::LT + t]) * (gk[a][3] + z4.w)));
      }
    }
  }
}

// ------------------------------------------------------------------ plan and launch
// Workspace: a 256-byte header (its status word is set when a tensor-core pass gives up a wait),
// the three slot arrays, the dM partials and, for shapes the tensor-core passes can take (d = 64,
// blocks of whole 128-token chunks), two arrays of bf16 d x d tiles and the rank-one parts mu.
struct BwdPlan {
  int M, X, XP, P;  // XP: dM ranges per slot, P = B * XP partials per head
  size_t slots, dm_part, tiles;  // byte sizes (tiles: one array, 0 without the tensor-core passes)
  size_t off_slots, off_mixed, off_dmixed, off_dm, off_tt, off_tn, off_mu, total;
};

BwdPlan bwd_plan(int B, int H, int N, int d, int block) {
  auto a256 = [](size_t x) { return (x + 255) & ~size_t(255); };
  BwdPlan p{};
  p.M = N / block;
  p.X = d * d + d;
  p.XP = (p.X + kDmRange - 1) / kDmRange;
  p.P = B * p.XP;
  p.slots = a256((size_t)B * H * p.M * p.X * sizeof(float));
  p.dm_part = a256((size_t)H * p.P * p.M * p.M * sizeof(float));
  p.tiles = tc_backward_supported(B, H, N, d, block, MHLA_BF16) ? (size_t)B * H * p.M * 8192 : 0;
  p.off_slots = sizeof(WorkspaceHeader);
  p.off_mixed = p.off_slots + p.slots;
  p.off_dmixed = p.off_mixed + p.slots;
  p.off_dm = p.off_dmixed + p.slots;
  p.off_tt = p.off_dm + p.dm_part;
  p.off_tn = p.off_tt + p.tiles;
  p.off_mu = p.off_tn + p.tiles;
  p.total = p.off_mu + (p.tiles ? (size_t)B * H * p.M * 64 * sizeof(float) : 0);
  return p;
}

template <int D>
constexpr size_t query_smem() {
  using G = BwdGeom<D>;
  return sizeof(float) * (2 * D * G::LD + D + 2 * G::TC * G::LD + 2 * D * G::LT + 2 * G::TC);
}
template <int D>
constexpr size_t key_smem() {
  using G = BwdGeom<D>;
  return sizeof(float) * (2 * D * G::LD + D + 2 * D * G::LT);
}
template <int D>
constexpr size_t summary_smem() {
  using G = BwdGeom<D>;
  return sizeof(float) * 2 * G::TC * G::LD;
}

template <typename T, int D>
cudaError_t backward_t(int B, int H, int N, int block, const void* q, const void* k, const void* v,
                       const float* mixing, const void* dy, void* dq, void* dk, void* dv, float* dm, float eps,
                       void* ws, cudaStream_t st) {
  static SmemOptIn opt_s, opt_q, opt_k;
  const BwdPlan p = bwd_plan(B, H, N, D, block);
  const int U = B * H, M = p.M, X = p.X;
  char* w = static_cast<char*>(ws);
  float* slots = reinterpret_cast<float*>(w + p.off_slots);    // S_b, z_b
  float* mixed = reinterpret_cast<float*>(w + p.off_mixed);    // S~, z~; then dS, dz
  float* dmixed = reinterpret_cast<float*>(w + p.off_dmixed);  // dS~, dz~
  float* dm_part = reinterpret_cast<float*>(w + p.off_dm);
  // the tensor-core token passes (bf16, d = 64, blocks of whole 128-token chunks)
  const bool tc = std::is_same<T, __nv_bfloat16>::value && tc_backward_supported(B, H, N, D, block, MHLA_BF16);
  uint8_t* tt = tc ? reinterpret_cast<uint8_t*>(w + p.off_tt) : nullptr;
  uint8_t* tn = tc ? reinterpret_cast<uint8_t*>(w + p.off_tn) : nullptr;
  float* mu = tc ? reinterpret_cast<float*>(w + p.off_mu) : nullptr;
  unsigned* status = &reinterpret_cast<WorkspaceHeader*>(w)->status;
  const T* tq = static_cast<const T*>(q);
  const T* tk = static_cast<const T*>(k);
  const T* tv = static_cast<const T*>(v);
  cudaError_t e;
  if ((e = opt_s.ensure((const void*)bwd_summary_kernel<T, D>, (int)summary_smem<D>())) != cudaSuccess) return e;
  if ((e = opt_q.ensure((const void*)bwd_query_kernel<T, D>, (int)query_smem<D>())) != cudaSuccess) return e;
  if ((e = opt_k.ensure((const void*)bwd_key_kernel<T, D>, (int)key_smem<D>())) != cudaSuccess) return e;
  const unsigned units_blocks = (unsigned)((size_t)U * M);
  const unsigned mix_grid = (unsigned)((size_t)U * ((X + kBT - 1) / kBT));
  if (tc) {
    if ((e = tc_backward_summary_launch(U, N, block, k, v, slots, status, st)) != cudaSuccess) return e;
  } else {
    bwd_summary_kernel<T, D><<<units_blocks, kBT, summary_smem<D>(), st>>>(tk, tv, slots, N, block, M);
  }
  bwd_mix_kernel<<<mix_grid, kBT, 0, st>>>(slots, mixing, mixed, H, M, X, 0);
  if (tc) {
    bwd_tiles_kernel<<<units_blocks, kBT, 0, st>>>(mixed, mu, tt, tn);
    if ((e = tc_backward_query_launch(U, N, block, q, dy, tt, tn, mu, mixed, dq, dmixed, eps, status, st)) !=
        cudaSuccess)
      return e;
  } else {
    bwd_query_kernel<T, D><<<units_blocks, kBT, query_smem<D>(), st>>>(tq, static_cast<const T*>(dy), mixed, dmixed,
                                                                     static_cast<T*>(dq), N, block, M, eps);
  }
  bwd_mix_kernel<<<mix_grid, kBT, 0, st>>>(dmixed, mixing, mixed, H, M, X, 1);
  if (tc) bwd_tiles_kernel<<<units_blocks, kBT, 0, st>>>(mixed, nullptr, tt, tn);
  const unsigned dm_grid = (unsigned)((size_t)H * p.P);
  switch ((M + 15) / 16) {
    case 1: bwd_dm_kernel<1><<<dm_grid, kBT, 0, st>>>(dmixed, slots, dm_part, B, H, M, X, p.XP); break;
    case 2: bwd_dm_kernel<2><<<dm_grid, kBT, 0, st>>>(dmixed, slots, dm_part, B, H, M, X, p.XP); break;
    case 3: bwd_dm_kernel<3><<<dm_grid, kBT, 0, st>>>(dmixed, slots, dm_part, B, H, M, X, p.XP); break;
    default: bwd_dm_kernel<4><<<dm_grid, kBT, 0, st>>>(dmixed, slots, dm_part, B, H, M, X, p.XP); break;
  }
  bwd_dm_sum_kernel<<<(unsigned)((H * M * M + kBT / 32 - 1) / (kBT / 32)), kBT, 0, st>>>(dm_part, dm, H, M, p.P);
  if (tc) {
    note_launch(6);  // the SIMT launches; the tensor-core passes count their own
    return tc_backward_key_launch(U, N, block, k, v, tt, tn, mixed, dk, dv, status, st);
  }
  bwd_key_kernel<T, D><<<units_blocks, kBT, key_smem<D>(), st>>>(tk, tv, mixed, static_cast<T*>(dk),
                                                               static_cast<T*>(dv), N, block, M);
  note_launch(7);
  return cudaGetLastError();
}

}  // namespace

size_t mhla_backward_workspace(int B, int H, int N, int d, int block) { return bwd_plan(B, H, N, d, block).total; }

mhla_path mhla_backward_kernel_path(int B, int H, int N, int d, int block, mhla_dtype dt) {
  return tc_backward_supported(B, H, N, d, block, dt) ? MHLA_PATH_TCGEN05 : MHLA_PATH_SIMT;
}

int mhla_backward_max_blocks() { return kMaxMixM; }

cudaError_t mhla_backward_launch(int B, int H, int N, int d, int block, mhla_dtype dt, const void* q, const void* k,
                                 const void* v, const float* mixing, const void* dy, void* dq, void* dk, void* dv,
                                 float* dm, float eps, void* ws, cudaStream_t st) {
#define MHLA_BWD_CASE(DV)                                                                                  \
  case DV:                                                                                                 \
    return dt == MHLA_F32 ? backward_t<float, DV>(B, H, N, block, q, k, v, mixing, dy, dq, dk, dv, dm, eps, ws, st) \
                          : backward_t<__nv_bfloat16, DV>(B, H, N, block, q, k, v, mixing, dy, dq, dk, dv, dm, eps, \
                                                          ws, st);
  switch (d) {
    MHLA_BWD_CASE(16)
    MHLA_BWD_CASE(32)
    MHLA_BWD_CASE(64)
    MHLA_BWD_CASE(128)
    default: return cudaErrorInvalidValue;
  }
#undef MHLA_BWD_CASE
}

}  // namespace mhla
