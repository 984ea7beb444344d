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
// Seven launches, everything in fp32 (bf16 inputs and gradients are converted
// at the loads and stores):
//   bwd_summary  (unit, block)   S_b, z_b                      from K, V
//   bwd_mix      (unit, columns) S~, z~  = M  applied to the slots
//   bwd_query    (unit, block)   dQ, dS~_i, dz~_i              from Q, dY, S~_i, z~_i
//   bwd_mix      (unit, columns) dS, dz  = M^T applied to the dS~ slots
//   bwd_dm       (head, range)   partial sums of dM over a range of the head's slot entries
//   bwd_dm_sum   (head)          dM = the partials summed in a fixed order (deterministic)
//   bwd_key      (unit, block)   dK, dV                        from K, V, dS_b, dz_b
// A slot is the d^2 + d floats (S then z) of one (unit, block).  The token
// passes walk a block in chunks of TC tokens staged in shared memory, both
// token-major ([t][c]) and feature-major ([c][t]), so that every product
// reads float4 / float2 vectors: a chunk product out[t][n] = sum_k X[k][t] W[k][n]
// gives a thread TT tokens x 4 columns, a d x d reduction sum_t A[t][c] B[t][e]
// gives it an R x R tile (R = d / 16).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace mhla {
namespace {

constexpr int kBT = 256;     // threads of every backward kernel
constexpr int kMaxMixM = 64; // blocks per sequence the mixing kernels stage
constexpr int kMixCols = 32; // slot entries per mixing CTA
constexpr int kDmK = 32;     // slot entries per stage of the dM kernel

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
  static_assert(TG * NQ == kBT && TT >= 1 && (TT & (TT - 1)) == 0, "chunk product layout");
  static_assert(16 * R == D, "reduction layout");
};

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

// Stage a chunk of TC tokens (rows t0 .. t0 + TC - 1 of a [L][D] block, `valid` of them real) into
// shared memory: token-major tok[t][c] and / or feature-major fea[c][t], through f (phi or identity);
// rows past `valid` are zero.
template <typename T, int D, typename F>
__device__ __forceinline__ void stage_chunk(const T* __restrict__ src, int valid, float* tok, float* fea, F f) {
  using G = BwdGeom<D>;
  for (int e = threadIdx.x; e < G::TC * D; e += kBT) {
    const int t = e / D, c = e - t * D;
    const float raw = to_f(src[(size_t)min(t, valid - 1) * D + c]);  // rows past the block: not read
    const float x = t < valid ? f(raw) : 0.f;
    if (tok) tok[t * G::LD + c] = x;
    if (fea) fea[c * G::LT + t] = x;
  }
}

struct PhiOp { __device__ float operator()(float x) const { return phi(x); } };
struct IdOp { __device__ float operator()(float x) const { return x; } };

// out[t][n] (+)= sum_{k < D} X[k][t] W[k][n]: this thread's TT tokens x 4 columns
template <int D>
__device__ __forceinline__ void chunk_product(float (&acc)[BwdGeom<D>::TT][4], const float* Xf, const float* W,
                                              int t0, int n0) {
  using G = BwdGeom<D>;
#pragma unroll 8
  for (int k = 0; k < D; ++k) {
    float x[G::TT];
    lds<G::TT>(x, Xf + k * G::LT + t0);
    const float4 w = *reinterpret_cast<const float4*>(W + k * G::LD + n0);
#pragma unroll
    for (int i = 0; i < G::TT; ++i) {
      acc[i][0] = fmaf(x[i], w.x, acc[i][0]);
      acc[i][1] = fmaf(x[i], w.y, acc[i][1]);
      acc[i][2] = fmaf(x[i], w.z, acc[i][2]);
      acc[i][3] = fmaf(x[i], w.w, acc[i][3]);
    }
  }
}

// acc[c][e] += sum_{t < TC} A[t][c0 + c] B[t][e0 + e]  (token-major tiles)
template <int D>
__device__ __forceinline__ void reduce_tokens(float (&acc)[BwdGeom<D>::R][BwdGeom<D>::R], const float* A,
                                              const float* B, int c0, int e0) {
  using G = BwdGeom<D>;
#pragma unroll 4
  for (int t = 0; t < G::TC; ++t) {
    float a[G::R], b[G::R];
    lds<G::R>(a, A + t * G::LD + c0);
    lds<G::R>(b, B + t * G::LD + e0);
#pragma unroll
    for (int i = 0; i < G::R; ++i)
#pragma unroll
      for (int j = 0; j < G::R; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
  }
}

// ------------------------------------------------------------------ S_b, z_b
template <typename T, int D>
__global__ void __launch_bounds__(kBT) bwd_summary_kernel(const T* __restrict__ k, const T* __restrict__ v,
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
  for (int t0 = 0; t0 < L; t0 += G::TC) {
    const int valid = min(G::TC, L - t0);
    __syncthreads();
    stage_chunk<T, D>(k + base + (size_t)t0 * D, valid, Kt, nullptr, PhiOp{});
    stage_chunk<T, D>(v + base + (size_t)t0 * D, valid, Vt, nullptr, IdOp{});
    __syncthreads();
    reduce_tokens<D>(acc, Kt, Vt, c0, e0);
    if (re == 0) {
      for (int t = 0; t < G::TC; ++t) {
        float a[G::R];
        lds<G::R>(a, Kt + t * G::LD + c0);
#pragma unroll
        for (int i = 0; i < G::R; ++i) zacc[i] += a[i];
      }
    }
  }
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
// w_ib = m[h][i][b] (transpose = 0) or m[h][b][i] (transpose = 1); a CTA takes kMixCols entries
// of every slot of one unit.
__global__ void __launch_bounds__(kBT) bwd_mix_kernel(const float* __restrict__ in, const float* __restrict__ mixing,
                                                      float* __restrict__ out, int H, int M, int X, int transpose) {
  __shared__ float sw[kMaxMixM * kMaxMixM];
  __shared__ float sin_[kMaxMixM][kMixCols];
  const int cols = (X + kMixCols - 1) / kMixCols;
  const int u = blockIdx.x / cols, x0 = (blockIdx.x % cols) * kMixCols;
  const float* mh = mixing + (size_t)(u % H) * M * M;
  for (int e = threadIdx.x; e < M * M; e += kBT) {
    const int i = e / M, b = e % M;
    sw[i * M + b] = transpose ? mh[(size_t)b * M + i] : mh[(size_t)i * M + b];
  }
  const int lane = threadIdx.x % 32, g = threadIdx.x / 32;
  const int x = x0 + lane;
  const float* ib = in + (size_t)u * M * X;
  for (int b = g; b < M; b += kBT / 32) sin_[b][lane] = x < X ? ib[(size_t)b * X + x] : 0.f;
  __syncthreads();
  if (x >= X) return;
  float* ob = out + (size_t)u * M * X;
  for (int i = g; i < M; i += kBT / 32) {
    float acc = 0.f;
    for (int b = 0; b < M; ++b) acc = fmaf(sw[i * M + b], sin_[b][lane], acc);
    ob[(size_t)i * X + x] = acc;
  }
}

// ------------------------------------------------------------------ query pass
template <typename T, int D>
__global__ void __launch_bounds__(kBT) bwd_query_kernel(const T* __restrict__ q, const T* __restrict__ dy,
                                                        const float* __restrict__ mixed, float* __restrict__ dmixed,
                                                        T* __restrict__ dq, int N, int L, int M, float eps) {
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
  const float* slot = mixed + ((size_t)u * M + i) * G::X;
  for (int e = threadIdx.x; e < D * D; e += kBT) {
    const int c = e / D, n = e % D;
    const float s = slot[e];
    St[c * G::LD + n] = s;
    Stt[n * G::LD + c] = s;
  }
  for (int c = threadIdx.x; c < D; c += kBT) zt[c] = slot[D * D + c];

  const int tg = threadIdx.x / G::NQ, nq = threadIdx.x % G::NQ;  // chunk products
  const int tp0 = tg * G::TT, n0 = nq * 4;
  const int rc = threadIdx.x / 16, re = threadIdx.x % 16, c0 = rc * G::R, e0 = re * G::R;  // dS~
  float ds[G::R][G::R] = {};
  float dz[G::R] = {};
  for (int t0 = 0; t0 < L; t0 += G::TC) {
    const int valid = min(G::TC, L - t0);
    __syncthreads();  // the previous chunk's tiles are no longer read
    stage_chunk<T, D>(q + base + (size_t)t0 * D, valid, Qk, Qf, PhiOp{});
    __syncthreads();
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
    float g[G::TT][4];
    float part[G::TT];
#pragma unroll
    for (int a = 0; a < G::TT; ++a) {
      const int t = tp0 + a;
      const bool ok = t < valid;
      const T* row = dy + base + (size_t)(t0 + (ok ? t : 0)) * D + n0;  // rows past the block: not read
      part[a] = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        g[a][j] = ok ? to_f(row[j]) : 0.f;
        part[a] = fmaf(g[a][j], num[a][j], part[a]);
      }
    }
#pragma unroll
    for (int a = 0; a < G::TT; ++a) {
#pragma unroll
      for (int o = G::NQ / 2; o > 0; o >>= 1) part[a] += __shfl_xor_sync(0xffffffffu, part[a], o);
      const int t = tp0 + a;
      const float inv = t < valid ? 1.f / den[t] : 0.f;  // rows past the block: no contribution
      if (nq == 0) dd[t] = -part[a] * inv * inv;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float dn = g[a][j] * inv;
        Nk[t * G::LD + n0 + j] = dn;
        Nf[(n0 + j) * G::LT + t] = dn;
      }
    }
    __syncthreads();
    // dphi(q) = S~ dnum + dden z~ (as dnum^T S~^T); dq = phi'(q) dphi(q)
    float dqf[G::TT][4] = {};
    chunk_product<D>(dqf, Nf, Stt, tp0, n0);
#pragma unroll
    for (int a = 0; a < G::TT; ++a) {
      const int t = tp0 + a;
      if (t < valid) {
        T* row = dq + base + (size_t)(t0 + t) * D + n0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float gq = fmaf(dd[t], zt[n0 + j], dqf[a][j]);
          row[j] = from_f<T>(fminf(1.f, Qk[t * G::LD + n0 + j]) * gq);
        }
      }
    }
    // dS~ += phi(Q)^T dnum, dz~ += phi(Q)^T dden
    reduce_tokens<D>(ds, Qk, Nk, c0, e0);
    if (re == 0) {
      for (int t = 0; t < G::TC; ++t) {
        float a[G::R];
        lds<G::R>(a, Qk + t * G::LD + c0);
        const float w = dd[t];
#pragma unroll
        for (int r = 0; r < G::R; ++r) dz[r] = fmaf(a[r], w, dz[r]);
      }
    }
  }
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
// part[h][p][i][b] = sum over entries x of range p of the head's slots (sample-major) of
// dS~[u][i][x] * S[u][b][x]; a thread owns a 4 x 4 tile of (i, b) in [0, 64)^2.
__global__ void __launch_bounds__(kBT) bwd_dm_kernel(const float* __restrict__ dmixed, const float* __restrict__ slots,
                                                     float* __restrict__ part, int B, int H, int M, int X, int P,
                                                     long long per) {
  __shared__ __align__(16) float sa[kDmK][kMaxMixM + 4];  // padded rows: fewer bank conflicts in the staging
  __shared__ __align__(16) float sb[kDmK][kMaxMixM + 4];
  const int h = blockIdx.x / P, p = blockIdx.x % P;
  const long long total = (long long)B * X;
  const long long x_begin = (long long)p * per, x_end = min(total, x_begin + per);
  const int ti = threadIdx.x / 16, tb = threadIdx.x % 16;
  float acc[4][4] = {};
  for (long long xs = x_begin; xs < x_end; xs += kDmK) {
    __syncthreads();
    for (int e = threadIdx.x; e < kDmK * kMaxMixM; e += kBT) {
      const int kk = e % kDmK, r = e / kDmK;  // consecutive threads: consecutive entries of one slot
      const long long xg = xs + kk;
      float a = 0.f, s = 0.f;
      if (r < M && xg < x_end) {
        const long long smp = xg / X, x = xg - smp * X;
        const size_t u = (size_t)smp * H + h;
        a = dmixed[(u * M + r) * X + x];
        s = slots[(u * M + r) * X + x];
      }
      sa[kk][r] = a;
      sb[kk][r] = s;
    }
    __syncthreads();
#pragma unroll 4
    for (int kk = 0; kk < kDmK; ++kk) {
      const float4 a = *reinterpret_cast<const float4*>(&sa[kk][ti * 4]);
      const float4 s = *reinterpret_cast<const float4*>(&sb[kk][tb * 4]);
      const float av[4] = {a.x, a.y, a.z, a.w}, sv[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(av[r], sv[c], acc[r][c]);
    }
  }
  float* out = part + ((size_t)h * P + p) * M * M;
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int i = ti * 4 + r, b = tb * 4 + c;
      if (i < M && b < M) out[i * M + b] = acc[r][c];
    }
}

__global__ void __launch_bounds__(kBT) bwd_dm_sum_kernel(const float* __restrict__ part, float* __restrict__ dm,
                                                         int H, int M, int P) {
  const int e = blockIdx.x * kBT + threadIdx.x;
  if (e >= H * M * M) return;
  const int h = e / (M * M), ib = e % (M * M);
  float s = 0.f;
  for (int p = 0; p < P; ++p) s += part[((size_t)h * P + p) * M * M + ib];
  dm[e] = s;
}

// ------------------------------------------------------------------ key pass
template <typename T, int D>
__global__ void __launch_bounds__(kBT) bwd_key_kernel(const T* __restrict__ k, const T* __restrict__ v,
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
    stage_chunk<T, D>(k + base + (size_t)t0 * D, valid, nullptr, Kf, PhiOp{});
    stage_chunk<T, D>(v + base + (size_t)t0 * D, valid, nullptr, Vf, IdOp{});
    __syncthreads();
    float gv[G::TT][4] = {}, gk[G::TT][4] = {};
    chunk_product<D>(gv, Kf, dS, tp0, n0);   // dv_t = dS^T phi(k_t):  sum_c phi(k)[c][t] dS[c][e]
    chunk_product<D>(gk, Vf, dSt, tp0, n0);  // dphi(k_t) = dS v_t:    sum_e v[e][t] dS^T[e][c]
#pragma unroll
    for (int a = 0; a < G::TT; ++a) {
      const int t = tp0 + a;
      if (t < valid) {
        T* rv = dv + base + (size_t)(t0 + t) * D + n0;
        T* rk = dk + base + (size_t)(t0 + t) * D + n0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          rv[j] = from_f<T>(gv[a][j]);
          rk[j] = from_f<T>(fminf(1.f, Kf[(n0 + j) * G::LT + t]) * (gk[a][j] + dzb[n0 + j]));
        }
      }
    }
  }
}

// ------------------------------------------------------------------ plan and launch
struct BwdPlan {
  int M, X, P;
  long long per;
  size_t slots, dm_part, total;  // byte offsets / sizes
};

BwdPlan bwd_plan(int B, int H, int N, int d, int block) {
  BwdPlan p{};
  p.M = N / block;
  p.X = d * d + d;
  const long long total = (long long)B * p.X;
  const long long want = std::max<long long>(1, (2 * 152 + H - 1) / std::max(H, 1));  // ~2 CTAs per SM
  p.P = (int)std::min<long long>(want, (total + kDmK - 1) / kDmK);
  p.per = ((total + p.P - 1) / p.P + kDmK - 1) / kDmK * kDmK;
  p.P = (int)((total + p.per - 1) / p.per);
  const size_t arr = ((size_t)B * H * p.M * p.X * sizeof(float) + 255) & ~size_t(255);
  p.slots = arr;  // one slot array
  p.dm_part = ((size_t)H * p.P * p.M * p.M * sizeof(float) + 255) & ~size_t(255);
  p.total = 3 * arr + p.dm_part;
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
  float* slots = reinterpret_cast<float*>(w);                 // S_b, z_b
  float* mixed = reinterpret_cast<float*>(w + p.slots);       // S~, z~; then dS, dz
  float* dmixed = reinterpret_cast<float*>(w + 2 * p.slots);  // dS~, dz~
  float* dm_part = reinterpret_cast<float*>(w + 3 * p.slots);
  const T* tq = static_cast<const T*>(q);
  const T* tk = static_cast<const T*>(k);
  const T* tv = static_cast<const T*>(v);
  cudaError_t e;
  if ((e = opt_s.ensure((const void*)bwd_summary_kernel<T, D>, (int)summary_smem<D>())) != cudaSuccess) return e;
  if ((e = opt_q.ensure((const void*)bwd_query_kernel<T, D>, (int)query_smem<D>())) != cudaSuccess) return e;
  if ((e = opt_k.ensure((const void*)bwd_key_kernel<T, D>, (int)key_smem<D>())) != cudaSuccess) return e;
  const unsigned units_blocks = (unsigned)((size_t)U * M);
  const unsigned mix_grid = (unsigned)((size_t)U * ((X + kMixCols - 1) / kMixCols));
  bwd_summary_kernel<T, D><<<units_blocks, kBT, summary_smem<D>(), st>>>(tk, tv, slots, N, block, M);
  bwd_mix_kernel<<<mix_grid, kBT, 0, st>>>(slots, mixing, mixed, H, M, X, 0);
  bwd_query_kernel<T, D><<<units_blocks, kBT, query_smem<D>(), st>>>(tq, static_cast<const T*>(dy), mixed, dmixed,
                                                                   static_cast<T*>(dq), N, block, M, eps);
  bwd_mix_kernel<<<mix_grid, kBT, 0, st>>>(dmixed, mixing, mixed, H, M, X, 1);
  bwd_dm_kernel<<<(unsigned)(H * p.P), kBT, 0, st>>>(dmixed, slots, dm_part, B, H, M, X, p.P, p.per);
  bwd_dm_sum_kernel<<<(unsigned)((H * M * M + kBT - 1) / kBT), kBT, 0, st>>>(dm_part, dm, H, M, p.P);
  bwd_key_kernel<T, D><<<units_blocks, kBT, key_smem<D>(), st>>>(tk, tv, mixed, static_cast<T*>(dk),
                                                               static_cast<T*>(dv), N, block, M);
  note_launch(7);
  return cudaGetLastError();
}

}  // namespace

size_t mhla_backward_workspace(int B, int H, int N, int d, int block) { return bwd_plan(B, H, N, d, block).total; }

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
