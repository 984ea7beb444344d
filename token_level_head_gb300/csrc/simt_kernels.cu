// SIMT (CUDA-core) kernels of the MHLA library.
//
// These carry the fp32 mode (fp32 FMA everywhere, which the 1e-4 parity bar
// needs: tensor-core tf32/bf16 products are ~1e-3 accurate) and every shape
// the tensor-core kernels do not take.  They follow the block form of
// "MHLA: Restoring Expressivity of Linear Attention via Token-Level
// Multi-Head" §4.1 in three stages: per-chunk summaries (S, z), mixing of
// the summaries per query block, and the normalised output.  The causal form
// (App. C of the same paper) adds the masked intra-chunk term in the output
// stage; the decode step follows "Linear Attention notes" §四; the RALA
// kernels follow "Breaking the Low-Rank Dilemma of Linear Attention", key
// designs 1 and 2.
#include <algorithm>
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace mhla {
namespace {

constexpr int kThreads = 256;
constexpr int kTokTile = 32;   // tokens staged per smem tile
constexpr int kOutTile = 32;   // max query tokens per output CTA

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Largest divisor of n that is <= cap.
inline int divisor_at_most(int n, int cap) {
  for (int c = std::min(n, cap); c >= 1; --c)
    if (n % c == 0) return c;
  return 1;
}

// Token of the j-th position of block b: blocks are the th x tw tiles, numbered row-major, of
// a grid of rows gw tokens wide (MHLA paper §4.1: blocks on a 2-D grid for images).
// Contiguous blocks of `block` tokens are the 1 x block tiles of a 1 x N grid.
struct TokMap {
  int gw, tw, th, bpr;  // grid width, tile width and height, tiles per grid row
  __device__ __forceinline__ int tok(int b, int j) const {
    const int lr = j / tw, lc = j - lr * tw;
    const int br = b / bpr, bc = b - br * bpr;
    return (br * th + lr) * gw + bc * tw + lc;
  }
};

TokMap tok_map(const MhlaShape& s) {
  if (s.grid()) return TokMap{s.gw, s.tw, s.th, s.gw / s.tw};
  return TokMap{s.N, s.block, 1, s.N / s.block};
}

// ---------------------------------------------------------------- summaries
// S_part[head][p] = sum_{t in chunk p} phi(K_t) V_t^T ; z_part[head][p] = sum phi(K_t)
// (MHLA paper §4.1, local KV summary; chunks subdivide the blocks; chunk p holds positions
// [(p % P) chunk, (p % P + 1) chunk) of block p / P).  With a decay gamma != 1 (plain causal
// linear attention, "Linear Attention notes" §七) each token is weighted gamma^(block - 1 - j),
// j its position in the block: the block's summary decayed to its last token.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
simt_summary_kernel(const T* __restrict__ K, const T* __restrict__ V, float* __restrict__ s_part,
                    float* __restrict__ z_part, int N, int chunk, int P, TokMap map, int phi_kind,
                    float gamma, int block) {
  constexpr int E = (D * D + kThreads - 1) / kThreads;
  __shared__ float sk[kTokTile][D];
  __shared__ float sv[kTokTile][D];
  const int head = blockIdx.y, part = blockIdx.x;
  const int blk = part / P, j0 = (part - blk * P) * chunk;
  const size_t hbase = (size_t)head * N * D;
  float acc[E];
#pragma unroll
  for (int j = 0; j < E; ++j) acc[j] = 0.f;
  float zacc = 0.f;
  for (int t0 = 0; t0 < chunk; t0 += kTokTile) {
    const int nt = min(kTokTile, chunk - t0);
    for (int i = threadIdx.x; i < nt * D; i += kThreads) {
      const int j = j0 + t0 + i / D;
      const size_t at = hbase + (size_t)map.tok(blk, j) * D + i % D;
      const float w = gamma == 1.f ? 1.f : powf(gamma, (float)(block - 1 - j));
      sk[i / D][i % D] = w * phi_k(to_f(K[at]), phi_kind);
      sv[i / D][i % D] = to_f(V[at]);
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < E; ++j) {
      const int idx = threadIdx.x + j * kThreads;
      if (idx < D * D) {
        const int c = idx / D, e = idx % D;
        float a = acc[j];
        for (int t = 0; t < nt; ++t) a = fmaf(sk[t][c], sv[t][e], a);
        acc[j] = a;
      }
    }
    if (threadIdx.x < D)
      for (int t = 0; t < nt; ++t) zacc += sk[t][threadIdx.x];
    __syncthreads();
  }
  float* sp = s_part + ((size_t)head * gridDim.x + part) * D * D;
#pragma unroll
  for (int j = 0; j < E; ++j) {
    const int idx = threadIdx.x + j * kThreads;
    if (idx < D * D) sp[idx] = acc[j];
  }
  if (threadIdx.x < D) z_part[((size_t)head * gridDim.x + part) * D + threadIdx.x] = zacc;
}

// ------------------------------------------------------------------- mixing
// For each head and query block i (MHLA paper §4.1 multi-head mixing, and the
// causal variants of §4.2 / App. C):
//   MIX_FULL:         S~_i = sum_j m_ij S_j
//   MIX_STRICT_LOWER: S~_i = sum_{j<i} m_ij S_j
//   MIX_PREFIX:       S~_i = sum_{j<i} S_j   (with decay: S~_i = gamma^block S~_{i-1} + S_{i-1},
//                     the state after block i - 1's last token)
// where S_j = sum of the P partials of block j.  Same for z.  One thread per
// entry of the (d*d + d) summary.
__global__ void __launch_bounds__(kThreads)
simt_mix_kernel(const float* __restrict__ s_part, const float* __restrict__ z_part,
                const float* __restrict__ mixing, float* __restrict__ s_mix,
                float* __restrict__ z_mix, int H, int M, int P, int D, int mode, float decay_block) {
  const int head = blockIdx.y;
  const int dd = D * D;
  const int ent = blockIdx.x * blockDim.x + threadIdx.x;
  if (ent >= dd + D) return;
  const bool isz = ent >= dd;
  const int col = isz ? ent - dd : ent;
  const size_t stride = isz ? (size_t)D : (size_t)dd;
  const float* src = (isz ? z_part + (size_t)head * M * P * D : s_part + (size_t)head * M * P * dd) + col;
  float* dst = (isz ? z_mix + (size_t)head * M * D : s_mix + (size_t)head * M * dd) + col;
  if (mode == MIX_PREFIX) {
    float run = 0.f;
    for (int b = 0; b < M; ++b) {
      dst[(size_t)b * stride] = run;
      float tsum = 0.f;
      for (int p = 0; p < P; ++p) tsum += src[(size_t)(b * P + p) * stride];
      run = fmaf(run, decay_block, tsum);
    }
    return;
  }
  const float* mh = mixing + (size_t)(head % H) * M * M;
  for (int i0 = 0; i0 < M; i0 += 16) {
    float acc[16];
#pragma unroll
    for (int ii = 0; ii < 16; ++ii) acc[ii] = 0.f;
    for (int b = 0; b < M; ++b) {
      float tsum = 0.f;
      for (int p = 0; p < P; ++p) tsum += src[(size_t)(b * P + p) * stride];
#pragma unroll
      for (int ii = 0; ii < 16; ++ii) {
        const int i = i0 + ii;
        if (i < M) {
          float w = mh[(size_t)i * M + b];
          if (mode == MIX_STRICT_LOWER && b >= i) w = 0.f;
          acc[ii] = fmaf(w, tsum, acc[ii]);
        }
      }
    }
#pragma unroll
    for (int ii = 0; ii < 16; ++ii)
      if (i0 + ii < M) dst[(size_t)(i0 + ii) * stride] = acc[ii];
  }
}

// ------------------------------------------------------------------- output
// Y_t = [phi(Q_t) S~_i + w_ii * sum_{s in block i, s<=t} (phi(Q_t).phi(K_s)) V_s]
//     / [phi(Q_t).z~_i + w_ii * sum_{s in block i, s<=t} phi(Q_t).phi(K_s) + eps]
// The intra-block terms are present only for the causal forms (intra_mode 1:
// w_ii = m_ii of the mixing, intra_mode 2: w_ii = 1); MHLA paper §4.1 output,
// App. C chunk form with the lower triangle including the diagonal.  A CTA takes
// positions t0 .. t0 + tile - 1 of block t0 / block (tokens by `map`; the causal
// forms have contiguous blocks, so there position and token coincide).
// Variants: the feature map phi_kind; normalise = 0 writes the numerator alone
// (MHLA paper §4.1: the normaliser may be left out), den_out still the
// denominator; a decay gamma != 1 (intra_mode 2 only) weights the state before
// the block by gamma^(j + 1) and the intra-block scores by gamma^(t - s).
template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
simt_out_kernel(const T* __restrict__ Q, const T* __restrict__ K, const T* __restrict__ V,
                const float* __restrict__ s_mix, const float* __restrict__ z_mix,
                const float* __restrict__ mixing, T* __restrict__ Y, float* __restrict__ den_out,
                int H, int N, int block, int tile, float eps, int intra_mode, TokMap map, int phi_kind,
                int normalise, float gamma) {
  constexpr int ROWS = kThreads / D;
  constexpr int PASSES = (kOutTile + ROWS - 1) / ROWS;
  extern __shared__ float smem[];
  float* sS = smem;                 // D*D
  float* sz = sS + D * D;           // D
  float* sq = sz + D;               // kOutTile*D   phi(q)
  float* sk = sq + kOutTile * D;    // kTokTile*D   phi(k)
  float* sv = sk + kTokTile * D;    // kTokTile*D   v
  float* ssc = sv + kTokTile * D;   // kOutTile*kTokTile scores
  const int head = blockIdx.y;
  const int t0 = blockIdx.x * tile;
  const int blk = t0 / block;
  const int M = N / block;
  const size_t hbase = (size_t)head * N * D;
  for (int i = threadIdx.x; i < D * D; i += kThreads) sS[i] = s_mix[((size_t)head * M + blk) * D * D + i];
  for (int i = threadIdx.x; i < D; i += kThreads) sz[i] = z_mix[((size_t)head * M + blk) * D + i];
  const int j0 = t0 - blk * block;
  for (int i = threadIdx.x; i < tile * D; i += kThreads)
    sq[i] = phi_k(to_f(Q[hbase + (size_t)map.tok(blk, j0 + i / D) * D + i % D]), phi_kind);
  __syncthreads();
  const int e = threadIdx.x % D, r = threadIdx.x / D;
  float num[PASSES], nin[PASSES], rs[PASSES];
#pragma unroll
  for (int p = 0; p < PASSES; ++p) {
    num[p] = 0.f; nin[p] = 0.f; rs[p] = 0.f;
    const int t = r + p * ROWS;
    if (t < tile)
      for (int c = 0; c < D; ++c) num[p] = fmaf(sq[t * D + c], sS[c * D + e], num[p]);
  }
  float w_ii = 1.f;
  if (intra_mode != 0) {
    if (intra_mode == 1) w_ii = mixing[((size_t)(head % H) * M + blk) * M + blk];
    const int last = t0 + tile - 1;
    for (int s0 = blk * block; s0 <= last; s0 += kTokTile) {
      const int ns = min(kTokTile, last + 1 - s0);
      for (int i = threadIdx.x; i < ns * D; i += kThreads) {
        sk[i] = phi_k(to_f(K[hbase + (size_t)s0 * D + i]), phi_kind);
        sv[i] = to_f(V[hbase + (size_t)s0 * D + i]);
      }
      __syncthreads();
      for (int idx = threadIdx.x; idx < tile * ns; idx += kThreads) {
        const int t = idx / ns, s = idx % ns;
        float dot = 0.f;
        for (int c = 0; c < D; ++c) dot = fmaf(sq[t * D + c], sk[s * D + c], dot);
        const int lag = (t0 + t) - (s0 + s);
        if (gamma != 1.f) dot *= powf(gamma, (float)lag);
        ssc[t * kTokTile + s] = lag >= 0 ? dot : 0.f;  // causal mask keeps s <= t
      }
      __syncthreads();
#pragma unroll
      for (int p = 0; p < PASSES; ++p) {
        const int t = r + p * ROWS;
        if (t < tile)
          for (int s = 0; s < ns; ++s) {
            const float sc = ssc[t * kTokTile + s];
            nin[p] = fmaf(sc, sv[s * D + e], nin[p]);
            rs[p] += sc;
          }
      }
      __syncthreads();
    }
  }
#pragma unroll
  for (int p = 0; p < PASSES; ++p) {
    const int t = r + p * ROWS;
    if (t < tile) {
      float den = 0.f;
      for (int c = 0; c < D; ++c) den = fmaf(sq[t * D + c], sz[c], den);
      const float gd = gamma == 1.f ? 1.f : powf(gamma, (float)(j0 + t + 1));  // state before the block
      den = fmaf(gd, den, w_ii * rs[p]) + eps;
      const float n = fmaf(gd, num[p], w_ii * nin[p]);
      const float y = normalise ? n / den : n;
      const int tok = map.tok(blk, j0 + t);
      Y[hbase + (size_t)tok * D + e] = from_f<T>(y);
      if (den_out != nullptr && e == 0) den_out[(size_t)head * N + tok] = den;
    }
  }
}

size_t out_smem_bytes(int D) {
  return sizeof(float) * ((size_t)D * D + D + (size_t)kOutTile * D + 2 * (size_t)kTokTile * D +
                          (size_t)kOutTile * kTokTile);
}

struct SimtPlan {
  int chunk, P, parts;  // summary chunk, partials per block, partials per head
  size_t off_spart, off_zpart, off_smix, off_zmix, total;
};

SimtPlan simt_plan(const MhlaShape& s) {
  SimtPlan p;
  p.chunk = divisor_at_most(s.block, 256);
  p.P = s.block / p.chunk;
  p.parts = s.N / p.chunk;
  const size_t heads = (size_t)s.heads(), dd = (size_t)s.d * s.d;
  size_t off = kWorkspacePrefix;
  p.off_spart = off; off = align256(off + heads * p.parts * dd * sizeof(float));
  p.off_zpart = off; off = align256(off + heads * p.parts * s.d * sizeof(float));
  p.off_smix = off;  off = align256(off + heads * s.M() * dd * sizeof(float));
  p.off_zmix = off;  off = align256(off + heads * s.M() * s.d * sizeof(float));
  p.total = off;
  return p;
}

template <typename T, int D>
cudaError_t mhla_launch_t(const MhlaShape& s, const SimtPlan& pl, const void* q, const void* k,
                          const void* v, const float* mixing, void* y, float* den_out, float eps,
                          MixMode mode, char* ws, cudaStream_t st) {
  float* s_part = reinterpret_cast<float*>(ws + pl.off_spart);
  float* z_part = reinterpret_cast<float*>(ws + pl.off_zpart);
  float* s_mix = reinterpret_cast<float*>(ws + pl.off_smix);
  float* z_mix = reinterpret_cast<float*>(ws + pl.off_zmix);
  const int heads = s.heads(), M = s.M();
  const TokMap map = tok_map(s);
  simt_summary_kernel<T, D><<<dim3(pl.parts, heads), kThreads, 0, st>>>(
      static_cast<const T*>(k), static_cast<const T*>(v), s_part, z_part, s.N, pl.chunk, pl.P, map, s.phi_kind,
      s.gamma, s.block);
  note_launch();
  const int ents = D * D + D;
  simt_mix_kernel<<<dim3((ents + kThreads - 1) / kThreads, heads), kThreads, 0, st>>>(
      s_part, z_part, mixing, s_mix, z_mix, s.H, M, pl.P, D, (int)mode,
      s.gamma == 1.f ? 1.f : std::pow(s.gamma, (float)s.block));
  note_launch();
  const int tile = divisor_at_most(s.block, kOutTile);
  const size_t smem = out_smem_bytes(D);
  static SmemOptIn opt_in;  // the first call on a device is eager (outside any graph capture)
  if (cudaError_t err = opt_in.ensure((const void*)simt_out_kernel<T, D>, (int)smem); err != cudaSuccess)
    return err;
  const int intra = mode == MIX_FULL ? 0 : (mode == MIX_STRICT_LOWER ? 1 : 2);
  simt_out_kernel<T, D><<<dim3(s.N / tile, heads), kThreads, smem, st>>>(
      static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v), s_mix, z_mix,
      mixing, static_cast<T*>(y), den_out, s.H, s.N, s.block, tile, eps, intra, map, s.phi_kind,
      s.normalise ? 1 : 0, s.gamma);
  note_launch();
  return cudaGetLastError();
}

// ------------------------------------------------------------------- decode
// One step for each (batch, head) unit ("Linear Attention notes" §四):
// S += phi(k) v^T, z += phi(k), out = phi(q) S / (phi(q).z + eps).
template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
simt_decode_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                   float* __restrict__ S, float* __restrict__ z, T* __restrict__ out,
                   float* __restrict__ den_out, float eps) {
  constexpr int G = kThreads / D;
  __shared__ float sq[D], sk[D], sv[D];
  __shared__ float red[G][D];
  __shared__ float sden;
  const int u = blockIdx.x, tid = threadIdx.x;
  if (tid < D) {
    sq[tid] = phi(to_f(q[(size_t)u * D + tid]));
    sk[tid] = phi(to_f(k[(size_t)u * D + tid]));
    sv[tid] = to_f(v[(size_t)u * D + tid]);
  }
  __syncthreads();
  const int e = tid % D, g = tid / D;
  float* su = S + (size_t)u * D * D;
  float acc = 0.f;
  for (int c = g; c < D; c += G) {
    const float snew = fmaf(sk[c], sv[e], su[c * D + e]);
    su[c * D + e] = snew;
    acc = fmaf(sq[c], snew, acc);
  }
  red[g][e] = acc;
  if (tid < 32) {
    float part = 0.f;
    for (int c = tid; c < D; c += 32) {
      const float zn = z[(size_t)u * D + c] + sk[c];
      z[(size_t)u * D + c] = zn;
      part = fmaf(sq[c], zn, part);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (tid == 0) sden = part + eps;
  }
  __syncthreads();
  if (tid < D) {
    float a = 0.f;
#pragma unroll
    for (int gg = 0; gg < G; ++gg) a += red[gg][tid];
    out[(size_t)u * D + tid] = from_f<T>(a / sden);
  }
  if (den_out != nullptr && tid == 0) den_out[u] = sden;
}

template <typename T, int D>
cudaError_t decode_t(int units, const void* q, const void* k, const void* v, float* S, float* z,
                     void* out, float* den_out, float eps, cudaStream_t st) {
  simt_decode_kernel<T, D><<<units, kThreads, 0, st>>>(
      static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v), S, z,
      static_cast<T*>(out), den_out, eps);
  note_launch();
  return cudaGetLastError();
}

// --------------------------------------------------------------------- RALA
// "Breaking the Low-Rank Dilemma of Linear Attention", key design 1:
//   Q_g = mean_t Q_t, l_j = Q_g.phi(K_j), alpha = softmax(l),
//   B = sum_j alpha_j phi(K_j) V_j^T;
// key design 2: Y_t = (X W)_t * (phi(Q_t) B).
// The softmax over all N tokens is split over token tiles: each tile keeps
// its own max m_t, sum s_t = sum exp(l - m_t) and B_t = sum exp(l - m_t)
// phi(k) v^T, and the combine step rescales them by exp(m_t - max).
constexpr int kRalaTile = 256;

template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
rala_qsum_kernel(const T* __restrict__ Q, float* __restrict__ qpart, int N) {
  constexpr int G = kThreads / D;
  __shared__ float red[G][D];
  const int head = blockIdx.y, tile = blockIdx.x;
  const int t0 = tile * kRalaTile, nt = min(kRalaTile, N - t0);
  const int c = threadIdx.x % D, g = threadIdx.x / D;
  const T* qh = Q + ((size_t)head * N + t0) * D;
  float a = 0.f;
  for (int t = g; t < nt; t += G) a += to_f(qh[(size_t)t * D + c]);
  red[g][c] = a;
  __syncthreads();
  if (threadIdx.x < D) {
    float s = 0.f;
    for (int gg = 0; gg < G; ++gg) s += red[gg][threadIdx.x];
    qpart[((size_t)head * gridDim.x + tile) * D + threadIdx.x] = s;
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
rala_tile_kernel(const T* __restrict__ K, const T* __restrict__ V, const float* __restrict__ qpart,
                 float* __restrict__ bpart, float* __restrict__ mpart, float* __restrict__ spart,
                 int N) {
  constexpr int E = (D * D + kThreads - 1) / kThreads;
  __shared__ float sqg[D];
  __shared__ float sk[kTokTile][D];
  __shared__ float sv[kTokTile][D];
  __shared__ float sl[kRalaTile];
  __shared__ float sw[kRalaTile];
  __shared__ float smax, ssum;
  const int head = blockIdx.y, tile = blockIdx.x, ntiles = gridDim.x;
  const int t0 = tile * kRalaTile, nt = min(kRalaTile, N - t0);
  const size_t hbase = ((size_t)head * N + t0) * D;
  if (threadIdx.x < D) {
    float s = 0.f;
    for (int i = 0; i < ntiles; ++i) s += qpart[((size_t)head * ntiles + i) * D + threadIdx.x];
    sqg[threadIdx.x] = s / (float)N;  // Q_g: mean of the raw queries
  }
  __syncthreads();
  // logits of this tile's keys
  for (int t = threadIdx.x; t < nt; t += kThreads) {
    float l = 0.f;
    for (int c = 0; c < D; ++c) l = fmaf(sqg[c], phi(to_f(K[hbase + (size_t)t * D + c])), l);
    sl[t] = l;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    float m = -INFINITY;
    for (int t = threadIdx.x; t < nt; t += 32) m = fmaxf(m, sl[t]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float s = 0.f;
    for (int t = threadIdx.x; t < nt; t += 32) {
      const float w = expf(sl[t] - m);
      sw[t] = w;
      s += w;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (threadIdx.x == 0) { smax = m; ssum = s; }
  }
  __syncthreads();
  float acc[E];
#pragma unroll
  for (int j = 0; j < E; ++j) acc[j] = 0.f;
  for (int s0 = 0; s0 < nt; s0 += kTokTile) {
    const int ns = min(kTokTile, nt - s0);
    for (int i = threadIdx.x; i < ns * D; i += kThreads) {
      sk[i / D][i % D] = sw[s0 + i / D] * phi(to_f(K[hbase + (size_t)s0 * D + i]));
      sv[i / D][i % D] = to_f(V[hbase + (size_t)s0 * D + i]);
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < E; ++j) {
      const int idx = threadIdx.x + j * kThreads;
      if (idx < D * D) {
        const int c = idx / D, e = idx % D;
        float a = acc[j];
        for (int t = 0; t < ns; ++t) a = fmaf(sk[t][c], sv[t][e], a);
        acc[j] = a;
      }
    }
    __syncthreads();
  }
  float* bp = bpart + ((size_t)head * ntiles + tile) * D * D;
#pragma unroll
  for (int j = 0; j < E; ++j) {
    const int idx = threadIdx.x + j * kThreads;
    if (idx < D * D) bp[idx] = acc[j];
  }
  if (threadIdx.x == 0) {
    mpart[(size_t)head * ntiles + tile] = smax;
    spart[(size_t)head * ntiles + tile] = ssum;
  }
}

__global__ void __launch_bounds__(kThreads)
rala_combine_kernel(const float* __restrict__ bpart, const float* __restrict__ mpart,
                    const float* __restrict__ spart, float* __restrict__ bkv, int ntiles, int D) {
  const int head = blockIdx.y;
  const int idx = blockIdx.x * kThreads + threadIdx.x;
  if (idx >= D * D) return;
  float m = -INFINITY;
  for (int i = 0; i < ntiles; ++i) m = fmaxf(m, mpart[(size_t)head * ntiles + i]);
  float tot = 0.f, acc = 0.f;
  for (int i = 0; i < ntiles; ++i) {
    const float sc = expf(mpart[(size_t)head * ntiles + i] - m);
    tot = fmaf(spart[(size_t)head * ntiles + i], sc, tot);
    acc = fmaf(bpart[((size_t)head * ntiles + i) * D * D + idx], sc, acc);
  }
  bkv[(size_t)head * D * D + idx] = acc / tot;
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
rala_out_kernel(const T* __restrict__ Q, const T* __restrict__ X, const T* __restrict__ W,
                const float* __restrict__ bkv, T* __restrict__ Y, int H, int N, int cx) {
  constexpr int ROWS = kThreads / D;
  extern __shared__ float smem[];
  float* sW = smem;             // cx * D
  float* sB = sW + cx * D;      // D * D
  const int head = blockIdx.y, b = head / H;
  const int t0 = blockIdx.x * kTokTile, nt = min(kTokTile, N - t0);
  for (int i = threadIdx.x; i < cx * D; i += kThreads) sW[i] = to_f(W[i]);
  for (int i = threadIdx.x; i < D * D; i += kThreads) sB[i] = bkv[(size_t)head * D * D + i];
  __syncthreads();
  const int e = threadIdx.x % D, r = threadIdx.x / D;
  for (int t = r; t < nt; t += ROWS) {
    const T* xr = X + ((size_t)b * N + t0 + t) * cx;
    float g = 0.f;
    for (int c = 0; c < cx; ++c) g = fmaf(to_f(xr[c]), sW[c * D + e], g);
    const T* qr = Q + ((size_t)head * N + t0 + t) * D;
    float a = 0.f;
    for (int c = 0; c < D; ++c) a = fmaf(phi(to_f(qr[c])), sB[c * D + e], a);
    Y[((size_t)head * N + t0 + t) * D + e] = from_f<T>(g * a);
  }
}

struct RalaPlan {
  int ntiles;
  size_t off_qpart, off_bpart, off_m, off_s, off_bkv, total;
};

RalaPlan rala_plan(int B, int H, int N, int d) {
  RalaPlan p;
  p.ntiles = (N + kRalaTile - 1) / kRalaTile;
  const size_t heads = (size_t)B * H;
  size_t off = kWorkspacePrefix;
  p.off_qpart = off; off = align256(off + heads * p.ntiles * d * sizeof(float));
  p.off_bpart = off; off = align256(off + heads * p.ntiles * (size_t)d * d * sizeof(float));
  p.off_m = off;     off = align256(off + heads * p.ntiles * sizeof(float));
  p.off_s = off;     off = align256(off + heads * p.ntiles * sizeof(float));
  p.off_bkv = off;   off = align256(off + heads * (size_t)d * d * sizeof(float));
  p.total = off;
  return p;
}

template <typename T, int D>
cudaError_t rala_t(int B, int H, int N, int cx, const void* q, const void* k, const void* v,
                   const void* x, const void* w, void* y, char* ws, cudaStream_t st) {
  const RalaPlan pl = rala_plan(B, H, N, D);
  float* qpart = reinterpret_cast<float*>(ws + pl.off_qpart);
  float* bpart = reinterpret_cast<float*>(ws + pl.off_bpart);
  float* mpart = reinterpret_cast<float*>(ws + pl.off_m);
  float* spart = reinterpret_cast<float*>(ws + pl.off_s);
  float* bkv = reinterpret_cast<float*>(ws + pl.off_bkv);
  const int heads = B * H;
  rala_qsum_kernel<T, D><<<dim3(pl.ntiles, heads), kThreads, 0, st>>>(static_cast<const T*>(q), qpart, N);
  note_launch();
  rala_tile_kernel<T, D><<<dim3(pl.ntiles, heads), kThreads, 0, st>>>(
      static_cast<const T*>(k), static_cast<const T*>(v), qpart, bpart, mpart, spart, N);
  note_launch();
  rala_combine_kernel<<<dim3((D * D + kThreads - 1) / kThreads, heads), kThreads, 0, st>>>(
      bpart, mpart, spart, bkv, pl.ntiles, D);
  note_launch();
  const size_t smem = sizeof(float) * ((size_t)cx * D + (size_t)D * D);
  static SmemOptIn opt_in;
  if (cudaError_t err = opt_in.ensure((const void*)rala_out_kernel<T, D>, (int)(sizeof(float) * (256 * D + D * D)));
      err != cudaSuccess)
    return err;
  rala_out_kernel<T, D><<<dim3((N + kTokTile - 1) / kTokTile, heads), kThreads, smem, st>>>(
      static_cast<const T*>(q), static_cast<const T*>(x), static_cast<const T*>(w), bkv,
      static_cast<T*>(y), H, N, cx);
  note_launch();
  return cudaGetLastError();
}

}  // namespace

// ------------------------------------------------------------ host entries
size_t simt_mhla_workspace(const MhlaShape& s) { return simt_plan(s).total; }

#define MHLA_DISPATCH_D(D_, CALL)                                     \
  switch (D_) {                                                       \
    case 16: { constexpr int DV = 16; return CALL; }                  \
    case 32: { constexpr int DV = 32; return CALL; }                  \
    case 64: { constexpr int DV = 64; return CALL; }                  \
    case 128: { constexpr int DV = 128; return CALL; }                \
    default: return cudaErrorInvalidValue;                            \
  }

cudaError_t simt_mhla_launch(const MhlaShape& s, mhla_dtype dt, const void* q, const void* k,
                             const void* v, const float* mixing, void* y, float* den_out,
                             float eps, MixMode mode, void* ws, cudaStream_t st) {
  const SimtPlan pl = simt_plan(s);
  char* w = static_cast<char*>(ws);
  if (dt == MHLA_F32) {
    MHLA_DISPATCH_D(s.d, (mhla_launch_t<float, DV>(s, pl, q, k, v, mixing, y, den_out, eps, mode, w, st)));
  }
  MHLA_DISPATCH_D(s.d, (mhla_launch_t<__nv_bfloat16, DV>(s, pl, q, k, v, mixing, y, den_out, eps, mode, w, st)));
}

cudaError_t simt_decode_launch(int units, int d, mhla_dtype dt, const void* q, const void* k,
                               const void* v, float* S, float* z, void* out, float* den_out,
                               float eps, cudaStream_t st) {
  if (dt == MHLA_F32) {
    MHLA_DISPATCH_D(d, (decode_t<float, DV>(units, q, k, v, S, z, out, den_out, eps, st)));
  }
  MHLA_DISPATCH_D(d, (decode_t<__nv_bfloat16, DV>(units, q, k, v, S, z, out, den_out, eps, st)));
}

size_t simt_rala_workspace(int B, int H, int N, int d, int cx) {
  (void)cx;
  return rala_plan(B, H, N, d).total;
}

cudaError_t simt_rala_launch(int B, int H, int N, int d, int cx, mhla_dtype dt, const void* q,
                             const void* k, const void* v, const void* x, const void* w, void* y,
                             void* ws, cudaStream_t st) {
  char* wsp = static_cast<char*>(ws);
  if (dt == MHLA_F32) {
    MHLA_DISPATCH_D(d, (rala_t<float, DV>(B, H, N, cx, q, k, v, x, w, y, wsp, st)));
  }
  MHLA_DISPATCH_D(d, (rala_t<__nv_bfloat16, DV>(B, H, N, cx, q, k, v, x, w, y, wsp, st)));
}

}  // namespace mhla
