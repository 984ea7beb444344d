// Internal host-side interfaces between the C-ABI layer and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "mhla.h"

namespace mhla {

// Counts every kernel launch (or graph-captured launch) issued by the library.
void note_launch(int n = 1);

// How the non-causal / causal MHLA work is split into summary partials.
struct MhlaShape {
  int B, H, N, d, block;  // block = block_size (non-causal) or chunk (causal)
  // 2-D blocks (non-causal only): tokens on a gh x gw grid in row-major order, blocks the
  // th x tw tiles numbered row-major; gw == 0 means contiguous blocks of `block` tokens.
  // With a grid, N = gh * gw and block = th * tw.
  int gh = 0, gw = 0, th = 0, tw = 0;
  // Variants: feature map (0 ELU + 1, 1 ReLU, 2 exp), whether Y is divided by the
  // denominator, and the decay gamma of plain causal linear attention (1 = none).
  int phi_kind = 0;
  bool normalise = true;
  float gamma = 1.f;
  int heads() const { return B * H; }
  bool plain_phi() const { return phi_kind == 0 && gamma == 1.f; }
  int M() const { return N / block; }
  bool grid() const { return gw > 0; }
};

// Mixing modes of the summary-mixing stage.
enum MixMode {
  MIX_FULL = 0,         // S~_i = sum_j m_ij S_j                (non-causal MHLA)
  MIX_STRICT_LOWER = 1, // S~_i = sum_{j<i} m_ij S_j            (causal MHLA)
  MIX_PREFIX = 2        // S~_i = sum_{j<i} S_j                 (plain causal linear attention)
};

// ---- tcgen05 path (bf16, d = 64, blocks of whole 128-token tiles)
bool tc_mhla_supported(const MhlaShape& s, mhla_dtype dt, MixMode mode);
size_t tc_mhla_workspace(const MhlaShape& s);
cudaError_t tc_mhla_launch(const MhlaShape& s, const void* q, const void* k, const void* v,
                           const float* mixing, void* y, float* den_out, float eps, MixMode mode,
                           void* ws, cudaStream_t st);

// The SUM and MIX passes of the tcgen05 kernel alone, with the weights m_ib for b < i only
// (causal MHLA's mixed prefix P_i = sum_{b<i} m_ib S_b, zeta_i likewise), into the workspace:
// S~_i^T as bf16 8 KB K-major 128-byte-swizzled tiles [heads * M], z~ [heads * M][64] fp32.
bool tc_mhla_prefix_supported(const MhlaShape& s, mhla_dtype dt);
cudaError_t tc_mhla_prefix_launch(const MhlaShape& s, const void* k, const void* v, const float* mixing, void* ws,
                                  cudaStream_t st);
void tc_mhla_mixed_summaries(const MhlaShape& s, void* ws, const uint8_t** smix, const float** zmix);
// Limit of every bounded device-side wait of the three-pass kernel (0 restores the default 0.5 s).
void tc_mhla_set_wait_limit(unsigned long long ns);

// ---- tcgen05 stream path (bf16, d = 64, blocks of whole 128-token tiles, at most 64 tiles a head):
// summaries, mixing and output as one ordered list of items with per-head readiness counters
bool tc_stream_supported(const MhlaShape& s, mhla_dtype dt, MixMode mode);
size_t tc_stream_workspace(const MhlaShape& s);
cudaError_t tc_stream_launch(const MhlaShape& s, const void* q, const void* k, const void* v,
                             const float* mixing, void* y, float* den_out, float eps, void* ws,
                             cudaStream_t st);
// Limit of every bounded device-side wait of the stream kernel (0 restores the default 0.5 s).
void tc_stream_set_wait_limit(unsigned long long ns);

// ---- tcgen05 causal path (bf16, d = 64, plain causal linear attention, N a multiple of 128)
bool tc_causal_supported(const MhlaShape& s, mhla_dtype dt, MixMode mode);
size_t tc_causal_workspace(const MhlaShape& s);
cudaError_t tc_causal_launch(const MhlaShape& s, const void* q, const void* k, const void* v, void* y,
                             float* den_out, float eps, void* ws, cudaStream_t st);

// ---- tcgen05 causal MHLA (mixing, chunk = block = 128, M <= 64): the prefix pass of the MHLA
// kernel, then the causal output kernel on its mixed prefixes
bool tc_causal_mhla_supported(const MhlaShape& s, mhla_dtype dt, MixMode mode);
size_t tc_causal_mhla_workspace(const MhlaShape& s);
cudaError_t tc_causal_mhla_launch(const MhlaShape& s, const void* q, const void* k, const void* v,
                                  const float* mixing, void* y, float* den_out, float eps, void* ws,
                                  cudaStream_t st);

// ---- tcgen05 RALA path (bf16, d = 32, Cx = 64, H <= 2, N a multiple of 64)
bool tc_rala_supported(int B, int H, int N, int d, int cx, mhla_dtype dt);
size_t tc_rala_workspace(int B, int H, int N);
cudaError_t tc_rala_launch(int B, int H, int N, const void* q, const void* k, const void* v, const void* x,
                           const void* w, void* y, void* ws, cudaStream_t st);

// ---- SIMT path (fp32 mode, and every shape the tensor-core path does not take)
size_t simt_mhla_workspace(const MhlaShape& s);
cudaError_t simt_mhla_launch(const MhlaShape& s, mhla_dtype dt, const void* q, const void* k,
                             const void* v, const float* mixing, void* y, float* den_out,
                             float eps, MixMode mode, void* ws, cudaStream_t st);
cudaError_t simt_decode_launch(int units, int d, mhla_dtype dt, const void* q, const void* k,
                               const void* v, float* S, float* z, void* out, float* den_out,
                               float eps, cudaStream_t st);
// ---- fused multi-step decode: T recurrent steps per launch, the state held on chip
cudaError_t decode_steps_launch(int T_steps, int units, int d, mhla_dtype dt, const void* q, const void* k,
                                const void* v, float* S, float* z, void* out, float* den_out, float eps,
                                float gamma, cudaStream_t st);
// ---- causal MHLA inference, token by token: one CTA per unit, running and mixed state in registers
cudaError_t causal_stream_launch(int t0, int T_steps, int units, int H, int d, int block, int M, mhla_dtype dt,
                                 const void* q, const void* k, const void* v, const float* mixing, float* S,
                                 float* z, void* out, float* den_out, float eps, cudaStream_t st);
// ---- backward of the non-causal block form (SIMT, any dtype, d in {16, 32, 64, 128}, M <= 64)
size_t mhla_backward_workspace(int B, int H, int N, int d, int block);
int mhla_backward_max_blocks();
cudaError_t mhla_backward_launch(int B, int H, int N, int d, int block, mhla_dtype dt, const void* q, const void* k,
                                 const void* v, const float* mixing, const void* dy, void* dq, void* dk, void* dv,
                                 float* dm, float eps, void* ws, cudaStream_t st);
// tensor-core token passes of the backward (bf16, d = 64, blocks of whole 128-token chunks)
bool tc_backward_supported(int B, int H, int N, int d, int block, mhla_dtype dt);
void tc_backward_set_wait_limit(unsigned long long ns);
cudaError_t tc_backward_query_launch(int units, int N, int block, const void* q, const void* dy,
                                     const uint8_t* tiles_t, const uint8_t* tiles_n, const float* mu,
                                     const float* mixed, void* dq, float* dmixed, float eps, unsigned* status,
                                     cudaStream_t st);
cudaError_t tc_backward_summary_launch(int units, int N, int block, const void* k, const void* v, float* slots,
                                       unsigned* status, cudaStream_t st);
cudaError_t tc_backward_key_launch(int units, int N, int block, const void* k, const void* v,
                                   const uint8_t* tiles_t, const uint8_t* tiles_n, const float* dslots, void* dk,
                                   void* dv, unsigned* status, cudaStream_t st);
mhla_path mhla_backward_kernel_path(int B, int H, int N, int d, int block, mhla_dtype dt);
size_t simt_rala_workspace(int B, int H, int N, int d, int cx);
cudaError_t simt_rala_launch(int B, int H, int N, int d, int cx, mhla_dtype dt, const void* q,
                             const void* k, const void* v, const void* x, const void* w, void* y,
                             void* ws, cudaStream_t st);

}  // namespace mhla
