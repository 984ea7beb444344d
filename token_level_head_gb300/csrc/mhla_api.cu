// C-ABI entry points: argument validation, workspace plans and dispatch.
// The operations and their sources are documented in include/mhla.h.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace mhla {

static std::atomic<unsigned long long> g_launches{0};
void note_launch(int n) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }

namespace {

bool valid_d(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t dtype_bytes(mhla_dtype dt) { return dt == MHLA_F32 ? 4 : 2; }

// [a, a+an) and [b, b+bn) overlap?
bool overlap(const void* a, size_t an, const void* b, size_t bn) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return an != 0 && bn != 0 && x < y + bn && y < x + an;
}

bool dims_ok(int B, int H, int N) { return B >= 0 && H >= 0 && N >= 0; }

size_t elems(int B, int H, int N, int d) { return (size_t)B * H * N * d; }

mhla_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MHLA_OK : MHLA_ERR_CUDA; }

// Workspace of the non-causal (causal = 0) or causal forms: the largest need
// of the kernel families either form may take for these sizes.
size_t mhla_ws(int B, int H, int N, int d, int block, int causal) {
  MhlaShape s{B, H, N, d, block};
  const size_t a = simt_mhla_workspace(s);
  size_t b = causal ? (tc_causal_supported(s, MHLA_BF16, MIX_PREFIX) ? tc_causal_workspace(s) : 0)
                    : (tc_mhla_supported(s, MHLA_BF16, MIX_FULL) ? tc_mhla_workspace(s) : 0);
  if (causal && tc_causal_mhla_supported(s, MHLA_BF16, MIX_STRICT_LOWER))
    b = std::max(b, tc_causal_mhla_workspace(s));
  const size_t c = !causal && tc_stream_supported(s, MHLA_BF16, MIX_FULL) ? tc_stream_workspace(s) : 0;
  return std::max(a, std::max(b, c));
}

// Shared validation of the Q/K/V/Y/den/workspace arguments of the MHLA entries.
mhla_status check_mhla(const void* q, const void* k, const void* v, const void* y,
                       const float* den_out, int B, int H, int N, int d, int block,
                       mhla_dtype dt, float eps, const void* ws, size_t ws_bytes, int causal) {
  if (!dims_ok(B, H, N) || !valid_d(d)) return MHLA_ERR_INVALID_ARG;
  if (dt != MHLA_F32 && dt != MHLA_BF16) return MHLA_ERR_INVALID_ARG;
  if (!std::isfinite(eps) || eps < 0.f) return MHLA_ERR_INVALID_ARG;
  if (block <= 0 || (N > 0 && N % block != 0)) return MHLA_ERR_INVALID_ARG;
  if ((size_t)B * H * N == 0) return MHLA_OK;
  if (!q || !k || !v || !y) return MHLA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(y)) return MHLA_ERR_INVALID_ARG;
  if (den_out && !aligned16(den_out)) return MHLA_ERR_INVALID_ARG;
  const size_t tb = elems(B, H, N, d) * dtype_bytes(dt);
  if (overlap(y, tb, q, tb) || overlap(y, tb, k, tb) || overlap(y, tb, v, tb))
    return MHLA_ERR_INVALID_ARG;
  if (den_out) {
    const size_t db = (size_t)B * H * N * sizeof(float);
    if (overlap(den_out, db, q, tb) || overlap(den_out, db, k, tb) || overlap(den_out, db, v, tb) ||
        overlap(den_out, db, y, tb))
      return MHLA_ERR_INVALID_ARG;
  }
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MHLA_ERR_INVALID_ARG;
  if (ws_bytes < mhla_ws(B, H, N, d, block, causal)) return MHLA_ERR_INVALID_ARG;
  return MHLA_OK;
}

}  // namespace
}  // namespace mhla

using namespace mhla;

extern "C" {

size_t mhla_workspace_bytes(int B, int H, int N, int d, int block_size, int causal) {
  if (!dims_ok(B, H, N) || !valid_d(d) || block_size <= 0 || (N > 0 && N % block_size != 0)) return 0;
  return mhla_ws(B, H, N, d, block_size, causal != 0);
}

mhla_path mhla_forward_path(int B, int H, int N, int d, int block_size, int causal,
                            mhla_dtype dt) {
  if (!dims_ok(B, H, N) || !valid_d(d) || block_size <= 0 || (N > 0 && N % block_size != 0) ||
      (dt != MHLA_F32 && dt != MHLA_BF16) || (causal != 0 && causal != 1))
    return MHLA_PATH_NONE;
  const MhlaShape s{B, H, N, d, block_size};
  if (causal) return tc_causal_supported(s, dt, MIX_PREFIX) ? MHLA_PATH_TCGEN05 : MHLA_PATH_SIMT;  // no mixing
  if (tc_stream_supported(s, dt, MIX_FULL)) return MHLA_PATH_TCGEN05_STREAM;
  return tc_mhla_supported(s, dt, MIX_FULL) ? MHLA_PATH_TCGEN05 : MHLA_PATH_SIMT;
}

// 2-D block geometry: tokens on a gh x gw grid, blocks th x tw tiles covering it.
static bool grid_ok(int gh, int gw, int th, int tw) {
  return gh >= 0 && gw > 0 && th > 0 && tw > 0 && gh % th == 0 && gw % tw == 0 &&
         (long long)gh * gw <= 0x7fffffffLL && (long long)th * tw <= 0x7fffffffLL;
}

// Options valid for this form (mode)?  Fills the variant fields of s.
static bool apply_options(MhlaShape& s, const mhla_options* opt, MixMode mode) {
  if (opt == nullptr) return true;
  if (opt->feature < MHLA_PHI_ELU1 || opt->feature > MHLA_PHI_EXP) return false;
  if (opt->normalise != 0 && opt->normalise != 1) return false;
  if (!std::isfinite(opt->gamma) || opt->gamma < 0.f || opt->gamma > 1.f) return false;
  if (opt->gamma != 1.f && mode != MIX_PREFIX) return false;  // decay: plain causal linear attention only
  s.phi_kind = opt->feature;
  s.normalise = opt->normalise != 0;
  s.gamma = opt->gamma;
  return true;
}

static mhla_status run_mhla(const void* q, const void* k, const void* v, const float* mixing,
                            void* y, float* den_out, int B, int H, int N, int d, int block,
                            MixMode mode, mhla_dtype dt, float eps, void* ws, size_t ws_bytes,
                            void* stream, const int* grid = nullptr, const mhla_options* opt = nullptr) {
  mhla_status st = check_mhla(q, k, v, y, den_out, B, H, N, d, block, dt, eps, ws, ws_bytes, mode != MIX_FULL);
  if (st != MHLA_OK || (size_t)B * H * N == 0) return st;
  if (mode != MIX_PREFIX && (!mixing || !aligned16(mixing))) return MHLA_ERR_INVALID_ARG;
  MhlaShape s{B, H, N, d, block};
  if (!apply_options(s, opt, mode)) return MHLA_ERR_INVALID_ARG;
  if (grid != nullptr) {  // {gh, gw, th, tw}, validated by the caller
    s.gh = grid[0];
    s.gw = grid[1];
    s.th = grid[2];
    s.tw = grid[3];
  }
  if (tc_causal_supported(s, dt, mode))
    return from_cuda(tc_causal_launch(s, q, k, v, y, den_out, eps, ws, static_cast<cudaStream_t>(stream)));
  if (tc_causal_mhla_supported(s, dt, mode))
    return from_cuda(tc_causal_mhla_launch(s, q, k, v, mixing, y, den_out, eps, ws, static_cast<cudaStream_t>(stream)));
  if (tc_stream_supported(s, dt, mode))
    return from_cuda(tc_stream_launch(s, q, k, v, mixing, y, den_out, eps, ws, static_cast<cudaStream_t>(stream)));
  if (tc_mhla_supported(s, dt, mode))
    return from_cuda(tc_mhla_launch(s, q, k, v, mixing, y, den_out, eps, mode, ws,
                                    static_cast<cudaStream_t>(stream)));
  return from_cuda(simt_mhla_launch(s, dt, q, k, v, mixing, y, den_out, eps, mode, ws,
                                    static_cast<cudaStream_t>(stream)));
}

mhla_status mhla_forward(const void* q, const void* k, const void* v, const float* mixing,
                         void* y, float* den_out, int B, int H, int N, int d, int block_size,
                         int causal, mhla_dtype dt, float eps, void* workspace,
                         size_t workspace_bytes, void* stream) {
  if (causal != 0 && causal != 1) return MHLA_ERR_INVALID_ARG;
  if (causal)
    return mhla_forward_causal(q, k, v, mixing, y, den_out, B, H, N, d, block_size, dt, eps,
                               workspace, workspace_bytes, stream);
  return run_mhla(q, k, v, mixing, y, den_out, B, H, N, d, block_size, MIX_FULL, dt, eps,
                  workspace, workspace_bytes, stream);
}

mhla_status mhla_forward_ex(const void* q, const void* k, const void* v, const float* mixing,
                            void* y, float* den_out, int B, int H, int N, int d, int block_size,
                            int causal, mhla_dtype dt, float eps, const mhla_options* opt,
                            void* workspace, size_t workspace_bytes, void* stream) {
  if (causal != 0 && causal != 1) return MHLA_ERR_INVALID_ARG;
  const MixMode mode = !causal ? MIX_FULL : mixing ? MIX_STRICT_LOWER : MIX_PREFIX;
  MhlaShape probe{B, H, N, d, block_size};
  if (!apply_options(probe, opt, mode)) return MHLA_ERR_INVALID_ARG;  // before the no-op exits
  return run_mhla(q, k, v, mixing, y, den_out, B, H, N, d, block_size, mode, dt, eps, workspace,
                  workspace_bytes, stream, nullptr, opt);
}

mhla_path mhla_forward_ex_path(int B, int H, int N, int d, int block_size, int causal, int with_mixing,
                               mhla_dtype dt, const mhla_options* opt) {
  if (!dims_ok(B, H, N) || !valid_d(d) || block_size <= 0 || (N > 0 && N % block_size != 0) ||
      (dt != MHLA_F32 && dt != MHLA_BF16) || (causal != 0 && causal != 1))
    return MHLA_PATH_NONE;
  const MixMode mode = !causal ? MIX_FULL : with_mixing ? MIX_STRICT_LOWER : MIX_PREFIX;
  MhlaShape s{B, H, N, d, block_size};
  if (!apply_options(s, opt, mode)) return MHLA_PATH_NONE;
  if (tc_causal_supported(s, dt, mode) || tc_causal_mhla_supported(s, dt, mode))
    return MHLA_PATH_TCGEN05;  // the order of run_mhla
  if (tc_stream_supported(s, dt, mode)) return MHLA_PATH_TCGEN05_STREAM;
  return tc_mhla_supported(s, dt, mode) ? MHLA_PATH_TCGEN05 : MHLA_PATH_SIMT;
}

mhla_status mhla_forward_grid(const void* q, const void* k, const void* v, const float* mixing,
                              void* y, float* den_out, int B, int H, int grid_h, int grid_w,
                              int tile_h, int tile_w, int d, mhla_dtype dt, float eps,
                              void* workspace, size_t workspace_bytes, void* stream) {
  if (!grid_ok(grid_h, grid_w, tile_h, tile_w)) return MHLA_ERR_INVALID_ARG;
  const int g[4] = {grid_h, grid_w, tile_h, tile_w};
  return run_mhla(q, k, v, mixing, y, den_out, B, H, grid_h * grid_w, d, tile_h * tile_w, MIX_FULL, dt,
                  eps, workspace, workspace_bytes, stream, g);
}

mhla_path mhla_forward_grid_path(int B, int H, int grid_h, int grid_w, int tile_h, int tile_w, int d,
                                 mhla_dtype dt) {
  if (!dims_ok(B, H, 0) || !valid_d(d) || !grid_ok(grid_h, grid_w, tile_h, tile_w) ||
      (dt != MHLA_F32 && dt != MHLA_BF16))
    return MHLA_PATH_NONE;
  MhlaShape s{B, H, grid_h * grid_w, d, tile_h * tile_w};
  s.gh = grid_h;
  s.gw = grid_w;
  s.th = tile_h;
  s.tw = tile_w;
  return tc_mhla_supported(s, dt, MIX_FULL) ? MHLA_PATH_TCGEN05 : MHLA_PATH_SIMT;
}

mhla_status mhla_locality_mixing(float* m, int blocks_h, int blocks_w) {
  if (!m || blocks_h <= 0 || blocks_w <= 0 || (long long)blocks_h * blocks_w > 65536) return MHLA_ERR_INVALID_ARG;
  const int M = blocks_h * blocks_w;
  for (int i = 0; i < M; ++i) {
    const int ri = i / blocks_w, ci = i % blocks_w;
    double far = 0.0;  // distance from block i to the farthest block
    for (int j = 0; j < M; ++j)
      far = std::max(far, std::hypot((double)(j / blocks_w - ri), (double)(j % blocks_w - ci)));
    // weight 1 - dist / far (a lone block: 1), each row normalised to sum to 1
    auto weight = [&](int j) {
      return far > 0.0 ? 1.0 - std::hypot((double)(j / blocks_w - ri), (double)(j % blocks_w - ci)) / far : 1.0;
    };
    double sum = 0.0;
    for (int j = 0; j < M; ++j) sum += weight(j);
    for (int j = 0; j < M; ++j) m[(size_t)i * M + j] = (float)(weight(j) / sum);
  }
  return MHLA_OK;
}

mhla_status mhla_forward_causal(const void* q, const void* k, const void* v, const float* mixing,
                                void* y, float* den_out, int B, int H, int N, int d, int chunk,
                                mhla_dtype dt, float eps, void* workspace, size_t workspace_bytes,
                                void* stream) {
  return run_mhla(q, k, v, mixing, y, den_out, B, H, N, d, chunk,
                  mixing ? MIX_STRICT_LOWER : MIX_PREFIX, dt, eps, workspace, workspace_bytes,
                  stream);
}

mhla_status linattn_decode_step(const void* q, const void* k, const void* v, float* S, float* z,
                                void* out, float* den_out, int B, int H, int d, mhla_dtype dt,
                                float eps, void* stream) {
  if (B < 0 || H < 0 || !valid_d(d)) return MHLA_ERR_INVALID_ARG;
  if (dt != MHLA_F32 && dt != MHLA_BF16) return MHLA_ERR_INVALID_ARG;
  if (!std::isfinite(eps) || eps < 0.f) return MHLA_ERR_INVALID_ARG;
  const size_t units = (size_t)B * H;
  if (units == 0) return MHLA_OK;
  if (!q || !k || !v || !S || !z || !out) return MHLA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(S) || !aligned16(z) ||
      !aligned16(out) || (den_out && !aligned16(den_out)))
    return MHLA_ERR_INVALID_ARG;
  const size_t vb = units * d * dtype_bytes(dt), sb = units * d * d * sizeof(float),
               zb = units * d * sizeof(float);
  if (overlap(out, vb, q, vb) || overlap(out, vb, k, vb) || overlap(out, vb, v, vb) ||
      overlap(out, vb, S, sb) || overlap(out, vb, z, zb) || overlap(S, sb, z, zb) ||
      overlap(S, sb, q, vb) || overlap(S, sb, k, vb) || overlap(S, sb, v, vb))
    return MHLA_ERR_INVALID_ARG;
  if (units > 0x7fffffffu) return MHLA_ERR_UNSUPPORTED;
  return from_cuda(simt_decode_launch((int)units, d, dt, q, k, v, S, z, out, den_out, eps,
                                      static_cast<cudaStream_t>(stream)));
}

mhla_status linattn_decode_steps(const void* q, const void* k, const void* v, float* S, float* z,
                                 void* out, float* den_out, int T, int B, int H, int d, mhla_dtype dt,
                                 float eps, float gamma, void* stream) {
  if (T < 0 || B < 0 || H < 0 || !valid_d(d)) return MHLA_ERR_INVALID_ARG;
  if (dt != MHLA_F32 && dt != MHLA_BF16) return MHLA_ERR_INVALID_ARG;
  if (!std::isfinite(eps) || eps < 0.f) return MHLA_ERR_INVALID_ARG;
  if (!std::isfinite(gamma) || gamma < 0.f || gamma > 1.f) return MHLA_ERR_INVALID_ARG;
  const size_t units = (size_t)B * H;
  if (units == 0) return MHLA_OK;
  if (!S || !z) return MHLA_ERR_INVALID_ARG;
  if (T > 0 && (!q || !k || !v || !out)) return MHLA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(S) || !aligned16(z) ||
      !aligned16(out) || (den_out && !aligned16(den_out)))
    return MHLA_ERR_INVALID_ARG;
  if (units > 0x7fffffffu / 4) return MHLA_ERR_UNSUPPORTED;
  const size_t vb = (size_t)T * units * d * dtype_bytes(dt), sb = units * d * d * sizeof(float),
               zb = units * d * sizeof(float), db = (size_t)T * units * sizeof(float);
  if (T > 0 && (overlap(out, vb, q, vb) || overlap(out, vb, k, vb) || overlap(out, vb, v, vb) ||
                overlap(out, vb, S, sb) || overlap(out, vb, z, zb) || overlap(S, sb, q, vb) ||
                overlap(S, sb, k, vb) || overlap(S, sb, v, vb) || overlap(z, zb, q, vb) ||
                overlap(z, zb, k, vb) || overlap(z, zb, v, vb)))
    return MHLA_ERR_INVALID_ARG;
  if (overlap(S, sb, z, zb)) return MHLA_ERR_INVALID_ARG;
  if (den_out && T > 0 &&
      (overlap(den_out, db, q, vb) || overlap(den_out, db, k, vb) || overlap(den_out, db, v, vb) ||
       overlap(den_out, db, out, vb) || overlap(den_out, db, S, sb) || overlap(den_out, db, z, zb)))
    return MHLA_ERR_INVALID_ARG;
  if (T == 0) return MHLA_OK;
  return from_cuda(decode_steps_launch(T, (int)units, d, dt, q, k, v, S, z, out, den_out, eps, gamma,
                                       static_cast<cudaStream_t>(stream)));
}

mhla_status mhla_causal_stream(const void* q, const void* k, const void* v, const float* mixing, float* S,
                               float* z, void* out, float* den_out, int t0, int T, int B, int H, int d,
                               int block, int M, mhla_dtype dt, float eps, void* stream) {
  if (T < 0 || B < 0 || H < 0 || t0 < 0 || block <= 0 || M <= 0 || !valid_d(d)) return MHLA_ERR_INVALID_ARG;
  if (dt != MHLA_F32 && dt != MHLA_BF16) return MHLA_ERR_INVALID_ARG;
  if (!std::isfinite(eps) || eps < 0.f) return MHLA_ERR_INVALID_ARG;
  if ((long long)t0 + T > (long long)M * block) return MHLA_ERR_INVALID_ARG;  // past the last block
  const size_t units = (size_t)B * H;
  if (units == 0 || T == 0) return MHLA_OK;
  if (!q || !k || !v || !mixing || !S || !z || !out) return MHLA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(mixing) || !aligned16(S) ||
      !aligned16(z) || !aligned16(out) || (den_out && !aligned16(den_out)))
    return MHLA_ERR_INVALID_ARG;
  if (units > 0x7fffffffu) return MHLA_ERR_UNSUPPORTED;
  const size_t vb = (size_t)T * units * d * dtype_bytes(dt), sb = units * M * (size_t)d * d * sizeof(float),
               zb = units * M * (size_t)d * sizeof(float), db = (size_t)T * units * sizeof(float),
               mb = (size_t)H * M * M * sizeof(float);
  const void* ins[] = {q, k, v, mixing};
  const size_t inb[] = {vb, vb, vb, mb};
  for (int i = 0; i < 4; ++i)
    if (overlap(out, vb, ins[i], inb[i]) || overlap(S, sb, ins[i], inb[i]) || overlap(z, zb, ins[i], inb[i]) ||
        (den_out && overlap(den_out, db, ins[i], inb[i])))
      return MHLA_ERR_INVALID_ARG;
  if (overlap(out, vb, S, sb) || overlap(out, vb, z, zb) || overlap(S, sb, z, zb) ||
      (den_out && (overlap(den_out, db, out, vb) || overlap(den_out, db, S, sb) || overlap(den_out, db, z, zb))))
    return MHLA_ERR_INVALID_ARG;
  return from_cuda(causal_stream_launch(t0, T, (int)units, H, d, block, M, dt, q, k, v, mixing, S, z, out, den_out,
                                        eps, static_cast<cudaStream_t>(stream)));
}

size_t mhla_backward_workspace_bytes(int B, int H, int N, int d, int block_size) {
  if (!dims_ok(B, H, N) || !valid_d(d) || block_size <= 0 || (N > 0 && N % block_size != 0)) return 0;
  if (N > 0 && N / block_size > mhla_backward_max_blocks()) return 0;
  return mhla_backward_workspace(B, H, N, d, block_size);
}

mhla_path mhla_backward_path(int B, int H, int N, int d, int block_size, mhla_dtype dt) {
  if (!dims_ok(B, H, N) || !valid_d(d) || block_size <= 0 || (N > 0 && N % block_size != 0) ||
      (dt != MHLA_F32 && dt != MHLA_BF16) || (N > 0 && N / block_size > mhla_backward_max_blocks()))
    return MHLA_PATH_NONE;
  return mhla_backward_kernel_path(B, H, N, d, block_size, dt);
}

mhla_status mhla_backward(const void* q, const void* k, const void* v, const float* mixing, const void* dy,
                          void* dq, void* dk, void* dv, float* dmixing, int B, int H, int N, int d, int block_size,
                          mhla_dtype dt, float eps, void* workspace, size_t workspace_bytes, void* stream) {
  if (!dims_ok(B, H, N) || !valid_d(d)) return MHLA_ERR_INVALID_ARG;
  if (dt != MHLA_F32 && dt != MHLA_BF16) return MHLA_ERR_INVALID_ARG;
  if (!std::isfinite(eps) || eps < 0.f) return MHLA_ERR_INVALID_ARG;
  if (block_size <= 0 || (N > 0 && N % block_size != 0)) return MHLA_ERR_INVALID_ARG;
  if ((size_t)B * H * N == 0) return MHLA_OK;
  const int M = N / block_size;
  if (M > mhla_backward_max_blocks()) return MHLA_ERR_UNSUPPORTED;
  if ((size_t)B * H * M > 0x7fffffffu) return MHLA_ERR_UNSUPPORTED;
  const void* bufs[] = {q, k, v, mixing, dy, dq, dk, dv, dmixing};
  for (const void* b : bufs)
    if (!b || !aligned16(b)) return MHLA_ERR_INVALID_ARG;
  const size_t tb = elems(B, H, N, d) * dtype_bytes(dt), mb = (size_t)H * M * M * sizeof(float);
  const void* ins[] = {q, k, v, dy, mixing};
  const size_t inb[] = {tb, tb, tb, tb, mb};
  void* outs[] = {dq, dk, dv, dmixing};
  const size_t outb[] = {tb, tb, tb, mb};
  for (int o = 0; o < 4; ++o) {
    for (int i = 0; i < 5; ++i)
      if (overlap(outs[o], outb[o], ins[i], inb[i])) return MHLA_ERR_INVALID_ARG;
    for (int j = o + 1; j < 4; ++j)
      if (overlap(outs[o], outb[o], outs[j], outb[j])) return MHLA_ERR_INVALID_ARG;
  }
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MHLA_ERR_INVALID_ARG;
  const size_t need = mhla_backward_workspace(B, H, N, d, block_size);
  if (workspace_bytes < need) return MHLA_ERR_INVALID_ARG;
  for (int o = 0; o < 4; ++o)
    if (overlap(outs[o], outb[o], workspace, need)) return MHLA_ERR_INVALID_ARG;
  for (int i = 0; i < 5; ++i)
    if (overlap(ins[i], inb[i], workspace, need)) return MHLA_ERR_INVALID_ARG;
  return from_cuda(mhla_backward_launch(B, H, N, d, block_size, dt, q, k, v, mixing, dy, dq, dk, dv, dmixing, eps,
                                        workspace, static_cast<cudaStream_t>(stream)));
}

size_t rala_workspace_bytes(int B, int H, int N, int d, int cx) {
  if (!dims_ok(B, H, N) || !valid_d(d) || cx <= 0 || cx % 16 != 0 || cx > 256) return 0;
  const size_t a = simt_rala_workspace(B, H, N, d, cx);
  const size_t b = tc_rala_supported(B, H, N, d, cx, MHLA_BF16) ? tc_rala_workspace(B, H, N) : 0;
  return std::max(a, b);
}

mhla_path rala_forward_path(int B, int H, int N, int d, int cx, mhla_dtype dt) {
  if (!dims_ok(B, H, N) || !valid_d(d) || cx <= 0 || cx % 16 != 0 || cx > 256 ||
      (dt != MHLA_F32 && dt != MHLA_BF16))
    return MHLA_PATH_NONE;
  return tc_rala_supported(B, H, N, d, cx, dt) ? MHLA_PATH_TCGEN05 : MHLA_PATH_SIMT;
}

mhla_status rala_forward(const void* q, const void* k, const void* v, const void* x,
                         const void* w, void* y, int B, int H, int N, int d, int cx,
                         mhla_dtype dt, void* workspace, size_t workspace_bytes, void* stream) {
  if (!dims_ok(B, H, N) || !valid_d(d) || cx <= 0 || cx % 16 != 0 || cx > 256)
    return MHLA_ERR_INVALID_ARG;
  if (dt != MHLA_F32 && dt != MHLA_BF16) return MHLA_ERR_INVALID_ARG;
  if ((size_t)B * H * N == 0) return MHLA_OK;
  if (!q || !k || !v || !x || !w || !y) return MHLA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(x) || !aligned16(w) ||
      !aligned16(y))
    return MHLA_ERR_INVALID_ARG;
  if ((size_t)cx * d > 16384) return MHLA_ERR_UNSUPPORTED;
  const size_t tb = elems(B, H, N, d) * dtype_bytes(dt);
  const size_t xb = (size_t)B * N * cx * dtype_bytes(dt), wb = (size_t)cx * d * dtype_bytes(dt);
  if (overlap(y, tb, q, tb) || overlap(y, tb, k, tb) || overlap(y, tb, v, tb) ||
      overlap(y, tb, x, xb) || overlap(y, tb, w, wb))
    return MHLA_ERR_INVALID_ARG;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MHLA_ERR_INVALID_ARG;
  if (workspace_bytes < rala_workspace_bytes(B, H, N, d, cx)) return MHLA_ERR_INVALID_ARG;
  if (tc_rala_supported(B, H, N, d, cx, dt))
    return from_cuda(tc_rala_launch(B, H, N, q, k, v, x, w, y, workspace, static_cast<cudaStream_t>(stream)));
  return from_cuda(simt_rala_launch(B, H, N, d, cx, dt, q, k, v, x, w, y, workspace,
                                    static_cast<cudaStream_t>(stream)));
}

mhla_status mhla_query_status(void* workspace, void* stream) {
  if (!workspace) return MHLA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return MHLA_ERR_CUDA;
  unsigned int flag = 0;
  auto* hdr = static_cast<WorkspaceHeader*>(workspace);
  if (cudaMemcpy(&flag, &hdr->status, sizeof(flag), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MHLA_ERR_CUDA;
  if (flag == 0) return MHLA_OK;
  const unsigned int zero = 0;
  if (cudaMemcpy(&hdr->status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
    return MHLA_ERR_CUDA;
  return MHLA_ERR_TIMEOUT;
}

const char* mhla_status_string(mhla_status s) {
  switch (s) {
    case MHLA_OK: return "ok";
    case MHLA_ERR_INVALID_ARG: return "invalid argument";
    case MHLA_ERR_UNSUPPORTED: return "unsupported argument combination";
    case MHLA_ERR_CUDA: return "CUDA error";
    case MHLA_ERR_TIMEOUT: return "a bounded device-side wait timed out";
  }
  return "unknown status";
}

unsigned long long mhla_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

void mhla_debug_set_wait_limit_ns(unsigned long long ns) {
  tc_stream_set_wait_limit(ns);
  tc_mhla_set_wait_limit(ns);
  tc_backward_set_wait_limit(ns);
}

}  // extern "C"
