/*
 * mhla.h — C ABI of the GB300 (sm_103a) token-level multi-head linear
 * attention (MHLA) forward library.
 *
 * Sources of the operations (cited by page title and section):
 *   [MHLA]  "MHLA: Restoring Expressivity of Linear Attention via Token-Level
 *           Multi-Head" — §4.1 (local KV summaries, multi-head mixing,
 *           output), §4.2 (token-level form, chunkwise-parallel causal form),
 *           App. C (causal chunked linear attention and causal inference).
 *   [LA]    "Linear Attention（线性注意力）笔记" — §二 (phi = ELU + 1),
 *           §四 (recurrent form, eps in the denominator), §五 (parallel form),
 *           §七 (RetNet decay), §八 (the constant-size state).
 *   [MASK]  "4. Attention" tutorial — "Mask": the causal mask removes only
 *           the future (strict upper triangle).
 *   [RALA]  "Breaking the Low-Rank Dilemma of Linear Attention" notes — key
 *           designs 1 (KV buffer rank augmentation) and 2 (output rank
 *           augmentation).
 *
 * Conventions shared by every entry point
 *   - phi(x) = ELU(x) + 1 = (x > 0 ? x + 1 : exp(x))            [LA §二]
 *   - Q, K, V, Y are dense row-major [B, H, N, d] (d innermost); the (b, h)
 *     slices are independent problems.  d must be 16, 32, 64 or 128.
 *   - dtype: MHLA_F32 (fp32 in/out, fp32 arithmetic) or MHLA_BF16 (bf16
 *     in/out, fp32 accumulation; summaries, normalisers and decode state are
 *     fp32).  Outputs have the input dtype.
 *   - Every pointer is a DEVICE pointer unless stated otherwise, 16-byte
 *     aligned; the caller owns all memory, including the workspace.  No call
 *     allocates memory (the one device-resident buffer of the library is the
 *     fixed scratch array of mhla_forward_noalloc, below) and no call keeps
 *     per-call state outside the workspace; calls are asynchronous on `stream`
 *     (a cudaStream_t, 0 = the legacy default stream) and do not synchronise
 *     the host.
 *   - Argument errors are detected on the host before any launch and return
 *     MHLA_ERR_INVALID_ARG (or MHLA_ERR_UNSUPPORTED for valid but
 *     unimplemented combinations) without touching device memory.  Launch
 *     failures return MHLA_ERR_CUDA.  Sizes with B*H*N == 0 are a no-op.
 *   - Workspace: at least the size returned by the matching *_workspace_bytes
 *     query, 256-byte aligned.  Before its FIRST use a workspace must be
 *     zero-filled (e.g. cudaMemsetAsync); the library leaves it ready for the
 *     next call.  Calls that share a workspace must not overlap on the GPU.
 *     A workspace may be reused across shapes as long as it is big enough.
 *   - Device-side waits (between the summary, mixing and output stages of
 *     one launch) are bounded; if one gives up, the output is incomplete and
 *     MHLA_ERR_TIMEOUT is latched in the workspace; mhla_query_status()
 *     reports it.
 */
#ifndef MHLA_GB300_H
#define MHLA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MHLA_OK = 0,
  MHLA_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size, aliasing, small workspace */
  MHLA_ERR_UNSUPPORTED = 2,  /* valid request this build does not implement */
  MHLA_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed */
  MHLA_ERR_TIMEOUT = 4       /* a bounded device-side wait gave up (latched in the workspace) */
} mhla_status;

typedef enum { MHLA_F32 = 0, MHLA_BF16 = 1 } mhla_dtype;

/* Which kernel family mhla_forward / mhla_forward_causal would run:
 * TCGEN05 the three-pass tensor-core kernel (summaries, grid-wide mixing,
 * output), TCGEN05_STREAM the tensor-core kernel that runs them as one stream
 * of work items with per-head readiness (bf16, d = 64, N / 128 not a multiple
 * of 16). */
typedef enum {
  MHLA_PATH_NONE = 0,
  MHLA_PATH_SIMT = 1,
  MHLA_PATH_TCGEN05 = 2,
  MHLA_PATH_TCGEN05_STREAM = 3
} mhla_path;

/* Workspace bytes for mhla_forward (causal = 0) or mhla_forward_causal
 * (causal = 1, block_size = chunk) with these sizes; 0 if the sizes are
 * invalid.  Valid for both dtypes. */
size_t mhla_workspace_bytes(int B, int H, int N, int d, int block_size, int causal);

/* MHLA forward, non-causal ([MHLA] §4.1; eps as in [LA] §五).
 *   Blocks are the M = N / block_size contiguous token ranges of block_size
 *   tokens.  For each (b, h) and block j:
 *     S_j = sum_{t in j} phi(K_t) V_t^T  (d x d, S_j[c][e]),  z_j = sum_{t in j} phi(K_t)
 *   for each query block i:  S~_i = sum_j m[h][i][j] S_j,   z~_i = sum_j m[h][i][j] z_j
 *   for token t in block i:  Y_t = phi(Q_t) S~_i / (phi(Q_t) . z~_i + eps)
 *   q, k, v : [B, H, N, d] (dtype dt)            — inputs
 *   mixing  : [H, M, M] fp32, row i = query block — input; not inspected
 *             (non-negative rows are the caller's contract, [MHLA] §4.2)
 *   y       : [B, H, N, d] (dtype dt)            — output, must not overlap q, k, v
 *   den_out : [B, H, N] fp32 or NULL             — optional output of the denominator
 *   block_size divides N; M = 1 is global linear attention ([LA] §五).
 *   causal  : 0 for the form above; 1 computes causal MHLA exactly as
 *             mhla_forward_causal(..., mixing, ..., chunk = block_size).
 *   eps     : finite, >= 0 (1e-6 in [LA]). */
mhla_status mhla_forward(const void* q, const void* k, const void* v, const float* mixing,
                         void* y, float* den_out, int B, int H, int N, int d, int block_size,
                         int causal, mhla_dtype dt, float eps, void* workspace,
                         size_t workspace_bytes, void* stream);

/* Causal chunked forward ([MHLA] App. C with the [MASK] convention and the
 * [LA] §四 normaliser).  Chunks are contiguous ranges of `chunk` tokens
 * (chunk divides N).  For token t in chunk i:
 *   mixing == NULL (plain causal linear attention):
 *     Y_t = [phi(Q_t) P_i + sum_{s in i, s<=t} (phi(Q_t).phi(K_s)) V_s]
 *         / [phi(Q_t) . zeta_i + sum_{s in i, s<=t} phi(Q_t).phi(K_s) + eps]
 *     with P_i = sum_{j<i} S_j, zeta_i = sum_{j<i} z_j (exclusive prefixes);
 *     equal to the recurrence S_t = S_{t-1} + phi(k_t) v_t^T of [LA] §四.
 *   mixing != NULL ([H, M, M] fp32, M = N / chunk; causal MHLA, [MHLA] §4.2
 *     chunkwise form): P_i = sum_{j<i} m[h][i][j] S_j, zeta_i likewise, and
 *     the intra-chunk sums are scaled by m[h][i][i]; entries above the
 *     diagonal are ignored.
 *   Other arguments as in mhla_forward. */
mhla_status mhla_forward_causal(const void* q, const void* k, const void* v, const float* mixing,
                                void* y, float* den_out, int B, int H, int N, int d, int chunk,
                                mhla_dtype dt, float eps, void* workspace, size_t workspace_bytes,
                                void* stream);

/* Variants of the forward (mhla_forward_ex). */
typedef enum {
  MHLA_PHI_ELU1 = 0, /* phi(x) = ELU(x) + 1 (the default everywhere)   [LA §二] */
  MHLA_PHI_RELU = 1, /* phi(x) = max(x, 0)                              [LA §二] */
  MHLA_PHI_EXP = 2   /* phi(x) = exp(x)                                 [LA §二] */
} mhla_feature;

typedef struct {
  int feature;   /* an mhla_feature */
  int normalise; /* 1: Y = numerator / (phi(q) . z~ + eps) (default);
                    0: Y = numerator alone ([MHLA] §4.1: the normalisation may be
                    omitted for long sequences); den_out, if given, still receives
                    the denominator */
  float gamma;   /* RetNet decay of plain causal linear attention ([LA] §七), in
                    [0, 1]; 1 = none.  Y_t = sum_{s<=t} gamma^(t-s) (phi(q_t).phi(k_s)) v_s
                    / (sum_{s<=t} gamma^(t-s) phi(q_t).phi(k_s) + eps) */
} mhla_options;

/* mhla_forward with variants (opt NULL = the defaults {ELU1, 1, 1.0}, exactly
 * mhla_forward).  gamma != 1 needs causal = 1 and mixing = NULL (plain causal
 * linear attention), else MHLA_ERR_INVALID_ARG; a feature outside the enum,
 * normalise not 0 / 1 or gamma outside [0, 1] are MHLA_ERR_INVALID_ARG.  The
 * tensor-core kernels take ELU + 1 without decay (normalise 0 or 1); the other
 * variants run on the SIMT kernels.  Same workspace as mhla_forward. */
mhla_status mhla_forward_ex(const void* q, const void* k, const void* v, const float* mixing,
                            void* y, float* den_out, int B, int H, int N, int d, int block_size,
                            int causal, mhla_dtype dt, float eps, const mhla_options* opt,
                            void* workspace, size_t workspace_bytes, void* stream);

/* Kernel family mhla_forward_ex would use for these arguments (no launch);
 * `with_mixing` says whether a mixing matrix is passed (it selects causal MHLA
 * or plain causal linear attention when causal = 1). */
mhla_path mhla_forward_ex_path(int B, int H, int N, int d, int block_size, int causal, int with_mixing,
                               mhla_dtype dt, const mhla_options* opt);

/* Non-causal MHLA with 2-D blocks ([MHLA] §4.1: for images the blocks lie on
 * a 2-D grid, Fig. 4b).  The N = grid_h * grid_w tokens of each (b, h) slice
 * are a grid_h x grid_w grid in row-major order (token t = row * grid_w + col,
 * the layout of the [B, H, N, d] tensors is unchanged); the blocks are the
 * tile_h x tile_w tiles of the grid, numbered row-major over the
 * (grid_h / tile_h) x (grid_w / tile_w) tile grid, M = their count; b(t) is
 * the tile holding token t.  Then, as in mhla_forward:
 *   S_b = sum_{t: b(t)=b} phi(K_t) V_t^T,  z_b likewise,
 *   S~_i = sum_b m[h][i][b] S_b,  Y_t = phi(Q_t) S~_{b(t)} / (phi(Q_t) . z~_{b(t)} + eps).
 *   mixing : [H, M, M] fp32 (mhla_locality_mixing gives the paper's initial value).
 *   tile_h must divide grid_h and tile_w grid_w, else MHLA_ERR_INVALID_ARG.
 *   workspace: mhla_workspace_bytes(B, H, grid_h * grid_w, d, tile_h * tile_w, 0).
 *   On a one-row grid (grid_h = tile_h = 1) the blocks are contiguous ranges
 *   of tile_w tokens and the result is that of mhla_forward.
 *   Other arguments as in mhla_forward. */
mhla_status mhla_forward_grid(const void* q, const void* k, const void* v, const float* mixing,
                              void* y, float* den_out, int B, int H, int grid_h, int grid_w,
                              int tile_h, int tile_w, int d, mhla_dtype dt, float eps,
                              void* workspace, size_t workspace_bytes, void* stream);

/* Kernel family mhla_forward_grid would use (no launch): the tensor-core
 * kernels take bf16, d = 64, tiles of a multiple of 128 tokens with tile_w
 * dividing 128 or a multiple of 128, M <= 64; else the SIMT kernels. */
mhla_path mhla_forward_grid_path(int B, int H, int grid_h, int grid_w, int tile_h, int tile_w, int d,
                                 mhla_dtype dt);

/* The locality-based initial mixing matrix of [MHLA] §4.2 for blocks on a
 * blocks_h x blocks_w grid (M = blocks_h * blocks_w, numbered row-major):
 * m[i][j] proportional to 1 - dist(i, j) / max_k dist(i, k), dist the
 * Euclidean distance between the blocks' grid positions, each row normalised
 * to sum to 1 (a single block: [[1]]).  `m` is a HOST array [M][M] fp32 that
 * the caller owns; computed on the host (a one-off initialisation, not part
 * of the forward).  M above 65536 returns MHLA_ERR_INVALID_ARG. */
mhla_status mhla_locality_mixing(float* m, int blocks_h, int blocks_w);

/* One recurrent decode step for B*H independent (batch, head) states
 * ([LA] §四; the fixed-size state of [LA] §八; [MHLA] App. C inference).
 *   q, k, v : [B, H, d] (dtype dt)       — this step's token
 *   S       : [B, H, d, d] fp32, in/out — S[c][e] = sum over past tokens of phi(k)_c v_e
 *   z       : [B, H, d] fp32, in/out    — sum over past tokens of phi(k)
 *   out     : [B, H, d] (dtype dt)      — output; must not overlap the inputs or the state
 *   den_out : [B, H] fp32 or NULL
 *   Order: S += phi(k) v^T; z += phi(k); out = phi(q) S / (phi(q) . z + eps),
 *   i.e. the token attends to itself.  No workspace. */
mhla_status linattn_decode_step(const void* q, const void* k, const void* v, float* S, float* z,
                                void* out, float* den_out, int B, int H, int d, mhla_dtype dt,
                                float eps, void* stream);

/* T consecutive recurrent decode steps in one call, for B*H independent
 * (batch, head) states ([LA] §四 recurrence; [LA] §七 RetNet decay; the
 * fixed-size state of [LA] §八).
 *   q, k, v : [T, B, H, d] (dtype dt)    — step t's tokens at [t]
 *   S       : [B, H, d, d] fp32, in/out — as in linattn_decode_step
 *   z       : [B, H, d] fp32, in/out
 *   out     : [T, B, H, d] (dtype dt)    — must not overlap the inputs or the state
 *   den_out : [T, B, H] fp32 or NULL     — each step's phi(q) . z + eps
 *   gamma   : decay in [0, 1]; 1 gives exactly the steps of linattn_decode_step.
 *   Per step: S <- gamma S + phi(k) v^T; z <- gamma z + phi(k);
 *   out = phi(q) S / (phi(q) . z + eps).  (The notes decay S; z decays with
 *   it so that the output stays a weighted mean of the values.)
 *   Equal, up to fp32 rounding, to T calls of linattn_decode_step when
 *   gamma = 1; the state is read once and written once per call.
 *   T = 0 or B*H = 0 returns MHLA_OK without a launch.  B*H above 2^29
 *   returns MHLA_ERR_UNSUPPORTED.  No workspace. */
mhla_status linattn_decode_steps(const void* q, const void* k, const void* v, float* S, float* z,
                                 void* out, float* den_out, int T, int B, int H, int d, mhla_dtype dt,
                                 float eps, float gamma, void* stream);

/* Causal MHLA inference, token by token ([MHLA] App. C, causal inference):
 * tokens t0 .. t0 + T - 1 of each (b, h) sequence, whose blocks are the
 * contiguous ranges of `block` tokens (block i holds tokens i*block ..).
 *   q, k, v : [T, B, H, d] (dtype dt) — token t0 + n at [n]
 *   mixing  : [H, M, M] fp32, read at and below the diagonal (m[h][i][b], b <= i)
 *   S       : [B, H, M, d, d] fp32, in/out — slot b: the summary sum phi(k) v^T of
 *             block b (S[c][e] = sum phi(k)_c v_e); slots of finished blocks are
 *             frozen, the slot of the block holding token t0 holds its running
 *             summary of the tokens before t0 (ignored, taken as zero, when t0
 *             starts the block)
 *   z       : [B, H, M, d] fp32, in/out — the same for sum phi(k)
 *   out     : [T, B, H, d] (dtype dt);  den_out : [T, B, H] fp32 or NULL
 *   Per token t in block i: S_i += phi(k) v^T; z_i += phi(k);
 *     out = phi(q) (sum_{b<i} m_ib S_b + m_ii S_i)
 *         / (phi(q) . (sum_{b<i} m_ib z_b + m_ii z_i) + eps);
 *   on return the slots of the blocks the call touched hold their summaries
 *   (running for the last one).  Token by token this equals
 *   mhla_forward_causal with this mixing and chunk = block.
 *   t0 + T must not pass M * block (MHLA_ERR_INVALID_ARG).  No workspace. */
mhla_status mhla_causal_stream(const void* q, const void* k, const void* v, const float* mixing, float* S,
                               float* z, void* out, float* den_out, int t0, int T, int B, int H, int d,
                               int block, int M, mhla_dtype dt, float eps, void* stream);

/* Workspace bytes for mhla_backward; 0 if the sizes are invalid or unsupported
 * (N / block_size above 64). */
size_t mhla_backward_workspace_bytes(int B, int H, int N, int d, int block_size);

/* Backward of the non-causal MHLA forward (mhla_forward with causal = 0:
 * contiguous blocks, phi = ELU + 1, with the normaliser) for training the
 * mixing end to end ([MHLA] §4.2; the pages give no backward formulas, these
 * are the chain rule through the steps of [MHLA] §4.1):
 *   dnum_t = dY_t / den_t,  dden_t = -(dY_t . Y_t) / den_t
 *   dS~_i = sum_{t in i} phi(q_t) dnum_t^T,  dz~_i = sum_{t in i} phi(q_t) dden_t
 *   dq_t = phi'(q_t) * (S~_i dnum_t + dden_t z~_i)
 *   dS_b = sum_i m_ib dS~_i,  dz_b = sum_i m_ib dz~_i
 *   dm[h][i][b] = sum over the samples of <dS~_i, S_b> + dz~_i . z_b
 *   dk_j = phi'(k_j) * (dS_b v_j + dz_b),  dv_j = dS_b^T phi(k_j)
 * with phi'(x) = 1 for x > 0 and exp(x) otherwise.  S, z, S~, z~, Y and den
 * are recomputed from q, k, v and the mixing (the forward saves nothing).
 *   q, k, v, dy     : [B, H, N, d] (dtype dt), as given to the forward; dy = dL/dY
 *   mixing          : [H, M, M] fp32, M = N / block_size <= 64
 *   dq, dk, dv      : [B, H, N, d] (dtype dt), written (not accumulated)
 *   dmixing         : [H, M, M] fp32, written (not accumulated); sums over the B samples
 *   workspace       : >= mhla_backward_workspace_bytes(...) device bytes,
 *                     256-byte aligned; must not overlap any argument
 *   workspace       : zero-filled before its first use (a status word at its
 *                     start, as for mhla_forward; the library leaves it zero
 *                     unless a device wait gave up, which mhla_query_status
 *                     reports as MHLA_ERR_TIMEOUT and clears)
 * Paths (mhla_backward_path): bf16 with d = 64 and block_size a multiple of
 * 128 runs the token passes on the tensor cores (bf16 operands: phi(Q),
 * phi(K), V, dY, dnum, dden and the bf16-rounded S~ and dS; fp32
 * accumulation); everything else, and the summaries, mixing and dM, run on
 * the SIMT cores in fp32 (bf16 values widened at the loads, gradients rounded
 * at the stores).  Outputs must not overlap the inputs or each other
 * (MHLA_ERR_INVALID_ARG).  M above 64 returns MHLA_ERR_UNSUPPORTED.
 * B*H*N = 0 returns MHLA_OK without a launch.  Deterministic: every sum has a
 * fixed order. */
mhla_status mhla_backward(const void* q, const void* k, const void* v, const float* mixing, const void* dy,
                          void* dq, void* dk, void* dv, float* dmixing, int B, int H, int N, int d, int block_size,
                          mhla_dtype dt, float eps, void* workspace, size_t workspace_bytes, void* stream);

/* Kernel family mhla_backward would use for these arguments (no launch):
 * MHLA_PATH_TCGEN05 for the tensor-core token passes, MHLA_PATH_SIMT
 * otherwise, MHLA_PATH_NONE for invalid or unsupported sizes. */
mhla_path mhla_backward_path(int B, int H, int N, int d, int block_size, mhla_dtype dt);

/* Workspace bytes for rala_forward; 0 if the sizes are invalid. */
size_t rala_workspace_bytes(int B, int H, int N, int d, int cx);

/* Rank-augmented linear attention forward ([RALA] key designs 1 and 2).
 * For each (b, h):
 *   Q_g = (1/N) sum_t Q_t (raw queries);  l_j = Q_g . phi(K_j);
 *   alpha = softmax_j(l);  Bkv = sum_j alpha_j phi(K_j) V_j^T  (d x d);
 *   G = X_b W  ([N, d], shared by the heads of sample b);
 *   Y_t = G_t * (phi(Q_t) Bkv)   (elementwise product; no normaliser).
 *   q, k, v : [B, H, N, d] (dtype dt);  x : [B, N, cx] (dtype dt);
 *   w : [cx, d] (dtype dt);  y : [B, H, N, d] (dtype dt).
 *   cx must be a multiple of 16 and at most 256. */
mhla_status rala_forward(const void* q, const void* k, const void* v, const void* x,
                         const void* w, void* y, int B, int H, int N, int d, int cx,
                         mhla_dtype dt, void* workspace, size_t workspace_bytes, void* stream);

/* Kernel family rala_forward would use for these arguments (no launch):
 * the tensor-core kernels take bf16 with d = 32, cx = 64, H <= 2 and N a
 * multiple of 64 (at most 8192); everything else runs the SIMT kernels. */
mhla_path rala_forward_path(int B, int H, int N, int d, int cx, mhla_dtype dt);

/* Scratch held by mhla_forward_noalloc on every GPU that loads the library. */
#define MHLA_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20) /* 32 MiB */

/* Non-causal MHLA forward that allocates nothing and takes no workspace.
 * The paper has no counterpart: this exists for callers that cannot obtain
 * device memory for a workspace (no allocator is available to them, or they
 * must not allocate after start-up, e.g. inside a host framework that owns a
 * fixed memory pool).  The result is that of mhla_forward(..., causal = 0,
 * ...) computed by the SIMT kernels; all arguments mean the same.
 *   Scratch: a file-scope device array of MHLA_NOALLOC_SCRATCH_BYTES per GPU,
 *   held until the process exits.  The CUDA runtime reserves it when it loads
 *   the library's device code on that GPU: with the default lazy module
 *   loading (CUDA_MODULE_LOADING=LAZY) that is the first call of this entry
 *   point on the device, which can therefore still fail for lack of device
 *   memory; make one warm-up call at start-up, while memory is known to be
 *   free (with CUDA_MODULE_LOADING=EAGER it happens at context creation).
 *   Sizes whose scratch need exceeds it return MHLA_ERR_UNSUPPORTED before
 *   any launch (the DiT-like B8 H6 N4096 d64 M16 case needs 25.2 MB).
 *   Set-up: the first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call
 *   outside any stream capture.
 *   Every call uses the same array; nothing in it needs to start at zero,
 *   but calls whose kernels overlap on the GPU (other streams, other host
 *   threads) race on it and must be serialised by the caller.
 *   Errors as for mhla_forward; no cudaMalloc/cudaFree is ever called. */
mhla_status mhla_forward_noalloc(const void* q, const void* k, const void* v, const float* mixing,
                                 void* y, float* den_out, int B, int H, int N, int d,
                                 int block_size, mhla_dtype dt, float eps, void* stream);

/* Kernel family mhla_forward would use for these arguments (no launch).
 * With causal = 1 the answer is for plain causal linear attention (mixing
 * NULL); mhla_forward_ex_path answers for causal MHLA with a mixing matrix,
 * which runs on the tensor cores for bf16, d = 64, chunk = 128 and
 * N / 128 <= 64 (the MHLA kernel's summary and mixing passes with the weights
 * below the diagonal, then the causal output kernel), else on the SIMT kernels. */
mhla_path mhla_forward_path(int B, int H, int N, int d, int block_size, int causal,
                            mhla_dtype dt);

/* Synchronises `stream`, then returns MHLA_ERR_TIMEOUT if a device-side wait
 * in a call that used this workspace gave up (and clears the flag), MHLA_OK
 * otherwise, or MHLA_ERR_CUDA if the synchronisation or read failed. */
mhla_status mhla_query_status(void* workspace, void* stream);

/* Static description of a status code (never NULL). */
const char* mhla_status_string(mhla_status s);

/* Number of kernels this library has launched (or captured into a graph) in
 * this process since it was loaded; a diagnostic counter. */
unsigned long long mhla_launch_count(void);

/* Diagnostic: sets the limit, in nanoseconds, of the bounded device-side
 * waits of the non-causal bf16 tensor-core kernels (every wait of the stream
 * path; the waits for the mixed summaries of the three-pass path) and of the
 * tensor-core passes of mhla_backward (every wait) for calls launched after it
 * (process
 * wide; 0 restores the default of 0.5 s).  With a limit too short for the
 * work in flight a call gives up: its output is incomplete, the kernel lets
 * its copies and MMAs in flight finish, leaves the workspace counters at
 * zero, and mhla_query_status() then reports MHLA_ERR_TIMEOUT.  The pages
 * describe no such control; it exists to exercise that failure path. */
void mhla_debug_set_wait_limit_ns(unsigned long long ns);

#ifdef __cplusplus
}
#endif

#endif /* MHLA_GB300_H */
