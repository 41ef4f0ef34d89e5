/*
 * dsv.h -- C ABI of libdsv.so: DSV's dynamic sparse 3D attention on one GB300 (sm_103a).
 *
 * Source of the method: "DSV: Exploiting Dynamic Sparsity to Accelerate Large-Scale
 * Video DiT Training" (German and Spanish technical summaries).  Per attention head
 * a low-rank pair (Q_lr, K_lr) estimates Q K^T (section 2A); one fused kernel forms
 * that estimate and selects the top-k keys without materialising the N x N scores
 * (section 2B, "Fused MM & Top-K"), once per group of 3D-neighbouring queries
 * (section 2B, "Query Grouping"); softmax attention forward and backward then run
 * over the selected keys only (Spanish summary section 3, custom fused kernels for
 * estimation and sparse attention; training needs the backward).
 *
 * Conventions shared by every call
 *   - Layout: contiguous [B][H][N][d] (bf16) for Q, K, V, dO, O, dQ, dK, dV;
 *     [B][H][N][r] (bf16) for Q_lr, K_lr; [B][H][N] fp32 for LSE;
 *     [B][H][N/block][k] int32 for idx.  Tokens are in block-major order: query
 *     block b of a head is rows [block*b, block*b + block).  The caller permutes
 *     tokens (3D cubes of neighbours) before the call; the kernels do not care how.
 *   - Every pointer is a DEVICE pointer owned by the caller, 16-byte aligned.  The
 *     library allocates nothing and frees nothing; it keeps no state between calls
 *     except the device status word read by dsv_last_device_status().
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Calls enqueue work and return at once; none synchronises except
 *     dsv_last_device_status().
 *   - Arguments are validated on the host before anything is launched; an invalid
 *     call returns an error code, launches nothing and writes nothing.
 *     dsv_last_error_message() then holds a one-line reason (per host thread).
 *   - Identical inputs give bitwise-identical outputs (no floating-point atomics).
 */
#ifndef DSV_H
#define DSV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DSV_OK = 0,
    DSV_ERR_INVALID_ARG = 1,   /* bad shape, null or misaligned pointer */
    DSV_ERR_UNSUPPORTED = 2,   /* valid but not built (e.g. d not in {64,128}) */
    DSV_ERR_WORKSPACE = 3,     /* workspace missing or smaller than required */
    DSV_ERR_CUDA = 4,          /* a CUDA runtime call failed (launch, attribute) */
    DSV_ERR_DEVICE_CHECK = 5   /* a kernel found an out-of-range key index */
} dsv_status;

/* Problem sizes.  block must be 64; N % block == 0; 1 <= k <= N;
 * d in {64, 128}; r in {16, 32, 48, 64} (only the estimate reads r);
 * scale <= 0 selects 1/sqrt(d) (the usual softmax scale; the pages give none). */
typedef struct {
    int64_t B, H, N;
    int64_t d, r;
    int64_t block;
    int64_t k;
    float scale;
} dsv_dims;

/* Bytes of device workspace dsv_estimate_topk needs (0: it needs none). */
size_t dsv_estimate_topk_workspace(const dsv_dims* dims);

/*
 * Low-rank estimate + top-k per query block (DSV section 2A/2B: fused MM & top-k
 * with query grouping).
 *   q_hat[b]  = sum of Q_lr over the `block` tokens of query block b;
 *   s[b, j]   = q_hat[b] . K_lr[j]   for every key j of the same head (never stored);
 *   idx[b, :] = the k keys of largest s[b, j], ties to the lower j, ascending order.
 * q_lr, k_lr: bf16 [B][H][N][r].  idx: int32 [B][H][N/block][k] (output).
 * Scores are formed in fp32 from q_hat held as an exact two-term bf16 sum; with
 * integer-valued factors (|q_hat| < 2^16, |s| < 2^24) every score is exact, so the
 * selection equals the exact-arithmetic one.  ws may be NULL when the workspace
 * size is 0.
 */
dsv_status dsv_estimate_topk(const dsv_dims* dims, const void* q_lr, const void* k_lr,
                             int32_t* idx, void* ws, size_t ws_bytes, void* stream);

/*
 * Mass-based adaptive k per query block (DSV German summary section 2A, stage 2, and
 * Spanish summary "Fase 2": the critical KV pairs are those that make up ~90 % of the
 * attention score).  A block's estimated attention distribution over keys is
 * softmax_j(tau s[b, j]) with s the block logits above; k_row[b] is the length of the
 * shortest prefix of its keys, in (s desc, key asc) order, whose mass reaches the fraction
 * mass_num / 2^16 of the total.  The mass is counted in integer weights
 *   w_j = floor(2^24 * 2^x_j),  x_j = tau_log2 * (s[b, j] - max_j s[b, j])  (fp32),
 * 2^x by a fixed fp32 recipe (x = n + f, n = floor(x); 2^f from its Taylor series to degree
 * 6 with coefficients (ln 2)^i / i! rounded to fp32, evaluated in Horner form with every
 * product and sum rounded separately; then scaled by 2^n), w_j = 0 when x_j < -30, and the
 * target is ceil(W * mass_num / 2^16) with W = sum_j w_j.  So the selection is exactly
 * reproducible (for integer-valued factors, as for dsv_estimate_topk).
 *   tau_log2: tau * log2(e) as fp32, > 0 (tau: the estimate's inverse temperature; for a
 *             block-summed logit of 64 queries, 1/64 takes the mean);
 *   mass_num: the mass fraction times 2^16, 1 .. 65536 (0.9 -> 58982);
 *   dense_num: the per-block sparse/dense switch (the pages decide per block, from its
 *             sparsity, whether sparse attention is used): 0 = off, else a block whose k
 *             exceeds the fraction dense_num / 2^16 of the keys (k * 2^16 > dense_num * N)
 *             attends to all N keys (k_row = N);
 *   k_row:    int32 [B][H][N/block] (output), 1 <= k_row[b] <= N;
 *   rowptr:   int64 [B*H*N/block + 1] (output), the CSR offsets: rowptr[0] = 0,
 *             rowptr[i + 1] = rowptr[i] + k_row[i] (rows in [B][H][N/block] order);
 *   order:    int32 [B*H*N/block] (output, may be NULL): the rows by descending
 *             ceil(k_row / 128), a launch order for the CSR attention calls below (the
 *             longest blocks start first); needs N <= 523,904.
 * dims->k is not used (it must still pass validation).  All buffers are device memory
 * owned by the caller; the call only enqueues work on `stream`.
 */
dsv_status dsv_estimate_mass_k(const dsv_dims* dims, const void* q_lr, const void* k_lr, float tau_log2,
                               uint32_t mass_num, uint32_t dense_num, int32_t* k_row, int64_t* rowptr, int32_t* order,
                               void* stream);

/*
 * A longest-first launch order for CSR rows with any per-block k (e.g. a different k per
 * head, all heads in one launch): order (int32 [B*H*N/block], output) lists the rows by
 * descending ceil(k / 128), where k = rowptr[i + 1] - rowptr[i].  Pass it to the CSR
 * attention calls below so the longest blocks start first.  Needs N <= 523,904.
 */
dsv_status dsv_csr_launch_order(const dsv_dims* dims, const int64_t* rowptr, int32_t* order, void* stream);

/*
 * The selected keys of every query block for per-block k (e.g. from dsv_estimate_mass_k),
 * in CSR form: row i's k_row[i] keys of largest s (ties to the lower key, ascending) at
 * cols[rowptr[i] .. rowptr[i + 1]).  k_row[i] must be in [1, N]; cols has rowptr[last]
 * entries (int32, device, caller-owned).  The same selection rule and exactness as
 * dsv_estimate_topk.
 */
dsv_status dsv_estimate_topk_csr(const dsv_dims* dims, const void* q_lr, const void* k_lr, const int32_t* k_row,
                                 const int64_t* rowptr, int32_t* cols, void* stream);

/* Bytes of device workspace dsv_sparse_attn_fwd needs: 0 for every shape at present (the
 * workspace arguments are reserved, so that a future forward may take scratch without an ABI
 * change). */
size_t dsv_sparse_attn_fwd_workspace(const dsv_dims* dims);

/*
 * Sparse attention forward over the selected keys (DSV Spanish summary section 3:
 * sparse attention kernels; page 1 section 2A: only the critical KV pairs are used).
 * For query i of block b:  l_ij = scale * Q_i . K_j for j in idx[b];
 *   LSE_i = max_j l_ij + ln sum_j exp(l_ij - max_j l_ij);  O_i = sum_j exp(l_ij - LSE_i) V_j.
 * q, k, v: bf16 [B][H][N][d].  idx: int32 [B][H][N/block][k], entries in [0, N)
 * (need not be sorted here).  With k = N every key is selected and idx is not read (the
 * dense path; idx may then be NULL).  o: bf16 [B][H][N][d] (output).  lse: fp32 [B][H][N] (output, natural log).
 * Accumulation in fp32.  ws, ws_bytes: a device workspace of at least
 * dsv_sparse_attn_fwd_workspace(dims) bytes (NULL and 0 while that is 0), 16-byte aligned.
 */
dsv_status dsv_sparse_attn_fwd(const dsv_dims* dims, const void* q, const void* k, const void* v,
                               const int32_t* idx, void* o, float* lse, void* ws, size_t ws_bytes, void* stream);

/* Recommended / minimum device workspace for dsv_sparse_attn_bwd.  With more
 * workspace the backward processes more query blocks per wave (fewer launches). */
size_t dsv_sparse_attn_bwd_workspace(const dsv_dims* dims);
size_t dsv_sparse_attn_bwd_workspace_min(const dsv_dims* dims);

/*
 * Sparse attention backward (needed for training, DSV page 1 section 2A stage 2).
 * Recomputes P_ij = exp(scale Q_i.K_j - LSE_i) from the stored LSE, then
 *   D_i = dO_i . O_i;  dS_ij = P_ij (dO_i . V_j - D_i);
 *   dQ_i = scale sum_j dS_ij K_j;
 *   dK_j = scale sum_{i: j in idx[block(i)]} dS_ij Q_i;  dV_j = sum_{same i} P_ij dO_i.
 * Keys no block selected get dK = dV = 0.  No gradient flows to Q_lr / K_lr.
 * The entries of one idx row must be distinct (dsv_estimate_topk writes them strictly
 * ascending); a repeated or out-of-range entry sets the device status word.
 * dK/dV are reduced per key in ascending query-block order from per-(block, key)
 * partial rows held in the workspace: deterministic, no float atomics.  With k = N (every key
 * selected: the pages' dense case) idx is not read and no partial rows exist: dK and dV of each
 * tile of 128 keys accumulate on chip over all query blocks in block order, dQ per query block
 * (idx may then be NULL);
 * the workspace then holds only D = rowsum(dO o O) (4 bytes per query row).
 * d_o, q, k, v, o: bf16 [B][H][N][d]; lse fp32 [B][H][N]; idx int32 [B][H][N/block][k];
 * dq, dk, dv: bf16 [B][H][N][d] (outputs).  ws: device workspace of ws_bytes >=
 * dsv_sparse_attn_bwd_workspace_min(dims), 256-byte aligned.
 */
dsv_status dsv_sparse_attn_bwd(const dsv_dims* dims, const void* d_o, const void* q, const void* k,
                               const void* v, const void* o, const float* lse, const int32_t* idx,
                               void* dq, void* dk, void* dv, void* ws, size_t ws_bytes, void* stream);

/*
 * The backward in two calls, so that its first part can run beside the forward.  The first part
 * (dsv_sparse_attn_bwd_prepare) builds the backward's key-major rank structure of idx in the
 * workspace -- which query blocks selected each key, and where each key's partial rows go -- and
 * reads nothing but idx; the second (dsv_sparse_attn_bwd_prepared) runs the rest of
 * dsv_sparse_attn_bwd on that workspace and gives bitwise the same dQ, dK, dV.  A training step
 * can call prepare on a second stream as soon as idx exists, after the forward is enqueued, so
 * that it fills the SMs the forward leaves idle, and order prepared after it with an event.
 *   - Both calls take the same dims, idx, ws and ws_bytes; ws must hold every head in one wave
 *     (dsv_sparse_attn_bwd_workspace(dims) does when it fits; otherwise DSV_ERR_WORKSPACE).
 *   - prepared must run after prepare has finished (same stream, or an event), and nothing may
 *     write the workspace in between.  Arguments as dsv_sparse_attn_bwd.
 */
dsv_status dsv_sparse_attn_bwd_prepare(const dsv_dims* dims, const int32_t* idx, void* ws, size_t ws_bytes,
                                       void* stream);
dsv_status dsv_sparse_attn_bwd_prepared(const dsv_dims* dims, const void* d_o, const void* q, const void* k,
                                        const void* v, const void* o, const float* lse, const int32_t* idx, void* dq,
                                        void* dk, void* dv, void* ws, size_t ws_bytes, void* stream);

/*
 * Backward without a caller workspace.  Some callers cannot allocate device memory
 * themselves: a host framework that owns every byte of the GPU through its own pool and
 * forbids outside allocations during a step, a plug-in whose memory budget is fixed when
 * its process starts, or a latency-critical loop where cudaMalloc/cudaFree would stall the
 * device.  This entry point computes exactly what dsv_sparse_attn_bwd computes, with the
 * library's own scratch: a fixed array of DSV_NOALLOC_SCRATCH_BYTES (32 MiB) in device
 * memory, held by every GPU that loads the library until the process exits.  It allocates
 * nothing.  (The DSV pages have no counterpart: this is a deployment convenience.)
 *   - Problems whose smallest backward workspace (dsv_sparse_attn_bwd_workspace_min) is
 *     above DSV_NOALLOC_SCRATCH_BYTES are rejected with DSV_ERR_WORKSPACE before anything
 *     runs; larger problems that fit are processed in several waves.  The smallest plan takes
 *     one query block per wave and chains a head's waves through an fp32 accumulator of
 *     8 d N bytes, next to k bf16 partial rows of 4 d bytes, so at d = 128 and the largest
 *     sparse k (N - 1) the limit is about N = 21,000 tokens per head (about N = 43,000 at
 *     d = 64); a head whose partial rows all fit (N/64 * k * 4 d bytes plus its rank structure)
 *     needs no accumulator, and k = N (the dense backward) needs only 4 bytes per query row.
 *     The long-video
 *     shape (N = 520,192, k = 52,019) is rejected: use dsv_sparse_attn_bwd there.
 *   - The first call on a device looks up that device's address of the array (with the
 *     device current); make that first call before any stream capture.
 *   - All calls share the one array, which keeps whatever the last call left there (every
 *     call rebuilds what it reads, so stale contents are never used); calls whose work
 *     overlaps on the GPU (other streams, other host threads) race on it and must be
 *     ordered by the caller.
 * Arguments and outputs are those of dsv_sparse_attn_bwd without ws / ws_bytes.
 */
#define DSV_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
dsv_status dsv_sparse_attn_bwd_noalloc(const dsv_dims* dims, const void* d_o, const void* q, const void* k,
                                       const void* v, const void* o, const float* lse, const int32_t* idx,
                                       void* dq, void* dk, void* dv, void* stream);

/*
 * Sparse attention over per-block key lists in CSR form (e.g. from dsv_estimate_mass_k and
 * dsv_estimate_topk_csr): query block i (rows in [B][H][N/block] order) attends to the keys
 * cols[rowptr[i] .. rowptr[i + 1]) (distinct, within [0, N); ascending order is not needed).
 * The same computation, layouts and outputs as dsv_sparse_attn_fwd / dsv_sparse_attn_bwd;
 * dims->k is not used (it must still pass validation).  A block with no keys gets O = 0,
 * LSE = -inf, dQ = 0.  rowptr: int64 [B*H*N/block + 1], cols: int32 [total_pairs], both
 * device memory owned by the caller.  order (may be NULL): a permutation of the rows in which
 * to launch them (e.g. dsv_estimate_mass_k's, longest first); results do not depend on it.
 * The backward runs as one wave over every head: its workspace must hold
 * dsv_sparse_attn_bwd_csr_workspace(dims, total_pairs) bytes (256-byte aligned), where
 * total_pairs = rowptr[B*H*N/block] (the caller knows it: it sized cols); otherwise
 * DSV_ERR_WORKSPACE.  total_pairs must fit int32.
 */
dsv_status dsv_sparse_attn_fwd_csr(const dsv_dims* dims, const void* q, const void* k, const void* v,
                                   const int64_t* rowptr, const int32_t* cols, const int32_t* order, void* o,
                                   float* lse, void* stream);
size_t dsv_sparse_attn_bwd_csr_workspace(const dsv_dims* dims, int64_t total_pairs);
dsv_status dsv_sparse_attn_bwd_csr(const dsv_dims* dims, const void* d_o, const void* q, const void* k, const void* v,
                                   const void* o, const float* lse, const int64_t* rowptr, const int32_t* cols,
                                   const int32_t* order, int64_t total_pairs, void* dq, void* dk, void* dv, void* ws,
                                   size_t ws_bytes, void* stream);

/* Human-readable name of a status code (static string). */
const char* dsv_status_string(dsv_status status);

/* One-line reason for the last non-OK status returned on this host thread. */
const char* dsv_last_error_message(void);

/* Synchronises `stream`, then reads and clears the current device's status word.
 * Returns DSV_ERR_DEVICE_CHECK if a kernel met a key index outside [0, N) since the
 * last read (the offending entry is skipped, never dereferenced), DSV_ERR_CUDA if
 * the synchronisation failed, DSV_OK otherwise. */
dsv_status dsv_last_device_status(void* stream);

/*
 * Optional per-kernel device timing, for measurement tools (not needed for use).
 * While enabled, every kernel launch the library makes is bracketed by two CUDA events
 * recorded on the launch's own stream (events come from a pool created at enable time;
 * no device memory is allocated).  dsv_profile_read() waits for the recorded events and
 * writes one line per kernel, "name launches total_ms\n", summed since the previous read,
 * into buf (NUL-terminated, truncated to buf_bytes); it returns the bytes needed.  With
 * buf == NULL it only reports the size and keeps the records.  Disabling drops unread
 * records.  Not thread-safe against concurrent launches from several host threads.
 */
dsv_status dsv_profile_enable(int on);
size_t dsv_profile_read(char* buf, size_t buf_bytes);

/* ---------------------------------------------------------------- fused AdaLN
 * LayerNorm + modulation in one pass over HBM, forward and backward (AdaptiveLoad page,
 * "AdaptiveLoad: Towards Efficient Video Diffusion Transformer Training", technical summary
 * section 2B: normalisation and modulation fused into one launch, statistics kept on chip,
 * and the modulation gradients reduced in (D tile, N tile) blocks so that reads stay
 * coalesced along D).  Per token n of sample b, over its D features:
 *   mean = sum_d x / D,  var = sum_d (x - mean)^2 / D,  rstd = 1 / sqrt(var + eps),
 *   xhat = (x - mean) * rstd,   y = xhat * (1 + scale[b]) + shift[b].
 * The backward recomputes mean and rstd from x (nothing is saved by the forward) and returns
 *   dx = rstd * (g - mean_d(g) - xhat * mean_d(g * xhat)),  g = dy * (1 + scale[b]),
 *   d_scale[b] = sum_n dy * xhat,   d_shift[b] = sum_n dy.
 * Arithmetic: bf16 inputs, fp32 statistics and sums, bf16 y / dx, fp32 d_scale / d_shift;
 * bitwise reproducible (fixed summation order, no float atomics).
 * Layouts (contiguous, device memory owned by the caller, 16-byte aligned):
 *   x, y, dy, dx: bf16 [B][N][D];  scale, shift: bf16 [B][D];  d_scale, d_shift: fp32 [B][D].
 * Validation before any launch: B, N >= 1; D a multiple of 8 in [8, 8192]; eps >= 0 and
 * finite; no NULL or misaligned pointer (DSV_ERR_INVALID_ARG).  With eps = 0 a constant row
 * has var = 0 and its y / dx are NaN, as the definition gives.  Asynchronous on `stream`.
 */
typedef struct {
  int64_t B;   /* samples */
  int64_t N;   /* tokens per sample */
  int64_t D;   /* features per token */
  float eps;   /* added to the variance inside the square root */
} dsv_adaln_dims;

dsv_status dsv_adaln_fwd(const dsv_adaln_dims* dims, const void* x, const void* scale, const void* shift,
                         void* y, void* stream);
/* Bytes of workspace dsv_adaln_bwd needs (per-tile partial sums of the modulation gradients). */
size_t dsv_adaln_bwd_workspace(const dsv_adaln_dims* dims);
/* ws: at least dsv_adaln_bwd_workspace(dims) bytes, 256-byte aligned (DSV_ERR_WORKSPACE otherwise).
 * It holds per-tile partial sums and the tickets that order their final sum, so one workspace
 * must not serve two backward calls that can run at the same time (other streams); calls in
 * order on one stream may share it.  The call runs two kernels, the second launched as a
 * programmatic dependent of the first (it waits for the first to finish before reading). */
dsv_status dsv_adaln_bwd(const dsv_adaln_dims* dims, const void* x, const void* scale, const void* dy, void* dx,
                         float* d_scale, float* d_shift, void* ws, size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DSV_H */
