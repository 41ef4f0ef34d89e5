// Host-side launch interface between the C ABI (dsv_api.cu) and the kernel files.
// Everything here is validated by the caller before a launch happens.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dsv {

using bf16 = __nv_bfloat16;

// Brackets one kernel launch with CUDA events when per-kernel timing is enabled
// (dsv_profile_enable); a no-op otherwise.
struct ProfScope {
  int slot;
  cudaStream_t stream;
  ProfScope(const char* name, cudaStream_t s);
  ~ProfScope();
};

struct EstimateParams {
  const bf16* q_lr;   // [BH][N][r]
  const bf16* k_lr;   // [BH][N][r]
  int32_t* idx;       // [BH][NB][k], or CSR columns when rowptr is set
  int64_t BH, N, NB, topk;
  int r;
  const int32_t* krow = nullptr;   // per-row k (adaptive selection), or null: topk for every row
  const int64_t* rowptr = nullptr; // CSR row offsets into idx, or null: row * topk
  unsigned int* status;
};
cudaError_t launch_estimate_topk(const EstimateParams& p, cudaStream_t stream);

// Mass-based adaptive k: per query block the length of the shortest (score desc, key asc)
// prefix of its keys whose integer weight reaches ceil(W * mass_num / 2^16); weights
// w = floor(2^24 * 2^x), x = tau_log2 * (s - max s) in fp32, 2^x by a fixed fp32 recipe
// (Taylor coefficients coef[0..6] of 2^f on [0, 1)).  Writes krow [BH][NB] and the CSR
// offsets rowptr [BH * NB + 1].
struct MassParams {
  const bf16* q_lr;
  const bf16* k_lr;
  int64_t BH, N, NB;
  int r;
  float tau_log2;
  uint32_t mass_num;
  uint32_t dense_num;  // 0, or: k * 2^16 > dense_num * N makes a block dense (k = N)
  float coef[7];
  int32_t* krow;
  int64_t* rowptr;
  int32_t* order = nullptr;  // optional: rows by descending chunk count (launch order)
  unsigned int* status;
};
cudaError_t launch_estimate_mass_k(const MassParams& p, cudaStream_t stream);
// rows (CSR offsets) by descending ceil(k / 128): a longest-first launch order
cudaError_t launch_csr_order(const int64_t* rowptr, int64_t rows, int64_t N, int32_t* order, cudaStream_t stream);

struct FwdParams {
  const bf16 *q, *k, *v;  // [BH][N][d]
  const int32_t* idx;     // [BH][NB][k]
  bf16* o;                // [BH][N][d]
  float* lse;             // [BH][N]
  int64_t BH, N, NB, topk;
  int d;
  float scale;
  unsigned int* status;
  const int64_t* rowptr = nullptr;  // CSR row offsets into idx (per-block k), or null: row * topk
  const int32_t* order = nullptr;   // optional launch order of the rows (CSR only)
};
cudaError_t launch_sparse_fwd_tc(const FwdParams& p, cudaStream_t stream);

// One wave of the backward: either whole heads [bh0, bh0 + nh) (blk0 = 0, nblk = NB)
// or the query blocks [blk0, blk0 + nblk) of the single head bh0 (nh = 1).
struct BwdWave {
  int64_t bh0, nh, blk0, nblk;
  bool first_of_head, last_of_head;  // for sub-head waves
};

struct BwdParams {
  const bf16 *d_o, *q, *k, *v, *o;
  const float* lse;
  const int32_t* idx;
  bf16 *dq, *dk, *dv;
  int64_t BH, N, NB, topk;
  int d;
  float scale;
  unsigned int* status;
  const int64_t* rowptr = nullptr;  // CSR row offsets into idx (per-block k), or null: row * topk
  const int32_t* order = nullptr;   // optional launch order of the rows (CSR, one wave over all heads)
  // workspace carve-out for one wave (sized for the largest wave)
  uint32_t* colbits;   // [nh][W32][N]   bit lb of word (lb / 32): block lb selected key j
  uint32_t* colpre;    // [nh][W32][N]   popcount of the words before
  uint32_t* count;     // [nh][N]
  int64_t* offsets;    // [nh][N]        first key-major position of key j (absolute within the wave)
  int64_t* tsum;       // [nh][N / 1024] sum of count over each 1024-key tile
  int32_t* lists;      // [pairs]        partial row of each key-major position: key j's rows in
                       //                ascending query-block order
  bf16* partial;       // [pairs][d]     BLOCK-major dK rows (CTA c's k rows at c k), times the
                       //                scale (bf16; summed in fp32); the 16-byte chunks of row n
                       //                are stored XOR (n & 7)
  bf16* partial_dv;    // [pairs][d]     the matching dV rows, laid out the same way
  float* acc;          // [N][2 d]       fp32 accumulator when a head spans several waves
  bool dense = false;       // k = N: the main kernel computes dQ only, no idx read, no partial rows
};
// Dense blocks (k = N): D_i = dO_i . O_i into delta [BH][N], then dK and dV of every key tile
// accumulated over all query blocks (dsv_dense_bwd.cu); dQ from launch_bwd_main_tc with dense set.
cudaError_t launch_dense_dkdv(const BwdParams& p, float* delta, cudaStream_t stream);
// parts: kBwdPrep (bitmaps, prefix, scan: reads idx only), kBwdFinish (main kernel and reduce on
// a workspace the prep filled), or both
constexpr int kBwdPrep = 1, kBwdFinish = 2, kBwdAll = 3;
cudaError_t launch_bwd_wave(const BwdParams& p, const BwdWave& w, cudaStream_t stream, int parts = kBwdAll);

// ---------------------------------------------------------------- fused AdaLN (adaln.cu)
struct AdalnParams {
  const void* x;         // bf16 [B][N][D]
  const void* scale;     // bf16 [B][D]
  const void* shift;     // bf16 [B][D] (forward)
  void* y;               // bf16 [B][N][D] (forward)
  const void* dy;        // bf16 [B][N][D] (backward)
  void* dx;              // bf16 [B][N][D] (backward)
  float* d_scale;        // fp32 [B][D] (backward)
  float* d_shift;        // fp32 [B][D] (backward)
  float* partial;        // backward workspace: fp32 [B * tiles][2][D] partials, fp32 [B * 8][2][D]
                         // group sums, u32 tickets (see adaln_tiling)
  int64_t B, N, D;
  float eps;
  unsigned int* status;  // device status word (timeout bit)
};
// Tokens per CTA tile: about this many tiles over all samples (three forward or two backward
// CTAs on each of the 152 SMs).
constexpr int64_t kAdalnFwdTiles = 3 * 152;
constexpr int64_t kAdalnBwdTiles = 2 * 152;
struct AdalnTiling {
  int64_t rows_per_tile, tiles_per_b;
  size_t partial_bytes, group_bytes, workspace_bytes;   // backward workspace layout
  int64_t tickets;
};
AdalnTiling adaln_tiling(int64_t B, int64_t N, int64_t D, bool backward);
cudaError_t launch_adaln_fwd(const AdalnParams& p, cudaStream_t stream);
cudaError_t launch_adaln_bwd(const AdalnParams& p, cudaStream_t stream);
cudaError_t launch_bwd_main_tc(const BwdParams& p, const BwdWave& w, int64_t W32, cudaStream_t stream);

}  // namespace dsv
