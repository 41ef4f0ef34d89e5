// Sparse attention backward (training needs it: DSV page 1, section 2A, stage 2).
//
// dQ is local to a query block; dK and dV of key j sum over every query block that
// selected j.  To stay deterministic without float atomics the per-(block, key)
// contributions are written as partial rows into the workspace, laid out KEY-MAJOR:
// key j's rows are contiguous and ordered by ascending query block, so the final
// reduction is a fixed-order segmented sum.  Per wave of query blocks:
//   1. colbits[w][j] bit b  <- block (32 w + b) selected key j      (integer atomicOr)
//   2. colpre[w][j]         <- popcount of words before w; count[j] <- total
//   3. offsets[j]           <- exclusive scan of count (per head)
//   4. main kernel (dsv_bwd_tc.cu): per query block, per 128-key chunk, on the tcgen05
//      tensor cores: recompute P from LSE, dP, dS; dQ accumulated in tensor memory;
//      dV_part = P^T dO, dK_part = scale dS^T Q written as bf16 to row offsets[j] + colpre
//      + popc(lower bits) -- the block's rank among the blocks that selected j.
//   5. reduce: dK_j, dV_j = sum of key j's rows in order (fp32), written as bf16.
// A head whose partial rows do not fit in the workspace is split into several waves
// whose sums are chained through an fp32 accumulator.
#include "dsv_common.cuh"
#include "dsv_internal.h"

namespace dsv {
namespace {


// ---------------------------------------------------------------- 1. column bitmaps
// k keys per block: one thread per (block, key) pair of the wave.
__global__ void set_bits_kernel(const int32_t* __restrict__ idx, uint32_t* __restrict__ colbits, int64_t N,
                                int64_t NB, int64_t kk, int64_t bh0, int64_t blk0, int64_t nblk, int64_t W32,
                                int64_t total, unsigned int* status) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t slot = i % kk;
    const int64_t lbh = i / kk;            // (head slot, local block)
    const int64_t hs = lbh / nblk, lb = lbh % nblk;
    const int64_t j = __ldg(idx + ((bh0 + hs) * NB + blk0 + lb) * kk + slot);
    if (j < 0 || j >= N) { flag_status(status, kStatusBadIndex); continue; }
    const uint32_t bit = 1u << (lb & 31);
    const uint32_t old = atomicOr(colbits + (hs * W32 + (lb >> 5)) * N + j, bit);
    if (old & bit) flag_status(status, kStatusBadIndex);  // duplicate key in one idx row
  }
}

// CSR rows: one warp per query block of the wave, over that block's key range.
__global__ void set_bits_csr_kernel(const int32_t* __restrict__ idx, const int64_t* __restrict__ rowptr,
                                uint32_t* __restrict__ colbits, int64_t N, int64_t NB, int64_t kk, int64_t bh0,
                                int64_t blk0, int64_t nblk, int64_t W32, int64_t rows, unsigned int* status) {
  const int lane = threadIdx.x & 31;
  for (int64_t r = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5; r < rows;
       r += (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5) {
    const int64_t hs = r / nblk, lb = r % nblk;
    const int64_t grow = (bh0 + hs) * NB + blk0 + lb;
    const int64_t first = rowptr ? rowptr[grow] : grow * kk;
    const int64_t last = rowptr ? rowptr[grow + 1] : first + kk;
    const uint32_t bit = 1u << (lb & 31);
    uint32_t* col = colbits + (hs * W32 + (lb >> 5)) * N;
    for (int64_t i = first + lane; i < last; i += 32) {
      const int64_t j = __ldg(idx + i);
      if (j < 0 || j >= N) { flag_status(status, kStatusBadIndex); continue; }
      const uint32_t old = atomicOr(col + j, bit);
      if (old & bit) flag_status(status, kStatusBadIndex);  // duplicate key in one idx row
    }
  }
}

// ---------------------------------------------------------------- 2. per-key word prefix
__global__ void colpre_kernel(const uint32_t* __restrict__ colbits, uint32_t* __restrict__ colpre,
                              uint32_t* __restrict__ count, int64_t N, int64_t W32, int64_t nh) {
  const int64_t total = nh * N;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t hs = i / N, j = i % N;
    uint32_t run = 0;
    for (int64_t w = 0; w < W32; ++w) {
      const int64_t a = (hs * W32 + w) * N + j;
      colpre[a] = run;
      run += __popc(colbits[a]);
    }
    count[i] = run;
  }
}

// ---------------------------------------------------------------- 3. exclusive scan per head slot
constexpr int kScanThreads = 1024;
__global__ void __launch_bounds__(kScanThreads)
scan_kernel(const uint32_t* __restrict__ count, int64_t* __restrict__ offsets, int64_t N, int64_t pairs_per_head,
            const int64_t* __restrict__ rowptr, int64_t NB, int64_t bh0, int64_t blk0) {
  __shared__ int64_t warp_sums[kScanThreads / 32];
  const int64_t hs = blockIdx.x;
  const uint32_t* c = count + hs * N;
  int64_t* off = offsets + hs * N;
  const int64_t per = (N + kScanThreads - 1) / kScanThreads;
  const int64_t lo_raw = static_cast<int64_t>(threadIdx.x) * per;
  const int64_t lo = lo_raw < N ? lo_raw : N, hi = lo + per < N ? lo + per : N;
  int64_t s = 0;
  for (int64_t i = lo; i < hi; ++i) s += c[i];
  // block-wide exclusive scan of s
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int64_t incl = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int64_t ws = warp_sums[lane];
    int64_t wi = ws;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t v = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += v;
    }
    warp_sums[lane] = wi - ws;
  }
  __syncthreads();
  // first key-major position of this head slot: its blocks' pairs come after the earlier slots'
  const int64_t base = rowptr ? rowptr[(bh0 + hs) * NB + blk0] - rowptr[bh0 * NB + blk0] : hs * pairs_per_head;
  int64_t run = base + warp_sums[warp] + incl - s;
  for (int64_t i = lo; i < hi; ++i) {
    off[i] = run;
    run += c[i];
  }
}

// ---------------------------------------------------------------- 4. main kernel: dsv_bwd_tc.cu

// ---------------------------------------------------------------- 5. segmented reduction per key
// One warp per key; lane l owns columns [4 l, 4 l + 4) (and + 128 when 2 D = 256).  The key's
// partial rows are gathered through its list (ascending query block: a fixed order), eight
// rows in flight; at d = 64 the row's 16-byte chunks sit XOR (row & 7).
template <int D>
__global__ void reduce_kernel(BwdParams p, int64_t bh0, int64_t nh, int mode /*0: write, 1: first, 2: middle, 3: last*/) {
  constexpr int W = 2 * D;       // columns per partial row
  constexpr int PER = W / 128;   // float4 per lane
  const int64_t N = p.N;
  const int lane = threadIdx.x & 31;
  const int64_t total = nh * N;
  for (int64_t key = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5; key < total;
       key += (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5) {
    const int64_t hs = key / N, j = key % N;
    const int64_t first = p.offsets[key];
    const int cnt = static_cast<int>(p.count[key]);
    float4 acc[PER];
#pragma unroll
    for (int u = 0; u < PER; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (mode == 2 || mode == 3) {
#pragma unroll
      for (int u = 0; u < PER; ++u) acc[u] = *reinterpret_cast<const float4*>(p.acc + j * W + u * 128 + lane * 4);
    }
    auto row_ptr = [&](int32_t row, int u) -> const uint2* {
      // element offset of this lane's 4 columns [u 128 + 4 lane, + 4) within partial row `row`
      int e = u * 128 + lane * 4;
      if (D == 64) e = ((((e >> 3) ^ (row & 7)) << 3) | (e & 7));
      return reinterpret_cast<const uint2*>(p.partial + static_cast<int64_t>(row) * W + e);
    };
    for (int r0 = 0; r0 < cnt; r0 += 32) {
      const int32_t mine = r0 + lane < cnt ? p.lists[first + r0 + lane] : 0;
      const int n = cnt - r0 < 32 ? cnt - r0 : 32;
      int i = 0;
      constexpr int kBatch = 8;  // rows in flight per warp
      for (; i + kBatch <= n; i += kBatch) {
        uint2 x[kBatch][PER];
#pragma unroll
        for (int q = 0; q < kBatch; ++q) {
          const int32_t row = __shfl_sync(0xffffffffu, mine, i + q);
#pragma unroll
          for (int u = 0; u < PER; ++u) x[q][u] = *row_ptr(row, u);
        }
#pragma unroll
        for (int q = 0; q < kBatch; ++q)
#pragma unroll
          for (int u = 0; u < PER; ++u) {
            acc[u].x += bf16_lo(x[q][u].x); acc[u].y += bf16_hi(x[q][u].x);
            acc[u].z += bf16_lo(x[q][u].y); acc[u].w += bf16_hi(x[q][u].y);
          }
      }
      for (; i < n; ++i) {
        const int32_t row = __shfl_sync(0xffffffffu, mine, i);
#pragma unroll
        for (int u = 0; u < PER; ++u) {
          const uint2 x = *row_ptr(row, u);
          acc[u].x += bf16_lo(x.x); acc[u].y += bf16_hi(x.x); acc[u].z += bf16_lo(x.y); acc[u].w += bf16_hi(x.y);
        }
      }
    }
    if (mode == 1 || mode == 2) {
#pragma unroll
      for (int u = 0; u < PER; ++u) *reinterpret_cast<float4*>(p.acc + j * W + u * 128 + lane * 4) = acc[u];
    } else {
      const int64_t bh = bh0 + hs;
#pragma unroll
      for (int u = 0; u < PER; ++u) {
        const int col = u * 128 + lane * 4;   // [0, D): dK, [D, 2D): dV
        bf16* dst = col < D ? p.dk + (bh * N + j) * D + col : p.dv + (bh * N + j) * D + (col - D);
        uint2 v;
        v.x = pack_bf16x2(acc[u].x, acc[u].y);
        v.y = pack_bf16x2(acc[u].z, acc[u].w);
        *reinterpret_cast<uint2*>(dst) = v;
      }
    }
  }
}

inline unsigned grid_for(int64_t work, int threads, int64_t cap = 152 * 16) {
  int64_t b = (work + threads - 1) / threads;
  if (b < 1) b = 1;
  if (b > cap) b = cap;
  return static_cast<unsigned>(b);
}

template <int D>
cudaError_t launch_wave_d(const BwdParams& p, const BwdWave& w, cudaStream_t stream) {
  const int64_t W32 = (w.nblk + 31) / 32;
  const int64_t N = p.N;
  cudaError_t e = cudaMemsetAsync(p.colbits, 0, sizeof(uint32_t) * w.nh * W32 * N, stream);
  if (e != cudaSuccess) return e;
  const int64_t rows = w.nh * w.nblk;
  { ProfScope prof("bwd_set_bits", stream);
  if (p.rowptr) {
    set_bits_csr_kernel<<<grid_for(rows * 32, 256), 256, 0, stream>>>(p.idx, p.rowptr, p.colbits, N, p.NB, p.topk,
                                                                       w.bh0, w.blk0, w.nblk, W32, rows, p.status);
  } else {
    const int64_t pairs = rows * p.topk;
    set_bits_kernel<<<grid_for(pairs, 256), 256, 0, stream>>>(p.idx, p.colbits, N, p.NB, p.topk, w.bh0, w.blk0,
                                                               w.nblk, W32, pairs, p.status);
  } }
  { ProfScope prof("bwd_colpre", stream);
  colpre_kernel<<<grid_for(w.nh * N, 256), 256, 0, stream>>>(p.colbits, p.colpre, p.count, N, W32, w.nh); }
  { ProfScope prof("bwd_scan", stream);
  scan_kernel<<<static_cast<unsigned>(w.nh), kScanThreads, 0, stream>>>(p.count, p.offsets, N, w.nblk * p.topk,
                                                                          p.rowptr, p.NB, w.bh0, w.blk0); }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  if ((e = launch_bwd_main_tc(p, w, W32, stream)) != cudaSuccess) return e;

  int mode = 0;
  if (w.nblk != p.NB) mode = w.first_of_head ? (w.last_of_head ? 0 : 1) : (w.last_of_head ? 3 : 2);
  { ProfScope prof("bwd_reduce", stream);
  reduce_kernel<D><<<grid_for(w.nh * N * 32, 256, 152 * 64), 256, 0, stream>>>(p, w.bh0, w.nh, mode); }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_wave(const BwdParams& p, const BwdWave& w, cudaStream_t stream) {
  switch (p.d) {
    case 64: return launch_wave_d<64>(p, w, stream);
    case 128: return launch_wave_d<128>(p, w, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dsv
