// Sparse attention backward (training needs it: DSV page 1, section 2A, stage 2).
//
// dQ is local to a query block; dK and dV of key j sum over every query block that
// selected j.  To stay deterministic without float atomics the per-(block, key)
// contributions are written as partial rows into the workspace (block-major: each query
// block's rows in its own chunk order), and a KEY-MAJOR list gives, for each key j, its
// rows in ascending query-block order, so the final reduction is a fixed-order segmented
// sum.  Per wave of query blocks:
//   1. colbits[w][j] bit b  <- block (32 w + b) selected key j   (shared-memory tiles)
//   2. colpre[w][j]         <- popcount of words before w; count[j] <- total
//   3. offsets[j]           <- exclusive scan of count (per head)
//   4. main kernel (dsv_bwd_tc.cu): per query block, per 128-key chunk, on the tcgen05
//      tensor cores: recompute P from LSE, dP, dS; dQ accumulated in tensor memory;
//      dV_part = P^T dO, dK_part = scale dS^T Q written as bf16 partial rows; the list
//      entry at offsets[j] + colpre + popc(lower bits) -- the block's rank among the
//      blocks that selected j -- is set to the row's index.
//   5. reduce: dK_j, dV_j = sum of key j's rows in list order (fp32), written as bf16.
// A head whose partial rows do not fit in the workspace is split into several waves
// whose sums are chained through an fp32 accumulator.
#include <climits>

#include "dsv_common.cuh"
#include "dsv_internal.h"

namespace dsv {
namespace {


// ---------------------------------------------------------------- 1. column bitmaps
// One CTA per (key tile, half of a 32-block word group, head slot) ORs each key's block bit into
// a shared-memory tile (16 bits per key, two keys per word) and then writes the tile out as its
// half-words of colbits.  Every word of the wave is written (zeros included): no clearing pass and
// no global atomics.  With fixed k, a first kernel records for every row where its keys cross each
// tile boundary (the selection writes rows strictly ascending), so a tile's CTA reads only its
// rows' runs in that tile; a row that is not strictly ascending is marked there, and the CTA
// filters all of that row's entries instead (the general method, which CSR rows always take: the
// half's 16 blocks are contiguous in idx, so the CTA walks that range flat).  A key outside
// [0, N) or a key twice in one row sets the bad-index status.
constexpr int kBitsThreads = 1024;
constexpr int64_t kBitsTile = 32768;  // keys per tile: 64 KB of shared memory

__device__ __forceinline__ void set_bit(uint32_t* tile, const int64_t* rp, int nrows, int64_t first, int64_t kk,
                                        bool csr, int64_t i, int32_t j, int64_t j0, int64_t tj, int64_t N,
                                        bool report_range, unsigned int* status) {
  if (j < 0 || j >= N) {
    if (report_range) flag_status(status, kStatusBadIndex);
    return;
  }
  const int64_t jj = j - j0;
  if (jj < 0 || jj >= tj) return;
  int r;
  if (csr) {  // largest r with rp[r] <= i
    int lo = 0, hi = nrows - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (rp[mid] <= i) lo = mid; else hi = mid - 1;
    }
    r = lo;
  } else {
    r = static_cast<int>(static_cast<uint32_t>(i - first) / static_cast<uint32_t>(kk));
  }
  const uint32_t bit = 1u << (r + 16 * static_cast<int>(jj & 1));
  const uint32_t old = atomicOr(tile + (jj >> 1), bit);
  if (old & bit) flag_status(status, kStatusBadIndex);  // duplicate key in one idx row
}

// Tile bounds of fixed-k rows: for row r of the wave (global row row0 + r) and tile t in [0, ntile],
// b[t] = the position of the row's first entry whose key is at least kBitsTile t (entries before
// b[0] have negative keys, entries from b[ntile] on keys past the last tile); b[ntile + 1] != 0
// when the row is not strictly ascending (the bounds then mean nothing).  Each entry is compared
// with the one before it: a boundary lies between two neighbouring entries, so every b[t] of an
// ascending row is written once.  The bounds are zeroed before.  A CTA covers kBoundsSpan entries
// of one row, a thread kBoundsPerThread of them.
constexpr int kBoundsThreads = 256;
constexpr int kBoundsPerThread = 8;
constexpr int kBoundsSpan = kBoundsThreads * kBoundsPerThread;
__global__ void __launch_bounds__(kBoundsThreads)
tile_bounds_kernel(const int32_t* __restrict__ idx, int32_t* __restrict__ bounds, int64_t kk, int64_t row0,
                   int64_t r0, int ntile) {
  const int64_t r = r0 + blockIdx.y;
  const int32_t* row = idx + (row0 + r) * kk;
  int32_t* b = bounds + r * (ntile + 2);
  auto tile_of = [&](int32_t key) -> int {
    return key < 0 ? -1 : ((key >> 15) < ntile ? (key >> 15) : ntile);  // kBitsTile = 2^15
  };
#pragma unroll
  for (int u = 0; u < kBoundsPerThread; ++u) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * kBoundsSpan + u * kBoundsThreads + threadIdx.x;
    if (i >= kk) break;
    const int32_t key = __ldg(row + i);
    const int32_t before = i > 0 ? __ldg(row + i - 1) : INT_MIN;
    const int pk = tile_of(key), pb = i > 0 ? tile_of(before) : -1;
    for (int t = pb + 1; t <= pk; ++t) b[t] = static_cast<int32_t>(i);
    if (i == kk - 1)
      for (int t = pk + 1; t <= ntile; ++t) b[t] = static_cast<int32_t>(kk);
    if (i > 0 && key <= before) b[ntile + 1] = 1;
  }
}
static_assert(kBitsTile == 32768, "tile_bounds_kernel divides keys by shifting");
// Below this many key tiles the general method reads each row only a few times: no bounds.
constexpr int kBoundsMinTiles = 8;

__global__ void __launch_bounds__(kBitsThreads)
set_bits_kernel(const int32_t* __restrict__ idx, const int64_t* __restrict__ rowptr, uint32_t* __restrict__ colbits,
                int64_t N, int64_t NB, int64_t kk, int64_t bh0, int64_t blk0, int64_t nblk, int64_t W32, int64_t hs0,
                const int32_t* __restrict__ bounds, int ntile, unsigned int* status) {
  extern __shared__ uint32_t tile[];  // word i: key 2 i in bits 0-15, key 2 i + 1 in bits 16-31
  __shared__ int64_t rp[17];
  __shared__ int32_t run0[16], runoff[17], irr[16];
  const int tid = threadIdx.x;
  const int64_t j0 = static_cast<int64_t>(blockIdx.x) * kBitsTile;
  const int64_t tj = N - j0 < kBitsTile ? N - j0 : kBitsTile;
  const int half = blockIdx.y & 1;
  const int64_t wg = blockIdx.y >> 1;
  const int64_t hs = hs0 + blockIdx.z;
  const int64_t lb0 = wg * 32 + half * 16;
  const int nrows = nblk - lb0 <= 0 ? 0 : (nblk - lb0 < 16 ? static_cast<int>(nblk - lb0) : 16);
  const int64_t g0 = (bh0 + hs) * NB + blk0 + lb0;  // global row of the half's first block
  for (int64_t i = tid; i < (tj + 1) / 2; i += kBitsThreads) tile[i] = 0;
  if (nrows > 0 && tid <= nrows) rp[tid] = rowptr ? rowptr[g0 + tid] : (g0 + tid) * kk;
  const int tt = static_cast<int>(blockIdx.x);
  if (bounds && tid < 16) {
    int32_t lo = 0, hi = 0, ir = 0;
    if (tid < nrows) {
      const int32_t* b = bounds + (hs * nblk + lb0 + tid) * (ntile + 2);
      lo = b[tt];
      hi = b[tt + 1];
      ir = b[ntile + 1];
      if (!ir && ((tt == 0 && b[0] > 0) || (tt == ntile - 1 && b[ntile] < kk)))
        flag_status(status, kStatusBadIndex);  // keys below 0 or past the last tile
      if (ir || hi < lo) lo = hi = 0;
    }
    run0[tid] = lo;
    runoff[tid] = hi - lo;  // length for now; the prefix below
    irr[tid] = ir;
  }
  __syncthreads();
  if (bounds && tid == 0) {
    int32_t acc = 0;
    for (int r = 0; r < 16; ++r) {
      const int32_t len = runoff[r];
      runoff[r] = acc;
      acc += len;
    }
    runoff[16] = acc;
  }
  __syncthreads();
  const bool csr = rowptr != nullptr;
  const bool report = blockIdx.x == 0;  // range errors are reported by the first key tile only
  if (bounds) {
    // every ascending row's run in this tile, as one flat range
    const int32_t total = runoff[16];
    int r = 0;  // the row of entry e: e only grows, so r is carried from one entry to the next
    for (int32_t e = tid; e < total; e += kBitsThreads) {
      while (r < 15 && runoff[r + 1] <= e) ++r;
      const int32_t key = __ldg(idx + rp[r] + run0[r] + (e - runoff[r]));
      const int64_t jj = static_cast<int64_t>(key) - j0;
      if (key >= N || jj < 0 || jj >= tj) {
        flag_status(status, kStatusBadIndex);  // past N inside the last tile
        continue;
      }
      const uint32_t bit = 1u << (r + 16 * static_cast<int>(jj & 1));
      if (atomicOr(tile + (jj >> 1), bit) & bit) flag_status(status, kStatusBadIndex);
    }
    // rows not strictly ascending: the general method, their entries filtered
    for (int r = 0; r < nrows; ++r)
      if (irr[r])
        for (int64_t i = rp[r] + tid; i < rp[r + 1]; i += kBitsThreads)
          set_bit(tile, rp, nrows, rp[0], kk, false, i, __ldg(idx + i), j0, tj, N, report, status);
  } else if (nrows > 0) {
    const int64_t first = rp[0], last = rp[nrows];
    // scalar head and tail, 16-byte loads in between
    const int64_t a0 = ((first + 3) & ~int64_t(3)) < last ? ((first + 3) & ~int64_t(3)) : last;
    const int64_t a1 = (last & ~int64_t(3)) > a0 ? (last & ~int64_t(3)) : a0;
    for (int64_t i = first + tid; i < a0; i += kBitsThreads)
      set_bit(tile, rp, nrows, first, kk, csr, i, __ldg(idx + i), j0, tj, N, report, status);
    for (int64_t i = a1 + tid; i < last; i += kBitsThreads)
      set_bit(tile, rp, nrows, first, kk, csr, i, __ldg(idx + i), j0, tj, N, report, status);
    const int4* v4 = reinterpret_cast<const int4*>(idx + a0);
    const int64_t n4 = (a1 - a0) >> 2;
    for (int64_t q = tid; q < n4; q += 2 * kBitsThreads) {
      const bool two = q + kBitsThreads < n4;
      const int4 x = __ldg(v4 + q);
      const int4 y = two ? __ldg(v4 + q + kBitsThreads) : make_int4(0, 0, 0, 0);
      const int64_t i = a0 + 4 * q, i2 = i + 4 * kBitsThreads;
      set_bit(tile, rp, nrows, first, kk, csr, i, x.x, j0, tj, N, report, status);
      set_bit(tile, rp, nrows, first, kk, csr, i + 1, x.y, j0, tj, N, report, status);
      set_bit(tile, rp, nrows, first, kk, csr, i + 2, x.z, j0, tj, N, report, status);
      set_bit(tile, rp, nrows, first, kk, csr, i + 3, x.w, j0, tj, N, report, status);
      if (two) {
        set_bit(tile, rp, nrows, first, kk, csr, i2, y.x, j0, tj, N, report, status);
        set_bit(tile, rp, nrows, first, kk, csr, i2 + 1, y.y, j0, tj, N, report, status);
        set_bit(tile, rp, nrows, first, kk, csr, i2 + 2, y.z, j0, tj, N, report, status);
        set_bit(tile, rp, nrows, first, kk, csr, i2 + 3, y.w, j0, tj, N, report, status);
      }
    }
  }
  __syncthreads();
  // bits 16 h .. 16 h + 15 of word j are the half-word at byte 2 h (little-endian)
  uint16_t* out = reinterpret_cast<uint16_t*>(colbits + (hs * W32 + wg) * N + j0) + half;
  for (int64_t i = tid; i < tj; i += kBitsThreads)
    out[2 * i] = static_cast<uint16_t>(tile[i >> 1] >> (16 * static_cast<int>(i & 1)));
}

// ---------------------------------------------------------------- 2. per-key word prefix
// One thread per key, 1024 keys per CTA: colpre[w][j] = popcount of the words before w,
// count[j] = the total, and the tile's sum of counts for the scan.
constexpr int kScanThreads = 1024;
__global__ void __launch_bounds__(kScanThreads)
colpre_kernel(const uint32_t* __restrict__ colbits, uint32_t* __restrict__ colpre, uint32_t* __restrict__ count,
              int64_t* __restrict__ tsum, int64_t N, int64_t W32, int64_t hs0) {
  __shared__ uint32_t warp_tot[kScanThreads / 32];
  const int64_t hs = hs0 + blockIdx.y;
  const int64_t j = static_cast<int64_t>(blockIdx.x) * kScanThreads + threadIdx.x;
  uint32_t run = 0;
  if (j < N) {
    for (int64_t w = 0; w < W32; ++w) {
      const int64_t a = (hs * W32 + w) * N + j;
      colpre[a] = run;
      run += __popc(colbits[a]);
    }
    count[hs * N + j] = run;
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t t = run;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  if (lane == 0) warp_tot[warp] = t;
  __syncthreads();
  if (warp == 0) {
    uint32_t u = warp_tot[lane];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) u += __shfl_xor_sync(0xffffffffu, u, o);
    if (lane == 0) tsum[hs * gridDim.x + blockIdx.x] = u;
  }
}

// ---------------------------------------------------------------- 3. exclusive scan per head slot
// One thread per key, 1024 keys per CTA: the tile's exclusive scan plus the sum of the
// earlier tiles of the same head slot plus the head slot's first key-major position.
__global__ void __launch_bounds__(kScanThreads)
scan_kernel(const uint32_t* __restrict__ count, const int64_t* __restrict__ tsum, int64_t* __restrict__ offsets,
            int64_t N, int64_t pairs_per_head, const int64_t* __restrict__ rowptr, int64_t NB, int64_t bh0,
            int64_t blk0, int64_t hs0) {
  __shared__ int64_t warp_sums[kScanThreads / 32];
  __shared__ int64_t tile_base;
  const int64_t hs = hs0 + blockIdx.y;
  const int64_t j = static_cast<int64_t>(blockIdx.x) * kScanThreads + threadIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t c = j < N ? count[hs * N + j] : 0;
  int64_t incl = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sums[warp] = incl;
  if (warp == 1) {  // sum of the earlier tiles, plus where this head slot starts
    int64_t b = 0;
    for (int64_t t = lane; t < blockIdx.x; t += 32) b += tsum[hs * gridDim.x + t];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) b += __shfl_xor_sync(0xffffffffu, b, o);
    if (lane == 0)
      tile_base = b + (rowptr ? rowptr[(bh0 + hs) * NB + blk0] - rowptr[bh0 * NB + blk0] : hs * pairs_per_head);
  }
  __syncthreads();
  if (warp == 0) {
    const int64_t ws = warp_sums[lane];
    int64_t wi = ws;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t v = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += v;
    }
    warp_sums[lane] = wi - ws;
  }
  __syncthreads();
  if (j < N) offsets[hs * N + j] = tile_base + warp_sums[warp] + incl - c;
}

// ---------------------------------------------------------------- 4. main kernel: dsv_bwd_tc.cu

// ---------------------------------------------------------------- 5. segmented reduction per key
// One warp per key; lane l owns columns [4 l, 4 l + 4) (and + 128 when 2 D = 256).  The key's
// partial rows are gathered through its list (ascending query block: a fixed order), eight
// rows in flight; a row is its dK half (columns [0, D)) and its dV half (columns [D, 2 D)), in
// two arrays, each half's 16-byte chunks XOR (row & 7).
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
      const bf16* half = e < D ? p.partial : p.partial_dv;
      e = e < D ? e : e - D;
      e = ((((e >> 3) ^ (row & 7)) << 3) | (e & 7));
      return reinterpret_cast<const uint2*>(half + static_cast<int64_t>(row) * D + e);
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

// Steps 1-3 (the key-major rank structure): they read only idx (and rowptr), so they may run
// as soon as the selection exists, e.g. beside the forward on another stream.
cudaError_t launch_wave_prep(const BwdParams& p, const BwdWave& w, cudaStream_t stream) {
  const int64_t W32 = (w.nblk + 31) / 32;
  const int64_t N = p.N;
  const int64_t ntile = (N + kBitsTile - 1) / kBitsTile;
  const int64_t nscan = (N + kScanThreads - 1) / kScanThreads;
  const size_t bits_smem = sizeof(uint32_t) * static_cast<size_t>(((N < kBitsTile ? N : kBitsTile) + 1) / 2);
  cudaError_t e = cudaFuncSetAttribute(set_bits_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(bits_smem));
  if (e != cudaSuccess) return e;
  // fixed k over many key tiles: tile bounds of every row of the wave, in the offsets array (written
  // only later, by the scan); with few tiles (each row then read only a few times), CSR rows, or
  // bounds that would not fit there, the general method
  const int nt = static_cast<int>(ntile);
  const int64_t rows = w.nh * w.nblk;
  const size_t bounds_bytes = sizeof(int32_t) * static_cast<size_t>(rows) * static_cast<size_t>(nt + 2);
  const int32_t* bounds = nullptr;
  if (nt >= kBoundsMinTiles && !p.rowptr && p.topk >= 1 && bounds_bytes <= sizeof(int64_t) * static_cast<size_t>(w.nh * N)) {
    int32_t* bw = reinterpret_cast<int32_t*>(p.offsets);
    if ((e = cudaMemsetAsync(bw, 0, bounds_bytes, stream)) != cudaSuccess) return e;
    ProfScope prof("bwd_tile_bounds", stream);
    for (int64_t r0 = 0; r0 < rows; r0 += 65535) {
      const unsigned nr = static_cast<unsigned>(rows - r0 < 65535 ? rows - r0 : 65535);
      tile_bounds_kernel<<<dim3(static_cast<unsigned>((p.topk + kBoundsSpan - 1) / kBoundsSpan), nr),
                           kBoundsThreads, 0, stream>>>(p.idx, bw, p.topk, w.bh0 * p.NB + w.blk0, r0, nt);
    }
    bounds = bw;
  }
  for (int64_t hs0 = 0; hs0 < w.nh; hs0 += 65535) {  // grid y / z limit
    const unsigned nh = static_cast<unsigned>(w.nh - hs0 < 65535 ? w.nh - hs0 : 65535);
    { ProfScope prof("bwd_set_bits", stream);
    set_bits_kernel<<<dim3(static_cast<unsigned>(ntile), static_cast<unsigned>(2 * W32), nh), kBitsThreads,
                      bits_smem, stream>>>(p.idx, p.rowptr, p.colbits, N, p.NB, p.topk, w.bh0, w.blk0, w.nblk, W32,
                                           hs0, bounds, nt, p.status); }
    { ProfScope prof("bwd_colpre", stream);
    colpre_kernel<<<dim3(static_cast<unsigned>(nscan), nh), kScanThreads, 0, stream>>>(
        p.colbits, p.colpre, p.count, p.tsum, N, W32, hs0); }
    { ProfScope prof("bwd_scan", stream);
    scan_kernel<<<dim3(static_cast<unsigned>(nscan), nh), kScanThreads, 0, stream>>>(
        p.count, p.tsum, p.offsets, N, w.nblk * p.topk, p.rowptr, p.NB, w.bh0, w.blk0, hs0); }
  }
  return cudaGetLastError();
}

// Steps 4-5 on a prepared workspace.
template <int D>
cudaError_t launch_wave_finish(const BwdParams& p, const BwdWave& w, cudaStream_t stream) {
  const int64_t W32 = (w.nblk + 31) / 32;
  const int64_t N = p.N;
  cudaError_t e;
  if ((e = launch_bwd_main_tc(p, w, W32, stream)) != cudaSuccess) return e;

  int mode = 0;
  if (w.nblk != p.NB) mode = w.first_of_head ? (w.last_of_head ? 0 : 1) : (w.last_of_head ? 3 : 2);
  { ProfScope prof("bwd_reduce", stream);
  reduce_kernel<D><<<grid_for(w.nh * N * 32, 256, 152 * 64), 256, 0, stream>>>(p, w.bh0, w.nh, mode); }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_wave(const BwdParams& p, const BwdWave& w, cudaStream_t stream, int parts) {
  if (p.d != 64 && p.d != 128) return cudaErrorInvalidValue;
  cudaError_t e;
  if ((parts & kBwdPrep) && (e = launch_wave_prep(p, w, stream)) != cudaSuccess) return e;
  if (parts & kBwdFinish) return p.d == 64 ? launch_wave_finish<64>(p, w, stream) : launch_wave_finish<128>(p, w, stream);
  return cudaSuccess;
}

}  // namespace dsv
