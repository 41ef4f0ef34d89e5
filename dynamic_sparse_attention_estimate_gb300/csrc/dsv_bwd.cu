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
//   4. main kernel: per query block, per 64-key chunk: recompute P from LSE, dP, dS,
//      dQ += dS K on the tensor cores; dV_part = P^T dO, dK_part = scale dS^T Q written
//      to row offsets[j] + colpre + popc(lower bits) -- the block's rank among the
//      blocks that selected j.
//   5. reduce: dK_j, dV_j = sum of key j's rows in order (fp32), written as bf16.
// A head whose partial rows do not fit in the workspace is split into several waves
// whose sums are chained through an fp32 accumulator.
#include "dsv_common.cuh"
#include "dsv_internal.h"

namespace dsv {
namespace {

constexpr int kChunk = 64;
constexpr int kThreads = 128;

// ---------------------------------------------------------------- 1. column bitmaps
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
scan_kernel(const uint32_t* __restrict__ count, int64_t* __restrict__ offsets, int64_t N, int64_t pairs_per_head) {
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
  int64_t run = hs * pairs_per_head + warp_sums[warp] + incl - s;
  for (int64_t i = lo; i < hi; ++i) {
    off[i] = run;
    run += c[i];
  }
}

// ---------------------------------------------------------------- 4. main kernel
template <int D>
struct BwdSmem {
  static constexpr int ROWB = D * 2;
  static constexpr int CH = ROWB / 16;
  static constexpr int T64 = 64 * ROWB;          // one 64-row tile of width D
  static constexpr int P_BYTES = 64 * 128;       // 64 x 64 bf16
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_DO = OFF_Q + T64;
  static constexpr int OFF_K = OFF_DO + T64;     // 2 stages
  static constexpr int OFF_V = OFF_K + 2 * T64;  // 2 stages
  static constexpr int OFF_P = OFF_V + 2 * T64;
  static constexpr int OFF_DS = OFF_P + P_BYTES;
  static constexpr int TOTAL = OFF_DS + P_BYTES;
};

template <int D>
__global__ void __launch_bounds__(kThreads)
sparse_bwd_main_kernel(BwdParams p, int64_t bh0, int64_t blk0, int64_t nblk, int64_t W32, float scale_log2) {
  using S = BwdSmem<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ int64_t s_pos[2][kChunk];
  __shared__ float s_lse[64];
  __shared__ float s_delta[64];
  const uint32_t base = smem_u32(smem);
  const uint32_t sQ = base + S::OFF_Q, sdO = base + S::OFF_DO;
  const uint32_t sK0 = base + S::OFF_K, sV0 = base + S::OFF_V;
  const uint32_t sP = base + S::OFF_P, sdS = base + S::OFF_DS;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int64_t N = p.N, NB = p.NB, kk = p.topk;
  const int64_t hs = blockIdx.x / nblk, lb = blockIdx.x % nblk;
  const int64_t bh = bh0 + hs, blk = blk0 + lb;
  const int64_t row0 = bh * N + blk * 64;
  const bf16* kh = p.k + bh * N * D;
  const bf16* vh = p.v + bh * N * D;
  const int32_t* ib = p.idx + (bh * NB + blk) * kk;
  const uint32_t* cbits = p.colbits + (hs * W32 + (lb >> 5)) * N;
  const uint32_t* cpre = p.colpre + (hs * W32 + (lb >> 5)) * N;
  const int64_t* offs = p.offsets + hs * N;
  const uint32_t lowmask = (1u << (lb & 31)) - 1u;
  const int nchunks = static_cast<int>((kk + kChunk - 1) / kChunk);

  for (int i = tid; i < 64 * S::CH; i += kThreads) {
    const int row = i / S::CH, ch = i % S::CH;
    cp_async_16(sQ + swz<S::ROWB>(row, ch), p.q + (row0 + row) * D + ch * 8, true);
    cp_async_16(sdO + swz<S::ROWB>(row, ch), p.d_o + (row0 + row) * D + ch * 8, true);
  }
  // D_i = dO_i . O_i (two threads per row), LSE in base 2
  {
    const int row = tid >> 1, half = tid & 1;
    const bf16* dor = p.d_o + (row0 + row) * D + half * (D / 2);
    const bf16* orow = p.o + (row0 + row) * D + half * (D / 2);
    float acc = 0.f;
    for (int c = 0; c < D / 2; c += 8) {
      const uint4 a = *reinterpret_cast<const uint4*>(dor + c);
      const uint4 b = *reinterpret_cast<const uint4*>(orow + c);
      const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) acc += bf16_lo(av[u]) * bf16_lo(bv[u]) + bf16_hi(av[u]) * bf16_hi(bv[u]);
    }
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    if (half == 0) {
      s_delta[row] = acc;
      s_lse[row] = p.lse[row0 + row] * kLog2e;
    }
  }

  auto load_chunk = [&](int c, int stage) {
    const uint32_t sK = sK0 + stage * S::T64, sV = sV0 + stage * S::T64;
    for (int i = tid; i < kChunk * S::CH; i += kThreads) {
      const int row = i / S::CH, ch = i % S::CH;
      const int64_t slot = static_cast<int64_t>(c) * kChunk + row;
      const int64_t j = slot < kk ? static_cast<int64_t>(__ldg(ib + slot)) : -1;
      const bool ok = j >= 0 && j < N;
      if (ch == 0) {
        int64_t pos = -1;
        if (ok) pos = offs[j] + cpre[j] + __popc(cbits[j] & lowmask);
        else if (slot < kk) flag_status(p.status, kStatusBadIndex);
        s_pos[stage][row] = pos;
      }
      const int64_t src = ok ? j : 0;
      cp_async_16(sK + swz<S::ROWB>(row, ch), kh + src * D + ch * 8, ok);
      cp_async_16(sV + swz<S::ROWB>(row, ch), vh + src * D + ch * 8, ok);
    }
  };

  load_chunk(0, 0);
  cp_async_commit();

  float dq[D / 8][4];
#pragma unroll
  for (int j = 0; j < D / 8; ++j) dq[j][0] = dq[j][1] = dq[j][2] = dq[j][3] = 0.f;

  for (int c = 0; c < nchunks; ++c) {
    const int stage = c & 1;
    if (c + 1 < nchunks) {
      load_chunk(c + 1, stage ^ 1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const uint32_t sK = sK0 + stage * S::T64, sV = sV0 + stage * S::T64;
    const int r_lo = warp * 16 + g, r_hi = r_lo + 8;

    // S = Q K^T and dP = dO V^T (16 x 64 per warp)
    float s[8][4], dp[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
      dp[j][0] = dp[j][1] = dp[j][2] = dp[j][3] = 0.f;
    }
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      uint32_t qa[4], da[4];
      ldsm_x4(sQ + swz<S::ROWB>(warp * 16 + (lane & 15), ks * 2 + (lane >> 4)), qa[0], qa[1], qa[2], qa[3]);
      ldsm_x4(sdO + swz<S::ROWB>(warp * 16 + (lane & 15), ks * 2 + (lane >> 4)), da[0], da[1], da[2], da[3]);
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t b0, b1, b2, b3;
        const int krow = np * 16 + (lane & 7) + 8 * (lane >> 4), kch = ks * 2 + ((lane >> 3) & 1);
        ldsm_x4(sK + swz<S::ROWB>(krow, kch), b0, b1, b2, b3);
        mma_bf16_16816(s[2 * np], qa, b0, b1);
        mma_bf16_16816(s[2 * np + 1], qa, b2, b3);
        ldsm_x4(sV + swz<S::ROWB>(krow, kch), b0, b1, b2, b3);
        mma_bf16_16816(dp[2 * np], da, b0, b1);
        mma_bf16_16816(dp[2 * np + 1], da, b2, b3);
      }
    }
    // P = exp2(S scale log2e - LSE2), dS = P (dP - D); masked slots give 0
    const float lse_lo = s_lse[r_lo], lse_hi = s_lse[r_hi];
    const float del_lo = s_delta[r_lo], del_hi = s_delta[r_hi];
    uint32_t dsf[4][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float pv[4], dsv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int col = 8 * j + 2 * t + (e & 1);
        const bool ok = s_pos[stage][col] >= 0;
        const float pe = ok ? fast_exp2(s[j][e] * scale_log2 - ((e >> 1) ? lse_hi : lse_lo)) : 0.f;
        pv[e] = pe;
        dsv[e] = pe * (dp[j][e] - ((e >> 1) ? del_hi : del_lo));
      }
      const uint32_t p01 = pack_bf16x2(pv[0], pv[1]), p23 = pack_bf16x2(pv[2], pv[3]);
      const uint32_t d01 = pack_bf16x2(dsv[0], dsv[1]), d23 = pack_bf16x2(dsv[2], dsv[3]);
      dsf[j >> 1][(j & 1) * 2 + 0] = d01;
      dsf[j >> 1][(j & 1) * 2 + 1] = d23;
      // P and dS tiles [query][key] for the key-side products
      asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(sP + swz<128>(r_lo, j) + 4 * t), "r"(p01));
      asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(sP + swz<128>(r_hi, j) + 4 * t), "r"(p23));
      asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(sdS + swz<128>(r_lo, j) + 4 * t), "r"(d01));
      asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(sdS + swz<128>(r_hi, j) + 4 * t), "r"(d23));
    }
    // dQ += dS K   (scale applied at the end)
#pragma unroll
    for (int kp = 0; kp < 4; ++kp) {
#pragma unroll
      for (int dn = 0; dn < D / 16; ++dn) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(sK + swz<S::ROWB>(kp * 16 + (lane & 7) + 8 * ((lane >> 3) & 1), dn * 2 + (lane >> 4)), b0, b1, b2,
                  b3);
        mma_bf16_16816(dq[2 * dn], dsf[kp], b0, b1);
        mma_bf16_16816(dq[2 * dn + 1], dsf[kp], b2, b3);
      }
    }
    __syncthreads();
    // key-side partials for keys [16 warp, 16 warp + 16): dV = P^T dO, dK = scale dS^T Q
    const int64_t pos_lo = s_pos[stage][warp * 16 + g], pos_hi = s_pos[stage][warp * 16 + g + 8];
#pragma unroll
    for (int which = 0; which < 2; ++which) {
      const uint32_t sA = which ? sP : sdS;    // which = 0: dK from dS and Q; 1: dV from P and dO
      const uint32_t sB = which ? sdO : sQ;
      const float mult = which ? 1.f : p.scale;
      float part[D / 8][4];
#pragma unroll
      for (int j = 0; j < D / 8; ++j) part[j][0] = part[j][1] = part[j][2] = part[j][3] = 0.f;
#pragma unroll
      for (int kq = 0; kq < 4; ++kq) {
        uint32_t a[4];
        ldsm_x4_t(sA + swz<128>(kq * 16 + (lane & 7) + 8 * (lane >> 4), warp * 2 + ((lane >> 3) & 1)), a[0], a[1],
                  a[2], a[3]);
#pragma unroll
        for (int dn = 0; dn < D / 16; ++dn) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(sB + swz<S::ROWB>(kq * 16 + (lane & 7) + 8 * ((lane >> 3) & 1), dn * 2 + (lane >> 4)), b0, b1,
                    b2, b3);
          mma_bf16_16816(part[2 * dn], a, b0, b1);
          mma_bf16_16816(part[2 * dn + 1], a, b2, b3);
        }
      }
      float* dst_lo = pos_lo >= 0 ? p.partial + pos_lo * (2 * D) + which * D : nullptr;
      float* dst_hi = pos_hi >= 0 ? p.partial + pos_hi * (2 * D) + which * D : nullptr;
#pragma unroll
      for (int j = 0; j < D / 8; ++j) {
        const int col = 8 * j + 2 * t;
        if (dst_lo) *reinterpret_cast<float2*>(dst_lo + col) = make_float2(part[j][0] * mult, part[j][1] * mult);
        if (dst_hi) *reinterpret_cast<float2*>(dst_hi + col) = make_float2(part[j][2] * mult, part[j][3] * mult);
      }
    }
    __syncthreads();
  }
  // dQ = scale * acc
  bf16* dqb = p.dq + (row0 + warp * 16) * D;
#pragma unroll
  for (int j = 0; j < D / 8; ++j) {
    const int col = 8 * j + 2 * t;
    *reinterpret_cast<uint32_t*>(dqb + g * D + col) = pack_bf16x2(dq[j][0] * p.scale, dq[j][1] * p.scale);
    *reinterpret_cast<uint32_t*>(dqb + (g + 8) * D + col) = pack_bf16x2(dq[j][2] * p.scale, dq[j][3] * p.scale);
  }
}

// ---------------------------------------------------------------- 5. segmented reduction per key
// One warp per key; lane l owns columns [4 l, 4 l + 4) (and + 128 when 2 D = 256).
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
    const int64_t cnt = p.count[key];
    float4 acc[PER];
#pragma unroll
    for (int u = 0; u < PER; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (mode == 2 || mode == 3) {
#pragma unroll
      for (int u = 0; u < PER; ++u) acc[u] = *reinterpret_cast<const float4*>(p.acc + j * W + u * 128 + lane * 4);
    }
    for (int64_t r = 0; r < cnt; ++r) {
      const float* row = p.partial + (first + r) * W;
#pragma unroll
      for (int u = 0; u < PER; ++u) {
        const float4 x = *reinterpret_cast<const float4*>(row + u * 128 + lane * 4);
        acc[u].x += x.x; acc[u].y += x.y; acc[u].z += x.z; acc[u].w += x.w;
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
  const int64_t pairs = w.nh * w.nblk * p.topk;
  { ProfScope prof("bwd_set_bits", stream);
  set_bits_kernel<<<grid_for(pairs, 256), 256, 0, stream>>>(p.idx, p.colbits, N, p.NB, p.topk, w.bh0, w.blk0, w.nblk,
                                                             W32, pairs, p.status); }
  { ProfScope prof("bwd_colpre", stream);
  colpre_kernel<<<grid_for(w.nh * N, 256), 256, 0, stream>>>(p.colbits, p.colpre, p.count, N, W32, w.nh); }
  { ProfScope prof("bwd_scan", stream);
  scan_kernel<<<static_cast<unsigned>(w.nh), kScanThreads, 0, stream>>>(p.count, p.offsets, N, w.nblk * p.topk); }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  const int smem = BwdSmem<D>::TOTAL;
  e = cudaFuncSetAttribute(sparse_bwd_main_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  { ProfScope prof("bwd_main", stream);
  sparse_bwd_main_kernel<D><<<static_cast<unsigned>(w.nh * w.nblk), kThreads, smem, stream>>>(
      p, w.bh0, w.blk0, w.nblk, W32, p.scale * kLog2e); }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

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
