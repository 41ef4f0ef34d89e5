// Fused low-rank estimate + exact top-k per query block (DSV technical summary,
// section 2B "Fused MM & Top-K" with "Query Grouping").
//
// One CTA owns 16 query blocks of one head (the M = 16 rows of an m16n8k16 MMA) and
// streams every key of that head.  Scores s[b, j] = q_hat[b] . K_lr[j] live only in
// registers: they are recomputed on each pass and never written anywhere.
//
// Selection is an exact radix select on the order-preserving 32-bit image of the
// fp32 score, per query block, in shared-memory histograms:
//   pass 1: 2048-bin histogram of bits [31:21] -> threshold bin, count above it;
//   pass 2: 2048-bin histogram of bits [20:10] among pass-1 bin members; if all of
//           them have zero bits [9:0] (every integer score below 2^14 does), the
//           threshold value is now exact;
//   pass 3 (only if needed): 1024-bin histogram of bits [9:0];
//   emit:   keys in ascending order, all with key > T and the first n_tie with key == T
//           (ties to the lower key index), written ascending with a CTA-wide prefix.
// q_hat is held as hi + lo bf16 (an exact split for |q_hat| < 2^16), so with
// integer-valued factors every fp32 score is the exact integer.
#include "dsv_common.cuh"
#include "dsv_internal.h"

namespace dsv {
namespace {

constexpr int kRows = 16;                       // query blocks per CTA
constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kTileKeys = kWarps * 32;          // keys per CTA-wide tile (32 per warp)
constexpr int kBins = 2048;
constexpr int kTieAll = 0x7fffffff;

struct RowState {
  uint32_t prefix;  // resolved high bits of the threshold
  int level;        // 0/1/2: pass (level + 1) pending; 3: resolved
  int rem;          // elements still to take inside the current prefix
  uint32_t T;       // threshold key (resolved)
  int n_tie;        // elements equal to T to take, lowest key first
  uint32_t orbits;  // OR of bits [9:0] over pass-1 bin members
  int out_pos;      // emit: elements written so far
  int tie_seen;     // emit: elements equal to T seen so far
};

DSV_DEVICE uint32_t order_key(float s) {
  s = __fadd_rn(s, 0.0f);  // -0 -> +0 so that equal scores get equal keys
  uint32_t u = __float_as_uint(s);
  return u ^ (static_cast<uint32_t>(static_cast<int32_t>(u) >> 31) | 0x80000000u);
}

// Warp-cooperative search over a histogram from the top bin down: the bin where the
// running count first reaches `need`, the count strictly above it and its own count.
DSV_DEVICE void warp_find_bin(const uint32_t* h, int nbins, int need, int lane, int& bin, int& above, int& cnt) {
  const int per = nbins / 32;
  const int hi = nbins - lane * per;  // this lane's bins: [hi - per, hi)
  int s = 0;
  for (int i = 0; i < per; ++i) s += h[hi - 1 - ((i + lane) % per)];  // staggered: no bank conflicts
  int incl = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  const unsigned m = __ballot_sync(0xffffffffu, incl >= need);
  const int L = m ? __ffs(m) - 1 : 31;
  int rb = 0, ra = 0, rc = 0;
  if (lane == L) {
    int acc = incl - s;
    for (int i = 0; i < per; ++i) {
      const int b = hi - 1 - i;
      const int c = static_cast<int>(h[b]);
      if (acc + c >= need || i == per - 1) { rb = b; ra = acc; rc = c; break; }
      acc += c;
    }
  }
  bin = __shfl_sync(0xffffffffu, rb, L);
  above = __shfl_sync(0xffffffffu, ra, L);
  cnt = __shfl_sync(0xffffffffu, rc, L);
}

template <int R>
struct Frags {
  static constexpr int KS = R / 16;
  uint32_t hi[KS][4];
  uint32_t lo[KS][4];
};

// Scores of this thread's 16 (row, key) pairs for the warp's 32 keys starting at kbase.
// sc[j][e]: row g + 8 (e >> 1), key kbase + 8 j + 2 t + (e & 1).
template <int R>
DSV_DEVICE void warp_scores(const Frags<R>& A, const bf16* __restrict__ kh, int64_t kbase, int64_t N, int g, int t,
                            float (&sc)[4][4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
    int64_t key = kbase + 8 * j + g;
    if (key >= N) key = N - 1;  // loads stay in bounds; the result is masked by the caller
    const uint2* src = reinterpret_cast<const uint2*>(kh + key * R) + t;
#pragma unroll
    for (int ks = 0; ks < Frags<R>::KS; ++ks) {
      const uint2 b = __ldg(src + ks * 4);
      mma_bf16_16816(sc[j], A.hi[ks], b.x, b.y);
      mma_bf16_16816(sc[j], A.lo[ks], b.x, b.y);
    }
  }
}

template <int R>
__global__ void __launch_bounds__(kThreads, 1)
estimate_topk_kernel(const bf16* __restrict__ q_lr, const bf16* __restrict__ k_lr, int32_t* __restrict__ idx,
                     int64_t N, int64_t NB, int64_t k, unsigned int* status) {
  extern __shared__ uint32_t hist[];  // [kRows][kBins]
  __shared__ float qhat[kRows][R];
  __shared__ RowState rs[kRows];
  __shared__ int wgt[kWarps][kRows];
  __shared__ int weq[kWarps][kRows];
  __shared__ int pending[3];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int64_t bh = blockIdx.y;
  const int64_t row0 = static_cast<int64_t>(blockIdx.x) * kRows;
  const int nrows = static_cast<int>(NB - row0 < kRows ? NB - row0 : kRows);
  const bf16* qh = q_lr + bh * N * R;
  const bf16* kh = k_lr + bh * N * R;
  int32_t* out = idx + (bh * NB + row0) * k;
  const int64_t ntiles = (N + kTileKeys - 1) / kTileKeys;

  // ---- query grouping: q_hat[row] = sum of the block's 64 Q_lr rows (fp32, exact for integers)
  for (int p = tid; p < kRows * R; p += kThreads) {
    const int row = p / R, c = p % R;
    float acc = 0.f;
    if (row < nrows) {
      const bf16* src = qh + (row0 + row) * 64 * R + c;
      for (int i = 0; i < 64; ++i) acc += __bfloat162float(src[i * R]);
    }
    qhat[row][c] = acc;
  }
  for (int i = tid; i < kRows * kBins; i += kThreads) hist[i] = 0u;
  if (tid < kRows) {
    RowState s;
    s.prefix = 0; s.level = 0; s.rem = static_cast<int>(k); s.T = 0; s.n_tie = 0; s.orbits = 0;
    s.out_pos = 0; s.tie_seen = 0;
    rs[tid] = s;
  }
  __syncthreads();

  // ---- A fragments: q_hat = hi + lo (bf16), with the k order permuted so each thread's
  // four k positions {2t, 2t+1, 2t+8, 2t+9} map to the contiguous channels 4t..4t+3.
  Frags<R> A;
#pragma unroll
  for (int ks = 0; ks < Frags<R>::KS; ++ks) {
    const int c0 = ks * 16 + 4 * t;
    const float x[4][2] = {{qhat[g][c0], qhat[g][c0 + 1]}, {qhat[g + 8][c0], qhat[g + 8][c0 + 1]},
                           {qhat[g][c0 + 2], qhat[g][c0 + 3]}, {qhat[g + 8][c0 + 2], qhat[g + 8][c0 + 3]}};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat16 h0 = __float2bfloat16_rn(x[i][0]), h1 = __float2bfloat16_rn(x[i][1]);
      const float l0 = x[i][0] - __bfloat162float(h0), l1 = x[i][1] - __bfloat162float(h1);
      A.hi[ks][i] = pack_bf16x2(__bfloat162float(h0), __bfloat162float(h1));
      A.lo[ks][i] = pack_bf16x2(l0, l1);
    }
  }

  // ---- histogram passes
  for (int level = 0; level < 3; ++level) {
    if (level > 0) {
      if (tid < 3) pending[tid] = 0;
      __syncthreads();
      if (tid < kRows && tid < nrows && rs[tid].level == level) atomicOr(&pending[level], 1);
      __syncthreads();
      if (!pending[level]) break;
      for (int i = tid; i < kRows * kBins; i += kThreads) hist[i] = 0u;
      __syncthreads();
    }
    // per-thread copy of the two rows' pass parameters
    uint32_t pre[2];
    bool act[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = g + 8 * h;
      act[h] = row < nrows && rs[row].level == level;
      pre[h] = rs[row].prefix;
    }
    for (int64_t tile = 0; tile < ntiles; ++tile) {
      const int64_t kbase = tile * kTileKeys + warp * 32;
      if (kbase >= N) continue;
      float sc[4][4];
      warp_scores<R>(A, kh, kbase, N, g, t, sc);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int h = e >> 1;
          const int64_t key_idx = kbase + 8 * j + 2 * t + (e & 1);
          if (!act[h] || key_idx >= N) continue;
          const uint32_t key = order_key(sc[j][e]);
          uint32_t* hrow = hist + (g + 8 * h) * kBins;
          if (level == 0) {
            atomicAdd(hrow + (key >> 21), 1u);
          } else if (level == 1) {
            if ((key >> 21) == pre[h]) {
              atomicAdd(hrow + ((key >> 10) & 2047u), 1u);
              if (key & 1023u) atomicOr(&rs[g + 8 * h].orbits, key & 1023u);
            }
          } else {
            if ((key >> 10) == pre[h]) atomicAdd(hrow + (key & 1023u), 1u);
          }
        }
      }
    }
    __syncthreads();
    // ---- resolve: warp w looks after row w
    if (warp < nrows && rs[warp].level == level) {
      RowState s = rs[warp];
      int bin, above, cnt;
      warp_find_bin(hist + warp * kBins, level == 2 ? 1024 : kBins, s.rem, lane, bin, above, cnt);
      const int rem = s.rem - above;  // 1 <= rem <= cnt
      if (level == 0) {
        if (rem == cnt) { s.T = static_cast<uint32_t>(bin) << 21; s.n_tie = kTieAll; s.level = 3; }
        else { s.prefix = bin; s.rem = rem; s.level = 1; }
      } else if (level == 1) {
        const uint32_t p = (s.prefix << 11) | static_cast<uint32_t>(bin);
        if (rem == cnt) { s.T = p << 10; s.n_tie = kTieAll; s.level = 3; }
        else if (s.orbits == 0) { s.T = p << 10; s.n_tie = rem; s.level = 3; }
        else { s.prefix = p; s.rem = rem; s.level = 2; }
      } else {
        s.T = (s.prefix << 10) | static_cast<uint32_t>(bin);
        s.n_tie = rem;
        s.level = 3;
      }
      __syncwarp();
      if (lane == 0) rs[warp] = s;
    }
    __syncthreads();
  }

  // ---- emit, keys in ascending order, one CTA-wide tile at a time
  uint32_t T[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) T[h] = rs[g + 8 * h].T;
  for (int64_t tile = 0; tile < ntiles; ++tile) {
    const int64_t kbase = tile * kTileKeys + warp * 32;
    uint32_t gtm[2] = {0u, 0u}, eqm[2] = {0u, 0u};
    if (kbase < N) {
      float sc[4][4];
      warp_scores<R>(A, kh, kbase, N, g, t, sc);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int h = e >> 1;
          const int pos = 8 * j + 2 * t + (e & 1);
          if (g + 8 * h >= nrows || kbase + pos >= N) continue;
          const uint32_t key = order_key(sc[j][e]);
          gtm[h] |= static_cast<uint32_t>(key > T[h]) << pos;
          eqm[h] |= static_cast<uint32_t>(key == T[h]) << pos;
        }
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      gtm[h] |= __shfl_xor_sync(0xffffffffu, gtm[h], 1);
      gtm[h] |= __shfl_xor_sync(0xffffffffu, gtm[h], 2);
      eqm[h] |= __shfl_xor_sync(0xffffffffu, eqm[h], 1);
      eqm[h] |= __shfl_xor_sync(0xffffffffu, eqm[h], 2);
    }
    if (t == 0) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        wgt[warp][g + 8 * h] = __popc(gtm[h]);
        weq[warp][g + 8 * h] = __popc(eqm[h]);
      }
    }
    __syncthreads();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = g + 8 * h;
      if (row >= nrows || (gtm[h] | eqm[h]) == 0u) continue;
      int bg = 0, be = 0;
      for (int w2 = 0; w2 < warp; ++w2) { bg += wgt[w2][row]; be += weq[w2][row]; }
      const int avail = max(0, rs[row].n_tie - rs[row].tie_seen);
      const int m = min(max(avail - be, 0), __popc(eqm[h]));
      const int base = rs[row].out_pos + bg + min(be, avail);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int pos = 8 * j + 2 * t + c;
          const uint32_t lt = (1u << pos) - 1u;
          const bool gt = (gtm[h] >> pos) & 1u;
          const bool eq = (eqm[h] >> pos) & 1u;
          const int eqb = __popc(eqm[h] & lt);
          if (gt || (eq && eqb < m)) {
            const int o = base + __popc(gtm[h] & lt) + min(eqb, m);
            if (o < k) out[row * k + o] = static_cast<int32_t>(kbase + pos);
            else flag_status(status, kStatusBadIndex);
          }
        }
      }
    }
    __syncthreads();
    if (tid < nrows) {
      int tg = 0, te = 0;
      for (int w2 = 0; w2 < kWarps; ++w2) { tg += wgt[w2][tid]; te += weq[w2][tid]; }
      const int avail = max(0, rs[tid].n_tie - rs[tid].tie_seen);
      rs[tid].out_pos += tg + min(te, avail);
      rs[tid].tie_seen += te;
    }
    __syncthreads();
  }
}

// k == N: every key of every block, ascending.
__global__ void arange_kernel(int32_t* __restrict__ idx, int64_t rows, int64_t k) {
  const int64_t total = rows * k;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    idx[i] = static_cast<int32_t>(i % k);
}

template <int R>
cudaError_t launch_r(const EstimateParams& p, cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(kRows) * kBins * sizeof(uint32_t);
  cudaError_t e = cudaFuncSetAttribute(estimate_topk_kernel<R>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>((p.NB + kRows - 1) / kRows), static_cast<unsigned>(p.BH));
  estimate_topk_kernel<R><<<grid, kThreads, smem, stream>>>(p.q_lr, p.k_lr, p.idx, p.N, p.NB, p.topk, p.status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_estimate_topk(const EstimateParams& p, cudaStream_t stream) {
  if (p.topk == p.N) {
    arange_kernel<<<4 * 152, 256, 0, stream>>>(p.idx, p.BH * p.NB, p.topk);
    return cudaGetLastError();
  }
  switch (p.r) {
    case 16: return launch_r<16>(p, stream);
    case 32: return launch_r<32>(p, stream);
    case 48: return launch_r<48>(p, stream);
    case 64: return launch_r<64>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dsv
