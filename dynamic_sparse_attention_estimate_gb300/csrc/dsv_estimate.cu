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
//   emit:   per segment of 32768 keys, bitmaps of "key > T" and "key == T" (the
//           histogram memory is reused), then one warp per query block turns them
//           into ascending key indices: every key > T, and the first n_tie keys == T
//           (ties go to the lower key index).
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
constexpr int kSegKeys = 32768;                 // keys per emit segment
constexpr int kSegWords = kSegKeys / 32;        // bitmap words per row per segment
constexpr int kTieAll = 0x7fffffff;
static_assert(2 * kRows * kSegWords <= kRows * kBins, "bitmaps reuse the histogram memory");

struct RowState {
  uint32_t prefix;  // resolved high bits of the threshold
  int level;        // 0/1/2: pass (level + 1) pending; 3: resolved
  int rem;          // elements still to take inside the current prefix
  uint32_t T;       // threshold key (resolved)
  int n_tie;        // elements equal to T to take, lowest key first
  uint32_t orbits;  // OR of bits [9:0] over pass-1 bin members
};

DSV_DEVICE uint32_t order_key(float s) {
  s = __fadd_rn(s, 0.0f);  // -0 -> +0 so that equal scores get equal keys
  const uint32_t u = __float_as_uint(s);
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
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
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

// B fragments of the warp's 32 keys [kbase, kbase + 32): thread (g, t) holds channels
// 4t..4t+3 (+16 ks) of key kbase + 8 j + g.
template <int R>
struct KeyFrags {
  uint2 b[4][R / 16];
};

template <int R>
DSV_DEVICE void load_keys(KeyFrags<R>& f, const bf16* __restrict__ kh, int kbase, int N, int g, int t) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    int key = kbase + 8 * j + g;
    key = key < N ? key : N - 1;  // stays in bounds; such keys are never used
    const uint2* src = reinterpret_cast<const uint2*>(kh + static_cast<int64_t>(key) * R) + t;
#pragma unroll
    for (int ks = 0; ks < R / 16; ++ks) f.b[j][ks] = __ldg(src + ks * 4);
  }
}

// sc[j][e]: row g + 8 (e >> 1), key kbase + 8 j + 2 t + (e & 1).
template <int R>
DSV_DEVICE void scores(const Frags<R>& A, const KeyFrags<R>& f, float (&sc)[4][4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < R / 16; ++ks) {
      mma_bf16_16816(sc[j], A.hi[ks], f.b[j][ks].x, f.b[j][ks].y);
      mma_bf16_16816(sc[j], A.lo[ks], f.b[j][ks].x, f.b[j][ks].y);
    }
  }
}

// Visit this warp's key groups in [k_begin, k_end) (32 keys each, tile stride), with the
// next group's K_lr fragments prefetched while the current one is consumed.
template <int R, typename F>
DSV_DEVICE void for_each_group(const Frags<R>& A, const bf16* __restrict__ kh, int N, int k_begin, int k_end, int warp,
                               int g, int t, F&& body) {
  int kbase = k_begin + warp * 32;
  if (kbase >= k_end) return;
  KeyFrags<R> cur, nxt;
  load_keys<R>(cur, kh, kbase, N, g, t);
  for (; kbase < k_end; kbase += kTileKeys) {
    const int knext = kbase + kTileKeys;
    if (knext < k_end) load_keys<R>(nxt, kh, knext, N, g, t);
    float sc[4][4];
    scores<R>(A, cur, sc);
    body(kbase, sc);
    cur = nxt;
  }
}

template <int LEVEL, int R>
DSV_DEVICE void hist_pass(const Frags<R>& A, const bf16* __restrict__ kh, int N, uint32_t* hist, RowState* rs,
                          int nrows, int warp, int g, int t) {
  bool act[2];
  uint32_t pre[2];
  uint32_t* hrow[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int row = g + 8 * h;
    act[h] = row < nrows && rs[row].level == LEVEL;
    pre[h] = rs[row].prefix;
    hrow[h] = hist + row * kBins;
  }
  for_each_group<R>(A, kh, N, 0, N, warp, g, t, [&](int kbase, const float (&sc)[4][4]) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int h = e >> 1;
        if (!act[h]) continue;
        const uint32_t key = order_key(sc[j][e]);
        if (LEVEL == 0) {
          atomicAdd(hrow[h] + (key >> 21), 1u);
        } else if (LEVEL == 1) {
          if ((key >> 21) == pre[h]) {
            atomicAdd(hrow[h] + ((key >> 10) & 2047u), 1u);
            if (key & 1023u) atomicOr(&rs[g + 8 * h].orbits, key & 1023u);
          }
        } else {
          if ((key >> 10) == pre[h]) atomicAdd(hrow[h] + (key & 1023u), 1u);
        }
      }
    }
  });
}

template <int R>
__global__ void __launch_bounds__(kThreads, 1)
estimate_topk_kernel(const bf16* __restrict__ q_lr, const bf16* __restrict__ k_lr, int32_t* __restrict__ idx,
                     int N, int NB, int k, unsigned int* status) {
  extern __shared__ uint32_t hist[];  // [kRows][kBins]; in the emit phase: gt / eq bitmaps
  __shared__ float qhat[kRows][R];
  __shared__ RowState rs[kRows];
  __shared__ int pending;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int64_t bh = blockIdx.y;
  const int row0 = blockIdx.x * kRows;
  const int nrows = NB - row0 < kRows ? NB - row0 : kRows;
  const bf16* qh = q_lr + bh * static_cast<int64_t>(N) * R;
  const bf16* kh = k_lr + bh * static_cast<int64_t>(N) * R;
  int32_t* out = idx + (bh * NB + row0) * static_cast<int64_t>(k);

  // ---- query grouping: q_hat[row] = sum of the block's 64 Q_lr rows (fp32, exact for integers)
  for (int p = tid; p < kRows * R; p += kThreads) {
    const int row = p / R, c = p % R;
    float acc = 0.f;
    if (row < nrows) {
      const bf16* src = qh + static_cast<int64_t>(row0 + row) * 64 * R + c;
      for (int i = 0; i < 64; ++i) acc += __bfloat162float(src[i * R]);
    }
    qhat[row][c] = acc;
  }
  for (int i = tid; i < kRows * kBins; i += kThreads) hist[i] = 0u;
  if (tid < kRows) rs[tid] = RowState{0u, 0, k, 0u, 0, 0u};
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
      const float h0 = __bfloat162float(__float2bfloat16_rn(x[i][0]));
      const float h1 = __bfloat162float(__float2bfloat16_rn(x[i][1]));
      A.hi[ks][i] = pack_bf16x2(h0, h1);
      A.lo[ks][i] = pack_bf16x2(x[i][0] - h0, x[i][1] - h1);
    }
  }

  // ---- histogram passes; warp w resolves row w after each
  auto resolve = [&](int level) {
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
  };
  auto next_level_pending = [&](int level) -> bool {
    if (tid == 0) pending = 0;
    __syncthreads();
    if (tid < nrows && rs[tid].level == level) atomicOr(&pending, 1);
    __syncthreads();
    const bool any = pending != 0;
    if (any)
      for (int i = tid; i < kRows * kBins; i += kThreads) hist[i] = 0u;
    __syncthreads();
    return any;
  };

  hist_pass<0, R>(A, kh, N, hist, rs, nrows, warp, g, t);
  __syncthreads();
  resolve(0);
  if (next_level_pending(1)) {
    hist_pass<1, R>(A, kh, N, hist, rs, nrows, warp, g, t);
    __syncthreads();
    resolve(1);
    if (next_level_pending(2)) {
      hist_pass<2, R>(A, kh, N, hist, rs, nrows, warp, g, t);
      __syncthreads();
      resolve(2);
    }
  }
  __syncthreads();

  // ---- emit, one segment of keys at a time
  uint32_t* gtb = hist;                        // [kRows][kSegWords]
  uint32_t* eqb = hist + kRows * kSegWords;    // [kRows][kSegWords]
  const uint32_t T0 = rs[g].T, T1 = rs[g + 8].T;
  int out_pos = 0, tie_seen = 0;               // row `warp`'s running counts (every lane holds them)
  const int n_tie = warp < nrows ? rs[warp].n_tie : 0;
  for (int seg = 0; seg < N; seg += kSegKeys) {
    const int seg_end = seg + kSegKeys < N ? seg + kSegKeys : N;
    for_each_group<R>(A, kh, N, seg, seg_end, warp, g, t, [&](int kbase, const float (&sc)[4][4]) {
      uint32_t gtm[2] = {0u, 0u}, eqm[2] = {0u, 0u};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int h = e >> 1;
          const int pos = 8 * j + 2 * t + (e & 1);
          const uint32_t key = order_key(sc[j][e]);
          const uint32_t T = h ? T1 : T0;
          gtm[h] |= static_cast<uint32_t>(key > T) << pos;
          eqm[h] |= static_cast<uint32_t>(key == T) << pos;
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
        const int w = (kbase - seg) >> 5;
        gtb[g * kSegWords + w] = gtm[0];
        eqb[g * kSegWords + w] = eqm[0];
        gtb[(g + 8) * kSegWords + w] = gtm[1];
        eqb[(g + 8) * kSegWords + w] = eqm[1];
      }
    });
    __syncthreads();
    if (warp < nrows) {
      const int nwords = (seg_end - seg) >> 5;
      const uint32_t* gw = gtb + warp * kSegWords;
      const uint32_t* ew = eqb + warp * kSegWords;
      int32_t* orow = out + static_cast<int64_t>(warp) * k;
      for (int w0 = 0; w0 < nwords; w0 += 32) {
        const int w = w0 + lane;
        const uint32_t gv = w < nwords ? gw[w] : 0u;
        const uint32_t ev = w < nwords ? ew[w] : 0u;
        // ties: this lane may take the lowest m of its equal keys
        const int ne = __popc(ev);
        int e_incl = ne;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int v = __shfl_up_sync(0xffffffffu, e_incl, o);
          if (lane >= o) e_incl += v;
        }
        const int avail = n_tie - tie_seen - (e_incl - ne);
        const int m = avail <= 0 ? 0 : (avail < ne ? avail : ne);
        uint32_t take = ev;
        if (m < ne) {
          take = 0u;
          uint32_t rest = ev;
          for (int i = 0; i < m; ++i) {
            const uint32_t b = rest & (0u - rest);
            take |= b;
            rest ^= b;
          }
        }
        uint32_t sel = gv | take;
        const int ns = __popc(sel);
        int s_incl = ns;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int v = __shfl_up_sync(0xffffffffu, s_incl, o);
          if (lane >= o) s_incl += v;
        }
        int o = out_pos + s_incl - ns;
        const int key0 = seg + (w << 5);
        while (sel) {
          const int b = __ffs(sel) - 1;
          sel &= sel - 1;
          if (o < k) orow[o] = key0 + b;
          else flag_status(status, kStatusBadIndex);
          ++o;
        }
        out_pos += __shfl_sync(0xffffffffu, s_incl, 31);
        tie_seen += __shfl_sync(0xffffffffu, e_incl, 31);
      }
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
  ProfScope prof("estimate_topk", stream);
  estimate_topk_kernel<R><<<grid, kThreads, smem, stream>>>(p.q_lr, p.k_lr, p.idx, static_cast<int>(p.N),
                                                             static_cast<int>(p.NB), static_cast<int>(p.topk),
                                                             p.status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_estimate_topk(const EstimateParams& p, cudaStream_t stream) {
  if (p.topk == p.N) {
    ProfScope prof("estimate_arange", stream);
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
