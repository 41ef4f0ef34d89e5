// Fused low-rank estimate + exact top-k per query block (DSV technical summary,
// section 2B "Fused MM & Top-K" with "Query Grouping").
//
// One CTA owns 16 query blocks of one head (the M = 16 rows of an m16n8k16 MMA) and
// streams every key of that head.  Scores s[b, j] = q_hat[b] . K_lr[j] live only in
// registers: they are recomputed on each pass and never written anywhere.
//
// Selection is an exact select on the order-preserving 32-bit image ("key") of the fp32
// score, per query block, in shared-memory histograms of 2048 bins:
//   sample: the scores of one 512-key tile in eight, histogrammed by key bits [31:21];
//           the sample's order statistics a few standard deviations on either side of
//           the k-th largest give a bracket [L, H] of keys that very likely holds it;
//   exact:  every key: those above H are counted (a register per row and thread, no
//           atomics), those inside the bracket histogrammed in 2048 bins of 2^sh keys.
//           If the k-th largest key lies outside the bracket the row falls back to the
//           whole key range; if its bin holds several distinct keys the bracket narrows
//           to that bin and the pass repeats (with integer scores below 2^13 one exact
//           pass suffices: their keys have zero low bits);
//   emit:   per segment of 32768 keys, bitmaps of "key > T" and "key == T" (the
//           histogram memory is reused), then one warp per query block turns them
//           into ascending key indices: every key > T, and the first n_tie keys == T
//           (ties go to the lower key index).
// The sample only decides how much work the exact passes take; the result is the exact
// top-k whatever it holds.
// q_hat is held as hi + lo bf16 (an exact split for |q_hat| < 2^16), so with
// integer-valued factors every fp32 score is the exact integer.
#include <stdint.h>

#include "dsv_common.cuh"
#include "dsv_internal.h"

namespace dsv {
namespace {

constexpr int kRows = 16;                       // query blocks per m16 row tile of the MMA
constexpr int kMaxRows2 = 27;                   // query blocks per CTA with two row tiles (shared memory)
constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kTileKeys = kWarps * 32;          // keys per CTA-wide tile (32 per warp)
constexpr int kBins = 2048;
constexpr int kSegKeys = 32768;                 // keys per emit segment
constexpr int kSegWords = kSegKeys / 32;        // bitmap words per row per segment
constexpr int kTieAll = 0x7fffffff;
constexpr int kSampleEvery = 8;                 // the sample: one key tile in this many
constexpr int kMaxExactPasses = 6;              // bracket, widen, and two narrowings at most
static_assert(2 * kRows * kSegWords <= kRows * kBins, "bitmaps reuse the histogram memory");

struct RowState {
  uint32_t L, H;    // the bracket of keys [L, H] the next exact pass histograms
  int sh;           // its bins hold 2^sh keys each
  int resolved;     // 0: an exact pass pending; 1: T and n_tie final
  int k;            // keys to select
  int above;        // keys > H (the exact pass counts them)
  uint32_t orbits;  // OR of (key - L) mod 2^sh over the bracket's members
  uint32_t T;       // threshold key (resolved)
  int n_tie;        // elements equal to T to take, lowest key first
};

DSV_DEVICE uint32_t order_key(float s) {
  s = __fadd_rn(s, 0.0f);  // -0 -> +0 so that equal scores get equal keys
  const uint32_t u = __float_as_uint(s);
  return u ^ (static_cast<uint32_t>(static_cast<int32_t>(u) >> 31) | 0x80000000u);
}

// Float bounds so that the passes compare scores directly instead of forming every score's key:
// for every score s that is not NaN, order_key(s) >= K  <=>  s >= ge_value(K), and
// order_key(s) > K  <=>  s >= gt_value(K).  Keys at or below that of -inf give -inf; keys above
// that of +inf (NaN patterns) give NaN, which no comparison passes; the key just below +0's
// (the image of -0, which order_key folds into +0) behaves like +0's; every other key is the
// image of exactly one float.
DSV_DEVICE float ge_value(uint32_t K) {
  if (K <= 0x007fffffu) return -__int_as_float(0x7f800000);
  if (K > 0xff800000u) return __int_as_float(0x7fc00000);
  if (K == 0x7fffffffu) K = 0x80000000u;
  return __uint_as_float((K & 0x80000000u) ? (K ^ 0x80000000u) : ~K);
}
DSV_DEVICE float gt_value(uint32_t K) { return K == 0xffffffffu ? __int_as_float(0x7fc00000) : ge_value(K + 1u); }

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
template <int R, int MT, typename F>
DSV_DEVICE void for_each_group(const Frags<R> (&A)[MT], const bf16* __restrict__ kh, int N, int k_begin, int k_end,
                               int warp, int g, int t, F&& body, int stride = kTileKeys) {
  int kbase = k_begin + warp * 32;
  if (kbase >= k_end) return;
  KeyFrags<R> cur, nxt;
  load_keys<R>(cur, kh, kbase, N, g, t);
  for (; kbase < k_end; kbase += stride) {
    const int knext = kbase + stride;
    if (knext < k_end) load_keys<R>(nxt, kh, knext, N, g, t);
    float sc[MT][4][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) scores<R>(A[mt], cur, sc[mt]);
    body(kbase, sc);
    cur = nxt;
  }
}

// One row tile (the mass kernel): sc[j][e] as above.
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

// The sample: tiles 0, kSampleEvery, 2 kSampleEvery, ... of every pending row, histogrammed by
// key bits [31:21].
template <int R, int MT>
DSV_DEVICE void sample_pass(const Frags<R> (&A)[MT], const bf16* __restrict__ kh, int N, uint32_t* hist,
                            const RowState* rs, int nrows, int warp, int g, int t) {
  bool act[MT][2];
  uint32_t* hrow[MT][2];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = kRows * mt + g + 8 * h;
      act[mt][h] = row < nrows && !rs[row].resolved;
      hrow[mt][h] = hist + row * kBins;
    }
  for_each_group<R, MT>(
      A, kh, N, 0, N, warp, g, t,
      [&](int, const float (&sc)[MT][4][4]) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (act[mt][e >> 1]) atomicAdd(hrow[mt][e >> 1] + (order_key(sc[mt][j][e]) >> 21), 1u);
      },
      kSampleEvery * kTileKeys);
}

// One exact pass over every key of the pending rows: keys above the bracket are counted in
// registers, keys inside it histogrammed.
template <int R, int MT>
DSV_DEVICE void exact_pass(const Frags<R> (&A)[MT], const bf16* __restrict__ kh, int N, uint32_t* hist, RowState* rs,
                           int nrows, int warp, int g, int t) {
  bool act[MT][2];
  uint32_t lo[MT][2], mask[MT][2], orb[MT][2];
  float vlo[MT][2], vhi[MT][2];  // key >= L  <=>  s >= vlo;  key > H  <=>  s >= vhi
  int sh[MT][2], above[MT][2];
  uint32_t* hrow[MT][2];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = kRows * mt + g + 8 * h;
      act[mt][h] = row < nrows && !rs[row].resolved;
      lo[mt][h] = rs[row].L;
      vlo[mt][h] = ge_value(rs[row].L);
      vhi[mt][h] = gt_value(rs[row].H);
      sh[mt][h] = rs[row].sh;
      mask[mt][h] = (1u << sh[mt][h]) - 1u;
      orb[mt][h] = 0u;
      above[mt][h] = 0;
      hrow[mt][h] = hist + row * kBins;
    }
  for_each_group<R, MT>(A, kh, N, 0, N, warp, g, t, [&](int, const float (&sc)[MT][4][4]) {
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int h = e >> 1;
          const float sv = sc[mt][j][e];
          const bool over = sv >= vhi[mt][h];
          above[mt][h] += over ? 1 : 0;
          if (!over && sv >= vlo[mt][h] && act[mt][h]) {
            const uint32_t off = order_key(sv) - lo[mt][h];
            atomicAdd(hrow[mt][h] + (off >> sh[mt][h]), 1u);
            orb[mt][h] |= off & mask[mt][h];
          }
        }
  });
  // the four lanes of a row group (t = 0..3) hold the same rows
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      int a = above[mt][h];
      uint32_t o = orb[mt][h];
      a += __shfl_xor_sync(0xffffffffu, a, 1);
      a += __shfl_xor_sync(0xffffffffu, a, 2);
      o |= __shfl_xor_sync(0xffffffffu, o, 1);
      o |= __shfl_xor_sync(0xffffffffu, o, 2);
      if (t == 0 && act[mt][h]) {
        RowState& r = rs[kRows * mt + g + 8 * h];
        if (a) atomicAdd(&r.above, a);
        if (o) atomicOr(&r.orbits, o);
      }
    }
}

// MT m16 row tiles of the MMA: `rows` query blocks per CTA (<= 16 MT; shared memory holds
// `rows` histograms), so that the grid can be sized to fill the GPU in whole waves.
template <int R, int MT>
__global__ void __launch_bounds__(kThreads, 1)
estimate_topk_kernel(const bf16* __restrict__ q_lr, const bf16* __restrict__ k_lr, int32_t* __restrict__ idx,
                     int N, int NB, int k, int rows, const int32_t* __restrict__ krow,
                     const int64_t* __restrict__ rowptr, unsigned int* status) {
  constexpr int kMax = kRows * MT;
  extern __shared__ uint32_t hist[];  // [rows][kBins]; in the emit phase: gt / eq bitmaps
  __shared__ float qhat[kMax][R];
  __shared__ RowState rs[kMax];
  __shared__ int pending;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int64_t bh = blockIdx.y;
  const int row0 = blockIdx.x * rows;
  const int nrows = NB - row0 < rows ? NB - row0 : rows;
  const bf16* qh = q_lr + bh * static_cast<int64_t>(N) * R;
  const bf16* kh = k_lr + bh * static_cast<int64_t>(N) * R;
  // per row: its k (krow, or the uniform k) and where its indices go (CSR offsets, or row * k)
  const int64_t grow0 = bh * NB + row0;
  auto row_k = [&](int row) -> int { return krow ? krow[grow0 + row] : k; };
  auto row_out = [&](int row) -> int32_t* {
    return idx + (rowptr ? rowptr[grow0 + row] : (grow0 + row) * static_cast<int64_t>(k));
  };

  // ---- query grouping: q_hat[row] = sum of the block's 64 Q_lr rows (fp32, exact for integers)
  for (int p = tid; p < kMax * R; p += kThreads) {
    const int row = p / R, c = p % R;
    float acc = 0.f;
    if (row < nrows) {
      const bf16* src = qh + static_cast<int64_t>(row0 + row) * 64 * R + c;
      for (int i = 0; i < 64; ++i) acc += __bfloat162float(src[i * R]);
    }
    qhat[row][c] = acc;
  }
  for (int i = tid; i < rows * kBins; i += kThreads) hist[i] = 0u;
  if (tid < kMax) {
    // k <= 0 selects nothing (no key is above the largest key), k >= N every key
    const int kr = tid < nrows ? row_k(tid) : 0;
    RowState r{0u, 0xffffffffu, 21, 0, kr, 0, 0u, 0u, 0};
    if (kr <= 0) { r.resolved = 1; r.T = 0xffffffffu; r.n_tie = 0; }
    else if (kr >= N) { r.resolved = 1; r.T = 0u; r.n_tie = kTieAll; }
    rs[tid] = r;
  }
  __syncthreads();

  // ---- A fragments: q_hat = hi + lo (bf16), with the k order permuted so each thread's
  // four k positions {2t, 2t+1, 2t+8, 2t+9} map to the contiguous channels 4t..4t+3.
  Frags<R> A[MT];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
  for (int ks = 0; ks < Frags<R>::KS; ++ks) {
    const int c0 = ks * 16 + 4 * t;
    const int r0 = kRows * mt + g, r1 = r0 + 8;
    const float x[4][2] = {{qhat[r0][c0], qhat[r0][c0 + 1]}, {qhat[r1][c0], qhat[r1][c0 + 1]},
                           {qhat[r0][c0 + 2], qhat[r0][c0 + 3]}, {qhat[r1][c0 + 2], qhat[r1][c0 + 3]}};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float h0 = __bfloat162float(__float2bfloat16_rn(x[i][0]));
      const float h1 = __bfloat162float(__float2bfloat16_rn(x[i][1]));
      A[mt].hi[ks][i] = pack_bf16x2(h0, h1);
      A[mt].lo[ks][i] = pack_bf16x2(x[i][0] - h0, x[i][1] - h1);
    }
  }

  // ---- the sample and the bracket of every row (warp w sets up rows w, w + 16, ...)
  auto any_pending = [&]() -> bool {  // also clears the histograms when a pass follows
    if (tid == 0) pending = 0;
    __syncthreads();
    if (tid < nrows && !rs[tid].resolved) atomicOr(&pending, 1);
    __syncthreads();
    const bool any = pending != 0;
    if (any)
      for (int i = tid; i < rows * kBins; i += kThreads) hist[i] = 0u;
    __syncthreads();
    return any;
  };
  if (any_pending()) {
    sample_pass<R, MT>(A, kh, N, hist, rs, nrows, warp, g, t);
    __syncthreads();
    int n_s = 0;  // sampled keys per row
    for (int t0 = 0; t0 < N; t0 += kSampleEvery * kTileKeys) n_s += N - t0 < kTileKeys ? N - t0 : kTileKeys;
#pragma unroll
    for (int q = 0; q < MT; ++q) {
      const int row = warp + kWarps * q;
      if (row < nrows && !rs[row].resolved) {
        RowState s = rs[row];
        // the k-th largest key sits near rank rho of the sample; take ranks about four
        // binomial standard deviations (plus a few) to either side
        const float frac = static_cast<float>(s.k) / static_cast<float>(N);
        const float rho = frac * static_cast<float>(n_s);
        const float m = 4.f * sqrtf(rho * (1.f - frac)) + 4.f;
        const int r_hi = static_cast<int>(floorf(rho - m)), r_lo = static_cast<int>(ceilf(rho + m));
        int bin_hi = kBins - 1, bin_lo = 0, above, cnt;
        if (r_hi >= 1) warp_find_bin(hist + row * kBins, kBins, r_hi, lane, bin_hi, above, cnt);
        if (r_lo <= n_s) warp_find_bin(hist + row * kBins, kBins, r_lo, lane, bin_lo, above, cnt);
        const int span = bin_hi - bin_lo + 1;  // bins of 2^21 keys
        int sh = 10;
        while ((1 << (sh - 10)) < span && sh < 21) ++sh;
        s.sh = sh;
        s.L = sh >= 21 ? 0u : static_cast<uint32_t>(bin_lo) << 21;
        const uint64_t h64 = static_cast<uint64_t>(s.L) + (static_cast<uint64_t>(kBins) << sh) - 1u;
        s.H = h64 > 0xffffffffull ? 0xffffffffu : static_cast<uint32_t>(h64);
        __syncwarp();
        if (lane == 0) rs[row] = s;
      }
    }
    __syncthreads();
    for (int pass = 0; pass < kMaxExactPasses && any_pending(); ++pass) {
      exact_pass<R, MT>(A, kh, N, hist, rs, nrows, warp, g, t);
      __syncthreads();
#pragma unroll
      for (int q = 0; q < MT; ++q) {
        const int row = warp + kWarps * q;
        if (row < nrows && !rs[row].resolved) {
          RowState s = rs[row];
          const uint32_t* hr = hist + row * kBins;
          int inside = 0;
          for (int b = lane; b < kBins; b += 32) inside += static_cast<int>(hr[b]);
#pragma unroll
          for (int o = 16; o >= 1; o >>= 1) inside += __shfl_xor_sync(0xffffffffu, inside, o);
          const int rem = s.k - s.above;  // to take at or below H
          if (rem < 1 || rem > inside) {
            // the k-th largest key is outside the bracket: the whole key range next
            s.L = 0u;
            s.H = 0xffffffffu;
            s.sh = 21;
          } else {
            int bin, abv, cnt;
            warp_find_bin(hr, kBins, rem, lane, bin, abv, cnt);
            const int rem2 = rem - abv;  // 1 <= rem2 <= cnt: to take inside the bin
            const uint32_t base = s.L + (static_cast<uint32_t>(bin) << s.sh);
            if (rem2 == cnt) {  // the whole bin: every key >= its lowest
              s.T = base;
              s.n_tie = kTieAll;
              s.resolved = 1;
            } else if (s.sh == 0 || s.orbits == 0u) {  // the bin holds one key value
              s.T = base;
              s.n_tie = rem2;
              s.resolved = 1;
            } else {  // narrow to the bin
              s.L = base;
              s.H = base + ((1u << s.sh) - 1u);
              s.sh = s.sh > 11 ? s.sh - 11 : 0;
            }
          }
          s.above = 0;
          s.orbits = 0u;
          __syncwarp();
          if (lane == 0) rs[row] = s;
        }
      }
    }
    if (tid < nrows && !rs[tid].resolved) {  // unreachable: every row resolves within the passes
      flag_status(status, kStatusBadIndex);
      rs[tid].T = 0xffffffffu;
      rs[tid].n_tie = 0;
    }
  }
  __syncthreads();

  // ---- emit, one segment of keys at a time
  uint32_t* gtb = hist;                      // [rows][kSegWords]
  uint32_t* eqb = hist + rows * kSegWords;   // [rows][kSegWords]
  float vgt[MT][2], vge[MT][2];  // key > T  <=>  s >= vgt;  key >= T  <=>  s >= vge
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t T = rs[kRows * mt + g + 8 * h].T;
      vgt[mt][h] = gt_value(T);
      vge[mt][h] = ge_value(T);
    }
  // rows warp and warp + 16: running counts (every lane holds them)
  int out_pos[MT], tie_seen[MT], n_tie[MT];
#pragma unroll
  for (int q = 0; q < MT; ++q) {
    const int row = warp + kWarps * q;
    out_pos[q] = tie_seen[q] = 0;
    n_tie[q] = row < nrows ? rs[row].n_tie : 0;
  }
  for (int seg = 0; seg < N; seg += kSegKeys) {
    const int seg_end = seg + kSegKeys < N ? seg + kSegKeys : N;
    for_each_group<R, MT>(A, kh, N, seg, seg_end, warp, g, t, [&](int kbase, const float (&sc)[MT][4][4]) {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        uint32_t gtm[2] = {0u, 0u}, eqm[2] = {0u, 0u};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int h = e >> 1;
            const int pos = 8 * j + (e & 1);  // + 2 t, applied below
            const float sv = sc[mt][j][e];
            const bool gt = sv >= vgt[mt][h];
            gtm[h] |= static_cast<uint32_t>(gt) << pos;
            eqm[h] |= static_cast<uint32_t>(!gt && sv >= vge[mt][h]) << pos;
          }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          gtm[h] <<= 2 * t;
          eqm[h] <<= 2 * t;
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
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int row = kRows * mt + g + 8 * h;
            if (row < nrows) {  // the bitmaps hold `rows` rows
              gtb[row * kSegWords + w] = gtm[h];
              eqb[row * kSegWords + w] = eqm[h];
            }
          }
        }
      }
    });
    __syncthreads();
#pragma unroll
    for (int q = 0; q < MT; ++q) {
      const int row = warp + kWarps * q;
      if (row >= nrows) continue;
      const int nwords = (seg_end - seg) >> 5;
      const uint32_t* gw = gtb + row * kSegWords;
      const uint32_t* ew = eqb + row * kSegWords;
      int32_t* orow = row_out(row);
      const int kw = row_k(row);
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
        const int avail = n_tie[q] - tie_seen[q] - (e_incl - ne);
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
        int o = out_pos[q] + s_incl - ns;
        const int key0 = seg + (w << 5);
        while (sel) {
          const int b = __ffs(sel) - 1;
          sel &= sel - 1;
          if (o < kw) orow[o] = key0 + b;
          else flag_status(status, kStatusBadIndex);
          ++o;
        }
        out_pos[q] += __shfl_sync(0xffffffffu, s_incl, 31);
        tie_seen[q] += __shfl_sync(0xffffffffu, e_incl, 31);
      }
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------- mass-based adaptive k
// Per query block the length of the shortest (score desc, key asc) prefix of its keys whose
// estimated attention mass reaches the fraction mass_num / 2^16 of the total (DSV pages,
// German summary section 2A stage 2 and Spanish "Fase 2": the critical pairs carry ~90 % of
// the attention score).  Mass is counted in integer weights w = floor(2^24 * 2^x), x =
// tau_log2 * (s - max s), with 2^x by one fixed fp32 recipe (x = n + f, 2^f from its Taylor
// series to degree 6, every product and sum rounded separately), so the integer decision is
// reproducible bit for bit.  The search is a radix select on the score's order-preserving
// key, with per-bin weight sums and counts instead of counts alone:
//   0. exact row maximum;  1. weights and counts per bin of key bits [31:21], total W;
//   2. inside the bin where the running weight from the top reaches ceil(W mass), bins of
//      bits [20:10] (exact when no member has bits [9:0] set: integer scores);
//   3. otherwise bits [9:0];
// then k = (keys above the threshold value T) + ceil((target - their weight) / w(T)).
constexpr int kMassRows = 8;  // query blocks per CTA (MMA rows 8..15 stay zero)

struct MassState {
  unsigned long long total, target, w_above;
  uint32_t c_above, maxkey, prefix, orbits;
  int level;
};

struct MassCoef {
  float c[7];
};

DSV_DEVICE float key_value(uint32_t key) {  // inverse of order_key
  return __uint_as_float((key & 0x80000000u) ? (key ^ 0x80000000u) : ~key);
}

DSV_DEVICE uint32_t mass_weight(float s, float smax, float tau_log2, const MassCoef& c) {
  const float x = __fmul_rn(tau_log2, __fsub_rn(s, smax));
  if (!(x >= -30.f)) return 0u;
  const float n = floorf(x);
  const float f = __fsub_rn(x, n);  // exact
  float p = c.c[6];
#pragma unroll
  for (int i = 5; i >= 0; --i) p = __fadd_rn(__fmul_rn(p, f), c.c[i]);
  return __float2uint_rz(ldexpf(p, static_cast<int>(n) + 24));
}

// Warp search over one row's per-bin weights hw and counts hc, from the top bin down: the
// bin where the running weight (starting at w0) first reaches `target`, the running weight
// before it and the count of this level's bins above it.
DSV_DEVICE void warp_find_mass_bin(const unsigned long long* hw, const uint32_t* hc, int nbins, unsigned long long w0,
                                   unsigned long long target, int lane, int& bin, unsigned long long& w_above,
                                   uint32_t& c_above) {
  const int per = nbins / 32;
  const int hi = nbins - lane * per;  // this lane's bins: [hi - per, hi)
  unsigned long long sw = 0;
  uint32_t sc = 0;
  for (int i = 0; i < per; ++i) {
    const int b = hi - 1 - ((i + lane) % per);
    sw += hw[b];
    sc += hc[b];
  }
  unsigned long long iw = sw;
  uint32_t ic = sc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long vw = __shfl_up_sync(0xffffffffu, iw, o);
    const uint32_t vc = __shfl_up_sync(0xffffffffu, ic, o);
    if (lane >= o) {
      iw += vw;
      ic += vc;
    }
  }
  const unsigned m = __ballot_sync(0xffffffffu, w0 + iw >= target);
  const int L = m ? __ffs(m) - 1 : 31;
  int rb = 0;
  unsigned long long rw = 0;
  uint32_t rc = 0;
  if (lane == L) {
    unsigned long long acc = w0 + iw - sw;
    uint32_t cacc = ic - sc;
    for (int i = 0; i < per; ++i) {
      const int b = hi - 1 - i;
      if (acc + hw[b] >= target || i == per - 1) {
        rb = b;
        rw = acc;
        rc = cacc;
        break;
      }
      acc += hw[b];
      cacc += hc[b];
    }
  }
  bin = __shfl_sync(0xffffffffu, rb, L);
  w_above = __shfl_sync(0xffffffffu, rw, L);
  c_above = __shfl_sync(0xffffffffu, rc, L);
}

template <int R>
__global__ void __launch_bounds__(kThreads, 1)
mass_k_kernel(const bf16* __restrict__ q_lr, const bf16* __restrict__ k_lr, int N, int NB, float tau_log2,
              uint32_t mass_num, uint32_t dense_num, MassCoef coef, int32_t* __restrict__ krow) {
  extern __shared__ unsigned long long mhw[];                            // [rows][kBins] weights
  uint32_t* mhc = reinterpret_cast<uint32_t*>(mhw + kMassRows * kBins);  // [rows][kBins] counts
  __shared__ float qhat[16][R];
  __shared__ MassState ms[kMassRows];
  __shared__ int pending;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int64_t bh = blockIdx.y;
  const int row0 = blockIdx.x * kMassRows;
  const int nrows = NB - row0 < kMassRows ? NB - row0 : kMassRows;
  const bf16* qh = q_lr + bh * static_cast<int64_t>(N) * R;
  const bf16* kh = k_lr + bh * static_cast<int64_t>(N) * R;

  for (int p = tid; p < 16 * R; p += kThreads) {
    const int row = p / R, c = p % R;
    float acc = 0.f;
    if (row < nrows) {
      const bf16* src = qh + static_cast<int64_t>(row0 + row) * 64 * R + c;
      for (int i = 0; i < 64; ++i) acc += __bfloat162float(src[i * R]);
    }
    qhat[row][c] = acc;
  }
  auto clear = [&]() {
    for (int i = tid; i < kMassRows * kBins; i += kThreads) {
      mhw[i] = 0ull;
      mhc[i] = 0u;
    }
  };
  clear();
  if (tid < kMassRows) ms[tid] = MassState{0ull, 0ull, 0ull, 0u, 0u, 0u, 0u, 0};
  __syncthreads();

  Frags<R> A;  // q_hat = hi + lo (bf16), as in the top-k kernel
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
  const bool act = g < nrows;  // this thread's row is g (MMA rows g + 8 are unused)
  uint32_t* hcr = mhc + g * kBins;
  unsigned long long* hwr = mhw + g * kBins;

  // ---- 0. exact row maximum
  uint32_t mk = 0u;
  for_each_group<R>(A, kh, N, 0, N, warp, g, t, [&](int, const float (&sc)[4][4]) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int e = 0; e < 2; ++e) mk = max(mk, order_key(sc[j][e]));
  });
  mk = max(mk, __shfl_xor_sync(0xffffffffu, mk, 1));
  mk = max(mk, __shfl_xor_sync(0xffffffffu, mk, 2));
  if (act && t == 0) atomicMax(&ms[g].maxkey, mk);
  __syncthreads();
  const float smax = key_value(ms[g].maxkey);

  // ---- 1. weights per bin of bits [31:21], and the total
  unsigned long long tot = 0ull;
  for_each_group<R>(A, kh, N, 0, N, warp, g, t, [&](int, const float (&sc)[4][4]) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const uint32_t w = act ? mass_weight(sc[j][e], smax, tau_log2, coef) : 0u;
        if (w == 0u) continue;
        const uint32_t key = order_key(sc[j][e]);
        atomicAdd(hwr + (key >> 21), static_cast<unsigned long long>(w));
        atomicAdd(hcr + (key >> 21), 1u);
        tot += w;
      }
  });
  tot += __shfl_xor_sync(0xffffffffu, tot, 1);
  tot += __shfl_xor_sync(0xffffffffu, tot, 2);
  if (act && t == 0) atomicAdd(&ms[g].total, tot);
  __syncthreads();
  if (warp < nrows) {
    MassState st = ms[warp];
    st.target = (st.total * mass_num + 65535ull) >> 16;
    int bin;
    unsigned long long wa;
    uint32_t ca;
    warp_find_mass_bin(mhw + warp * kBins, mhc + warp * kBins, kBins, 0ull, st.target, lane, bin, wa, ca);
    st.prefix = static_cast<uint32_t>(bin);
    st.w_above = wa;
    st.c_above = ca;
    st.level = 1;
    __syncwarp();
    if (lane == 0) ms[warp] = st;
    __syncwarp();
  }
  __syncthreads();
  clear();
  __syncthreads();

  // ---- 2. inside that bin: bits [20:10]
  {
    const uint32_t pre = ms[g].prefix;
    for_each_group<R>(A, kh, N, 0, N, warp, g, t, [&](int, const float (&sc)[4][4]) {
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const uint32_t key = order_key(sc[j][e]);
          if (!act || (key >> 21) != pre) continue;
          const uint32_t w = mass_weight(sc[j][e], smax, tau_log2, coef);
          if (w == 0u) continue;
          atomicAdd(hwr + ((key >> 10) & 2047u), static_cast<unsigned long long>(w));
          atomicAdd(hcr + ((key >> 10) & 2047u), 1u);
          if (key & 1023u) atomicOr(&ms[g].orbits, key & 1023u);
        }
    });
  }
  __syncthreads();
  if (warp < nrows) {
    MassState st = ms[warp];
    int bin;
    unsigned long long wa;
    uint32_t ca;
    warp_find_mass_bin(mhw + warp * kBins, mhc + warp * kBins, kBins, st.w_above, st.target, lane, bin, wa, ca);
    st.prefix = (st.prefix << 11) | static_cast<uint32_t>(bin);
    st.w_above = wa;
    st.c_above += ca;
    st.level = st.orbits == 0u ? 3 : 2;  // no member below bit 10: the key is exact
    __syncwarp();
    if (lane == 0) ms[warp] = st;
    __syncwarp();
  }
  if (tid == 0) pending = 0;
  __syncthreads();
  if (tid < nrows && ms[tid].level == 2) atomicOr(&pending, 1);
  __syncthreads();

  // ---- 3. if needed: bits [9:0]
  if (pending) {
    clear();
    __syncthreads();
    const uint32_t pre = ms[g].prefix;
    const bool need = act && ms[g].level == 2;
    for_each_group<R>(A, kh, N, 0, N, warp, g, t, [&](int, const float (&sc)[4][4]) {
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const uint32_t key = order_key(sc[j][e]);
          if (!need || (key >> 10) != pre) continue;
          const uint32_t w = mass_weight(sc[j][e], smax, tau_log2, coef);
          if (w == 0u) continue;
          atomicAdd(hwr + (key & 1023u), static_cast<unsigned long long>(w));
          atomicAdd(hcr + (key & 1023u), 1u);
        }
    });
    __syncthreads();
    if (warp < nrows && ms[warp].level == 2) {
      MassState st = ms[warp];
      int bin;
      unsigned long long wa;
      uint32_t ca;
      warp_find_mass_bin(mhw + warp * kBins, mhc + warp * kBins, 1024, st.w_above, st.target, lane, bin, wa, ca);
      st.prefix = (st.prefix << 10) | static_cast<uint32_t>(bin);
      st.w_above = wa;
      st.c_above += ca;
      st.level = 4;
      __syncwarp();
      if (lane == 0) ms[warp] = st;
      __syncwarp();
    }
    __syncthreads();
  }

  // ---- k = keys above T + the keys equal to T needed to reach the target
  if (warp < nrows && lane == 0) {
    const MassState st = ms[warp];
    const uint32_t T = st.level == 3 ? (st.prefix << 10) : st.prefix;
    const unsigned long long wt = mass_weight(key_value(T), key_value(st.maxkey), tau_log2, coef);
    const unsigned long long n_tie = wt ? (st.target - st.w_above + wt - 1ull) / wt : 0ull;
    unsigned long long kb = st.c_above + n_tie;
    // sparse/dense switch: a block whose k exceeds dense_num / 2^16 of the keys takes them all
    if (dense_num && kb * 65536ull > static_cast<unsigned long long>(dense_num) * static_cast<unsigned long long>(N))
      kb = static_cast<unsigned long long>(N);
    krow[bh * NB + row0 + warp] = static_cast<int32_t>(kb);
  }
}

// CSR row offsets: rowptr[0] = 0, rowptr[i + 1] = krow[0] + ... + krow[i] (one CTA).
__global__ void __launch_bounds__(1024) csr_scan_kernel(const int32_t* __restrict__ krow, int64_t rows,
                                                        int64_t* __restrict__ rowptr) {
  __shared__ long long part[1024];
  const int t = threadIdx.x;
  const int64_t per = (rows + 1023) / 1024;
  const int64_t b = t * per, e = b + per < rows ? b + per : rows;
  long long s = 0;
  for (int64_t i = b; i < e; ++i) s += krow[i];
  part[t] = s;
  __syncthreads();
  for (int o = 1; o < 1024; o <<= 1) {
    const long long v = t >= o ? part[t - o] : 0;
    __syncthreads();
    part[t] += v;
    __syncthreads();
  }
  long long run = part[t] - s;
  if (t == 0) rowptr[0] = 0;
  for (int64_t i = b; i < e; ++i) {
    run += krow[i];
    rowptr[i + 1] = run;
  }
}

// Launch order for the attention over CSR rows: rows by descending chunk count (ceil(k / 128)),
// so the longest blocks start first and the grid's tail is short (the order inside a class is
// whatever the shared-memory atomics give; results do not depend on it).  One CTA; the
// per-class counters live in shared memory (nclass <= 4096).
__global__ void __launch_bounds__(1024) csr_order_kernel(const int64_t* __restrict__ rowptr, int64_t rows, int nclass,
                                                         int32_t* __restrict__ order) {
  __shared__ int start[4096];
  const int t = threadIdx.x;
  for (int c = t; c < nclass; c += 1024) start[c] = 0;
  __syncthreads();
  auto cls = [&](int64_t i) {
    const int64_t nch = (rowptr[i + 1] - rowptr[i] + 127) / 128;
    return static_cast<int>(nch < nclass - 1 ? nch : nclass - 1);
  };
  for (int64_t i = t; i < rows; i += 1024) atomicAdd(&start[cls(i)], 1);
  __syncthreads();
  if (t == 0) {  // exclusive scan from the heaviest class down
    int run = 0;
    for (int c = nclass - 1; c >= 0; --c) {
      const int n = start[c];
      start[c] = run;
      run += n;
    }
  }
  __syncthreads();
  for (int64_t i = t; i < rows; i += 1024) order[atomicAdd(&start[cls(i)], 1)] = static_cast<int32_t>(i);
}

template <int R>
cudaError_t launch_mass_r(const MassParams& p, cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(kMassRows) * kBins * (sizeof(unsigned long long) + sizeof(uint32_t));
  cudaError_t e = cudaFuncSetAttribute(mass_k_kernel<R>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  MassCoef coef;
  for (int i = 0; i < 7; ++i) coef.c[i] = p.coef[i];
  dim3 grid(static_cast<unsigned>((p.NB + kMassRows - 1) / kMassRows), static_cast<unsigned>(p.BH));
  ProfScope prof("estimate_mass_k", stream);
  mass_k_kernel<R><<<grid, kThreads, smem, stream>>>(p.q_lr, p.k_lr, static_cast<int>(p.N), static_cast<int>(p.NB),
                                                     p.tau_log2, p.mass_num, p.dense_num, coef, p.krow);
  return cudaGetLastError();
}

// Query blocks per CTA.  One CTA runs per SM and the grid has ceil(NB / rows) CTAs per head.
// Measured on the short clip (12 heads x 256 blocks, r = 16): a CTA's time hardly depends on its
// rows (8..16 rows: 103 us a wave; the per-key work -- streaming the head's K_lr, the MMA tile,
// the compares -- dominates), and a CTA with two row tiles (17..27 rows) takes about 1.75 times
// as long as one with a single tile.  So: with one tile, the most rows (fewest CTAs, fewest
// waves); with two tiles, the fewest rows that reach their fewest waves; two tiles only when
// that saves at least 10 % (waves x 175 against waves x 100), and only when the low-rank dim
// leaves room in registers.
int estimate_rows_per_cta(int64_t BH, int64_t NB, bool two_tiles_ok) {
  constexpr int64_t kSMs = 152;
  auto waves = [&](int r) { return (BH * ((NB + r - 1) / r) + kSMs - 1) / kSMs; };
  const int one = NB < kRows ? static_cast<int>(NB < 1 ? 1 : NB) : kRows;
  if (!two_tiles_ok || NB <= kRows) return one;
  const int64_t w1 = waves(one);
  int two = kMaxRows2;
  for (int r = kMaxRows2; r > kRows; --r)
    if (waves(r) == waves(kMaxRows2)) two = r;   // the fewest rows with the fewest waves
  return waves(two) * 175 * 10 <= w1 * 100 * 9 ? two : one;
}

// k == N: every key of every block, ascending.
__global__ void arange_kernel(int32_t* __restrict__ idx, int64_t rows, int64_t k) {
  const int64_t total = rows * k;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    idx[i] = static_cast<int32_t>(i % k);
}

template <int R, int MT>
cudaError_t launch_rt(const EstimateParams& p, int rows, cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(rows) * kBins * sizeof(uint32_t);
  cudaError_t e = cudaFuncSetAttribute(estimate_topk_kernel<R, MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>((p.NB + rows - 1) / rows), static_cast<unsigned>(p.BH));
  ProfScope prof("estimate_topk", stream);
  estimate_topk_kernel<R, MT><<<grid, kThreads, smem, stream>>>(p.q_lr, p.k_lr, p.idx, static_cast<int>(p.N),
                                                                 static_cast<int>(p.NB), static_cast<int>(p.topk), rows,
                                                                 p.krow, p.rowptr, p.status);
  return cudaGetLastError();
}

template <int R>
cudaError_t launch_r(const EstimateParams& p, cudaStream_t stream) {
  const int rows = estimate_rows_per_cta(p.BH, p.NB, R <= 32);
  return rows > kRows ? launch_rt<R, (R <= 32 ? 2 : 1)>(p, rows, stream) : launch_rt<R, 1>(p, rows, stream);
}

}  // namespace

cudaError_t launch_estimate_mass_k(const MassParams& p, cudaStream_t stream) {
  cudaError_t e;
  switch (p.r) {
    case 16: e = launch_mass_r<16>(p, stream); break;
    case 32: e = launch_mass_r<32>(p, stream); break;
    case 48: e = launch_mass_r<48>(p, stream); break;
    case 64: e = launch_mass_r<64>(p, stream); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  {
    ProfScope prof("csr_scan", stream);
    csr_scan_kernel<<<1, 1024, 0, stream>>>(p.krow, p.BH * p.NB, p.rowptr);
  }
  if (p.order) return launch_csr_order(p.rowptr, p.BH * p.NB, p.N, p.order, stream);
  return cudaGetLastError();
}

cudaError_t launch_csr_order(const int64_t* rowptr, int64_t rows, int64_t N, int32_t* order, cudaStream_t stream) {
  const int64_t nclass = (N + 127) / 128 + 1;
  if (nclass > 4096) return cudaErrorInvalidValue;
  ProfScope prof("csr_order", stream);
  csr_order_kernel<<<1, 1024, 0, stream>>>(rowptr, rows, static_cast<int>(nclass), order);
  return cudaGetLastError();
}

cudaError_t launch_estimate_topk(const EstimateParams& p, cudaStream_t stream) {
  if (p.topk == p.N && !p.krow) {
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
