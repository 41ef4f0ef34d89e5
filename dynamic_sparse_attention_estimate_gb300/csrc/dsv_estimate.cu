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
template <int R, int MT, typename F>
DSV_DEVICE void for_each_group(const Frags<R> (&A)[MT], const bf16* __restrict__ kh, int N, int k_begin, int k_end,
                               int warp, int g, int t, F&& body) {
  int kbase = k_begin + warp * 32;
  if (kbase >= k_end) return;
  KeyFrags<R> cur, nxt;
  load_keys<R>(cur, kh, kbase, N, g, t);
  for (; kbase < k_end; kbase += kTileKeys) {
    const int knext = kbase + kTileKeys;
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

template <int LEVEL, int R, int MT>
DSV_DEVICE void hist_pass(const Frags<R> (&A)[MT], const bf16* __restrict__ kh, int N, uint32_t* hist, RowState* rs,
                          int nrows, int warp, int g, int t) {
  bool act[MT][2];
  uint32_t pre[MT][2];
  uint32_t* hrow[MT][2];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = kRows * mt + g + 8 * h;
      act[mt][h] = row < nrows && rs[row].level == LEVEL;
      pre[mt][h] = rs[row].prefix;
      hrow[mt][h] = hist + row * kBins;
    }
  for_each_group<R, MT>(A, kh, N, 0, N, warp, g, t, [&](int kbase, const float (&sc)[MT][4][4]) {
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int h = e >> 1;
        if (!act[mt][h]) continue;
        const uint32_t key = order_key(sc[mt][j][e]);
        if (LEVEL == 0) {
          atomicAdd(hrow[mt][h] + (key >> 21), 1u);
        } else if (LEVEL == 1) {
          if ((key >> 21) == pre[mt][h]) {
            atomicAdd(hrow[mt][h] + ((key >> 10) & 2047u), 1u);
            if (key & 1023u) atomicOr(&rs[kRows * mt + g + 8 * h].orbits, key & 1023u);
          }
        } else {
          if ((key >> 10) == pre[mt][h]) atomicAdd(hrow[mt][h] + (key & 1023u), 1u);
        }
      }
    }
  });
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
  if (tid < kMax) rs[tid] = RowState{0u, 0, tid < nrows ? row_k(tid) : k, 0u, 0, 0u};
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

  // ---- histogram passes; warp w resolves rows w and w + 16 after each
  auto resolve = [&](int level) {
#pragma unroll
    for (int q = 0; q < MT; ++q) {
      const int row = warp + kWarps * q;
      if (row < nrows && rs[row].level == level) {
        RowState s = rs[row];
        int bin, above, cnt;
        warp_find_bin(hist + row * kBins, level == 2 ? 1024 : kBins, s.rem, lane, bin, above, cnt);
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
        if (lane == 0) rs[row] = s;
      }
    }
  };
  auto next_level_pending = [&](int level) -> bool {
    if (tid == 0) pending = 0;
    __syncthreads();
    if (tid < nrows && rs[tid].level == level) atomicOr(&pending, 1);
    __syncthreads();
    const bool any = pending != 0;
    if (any)
      for (int i = tid; i < rows * kBins; i += kThreads) hist[i] = 0u;
    __syncthreads();
    return any;
  };

  hist_pass<0, R, MT>(A, kh, N, hist, rs, nrows, warp, g, t);
  __syncthreads();
  resolve(0);
  if (next_level_pending(1)) {
    hist_pass<1, R, MT>(A, kh, N, hist, rs, nrows, warp, g, t);
    __syncthreads();
    resolve(1);
    if (next_level_pending(2)) {
      hist_pass<2, R, MT>(A, kh, N, hist, rs, nrows, warp, g, t);
      __syncthreads();
      resolve(2);
    }
  }
  __syncthreads();

  // ---- emit, one segment of keys at a time
  uint32_t* gtb = hist;                      // [rows][kSegWords]
  uint32_t* eqb = hist + rows * kSegWords;   // [rows][kSegWords]
  uint32_t T[MT][2];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    T[mt][0] = rs[kRows * mt + g].T;
    T[mt][1] = rs[kRows * mt + g + 8].T;
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
            const int pos = 8 * j + 2 * t + (e & 1);
            const uint32_t key = order_key(sc[mt][j][e]);
            gtm[h] |= static_cast<uint32_t>(key > T[mt][h]) << pos;
            eqm[h] |= static_cast<uint32_t>(key == T[mt][h]) << pos;
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
