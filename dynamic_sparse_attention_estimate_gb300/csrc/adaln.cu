// Fused AdaLN: LayerNorm + modulation, forward and backward (AdaptiveLoad page, technical
// summary section 2B).  y = (x - mean) * rstd * (1 + scale[b]) + shift[b] per token, with
// mean and the biased variance over the D features and rstd = 1 / sqrt(var + eps).
//
// The row mean is sum * (1/D) corrected once by its exact FMA residual, which makes it exact for
// a constant row (whose normalised row is then exactly 0 and whose output is exactly the shift).
//
// Layout: a 256-thread CTA owns a tile of consecutive tokens of one sample.  The tile is
// contiguous in HBM and streams through shared-memory stages filled by bulk copies of the tensor
// memory accelerator (mbarrier completion, bounded waits).  A token's D features are D / 8
// 16-byte vectors spread over W warps (W = 1 while D <= 1024, up to 8 at D = 8192); the CTA's 8
// warps form 8 / W row groups that take the stage's tokens in turn (two at a time in the
// forward).  A token is read from shared memory once into registers for its passes (mean,
// variance, output); the reductions are warp shuffles plus, when W > 1, a shared-memory level
// across the row's warps behind a named barrier of that row group.  Elementwise arithmetic runs
// on packed fp32 pairs; the modulation is held as fp32 in shared memory.
//
// Backward: the statistics are recomputed from x (nothing is saved between the passes).  Per
// token dx = rstd * (g - mean(g) - xhat * mean(g * xhat)) with g = dy * (1 + scale); the
// modulation gradients d_scale = sum_n dy * xhat and d_shift = sum_n dy are accumulated per
// feature in registers by the lanes that own that feature over the CTA's tile (the (D tile,
// N tile) blocking: loads stay coalesced along D), reduced across the row groups in a fixed
// order, and written as one partial row per tile; a second kernel sums the tiles in a fixed
// order.  No float atomics: the results are bitwise reproducible.
#include "dsv_common.cuh"
#include "dsv_internal.h"
#include "dsv_tc.cuh"

namespace dsv {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxStages = 4;

struct RowGeom {
  int nvec;   // 16-byte vectors per row (D / 8)
  int W;      // warps per row
  int slab;   // vectors per warp: ceil(nvec / W)
  int RG;     // row groups per CTA: kWarps / W
};

DSV_DEVICE float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Barrier of the W warps that share a row (named barrier 1 + row group; barrier 0 is the
// CTA-wide one that releases a stage).
DSV_DEVICE void row_group_sync(int W, int rg) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(1 + rg), "r"(32 * W) : "memory");
}

// Sum of v over the W warps of this warp's row: a warp shuffle, then (W > 1) the row's W
// warp totals from shared memory in warp order.  Called by every warp of a row group the same
// number of times (it contains the row group's barrier when W > 1).
DSV_DEVICE float row_sum(float v, float* slot, int W, int rg, int warp, int lane) {
  v = warp_sum(v);
  if (W == 1) return v;
  if (lane == 0) slot[warp] = v;
  row_group_sync(W, rg);
  float t = 0.f;
  for (int p = 0; p < W; ++p) t += slot[rg * W + p];
  return t;
}

// ---------------------------------------------------------------- packed fp32 pairs
// Elementwise work runs on float pairs with Blackwell's packed f32x2 instructions (one
// instruction for two IEEE round-to-nearest FMAs / adds): a bf16x2 word unpacks to one pair.
DSV_DEVICE float2 pair(uint32_t w) { return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u)); }
DSV_DEVICE uint64_t as_u64(float2 v) { return *reinterpret_cast<uint64_t*>(&v); }
DSV_DEVICE float2 as_f2(uint64_t v) { return *reinterpret_cast<float2*>(&v); }
DSV_DEVICE float2 fma2(float2 a, float2 b, float2 c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;\n" : "=l"(d) : "l"(as_u64(a)), "l"(as_u64(b)), "l"(as_u64(c)));
  return as_f2(d);
}
DSV_DEVICE float2 add2(float2 a, float2 b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;\n" : "=l"(d) : "l"(as_u64(a)), "l"(as_u64(b)));
  return as_f2(d);
}
DSV_DEVICE float2 mul2(float2 a, float2 b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;\n" : "=l"(d) : "l"(as_u64(a)), "l"(as_u64(b)));
  return as_f2(d);
}
DSV_DEVICE float2 bcast(float v) { return make_float2(v, v); }
DSV_DEVICE uint32_t word(const uint4& u, int j) { return j == 0 ? u.x : j == 1 ? u.y : j == 2 ? u.z : u.w; }

// Sum of (a, b) over the W warps of this warp's row, both in one shuffle chain (see row_sum).
DSV_DEVICE float2 row_sum2(float2 v, float2* slot, int W, int rg, int warp, int lane) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    v.x += __shfl_xor_sync(0xffffffffu, v.x, o);
    v.y += __shfl_xor_sync(0xffffffffu, v.y, o);
  }
  if (W == 1) return v;
  if (lane == 0) slot[warp] = v;
  row_group_sync(W, rg);
  float2 t = make_float2(0.f, 0.f);
  for (int p = 0; p < W; ++p) {
    t.x += slot[rg * W + p].x;
    t.y += slot[rg * W + p].y;
  }
  return t;
}

// Row mean and rstd of a packed row (two passes over the registers: the mean, then the
// squares about it).  The mean is sum * (1/D) corrected once by its exact FMA residual
// sum - mean * D, which makes it exact whenever sum / D is representable (a constant row).
template <int VPL>
DSV_DEVICE void row_stats(const uint4 (&r)[VPL], const bool (&valid)[VPL], float* red0, float* red1, const RowGeom& g,
                          int rg, int warp, int lane, float Df, float invD, float eps, float& mean, float& rstd) {
  float2 s = make_float2(0.f, 0.f);
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    if (!valid[i]) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) s = add2(s, pair(word(r[i], j)));
  }
  const float sum = row_sum(s.x + s.y, red0, g.W, rg, warp, lane);
  const float m0 = sum * invD;
  mean = fmaf(fmaf(-m0, Df, sum), invD, m0);
  const float2 nm = bcast(-mean);
  float2 q = make_float2(0.f, 0.f);
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    if (!valid[i]) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 c = add2(pair(word(r[i], j)), nm);
      q = fma2(c, c, q);
    }
  }
  rstd = rsqrtf(fmaf(row_sum(q.x + q.y, red1, g.W, rg, warp, lane), invD, eps));
}

// Mean and rstd of two packed rows at once (two tokens per warp): both rows' sums share one
// shuffle chain (and, for W > 1, one row-group barrier), which halves the dependent latency per
// token.  Same arithmetic per row as row_stats.
template <int VPL>
DSV_DEVICE void row_stats_pair(const uint4 (&ra)[VPL], const uint4 (&rb)[VPL], const bool (&valid)[VPL], float2* red0,
                               float2* red1, const RowGeom& g, int rg, int warp, int lane, float Df, float invD,
                               float eps, float2& mean, float2& rstd) {
  float2 sa = make_float2(0.f, 0.f), sb = make_float2(0.f, 0.f);
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    if (!valid[i]) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      sa = add2(sa, pair(word(ra[i], j)));
      sb = add2(sb, pair(word(rb[i], j)));
    }
  }
  const float2 sum = row_sum2(make_float2(sa.x + sa.y, sb.x + sb.y), red0, g.W, rg, warp, lane);
  const float m0a = sum.x * invD, m0b = sum.y * invD;
  mean.x = fmaf(fmaf(-m0a, Df, sum.x), invD, m0a);
  mean.y = fmaf(fmaf(-m0b, Df, sum.y), invD, m0b);
  const float2 na = bcast(-mean.x), nb = bcast(-mean.y);
  float2 qa = make_float2(0.f, 0.f), qb = make_float2(0.f, 0.f);
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    if (!valid[i]) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 ca = add2(pair(word(ra[i], j)), na);
      const float2 cb = add2(pair(word(rb[i], j)), nb);
      qa = fma2(ca, ca, qa);
      qb = fma2(cb, cb, qb);
    }
  }
  const float2 q = row_sum2(make_float2(qa.x + qa.y, qb.x + qb.y), red1, g.W, rg, warp, lane);
  rstd.x = rsqrtf(fmaf(q.x, invD, eps));
  rstd.y = rsqrtf(fmaf(q.y, invD, eps));
}

// ---------------------------------------------------------------- tensor-memory-accelerator staging
// A CTA's tile of tokens is contiguous in HBM; it streams through NS shared-memory stages of R
// rows each, filled by bulk copies that complete on one mbarrier per stage.  Thread 0 issues the
// copies; after every warp has finished a stage (a CTA barrier) it refills that stage with the
// chunk NS ahead.  Waits are bounded: a copy that never lands sets the timeout status bit and
// the CTA winds down without storing, after a second bounded wait for its copies in flight.
DSV_DEVICE void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
}
DSV_DEVICE void bulk_load(uint32_t sdst, const void* gsrc, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n"
               ::"r"(sdst), "l"(gsrc), "r"(bytes), "r"(bar)
               : "memory");
}

struct Staging {
  int R;    // rows per stage (a multiple of the row groups)
  int NS;   // stages
};

// ---------------------------------------------------------------- forward
template <int VPL>
__global__ void __launch_bounds__(kThreads, 3)
adaln_fwd_kernel(const uint4* __restrict__ x, const uint4* __restrict__ scale, const uint4* __restrict__ shift,
                 uint4* __restrict__ y, int64_t N, RowGeom g, Staging st, float Df, float invD, float eps,
                 int64_t rows_per_tile, int64_t tiles_per_b, unsigned int* status) {
  // [NS][R][nvec] x rows, then the sample's modulation as fp32 pairs: (1 + scale) and shift,
  // each [4][nvec] (pair j of vector v at j * nvec + v: consecutive lanes, consecutive words)
  extern __shared__ __align__(128) uint4 sbuf[];
  __shared__ __align__(8) uint64_t full[kMaxStages];
  __shared__ float2 red[2][kWarps];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rg = warp / g.W, part = warp % g.W;
  const int64_t b = blockIdx.x / tiles_per_b, tile = blockIdx.x % tiles_per_b;
  const int64_t r0 = tile * rows_per_tile;
  const int64_t r1 = r0 + rows_per_tile < N ? r0 + rows_per_tile : N;
  const int nchunk = static_cast<int>((r1 - r0 + st.R - 1) / st.R);
  const size_t stage_vecs = static_cast<size_t>(st.R) * g.nvec;

  if (tid == 0) {
    for (int s = 0; s < st.NS; ++s) tc::mbar_init(smem_u32(&full[s]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();
  int issued = 0, waited = 0;   // chunks issued (thread 0) and chunks whose copy this thread saw land
  auto issue = [&](int c) {
    issued = c + 1;
    const int s = c % st.NS;
    const int64_t rs = r0 + static_cast<int64_t>(c) * st.R;
    const int64_t nr = r1 - rs < st.R ? r1 - rs : st.R;
    const uint32_t bytes = static_cast<uint32_t>(nr * g.nvec * 16);
    mbar_expect_tx(smem_u32(&full[s]), bytes);
    bulk_load(smem_u32(sbuf + s * stage_vecs), x + (b * N + rs) * g.nvec, bytes, smem_u32(&full[s]));
  };
  if (tid == 0)
    for (int c = 0; c < st.NS && c < nchunk; ++c) issue(c);

  float2* mod_s = reinterpret_cast<float2*>(sbuf + st.NS * stage_vecs);   // 1 + scale
  float2* mod_h = mod_s + 4 * g.nvec;                                      // shift
  for (int v = tid; v < g.nvec; v += kThreads) {
    const uint4 a = __ldg(scale + b * g.nvec + v), h = __ldg(shift + b * g.nvec + v);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      mod_s[j * g.nvec + v] = add2(pair(word(a, j)), bcast(1.f));
      mod_h[j * g.nvec + v] = pair(word(h, j));
    }
  }
  __syncthreads();

  int vec[VPL];
  bool valid[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int local = lane + 32 * i;
    vec[i] = part * g.slab + local;
    valid[i] = local < g.slab && vec[i] < g.nvec;
  }

  bool ok = true;
  for (int c = 0; c < nchunk; ++c) {
    const int s = c % st.NS;
    if (ok) ok = tc::mbar_wait(smem_u32(&full[s]), (c / st.NS) & 1);
    if (ok) waited = c + 1;
    const uint4* stage = sbuf + s * stage_vecs;
    const int64_t rs = r0 + static_cast<int64_t>(c) * st.R;
    // two tokens per warp: local rows lr and lr + RG of the stage (the same trip count for every
    // warp of a row group)
    for (int lr = rg; lr < st.R; lr += 2 * g.RG) {
      const int lr2 = lr + g.RG;
      const int64_t row_a = rs + lr, row_b = rs + lr2;
      const bool act_a = row_a < r1, act_b = lr2 < st.R && row_b < r1;
      uint4 xa[VPL], xb[VPL];
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        xa[i] = (act_a && valid[i]) ? stage[static_cast<size_t>(lr) * g.nvec + vec[i]] : make_uint4(0, 0, 0, 0);
        xb[i] = (act_b && valid[i]) ? stage[static_cast<size_t>(lr2) * g.nvec + vec[i]] : make_uint4(0, 0, 0, 0);
      }
      float2 mean, rstd;
      row_stats_pair<VPL>(xa, xb, valid, red[0], red[1], g, rg, warp, lane, Df, invD, eps, mean, rstd);
      if (ok) {
        // y = fma(xhat, 1 + scale, shift), xhat = fma(x, rstd, -mean rstd)
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          if (!(q ? act_b : act_a)) continue;
          const float m = q ? mean.y : mean.x, r = q ? rstd.y : rstd.x;
          const float2 rs2 = bcast(r), nmr = bcast(-m * r);
          uint4* yr = y + (b * N + (q ? row_b : row_a)) * g.nvec;
#pragma unroll
          for (int i = 0; i < VPL; ++i) {
            if (!valid[i]) continue;
            const uint4 xv = q ? xb[i] : xa[i];
            uint32_t o[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float2 xh = fma2(pair(word(xv, j)), rs2, nmr);
              const float2 v = fma2(xh, mod_s[j * g.nvec + vec[i]], mod_h[j * g.nvec + vec[i]]);
              o[j] = pack_bf16x2(v.x, v.y);
            }
            __stcs(yr + vec[i], make_uint4(o[0], o[1], o[2], o[3]));
          }
        }
      }
    }
    __syncthreads();   // every warp is done with stage s
    if (tid == 0 && ok && c + st.NS < nchunk) issue(c + st.NS);
  }
  if (!ok && lane == 0) flag_status(status, kStatusTimeout);
  // error path: before this CTA's shared memory can go away, wait (again bounded) for the copies
  // thread 0 issued that nobody saw land
  if (!ok && tid == 0)
    for (int cc = waited; cc < issued; ++cc) tc::mbar_wait(smem_u32(&full[cc % st.NS]), (cc / st.NS) & 1);
}

// ---------------------------------------------------------------- backward: dx + per-tile partials
// Two CTAs per SM up to three vectors per lane (at most 128 registers without spills).
template <int VPL>
__global__ void __launch_bounds__(kThreads, VPL <= 3 ? 2 : 1)
adaln_bwd_kernel(const uint4* __restrict__ x, const uint4* __restrict__ scale, const uint4* __restrict__ dy,
                 uint4* __restrict__ dx, float* __restrict__ part_out, unsigned int* __restrict__ tickets,
                 int tickets_n, int64_t N, RowGeom g, Staging st, int D, float Df, float invD, float eps,
                 int64_t rows_per_tile, int64_t tiles_per_b, unsigned int* status) {
  // [NS][2][R][nvec]: x rows then dy rows per stage, then (1 + scale) as fp32 pairs [4][nvec];
  // after the loop the stages hold the row groups' modulation-gradient partials [RG][2][D]
  extern __shared__ __align__(128) uint4 sbuf[];
  __shared__ __align__(8) uint64_t full[kMaxStages];
  __shared__ float red[2][kWarps];
  __shared__ float2 red2[kWarps];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rg = warp / g.W, part = warp % g.W;
  const int64_t b = blockIdx.x / tiles_per_b, tile = blockIdx.x % tiles_per_b;
  const int64_t r0 = tile * rows_per_tile;
  const int64_t r1 = r0 + rows_per_tile < N ? r0 + rows_per_tile : N;
  const int nchunk = static_cast<int>((r1 - r0 + st.R - 1) / st.R);
  const size_t half_vecs = static_cast<size_t>(st.R) * g.nvec;

  if (tid == 0) {
    for (int s = 0; s < st.NS; ++s) tc::mbar_init(smem_u32(&full[s]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();
  int issued = 0, waited = 0;   // chunks issued (thread 0) and chunks whose copy this thread saw land
  auto issue = [&](int c) {
    issued = c + 1;
    const int s = c % st.NS;
    const int64_t rs = r0 + static_cast<int64_t>(c) * st.R;
    const int64_t nr = r1 - rs < st.R ? r1 - rs : st.R;
    const uint32_t bytes = static_cast<uint32_t>(nr * g.nvec * 16);
    const uint32_t bar = smem_u32(&full[s]);
    mbar_expect_tx(bar, 2 * bytes);
    bulk_load(smem_u32(sbuf + (2 * s) * half_vecs), x + (b * N + rs) * g.nvec, bytes, bar);
    bulk_load(smem_u32(sbuf + (2 * s + 1) * half_vecs), dy + (b * N + rs) * g.nvec, bytes, bar);
  };
  if (tid == 0)
    for (int c = 0; c < st.NS && c < nchunk; ++c) issue(c);
  // the column-sum kernel may be scheduled once every CTA of this grid has started; it waits
  // for this grid's completion before reading anything
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  // the column-sum kernel's tickets start at zero (it runs after this kernel on the stream)
  if (blockIdx.x == 0)
    for (int i = tid; i < tickets_n; i += kThreads) tickets[i] = 0u;

  float2* mod_s = reinterpret_cast<float2*>(sbuf + st.NS * 2 * half_vecs);   // 1 + scale
  for (int v = tid; v < g.nvec; v += kThreads) {
    const uint4 a = __ldg(scale + b * g.nvec + v);
#pragma unroll
    for (int j = 0; j < 4; ++j) mod_s[j * g.nvec + v] = add2(pair(word(a, j)), bcast(1.f));
  }
  __syncthreads();

  int vec[VPL];
  bool valid[VPL];
  float2 acc_s[VPL][4], acc_b[VPL][4];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int local = lane + 32 * i;
    vec[i] = part * g.slab + local;
    valid[i] = local < g.slab && vec[i] < g.nvec;
#pragma unroll
    for (int j = 0; j < 4; ++j) acc_s[i][j] = acc_b[i][j] = make_float2(0.f, 0.f);
  }

  bool ok = true;
  for (int c = 0; c < nchunk; ++c) {
    const int s = c % st.NS;
    if (ok) ok = tc::mbar_wait(smem_u32(&full[s]), (c / st.NS) & 1);
    if (ok) waited = c + 1;
    const uint4* sx = sbuf + (2 * s) * half_vecs;
    const uint4* sd = sbuf + (2 * s + 1) * half_vecs;
    const int64_t rs = r0 + static_cast<int64_t>(c) * st.R;
    for (int lr = rg; lr < st.R; lr += g.RG) {
      const int64_t row = rs + lr;
      const bool active = row < r1 && ok;
      uint4 cx[VPL], cd[VPL];
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        const size_t o = static_cast<size_t>(lr) * g.nvec + vec[i];
        cx[i] = (active && valid[i]) ? sx[o] : make_uint4(0, 0, 0, 0);
        cd[i] = (active && valid[i]) ? sd[o] : make_uint4(0, 0, 0, 0);
      }
      float mean, rstd;
      row_stats<VPL>(cx, valid, red[0], red[1], g, rg, warp, lane, Df, invD, eps, mean, rstd);
      // a padding row (not active) has x = dy = 0; its rstd may be inf when eps = 0, so it enters
      // through rs2 = 0 and nothing below multiplies an inf
      const float2 rs2 = bcast(active ? rstd : 0.f), nmr = bcast(active ? -mean * rstd : 0.f);
      float2 sg = make_float2(0.f, 0.f), sgx = make_float2(0.f, 0.f);
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        if (!valid[i]) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 d = pair(word(cd[i], j));
          const float2 xh = fma2(pair(word(cx[i], j)), rs2, nmr);
          const float2 gg = mul2(d, mod_s[j * g.nvec + vec[i]]);     // dy * (1 + scale)
          sg = add2(sg, gg);
          sgx = fma2(gg, xh, sgx);
          acc_s[i][j] = fma2(d, xh, acc_s[i][j]);
          acc_b[i][j] = add2(acc_b[i][j], d);
        }
      }
      const float2 m = row_sum2(make_float2(sg.x + sg.y, sgx.x + sgx.y), red2, g.W, rg, warp, lane);
      if (active) {
        // dx = rstd (g - mean g - xhat mean(g xhat)) = fma(rstd, g, fma(-rstd mean(g xhat), xhat, -rstd mean g))
        const float mg = m.x * invD, mgx = m.y * invD;
        const float2 a2 = bcast(rstd), b2 = bcast(-rstd * mgx), c2 = bcast(-rstd * mg);
        uint4* dxr = dx + (b * N + row) * g.nvec;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
          if (!valid[i]) continue;
          uint32_t o[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 d = pair(word(cd[i], j));
            const float2 xh = fma2(pair(word(cx[i], j)), rs2, nmr);
            const float2 gg = mul2(d, mod_s[j * g.nvec + vec[i]]);
            const float2 v = fma2(a2, gg, fma2(b2, xh, c2));
            o[j] = pack_bf16x2(v.x, v.y);
          }
          __stcs(dxr + vec[i], make_uint4(o[0], o[1], o[2], o[3]));
        }
      }
    }
    __syncthreads();   // every warp is done with stage s
    if (tid == 0 && ok && c + st.NS < nchunk) issue(c + st.NS);
  }
  if (!ok && lane == 0) flag_status(status, kStatusTimeout);
  // Error path (any thread of the CTA gave up on a stage): the tile's results are invalid and
  // the status word says so.  Thread 0 waits (again bounded) for the copies it issued that it
  // has not seen land, so that none can still write into the stages; then the CTA leaves
  // without reusing the stages for the partial sums (shared memory lives until its last thread
  // exits).
  if (__syncthreads_or(!ok)) {
    if (tid == 0)
      for (int cc = waited; cc < issued; ++cc) tc::mbar_wait(smem_u32(&full[cc % st.NS]), (cc / st.NS) & 1);
    return;
  }

  // row groups' partials -> shared memory (the stages are free: every copy has landed and every
  // warp passed the last barrier) -> one fixed-order sum per feature
  float* acc_smem = reinterpret_cast<float*>(sbuf);
  float* mine = acc_smem + static_cast<size_t>(rg) * 2 * D;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    if (!valid[i]) continue;
    float4* ps = reinterpret_cast<float4*>(mine + 8 * vec[i]);
    float4* pb = reinterpret_cast<float4*>(mine + D + 8 * vec[i]);
    ps[0] = make_float4(acc_s[i][0].x, acc_s[i][0].y, acc_s[i][1].x, acc_s[i][1].y);
    ps[1] = make_float4(acc_s[i][2].x, acc_s[i][2].y, acc_s[i][3].x, acc_s[i][3].y);
    pb[0] = make_float4(acc_b[i][0].x, acc_b[i][0].y, acc_b[i][1].x, acc_b[i][1].y);
    pb[1] = make_float4(acc_b[i][2].x, acc_b[i][2].y, acc_b[i][3].x, acc_b[i][3].y);
  }
  __syncthreads();
  float* out = part_out + static_cast<size_t>(blockIdx.x) * 2 * D;
  for (int f = tid; f < 2 * D; f += kThreads) {
    float t = 0.f;
    for (int r = 0; r < g.RG; ++r) t += acc_smem[static_cast<size_t>(r) * 2 * D + f];
    out[f] = t;
  }
}

// ---------------------------------------------------------------- backward: sum of the tiles
// One 256-thread CTA per (sample, 32 consecutive entries of the [2][D] partial row, group of
// tiles): warp w sums the group's tiles w, w + 8, ... for its 32 entries (one per lane,
// coalesced; eight loads issued before their in-order adds), the 8 warp sums are added in warp
// order and the group's sum is stored.  The group CTAs of an entry slab then take an integer
// ticket; the last to arrive (all groups' sums are visible to it) adds the kColGroups sums in
// group order and resets the ticket.  The order of every addition is fixed: the result does
// not depend on which CTA finishes last.
constexpr int kColGroups = 8;
__global__ void __launch_bounds__(kThreads)
adaln_colsum_kernel(const float* __restrict__ part, float* __restrict__ group_sums, unsigned int* __restrict__ tickets,
                    float* __restrict__ d_scale, float* __restrict__ d_shift, int D, int64_t tiles_per_b) {
  __shared__ float red[kWarps][33];
  __shared__ bool last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t slabs = (2 * D + 31) / 32;
  const int64_t grp = blockIdx.x % kColGroups;
  const int64_t bs = blockIdx.x / kColGroups;          // (sample, slab)
  const int64_t b = bs / slabs;
  const int f = static_cast<int>(bs % slabs) * 32 + lane;
  const int64_t t_lo = grp * tiles_per_b / kColGroups, t_hi = (grp + 1) * tiles_per_b / kColGroups;
  // launched early (programmatic dependent launch): wait until the backward grid has finished
  // and its partial rows are visible
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  float t = 0.f;
  if (f < 2 * D) {
    const float* p = part + static_cast<size_t>(b) * tiles_per_b * 2 * D + f;
    for (int64_t t0 = t_lo + warp; t0 < t_hi; t0 += 8 * kWarps) {
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int64_t tl = t0 + static_cast<int64_t>(u) * kWarps;
        v[u] = tl < t_hi ? p[static_cast<size_t>(tl) * 2 * D] : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) t += v[u];
    }
  }
  red[warp][lane] = t;
  __syncthreads();
  float* gs = group_sums + (static_cast<size_t>(b) * kColGroups) * 2 * D;
  if (warp == 0) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) s += red[w][lane];
    if (f < 2 * D) gs[grp * 2 * D + f] = s;
    __threadfence();
  }
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(tickets + bs, 1u) == kColGroups - 1;
  __syncthreads();
  if (!last || warp != 0) return;
  __threadfence();
  if (f < 2 * D) {
    float s = 0.f;
#pragma unroll
    for (int g2 = 0; g2 < kColGroups; ++g2) s += __ldcg(gs + g2 * 2 * D + f);
    if (f < D) d_scale[b * D + f] = s;
    else d_shift[b * D + (f - D)] = s;
  }
  if (lane == 0) tickets[bs] = 0u;
}

RowGeom geom_for(int64_t D) {
  RowGeom g;
  g.nvec = static_cast<int>(D / 8);
  g.W = 1;
  while ((g.nvec + g.W - 1) / g.W > 128) g.W *= 2;
  g.slab = (g.nvec + g.W - 1) / g.W;
  g.RG = kWarps / g.W;
  return g;
}

template <typename K>
cudaError_t pick_vpl(int slab, K k1, K k2, K k3, K k4, K* out) {
  const int vpl = (slab + 31) / 32;
  *out = vpl == 1 ? k1 : vpl == 2 ? k2 : vpl == 3 ? k3 : k4;
  return vpl >= 1 && vpl <= 4 ? cudaSuccess : cudaErrorInvalidValue;
}

// Rows per stage: about `stage_bytes` of rows (bytes_per_row each), a multiple of the row
// groups, no more than the tile needs.
Staging staging_for(const RowGeom& g, int64_t bytes_per_row, int64_t rows_per_tile, int64_t stage_bytes, int ns) {
  int64_t u = stage_bytes / (g.RG * bytes_per_row);
  const int64_t u_max = (rows_per_tile + g.RG - 1) / g.RG;
  if (u > u_max) u = u_max;
  if (u < 1) u = 1;
  Staging st;
  st.R = static_cast<int>(u * g.RG);
  st.NS = ns;
  return st;
}

// Forward stages hold two tokens per row group where rows are short enough (the pairs above).
constexpr int64_t kFwdStageBytes = 24 << 10, kBwdStageBytes = 24 << 10;
constexpr int kFwdStages = 2, kBwdStages = 3;

}  // namespace

AdalnTiling adaln_tiling(int64_t B, int64_t N, int64_t D, bool backward) {
  const RowGeom g = geom_for(D);
  AdalnTiling t;
  const int64_t target = backward ? kAdalnBwdTiles : kAdalnFwdTiles;
  int64_t per_b = (target + B - 1) / B;
  const int64_t max_tiles = (N + g.RG - 1) / g.RG;   // at least one row per row group
  if (per_b > max_tiles) per_b = max_tiles;
  if (per_b < 1) per_b = 1;
  t.rows_per_tile = (N + per_b - 1) / per_b;
  t.tiles_per_b = (N + t.rows_per_tile - 1) / t.rows_per_tile;
  // backward workspace: per-tile partial rows, per-group sums, one ticket per (sample, slab)
  t.partial_bytes = static_cast<size_t>(B * t.tiles_per_b) * 2 * D * sizeof(float);
  t.group_bytes = static_cast<size_t>(B * kColGroups) * 2 * D * sizeof(float);
  t.tickets = B * ((2 * D + 31) / 32);
  t.workspace_bytes = backward ? t.partial_bytes + t.group_bytes + static_cast<size_t>(t.tickets) * 4 : 0;
  return t;
}

cudaError_t launch_adaln_fwd(const AdalnParams& p, cudaStream_t stream) {
  const RowGeom g = geom_for(p.D);
  const AdalnTiling t = adaln_tiling(p.B, p.N, p.D, false);
  const Staging st = staging_for(g, 2 * p.D, t.rows_per_tile, kFwdStageBytes, kFwdStages);
  using Kern = void (*)(const uint4*, const uint4*, const uint4*, uint4*, int64_t, RowGeom, Staging, float, float,
                        float, int64_t, int64_t, unsigned int*);
  Kern k = nullptr;
  cudaError_t e = pick_vpl<Kern>(g.slab, adaln_fwd_kernel<1>, adaln_fwd_kernel<2>, adaln_fwd_kernel<3>,
                                 adaln_fwd_kernel<4>, &k);
  if (e != cudaSuccess) return e;
  const size_t smem = static_cast<size_t>(st.NS) * st.R * 2 * p.D + 2 * static_cast<size_t>(p.D) * sizeof(float);
  if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem))) !=
      cudaSuccess)
    return e;
  ProfScope prof("adaln_fwd", stream);
  k<<<static_cast<unsigned>(p.B * t.tiles_per_b), kThreads, smem, stream>>>(
      static_cast<const uint4*>(p.x), static_cast<const uint4*>(p.scale), static_cast<const uint4*>(p.shift),
      static_cast<uint4*>(p.y), p.N, g, st, static_cast<float>(p.D), 1.0f / static_cast<float>(p.D), p.eps,
      t.rows_per_tile, t.tiles_per_b, p.status);
  return cudaGetLastError();
}

cudaError_t launch_adaln_bwd(const AdalnParams& p, cudaStream_t stream) {
  const RowGeom g = geom_for(p.D);
  const AdalnTiling t = adaln_tiling(p.B, p.N, p.D, true);
  const Staging st = staging_for(g, 4 * p.D, t.rows_per_tile, kBwdStageBytes, kBwdStages);
  using Kern = void (*)(const uint4*, const uint4*, const uint4*, uint4*, float*, unsigned int*, int, int64_t, RowGeom,
                        Staging, int, float, float, float, int64_t, int64_t, unsigned int*);
  Kern k = nullptr;
  cudaError_t e = pick_vpl<Kern>(g.slab, adaln_bwd_kernel<1>, adaln_bwd_kernel<2>, adaln_bwd_kernel<3>,
                                 adaln_bwd_kernel<4>, &k);
  if (e != cudaSuccess) return e;
  // the stages (x and dy) also hold the row groups' partials after the loop: NS R >= 2 RG
  const size_t stages = static_cast<size_t>(st.NS) * st.R * 4 * p.D;
  const size_t partials = static_cast<size_t>(g.RG) * 2 * p.D * sizeof(float);
  const size_t smem = (stages > partials ? stages : partials) + static_cast<size_t>(p.D) * sizeof(float);
  float* group_sums = p.partial + t.partial_bytes / sizeof(float);
  unsigned int* tickets = reinterpret_cast<unsigned int*>(group_sums + t.group_bytes / sizeof(float));
  if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem))) !=
      cudaSuccess)
    return e;
  { ProfScope prof("adaln_bwd", stream);
  k<<<static_cast<unsigned>(p.B * t.tiles_per_b), kThreads, smem, stream>>>(
      static_cast<const uint4*>(p.x), static_cast<const uint4*>(p.scale), static_cast<const uint4*>(p.dy),
      static_cast<uint4*>(p.dx), p.partial, tickets, static_cast<int>(t.tickets), p.N, g, st, static_cast<int>(p.D),
      static_cast<float>(p.D), 1.0f / static_cast<float>(p.D), p.eps, t.rows_per_tile, t.tiles_per_b, p.status); }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int64_t slabs = (2 * p.D + 31) / 32;
  { ProfScope prof("adaln_colsum", stream);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.B * slabs * kColGroups));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, adaln_colsum_kernel, static_cast<const float*>(p.partial), group_sums, tickets,
                         p.d_scale, p.d_shift, static_cast<int>(p.D), t.tiles_per_b);
  if (e != cudaSuccess) return e; }
  return cudaGetLastError();
}

}  // namespace dsv
