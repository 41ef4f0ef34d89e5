// Backward of DENSE blocks (every key selected, k = N: the per-block sparse/dense switch of the
// DSV pages, German summary section 2A stage 2, taken to a whole head), without partial rows.
//
// With every query block selecting every key, a tile of 128 consecutive keys sees the same
// queries in every block, so dK and dV of the tile are dense products accumulated in tensor
// memory over all query blocks (key-stationary), in block order; nothing per (block, key)
// leaves the SM.  dQ comes from the query-centric main kernel in its dense, dQ-only form
// (dsv_bwd_tc.cu), and D_i = dO_i . O_i from dense_delta_kernel below.  Per query block b of
// the head, with keys on the MMA's M dimension:
//     S^T = K_t . Q_b^T,   dP^T = V_t . dO_b^T                   (M=128, N=64,  K=d)
//     P = exp2(S scale log2e - LSE2_b),  dS = P (dP - D_b)       (compute warps, fp32)
//     dV_t += P^T . dO_b,  dK_t += dS^T . Q_b                     (M=128, N=d,   K=64)
// Roles (416 threads): warps 0-7 compute P and dS (two warps per TMEM lane quadrant, each on 32
// of the 64 query columns; thread = key lane); warps 8, 10, 11 and 12 load the key tile once and
// then each query block's Q, dO, LSE and D into a three-stage ring with cp.async (contiguous rows,
// a quarter of every tile per warp: one warp alone cannot keep enough loads in flight); one
// thread of warp 9 issues the MMAs (S / dP of block b + 1 ahead of the gradients of block b,
// into two TMEM buffers).  At the end warps 0-3 move dK (times the scale) and dV out of tensor
// memory through shared memory and write them row by row.  Every wait is bounded.
#include "dsv_common.cuh"
#include "dsv_internal.h"
#include "dsv_tc.cuh"

namespace dsv {
namespace {

constexpr int kKeys = 128;     // keys per CTA (the MMA's M)
constexpr int kProducers = 4;  // warp 8 and warps 10.. copy tiles
constexpr int kThreads = 320 + 32 * (kProducers - 1);
constexpr int kCompute = 256;
constexpr uint32_t kWaitLimit = 1u << 22;
// TMEM columns: S^T (two buffers of 64), dP^T (two of 64), dV_t (d), dK_t (d)
constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kTmemCols = 512;

template <int D>
struct DSm {
  static constexpr int BLK = D / 64;
  static constexpr int T64 = BLK * 64 * 128;      // a [64 rows][D] tile (Q_b or dO_b)
  static constexpr int KV = BLK * kKeys * 128;    // a [128 rows][D] tile (K_t or V_t)
  static constexpr int P = kKeys * 128;           // [128 keys][64 q] bf16
  static constexpr int QST = 3;                    // Q / dO stages
  static constexpr int OFF_K = 0, OFF_V = KV, OFF_Q = 2 * KV, OFF_DO = OFF_Q + QST * T64,
                       OFF_P = OFF_DO + QST * T64,
                       OFF_LD = OFF_P + 2 * P,  // per stage: LSE (64 floats), then D (64 floats)
                       TOTAL = OFF_LD + QST * 2 * 64 * 4;
  static_assert(4 * T64 >= kKeys * 2 * D * 2, "the epilogue stages dK and dV in the Q / dO stages");
};

struct DBars {
  uint64_t kv_full;                  // K_t and V_t landed
  uint64_t q_full[3], q_empty[3];    // per stage: Q_b, dO_b, LSE_b, D_b landed / no longer read
  uint64_t s_full[2], s_empty[2];    // per TMEM buffer: S^T, dP^T ready / read
  uint64_t p_full, pds_empty;        // P, dS written / read by the gradient MMAs
  uint64_t acc_full;                 // last dV_t, dK_t update done
  uint64_t drain;                    // every MMA issued is done
};

DSV_DEVICE void cp_async_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(bar) : "memory");
}

// tile rows [r_begin, r_end) of a 128-byte-swizzled tile of tile_rows rows from rows row0 + r of a
// [*][D] bf16 tensor (rows >= limit are zero-filled); whole rows per warp-wide copy
template <int D>
DSV_DEVICE void copy_tile(uint32_t dst, int tile_rows, const bf16* base, int64_t row0, int r_begin, int r_end,
                          int64_t limit, int lane) {
  constexpr int LPR = D / 8, RPI = 32 / LPR;
  const int sub = lane % LPR, rsub = lane / LPR;
  const int e = sub * 8;
  for (int r0 = r_begin; r0 < r_end; r0 += RPI) {
    const int row = r0 + rsub;
    const bool ok = row0 + row < limit;
    cp_async_16(dst + (e >> 6) * (tile_rows * 128) + tc::sw128(row, e & 63), base + (ok ? row0 + row : 0) * D + e, ok);
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
dense_dkdv_kernel(const bf16* __restrict__ q, const bf16* __restrict__ k, const bf16* __restrict__ v,
                  const bf16* __restrict__ d_o, const float* __restrict__ lse, const float* __restrict__ delta,
                  bf16* __restrict__ dk, bf16* __restrict__ dv, int64_t N, float scale, float scale_log2,
                  unsigned int* status) {
  using S = DSm<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ __align__(8) DBars bars;
  __shared__ uint32_t tmem_base_s;
  __shared__ int fail_s;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t bh = blockIdx.y;
  const int64_t key0 = static_cast<int64_t>(blockIdx.x) * kKeys;
  const int NB = static_cast<int>(N / 64);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sK = sbase + S::OFF_K, sV = sbase + S::OFF_V, sQ = sbase + S::OFF_Q, sDO = sbase + S::OFF_DO;
  const uint32_t sP = sbase + S::OFF_P, sDS = sP + S::P;
  float* ld_s = reinterpret_cast<float*>(smem + S::OFF_LD);  // [stage][LSE 64, D 64]
  auto bar = [](uint64_t& b) { return smem_u32(&b); };

  if (sbase & 1023u) {  // swizzled tiles need 1024-byte alignment
    if (tid == 0) flag_status(status, kStatusTimeout);
    return;
  }
  if (warp == 0) {
    tc::tmem_alloc(smem_u32(&tmem_base_s), kTmemCols);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    tc::mbar_init(bar(bars.kv_full), 32 * kProducers);
    for (int s = 0; s < S::QST; ++s) {
      tc::mbar_init(bar(bars.q_full[s]), 32 * kProducers);
      tc::mbar_init(bar(bars.q_empty[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(bar(bars.s_full[s]), 1);
      tc::mbar_init(bar(bars.s_empty[s]), kCompute);
    }
    tc::mbar_init(bar(bars.p_full), kCompute);
    tc::mbar_init(bar(bars.pds_empty), 1);
    tc::mbar_init(bar(bars.acc_full), 1);
    tc::mbar_init(bar(bars.drain), 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    fail_s = 0;
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  const int64_t hrow = bh * N;  // first row of this head

  if (warp == 8 || warp >= 10) {
    // ================================================================ producers (cp.async), each
    // on its own quarter of every tile's rows
    const int pr = warp == 8 ? 0 : warp - 9;
    const int kr0 = pr * (kKeys / kProducers), qr0 = pr * (64 / kProducers);
    copy_tile<D>(sK, kKeys, k + hrow * D, key0, kr0, kr0 + kKeys / kProducers, N, lane);
    copy_tile<D>(sV, kKeys, v + hrow * D, key0, kr0, kr0 + kKeys / kProducers, N, lane);
    cp_async_arrive(bar(bars.kv_full));
    bool ok_run = true;
    for (int b = 0; b < NB && ok_run; ++b) {
      const int st = b % S::QST;
      if (b >= S::QST) ok_run = tc::mbar_wait(bar(bars.q_empty[st]), ((b / S::QST) - 1) & 1, kWaitLimit);
      ok_run = __all_sync(0xffffffffu, ok_run);
      if (!ok_run) break;
      copy_tile<D>(sQ + st * S::T64, 64, q + hrow * D, static_cast<int64_t>(b) * 64, qr0, qr0 + 64 / kProducers, N,
                   lane);
      copy_tile<D>(sDO + st * S::T64, 64, d_o + hrow * D, static_cast<int64_t>(b) * 64, qr0, qr0 + 64 / kProducers,
                   N, lane);
      // LSE and D of the block's 64 queries: 16 lanes x 16 bytes each
      const uint32_t ldst = smem_u32(ld_s + st * 128);
      if (pr == 0) {
        if (lane < 16) cp_async_16(ldst + lane * 16, lse + hrow + b * 64 + lane * 4, true);
        else cp_async_16(ldst + 256 + (lane - 16) * 16, delta + hrow + b * 64 + (lane - 16) * 4, true);
      }
      cp_async_arrive(bar(bars.q_full[st]));
    }
    cp_async_wait<0>();
    if (!ok_run && lane == 0) atomicOr(&fail_s, 1);
  } else if (warp == 9) {
    // ================================================================ MMA issue (one thread)
    if (lane == 0) {
      constexpr uint32_t idS = tc::idesc_bf16(128, 64, 0, 0);   // S^T, dP^T: both K-major
      constexpr uint32_t idKV = tc::idesc_bf16(128, D, 0, 1);   // dV_t, dK_t: A K-major, B MN-major
      auto issue_s = [&](int b) {  // S^T and dP^T of block b into TMEM buffer b & 1
        tc::tc_fence_after();
        const int st = b % S::QST;
        const uint32_t col = (b & 1) * 64;
#pragma unroll
        for (int j = 0; j < D / 16; ++j) {
          const uint32_t off_a = (j >> 2) * (kKeys * 128) + (j & 3) * 32;
          const uint32_t off_b = (j >> 2) * (64 * 128) + (j & 3) * 32;
          tc::mma_ss(tmem + kColS + col, tc::smem_desc(sK + off_a, 16, 1024),
                     tc::smem_desc(sQ + st * S::T64 + off_b, 16, 1024), idS, j > 0 ? 1u : 0u);
          tc::mma_ss(tmem + kColDP + col, tc::smem_desc(sV + off_a, 16, 1024),
                     tc::smem_desc(sDO + st * S::T64 + off_b, 16, 1024), idS, j > 0 ? 1u : 0u);
        }
        tc::mma_commit(bar(bars.s_full[b & 1]));
      };
      auto s_ready = [&](int b) {
        return tc::mbar_wait(bar(bars.q_full[b % S::QST]), (b / S::QST) & 1, kWaitLimit) &&
               (b < 2 || tc::mbar_wait(bar(bars.s_empty[b & 1]), ((b >> 1) - 1) & 1, kWaitLimit));
      };
      bool ok_run = tc::mbar_wait(bar(bars.kv_full), 0, kWaitLimit) && s_ready(0);
      if (ok_run) issue_s(0);
      for (int b = 0; b < NB && ok_run; ++b) {
        if (b + 1 < NB) {
          ok_run = s_ready(b + 1);
          if (!ok_run) break;
          issue_s(b + 1);
        }
        ok_run = tc::mbar_wait(bar(bars.p_full), b & 1, kWaitLimit);
        if (!ok_run) break;
        tc::tc_fence_after();
        const int st = b % S::QST;
#pragma unroll
        for (int j = 0; j < 4; ++j) {  // K = 64 queries
          tc::mma_ss(tmem + kColDV, tc::smem_desc(sP + j * 32, 16, 1024),
                     tc::smem_desc(sDO + st * S::T64 + j * 2048, 64 * 128, 1024), idKV, (b > 0 || j > 0) ? 1u : 0u);
          tc::mma_ss(tmem + kColDV + D, tc::smem_desc(sDS + j * 32, 16, 1024),
                     tc::smem_desc(sQ + st * S::T64 + j * 2048, 64 * 128, 1024), idKV, (b > 0 || j > 0) ? 1u : 0u);
        }
        tc::mma_commit(bar(bars.pds_empty));
        tc::mma_commit(bar(bars.q_empty[st]));
        if (b == NB - 1) tc::mma_commit(bar(bars.acc_full));
      }
      if (!ok_run) atomicOr(&fail_s, 1);
      tc::mma_commit(bar(bars.drain));
      if (!tc::mbar_wait(bar(bars.drain), 0, kWaitLimit)) atomicOr(&fail_s, 1);
    }
  } else {
    // ================================================================ P and dS (threads 0..255)
    const int t = tid & 127;          // key lane
    const int hq = tid >> 7;          // query columns [32 hq, 32 hq + 32)
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const bool valid = key0 + t < N;
    bool ok_run = true;
    for (int b = 0; b < NB; ++b) {
      const int st = b & 1;
      ok_run = ok_run && tc::mbar_wait(bar(bars.s_full[st]), (b >> 1) & 1, kWaitLimit);
      tc::tc_fence_after();
      uint32_t sr[2][16], dr[2][16];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        tc::tmem_ld16(tmem + lane_base + kColS + st * 64 + hq * 32 + h * 16, sr[h]);
        tc::tmem_ld16(tmem + lane_base + kColDP + st * 64 + hq * 32 + h * 16, dr[h]);
      }
      tc::tmem_wait_ld();
      tc::tc_fence_before();
      tc::mbar_arrive(bar(bars.s_empty[st]));
      const float* lsb = ld_s + (b % S::QST) * 128;
      uint32_t pw[16], dw[16];  // packed bf16 pairs of P and dS
#pragma unroll
      for (int i4 = 0; i4 < 8; ++i4) {
        const float4 l4 = reinterpret_cast<const float4*>(lsb)[hq * 8 + i4];
        const float4 d4 = reinterpret_cast<const float4*>(lsb + 64)[hq * 8 + i4];
        const float ll[4] = {l4.x * kLog2e, l4.y * kLog2e, l4.z * kLog2e, l4.w * kLog2e};
        const float dd[4] = {d4.x, d4.y, d4.z, d4.w};
        float pv[4], dv4[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = i4 * 4 + u;
          const float sv = __uint_as_float(sr[i >> 4][i & 15]);
          const float dpv = __uint_as_float(dr[i >> 4][i & 15]);
          pv[u] = valid ? fast_exp2(sv * scale_log2 - ll[u]) : 0.f;
          dv4[u] = pv[u] * (dpv - dd[u]);
        }
        pw[i4 * 2] = pack_bf16x2(pv[0], pv[1]);
        pw[i4 * 2 + 1] = pack_bf16x2(pv[2], pv[3]);
        dw[i4 * 2] = pack_bf16x2(dv4[0], dv4[1]);
        dw[i4 * 2 + 1] = pack_bf16x2(dv4[2], dv4[3]);
      }
      if (b >= 1) ok_run = ok_run && tc::mbar_wait(bar(bars.pds_empty), (b - 1) & 1, kWaitLimit);
      const uint32_t prow = sP + t * 128, drow = sDS + t * 128;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        const int ch = hq * 4 + cc;
        const uint32_t off = ((ch ^ t) & 7) << 4;
        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(prow + off), "r"(pw[cc * 4]), "r"(pw[cc * 4 + 1]),
                     "r"(pw[cc * 4 + 2]), "r"(pw[cc * 4 + 3]));
        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(drow + off), "r"(dw[cc * 4]), "r"(dw[cc * 4 + 1]),
                     "r"(dw[cc * 4 + 2]), "r"(dw[cc * 4 + 3]));
      }
      tc::fence_async_shared();
      tc::tc_fence_before();
      tc::mbar_arrive(bar(bars.p_full));
    }
    if (!ok_run) atomicOr(&fail_s, 1);
    // ---- epilogue (warps 0-3, one key lane each): dK_t (times the scale) and dV_t as bf16 rows,
    // staged in the Q / dO stages (free once the last gradients are done), then written out
    // coalesced
    if (warp < 4) {
      ok_run = ok_run && tc::mbar_wait(bar(bars.acc_full), 0, kWaitLimit);
      if (!ok_run) atomicOr(&fail_s, 1);
    }
  }
  __syncthreads();
  const bool failed = fail_s != 0;
  if (!failed && warp < 4) {
    tc::tc_fence_after();
    const int t = tid;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    uint8_t* stage = smem + S::OFF_Q;  // [128 keys][dK row, dV row]: 4 D bytes per key
#pragma unroll 1
    for (int part = 0; part < 2 * D / 16; ++part) {  // 16-column parts: dV first, then dK
      uint32_t r[16];
      tc::tmem_ld16(tmem + lane_base + kColDV + part * 16, r);
      tc::tmem_wait_ld();
      const bool is_dk = part >= D / 16;
      const float mult = is_dk ? scale : 1.f;
      uint32_t w[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        w[i] = pack_bf16x2(__uint_as_float(r[2 * i]) * mult, __uint_as_float(r[2 * i + 1]) * mult);
      const int col = (part % (D / 16)) * 16;  // first column of this part within the row
      uint4* dst = reinterpret_cast<uint4*>(stage + t * (4 * D) + (is_dk ? 0 : 2 * D) + col * 2);
      dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
      dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
    asm volatile("bar.sync 1, 128;\n" ::: "memory");
    // rows key0 + r (r < 128, key < N): dK from stage[r][0, 2 D), dV from stage[r][2 D, 4 D)
    constexpr int VPR = D / 8;  // 16-byte vectors per output row
    for (int i = t; i < kKeys * 2 * VPR; i += 128) {
      const int r = i / (2 * VPR), rest = i % (2 * VPR);
      const int which = rest / VPR, vec = rest % VPR;  // 0: dK, 1: dV
      if (key0 + r >= N) continue;
      const uint4 val = *reinterpret_cast<const uint4*>(stage + r * (4 * D) + which * (2 * D) + vec * 16);
      bf16* out = (which ? dv : dk) + (hrow + key0 + r) * D;
      reinterpret_cast<uint4*>(out)[vec] = val;
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (fail_s && tid == 0) flag_status(status, kStatusTimeout);
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// D_i = dO_i . O_i for every row (dense blocks; the sparse main kernel forms it per block itself):
// a warp per row group, 16-byte loads, fp32 sums in a fixed order.
template <int D>
__global__ void dense_delta_kernel(const bf16* __restrict__ d_o, const bf16* __restrict__ o, float* __restrict__ delta,
                                   int64_t rows) {
  constexpr int LPR = D / 8;  // lanes per row (16-byte vectors)
  constexpr int RPW = 32 / LPR;
  const int lane = threadIdx.x & 31;
  const int64_t warp_g = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t r0 = warp_g * RPW; r0 < rows; r0 += nwarps * RPW) {
    const int64_t row = r0 + lane / LPR;
    float acc = 0.f;
    if (row < rows) {
      const uint4 a = reinterpret_cast<const uint4*>(d_o + row * D)[lane % LPR];
      const uint4 b = reinterpret_cast<const uint4*>(o + row * D)[lane % LPR];
      const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) acc += bf16_lo(av[u]) * bf16_lo(bv[u]) + bf16_hi(av[u]) * bf16_hi(bv[u]);
    }
#pragma unroll
    for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (row < rows && lane % LPR == 0) delta[row] = acc;
  }
}

template <int D>
cudaError_t launch_d(const BwdParams& p, float* delta, cudaStream_t stream) {
  {
    ProfScope prof("dense_delta", stream);
    const int64_t rows = p.BH * p.N;
    int64_t blocks = (rows / (32 / (D / 8)) + 7) / 8;
    if (blocks > 152 * 32) blocks = 152 * 32;
    if (blocks < 1) blocks = 1;
    dense_delta_kernel<D><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p.d_o, p.o, delta, rows);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const int smem = DSm<D>::TOTAL;
  cudaError_t e = cudaFuncSetAttribute(dense_dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>((p.N + kKeys - 1) / kKeys), static_cast<unsigned>(p.BH));
  ProfScope prof("dense_dkdv", stream);
  dense_dkdv_kernel<D><<<grid, kThreads, smem, stream>>>(p.q, p.k, p.v, p.d_o, p.lse, delta, p.dk, p.dv, p.N, p.scale,
                                                         p.scale * kLog2e, p.status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dense_dkdv(const BwdParams& p, float* delta, cudaStream_t stream) {
  switch (p.d) {
    case 64: return launch_d<64>(p, delta, stream);
    case 128: return launch_d<128>(p, delta, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dsv
