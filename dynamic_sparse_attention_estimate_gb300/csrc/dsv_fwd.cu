// Sparse attention forward over the selected keys (DSV, Spanish technical summary
// section 3: custom fused kernels for sparse attention; page 1 section 2A: only the
// critical KV pairs take part).
//
// One CTA = one query block (64 queries) of one head, 4 warps x 16 query rows.  The
// block's selected keys are processed in chunks of 64: their K and V rows are gathered
// from HBM/L2 by cp.async into swizzled shared memory (double buffered), S = Q K^T and
// O += P V run on the tensor cores (mma.sync m16n8k16, bf16 in, fp32 accumulate), and
// the softmax is online in fp32, base 2, with the scale folded in.
#include "dsv_common.cuh"
#include "dsv_internal.h"

#include <math_constants.h>

namespace dsv {
namespace {

constexpr int kChunk = 64;
constexpr int kThreads = 128;

template <int D>
struct FwdSmem {
  static constexpr int ROWB = D * 2;
  static constexpr int CH = ROWB / 16;
  static constexpr int Q_BYTES = 64 * ROWB;
  static constexpr int KV_BYTES = kChunk * ROWB;
  static constexpr int TOTAL = Q_BYTES + 4 * KV_BYTES;  // Q, K[2], V[2]
};

template <int D>
__global__ void __launch_bounds__(kThreads)
sparse_fwd_kernel(const bf16* __restrict__ q, const bf16* __restrict__ k, const bf16* __restrict__ v,
                  const int32_t* __restrict__ idx, bf16* __restrict__ o, float* __restrict__ lse,
                  int64_t N, int64_t NB, int64_t kk, float scale_log2, unsigned int* status) {
  using S = FwdSmem<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ int s_valid[2][kChunk];
  const uint32_t sQ = smem_u32(smem);
  const uint32_t sK0 = sQ + S::Q_BYTES;
  const uint32_t sV0 = sK0 + 2 * S::KV_BYTES;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int64_t bh = blockIdx.y, blk = blockIdx.x;
  const bf16* qb = q + (bh * N + blk * 64) * D;
  const bf16* kh = k + bh * N * D;
  const bf16* vh = v + bh * N * D;
  const int32_t* ib = idx + (bh * NB + blk) * kk;
  const int nchunks = static_cast<int>((kk + kChunk - 1) / kChunk);

  for (int i = tid; i < 64 * S::CH; i += kThreads) {
    const int row = i / S::CH, ch = i % S::CH;
    cp_async_16(sQ + swz<S::ROWB>(row, ch), qb + row * D + ch * 8, true);
  }

  auto load_chunk = [&](int c, int stage) {
    const uint32_t sK = sK0 + stage * S::KV_BYTES, sV = sV0 + stage * S::KV_BYTES;
    for (int i = tid; i < kChunk * S::CH; i += kThreads) {
      const int row = i / S::CH, ch = i % S::CH;
      const int64_t slot = static_cast<int64_t>(c) * kChunk + row;
      int64_t j = slot < kk ? static_cast<int64_t>(__ldg(ib + slot)) : -1;
      bool ok = j >= 0 && j < N;
      if (slot < kk && !ok && ch == 0) flag_status(status, kStatusBadIndex);
      if (ch == 0) s_valid[stage][row] = ok;
      const int64_t src = ok ? j : 0;
      cp_async_16(sK + swz<S::ROWB>(row, ch), kh + src * D + ch * 8, ok);
      cp_async_16(sV + swz<S::ROWB>(row, ch), vh + src * D + ch * 8, ok);
    }
  };

  load_chunk(0, 0);
  cp_async_commit();

  float acc[D / 8][4];
#pragma unroll
  for (int j = 0; j < D / 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
  float m_run[2] = {-CUDART_INF_F, -CUDART_INF_F};
  float l_run[2] = {0.f, 0.f};
  uint32_t qf[D / 16][4];

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
    if (c == 0) {
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        ldsm_x4(sQ + swz<S::ROWB>(warp * 16 + (lane & 15), ks * 2 + (lane >> 4)), qf[ks][0], qf[ks][1], qf[ks][2],
                qf[ks][3]);
    }
    const uint32_t sK = sK0 + stage * S::KV_BYTES, sV = sV0 + stage * S::KV_BYTES;

    // S = Q K^T  (16 x 64 per warp)
    float s[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
    for (int np = 0; np < 4; ++np) {
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(sK + swz<S::ROWB>(np * 16 + (lane & 7) + 8 * (lane >> 4), ks * 2 + ((lane >> 3) & 1)), b0, b1, b2, b3);
        mma_bf16_16816(s[2 * np], qf[ks], b0, b1);
        mma_bf16_16816(s[2 * np + 1], qf[ks], b2, b3);
      }
    }
    // mask, scale, row max
    float mx[2] = {m_run[0], m_run[1]};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int col = 8 * j + 2 * t + (e & 1);
        const bool ok = (static_cast<int64_t>(c) * kChunk + col < kk) && s_valid[stage][col];
        const float x = ok ? s[j][e] * scale_log2 : -CUDART_INF_F;
        s[j][e] = x;
        mx[e >> 1] = fmaxf(mx[e >> 1], x);
      }
    }
    float alpha[2], base[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
      mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
      base[h] = mx[h] == -CUDART_INF_F ? 0.f : mx[h];
      alpha[h] = fast_exp2(m_run[h] - base[h]);  // exp2(-inf) = 0 on the first chunk
      m_run[h] = mx[h];
      l_run[h] *= alpha[h];
    }
#pragma unroll
    for (int j = 0; j < D / 8; ++j) {
      acc[j][0] *= alpha[0]; acc[j][1] *= alpha[0];
      acc[j][2] *= alpha[1]; acc[j][3] *= alpha[1];
    }
    uint32_t pf[4][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float p0 = fast_exp2(s[j][0] - base[0]), p1 = fast_exp2(s[j][1] - base[0]);
      const float p2 = fast_exp2(s[j][2] - base[1]), p3 = fast_exp2(s[j][3] - base[1]);
      l_run[0] += p0 + p1;
      l_run[1] += p2 + p3;
      pf[j >> 1][(j & 1) * 2 + 0] = pack_bf16x2(p0, p1);
      pf[j >> 1][(j & 1) * 2 + 1] = pack_bf16x2(p2, p3);
    }
    // O += P V
#pragma unroll
    for (int kp = 0; kp < 4; ++kp) {
#pragma unroll
      for (int dn = 0; dn < D / 16; ++dn) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(sV + swz<S::ROWB>(kp * 16 + (lane & 7) + 8 * ((lane >> 3) & 1), dn * 2 + (lane >> 4)), b0, b1, b2,
                  b3);
        mma_bf16_16816(acc[2 * dn], pf[kp], b0, b1);
        mma_bf16_16816(acc[2 * dn + 1], pf[kp], b2, b3);
      }
    }
    __syncthreads();
  }

  // finalize: O = acc / l, LSE = (m + log2 l) ln 2
  float inv[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
    inv[h] = l_run[h] > 0.f ? 1.f / l_run[h] : 0.f;
  }
  bf16* ob = o + (bh * N + blk * 64 + warp * 16) * D;
#pragma unroll
  for (int j = 0; j < D / 8; ++j) {
    const int col = 8 * j + 2 * t;
    *reinterpret_cast<uint32_t*>(ob + g * D + col) = pack_bf16x2(acc[j][0] * inv[0], acc[j][1] * inv[0]);
    *reinterpret_cast<uint32_t*>(ob + (g + 8) * D + col) = pack_bf16x2(acc[j][2] * inv[1], acc[j][3] * inv[1]);
  }
  if (t == 0) {
    float* lb = lse + bh * N + blk * 64 + warp * 16;
#pragma unroll
    for (int h = 0; h < 2; ++h)
      lb[g + 8 * h] = l_run[h] > 0.f ? (m_run[h] + __log2f(l_run[h])) * kLn2 : -CUDART_INF_F;
  }
}

template <int D>
cudaError_t launch_d(const FwdParams& p, cudaStream_t stream) {
  const int smem = FwdSmem<D>::TOTAL;
  cudaError_t e = cudaFuncSetAttribute(sparse_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>(p.NB), static_cast<unsigned>(p.BH));
  ProfScope prof("sparse_fwd", stream);
  sparse_fwd_kernel<D><<<grid, kThreads, smem, stream>>>(p.q, p.k, p.v, p.idx, p.o, p.lse, p.N, p.NB, p.topk,
                                                          p.scale * kLog2e, p.status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_sparse_fwd(const FwdParams& p, cudaStream_t stream) {
  switch (p.d) {
    case 64: return launch_d<64>(p, stream);
    case 128: return launch_d<128>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dsv
