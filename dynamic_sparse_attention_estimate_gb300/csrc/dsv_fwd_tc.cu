// Sparse attention forward on the tcgen05 tensor cores (DSV, Spanish technical summary
// section 3: custom fused kernels for sparse attention over the critical keys).
//
// One CTA = one query block (64 queries) of one head.  Its selected keys are processed in
// chunks of 128 with keys on the MMA's M dimension (the "transposed" formulation):
//     S^T[128 keys x 64 q]  = K_c . Q^T           (tcgen05, M=128, N=64, K=d)
//     O^T[d x 64 q]        += V_c^T . P^T         (tcgen05, M=d,   N=64, K=128)
// so both products keep M = 128 although a block has 64 queries (for d = 64 the PV operand
// carries an extra row of ones that yields the softmax row sums; see kOnesRow).
// Roles (192 threads at d = 64, 416 at d = 128):
//   warps 0-3  softmax (with warps 9-12 at d = 128, each pair of warps on one TMEM lane
//              quadrant taking 32 of the 64 query columns): a thread owns a key lane of S^T in
//              tensor memory (TMEM); it forms P = exp2(S scale log2e - m_q) and writes its part
//              of the key's P^T row (64 bf16, one 128-byte row) to shared memory as the B
//              operand of the PV product;
//   warp 4     producer (with warps 6-8 at d = 128, each taking 32 of a chunk's rows):
//              gathers the chunk's K and V rows with cp.async (16 bytes per copy, into
//              128-byte-swizzled tiles) into a ring of stages and lets the stage's mbarriers
//              count the copies' completion (cp.async.mbarrier.arrive), so it never waits for
//              its own copies; K and V of a stage have barriers of their own, so a chunk's K
//              rows are gathered as soon as the S^T product two chunks back has read the
//              stage's K, while its V rows wait for that chunk's PV product; keys past k or
//              out of range are zero-filled;
//   warp 5     one thread issues every MMA as soon as its inputs are ready, an S^T product
//              before a PV product when both are (the softmax waits for S^T, while a PV product
//              has until the softmax writes P^T two chunks later): it checks the S^T product's
//              barriers, then waits in the hardware, for a short bounded time, on the PV
//              product's.
// Dense blocks (every key selected, k = N): the DENSE instantiation reads no idx; chunk c holds
// keys 128 c .. 128 c + 127 (contiguous rows, the same arithmetic otherwise).
// The running max m_q is kept STALE: a chunk only triggers the cross-thread column max and
// an O/L rescale when one of its logits exceeds m_q by more than 8 (in log2 units; the
// first chunk always does).  Otherwise P <= 2^8, and softmax is invariant to the
// subtracted constant.  Row sums accumulate per key lane in TMEM and are reduced once.
#include "dsv_common.cuh"
#include "dsv_internal.h"
#include "dsv_tc.cuh"

#include <math_constants.h>

namespace dsv {
namespace {

constexpr int kChunk = 128;
// Producer warps per CTA.  Gathers of random rows are bound by the loads a warp keeps in
// flight: measured on this GPU, one issuing warp per SM moves about 3.8 TB/s of 256-byte rows
// out of L2 over the whole GPU, four move about 14 TB/s.  At d = 128 (one CTA per SM) four warps
// gather, each 32 of a chunk's 128 rows; at d = 64 (two CTAs per SM, registers for 192 threads
// each) one warp per CTA.  Producers are warp 4 and warps 6, 7, 8.
template <int D>
constexpr int kProducers = D == 128 ? 4 : 1;
// Softmax warps: four (one per TMEM lane quadrant, 64 query columns each) at d = 64; eight at
// d = 128 (two per quadrant, 32 query columns each: the softmax is the forward's critical path
// there, and two warps per quadrant halve each thread's chain of dependent work).  Softmax warps
// are 0-3 and, at d = 128, 9-12.
template <int D>
constexpr int kSoftmaxWarps = D == 128 ? 8 : 4;
template <int D>
constexpr int kThreadsFor = 32 * (1 + kProducers<D> + kSoftmaxWarps<D>);  // + the MMA warp
DSV_DEVICE int producer_index(int warp) { return warp == 4 ? 0 : (warp >= 6 && warp <= 8 ? warp - 5 : -1); }
DSV_DEVICE int softmax_index(int warp) { return warp < 4 ? warp : (warp >= 9 ? warp - 5 : -1); }
constexpr float kStaleLimit = 8.f;  // log2 units
constexpr uint32_t kWaitLimit = 1u << 22;
constexpr uint32_t kPollLimit = 1u << 24;  // rounds of bounded waits before giving up

// TMEM columns
constexpr uint32_t kColS0 = 0, kColS1 = 64, kColO = 128, kColL = 192, kTmemCols = 256;

template <int D, int NST>
struct Smem {
  static constexpr int BLK = D / 64;                 // 64-element column blocks
  static constexpr int Q_BYTES = BLK * 64 * 128;
  static constexpr int KV_BYTES = BLK * kChunk * 128;
  static constexpr int P_BYTES = kChunk * 128;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int OFF_V = OFF_K + NST * KV_BYTES;
  static constexpr int OFF_P = OFF_V + NST * KV_BYTES;
  // d = 64: a constant 16-key tile whose first M column is 1, the second 64-row block of the
  // PV product's A operand (see kOnesRow)
  static constexpr int OFF_ONES = OFF_P + 2 * P_BYTES;
  static constexpr int ONES_BYTES = D == 64 ? 2048 : 0;
  static constexpr int TOTAL = OFF_ONES + ONES_BYTES;
};

template <int NST>
struct Bars {
  uint64_t full_k[NST];     // cp.async completion: K rows of a stage (and Q, with stage 0) landed
  uint64_t full_v[NST];     // cp.async completion: V rows of a stage landed
  uint64_t empty_k[NST];    // MMA commit: the S^T product that read a stage's K rows is done
  uint64_t empty_v[NST];    // MMA commit: the PV product that read a stage's V rows is done
  uint64_t s_full[2];       // MMA commit: S^T in TMEM buffer b is ready
  uint64_t s_empty[2];      // softmax: S^T buffer b has been read
  uint64_t p_full[2];       // softmax: P^T tile b written
  uint64_t pv_done[2];      // MMA commit: PV with P^T tile b done
  uint64_t o_full;          // MMA commit: last PV done
  uint64_t drain;           // MMA commit at the end: every MMA the issuing thread started is done
};

// Barrier over the NT softmax threads.
template <int NT>
DSV_DEVICE void named_sync_softmax() { asm volatile("bar.sync 1, %0;\n" ::"r"(NT) : "memory"); }
// The same barrier, ORing a flag across the softmax threads (uniform result).
template <int NT>
DSV_DEVICE bool named_sync_or(bool v) {
  uint32_t r;
  asm volatile("{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, 1, %2, p;\n selp.u32 %0, 1, 0, q;\n}\n"
               : "=r"(r)
               : "r"(static_cast<uint32_t>(v)), "r"(NT)
               : "memory");
  return r != 0;
}

DSV_DEVICE bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for the phase with the given parity to complete, suspended in the hardware for at most
// about `ns` nanoseconds (returns false if it has not completed by then).
DSV_DEVICE bool mbar_try_wait_ns(uint32_t bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}
// Arrive on `bar` once all cp.async copies this thread issued so far have landed.
DSV_DEVICE void cp_async_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(bar) : "memory");
}

// d = 64: the PV product runs with M = 128 instead of 64 (the same tensor-core time: M = 64
// runs at half rate), its A operand extended past V_c^T by a row of ones, so TMEM lane 64 of
// O^T accumulates sum_keys P^T = the softmax row sums L, and the softmax threads keep no
// sums of their own.  L is then the sum of the same bf16 P values that weight V.
template <int D>
constexpr bool kOnesRow = D == 64;

// Column reduction over the key lanes of the softmax threads: each thread holds C consecutive
// query columns (v[c] for column c0 + c, c0 = C times its half); the four warps of a half cover
// the 128 key lanes.  Fixed order, so the result is deterministic.  Returns through red[64] in
// shared memory (visible after the trailing barrier).
template <bool MAX, int C, int NSMW>
DSV_DEVICE void column_reduce(float (&v)[C], float* red_w /*[NSMW][C]*/, float* red, int sw, int lane) {
  constexpr int K = C / 32;  // columns per lane after the exchange
  float cur[C];
#pragma unroll
  for (int i = 0; i < C; ++i) cur[i] = v[i];
  int n = C;
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) {  // after the step with mask m each lane keeps half its columns
    const bool upper = (lane & m) != 0;
    n >>= 1;
#pragma unroll
    for (int i = 0; i < C / 2; ++i) {
      if (i < n) {
        const float mine = upper ? cur[i + n] : cur[i];
        const float other = upper ? cur[i] : cur[i + n];
        const float recv = __shfl_xor_sync(0xffffffffu, other, m);
        cur[i] = MAX ? fmaxf(mine, recv) : mine + recv;
      }
    }
  }
#pragma unroll
  for (int i = 0; i < K; ++i) red_w[sw * C + K * lane + i] = cur[i];  // lane holds columns K lane + i
  named_sync_softmax<32 * NSMW>();
  const int hq = sw >> 2, loc = (sw & 3) * 32 + lane;
  if (loc < C) {
    float r = red_w[(hq * 4) * C + loc];
#pragma unroll
    for (int w = 1; w < 4; ++w) r = MAX ? fmaxf(r, red_w[(hq * 4 + w) * C + loc]) : r + red_w[(hq * 4 + w) * C + loc];
    red[hq * C + loc] = r;
  }
  named_sync_softmax<32 * NSMW>();
}

// CSR: per-block key counts from row offsets (and an optional launch order); otherwise k for
// every block, compiled without those loads.
template <int D, int NST, int MINB, bool CSR, bool DENSE>
__global__ void __launch_bounds__(kThreadsFor<D>, MINB)
sparse_fwd_tc_kernel(const bf16* __restrict__ q, const bf16* __restrict__ k, const bf16* __restrict__ v,
                     const int32_t* __restrict__ idx, const int64_t* __restrict__ rowptr,
                     const int32_t* __restrict__ order, bf16* __restrict__ o,
                     float* __restrict__ lse, int64_t N, int64_t NB, int64_t k_uniform, float scale_log2,
                     unsigned int* status) {
  using S = Smem<D, NST>;
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ __align__(8) Bars<NST> bars;
  __shared__ uint32_t tmem_base_s;
  // m_s is read as float4: every array here is 16-byte aligned explicitly
  __shared__ __align__(16) float m_s[64];
  __shared__ __align__(16) float alpha_s[64];
  __shared__ __align__(16) float red_w[4 * 64];
  __shared__ __align__(16) float red_s[64];
  __shared__ int flag_s[2];
  __shared__ int fail_s;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // this CTA's query block (in launch order when one is given), and its keys: k of them, or
  // its CSR row
  const int64_t lin = static_cast<int64_t>(blockIdx.y) * NB + blockIdx.x;
  const bool ordered = CSR && order != nullptr;
  const int64_t grow = ordered ? order[lin] : lin;
  const int64_t bh = ordered ? grow / NB : blockIdx.y, blk = ordered ? grow % NB : blockIdx.x;
  const int64_t kk = CSR ? rowptr[grow + 1] - rowptr[grow] : k_uniform;
  const int nchunks = static_cast<int>((kk + kChunk - 1) / kChunk);
  if (CSR && nchunks == 0) {  // a block with no keys: O = 0, LSE = -inf (uniform for the CTA, before any barrier)
    for (int i = tid; i < 64 * D / 8; i += kThreadsFor<D>)
      reinterpret_cast<uint4*>(o + (bh * N + blk * 64) * D)[i] = make_uint4(0u, 0u, 0u, 0u);
    if (tid < 64) lse[bh * N + blk * 64 + tid] = -CUDART_INF_F;
    return;
  }
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + S::OFF_Q, sK = sbase + S::OFF_K, sV = sbase + S::OFF_V, sP = sbase + S::OFF_P;
  const int32_t* ib = DENSE ? nullptr : idx + (CSR ? rowptr[grow] : grow * k_uniform);
  // the key at slot i (dense: the key position itself)
  auto key_at = [&](int64_t i) -> int32_t { return DENSE ? static_cast<int32_t>(i) : __ldg(ib + i); };
  auto bar = [](uint64_t& b) { return smem_u32(&b); };

  // the 128-byte swizzle of TMA and of the MMA descriptors both follow address bits, so the
  // tiles must start on 1024-byte boundaries
  if (sbase & 1023u) {
    if (tid == 0) flag_status(status, kStatusTimeout);
    return;
  }
  if (warp == 0) {
    tc::tmem_alloc(smem_u32(&tmem_base_s), kTmemCols);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    for (int s = 0; s < NST; ++s) {
      tc::mbar_init(bar(bars.full_k[s]), 32 * kProducers<D>);
      tc::mbar_init(bar(bars.full_v[s]), 32 * kProducers<D>);
      tc::mbar_init(bar(bars.empty_k[s]), 1);
      tc::mbar_init(bar(bars.empty_v[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(bar(bars.s_full[b]), 1);
      tc::mbar_init(bar(bars.s_empty[b]), 32 * kSoftmaxWarps<D>);
      tc::mbar_init(bar(bars.p_full[b]), 32 * kSoftmaxWarps<D>);
      tc::mbar_init(bar(bars.pv_done[b]), 1);
    }
    tc::mbar_init(bar(bars.o_full), 1);
    tc::mbar_init(bar(bars.drain), 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    flag_s[0] = flag_s[1] = 0;
    fail_s = 0;
  }
  if (tid < 64) m_s[tid] = -CUDART_INF_F;
  if (kOnesRow<D> && tid < 128) {  // 16 rows x 128 bytes, 128-byte swizzle: element 0 of row r
    const int row = tid >> 3, ch = tid & 7;  // sits in 16-byte chunk (r & 7)
    *reinterpret_cast<uint4*>(smem + S::OFF_ONES + tid * 16) = make_uint4(ch == (row & 7) ? 0x3f80u : 0u, 0u, 0u, 0u);
    tc::fence_async_shared();  // visible to the tensor core
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = tmem_base_s;

  if (producer_index(warp) >= 0) {
    // ================================================================ producers (cp.async)
    // Producer p copies the row groups g = p, p + NP, ... (rows 32 g .. 32 g + 31) of each chunk;
    // lane l holds the key index of row 32 g + l.  Whole rows, 16 bytes a copy.
    constexpr int NP = kProducers<D>, NG = 4 / NP;  // row groups per producer
    const int pidx = producer_index(warp);
    const bf16* qb = q + (bh * N + blk * 64) * D;
    const bf16* kh = k + bh * N * D;
    const bf16* vh = v + bh * N * D;
    if (pidx == 0) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int row = lane + 32 * h;
#pragma unroll
        for (int e = 0; e < D; e += 8)
          cp_async_16(sQ + (e >> 6) * (64 * 128) + tc::sw128(row, e & 63), qb + row * D + e, true);
      }
    }
    bool ok_run = true;
    int32_t nxt[NG];
    auto load_rows = [&](int c, int32_t (&rr)[NG]) {
#pragma unroll
      for (int h = 0; h < NG; ++h) {
        const int64_t slot = static_cast<int64_t>(c) * kChunk + 32 * (pidx + NP * h) + lane;
        rr[h] = (c < nchunks && slot < kk) ? key_at(slot) : -1;
      }
    };
    load_rows(0, nxt);
    for (int c = 0; c < nchunks && ok_run; ++c) {
      const int st = c % NST;
      int32_t cur[NG];
#pragma unroll
      for (int h = 0; h < NG; ++h) cur[h] = nxt[h];
      load_rows(c + 1, nxt);
      // K rows as soon as the S^T product two chunks back has read the stage's K, V rows once the
      // PV product has read its V (later: the softmax and P^T lie between them)
      if (c >= NST) ok_run = tc::mbar_wait(bar(bars.empty_k[st]), ((c / NST) - 1) & 1, kWaitLimit);
      ok_run = __all_sync(0xffffffffu, ok_run);
      if (!ok_run) break;
      const uint32_t dK = sK + st * S::KV_BYTES, dV = sV + st * S::KV_BYTES;
#pragma unroll
      for (int h = 0; h < NG; ++h) {  // validity of the rows this lane holds the index of
        const int64_t slot = static_cast<int64_t>(c) * kChunk + 32 * (pidx + NP * h) + lane;
        if (slot < kk && !(cur[h] >= 0 && cur[h] < N)) flag_status(status, kStatusBadIndex);
      }
      // each warp-wide copy covers whole rows: LPR lanes per row (8 for d = 64, 16 for d = 128),
      // so every 32-byte sector is fetched once; a row's index comes from the lane holding it
      constexpr int LPR = D / 8, RPI = 32 / LPR;
      const int sub = lane % LPR, rsub = lane / LPR;
      const int e = sub * 8;
      auto copy_rows = [&](uint32_t dst, const bf16* src_head) {
#pragma unroll
        for (int h = 0; h < NG; ++h) {
#pragma unroll
          for (int it = 0; it < 32 / RPI; ++it) {
            const int rg = it * RPI + rsub;                       // row within the group
            const int row = 32 * (pidx + NP * h) + rg;
            const int32_t j = __shfl_sync(0xffffffffu, cur[h], rg);
            const bool ok = j >= 0 && j < N;
            const int64_t src = (ok ? static_cast<int64_t>(j) : 0) * D + e;
            cp_async_16(dst + (e >> 6) * (kChunk * 128) + tc::sw128(row, e & 63), src_head + src, ok);
          }
        }
      };
      copy_rows(dK, kh);
      cp_async_arrive(bar(bars.full_k[st]));
      if (c >= NST) ok_run = tc::mbar_wait(bar(bars.empty_v[st]), ((c / NST) - 1) & 1, kWaitLimit);
      ok_run = __all_sync(0xffffffffu, ok_run);
      if (!ok_run) break;
      copy_rows(dV, vh);
      cp_async_arrive(bar(bars.full_v[st]));
    }
    cp_async_wait<0>();
    if (!ok_run && lane == 0) atomicOr(&fail_s, 1);
  } else if (warp == 5) {
    // ================================================================ MMA issue (one thread)
    if (lane == 0) {
      constexpr uint32_t idS = tc::idesc_bf16(128, 64, 0, 0);
      constexpr uint32_t idO = tc::idesc_bf16(kOnesRow<D> ? 128 : D, 64, 1, 1);
      const uint32_t sOnes = sbase + S::OFF_ONES;
      bool ok_run = true;
      int cs = 0, cp = 0;
      uint32_t idle = 0;
      while (ok_run && cp < nchunks) {
        // S(cs) whenever its K rows have landed and its TMEM buffer is free (a softmax that waits
        // for S^T must not find it queued behind a PV product), otherwise PV(cp) once S(cp) exists,
        // waiting for it in the hardware for a short bounded time
        const bool pv_next = cp < cs;
        if (cs < nchunks &&
            (pv_next ? mbar_test(bar(bars.full_k[cs % NST]), (cs / NST) & 1)
                     : mbar_try_wait_ns(bar(bars.full_k[cs % NST]), (cs / NST) & 1, 64)) &&
            (cs < 2 || mbar_test(bar(bars.s_empty[cs & 1]), ((cs - 2) >> 1) & 1))) {
          // S(cs): S^T = K_c Q^T.  The stage was written with cp.async (generic proxy):
          // order those writes before the tensor core's reads.
          tc::fence_async_shared();
          tc::tc_fence_after();
          const uint32_t aK = sK + (cs % NST) * S::KV_BYTES;
#pragma unroll
          for (int j = 0; j < D / 16; ++j) {
            const uint32_t off_a = (j >> 2) * (kChunk * 128) + (j & 3) * 32;
            const uint32_t off_b = (j >> 2) * (64 * 128) + (j & 3) * 32;
            tc::mma_ss(tmem + ((cs & 1) ? kColS1 : kColS0), tc::smem_desc(aK + off_a, 16, 1024),
                       tc::smem_desc(sQ + off_b, 16, 1024), idS, j > 0 ? 1u : 0u);
          }
          tc::mma_commit(bar(bars.s_full[cs & 1]));
          tc::mma_commit(bar(bars.empty_k[cs % NST]));
          ++cs;
          idle = 0;
        } else if (pv_next && mbar_try_wait_ns(bar(bars.p_full[cp & 1]), (cp >> 1) & 1, 64) &&
                   mbar_try_wait_ns(bar(bars.full_v[cp % NST]), (cp / NST) & 1, 64)) {
          // PV(cp): O^T += V_c^T P^T
          tc::tc_fence_after();
          const uint32_t aV = sV + (cp % NST) * S::KV_BYTES, bP = sP + (cp & 1) * S::P_BYTES;
#pragma unroll
          for (int j = 0; j < kChunk / 16; ++j) {
            // second 64-row block of A: the next 64 head dims (d = 128) or the ones tile
            const uint32_t a = aV + j * 2048, lbo = kOnesRow<D> ? sOnes - a : kChunk * 128;
            tc::mma_ss(tmem + kColO, tc::smem_desc(a, lbo, 1024), tc::smem_desc(bP + j * 2048, 8192, 1024), idO,
                       (cp > 0 || j > 0) ? 1u : 0u);
          }
          tc::mma_commit(bar(bars.pv_done[cp & 1]));
          tc::mma_commit(bar(bars.empty_v[cp % NST]));
          if (cp == nchunks - 1) tc::mma_commit(bar(bars.o_full));
          ++cp;
          idle = 0;
        } else if (++idle > kPollLimit) {
          ok_run = false;
        }
      }
      if (!ok_run) atomicOr(&fail_s, 1);
      // Before the CTA frees its tensor memory and shared memory, every MMA issued here must
      // have finished, also after a wait gave up with MMAs still in flight: one more commit
      // tracks all of them.
      tc::mma_commit(bar(bars.drain));
      if (!tc::mbar_wait(bar(bars.drain), 0, kWaitLimit)) atomicOr(&fail_s, 1);
    }
  } else {
    // ================================================================ softmax
    // Every softmax thread runs every iteration and reaches every named barrier, also after
    // a timed-out wait (later waits are then skipped and the results are discarded).
    constexpr int SMW = kSoftmaxWarps<D>, NSM = 32 * SMW;
    constexpr int QC = 256 / SMW;  // query columns per thread: 64 or 32
    constexpr int NH = QC / 16;    // 16-column TMEM loads per matrix row
    const int sw = softmax_index(warp), hq = sw >> 2, quad = warp & 3;
    const int t = quad * 32 + lane;  // key lane (TMEM lane) of this thread
    const int sidx = sw * 32 + lane;  // 0 .. NSM - 1
    const int c0 = hq * QC;           // this thread's first query column
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    bool ok_run = true;
    int32_t jnext = t < kk ? key_at(t) : -1;  // this lane's key index, one chunk ahead
    for (int c = 0; c < nchunks; ++c) {
      const int b = c & 1;
      const bool valid = jnext >= 0 && jnext < N;
      {
        const int64_t slot = static_cast<int64_t>(c + 1) * kChunk + t;
        jnext = slot < kk ? key_at(slot) : -1;
      }
      ok_run = ok_run && tc::mbar_wait(bar(bars.s_full[b]), (c >> 1) & 1, kWaitLimit);
      tc::tc_fence_after();
      // ---- one pass over this thread's part of the S^T row: probabilities against the stale
      // max, and the vote on "some logit exceeds the stale max by more than 8" (the S buffer is
      // released after it)
      const uint32_t s_col = tmem + lane_base + (b ? kColS1 : kColS0) + c0;
      bool over = false;
      float p[QC];
      {
        uint32_t r[NH][16];
#pragma unroll
        for (int h = 0; h < NH; ++h) tc::tmem_ld16(s_col + h * 16, r[h]);
        tc::tmem_wait_ld();
#pragma unroll
        for (int i4 = 0; i4 < QC / 4; ++i4) {
          const float4 m4 = reinterpret_cast<const float4*>(m_s + c0)[i4];
          const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int i = i4 * 4 + u;
            const float dlt = __uint_as_float(r[i >> 4][i & 15]) * scale_log2 - mm[u];
            over |= dlt > kStaleLimit;
            p[i] = valid ? fast_exp2(dlt) : 0.f;
          }
        }
      }
      over &= valid;
      if (__any_sync(0xffffffffu, over) && lane == 0) atomicOr(&flag_s[c & 1], 1);
      if (sidx == 0) flag_s[(c + 1) & 1] = 0;
      named_sync_softmax<NSM>();
      if (flag_s[c & 1]) {
        // ---- new running max for this chunk; rescale O and L; redo the probabilities
        float x[QC];
        {
          uint32_t r[NH][16];
#pragma unroll
          for (int h = 0; h < NH; ++h) tc::tmem_ld16(s_col + h * 16, r[h]);
          tc::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < QC; ++i) x[i] = valid ? __uint_as_float(r[i >> 4][i & 15]) * scale_log2 : -CUDART_INF_F;
        }
        column_reduce<true, QC, SMW>(x, red_w, red_s, sw, lane);
        if (sidx < 64) {
          const float mo = m_s[sidx];
          const float mn = fmaxf(mo, red_s[sidx]);
          alpha_s[sidx] = mn == -CUDART_INF_F ? 1.f : fast_exp2(mo - mn);
          m_s[sidx] = mn;
        }
        named_sync_softmax<NSM>();
        if (c > 0) {
          ok_run = ok_run && tc::mbar_wait(bar(bars.pv_done[(c - 1) & 1]), ((c - 1) >> 1) & 1, kWaitLimit);
          tc::tc_fence_after();
#pragma unroll
          for (int col = 0; col < (kOnesRow<D> ? 1 : 2); ++col) {  // O^T (and L with it), then L
            const uint32_t base = tmem + lane_base + (col ? kColL : kColO) + c0;
#pragma unroll
            for (int h = 0; h < NH; ++h) {
              uint32_t r[16];
              tc::tmem_ld16(base + h * 16, r);
              tc::tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha_s[c0 + h * 16 + i]);
              tc::tmem_st16(base + h * 16, r);
            }
          }
          tc::tmem_wait_st();
        }
#pragma unroll
        for (int i = 0; i < QC; ++i) p[i] = x[i] == -CUDART_INF_F ? 0.f : fast_exp2(x[i] - m_s[c0 + i]);
      }
      tc::tc_fence_before();
      tc::mbar_arrive(bar(bars.s_empty[b]));
      // ---- this thread's columns of the key's P^T row in the B tile (64 queries = one 128-byte
      // row; 16-byte pieces XOR-swizzled by the row)
      if (c >= 2) ok_run = ok_run && tc::mbar_wait(bar(bars.pv_done[b]), ((c - 2) >> 1) & 1, kWaitLimit);
      const uint32_t prow = sP + b * S::P_BYTES + t * 128;
#pragma unroll
      for (int cl = 0; cl < QC / 8; ++cl) {
        const int ch = hq * (QC / 8) + cl;
        const uint32_t w0 = pack_bf16x2(p[cl * 8 + 0], p[cl * 8 + 1]), w1 = pack_bf16x2(p[cl * 8 + 2], p[cl * 8 + 3]);
        const uint32_t w2 = pack_bf16x2(p[cl * 8 + 4], p[cl * 8 + 5]), w3 = pack_bf16x2(p[cl * 8 + 6], p[cl * 8 + 7]);
        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(prow + (((ch ^ t) & 7) << 4)), "r"(w0), "r"(w1),
                     "r"(w2), "r"(w3));
      }
      // ---- d = 128: row sums of this key lane, accumulated in TMEM
      if (!kOnesRow<D>) {
        const uint32_t base = tmem + lane_base + kColL + c0;
        uint32_t r[NH][16];
        if (c > 0) {
#pragma unroll
          for (int h = 0; h < NH; ++h) tc::tmem_ld16(base + h * 16, r[h]);
          tc::tmem_wait_ld();
        }
#pragma unroll
        for (int h = 0; h < NH; ++h) {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            r[h][i] = __float_as_uint((c > 0 ? __uint_as_float(r[h][i]) : 0.f) + p[h * 16 + i]);
          tc::tmem_st16(base + h * 16, r[h]);
        }
        tc::tmem_wait_st();
      }
      tc::fence_async_shared();
      tc::tc_fence_before();
      tc::mbar_arrive(bar(bars.p_full[b]));
    }
    // ---- epilogue: l = row sums (lane 64 of O^T, or column sums of L), O = O^T / l,
    // LSE = (m + log2 l) ln 2
    ok_run = ok_run && tc::mbar_wait(bar(bars.o_full), 0, kWaitLimit);
    if (!ok_run) atomicOr(&fail_s, 1);
    const bool failed = named_sync_or<NSM>(!ok_run);
    if (!failed) {
      tc::tc_fence_after();
      if (kOnesRow<D>) {
        if (warp == 2) {  // lane 64 of O^T holds l for all 64 query columns
          uint32_t r[4][16];
#pragma unroll
          for (int h = 0; h < 4; ++h) tc::tmem_ld16(tmem + lane_base + kColO + h * 16, r[h]);
          tc::tmem_wait_ld();
          if (lane == 0) {
#pragma unroll
            for (int h = 0; h < 4; ++h)
#pragma unroll
              for (int i = 0; i < 16; ++i) red_s[h * 16 + i] = __uint_as_float(r[h][i]);
          }
        }
        named_sync_softmax<NSM>();
      } else {
        float lsum[QC];
        {
          uint32_t r[NH][16];
#pragma unroll
          for (int h = 0; h < NH; ++h) tc::tmem_ld16(tmem + lane_base + kColL + c0 + h * 16, r[h]);
          tc::tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < NH; ++h)
#pragma unroll
            for (int i = 0; i < 16; ++i) lsum[h * 16 + i] = __uint_as_float(r[h][i]);
        }
        column_reduce<false, QC, SMW>(lsum, red_w, red_s, sw, lane);
      }
      // O^T lane -> head dim (M = 128: lane = row; lanes 64.. of the d = 64 product are the
      // row sums and the zero rows of the ones tile)
      const int dim = t < D ? t : -1;
      const int64_t qrow0 = bh * N + blk * 64;
      bf16* stage = reinterpret_cast<bf16*>(smem + S::OFF_K);  // [64 q][D]: K stage 0 is free now
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        uint32_t r[16];
        tc::tmem_ld16(tmem + lane_base + kColO + c0 + h * 16, r);  // whole warp, converged
        tc::tmem_wait_ld();
        if (dim >= 0) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int qq = c0 + h * 16 + i;
            const float l = red_s[qq];
            stage[qq * D + dim] = __float2bfloat16_rn(l > 0.f ? __uint_as_float(r[i]) / l : 0.f);
          }
        }
      }
      named_sync_softmax<NSM>();
      bf16* ob = o + qrow0 * D;
      for (int i = sidx; i < 64 * D / 8; i += NSM)
        reinterpret_cast<uint4*>(ob)[i] = reinterpret_cast<const uint4*>(stage)[i];
      if (sidx < 64) {
        const float l = red_s[sidx];
        lse[qrow0 + sidx] = l > 0.f ? (m_s[sidx] + __log2f(l)) * kLn2 : -CUDART_INF_F;
      }
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

// ---------------------------------------------------------------- host side
#ifndef DSV_FWD64_STAGES
#define DSV_FWD64_STAGES 2
#endif
#ifndef DSV_FWD64_MIN_BLOCKS
#define DSV_FWD64_MIN_BLOCKS 2
#endif

template <int D, int NST, int MINB>
cudaError_t launch_d(const FwdParams& p, cudaStream_t stream) {
  const int smem = Smem<D, NST>::TOTAL;
  // k = N without CSR rows: every block attends to every key, in key order; idx is not read
  const bool dense = !p.rowptr && p.topk == p.N;
  auto kern = p.rowptr ? sparse_fwd_tc_kernel<D, NST, MINB, true, false>
                       : (dense ? sparse_fwd_tc_kernel<D, NST, MINB, false, true>
                                : sparse_fwd_tc_kernel<D, NST, MINB, false, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>(p.NB), static_cast<unsigned>(p.BH));
  ProfScope prof("sparse_fwd", stream);
  kern<<<grid, kThreadsFor<D>, smem, stream>>>(p.q, p.k, p.v, p.idx, p.rowptr, p.order, p.o, p.lse, p.N, p.NB, p.topk,
                                               p.scale * kLog2e, p.status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_sparse_fwd_tc(const FwdParams& p, cudaStream_t stream) {
  switch (p.d) {
    case 64: return launch_d<64, DSV_FWD64_STAGES, DSV_FWD64_MIN_BLOCKS>(p, stream);
    case 128: return launch_d<128, 2, 1>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dsv
