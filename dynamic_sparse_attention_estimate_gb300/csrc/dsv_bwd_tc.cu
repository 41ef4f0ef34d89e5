// Sparse attention backward, main kernel, on the tcgen05 tensor cores (training needs the
// backward: DSV page 1, technical summary section 2A, stage 2).
//
// One CTA = one query block (64 queries).  For every chunk of 128 selected keys, with keys
// on the MMA's M dimension:
//     S^T  = K_c . Q^T            dP^T = V_c . dO^T           (M=128, N=64,  K=d)
//     P = exp2(S scale log2e - LSE2),  dS = P (dP - D)         (compute warps, fp32)
//     dV_c = P^T . dO             dK_c = dS^T . Q             (M=128, N=d,   K=64)
//     dQ^T += K_c^T . dS^T                                    (M=d,   N=64,  K=128)
// dQ accumulates in tensor memory (TMEM) across chunks; dV_c and dK_c (one row per key) go
// out as bf16 partial rows, block-major (this CTA's k rows are contiguous), and the list of
// every key's rows in ascending block order is written alongside; a separate kernel sums
// every key's rows in that fixed order (deterministic, no float atomics).
// P^T and dS^T go to tensor memory as bf16 pairs (a key's row in its own TMEM lane, where the
// thread that computed it writes it): the A operands of dV_c and dK_c, read by the tensor core
// without a trip through shared memory.  dS is also written to shared memory as bf16 128-byte
// rows (one per key), the MN-major B operand of dQ^T.
// Roles (512 threads): warps 0-7 compute P and dS (two warps per TMEM lane quadrant, each
// on 32 of the 64 query columns; thread = key lane of S^T / dP^T); warps 8-11 read dV_c /
// dK_c out of TMEM into shared-memory staging rows and write the key lists (and dQ at the
// end); one thread of warp 13 issues the MMAs, each group as soon as its inputs are there
// (dP^T before S^T, and S^T of the next chunk or the gradients of the current one, whichever
// is ready first; the results do not depend on the order).  Partial rows leave shared
// memory through the tensor memory accelerator (bulk copies, no load/store-unit work): at d = 64
// one thread of warp 14 sends each chunk's staged rows as two copies (the dK half-rows and the
// dV half-rows, 16 KB each: they go to two arrays) from two alternating staging buffers; at
// d = 128 each readout warp stages its 32 dK half-rows (8 KB), sends them as one copy, waits for
// the copy to have read them, then does the same with its dV half-rows (a half-size staging
// area, which leaves room for a second V stage).  dV_c / dK_c sit in two TMEM buffers at d = 64 (one at d = 128, released as soon as the
// readout has loaded it), so that readout and stores of chunk c overlap the MMAs of chunk c + 1.
// Every wait is bounded.
// Gathers.  Random-row gathers run at the rate of the copies the issuing warps keep in flight
// (measured here: 256-byte rows out of L2 at about 3.8 TB/s over the GPU with one issuing warp
// per SM, 14 TB/s with four), and a stage can be refilled the moment its last reader is done.
// So the warps that learn of that moment first issue the copies, each for its own rows: the
// compute warps gather chunk c + 1's V rows (16 each) right after reading S^T / dP^T of chunk c
// (dP of chunk c was the last reader of the stage), and the readout warps gather chunk
// c + KST's K rows (32 each) as soon as dQ of chunk c has read its stage (and, before the first
// chunk, Q, dO and the first K stages).  Each ring's "landed" barrier counts its copies.
// Dense blocks (k = N, the DENSE instantiation): chunk c holds keys 128 c .. 128 c + 127 and
// no idx is read; the kernel computes dQ only (no dV_c / dK_c products, no partial rows): dK and
// dV of dense blocks come from the key-stationary kernel of dsv_dense_bwd.cu.
#include "dsv_common.cuh"
#include "dsv_internal.h"
#include "dsv_tc.cuh"

namespace dsv {
namespace {

constexpr int kChunk = 128;
constexpr int kThreads = 512;
constexpr int kCompute = 256;  // threads computing P and dS
constexpr uint32_t kWaitLimit = 1u << 22;

// TMEM columns: S^T, dP^T, dQ^T (64 each), then dV_c, dK_c (d each) in one buffer (d = 128)
// or two (d = 64: the MMAs of the next chunk fill one while the partial rows leave the other)
constexpr uint32_t kColS = 0, kColDP = 64, kColDQ = 128, kTmemCols = 512;
// P^T and dS^T of the current chunk: 128 key lanes x 64 queries, two bf16 per column (the even
// query in the low half), the A operands of dV_c and dK_c
constexpr uint32_t kColP = 448, kColDS = 480;

template <int D>
struct Sm {
  static constexpr int KST = D == 64 ? 4 : 2;         // K stages (held until dQ)
  static constexpr int VST = 2;                       // V stages (held until dP, which is issued
                                                      // a chunk ahead of the gradients)
  static constexpr int NPDS = 1;                      // dS tiles (and P^T / dS^T TMEM sets)
  static constexpr int NST = D == 64 ? 2 : 1;         // staging buffers (d = 64: the store thread
                                                      // drains one while the other fills; d = 128:
                                                      // each readout warp sends its own rows)
  static constexpr int NDVK = D == 64 ? 2 : 1;       // dV_c / dK_c accumulator buffers
  static constexpr uint32_t COL_DV = kColDQ + 64;     // first buffer; buffer b at + b * 2d
  static constexpr int ROWB = 2 * D;                  // staging bytes per key: one bf16 half-row
                                                      // (the dK part or the dV part)
  static constexpr int STB = D == 64 ? 2 * kChunk * ROWB : kChunk * ROWB;  // bytes per staging
                                                      // buffer: d = 64 the chunk's dK then dV
                                                      // half-rows; d = 128 one half at a time
  static constexpr int BLK = D / 64;
  static constexpr int T64 = BLK * 64 * 128;          // a [64 rows][D] tile
  static constexpr int KV = BLK * kChunk * 128;       // a [128 rows][D] tile
  static constexpr int P = kChunk * 128;              // [128 keys][64 q] bf16 (a dS tile)
  static constexpr int OFF_Q = 0, OFF_DO = OFF_Q + T64, OFF_K = OFF_DO + T64, OFF_V = OFF_K + KST * KV,
                       OFF_DS = OFF_V + VST * KV, OFF_ST = OFF_DS + NPDS * P,
                       TOTAL = OFF_ST + NST * STB;
};

struct Bars {
  uint64_t full_k[4], full_v[4];    // per ring slot: K rows (and Q, dO with chunk 0) / V rows landed
  uint64_t empty_k[4], empty_v[4];  // per ring slot: K free (after dQ) / V free (after dP)
  uint64_t s_full, s_empty;        // S^T, dP^T in TMEM ready / read
  uint64_t p_full[2], pds_empty[2];  // per tile pair: P, dS written / no longer read by any MMA
  uint64_t dvk_full[2], dvk_empty[2];  // per buffer: dV_c, dK_c in TMEM ready / read
  uint64_t dq_full;                // last dQ^T update done
  uint64_t st_full[2], st_empty[2];  // per staging buffer: rows written / copied out (d = 64)
  uint64_t drain;                  // MMA commit at the end: every MMA issued is done
};

// D[tmem] (+)= A[tmem] * B[smem]; issued by one thread.  A (M = 128) sits K-major in TMEM: row m
// in lane m, two bf16 per 32-bit column (the even K element in the low half), K elements
// 16 j .. 16 j + 15 in columns 8 j .. 8 j + 7 from a_tmem.
DSV_DEVICE void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate));
}
DSV_DEVICE void sync_group(int id) { asm volatile("bar.sync %0, 128;\n" ::"r"(id) : "memory"); }
DSV_DEVICE bool sync_group_or(int id, bool v) {
  uint32_t r;
  asm volatile("{\n .reg .pred p, q;\n setp.ne.u32 p, %2, 0;\n bar.red.or.pred q, %1, 128, p;\n selp.u32 %0, 1, 0, q;\n}\n"
               : "=r"(r)
               : "r"(id), "r"(static_cast<uint32_t>(v))
               : "memory");
  return r != 0;
}
// Wait for this thread's TMEM loads, and make the 32 destination registers depend on the
// wait so no use of them is scheduled ahead of it.
DSV_DEVICE void tmem_wait_ld_into(uint32_t (&r)[2][16]) {
  tc::tmem_wait_ld();
#pragma unroll
  for (int h = 0; h < 2; ++h)
    asm volatile("" : "+r"(r[h][0]), "+r"(r[h][1]), "+r"(r[h][2]), "+r"(r[h][3]), "+r"(r[h][4]), "+r"(r[h][5]),
                 "+r"(r[h][6]), "+r"(r[h][7]), "+r"(r[h][8]), "+r"(r[h][9]), "+r"(r[h][10]), "+r"(r[h][11]),
                 "+r"(r[h][12]), "+r"(r[h][13]), "+r"(r[h][14]), "+r"(r[h][15]));
}
// Shared -> global bulk copy by the tensor memory accelerator, tracked by this thread's
// bulk-async groups.
DSV_DEVICE void bulk_store(void* gdst, uint32_t ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n" ::"l"(gdst), "r"(ssrc), "r"(bytes)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;\n" ::: "memory");
}
DSV_DEVICE void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory"); }
DSV_DEVICE void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory"); }
DSV_DEVICE bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
DSV_DEVICE void cp_async_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(bar) : "memory");
}

// NROWS rows of a 128-byte-swizzled [TILE_ROWS][D] tile, starting at tile row row0, gathered with
// cp.async from the head's rows: tile row row0 + i takes source row j = the key held by lane
// key_lane0 + i of this warp (j outside [0, N): zeros).  LPR lanes per row, so each warp-wide
// copy moves whole rows and every 32-byte sector is fetched once.
template <int D, int NROWS, int TILE_ROWS = kChunk>
DSV_DEVICE void gather_rows(uint32_t tile, const bf16* head, int32_t my_key, int key_lane0, int row0, int lane,
                            int64_t N) {
  constexpr int LPR = D / 8, RPI = 32 / LPR;
  const int sub = lane % LPR, rsub = lane / LPR, e = sub * 8;
  const uint32_t dcol = tile + (e >> 6) * (TILE_ROWS * 128);  // 64-column blocks are TILE_ROWS rows apart
#pragma unroll
  for (int it = 0; it < NROWS / RPI; ++it) {
    const int i = it * RPI + rsub;
    const int32_t j = __shfl_sync(0xffffffffu, my_key, key_lane0 + i);
    const bool ok = j >= 0 && j < N;
    cp_async_16(dcol + tc::sw128(row0 + i, e & 63), head + (ok ? static_cast<int64_t>(j) : 0) * D + e, ok);
  }
}

// CSR: per-block key counts from row offsets (and an optional launch order); otherwise k for
// every block, compiled without those loads.
template <int D, bool CSR, bool DENSE>
__global__ void __launch_bounds__(kThreads, 1)
sparse_bwd_tc_kernel(BwdParams p, int64_t bh0, int64_t blk0, int64_t nblk, int64_t W32, float scale_log2) {
  using S = Sm<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ __align__(8) Bars bars;
  __shared__ uint32_t tmem_base_s;
  __shared__ __align__(16) float lse2_s[64];
  __shared__ __align__(16) float delta_s[64];
  __shared__ int fail_s;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t N = p.N, NB = p.NB;
  const int64_t cta_row = (CSR && p.order) ? p.order[blockIdx.x] : static_cast<int64_t>(blockIdx.x);  // launch order
  const int64_t hs = cta_row / nblk, lb = cta_row % nblk;
  const int64_t bh = bh0 + hs, blk = blk0 + lb;
  const int64_t row0 = bh * N + blk * 64;
  // this block's keys: k of them (or its CSR row), and its first partial row in the wave
  const int64_t grow = bh * NB + blk;
  const int64_t kk = CSR ? p.rowptr[grow + 1] - p.rowptr[grow] : p.topk;
  const int32_t* ib = DENSE ? nullptr : p.idx + (CSR ? p.rowptr[grow] : grow * p.topk);
  // the key at slot i (dense: the key position itself)
  auto key_at = [&](int64_t i) -> int32_t { return DENSE ? static_cast<int32_t>(i) : __ldg(ib + i); };
  const int64_t prow0 = CSR ? p.rowptr[grow] - p.rowptr[bh0 * NB + blk0] : cta_row * kk;
  const int nchunks = static_cast<int>((kk + kChunk - 1) / kChunk);
  if (CSR && nchunks == 0) {  // a block with no keys: dQ = 0 (uniform for the CTA, before any barrier)
    for (int i = tid; i < 64 * D / 8; i += kThreads)
      reinterpret_cast<uint4*>(p.dq + row0 * D)[i] = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + S::OFF_Q, sDO = sbase + S::OFF_DO, sK = sbase + S::OFF_K, sV = sbase + S::OFF_V;
  const uint32_t sDS0 = sbase + S::OFF_DS;  // dS tile b at sDS0 + b * S::P
  auto bar = [](uint64_t& b) { return smem_u32(&b); };

  if (sbase & 1023u) {  // swizzled tiles need 1024-byte alignment
    if (tid == 0) flag_status(p.status, kStatusTimeout);
    return;
  }
  if (warp == 0) {
    tc::tmem_alloc(smem_u32(&tmem_base_s), kTmemCols);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    for (int s = 0; s < 4; ++s) {
      tc::mbar_init(bar(bars.full_k[s]), 128);   // the 4 readout warps' copies
      tc::mbar_init(bar(bars.full_v[s]), 256);   // the 8 compute warps' copies
      tc::mbar_init(bar(bars.empty_k[s]), 1);
      tc::mbar_init(bar(bars.empty_v[s]), 1);
    }
    tc::mbar_init(bar(bars.s_full), 1);
    tc::mbar_init(bar(bars.s_empty), kCompute);
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(bar(bars.p_full[s]), kCompute);
      tc::mbar_init(bar(bars.pds_empty[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(bar(bars.dvk_full[s]), 1);
      tc::mbar_init(bar(bars.dvk_empty[s]), 128);
    }
    tc::mbar_init(bar(bars.dq_full), 1);
    tc::mbar_init(bar(bars.drain), 1);
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(bar(bars.st_full[s]), 128);
      tc::mbar_init(bar(bars.st_empty[s]), 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    fail_s = 0;
  }
  // D_i = dO_i . O_i and LSE in base 2 (compute warps: two threads per query row)
  if (warp < 4) {
    const int row = tid >> 1, half = tid & 1;
    const bf16* dor = p.d_o + (row0 + row) * D + half * (D / 2);
    const bf16* orow = p.o + (row0 + row) * D + half * (D / 2);
    float acc = 0.f;
#pragma unroll
    for (int c = 0; c < D / 2; c += 8) {
      const uint4 a = *reinterpret_cast<const uint4*>(dor + c);
      const uint4 b = *reinterpret_cast<const uint4*>(orow + c);
      const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) acc += bf16_lo(av[u]) * bf16_lo(bv[u]) + bf16_hi(av[u]) * bf16_hi(bv[u]);
    }
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    if (half == 0) {
      delta_s[row] = acc;
      lse2_s[row] = p.lse[row0 + row] * kLog2e;
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = tmem_base_s;

  constexpr int KST = S::KST, VST = S::VST;
  constexpr int NDVK = S::NDVK, NPDS = S::NPDS;
  // d = 64: a chunk's staged partial rows leave as one bulk copy (block-major rows are
  // contiguous); d = 128 stages half rows, which the readout warps copy out themselves
  constexpr bool kStoreWarps = D == 64 && !DENSE;
  if (warp == 12 || warp == 15) {
    // idle
  } else if (warp == 13) {
    // ================================================================ MMA issue (one thread)
    if (lane == 0) {
      constexpr uint32_t idS = tc::idesc_bf16(128, 64, 0, 0);   // S^T, dP^T
      constexpr uint32_t idKV = tc::idesc_bf16(128, D, 0, 1);   // dV_c, dK_c: A K-major, B MN-major
      constexpr uint32_t idQ = tc::idesc_bf16(D, 64, 1, 1);     // dQ^T: A, B MN-major
      // S^T / dP^T of chunk c
      auto issue_dp = [&](int c) {  // dP^T of chunk c (frees its V stage)
        tc::fence_async_shared();  // the stage was written with cp.async (generic proxy)
        tc::tc_fence_after();
        const uint32_t aV = sV + (c % VST) * S::KV;
#pragma unroll
        for (int j = 0; j < D / 16; ++j) {
          const uint32_t off_a = (j >> 2) * (kChunk * 128) + (j & 3) * 32;
          const uint32_t off_b = (j >> 2) * (64 * 128) + (j & 3) * 32;
          tc::mma_ss(tmem + kColDP, tc::smem_desc(aV + off_a, 16, 1024), tc::smem_desc(sDO + off_b, 16, 1024), idS,
                     j > 0 ? 1u : 0u);
        }
        tc::mma_commit(bar(bars.empty_v[c % VST]));
      };
      auto issue_sdp = [&](int c) {  // S^T and dP^T of chunk c together (d = 64)
        tc::fence_async_shared();
        tc::tc_fence_after();
        const uint32_t aK = sK + (c % KST) * S::KV, aV = sV + (c % VST) * S::KV;
#pragma unroll
        for (int j = 0; j < D / 16; ++j) {
          const uint32_t off_a = (j >> 2) * (kChunk * 128) + (j & 3) * 32;
          const uint32_t off_b = (j >> 2) * (64 * 128) + (j & 3) * 32;
          tc::mma_ss(tmem + kColS, tc::smem_desc(aK + off_a, 16, 1024), tc::smem_desc(sQ + off_b, 16, 1024), idS,
                     j > 0 ? 1u : 0u);
          tc::mma_ss(tmem + kColDP, tc::smem_desc(aV + off_a, 16, 1024), tc::smem_desc(sDO + off_b, 16, 1024), idS,
                     j > 0 ? 1u : 0u);
        }
        tc::mma_commit(bar(bars.s_full));
        tc::mma_commit(bar(bars.empty_v[c % VST]));
      };
      auto issue_s = [&](int c) {  // S^T of chunk c; s_full then covers dP^T too
        tc::fence_async_shared();
        tc::tc_fence_after();
        const uint32_t aK = sK + (c % KST) * S::KV;
#pragma unroll
        for (int j = 0; j < D / 16; ++j) {
          const uint32_t off_a = (j >> 2) * (kChunk * 128) + (j & 3) * 32;
          const uint32_t off_b = (j >> 2) * (64 * 128) + (j & 3) * 32;
          tc::mma_ss(tmem + kColS, tc::smem_desc(aK + off_a, 16, 1024), tc::smem_desc(sQ + off_b, 16, 1024), idS,
                     j > 0 ? 1u : 0u);
        }
        tc::mma_commit(bar(bars.s_full));
      };
      // the dQ^T update of chunk c, then dV_c, dK_c (so the K stage frees first)
      auto issue_grads = [&](int c) {
        tc::tc_fence_after();
        const uint32_t cdv = S::COL_DV + (c % NDVK) * 2 * D;
        const uint32_t sDS = sDS0 + (c % NPDS) * S::P;
        const uint32_t aK = sK + (c % KST) * S::KV;
#pragma unroll
        for (int j = 0; j < kChunk / 16; ++j)  // K = 128 keys
          tc::mma_ss(tmem + kColDQ, tc::smem_desc(aK + j * 2048, kChunk * 128, 1024),
                     tc::smem_desc(sDS + j * 2048, 8192, 1024), idQ, (c > 0 || j > 0) ? 1u : 0u);
        tc::mma_commit(bar(bars.empty_k[c % KST]));  // the K stage is free once dQ^T has read it
        if (!DENSE) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {  // K = 64 queries
            mma_ts(tmem + cdv, tmem + kColP + j * 8, tc::smem_desc(sDO + j * 2048, 64 * 128, 1024), idKV,
                       j > 0 ? 1u : 0u);
            mma_ts(tmem + cdv + D, tmem + kColDS + j * 8, tc::smem_desc(sQ + j * 2048, 64 * 128, 1024), idKV,
                       j > 0 ? 1u : 0u);
          }
          tc::mma_commit(bar(bars.dvk_full[c % NDVK]));
        }
        tc::mma_commit(bar(bars.pds_empty[c % NPDS]));
        if (c == nchunks - 1) tc::mma_commit(bar(bars.dq_full));
      };
      // Issue order per chunk c: dP^T(c+1) as soon as S^T/dP^T(c) have been read and V(c+1)
      // has landed (the V rows are gathered two chunks ahead), then S^T(c+1) and the gradients
      // of chunk c in whichever order their inputs arrive: S^T(c+1) waits for the K rows of
      // chunk c+1, which can only be gathered once dQ of chunk c-1 has read their stage, and
      // the gradients of chunk c free chunk c's K stage for chunk c+2.
      auto wait_v = [&](int c) { return tc::mbar_wait(bar(bars.full_v[c % VST]), (c / VST) & 1, kWaitLimit); };
      auto wait_k = [&](int c) { return tc::mbar_wait(bar(bars.full_k[c % KST]), (c / KST) & 1, kWaitLimit); };
      // chunk 0: Q and dO land with the first K stage
      bool ok_run = wait_v(0) && wait_k(0);
      if (ok_run && D == 64) issue_sdp(0);
      if (ok_run && D == 128) {
        issue_dp(0);
        issue_s(0);
      }
      for (int c = 0; c < nchunks && ok_run; ++c) {
        if (c + 1 < nchunks && D == 64) {  // four K stages: the K rows are never late
          ok_run = wait_k(c + 1) && wait_v(c + 1) && tc::mbar_wait(bar(bars.s_empty), c & 1, kWaitLimit);
          if (!ok_run) break;
          issue_sdp(c + 1);
        } else if (c + 1 < nchunks) {
          ok_run = tc::mbar_wait(bar(bars.s_empty), c & 1, kWaitLimit) && wait_v(c + 1);
          if (!ok_run) break;
          issue_dp(c + 1);
          // S^T(c + 1) waits for its K rows, the gradients of chunk c for P/dS(c): issue whichever
          // is ready first (the gradients free chunk c's K stage for the rows of chunk c + 2)
          bool s_done = false, g_done = false;
          uint32_t spins = 0;
          while (!(s_done && g_done)) {
            if (!s_done && mbar_test(bar(bars.full_k[(c + 1) % KST]), ((c + 1) / KST) & 1)) {
              issue_s(c + 1);
              s_done = true;
            } else if (!g_done && mbar_test(bar(bars.p_full[c % NPDS]), (c / NPDS) & 1) &&
                       (DENSE || c < NDVK || mbar_test(bar(bars.dvk_empty[c % NDVK]), ((c / NDVK) - 1) & 1))) {
              issue_grads(c);
              g_done = true;
            } else if (++spins > kWaitLimit) {
              break;
            }
          }
          ok_run = s_done && g_done;
          continue;
        }
        ok_run = tc::mbar_wait(bar(bars.p_full[c % NPDS]), (c / NPDS) & 1, kWaitLimit) &&
                 (DENSE || c < NDVK || tc::mbar_wait(bar(bars.dvk_empty[c % NDVK]), ((c / NDVK) - 1) & 1, kWaitLimit));
        if (!ok_run) break;
        issue_grads(c);
      }
      if (!ok_run) atomicOr(&fail_s, 1);
      // Every MMA issued here must be done before the CTA frees its tensor and shared memory,
      // also when a wait gave up with MMAs still in flight: one more commit tracks them all.
      tc::mma_commit(bar(bars.drain));
      if (!tc::mbar_wait(bar(bars.drain), 0, kWaitLimit)) atomicOr(&fail_s, 1);
    }
  } else if (warp < 8) {
    // ================================================================ P and dS (threads 0..255)
    const int t = tid & 127;          // key lane
    const int hq = tid >> 7;          // query columns [32 hq, 32 hq + 32)
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    bool ok_run = true;
    int32_t jnext = t < kk ? key_at(t) : -1;
    // this warp's 16 V rows of each chunk: rows 32 (warp & 3) + 16 hq + i, keys in lanes 16 hq + i
    const bf16* vhead = p.v + bh * N * D;
    const int vrow0 = 32 * (warp & 3) + 16 * hq;
    // chunks 0 .. VST - 1 (every V stage is free); then chunk c + VST once dP of chunk c, the last
    // reader of its stage, is done -- which is before this warp sees S^T / dP^T of chunk c
    for (int c0 = 0; c0 < VST && c0 < nchunks; ++c0) {
      const int64_t slot = static_cast<int64_t>(c0) * kChunk + t;
      gather_rows<D, 16>(sV + c0 * S::KV, vhead, slot < kk ? key_at(slot) : -1, 16 * hq, vrow0, lane, N);
      cp_async_arrive(bar(bars.full_v[c0]));
    }
    for (int c = 0; c < nchunks; ++c) {
      const bool valid = jnext >= 0 && jnext < N;
      {
        const int64_t slot = static_cast<int64_t>(c + 1) * kChunk + t;
        jnext = slot < kk ? key_at(slot) : -1;
      }
      ok_run = ok_run && tc::mbar_wait(bar(bars.s_full), c & 1, kWaitLimit);
      tc::tc_fence_after();
      uint32_t sr[2][16], dr[2][16];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        tc::tmem_ld16(tmem + lane_base + kColS + hq * 32 + h * 16, sr[h]);
        tc::tmem_ld16(tmem + lane_base + kColDP + hq * 32 + h * 16, dr[h]);
      }
      tc::tmem_wait_ld();
      tc::tc_fence_before();
      tc::mbar_arrive(bar(bars.s_empty));
      if (c + VST < nchunks) {  // chunk c + VST's V rows, into chunk c's stage (dP of chunk c is done)
        const int sv = c % VST;
        const int64_t slot = static_cast<int64_t>(c + VST) * kChunk + t;
        const int32_t vkey = slot < kk ? key_at(slot) : -1;
        ok_run = ok_run && tc::mbar_wait(bar(bars.empty_v[sv]), (c / VST) & 1, kWaitLimit);
        gather_rows<D, 16>(sV + sv * S::KV, vhead, vkey, 16 * hq, vrow0, lane, N);
        cp_async_arrive(bar(bars.full_v[sv]));
      }
      uint32_t pw[16], dw[16];  // packed bf16 pairs of P and dS
#pragma unroll
      for (int i4 = 0; i4 < 8; ++i4) {
        const float4 l4 = reinterpret_cast<const float4*>(lse2_s)[hq * 8 + i4];
        const float4 d4 = reinterpret_cast<const float4*>(delta_s)[hq * 8 + i4];
        const float ll[4] = {l4.x, l4.y, l4.z, l4.w}, dd[4] = {d4.x, d4.y, d4.z, d4.w};
        float pv[4], dv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = i4 * 4 + u;
          const float sv = __uint_as_float(sr[i >> 4][i & 15]);
          const float dpv = __uint_as_float(dr[i >> 4][i & 15]);
          pv[u] = valid ? fast_exp2(sv * scale_log2 - ll[u]) : 0.f;
          dv[u] = pv[u] * (dpv - dd[u]);
        }
        pw[i4 * 2] = pack_bf16x2(pv[0], pv[1]);
        pw[i4 * 2 + 1] = pack_bf16x2(pv[2], pv[3]);
        dw[i4 * 2] = pack_bf16x2(dv[0], dv[1]);
        dw[i4 * 2 + 1] = pack_bf16x2(dv[2], dv[3]);
      }
      const int pb = c % NPDS;
      if (c >= NPDS) ok_run = ok_run && tc::mbar_wait(bar(bars.pds_empty[pb]), ((c / NPDS) - 1) & 1, kWaitLimit);
      const uint32_t drow = sDS0 + pb * S::P + t * 128;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        const int ch = hq * 4 + cc;
        const uint32_t off = ((ch ^ t) & 7) << 4;
        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(drow + off), "r"(dw[cc * 4]), "r"(dw[cc * 4 + 1]),
                     "r"(dw[cc * 4 + 2]), "r"(dw[cc * 4 + 3]));
      }
      if (!DENSE) {  // this key lane's P^T and dS^T columns (query pairs 16 hq .. 16 hq + 15) in TMEM
        tc::tmem_st16(tmem + lane_base + kColP + hq * 16, pw);
        tc::tmem_st16(tmem + lane_base + kColDS + hq * 16, dw);
        tc::tmem_wait_st();
      }
      tc::fence_async_shared();
      tc::tc_fence_before();
      tc::mbar_arrive(bar(bars.p_full[pb]));
    }
    cp_async_wait<0>();
    if (!ok_run) atomicOr(&fail_s, 1);
  } else if (warp == 14) {
    // ================================================================ partial-row stores (d = 64)
    // One thread hands each chunk's staged rows (one contiguous run of block-major partial
    // rows: 128 x 256 bytes) to the tensor memory accelerator as a single bulk copy, so the
    // stores take no load/store-unit bandwidth from the gathers.
    if (kStoreWarps && lane == 0) {
      bool ok_run = true;
      for (int c = 0; c < nchunks && ok_run; ++c) {
        const int b = c & 1;
        ok_run = tc::mbar_wait(bar(bars.st_full[b]), (c >> 1) & 1, kWaitLimit);
        if (!ok_run) break;
        const int64_t row0_c = prow0 + static_cast<int64_t>(c) * kChunk;
        const int64_t nrows = kk - static_cast<int64_t>(c) * kChunk < kChunk ? kk - static_cast<int64_t>(c) * kChunk : kChunk;
        const uint32_t sbuf = sbase + S::OFF_ST + b * S::STB;
        bulk_store(p.partial + row0_c * D, sbuf, static_cast<uint32_t>(nrows * S::ROWB));
        bulk_store(p.partial_dv + row0_c * D, sbuf + kChunk * S::ROWB, static_cast<uint32_t>(nrows * S::ROWB));
        bulk_wait_read();                        // the staging buffer has been read
        tc::mbar_arrive(bar(bars.st_empty[b]));
      }
      bulk_wait_all();  // the partial rows are written before the CTA ends
      if (!ok_run) atomicOr(&fail_s, 1);
    }
  } else {
    // ================================================================ partial rows and dQ (threads 256..383)
    const int te = tid - 256;
    const uint32_t lane_base = static_cast<uint32_t>((warp - 8) * 32) << 16;
    const uint32_t* cbits = p.colbits + (hs * W32 + (lb >> 5)) * N;
    const uint32_t* cpre = p.colpre + (hs * W32 + (lb >> 5)) * N;
    const int64_t* offs = p.offsets + hs * N;
    const uint32_t lowmask = (1u << (lb & 31)) - 1u;
    auto key_of = [&](int c) -> int32_t {
      const int64_t slot = static_cast<int64_t>(c) * kChunk + te;
      return (c < nchunks && slot < kk) ? key_at(slot) : -1;
    };
    // a key's partial row: offsets[j] + (blocks of this wave before this one that selected j);
    // the three loads are issued one chunk before the row is needed
    struct PosParts {
      int64_t off;
      uint32_t pre, bits;
      bool valid;
    };
    auto pos_load = [&](int32_t j) -> PosParts {
      PosParts q{0, 0u, 0u, j >= 0 && j < N};
      if (q.valid) {
        q.off = offs[j];
        q.pre = cpre[j];
        q.bits = cbits[j];
      }
      return q;
    };
    // Q and dO (16 rows each per warp) and the first KST K stages (32 rows per warp)
    const int wr = warp - 8;
    const bf16* khead = p.k + bh * N * D;
    {
      const int32_t qkey = static_cast<int32_t>(blk * 64) + 16 * wr + (lane & 15);
      gather_rows<D, 16, 64>(sQ, p.q + bh * N * D, qkey, 0, 16 * wr, lane, N);  // [64 rows][D] tiles
      gather_rows<D, 16, 64>(sDO, p.d_o + bh * N * D, qkey, 0, 16 * wr, lane, N);
      for (int s0 = 0; s0 < KST && s0 < nchunks; ++s0) {
        gather_rows<D, 32>(sK + s0 * S::KV, khead, key_of(s0), 0, 32 * wr, lane, N);
        cp_async_arrive(bar(bars.full_k[s0]));
      }
    }
    PosParts pos_next = pos_load(DENSE ? -1 : key_of(0));
    int32_t j_next2 = DENSE ? -1 : key_of(1);
    bool ok_run = true;
    for (int c = 0; c < nchunks; ++c) {
      // chunk c + KST's K rows, into chunk c's stage once dQ of chunk c has read it
      if (c + KST < nchunks) {
        const int32_t kkey = key_of(c + KST);
        ok_run = ok_run && tc::mbar_wait(bar(bars.empty_k[c % KST]), (c / KST) & 1, kWaitLimit);
        gather_rows<D, 32>(sK + (c % KST) * S::KV, khead, kkey, 0, 32 * wr, lane, N);
        cp_async_arrive(bar(bars.full_k[c % KST]));
      }
      if (DENSE) continue;  // dense: no partial rows, dQ only
      const int64_t pos = pos_next.valid ? pos_next.off + pos_next.pre + __popc(pos_next.bits & lowmask) : -1;
      pos_next = pos_load(j_next2);
      j_next2 = key_of(c + 2);
      const int buf = c % NDVK;
      ok_run = ok_run && tc::mbar_wait(bar(bars.dvk_full[buf]), (c / NDVK) & 1, kWaitLimit);
      tc::tc_fence_after();
      // dK (times scale) then dV, as bf16, into this key's staging row (16-byte chunks XOR-
      // swizzled by the partial row index, so a warp's stores hit distinct banks; the reduction
      // undoes it).  d = 64: the store thread copies the chunk's rows out; d = 128: the warp's
      // elected lane copies the warp's rows out.  The TMEM load of the next 32 columns is in
      // flight while the current ones are converted.
      const uint32_t cdv = S::COL_DV + buf * 2 * D;
      const int sb = kStoreWarps ? (c & 1) : 0;  // staging buffer
      // staging half-row of this key: d = 64 row te of buffer sb's dK area (its dV area follows);
      // d = 128 row te of the one area, dK half first, then (after its copy has read it) dV half
      const uint32_t srow = sbase + S::OFF_ST + sb * S::STB + te * S::ROWB;
      const uint32_t swarp = sbase + S::OFF_ST + (te & ~31) * S::ROWB;
      constexpr int NPART = 2 * D / 32;             // 32-column parts: dK columns first, then dV
      auto part_col = [&](int part) -> uint32_t {
        return part < D / 32 ? cdv + D + part * 32 : cdv + (part - D / 32) * 32;
      };
      uint32_t r[2][2][16];
      tc::tmem_ld16(tmem + lane_base + part_col(0), r[0][0]);
      tc::tmem_ld16(tmem + lane_base + part_col(0) + 16, r[0][1]);
      tmem_wait_ld_into(r[0]);
      // this pair's partial row, for the reduction of key j: the list of key j's rows is in
      // ascending block order at key-major position pos
      const int64_t prow_index = prow0 + static_cast<int64_t>(c) * kChunk + te;
      if (pos >= 0) p.lists[pos] = static_cast<int32_t>(prow_index);
      // 16-byte chunk q of the row is staged at q ^ swz: distinct for 8 consecutive keys (no
      // bank conflicts), keyed on the partial row index, which the reduction undoes
      const int swz = static_cast<int>(prow_index & 7);
      if (kStoreWarps && c >= 2)  // the bulk copy has read this buffer's previous chunk
        ok_run = ok_run && tc::mbar_wait(bar(bars.st_empty[sb]), ((c >> 1) - 1) & 1, kWaitLimit);
      if (!kStoreWarps && c >= 1) {  // this warp's copy of the previous chunk has read its rows
        if (lane == 0) bulk_wait_read();
        __syncwarp();
      }
#pragma unroll
      for (int part = 0; part < NPART; ++part) {
        const int cur = part & 1;
        if (part + 1 < NPART) {
          tc::tmem_ld16(tmem + lane_base + part_col(part + 1), r[cur ^ 1][0]);
          tc::tmem_ld16(tmem + lane_base + part_col(part + 1) + 16, r[cur ^ 1][1]);
        }
        const float mult = part < D / 32 ? p.scale : 1.f;
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = pack_bf16x2(__uint_as_float(r[cur][i >> 3][(2 * i) & 15]) * mult,
                             __uint_as_float(r[cur][i >> 3][(2 * i + 1) & 15]) * mult);
        const bool dv_part = part >= D / 32;
        // 16-byte chunks within the staging half-row (d = 64: the dV half-rows follow the dK area)
        const int base_chunk = (dv_part ? part - D / 32 : part) * 4;
        const uint32_t hrow = srow + ((kStoreWarps && dv_part) ? kChunk * S::ROWB : 0);
#pragma unroll
        for (int v = 0; v < 4; ++v)
          asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(hrow + (((base_chunk + v) ^ swz) << 4)),
                       "r"(w[4 * v]), "r"(w[4 * v + 1]), "r"(w[4 * v + 2]), "r"(w[4 * v + 3]));
        if (part + 1 < NPART) tmem_wait_ld_into(r[cur ^ 1]);
        if (part + 2 == NPART) {  // every TMEM load of this chunk has completed: release the buffer
          tc::tc_fence_before();
          tc::mbar_arrive(bar(bars.dvk_empty[buf]));
        }
        if (!kStoreWarps && (part == D / 32 - 1 || part == NPART - 1)) {
          // d = 128: the warp's 32 half-rows are consecutive: one bulk copy (8 KB) by one lane, into
          // the dK array after the dK parts, the dV array after the dV parts; the dV parts reuse
          // the area once the dK copy has read it
          tc::fence_async_shared();  // staged rows visible to the bulk copy
          __syncwarp();
          const int64_t wslot = static_cast<int64_t>(c) * kChunk + (te & ~31);
          const int64_t nr = kk - wslot < 32 ? kk - wslot : 32;
          if (lane == 0 && nr > 0)
            bulk_store((dv_part ? p.partial_dv : p.partial) + (prow0 + wslot) * D, swarp,
                       static_cast<uint32_t>(nr * S::ROWB));
          if (!dv_part) {
            if (lane == 0) bulk_wait_read();
            __syncwarp();
          }
        }
      }
      if (NPART < 2) {
        tc::tc_fence_before();
        tc::mbar_arrive(bar(bars.dvk_empty[buf]));
      }
      if (kStoreWarps) {
        tc::fence_async_shared();  // staged rows visible to the bulk copy
        tc::mbar_arrive(bar(bars.st_full[sb]));
      }
    }
    if (!kStoreWarps) {  // the rows are written before the CTA ends
      if (lane == 0) bulk_wait_all();
      __syncwarp();
    }
    cp_async_wait<0>();  // the K copies this warp issued have landed
    // ---- dQ = scale * (dQ^T)^T, through a shared-memory transpose
    ok_run = ok_run && tc::mbar_wait(bar(bars.dq_full), 0, kWaitLimit);
    if (!ok_run) atomicOr(&fail_s, 1);
    const bool failed = sync_group_or(2, !ok_run);
    if (!failed) {
      tc::tc_fence_after();
      const int dim = D == 128 ? te : ((lane < 16) ? (warp - 8) * 16 + lane : -1);
      bf16* stage = reinterpret_cast<bf16*>(smem + S::OFF_K);  // [64 q][D]: stage 0 is free now
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        uint32_t r[16];
        tc::tmem_ld16(tmem + lane_base + kColDQ + h * 16, r);  // whole warp, converged
        tc::tmem_wait_ld();
        if (dim >= 0) {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            stage[(h * 16 + i) * D + dim] = __float2bfloat16_rn(__uint_as_float(r[i]) * p.scale);
        }
      }
      sync_group(2);
      bf16* dqb = p.dq + row0 * D;
      for (int i = te; i < 64 * D / 8; i += 128)
        reinterpret_cast<uint4*>(dqb)[i] = reinterpret_cast<const uint4*>(stage)[i];
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (fail_s && tid == 0) flag_status(p.status, kStatusTimeout);
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D>
cudaError_t launch_d(const BwdParams& p, const BwdWave& w, int64_t W32, cudaStream_t stream) {
  const int smem = Sm<D>::TOTAL;
  auto kern = p.rowptr ? sparse_bwd_tc_kernel<D, true, false>
                       : (p.dense ? sparse_bwd_tc_kernel<D, false, true> : sparse_bwd_tc_kernel<D, false, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  ProfScope prof("bwd_main", stream);
  kern<<<static_cast<unsigned>(w.nh * w.nblk), kThreads, smem, stream>>>(p, w.bh0, w.blk0, w.nblk, W32,
                                                                          p.scale * kLog2e);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_main_tc(const BwdParams& p, const BwdWave& w, int64_t W32, cudaStream_t stream) {
  switch (p.d) {
    case 64: return launch_d<64>(p, w, W32, stream);
    case 128: return launch_d<128>(p, w, W32, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dsv
