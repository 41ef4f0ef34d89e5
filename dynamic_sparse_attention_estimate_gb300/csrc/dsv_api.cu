// C ABI of libdsv.so (declared in include/dsv.h): host-side validation, workspace
// planning and launches.  Nothing here allocates device memory.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <map>
#include <string>
#include <vector>

#include "../../include/dsv.h"
#include "dsv_internal.h"

// Device status word: kernels OR in kStatusBadIndex when they meet a key index outside
// [0, N) or a repeated key in one idx row.  Read and cleared by dsv_last_device_status.
__device__ unsigned int g_dsv_status;

namespace {

thread_local char g_msg[512] = "";

dsv_status fail(dsv_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return s;
}

dsv_status ok() {
  g_msg[0] = '\0';
  return DSV_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int kMaxDevices = 64;
// Per-device address of g_dsv_status, looked up on first use with that device current (host
// threads racing on the first look-up all find the same address).
std::atomic<unsigned int*> g_status_ptr[kMaxDevices];

dsv_status status_word(unsigned int** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(DSV_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(DSV_ERR_CUDA, "device ordinal %d out of range", dev);
  unsigned int* ptr = g_status_ptr[dev].load(std::memory_order_acquire);
  if (!ptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_dsv_status);
    if (e != cudaSuccess) return fail(DSV_ERR_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    ptr = static_cast<unsigned int*>(p);
    g_status_ptr[dev].store(ptr, std::memory_order_release);
  }
  *out = ptr;
  return DSV_OK;
}

dsv_status check_dims(const dsv_dims* d, bool need_d, bool need_r) {
  if (!d) return fail(DSV_ERR_INVALID_ARG, "dims is NULL");
  if (d->B < 1 || d->H < 1 || d->N < 1) return fail(DSV_ERR_INVALID_ARG, "B, H, N must be >= 1");
  if (d->block != 64) return fail(DSV_ERR_UNSUPPORTED, "block must be 64 (got %lld)", (long long)d->block);
  if (d->N % d->block) return fail(DSV_ERR_INVALID_ARG, "N (%lld) must be a multiple of block", (long long)d->N);
  if (d->N > 0x7fffffffLL) return fail(DSV_ERR_INVALID_ARG, "N must fit int32 key indices");
  if (d->k < 1 || d->k > d->N) return fail(DSV_ERR_INVALID_ARG, "need 1 <= k <= N (k=%lld)", (long long)d->k);
  if (d->B * d->H > (1LL << 31) - 1) return fail(DSV_ERR_INVALID_ARG, "B*H too large");
  if (d->B * d->H * d->N > 0x7fffffffLL)
    return fail(DSV_ERR_INVALID_ARG, "B*H*N must fit int32 row coordinates (split the heads over calls)");
  if (need_d && d->d != 64 && d->d != 128)
    return fail(DSV_ERR_UNSUPPORTED, "head dim d must be 64 or 128 (got %lld)", (long long)d->d);
  if (need_r && (d->r < 16 || d->r > 64 || d->r % 16))
    return fail(DSV_ERR_UNSUPPORTED, "low-rank dim r must be 16, 32, 48 or 64 (got %lld)", (long long)d->r);
  if (!(d->scale == d->scale)) return fail(DSV_ERR_INVALID_ARG, "scale is NaN");
  return DSV_OK;
}

#define DSV_NEED_PTR(p)                                                                \
  do {                                                                                 \
    if (!(p)) return fail(DSV_ERR_INVALID_ARG, "%s is NULL", #p);                     \
    if (!aligned16(p)) return fail(DSV_ERR_INVALID_ARG, "%s is not 16-byte aligned", #p); \
  } while (0)

float eff_scale(const dsv_dims* d) { return d->scale > 0.f ? d->scale : 1.0f / sqrtf(static_cast<float>(d->d)); }

// ---------------------------------------------------------------- backward workspace planning
constexpr size_t kAlign = 256;
size_t up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct WavePlan {
  int64_t nh = 0, nblk = 0;  // heads per wave (whole-head waves) or blocks per wave (sub-head)
  bool sub = false;
};

struct Carve {
  size_t colbits, colpre, count, offsets, tsum, lists, partial, partial_dv, acc, total;
};

// pairs: the (block, key) pairs of the largest wave (-1: nh * nblk * k)
Carve carve(const dsv_dims* d, int64_t nh, int64_t nblk, bool sub, int64_t pairs = -1) {
  const int64_t W32 = (nblk + 31) / 32;
  if (pairs < 0) pairs = nh * nblk * d->k;
  Carve c;
  size_t o = 0;
  c.colbits = o; o += up(sizeof(uint32_t) * nh * W32 * d->N);
  c.colpre = o;  o += up(sizeof(uint32_t) * nh * W32 * d->N);
  c.count = o;   o += up(sizeof(uint32_t) * nh * d->N);
  c.offsets = o; o += up(sizeof(int64_t) * nh * d->N);
  c.tsum = o;    o += up(sizeof(int64_t) * nh * ((d->N + 1023) / 1024));
  c.lists = o;   o += up(sizeof(int32_t) * pairs);
  c.partial = o; o += up(sizeof(uint16_t) * d->d * pairs);       // bf16 dK half-rows
  c.partial_dv = o; o += up(sizeof(uint16_t) * d->d * pairs);    // bf16 dV half-rows
  c.acc = o;     o += sub ? up(sizeof(float) * 2 * d->d * d->N) : 0;
  c.total = o;
  return c;
}

size_t plan_bytes(const dsv_dims* d, const WavePlan& w) { return carve(d, w.nh, w.nblk, w.sub).total; }

// Largest plan that fits `budget` bytes (whole heads first, then blocks of one head).
bool plan_for(const dsv_dims* d, size_t budget, WavePlan* out) {
  const int64_t BH = d->B * d->H, NB = d->N / 64;
  for (int64_t nh = BH; nh >= 1; nh = (nh == 1 ? 0 : (nh + 1) / 2)) {
    WavePlan w{nh, NB, false};
    if (plan_bytes(d, w) <= budget) {
      // grow back towards BH while it still fits (the halving may undershoot)
      while (w.nh < BH) {
        WavePlan w2{w.nh + 1, NB, false};
        if (plan_bytes(d, w2) > budget) break;
        w = w2;
      }
      *out = w;
      return true;
    }
    if (nh == 1) break;
  }
  // blocks of one head per wave: the largest even split that fits, rounded down to whole waves of
  // the main kernel's CTAs (one per SM), so that only a head's last wave ends in a partial one
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    sms = 0;
    (void)cudaGetLastError();  // no device (a size query on a host without one): no rounding
  }
  for (int64_t s = 2; s <= NB; s = (s < 64 ? s + 1 : s + s / 8)) {
    int64_t nblk = (NB + s - 1) / s;
    WavePlan w{1, nblk, true};
    if (plan_bytes(d, w) <= budget) {
      if (sms > 0 && nblk > sms) w.nblk = nblk / sms * sms;
      *out = w;
      return true;
    }
  }
  WavePlan w{1, 1, NB > 1};
  if (plan_bytes(d, w) <= budget) { *out = w; return true; }
  return false;
}

constexpr size_t kRecommendedPartialBytes = size_t(16) << 30;

// ---------------------------------------------------------------- optional per-kernel timing
struct ProfRecord {
  const char* name;
  cudaEvent_t begin, end;
};
constexpr int kProfPool = 16384;
bool g_prof_on = false;
std::vector<cudaEvent_t> g_prof_events;   // 2 * kProfPool, created at enable time
std::vector<ProfRecord> g_prof_records;
size_t g_prof_dropped = 0;

}  // namespace

namespace dsv {
ProfScope::ProfScope(const char* name, cudaStream_t s) : slot(-1), stream(s) {
  if (!g_prof_on) return;
  const size_t n = g_prof_records.size();
  if (n >= static_cast<size_t>(kProfPool)) { ++g_prof_dropped; return; }
  ProfRecord r{name, g_prof_events[2 * n], g_prof_events[2 * n + 1]};
  if (cudaEventRecord(r.begin, s) != cudaSuccess) return;
  g_prof_records.push_back(r);
  slot = static_cast<int>(n);
}
ProfScope::~ProfScope() {
  if (slot >= 0) cudaEventRecord(g_prof_records[slot].end, stream);
}
}  // namespace dsv

extern "C" {

const char* dsv_status_string(dsv_status s) {
  switch (s) {
    case DSV_OK: return "DSV_OK";
    case DSV_ERR_INVALID_ARG: return "DSV_ERR_INVALID_ARG";
    case DSV_ERR_UNSUPPORTED: return "DSV_ERR_UNSUPPORTED";
    case DSV_ERR_WORKSPACE: return "DSV_ERR_WORKSPACE";
    case DSV_ERR_CUDA: return "DSV_ERR_CUDA";
    case DSV_ERR_DEVICE_CHECK: return "DSV_ERR_DEVICE_CHECK";
  }
  return "DSV_ERR_UNKNOWN";
}

const char* dsv_last_error_message(void) { return g_msg; }

size_t dsv_estimate_topk_workspace(const dsv_dims* dims) {
  (void)dims;
  return 0;
}

dsv_status dsv_estimate_topk(const dsv_dims* dims, const void* q_lr, const void* k_lr, int32_t* idx, void* ws,
                             size_t ws_bytes, void* stream) {
  (void)ws;
  (void)ws_bytes;
  dsv_status s = check_dims(dims, false, true);
  if (s != DSV_OK) return s;
  DSV_NEED_PTR(q_lr);
  DSV_NEED_PTR(k_lr);
  DSV_NEED_PTR(idx);
  unsigned int* status = nullptr;
  if ((s = status_word(&status)) != DSV_OK) return s;
  dsv::EstimateParams p;
  p.q_lr = static_cast<const dsv::bf16*>(q_lr);
  p.k_lr = static_cast<const dsv::bf16*>(k_lr);
  p.idx = idx;
  p.BH = dims->B * dims->H;
  p.N = dims->N;
  p.NB = dims->N / dims->block;
  p.topk = dims->k;
  p.r = static_cast<int>(dims->r);
  p.status = status;
  cudaError_t e = dsv::launch_estimate_topk(p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(DSV_ERR_CUDA, "estimate launch: %s", cudaGetErrorString(e));
  return ok();
}

dsv_status dsv_estimate_mass_k(const dsv_dims* dims, const void* q_lr, const void* k_lr, float tau_log2,
                               uint32_t mass_num, uint32_t dense_num, int32_t* k_row, int64_t* rowptr, int32_t* order,
                               void* stream) {
  dsv_status s = check_dims(dims, false, true);
  if (s != DSV_OK) return s;
  DSV_NEED_PTR(q_lr);
  DSV_NEED_PTR(k_lr);
  if (!k_row) return fail(DSV_ERR_INVALID_ARG, "k_row is NULL");
  if (!rowptr) return fail(DSV_ERR_INVALID_ARG, "rowptr is NULL");
  if (!(tau_log2 > 0.f) || !(tau_log2 < 3.0e38f)) return fail(DSV_ERR_INVALID_ARG, "tau_log2 must be finite and > 0");
  if (mass_num < 1 || mass_num > 65536) return fail(DSV_ERR_INVALID_ARG, "mass_num must be in [1, 65536] (got %u)", mass_num);
  if (dense_num > 65536) return fail(DSV_ERR_INVALID_ARG, "dense_num must be in [0, 65536] (got %u)", dense_num);
  if (dims->N > (1LL << 20))
    return fail(DSV_ERR_UNSUPPORTED, "mass selection supports N <= 2^20 (the weight sums are 64-bit)");
  if (order && (dims->N + 127) / 128 + 1 > 4096)
    return fail(DSV_ERR_UNSUPPORTED, "a launch order needs N <= 523904");
  unsigned int* status = nullptr;
  if ((s = status_word(&status)) != DSV_OK) return s;
  dsv::MassParams p;
  p.q_lr = static_cast<const dsv::bf16*>(q_lr);
  p.k_lr = static_cast<const dsv::bf16*>(k_lr);
  p.BH = dims->B * dims->H;
  p.N = dims->N;
  p.NB = dims->N / dims->block;
  p.r = static_cast<int>(dims->r);
  p.tau_log2 = tau_log2;
  p.mass_num = mass_num;
  p.dense_num = dense_num;
  double fact = 1.0;
  for (int i = 0; i < 7; ++i) {  // Taylor coefficients of 2^f: (ln 2)^i / i!, rounded to fp32
    if (i > 0) fact *= i;
    p.coef[i] = static_cast<float>(std::pow(std::log(2.0), i) / fact);
  }
  p.krow = k_row;
  p.rowptr = rowptr;
  p.order = order;
  p.status = status;
  cudaError_t e = dsv::launch_estimate_mass_k(p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(DSV_ERR_CUDA, "mass selection launch: %s", cudaGetErrorString(e));
  return ok();
}

dsv_status dsv_csr_launch_order(const dsv_dims* dims, const int64_t* rowptr, int32_t* order, void* stream) {
  dsv_status s = check_dims(dims, false, false);
  if (s != DSV_OK) return s;
  if (!rowptr || !order) return fail(DSV_ERR_INVALID_ARG, "rowptr and order must be non-NULL");
  if ((dims->N + 127) / 128 + 1 > 4096) return fail(DSV_ERR_UNSUPPORTED, "a launch order needs N <= 523904");
  cudaError_t e = dsv::launch_csr_order(rowptr, dims->B * dims->H * (dims->N / dims->block), dims->N, order,
                                        static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(DSV_ERR_CUDA, "launch order: %s", cudaGetErrorString(e));
  return ok();
}

dsv_status dsv_estimate_topk_csr(const dsv_dims* dims, const void* q_lr, const void* k_lr, const int32_t* k_row,
                                 const int64_t* rowptr, int32_t* cols, void* stream) {
  dsv_status s = check_dims(dims, false, true);
  if (s != DSV_OK) return s;
  DSV_NEED_PTR(q_lr);
  DSV_NEED_PTR(k_lr);
  if (!k_row || !rowptr || !cols) return fail(DSV_ERR_INVALID_ARG, "k_row, rowptr and cols must be non-NULL");
  unsigned int* status = nullptr;
  if ((s = status_word(&status)) != DSV_OK) return s;
  dsv::EstimateParams p;
  p.q_lr = static_cast<const dsv::bf16*>(q_lr);
  p.k_lr = static_cast<const dsv::bf16*>(k_lr);
  p.idx = cols;
  p.BH = dims->B * dims->H;
  p.N = dims->N;
  p.NB = dims->N / dims->block;
  p.topk = dims->N;
  p.r = static_cast<int>(dims->r);
  p.krow = k_row;
  p.rowptr = rowptr;
  p.status = status;
  cudaError_t e = dsv::launch_estimate_topk(p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(DSV_ERR_CUDA, "estimate launch: %s", cudaGetErrorString(e));
  return ok();
}

// The forward needs no scratch at present (its workspace arguments are reserved).
size_t fwd_workspace_bytes(const dsv_dims*) { return 0; }

dsv_status fwd_impl(const dsv_dims* dims, const void* q, const void* k, const void* v, const int32_t* idx,
                    const int64_t* rowptr, const int32_t* order, void* o, float* lse, void* ws, size_t ws_bytes,
                    void* stream) {
  dsv_status s = check_dims(dims, true, false);
  if (s != DSV_OK) return s;
  if (ws && !aligned16(ws)) return fail(DSV_ERR_WORKSPACE, "workspace must be 16-byte aligned");
  DSV_NEED_PTR(q);
  DSV_NEED_PTR(k);
  DSV_NEED_PTR(v);
  if (rowptr || dims->k != dims->N) DSV_NEED_PTR(idx);  // k = N: every key, idx is not read
  DSV_NEED_PTR(o);
  DSV_NEED_PTR(lse);
  unsigned int* status = nullptr;
  if ((s = status_word(&status)) != DSV_OK) return s;
  dsv::FwdParams p;
  p.q = static_cast<const dsv::bf16*>(q);
  p.k = static_cast<const dsv::bf16*>(k);
  p.v = static_cast<const dsv::bf16*>(v);
  p.idx = idx;
  p.o = static_cast<dsv::bf16*>(o);
  p.lse = lse;
  p.BH = dims->B * dims->H;
  p.N = dims->N;
  p.NB = dims->N / dims->block;
  p.topk = dims->k;
  p.d = static_cast<int>(dims->d);
  p.scale = eff_scale(dims);
  p.status = status;
  p.rowptr = rowptr;
  p.order = order;
  (void)ws_bytes;
  cudaError_t e = dsv::launch_sparse_fwd_tc(p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(DSV_ERR_CUDA, "forward launch: %s", cudaGetErrorString(e));
  return ok();
}

size_t dsv_sparse_attn_fwd_workspace(const dsv_dims* dims) {
  if (check_dims(dims, true, false) != DSV_OK) return 0;
  return fwd_workspace_bytes(dims);
}

dsv_status dsv_sparse_attn_fwd(const dsv_dims* dims, const void* q, const void* k, const void* v, const int32_t* idx,
                               void* o, float* lse, void* ws, size_t ws_bytes, void* stream) {
  return fwd_impl(dims, q, k, v, idx, nullptr, nullptr, o, lse, ws, ws_bytes, stream);
}

dsv_status dsv_sparse_attn_fwd_csr(const dsv_dims* dims, const void* q, const void* k, const void* v,
                                   const int64_t* rowptr, const int32_t* cols, const int32_t* order, void* o,
                                   float* lse, void* stream) {
  if (!rowptr) return fail(DSV_ERR_INVALID_ARG, "rowptr is NULL");
  return fwd_impl(dims, q, k, v, cols, rowptr, order, o, lse, nullptr, 0, stream);
}

// k = N (every key selected): the dense backward needs only D = rowsum(dO o O) per query row;
// no partial rows at all.
size_t dense_bwd_bytes(const dsv_dims* d) { return up(sizeof(float) * static_cast<size_t>(d->B * d->H * d->N)); }

size_t dsv_sparse_attn_bwd_workspace_min(const dsv_dims* dims) {
  if (check_dims(dims, true, false) != DSV_OK) return 0;
  if (dims->k == dims->N) return dense_bwd_bytes(dims);
  WavePlan w{1, 1, dims->N / 64 > 1};
  return plan_bytes(dims, w);
}

size_t dsv_sparse_attn_bwd_workspace(const dsv_dims* dims) {
  if (check_dims(dims, true, false) != DSV_OK) return 0;
  if (dims->k == dims->N) return dense_bwd_bytes(dims);
  // the largest plan whose partial rows stay within the recommended budget
  const size_t per_block = sizeof(uint16_t) * 2 * dims->d * dims->k;
  const int64_t BH = dims->B * dims->H, NB = dims->N / 64;
  const int64_t blocks = static_cast<int64_t>(kRecommendedPartialBytes / (per_block ? per_block : 1));
  WavePlan w;
  if (blocks >= BH * NB) w = WavePlan{BH, NB, false};
  else if (blocks >= NB) w = WavePlan{blocks / NB, NB, false};
  else {
    const int64_t nblk = blocks < 1 ? 1 : blocks;
    const int64_t s = (NB + nblk - 1) / nblk;
    w = WavePlan{1, (NB + s - 1) / s, true};
  }
  return plan_bytes(dims, w);
}

// rowptr == nullptr: k keys per block, waves planned from the workspace; otherwise CSR rows
// with total_pairs keys in all, one wave over every head (the workspace must hold it).
// parts: dsv::kBwdAll, or one of the two halves of a split backward (kBwdPrep reads idx only;
// kBwdFinish expects the workspace a kBwdPrep call filled); the halves need a single wave.
dsv_status bwd_impl(const dsv_dims* dims, const void* d_o, const void* q, const void* k, const void* v,
                    const void* o, const float* lse, const int32_t* idx, const int64_t* rowptr,
                    const int32_t* order, int64_t total_pairs, void* dq, void* dk, void* dv, void* ws,
                    size_t ws_bytes, void* stream, int parts = dsv::kBwdAll) {
  dsv_status s = check_dims(dims, true, false);
  if (s != DSV_OK) return s;
  if (rowptr || dims->k != dims->N) DSV_NEED_PTR(idx);  // k = N: every key, idx is not read
  if (parts & dsv::kBwdFinish) {
    DSV_NEED_PTR(d_o);
    DSV_NEED_PTR(q);
    DSV_NEED_PTR(k);
    DSV_NEED_PTR(v);
    DSV_NEED_PTR(o);
    DSV_NEED_PTR(lse);
    DSV_NEED_PTR(dq);
    DSV_NEED_PTR(dk);
    DSV_NEED_PTR(dv);
  }
  if (!ws) return fail(DSV_ERR_WORKSPACE, "workspace is NULL");
  if (reinterpret_cast<uintptr_t>(ws) % kAlign) return fail(DSV_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  if (!rowptr && dims->k == dims->N) {
    // every key selected: the dense backward (dK, dV key-stationary; dQ query-centric), which
    // reads no idx and writes no partial rows; the split backward's first part has nothing to do
    const size_t need = dense_bwd_bytes(dims);
    if (ws_bytes < need)
      return fail(DSV_ERR_WORKSPACE, "workspace of %zu bytes is below the %zu the dense backward needs", ws_bytes, need);
    if (parts == dsv::kBwdPrep) return ok();
    unsigned int* status = nullptr;
    if ((s = status_word(&status)) != DSV_OK) return s;
    dsv::BwdParams p{};
    p.d_o = static_cast<const dsv::bf16*>(d_o);
    p.q = static_cast<const dsv::bf16*>(q);
    p.k = static_cast<const dsv::bf16*>(k);
    p.v = static_cast<const dsv::bf16*>(v);
    p.o = static_cast<const dsv::bf16*>(o);
    p.lse = lse;
    p.idx = idx;
    p.dq = static_cast<dsv::bf16*>(dq);
    p.dk = static_cast<dsv::bf16*>(dk);
    p.dv = static_cast<dsv::bf16*>(dv);
    p.BH = dims->B * dims->H;
    p.N = dims->N;
    p.NB = dims->N / dims->block;
    p.topk = dims->k;
    p.d = static_cast<int>(dims->d);
    p.scale = eff_scale(dims);
    p.status = status;
    p.dense = true;
    float* delta = static_cast<float*>(ws);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = dsv::launch_dense_dkdv(p, delta, st);
    if (e == cudaSuccess) e = dsv::launch_bwd_main_tc(p, dsv::BwdWave{0, p.BH, 0, p.NB, true, true}, 1, st);
    if (e != cudaSuccess) return fail(DSV_ERR_CUDA, "dense backward launch: %s", cudaGetErrorString(e));
    return ok();
  }
  WavePlan plan;
  if (rowptr) {
    plan = WavePlan{dims->B * dims->H, dims->N / 64, false};
    const size_t need = carve(dims, plan.nh, plan.nblk, false, total_pairs).total;
    if (ws_bytes < need)
      return fail(DSV_ERR_WORKSPACE, "workspace of %zu bytes is below the %zu the CSR backward needs", ws_bytes, need);
  } else if (!plan_for(dims, ws_bytes, &plan)) {
    return fail(DSV_ERR_WORKSPACE, "workspace of %zu bytes is below the minimum %zu", ws_bytes,
                dsv_sparse_attn_bwd_workspace_min(dims));
  }
  if (parts != dsv::kBwdAll && (plan.sub || plan.nh < dims->B * dims->H))
    return fail(DSV_ERR_WORKSPACE, "a split backward needs a workspace that holds every head in one wave "
                "(dsv_sparse_attn_bwd_workspace)");
  unsigned int* status = nullptr;
  if ((s = status_word(&status)) != DSV_OK) return s;

  const Carve c = rowptr ? carve(dims, plan.nh, plan.nblk, false, total_pairs) : carve(dims, plan.nh, plan.nblk, plan.sub);
  uint8_t* base = static_cast<uint8_t*>(ws);
  dsv::BwdParams p;
  p.d_o = static_cast<const dsv::bf16*>(d_o);
  p.q = static_cast<const dsv::bf16*>(q);
  p.k = static_cast<const dsv::bf16*>(k);
  p.v = static_cast<const dsv::bf16*>(v);
  p.o = static_cast<const dsv::bf16*>(o);
  p.lse = lse;
  p.idx = idx;
  p.dq = static_cast<dsv::bf16*>(dq);
  p.dk = static_cast<dsv::bf16*>(dk);
  p.dv = static_cast<dsv::bf16*>(dv);
  p.BH = dims->B * dims->H;
  p.N = dims->N;
  p.NB = dims->N / dims->block;
  p.topk = dims->k;
  p.d = static_cast<int>(dims->d);
  p.scale = eff_scale(dims);
  p.status = status;
  p.colbits = reinterpret_cast<uint32_t*>(base + c.colbits);
  p.colpre = reinterpret_cast<uint32_t*>(base + c.colpre);
  p.count = reinterpret_cast<uint32_t*>(base + c.count);
  p.offsets = reinterpret_cast<int64_t*>(base + c.offsets);
  p.tsum = reinterpret_cast<int64_t*>(base + c.tsum);
  p.lists = reinterpret_cast<int32_t*>(base + c.lists);
  p.partial = reinterpret_cast<dsv::bf16*>(base + c.partial);
  p.partial_dv = reinterpret_cast<dsv::bf16*>(base + c.partial_dv);
  p.acc = plan.sub ? reinterpret_cast<float*>(base + c.acc) : nullptr;
  p.rowptr = rowptr;
  p.order = order;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  std::vector<dsv::BwdWave> waves;
  if (!plan.sub) {
    for (int64_t bh0 = 0; bh0 < p.BH; bh0 += plan.nh)
      waves.push_back(dsv::BwdWave{bh0, plan.nh < p.BH - bh0 ? plan.nh : p.BH - bh0, 0, p.NB, true, true});
  } else {
    for (int64_t bh = 0; bh < p.BH; ++bh)
      for (int64_t b0 = 0; b0 < p.NB; b0 += plan.nblk) {
        const int64_t n = plan.nblk < p.NB - b0 ? plan.nblk : p.NB - b0;
        waves.push_back(dsv::BwdWave{bh, 1, b0, n, b0 == 0, b0 + n == p.NB});
      }
  }
  for (const dsv::BwdWave& w : waves) {
    cudaError_t e = dsv::launch_bwd_wave(p, w, st, parts);
    if (e != cudaSuccess) return fail(DSV_ERR_CUDA, "backward launch: %s", cudaGetErrorString(e));
  }
  return ok();
}

dsv_status dsv_sparse_attn_bwd(const dsv_dims* dims, const void* d_o, const void* q, const void* k, const void* v,
                               const void* o, const float* lse, const int32_t* idx, void* dq, void* dk, void* dv,
                               void* ws, size_t ws_bytes, void* stream) {
  return bwd_impl(dims, d_o, q, k, v, o, lse, idx, nullptr, nullptr, 0, dq, dk, dv, ws, ws_bytes, stream);
}

dsv_status dsv_sparse_attn_bwd_prepare(const dsv_dims* dims, const int32_t* idx, void* ws, size_t ws_bytes,
                                       void* stream) {
  return bwd_impl(dims, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, idx, nullptr, nullptr, 0, nullptr,
                  nullptr, nullptr, ws, ws_bytes, stream, dsv::kBwdPrep);
}

dsv_status dsv_sparse_attn_bwd_prepared(const dsv_dims* dims, const void* d_o, const void* q, const void* k,
                                        const void* v, const void* o, const float* lse, const int32_t* idx, void* dq,
                                        void* dk, void* dv, void* ws, size_t ws_bytes, void* stream) {
  return bwd_impl(dims, d_o, q, k, v, o, lse, idx, nullptr, nullptr, 0, dq, dk, dv, ws, ws_bytes, stream,
                  dsv::kBwdFinish);
}

size_t dsv_sparse_attn_bwd_csr_workspace(const dsv_dims* dims, int64_t total_pairs) {
  if (check_dims(dims, true, false) != DSV_OK || total_pairs < 0) return 0;
  return carve(dims, dims->B * dims->H, dims->N / 64, false, total_pairs).total;
}

dsv_status dsv_sparse_attn_bwd_csr(const dsv_dims* dims, const void* d_o, const void* q, const void* k, const void* v,
                                   const void* o, const float* lse, const int64_t* rowptr, const int32_t* cols,
                                   const int32_t* order, int64_t total_pairs, void* dq, void* dk, void* dv, void* ws,
                                   size_t ws_bytes, void* stream) {
  if (!rowptr) return fail(DSV_ERR_INVALID_ARG, "rowptr is NULL");
  if (total_pairs < 0) return fail(DSV_ERR_INVALID_ARG, "total_pairs must be >= 0");
  if (total_pairs > 0x7fffffffLL) return fail(DSV_ERR_UNSUPPORTED, "total_pairs must fit int32 partial-row indices");
  return bwd_impl(dims, d_o, q, k, v, o, lse, cols, rowptr, order, total_pairs, dq, dk, dv, ws, ws_bytes, stream);
}

dsv_status dsv_profile_enable(int on) {
  if (on && !g_prof_on) {
    if (g_prof_events.empty()) {
      g_prof_events.resize(2 * kProfPool);
      for (auto& e : g_prof_events) {
        cudaError_t err = cudaEventCreate(&e);
        if (err != cudaSuccess) {
          g_prof_events.clear();
          return fail(DSV_ERR_CUDA, "cudaEventCreate: %s", cudaGetErrorString(err));
        }
      }
    }
    g_prof_records.clear();
    g_prof_dropped = 0;
  }
  if (!on) g_prof_records.clear();
  g_prof_on = on != 0;
  return ok();
}

size_t dsv_profile_read(char* buf, size_t buf_bytes) {
  std::map<std::string, std::pair<long long, double>> agg;
  for (const auto& r : g_prof_records) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.end) == cudaSuccess && cudaEventElapsedTime(&ms, r.begin, r.end) == cudaSuccess) {
      auto& a = agg[r.name];
      a.first += 1;
      a.second += ms;
    }
  }
  const bool consume = buf != nullptr && buf_bytes > 0;   // a size query keeps the records
  if (consume) g_prof_records.clear();
  std::string out;
  char line[256];
  for (const auto& kv : agg) {
    snprintf(line, sizeof(line), "%s %lld %.6f\n", kv.first.c_str(), kv.second.first, kv.second.second);
    out += line;
  }
  if (g_prof_dropped) {
    snprintf(line, sizeof(line), "dropped %zu 0\n", g_prof_dropped);
    out += line;
    if (consume) g_prof_dropped = 0;
  }
  if (consume) {
    const size_t n = out.size() < buf_bytes - 1 ? out.size() : buf_bytes - 1;
    memcpy(buf, out.data(), n);
    buf[n] = '\0';
  }
  return out.size() + 1;
}

dsv_status dsv_last_device_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(DSV_ERR_CUDA, "stream synchronize: %s", cudaGetErrorString(e));
  unsigned int v = 0, zero = 0;
  e = cudaMemcpyFromSymbol(&v, g_dsv_status, sizeof(v));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_dsv_status, &zero, sizeof(zero));
  if (e != cudaSuccess) return fail(DSV_ERR_CUDA, "status word: %s", cudaGetErrorString(e));
  if (v)
    return fail(DSV_ERR_DEVICE_CHECK, "device status 0x%x:%s%s", v,
                (v & 1u) ? " an out-of-range or repeated key index" : "",
                (v & 2u) ? " a kernel gave up waiting on its own barrier" : "");
  return ok();
}

// ---------------------------------------------------------------- fused AdaLN
static dsv_status check_adaln(const dsv_adaln_dims* d) {
  if (!d) return fail(DSV_ERR_INVALID_ARG, "dims is NULL");
  if (d->B < 1 || d->N < 1) return fail(DSV_ERR_INVALID_ARG, "B and N must be >= 1");
  if (d->D < 8 || d->D > 8192 || d->D % 8)
    return fail(DSV_ERR_INVALID_ARG, "D must be a multiple of 8 in [8, 8192] (got %lld)", (long long)d->D);
  if (d->B * d->N > (1LL << 40)) return fail(DSV_ERR_INVALID_ARG, "B*N too large");
  if (!(d->eps >= 0.f) || d->eps > 3.0e38f) return fail(DSV_ERR_INVALID_ARG, "eps must be finite and >= 0");
  return DSV_OK;
}

dsv_status dsv_adaln_fwd(const dsv_adaln_dims* dims, const void* x, const void* scale, const void* shift, void* y,
                         void* stream) {
  dsv_status s = check_adaln(dims);
  if (s != DSV_OK) return s;
  DSV_NEED_PTR(x);
  DSV_NEED_PTR(scale);
  DSV_NEED_PTR(shift);
  DSV_NEED_PTR(y);
  dsv::AdalnParams p{};
  p.x = x;
  p.scale = scale;
  p.shift = shift;
  p.y = y;
  p.B = dims->B;
  p.N = dims->N;
  p.D = dims->D;
  p.eps = dims->eps;
  if ((s = status_word(&p.status)) != DSV_OK) return s;
  cudaError_t e = dsv::launch_adaln_fwd(p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(DSV_ERR_CUDA, "adaln forward launch: %s", cudaGetErrorString(e));
  return ok();
}

size_t dsv_adaln_bwd_workspace(const dsv_adaln_dims* dims) {
  if (check_adaln(dims) != DSV_OK) return 0;
  return up(dsv::adaln_tiling(dims->B, dims->N, dims->D, true).workspace_bytes);
}

dsv_status dsv_adaln_bwd(const dsv_adaln_dims* dims, const void* x, const void* scale, const void* dy, void* dx,
                         float* d_scale, float* d_shift, void* ws, size_t ws_bytes, void* stream) {
  dsv_status s = check_adaln(dims);
  if (s != DSV_OK) return s;
  DSV_NEED_PTR(x);
  DSV_NEED_PTR(scale);
  DSV_NEED_PTR(dy);
  DSV_NEED_PTR(dx);
  DSV_NEED_PTR(d_scale);
  DSV_NEED_PTR(d_shift);
  const size_t need = dsv::adaln_tiling(dims->B, dims->N, dims->D, true).workspace_bytes;
  if (!ws) return fail(DSV_ERR_WORKSPACE, "workspace is NULL");
  if (reinterpret_cast<uintptr_t>(ws) % kAlign) return fail(DSV_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  if (ws_bytes < need) return fail(DSV_ERR_WORKSPACE, "workspace of %zu bytes is below the %zu needed", ws_bytes, need);
  dsv::AdalnParams p{};
  p.x = x;
  p.scale = scale;
  p.dy = dy;
  p.dx = dx;
  p.d_scale = d_scale;
  p.d_shift = d_shift;
  p.partial = static_cast<float*>(ws);
  p.B = dims->B;
  p.N = dims->N;
  p.D = dims->D;
  p.eps = dims->eps;
  if ((s = status_word(&p.status)) != DSV_OK) return s;
  cudaError_t e = dsv::launch_adaln_bwd(p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(DSV_ERR_CUDA, "adaln backward launch: %s", cudaGetErrorString(e));
  return ok();
}

// ---------------------------------------------------------------- backward with library-held scratch
// For callers that cannot allocate device memory (see include/dsv.h).  The scratch is a
// fixed device array; host code only ever uses the address looked up per device below.
}  // extern "C"

namespace {
static __device__ __align__(256) unsigned char g_noalloc_scratch[DSV_NOALLOC_SCRATCH_BYTES];
// Per-device address of g_noalloc_scratch, looked up once per device.  Several host threads may
// race on the first look-up; they all find the same address, and the atomic makes the store and
// the loads well defined.
std::atomic<void*> g_noalloc_ptr[kMaxDevices];
}  // namespace

extern "C" {

dsv_status dsv_sparse_attn_bwd_noalloc(const dsv_dims* dims, const void* d_o, const void* q, const void* k,
                                       const void* v, const void* o, const float* lse, const int32_t* idx,
                                       void* dq, void* dk, void* dv, void* stream) {
  dsv_status s = check_dims(dims, true, false);
  if (s != DSV_OK) return s;
  const size_t need = dsv_sparse_attn_bwd_workspace_min(dims);
  if (need > DSV_NOALLOC_SCRATCH_BYTES)
    return fail(DSV_ERR_WORKSPACE,
                "this backward needs at least %zu bytes of scratch but the no-allocation variant holds %zu; "
                "call dsv_sparse_attn_bwd with a caller workspace instead",
                need, static_cast<size_t>(DSV_NOALLOC_SCRATCH_BYTES));
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(DSV_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(DSV_ERR_CUDA, "device ordinal %d out of range", dev);
  void* scratch = g_noalloc_ptr[dev].load(std::memory_order_acquire);
  if (!scratch) {  // set-up, once per device, with that device current
    e = cudaGetSymbolAddress(&scratch, g_noalloc_scratch);
    if (e != cudaSuccess) return fail(DSV_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
    g_noalloc_ptr[dev].store(scratch, std::memory_order_release);
  }
  // Every word of the scratch that the backward reads in a wave is written earlier in the same
  // wave (the bitmap kernel writes all of its words, zeros included; the scans, lists, partial
  // rows and the accumulator are written before they are read), so what an earlier call left
  // there is never used and nothing needs clearing.
  return dsv_sparse_attn_bwd(dims, d_o, q, k, v, o, lse, idx, dq, dk, dv, scratch, DSV_NOALLOC_SCRATCH_BYTES,
                             stream);
}

}  // extern "C"
