// Device helpers shared by the DSV kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define DSV_DEVICE __device__ __forceinline__

namespace dsv {

// Bit set in the device status word when a kernel meets a key index outside [0, N).
constexpr unsigned int kStatusBadIndex = 1u;
// Bit set when a kernel gave up waiting on one of its own mbarriers (bounded waits).
constexpr unsigned int kStatusTimeout = 2u;

// log2(e): softmax runs in base 2 with the scale folded in.
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

DSV_DEVICE uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- packing
DSV_DEVICE uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
DSV_DEVICE float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
DSV_DEVICE float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// ---------------------------------------------------------------- mma.sync m16n8k16 (bf16 in, fp32 acc)
DSV_DEVICE void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------- ldmatrix
DSV_DEVICE void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
DSV_DEVICE void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

// ---------------------------------------------------------------- cp.async (16 B, zero-fill when !valid)
DSV_DEVICE void cp_async_16(uint32_t dst, const void* src, bool valid) {
  int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n));
}
DSV_DEVICE void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
DSV_DEVICE void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

// ---------------------------------------------------------------- smem tile addressing
// Tiles of rows of ROW_BYTES (a multiple of 128); 16-byte chunk c of row r is stored at
// chunk c ^ (r & 7) so that 8 consecutive rows read at one logical chunk hit 32 banks.
template <int ROW_BYTES>
DSV_DEVICE uint32_t swz(int row, int chunk) {
  return static_cast<uint32_t>(row * ROW_BYTES + ((chunk ^ (row & 7)) << 4));
}

// 2^x with the hardware approximation (relative error about 2^-22; results below 2^-126
// flush to zero, and 2^-inf = 0), which is all a softmax needs.
DSV_DEVICE float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

DSV_DEVICE void flag_status(unsigned int* status, unsigned int bits) {
  if (status) atomicOr(status, bits);
}

}  // namespace dsv
