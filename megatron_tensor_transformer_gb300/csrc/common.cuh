// Shared device helpers for the tpx kernels (sm_103a).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/tpx.h"

namespace tpx {

// Launch counter (host side), bumped by every launch the library makes.
void note_launch();

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ uint16_t f2bf(float f) {
  __nv_bfloat16 b = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&b);
}

// 16-byte streaming load that bypasses L1 allocation: weights are read exactly once.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// 16-byte read-only load through L1 (activations, reused by many warps).
__device__ __forceinline__ uint4 ld_ro16(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

// D = A * B + D, m16n8k16, bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two e4m3 codes (low 16 bits of v) -> packed bf16x2; exact (every e4m3 value is a bf16 value).
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint16_t v) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(v), __NV_E4M3);
  __half2 hh = *reinterpret_cast<__half2*>(&h);
  float2 f = __half22float2(hh);
  __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
  return *reinterpret_cast<uint32_t*>(&b);
}

// Four e4m3 codes (byte i of w = element i) -> four bf16 values (.x = elements 0,1; .y =
// elements 2,3), exactly, with integer ops and one bf16x2 multiply per pair (no conversion
// instructions).  Each code's sign goes to bit 15 of a 16-bit half and its 7 exponent+mantissa
// bits to bits 10..4: read as bf16 that is the code's value times 2^-120 (a normal code's
// exponent field reads e against bias 127 instead of 7; a subnormal code and zero line their
// 3 mantissa bits up under a zero exponent field in both formats).  Multiplying by 2^120 is
// exact.  Even elements are placed with left shifts, odd ones with right shifts; a byte
// permute puts the pairs back in order.
__device__ __forceinline__ uint2 e4m3x4_to_bf16x4(uint32_t w) {
  const uint32_t k = 0x7B807B80u;  // bf16x2 (2^120, 2^120)
  const uint32_t ev = ((w << 4) & 0x07F007F0u) | ((w << 8) & 0x80008000u);  // elements 0, 2
  const uint32_t od = ((w >> 4) & 0x07F007F0u) | (w & 0x80008000u);         // elements 1, 3
  uint32_t e2, o2;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(e2) : "r"(ev), "r"(k));
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(o2) : "r"(od), "r"(k));
  return make_uint2(__byte_perm(e2, o2, 0x5410), __byte_perm(e2, o2, 0x7632));
}

// silu(z) = z / (1 + e^-z) with the fast exponential and divide (a few ulp in fp32, far below
// the bf16 rounding of h); for very negative z the divisor overflows and the result is 0.
__device__ __forceinline__ float silu_f(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace tpx
