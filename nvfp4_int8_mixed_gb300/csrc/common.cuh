// Shared device helpers of the sixbit library (sm_103a).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace sixbit {

// Error codes mirrored from include/sixbit.h.
constexpr int kOk = 0, kEInval = -1, kEShape = -2, kEAlign = -3, kELaunch = -4, kEDevice = -5;

// Device error word (defined in api.cu); kernels get its address as an argument.
enum DeviceError : int { kErrNone = 0, kErrWaitTimeout = 1 };

__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// float -> bf16 bits, round to nearest even (hardware cvt).
__device__ __forceinline__ uint16_t f32_to_bf16(float x) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(x));
  return r;
}
// two floats -> packed bf16x2 (lo in bits 0..15).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// E2M1 x2: returns a byte with cvt(lo) in bits 0..3 and cvt(hi) in bits 4..7.
// Round to nearest even, saturate to +-6, keep the sign of a zero result.
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
  uint16_t r;
  asm("{ .reg .b8 t; cvt.rn.satfinite.e2m1x2.f32 t, %1, %2; cvt.u16.u8 %0, t; }" : "=h"(r) : "f"(hi), "f"(lo));
  return r & 0xFFu;
}

// Eight floats -> eight E2M1 codes in one 32-bit word, element i in nibble i
// (round to nearest even, saturating at 6).
__device__ __forceinline__ uint32_t e2m1x8(float f0, float f1, float f2, float f3, float f4, float f5, float f6,
                                           float f7) {
  uint32_t r;
  asm("{ .reg .b8 t0, t1, t2, t3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 t0, %2, %1;\n"
      " cvt.rn.satfinite.e2m1x2.f32 t1, %4, %3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 t2, %6, %5;\n"
      " cvt.rn.satfinite.e2m1x2.f32 t3, %8, %7;\n"
      " mov.b32 %0, {t0, t1, t2, t3}; }"
      : "=r"(r)
      : "f"(f0), "f"(f1), "f"(f2), "f"(f3), "f"(f4), "f"(f5), "f"(f6), "f"(f7));
  return r;
}

// float >= 0 -> E4M3 byte, round to nearest even, saturate at 448.
__device__ __forceinline__ uint32_t e4m3_encode(float x) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(x));
  return r & 0xFFu;
}
// E4M3 byte -> float (exact: every E4M3 value is an fp16 value).
__device__ __forceinline__ float e4m3_decode(uint32_t b) {
  uint32_t h2;
  uint16_t in = uint16_t(b & 0xFF);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
  float f;
  const uint16_t lo = uint16_t(h2 & 0xFFFF);
  asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(lo));
  return f;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// max of non-negative floats through their bit patterns (monotone for x >= 0).
__device__ __forceinline__ void atomic_max_nonneg(float* p, float v) {
  atomicMax(reinterpret_cast<unsigned int*>(p), __float_as_uint(v));
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}
__device__ __forceinline__ uint4 ldg_v4(const void* p) {
  return *reinterpret_cast<const uint4*>(p);
}

__host__ __device__ __forceinline__ int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Swizzled scale-factor byte offset: 128x4 atoms of 512 bytes.
__host__ __device__ __forceinline__ int64_t sf_offset(int64_t m, int64_t c, int64_t kc4) {
  return ((m >> 7) * (kc4 >> 2) + (c >> 2)) * 512 + (m & 31) * 16 + ((m & 127) >> 5) * 4 + (c & 3);
}

}  // namespace sixbit
