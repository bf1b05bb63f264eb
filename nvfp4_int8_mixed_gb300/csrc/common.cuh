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

// ---------------------------------------------- packed fp32 pair arithmetic
// sm_100-class f32x2 instructions: two IEEE round-to-nearest fp32 operations
// (no flush to zero) per instruction on a pair held in one 64-bit register.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
__device__ __forceinline__ void f2_unpack(uint64_t d, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(d));
}
__device__ __forceinline__ uint64_t f2_from_bf16x2(uint32_t w) { return f2_pack(bf16lo(w), bf16hi(w)); }
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
// bf16x2 word of a pair (lo in bits 0..15), round to nearest even.
__device__ __forceinline__ uint32_t f2_to_bf16x2(uint64_t d) {
  float lo, hi;
  f2_unpack(d, lo, hi);
  return pack_bf16x2(lo, hi);
}

// ------------------------------------------------------- NVFP4 arithmetic
// g = amax_t / 2688 (6 * 448), 1 when amax_t = 0.
__device__ __forceinline__ float nvfp4_global_scale(float amax_t) {
  return amax_t == 0.f ? 1.f : __fdiv_rn(amax_t, 2688.f);
}
// Scale of one 16-element block: S = E4M3(amax_b * 448 / amax_t) (0 when
// amax_t = 0), d = S * g.  Returns S's byte; r = 1/d, or 0 when d = 0 (the
// block's codes are then all +0, which the caller must write as 0).
__device__ __forceinline__ uint32_t nvfp4_block_scale(float amax_b, float amax_t, float g, float& r) {
  const float s = (amax_t == 0.f) ? 0.f : __fdiv_rn(__fmul_rn(amax_b, 448.f), amax_t);
  const uint32_t sb = e4m3_encode(s);
  const float d = __fmul_rn(e4m3_decode(sb), g);
  r = d != 0.f ? __frcp_rn(d) : 0.f;
  return sb;
}
// Eight bf16 values (four packed words) times r -> eight E2M1 codes; 0 when r = 0.
__device__ __forceinline__ uint32_t nvfp4_codes8(const uint32_t* pw, float r) {
  if (r == 0.f) return 0u;
  const uint64_t r2 = f2_pack(r, r);
  float y[8];
#pragma unroll
  for (int e = 0; e < 4; ++e) f2_unpack(f2_mul(f2_from_bf16x2(pw[e]), r2), y[2 * e], y[2 * e + 1]);
  return e2m1x8(y[0], y[1], y[2], y[3], y[4], y[5], y[6], y[7]);
}
// max(|a|, |b|) of each bf16 half in one instruction.  The magnitude is one
// of the inputs' magnitudes, unrounded; the sign bit of each half is the XOR
// of the inputs' signs, so callers mask it off once at the end.  Finite
// inputs only (a NaN gives the canonical NaN).
__device__ __forceinline__ uint32_t bf16x2_maxabs(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// |x| max of eight bf16 values (four packed words), as a float.
__device__ __forceinline__ float bf16x8_absmax(const uint32_t* pw) {
  const uint32_t a = bf16x2_maxabs(bf16x2_maxabs(pw[0], pw[1]), bf16x2_maxabs(pw[2], pw[3])) & 0x7FFF7FFFu;
  return __uint_as_float(max(a & 0xFFFFu, a >> 16) << 16);
}

// -------------------------------------------------------- INT8 arithmetic
// E2M1 code of an integer in [-4, 4].
__device__ __forceinline__ uint32_t digit_code(int d) {
  const uint32_t mag = (0x65420u >> (4 * (d < 0 ? -d : d))) & 0xFu;
  return mag | (d < 0 ? 8u : 0u);
}
// Digit split of an INT8 code q in [-128, 127]: byte 0 = E2M1 code of a,
// byte 1 = of b, byte 2 = of c, q = 64a + 8b + c, c = q mod 8 in [-3, 4],
// b likewise for (q - c)/8, a the rest.
__device__ __forceinline__ uint32_t digit_entry(int q) {
  const int c = ((q + 3) & 7) - 3;
  const int q1 = (q - c) >> 3;                 // exact: q - c is a multiple of 8
  const int b = ((q1 + 3) & 7) - 3;
  const int a = (q1 - b) >> 3;
  return digit_code(a) | (digit_code(b) << 8) | (digit_code(c) << 16);
}
// Eight bf16 values (four packed words) -> q = rne(x * inv), clamped to
// +-127 when CLAMP, returned as the bits of q + 1.5 * 2^23 (the low byte of
// each word is q as a two's complement byte).
template <bool CLAMP>
__device__ __forceinline__ void int8_encode8(const uint32_t* pw, float inv, uint32_t* qb) {
  constexpr float kMagic = 12582912.0f;        // 1.5 * 2^23
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float lo = __fmul_rn(bf16lo(pw[e]), inv), hi = __fmul_rn(bf16hi(pw[e]), inv);
    if (CLAMP) {
      lo = fminf(fmaxf(lo, -127.f), 127.f);
      hi = fminf(fmaxf(hi, -127.f), 127.f);
    }
    qb[2 * e] = __float_as_uint(__fadd_rn(lo, kMagic));
    qb[2 * e + 1] = __float_as_uint(__fadd_rn(hi, kMagic));
  }
}
// The three digit-plane words of eight consecutive codes (element 2j in the
// low nibble of byte j), from qb of int8_encode8 and a 256-entry digit_entry
// table indexed by the code's byte.
__device__ __forceinline__ void int8_planes8(const uint32_t* qb, const uint32_t* lut, uint32_t& p0, uint32_t& p1,
                                             uint32_t& p2) {
  uint32_t p[4];                               // byte k of p[j] = digit-k codes of elements 2j, 2j+1
#pragma unroll
  for (int j = 0; j < 4; ++j) p[j] = lut[qb[2 * j] & 0xFFu] | (lut[qb[2 * j + 1] & 0xFFu] << 4);
  const uint32_t x01 = __byte_perm(p[0], p[1], 0x5140);   // a01 a23 b01 b23
  const uint32_t x23 = __byte_perm(p[2], p[3], 0x5140);   // a45 a67 b45 b67
  const uint32_t c01 = __byte_perm(p[0], p[1], 0x0062);   // c01 c23
  const uint32_t c23 = __byte_perm(p[2], p[3], 0x0062);   // c45 c67
  p0 = __byte_perm(x01, x23, 0x5410);
  p1 = __byte_perm(x01, x23, 0x7632);
  p2 = __byte_perm(c01, c23, 0x5410);
}

// ------------------------------------------- delayed-scaling amax history
// A producer that quantizes its own output to NVFP4 in one pass cannot know
// that output's tensor amax; it scales by headroom * the amax its previous
// call recorded.  History word layout, uint32[4]: {previous call's amax
// (float bits), this call's running amax, CTA arrival ticket, unused};
// zero-initialised before the first call.  The last CTA of a call to arrive
// moves the running amax into the previous-amax word and clears the other
// two, so consecutive calls need no other kernel.
__device__ __forceinline__ float hist_prev(const uint32_t* h) { return __uint_as_float(__ldcg(h)); }
// One call per warp (or thread) holding a partial amax; fences its atomic.
__device__ __forceinline__ void hist_accumulate(uint32_t* h, float amax) {
  if (amax > 0.f) atomicMax(h + 1, __float_as_uint(amax));
  __threadfence();
}
// One thread per CTA, after a CTA barrier that follows every
// hist_accumulate of the CTA (or with the CTA's whole amax in cta_amax).
__device__ __forceinline__ void hist_arrive(uint32_t* h, float cta_amax = 0.f) {
  if (cta_amax > 0.f) atomicMax(h + 1, __float_as_uint(cta_amax));
  __threadfence();
  if (atomicAdd(h + 2, 1u) == gridDim.x * gridDim.y * gridDim.z - 1) {
    __threadfence();
    const uint32_t a = atomicExch(h + 1, 0u);
    atomicExch(h, a);
    atomicExch(h + 2, 0u);
  }
}

// ------------------------------------------- compressed update cache (MX)
// A block update cached as E4M3 codes with one power-of-two scale per 32
// consecutive elements: scale byte k + 127, k the smallest integer with the
// block's max |v| <= 448 * 2^k, clamped to [-127, 127] (-127 for a zero
// block); code = E4M3(v * 2^-k); value = E4M3(code) * 2^k.  Layout: n code
// bytes, then n/32 scale bytes.
__device__ __forceinline__ int mx_scale_exp(float amax) {
  const uint32_t b = __float_as_uint(amax);
  const int e = int((b >> 23) & 0xFFu);
  if (!(amax > 0.f) || e == 0) return -127;    // zero (or fp32-subnormal) maximum
  const int k = (e - 127) - 8 + ((b & 0x7FFFFFu) > 0x600000u ? 1 : 0);   // mantissa 1.75 = 0x600000
  return k < -127 ? -127 : (k > 127 ? 127 : k);
}
// 2^k exactly, k in [-127, 127] (2^-127 is an fp32 subnormal).
__device__ __forceinline__ float exp2i(int k) {
  return k >= -126 ? __uint_as_float(uint32_t(k + 127) << 23) : __uint_as_float(0x00400000u);
}
// Four floats -> four E4M3 codes (f0 in the low byte), round to nearest even, saturating.
__device__ __forceinline__ uint32_t e4m3x4(float f0, float f1, float f2, float f3) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(f1), "f"(f0));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(f3), "f"(f2));
  return uint32_t(lo) | (uint32_t(hi) << 16);
}
// Two E4M3 codes (low byte first) -> two floats (exact).
__device__ __forceinline__ void e4m3x2_to_f32(uint32_t two, float& lo, float& hi) {
  uint32_t h2;
  const uint16_t in = uint16_t(two & 0xFFFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
  asm("{ .reg .f16 a, b;\n mov.b32 {a, b}, %2;\n cvt.f32.f16 %0, a;\n cvt.f32.f16 %1, b; }"
      : "=f"(lo), "=f"(hi)
      : "r"(h2));
}
// Eight cached values: codes (two words, element 0 in the low byte) times 2^k.
__device__ __forceinline__ void mx_decode8(uint2 codes, float scale, float* v) {
  e4m3x2_to_f32(codes.x, v[0], v[1]);
  e4m3x2_to_f32(codes.x >> 16, v[2], v[3]);
  e4m3x2_to_f32(codes.y, v[4], v[5]);
  e4m3x2_to_f32(codes.y >> 16, v[6], v[7]);
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __fmul_rn(v[i], scale);
}

// Swizzled scale-factor byte offset: 128x4 atoms of 512 bytes.
__host__ __device__ __forceinline__ int64_t sf_offset(int64_t m, int64_t c, int64_t kc4) {
  return ((m >> 7) * (kc4 >> 2) + (c >> 2)) * 512 + (m & 31) * 16 + ((m & 127) >> 5) * 4 + (c & 3);
}

}  // namespace sixbit
