// Activation / weight quantizers: tensor and row amax (a1), NVFP4 (a2, a4),
// per-token INT8 with its E2M1 digit planes (a3).
//
// Method: 6Bit-Diffusion ("Abstract", mlsanity.com page) quantizes each
// linear layer's activations on the fly to NVFP4 or INT8.  The encodings:
//  NVFP4: g = amax/2688; per 16-element block S = E4M3(amax_b*448/amax),
//         code = E2M1(x * (1/(S*g))), all float32 round-to-nearest.
//  INT8:  per row inv = 127/amax_m, q = clamp(rne(x*inv), +-127), s = amax_m/127.
// All kernels are HBM-bound streaming passes: 16-byte vector loads issued
// several at a time per thread, coalesced across the warp, grids sized as a
// multiple of the SM count.
#include "common.cuh"
#include "kernels.h"

namespace sixbit {

namespace {

constexpr int kThreads = 256;

template <typename T> struct In;
template <> struct In<uint16_t> {   // bf16 bits
  __device__ static void load8(const uint16_t* p, float* f) {
    uint4 v = ldg_nc_v4(p);
    f[0] = bf16lo(v.x); f[1] = bf16hi(v.x); f[2] = bf16lo(v.y); f[3] = bf16hi(v.y);
    f[4] = bf16lo(v.z); f[5] = bf16hi(v.z); f[6] = bf16lo(v.w); f[7] = bf16hi(v.w);
  }
};
template <> struct In<float> {
  __device__ static void load8(const float* p, float* f) {
    uint4 a = ldg_nc_v4(p), b = ldg_nc_v4(p + 4);
    f[0] = __uint_as_float(a.x); f[1] = __uint_as_float(a.y); f[2] = __uint_as_float(a.z); f[3] = __uint_as_float(a.w);
    f[4] = __uint_as_float(b.x); f[5] = __uint_as_float(b.y); f[6] = __uint_as_float(b.z); f[7] = __uint_as_float(b.w);
  }
};

// ---------------------------------------------------------------- amax (a1)
// One warp per row: row max |x| (optional) and the tensor max via an atomic
// max on the float bits (values are >= 0, so the bit order is the value order).
template <typename T>
__global__ void __launch_bounds__(kThreads) amax_rows_kernel(const T* __restrict__ x, int64_t M, int64_t K, int64_t ldx,
                                                             float* amax_out, float* row_amax_out) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * kThreads) >> 5;
  float tmax = 0.f;
  const int64_t nvec = K / 8;
  for (int64_t m = warp; m < M; m += nwarps) {
    const T* row = x + m * ldx;
    float rmax = 0.f;
    int64_t j = lane;
    for (; j + 96 < nvec; j += 128) {          // 4 vectors in flight per lane
      float f[4][8];
#pragma unroll
      for (int u = 0; u < 4; ++u) In<T>::load8(row + (j + 32 * u) * 8, f[u]);
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int e = 0; e < 8; ++e) rmax = fmaxf(rmax, fabsf(f[u][e]));
    }
    for (; j < nvec; j += 32) {
      float f[8];
      In<T>::load8(row + j * 8, f);
#pragma unroll
      for (int e = 0; e < 8; ++e) rmax = fmaxf(rmax, fabsf(f[e]));
    }
    rmax = warp_max(rmax);
    if (row_amax_out && lane == 0) row_amax_out[m] = rmax;
    tmax = fmaxf(tmax, rmax);
  }
  if (amax_out && lane == 0) atomic_max_nonneg(amax_out, tmax);
}

// ------------------------------------------------------------ NVFP4 (a2/a4)
// The tensor is walked as 64-element groups (4 scale blocks).  A warp takes
// 4 groups per step: lanes 8j..8j+7 hold the 8 vectors of group j, a lane
// pair holds one 16-element block.  Each lane writes its 8 codes as one
// 32-bit word; lane 8j assembles the group's 4 scale bytes into one 32-bit
// word of the swizzled scale buffer.
template <typename T>
__global__ void __launch_bounds__(kThreads) nvfp4_quant_kernel(const T* __restrict__ x, int64_t M, int64_t K, int64_t ldx,
                                                               const float* __restrict__ amax_ptr,
                                                               uint8_t* __restrict__ codes, uint8_t* __restrict__ sf,
                                                               float* g_out, const uint8_t* pred, int64_t Mpad) {
  if (pred && *pred == 0) return;
  const float amax_t = *amax_ptr;
  const float g = (amax_t == 0.f) ? 1.f : __fdiv_rn(amax_t, 2688.f);
  if (blockIdx.x == 0 && threadIdx.x == 0) *g_out = g;
  const int lane = threadIdx.x & 31;
  const int sub = lane >> 3, vec = lane & 7;
  const int64_t gpr = K / 64;
  const int64_t kc4 = K / 16;               // K % 64 == 0 -> already a multiple of 4
  const int64_t total = Mpad * gpr;
  const int64_t warp = (int64_t(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * kThreads) >> 5;
  constexpr int kU = 2;                     // warp steps unrolled (loads in flight)
  for (int64_t G0 = warp * 4 * kU; G0 < total; G0 += nwarps * 4 * kU) {
    float f[kU][8];
    int64_t mm[kU], gg[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int64_t G = G0 + u * 4 + sub;
      mm[u] = G / gpr;
      gg[u] = G - mm[u] * gpr;
      if (G < total && mm[u] < M) In<T>::load8(x + mm[u] * ldx + gg[u] * 64 + vec * 8, f[u]);
      else {
#pragma unroll
        for (int e = 0; e < 8; ++e) f[u][e] = 0.f;
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int64_t G = G0 + u * 4 + sub;
      float am = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) am = fmaxf(am, fabsf(f[u][e]));
      am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));        // block of 16 = lane pair
      const float s = (amax_t == 0.f) ? 0.f : __fdiv_rn(__fmul_rn(am, 448.f), amax_t);
      const uint32_t sb = e4m3_encode(s);
      const float d = __fmul_rn(e4m3_decode(sb), g);
      uint32_t w = 0;
      if (d != 0.f) {
        const float r = __frcp_rn(d);
#pragma unroll
        for (int e = 0; e < 4; ++e)
          w |= e2m1x2(__fmul_rn(f[u][2 * e], r), __fmul_rn(f[u][2 * e + 1], r)) << (8 * e);
      }
      // scale bytes of blocks 0..3 of this group live in lanes 8j, 8j+2, 8j+4, 8j+6
      const uint32_t s0 = __shfl_sync(0xffffffffu, sb, (lane & ~7) + 0);
      const uint32_t s1 = __shfl_sync(0xffffffffu, sb, (lane & ~7) + 2);
      const uint32_t s2 = __shfl_sync(0xffffffffu, sb, (lane & ~7) + 4);
      const uint32_t s3 = __shfl_sync(0xffffffffu, sb, (lane & ~7) + 6);
      if (G < total) {
        const int64_t m = mm[u], grp = gg[u];
        if (m < M) *reinterpret_cast<uint32_t*>(codes + m * (K / 2) + grp * 32 + vec * 4) = w;
        if (vec == 0) {
          const uint32_t word = (m < M) ? (s0 | (s1 << 8) | (s2 << 16) | (s3 << 24)) : 0u;
          *reinterpret_cast<uint32_t*>(sf + sf_offset(m, grp * 4, kc4)) = word;
        }
      }
    }
  }
}

// ------------------------------------------------------------------ INT8 (a3)
__device__ __forceinline__ uint32_t digit_code(int d) {    // integer in [-4, 4] -> E2M1 code
  const uint32_t mag = (0x65420u >> (4 * (d < 0 ? -d : d))) & 0xFu;
  return mag | (d < 0 ? 8u : 0u);
}

// One warp per row.  Pass 1 finds the row amax (unless given); pass 2
// re-reads the row (an L2 hit) and writes codes and/or digit planes.
__global__ void __launch_bounds__(kThreads) int8_quant_kernel(const uint16_t* __restrict__ x, int64_t M, int64_t K, int64_t ldx,
                                                              const float* __restrict__ row_amax_in,
                                                              int8_t* __restrict__ q, uint8_t* __restrict__ planes,
                                                              float* __restrict__ row_scale, const uint8_t* pred) {
  if (pred && *pred == 0) return;
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * kThreads) >> 5;
  const int64_t nvec = K / 8;
  const int64_t plane_stride = M * (K / 2);
  for (int64_t m = warp; m < M; m += nwarps) {
    const uint16_t* row = x + m * ldx;
    float amax;
    if (row_amax_in) {
      amax = row_amax_in[m];
    } else {
      float rmax = 0.f;
      int64_t j = lane;
      for (; j + 96 < nvec; j += 128) {
        float f[4][8];
#pragma unroll
        for (int u = 0; u < 4; ++u) In<uint16_t>::load8(row + (j + 32 * u) * 8, f[u]);
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int e = 0; e < 8; ++e) rmax = fmaxf(rmax, fabsf(f[u][e]));
      }
      for (; j < nvec; j += 32) {
        float f[8];
        In<uint16_t>::load8(row + j * 8, f);
#pragma unroll
        for (int e = 0; e < 8; ++e) rmax = fmaxf(rmax, fabsf(f[e]));
      }
      amax = warp_max(rmax);
    }
    const bool nz = amax > 0.f;
    const float inv = nz ? __fdiv_rn(127.f, amax) : 0.f;
    if (lane == 0) row_scale[m] = nz ? __fdiv_rn(amax, 127.f) : 0.f;
    for (int64_t j = lane; j < nvec; j += 32) {
      float f[8];
      In<uint16_t>::load8(row + j * 8, f);
      int qi[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        int v = __float2int_rn(__fmul_rn(f[e], inv));
        qi[e] = nz ? max(-127, min(127, v)) : 0;
      }
      if (q) {
        uint2 w;
        w.x = (qi[0] & 0xFF) | ((qi[1] & 0xFF) << 8) | ((qi[2] & 0xFF) << 16) | (uint32_t(qi[3] & 0xFF) << 24);
        w.y = (qi[4] & 0xFF) | ((qi[5] & 0xFF) << 8) | ((qi[6] & 0xFF) << 16) | (uint32_t(qi[7] & 0xFF) << 24);
        *reinterpret_cast<uint2*>(q + m * K + j * 8) = w;
      }
      if (planes) {
        uint32_t pa = 0, pb = 0, pc = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int c = ((qi[e] + 3) & 7) - 3;          // q mod 8 in [-3, 4]
          const int q1 = (qi[e] - c) >> 3;              // exact: q - c is a multiple of 8
          const int b = ((q1 + 3) & 7) - 3;
          const int a = (q1 - b) >> 3;                  // in [-2, 2]
          pa |= digit_code(a) << (4 * e);
          pb |= digit_code(b) << (4 * e);
          pc |= digit_code(c) << (4 * e);
        }
        uint8_t* base = planes + m * (K / 2) + j * 4;
        *reinterpret_cast<uint32_t*>(base) = pa;
        *reinterpret_cast<uint32_t*>(base + plane_stride) = pb;
        *reinterpret_cast<uint32_t*>(base + 2 * plane_stride) = pc;
      }
    }
  }
}

int grid_for(int64_t work_items, int per_block, int num_sms, int waves = 8) {
  int64_t want = cdiv(work_items, per_block);
  int64_t cap = int64_t(num_sms) * waves;
  return int(want < 1 ? 1 : (want < cap ? want : cap));
}

}  // namespace

int launch_amax(const void* x, int dtype, int64_t M, int64_t K, int64_t ldx, float* amax_out, float* row_amax_out,
                int num_sms, cudaStream_t s) {
  if (amax_out && cudaMemsetAsync(amax_out, 0, sizeof(float), s) != cudaSuccess) return kELaunch;
  const int grid = grid_for(M, kThreads / 32, num_sms);
  if (dtype == 1)
    amax_rows_kernel<uint16_t><<<grid, kThreads, 0, s>>>(static_cast<const uint16_t*>(x), M, K, ldx, amax_out, row_amax_out);
  else
    amax_rows_kernel<float><<<grid, kThreads, 0, s>>>(static_cast<const float*>(x), M, K, ldx, amax_out, row_amax_out);
  return cudaGetLastError() == cudaSuccess ? kOk : kELaunch;
}

int launch_nvfp4_quant(const void* x, int dtype, int64_t M, int64_t K, int64_t ldx, const float* amax,
                       uint8_t* codes, uint8_t* sf, float* g_out, const uint8_t* pred, int num_sms, cudaStream_t s) {
  const int64_t Mpad = cdiv(M, 128) * 128;
  const int64_t warps_needed = cdiv(Mpad * (K / 64), 8);
  const int grid = grid_for(warps_needed, kThreads / 32, num_sms);
  if (dtype == 1)
    nvfp4_quant_kernel<uint16_t><<<grid, kThreads, 0, s>>>(static_cast<const uint16_t*>(x), M, K, ldx, amax, codes, sf,
                                                           g_out, pred, Mpad);
  else
    nvfp4_quant_kernel<float><<<grid, kThreads, 0, s>>>(static_cast<const float*>(x), M, K, ldx, amax, codes, sf, g_out,
                                                        pred, Mpad);
  return cudaGetLastError() == cudaSuccess ? kOk : kELaunch;
}

int launch_int8_quant(const void* x, int64_t M, int64_t K, int64_t ldx, const float* row_amax_in, int8_t* q,
                      uint8_t* planes, float* row_scale, const uint8_t* pred, int num_sms, cudaStream_t s) {
  const int grid = grid_for(M, kThreads / 32, num_sms);
  int8_quant_kernel<<<grid, kThreads, 0, s>>>(static_cast<const uint16_t*>(x), M, K, ldx, row_amax_in, q, planes,
                                              row_scale, pred);
  return cudaGetLastError() == cudaSuccess ? kOk : kELaunch;
}

}  // namespace sixbit
