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
#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace sixbit {

namespace {

constexpr int kThreads = 256;

// ---------------------------------------------------------------- amax (a1)
// |x| maxima through bit patterns: for x >= 0 the IEEE bit order is the value
// order, so |x| = bits & ~sign and the max is an unsigned max (two bf16 per
// 32-bit word with a halfword max).  NaN inputs are not supported.
__device__ __forceinline__ uint32_t absmax_word(uint32_t acc, uint32_t w, uint16_t) {
  return __vmaxu2(acc, w & 0x7FFF7FFFu);
}
__device__ __forceinline__ uint32_t absmax_word(uint32_t acc, uint32_t w, float) {
  return max(acc, w & 0x7FFFFFFFu);
}
__device__ __forceinline__ float absmax_value(uint32_t acc, uint16_t) {
  return __uint_as_float(max(acc & 0xFFFFu, acc >> 16) << 16);
}
__device__ __forceinline__ float absmax_value(uint32_t acc, float) { return __uint_as_float(acc); }

// Contiguous tensor: every thread keeps 8 independent 16-byte loads in
// flight; one atomic max per CTA.
template <typename T>
__global__ void __launch_bounds__(kThreads) amax_flat_kernel(const T* __restrict__ x, int64_t nvec16, float* amax_out,
                                                             const uint8_t* pred) {
  if (pred && *pred == 0) return;
  __shared__ uint32_t red[kThreads / 32];
  constexpr int kU = 8;
  uint32_t acc = 0;
  const uint4* p = reinterpret_cast<const uint4*>(x);
  const int64_t stride = int64_t(gridDim.x) * kThreads;
  int64_t i = int64_t(blockIdx.x) * kThreads + threadIdx.x;
  // The last batch is predicated rather than finished one load at a time, so
  // a thread never waits on more than one memory round trip per kU vectors.
  for (; i < nvec16; i += kU * stride) {
    uint4 v[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u)
      v[u] = i + u * stride < nvec16 ? ldg_nc_v4(p + i + u * stride) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      acc = absmax_word(acc, v[u].x, T()); acc = absmax_word(acc, v[u].y, T());
      acc = absmax_word(acc, v[u].z, T()); acc = absmax_word(acc, v[u].w, T());
    }
  }
  float m = warp_max(absmax_value(acc, T()));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = __float_as_uint(m);
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t b = 0;
    for (int w = 0; w < kThreads / 32; ++w) b = max(b, red[w]);
    atomic_max_nonneg(amax_out, __uint_as_float(b));
  }
}

// Strided rows and/or per-row maxima: one warp per row, 8 vectors of 16
// bytes per lane in flight.
template <typename T>
__global__ void __launch_bounds__(kThreads) amax_rows_kernel(const T* __restrict__ x, int64_t M, int64_t K, int64_t ldx,
                                                             float* amax_out, float* row_amax_out, const uint8_t* pred) {
  if (pred && *pred == 0) return;
  constexpr int kE = 16 / sizeof(T);          // elements per 16-byte vector
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * kThreads) >> 5;
  const int64_t nvec = K / kE;
  float tmax = 0.f;
  for (int64_t m = warp; m < M; m += nwarps) {
    const uint4* row = reinterpret_cast<const uint4*>(x + m * ldx);
    uint32_t acc = 0;
    for (int64_t j0 = 0; j0 < nvec; j0 += 8 * 32) {
      uint4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int64_t j = j0 + u * 32 + lane;
        v[u] = j < nvec ? ldg_nc_v4(row + j) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        acc = absmax_word(acc, v[u].x, T()); acc = absmax_word(acc, v[u].y, T());
        acc = absmax_word(acc, v[u].z, T()); acc = absmax_word(acc, v[u].w, T());
      }
    }
    const float rmax = warp_max(absmax_value(acc, T()));
    if (row_amax_out && lane == 0) row_amax_out[m] = rmax;
    tmax = fmaxf(tmax, rmax);
  }
  if (amax_out && lane == 0) atomic_max_nonneg(amax_out, tmax);
}

// ------------------------------------------------------------ NVFP4 (a2/a4)
// One warp per row; one lane owns one 16-element scale block: the block
// amax, the E4M3 scale, the reciprocal and the 16 codes are computed once per
// block.  A warp covers 32 consecutive blocks (512 elements) of a row per
// step and keeps two steps of loads in flight.  Each lane writes its block's
// 16 codes as one 8-byte store; lanes 4j..4j+3 assemble their group's 4 scale
// bytes into one 32-bit word of the swizzled scale buffer, written by lane
// 4j.  Rows M..Mpad-1 get zero scales.
template <typename T> struct Block16;           // the raw 16 elements of one block
template <> struct Block16<uint16_t> {
  uint4 v[2];
  __device__ void load(const uint16_t* p) { v[0] = ldg_v4(p); v[1] = ldg_v4(p + 8); }
  __device__ void zero() { v[0] = v[1] = make_uint4(0, 0, 0, 0); }
  __device__ float amax() const {
    const uint32_t a0 = bf16x2_maxabs(bf16x2_maxabs(v[0].x, v[0].y), bf16x2_maxabs(v[0].z, v[0].w));
    const uint32_t a1 = bf16x2_maxabs(bf16x2_maxabs(v[1].x, v[1].y), bf16x2_maxabs(v[1].z, v[1].w));
    const uint32_t a = bf16x2_maxabs(a0, a1) & 0x7FFF7FFFu;
    return __uint_as_float(max(a & 0xFFFFu, a >> 16) << 16);
  }
  __device__ float at(int i) const {               // element i (compile-time i after unrolling)
    const uint32_t* w = &v[i >> 3].x;
    return (i & 1) ? bf16hi(w[(i & 7) >> 1]) : bf16lo(w[(i & 7) >> 1]);
  }
};
template <> struct Block16<float> {
  uint4 v[4];
  __device__ void load(const float* p) {
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = ldg_v4(p + 4 * i);
  }
  __device__ void zero() {
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = make_uint4(0, 0, 0, 0);
  }
  __device__ float amax() const {
    uint32_t a = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      a = max(a, v[i].x & 0x7FFFFFFFu); a = max(a, v[i].y & 0x7FFFFFFFu);
      a = max(a, v[i].z & 0x7FFFFFFFu); a = max(a, v[i].w & 0x7FFFFFFFu);
    }
    return __uint_as_float(a);
  }
  __device__ float at(int i) const { return __uint_as_float((&v[i >> 2].x)[i & 3]); }
};

// Work item = (row, pair of 32-block spans): a warp's two 16-byte loads per
// lane per block for 2 x 32 consecutive blocks (2 KB of bf16).  Warps are
// persistent and walk the items t = warp, warp + nwarps, ...; the next
// item's loads are issued before the current item is encoded and stored, so
// every warp always has a load in flight.  Consecutive warps take
// consecutive items (adjacent memory).
template <typename T>
__device__ __forceinline__ void nvfp4_load_item(const T* __restrict__ x, int64_t m, int sp0, int nspan, int nblk,
                                                int64_t M, int64_t ldx, int lane, Block16<T> (&blk)[2]) {
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int b = (sp0 + u) * 32 + lane;
    if (m < M && sp0 + u < nspan && b < nblk) blk[u].load(x + m * ldx + int64_t(b) * 16);
    else blk[u].zero();
  }
}

template <typename T>
__global__ void __launch_bounds__(kThreads) nvfp4_quant_kernel(const T* __restrict__ x, int64_t M, int64_t K, int64_t ldx,
                                                               const float* __restrict__ amax_ptr,
                                                               uint8_t* __restrict__ codes, uint8_t* __restrict__ sf,
                                                               float* g_out, const uint8_t* pred, int64_t Mpad) {
  if (pred && *pred == 0) return;
  const float amax_t = *amax_ptr;
  const float g = nvfp4_global_scale(amax_t);
  if (blockIdx.x == 0 && threadIdx.x == 0) *g_out = g;
  // 1 / (S g) for every E4M3 scale a satfinite encode can give (codes
  // 0..126), computed once per CTA exactly as the per-block form would
  __shared__ float rtab[128];
  if (threadIdx.x < 128) {
    const float d = __fmul_rn(e4m3_decode(threadIdx.x), g);
    rtab[threadIdx.x] = d != 0.f ? __frcp_rn(d) : 0.f;
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int64_t kc4 = K / 16;                 // K % 64 == 0 -> a multiple of 4
  const int nblk = int(K / 16);
  const int nspan = (nblk + 31) / 32;
  const int64_t ppr = (nspan + 1) / 2;        // items (span pairs) per row
  const int64_t items = Mpad * ppr;
  const int64_t warp = (int64_t(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * kThreads) >> 5;
  // Item it = (row m, span pair pr), it = m * ppr + pr.  A warp's items are
  // nwarps apart, i.e. dq rows and dr pairs: (m, pr) advance by additions.
  const int64_t dq = nwarps / ppr;
  const int dr = int(nwarps - dq * ppr);
  int64_t m = warp / ppr;
  int pr = int(warp - m * ppr);
  Block16<T> cur[2], nxt[2];
  if (warp < items) nvfp4_load_item(x, m, 2 * pr, nspan, nblk, M, ldx, lane, cur);
  for (int64_t it = warp; it < items; it += nwarps) {
    int64_t mn = m + dq;                      // the next item, it + nwarps
    int prn = pr + dr;
    if (prn >= int(ppr)) { prn -= int(ppr); ++mn; }
    if (it + nwarps < items) nvfp4_load_item(x, mn, 2 * prn, nspan, nblk, M, ldx, lane, nxt);
    const int sp0 = 2 * pr;
    const bool row_ok = m < M;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (sp0 + u >= nspan) break;            // warp-uniform
      const int b = (sp0 + u) * 32 + lane;
      float r;
      const float amax_b = cur[u].amax();
      const uint32_t sb = e4m3_encode(amax_t == 0.f ? 0.f : __fdiv_rn(__fmul_rn(amax_b, 448.f), amax_t));
      r = rtab[sb];
      uint32_t w0 = 0, w1 = 0;
      if constexpr (sizeof(T) == 2) {
        // bf16 pairs times r on the f32x2 pipe (no add follows, so no fusion)
        w0 = nvfp4_codes8(&cur[u].v[0].x, r);
        w1 = nvfp4_codes8(&cur[u].v[1].x, r);
      } else if (r != 0.f) {
        float y[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) y[e] = __fmul_rn(cur[u].at(e), r);
        w0 = e2m1x8(y[0], y[1], y[2], y[3], y[4], y[5], y[6], y[7]);
        w1 = e2m1x8(y[8], y[9], y[10], y[11], y[12], y[13], y[14], y[15]);
      }
      // 4 consecutive blocks (lanes 4j..4j+3) form one 32-bit word of the swizzled scale buffer
      uint32_t word = sb | (__shfl_down_sync(0xffffffffu, sb, 1) << 8);
      word |= __shfl_down_sync(0xffffffffu, word, 2) << 16;
      if (b < nblk) {
        if (row_ok) *reinterpret_cast<uint2*>(codes + m * (K / 2) + int64_t(b) * 8) = make_uint2(w0, w1);
        if ((lane & 3) == 0) *reinterpret_cast<uint32_t*>(sf + sf_offset(m, b, kc4)) = row_ok ? word : 0u;
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) cur[u] = nxt[u];
    m = mn;
    pr = prn;
  }
}

// ------------------------------------------------------------------ INT8 (a3)
// WPR warps per row, NVL 16-byte vectors (8 bf16) per lane: the whole row
// stays in registers between the amax reduction and the encode, so the input
// is read from HBM once.  Rows of up to 7680 elements take one warp each
// (independent warps, no CTA barrier); wider rows split over the CTA's 4
// warps, which exchange their partial row amax through shared memory.  Vector v of the row sits in warp v / (32*NVL) of
// the row's group, register slot (v / 32) % NVL, lane v % 32.  CTAs of 4
// warps take 4 / WPR rows per step.
// Encode: v = clamp(x * inv, +-127) rounded to nearest even by adding
// 1.5 * 2^23 (the low byte of the sum's bits is then q as a two's complement
// byte); the digit planes come from a 256-entry shared table.
// kClamp: a caller-given row amax may be below the true one, so x * inv is
// clamped to +-127; with the kernel's own amax |x * inv| already rounds to
// at most 127 and the clamp is skipped.
template <int NVL, int WPR, bool kClamp>
__global__ void __launch_bounds__(128) int8_quant_kernel(const uint16_t* __restrict__ x, int64_t M, int64_t K, int64_t ldx,
                                                         const float* __restrict__ row_amax_in,
                                                         int8_t* __restrict__ q, uint8_t* __restrict__ planes,
                                                         float* __restrict__ row_scale, const uint8_t* pred) {
  if (pred && *pred == 0) return;
  constexpr int RPC = 4 / WPR;
  __shared__ float red[4];
  __shared__ uint32_t lut[256];
  for (int i = threadIdx.x; i < 256; i += 128) lut[i] = digit_entry(int(int8_t(uint8_t(i))));
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rloc = warp / WPR, wpart = warp % WPR;
  const int64_t nvec = K / 8;
  const int64_t plane_stride = M * (K / 2);
  for (int64_t m0 = int64_t(blockIdx.x) * RPC; m0 < M; m0 += int64_t(gridDim.x) * RPC) {
    const int64_t m = m0 + rloc;
    const bool row_ok = m < M;
    const uint16_t* row = x + m * ldx;
    uint4 v[NVL];
#pragma unroll
    for (int i = 0; i < NVL; ++i) {
      const int64_t vi = int64_t(wpart * NVL + i) * 32 + lane;
      v[i] = (row_ok && vi < nvec) ? ldg_nc_v4(row + vi * 8) : make_uint4(0, 0, 0, 0);
    }
    float amax;
    if (row_amax_in) {
      amax = row_ok ? row_amax_in[m] : 0.f;
    } else {
      uint32_t acc = 0;
#pragma unroll
      for (int i = 0; i < NVL; ++i)
        acc = bf16x2_maxabs(acc, bf16x2_maxabs(bf16x2_maxabs(v[i].x, v[i].y), bf16x2_maxabs(v[i].z, v[i].w)));
      acc &= 0x7FFF7FFFu;
      amax = warp_max(__uint_as_float(max(acc & 0xFFFFu, acc >> 16) << 16));
      if (WPR > 1) {
        if (lane == 0) red[warp] = amax;
        __syncthreads();
#pragma unroll
        for (int w = 0; w < WPR; ++w) amax = fmaxf(amax, red[rloc * WPR + w]);
        __syncthreads();
      }
    }
    if (!row_ok) continue;                     // uniform per row group (after the barriers)
    const bool nz = amax > 0.f;
    const float inv = nz ? __fdiv_rn(127.f, amax) : 0.f;
    if (lane == 0 && wpart == 0) row_scale[m] = nz ? __fdiv_rn(amax, 127.f) : 0.f;
#pragma unroll
    for (int i = 0; i < NVL; ++i) {
      const int64_t vi = int64_t(wpart * NVL + i) * 32 + lane;
      if (vi >= nvec) continue;
      uint32_t qb[8];                          // bits of (v + magic): low byte = q
      int8_encode8<kClamp>(&v[i].x, inv, qb);
      if (q) {
        uint2 w;
        w.x = __byte_perm(__byte_perm(qb[0], qb[1], 0x0040), __byte_perm(qb[2], qb[3], 0x0040), 0x5410);
        w.y = __byte_perm(__byte_perm(qb[4], qb[5], 0x0040), __byte_perm(qb[6], qb[7], 0x0040), 0x5410);
        *reinterpret_cast<uint2*>(q + m * K + vi * 8) = w;
      }
      if (planes) {
        uint32_t p0, p1, p2;
        int8_planes8(qb, lut, p0, p1, p2);
        uint8_t* base = planes + m * (K / 2) + vi * 4;
        *reinterpret_cast<uint32_t*>(base) = p0;
        *reinterpret_cast<uint32_t*>(base + plane_stride) = p1;
        *reinterpret_cast<uint32_t*>(base + 2 * plane_stride) = p2;
      }
    }
  }
}

// Plain INT8 codes -> the three E2M1 digit planes the W4A8 GEMM reads (for
// callers that hold int8 activations from elsewhere).  Exact: a table
// lookup per code.  One thread per 16 codes (a 16-byte load, three 8-byte
// stores), grid-stride over rows of K/16 groups.
__global__ void __launch_bounds__(kThreads) int8_planes_kernel(const int8_t* __restrict__ q, int64_t M, int64_t K,
                                                               int64_t ldq, uint8_t* __restrict__ planes) {
  __shared__ uint32_t lut[256];
  for (int i = threadIdx.x; i < 256; i += kThreads) lut[i] = digit_entry(int(int8_t(uint8_t(i))));
  __syncthreads();
  const int64_t gpr = K / 16;                      // 16-code groups per row
  const int64_t total = M * gpr;
  const int64_t plane_stride = M * (K / 2);
  // group gi = (row m, group c), gi = m * gpr + c; the grid stride is dq rows
  // and dc groups, so (m, c) advance by additions
  const int64_t stride = int64_t(gridDim.x) * kThreads;
  const int64_t dq = stride / gpr, dc = stride - dq * gpr;
  const int64_t g0 = int64_t(blockIdx.x) * kThreads + threadIdx.x;
  int64_t m = g0 / gpr, c = g0 - m * gpr;
  for (int64_t gi = g0; gi < total; gi += stride) {
    const uint4 v = ldg_nc_v4(q + m * ldq + c * 16);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t p0[2], p1[2], p2[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t qb[8];                              // int8_planes8 reads the code from each entry's low byte
#pragma unroll
      for (int e = 0; e < 8; ++e) qb[e] = (w[2 * h + (e >> 2)] >> (8 * (e & 3))) & 0xFFu;
      int8_planes8(qb, lut, p0[h], p1[h], p2[h]);
    }
    uint8_t* base = planes + m * (K / 2) + c * 8;
    *reinterpret_cast<uint2*>(base) = make_uint2(p0[0], p0[1]);
    *reinterpret_cast<uint2*>(base + plane_stride) = make_uint2(p1[0], p1[1]);
    *reinterpret_cast<uint2*>(base + 2 * plane_stride) = make_uint2(p2[0], p2[1]);
    m += dq;
    c += dc;
    if (c >= gpr) {
      c -= gpr;
      ++m;
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
                const uint8_t* pred, int num_sms, cudaStream_t s) {
  if (amax_out && cudaMemsetAsync(amax_out, 0, sizeof(float), s) != cudaSuccess) return kELaunch;
  const int esz = dtype == 1 ? 2 : 4;
  const bool flat = !row_amax_out && ldx == K && (M * K * esz) % 16 == 0;
  if (flat) {
    const int64_t nvec16 = M * K * esz / 16;
    const int grid = grid_for(nvec16, kThreads * 8, num_sms, 8);
    if (dtype == 1)
      amax_flat_kernel<uint16_t><<<grid, kThreads, 0, s>>>(static_cast<const uint16_t*>(x), nvec16, amax_out, pred);
    else
      amax_flat_kernel<float><<<grid, kThreads, 0, s>>>(static_cast<const float*>(x), nvec16, amax_out, pred);
  } else {
    const int grid = grid_for(M, kThreads / 32, num_sms, 16);
    if (dtype == 1)
      amax_rows_kernel<uint16_t><<<grid, kThreads, 0, s>>>(static_cast<const uint16_t*>(x), M, K, ldx, amax_out, row_amax_out, pred);
    else
      amax_rows_kernel<float><<<grid, kThreads, 0, s>>>(static_cast<const float*>(x), M, K, ldx, amax_out, row_amax_out, pred);
  }
  return cudaGetLastError() == cudaSuccess ? kOk : kELaunch;
}

int launch_nvfp4_quant(const void* x, int dtype, int64_t M, int64_t K, int64_t ldx, const float* amax,
                       uint8_t* codes, uint8_t* sf, float* g_out, const uint8_t* pred, int num_sms, cudaStream_t s) {
  const int64_t Mpad = cdiv(M, 128) * 128;
  const int64_t items = Mpad * cdiv(cdiv(K / 16, 32), 2);
  // persistent: as many CTAs as are resident (each warp walks many items);
  // the residency is looked up once per input type (thread-safe statics)
  auto resident = [](const void* kern) {
    int n = 0;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kThreads, 0) == cudaSuccess && n > 0 ? n : 1;
  };
  static const int ps_bf16 = resident(reinterpret_cast<const void*>(nvfp4_quant_kernel<uint16_t>));
  static const int ps_f32 = resident(reinterpret_cast<const void*>(nvfp4_quant_kernel<float>));
  const int ps = dtype == 1 ? ps_bf16 : ps_f32;
  const int grid = grid_for(items, kThreads / 32, num_sms, ps);
  if (dtype == 1)
    nvfp4_quant_kernel<uint16_t><<<grid, kThreads, 0, s>>>(static_cast<const uint16_t*>(x), M, K, ldx, amax, codes, sf,
                                                           g_out, pred, Mpad);
  else
    nvfp4_quant_kernel<float><<<grid, kThreads, 0, s>>>(static_cast<const float*>(x), M, K, ldx, amax, codes, sf, g_out,
                                                        pred, Mpad);
  return cudaGetLastError() == cudaSuccess ? kOk : kELaunch;
}

int launch_int8_planes(const int8_t* q, int64_t M, int64_t K, int64_t ldq, uint8_t* planes, int num_sms,
                       cudaStream_t s) {
  int8_planes_kernel<<<grid_for(M * (K / 16), kThreads, num_sms, 8), kThreads, 0, s>>>(q, M, K, ldq, planes);
  return cudaGetLastError() == cudaSuccess ? kOk : kELaunch;
}

int launch_int8_quant(const void* x, int64_t M, int64_t K, int64_t ldx, const float* row_amax_in, int8_t* q,
                      uint8_t* planes, float* row_scale, const uint8_t* pred, int num_sms, cudaStream_t s) {
  auto xs = static_cast<const uint16_t*>(x);
  // rows per CTA step = 4 / warps-per-row
  auto go = [&](auto clamp) {
    constexpr bool C = decltype(clamp)::value;
    if (K <= 2048)
      int8_quant_kernel<8, 1, C><<<grid_for(M, 4, num_sms, 16), 128, 0, s>>>(xs, M, K, ldx, row_amax_in, q, planes, row_scale, pred);
    else if (K <= 3072)    // one warp a row: no CTA barrier per row (K = 3072: 37.5 us vs 49.8 for 8 x 2)
      int8_quant_kernel<12, 1, C><<<grid_for(M, 4, num_sms, 16), 128, 0, s>>>(xs, M, K, ldx, row_amax_in, q, planes, row_scale, pred);
    else if (K <= 4096)
      int8_quant_kernel<8, 2, C><<<grid_for(M, 2, num_sms, 16), 128, 0, s>>>(xs, M, K, ldx, row_amax_in, q, planes, row_scale, pred);
    else if (K <= 7680)    // one warp a row again: 12 rows in flight per SM, no barrier (K = 7680: 90.8 vs 101 us)
      int8_quant_kernel<30, 1, C><<<grid_for(M, 4, num_sms, 16), 128, 0, s>>>(xs, M, K, ldx, row_amax_in, q, planes, row_scale, pred);
    else if (K <= 8192)
      int8_quant_kernel<8, 4, C><<<grid_for(M, 1, num_sms, 16), 128, 0, s>>>(xs, M, K, ldx, row_amax_in, q, planes, row_scale, pred);
    else if (K <= 12288)   // 12 vectors a lane: fewer registers than 16, more CTAs resident
      int8_quant_kernel<12, 4, C><<<grid_for(M, 1, num_sms, 16), 128, 0, s>>>(xs, M, K, ldx, row_amax_in, q, planes, row_scale, pred);
    else
      int8_quant_kernel<16, 4, C><<<grid_for(M, 1, num_sms, 12), 128, 0, s>>>(xs, M, K, ldx, row_amax_in, q, planes, row_scale, pred);
  };
  if (row_amax_in) go(std::true_type{});
  else go(std::false_type{});
  return cudaGetLastError() == cudaSuccess ? kOk : kELaunch;
}

}  // namespace sixbit
