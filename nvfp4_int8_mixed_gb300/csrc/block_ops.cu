// Block-level kernels: Gamma/Delta/r2 pass (a7), DMPQ assignment (a8),
// TDC decision and reuse (a9), and the LayerNorm of the block harness; the
// compressed-update-cache versions of a7 / a9, the LayerNorm that quantizes
// its own output (NVFP4 by delayed scaling, INT8 exact), and the pair
// statistics of the DMPQ calibration side (E_rel, update similarity).
//
// Method: 6Bit-Diffusion, thelatestinai.com page -- Figure 2 (Gamma = block
// relative L1 input/output distance at the preceding step drives DMPQ; TDC
// decides from the updates of the two preceding steps), Figure 3 (per-layer
// line alpha*Gamma + beta), Figure 4 (updates compared by relative L2).
// Decisions are computed and consumed on the device: no host round trip.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace sixbit {

// Test switch (set through sixbit_debug_stall_staging): nonzero makes every
// warp of the LayerNorm producer's row-prefetch form, and every CTA of the
// Gamma passes, wait for its first row or tile on a barrier that is never
// signalled, so that bounded wait expires and the device-error path runs.
__device__ int g_sixbit_stall_stage = 0;

int set_stage_stall(int on) {
  return cudaMemcpyToSymbol(g_sixbit_stall_stage, &on, sizeof(on)) == cudaSuccess ? kOk : kELaunch;
}

namespace {

constexpr int kThreads = 256;
constexpr int kTile = 8192;                   // elements per tile of the Gamma pass
constexpr int kVecPerThread = kTile / (8 * kThreads);   // 4 x 16-byte vectors per operand
constexpr int kGammaCtasPerSm = 2;          // 256 CTAs on 152 SMs: at most two per SM

struct GammaWs {                              // layout of the scratch buffer
  unsigned int counter;                       // CTAs finished (reset by the last one)
  unsigned int pad[3];
};

// The fixed reduction tree of the Gamma pass (and of the pair statistics).
// Its result depends only on the input, never on the device:
//   * lane t of a tile (t = 0..255) owns elements j*2048 + 8t + e (j = 0..3,
//     e = 0..7) and adds their terms one at a time in increasing element
//     order, in float32 (round to nearest, no contraction);
//   * the 256 lane sums: a butterfly inside each warp (partners t^16, t^8,
//     t^4, t^2, t^1), then the 8 warp sums by w + (w+4), + (w+2), + (w+1);
//   * the float32 tile sums are widened to float64 and added in order into
//     256 chains, chain k holding tiles k, k+256, ... (starting from +0);
//   * the 256 chain sums are halved (k + (k+128), ..., + (k+1)).
// The grid is min(tiles, 256) CTAs and CTA k walks exactly the tiles of
// chain k, so it adds them into its chain as it goes; the last CTA to finish
// only halves the 256 chain sums.  (Reading every tile partial back in one
// CTA had cost 13 us at 34M elements: float64 throughput on one SM.)
constexpr int kChains = 256;
static_assert(kChains == kThreads, "the last CTA halves one chain sum per thread");

// Per-tile combine of 4 lane sums, batched: each warp's butterfly result
// goes to shared memory slot `it % kBatch` (it = the CTA's tile counter);
// after every kBatch tiles (and after the last) one CTA barrier, threads
// 0..4*kBatch-1 each combine one (tile, sum) over the 8 warps into `part`,
// and a second barrier frees the slots; then threads 0..3 add the batch's
// tile sums, in tile order, into this CTA's chain.  Two barriers per kBatch
// tiles instead of one per tile.  `part` is next written after the next
// batch's first barrier, which threads 0..3 reach only after reading it.
constexpr int kBatch = 32;
struct TileRed {
  float w[kBatch][kThreads / 32][4];
  float part[kBatch][4];
};
__device__ __forceinline__ void tile_combine4(float v[4], TileRed& red, int it, bool flush, double& chain) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v[i] = __fadd_rn(v[i], __shfl_xor_sync(0xffffffffu, v[i], o));
  const int slot = it % kBatch;
  if (lane == 0)
#pragma unroll
    for (int i = 0; i < 4; ++i) red.w[slot][w][i] = v[i];
  if (slot == kBatch - 1 || flush) {
    __syncthreads();
    if (threadIdx.x < 4 * (slot + 1)) {
      const int b = threadIdx.x >> 2, i = threadIdx.x & 3;
      float g[kThreads / 32];
#pragma unroll
      for (int k = 0; k < kThreads / 32; ++k) g[k] = red.w[b][k][i];
#pragma unroll
      for (int h = kThreads / 64; h > 0; h >>= 1)
#pragma unroll
        for (int k = 0; k < h; ++k) g[k] = __fadd_rn(g[k], g[k + h]);
      red.part[b][i] = g[0];
    }
    __syncthreads();
    if (threadIdx.x < 4)
      for (int b = 0; b <= slot; ++b) chain = __dadd_rn(chain, double(red.part[b][threadIdx.x]));
  }
}

// End of a pass: every CTA stores its 4 chain sums (threads 0..3 hold them);
// the last CTA to finish halves the 256 chains' sums (chains of CTAs that do
// not exist, when tiles < 256, are +0) and returns true in thread 0 with the
// 4 sums.
__device__ __forceinline__ bool tiles_finish(GammaWs* ws, double* chains, double chain, double out[4]) {
  __shared__ bool is_last;
  __shared__ double dsm[kThreads][4];
  if (threadIdx.x < 4) {
    chains[4 * blockIdx.x + threadIdx.x] = chain;
    __threadfence();                          // this CTA's chain sums, before the ticket
  }
  __syncthreads();
  if (threadIdx.x == 0) is_last = atomicAdd(&ws->counter, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!is_last) return false;
  __threadfence();
#pragma unroll
  for (int i = 0; i < 4; ++i) dsm[threadIdx.x][i] = threadIdx.x < gridDim.x ? __ldcg(chains + 4 * threadIdx.x + i) : 0.0;
  __syncthreads();
  // halving: partners 128, 64, 32 apart through shared memory, then 16..1
  // apart by shuffles inside warp 0 (lane k adds lane k + h; lanes >= h
  // compute values that no later level reads)
  for (int h = kThreads / 2; h >= 32; h >>= 1) {
    if (threadIdx.x < h)
#pragma unroll
      for (int i = 0; i < 4; ++i) dsm[threadIdx.x][i] = __dadd_rn(dsm[threadIdx.x][i], dsm[threadIdx.x + h][i]);
    __syncthreads();
  }
  if (threadIdx.x >= 32) return false;
  double r[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) r[i] = dsm[threadIdx.x][i];
#pragma unroll
  for (int h = 16; h > 0; h >>= 1)
#pragma unroll
    for (int i = 0; i < 4; ++i) r[i] = __dadd_rn(r[i], __shfl_down_sync(0xffffffffu, r[i], h));
  if (threadIdx.x != 0) return false;
#pragma unroll
  for (int i = 0; i < 4; ++i) out[i] = r[i];
  ws->counter = 0u;
  return true;
}

// Gamma / r2 from the four sums; TDC counters advanced.
__device__ __forceinline__ void gamma_publish(const double S[4], bool do_r2, bool computed, float* gamma_out,
                                              float* r2_out, int32_t* tdc_state) {
  if (gamma_out) *gamma_out = (S[1] == 0.0) ? 0.f : __double2float_rn(__ddiv_rn(S[0], S[1]));
  if (do_r2) *r2_out = (S[3] == 0.0) ? __int_as_float(0x7f800000) : __double2float_rn(__ddiv_rn(S[2], S[3]));
  if (tdc_state) {
    if (computed) { tdc_state[0] += 1; tdc_state[1] = 0; }
    else tdc_state[1] += 1;
  }
}

// acc + x*x with the product rounded once (no contraction into an FMA).
__device__ __forceinline__ float add_sq(float acc, float x) { return __fadd_rn(acc, __fmul_rn(x, x)); }

// Tile staging of the Gamma passes: thread 0 copies a tile's inputs into
// shared memory with bulk copies (the TMA engine), completing on one mbarrier
// per stage, two stages deep, so a CTA's next tile is in flight while it
// works on the current one (at most two CTAs share an SM, and one CTA alone
// on an SM would otherwise wait for every tile).  Each wait is bounded; a CTA
// that gives up records the device error, lets its copies in flight land and
// leaves its tile loop (its sums are then meaningless, the error says so).
constexpr uint32_t kStageSpinCap = 1u << 22;  // polls of a bounded stage wait
__device__ __forceinline__ void stage_bar_init(uint32_t bar) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar));
}
__device__ __forceinline__ bool stage_bar_wait(uint32_t bar, uint32_t parity) {
  for (uint32_t i = 0; i < kStageSpinCap; ++i) {
    uint32_t ok;
    asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity)
                 : "memory");
    if (ok) return true;
  }
  return false;
}
__device__ __forceinline__ void stage_expect(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// bytes % 16 == 0, both addresses 16-byte aligned
__device__ __forceinline__ void stage_copy(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// a7: one pass over (in, out, previous Delta).  Per element:
//   d = f32(out) - f32(in); S1 += |d|; S0 += |in|;
//   if computed: D_new = bf16(d) (stored over D_old); if r2 wanted:
//   e = f32(D_new) - f32(D_old); Sd += e*e; So += D_old^2.
// The sums follow the fixed tree above: CTA k walks the tiles of chain k
// (t = k, k + 256, ...) and the last CTA to finish halves the chain sums,
// writes Gamma / r2 and advances the TDC counters.  A tile's whole 8-element
// groups arrive through the shared-memory stages; a partial last group is
// read directly.
constexpr size_t kGammaStage = size_t(3) * kTile * 2;    // in, out, Delta_old: 16 KB each
constexpr size_t kGammaSmem = 2 * kGammaStage;             // 96 KB of dynamic shared memory
__global__ void __launch_bounds__(kThreads, kGammaCtasPerSm) gamma_kernel(
    const uint16_t* __restrict__ xin, const uint16_t* __restrict__ xout, int64_t n, uint16_t* delta, float* gamma_out,
    float* r2_out, int32_t* tdc_state, const uint8_t* computed_ptr, GammaWs* ws, double* chains, int* err) {
  __shared__ TileRed red;
  __shared__ __align__(8) uint64_t sbar[3];   // two stages + one never signalled (test switch)
  extern __shared__ __align__(128) uint8_t gstage[];   // [2 stages][in | out | Delta_old][kTile bf16]
  const bool computed = computed_ptr ? (*computed_ptr != 0) : true;
  const bool do_delta = computed && delta != nullptr;
  const bool do_r2 = do_delta && r2_out != nullptr && (tdc_state ? tdc_state[0] >= 1 : true);
  const int64_t ntiles = cdiv(n, kTile);
  const uint32_t bar0 = uint32_t(__cvta_generic_to_shared(&sbar[0]));
  const uint32_t sbase = uint32_t(__cvta_generic_to_shared(gstage));
  auto issue = [&](int64_t t, int s) {       // tile t's whole 8-element groups into stage s
    const int64_t base = t * kTile;
    const uint32_t nb = uint32_t((n - base < kTile ? n - base : kTile) / 8 * 8) * 2u;
    const uint32_t bar = bar0 + 8u * uint32_t(s), dst = sbase + uint32_t(s) * uint32_t(kGammaStage);
    stage_expect(bar, nb * (do_r2 ? 3u : 2u));
    if (nb) {
      stage_copy(dst, xin + base, nb, bar);
      stage_copy(dst + kTile * 2u, xout + base, nb, bar);
      if (do_r2) stage_copy(dst + 2u * kTile * 2u, delta + base, nb, bar);
    }
  };
  if (threadIdx.x == 0) {
    stage_bar_init(bar0);
    stage_bar_init(bar0 + 8u);
    stage_bar_init(bar0 + 16u);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    if (blockIdx.x < ntiles) issue(blockIdx.x, 0);
  }
  __syncthreads();
  int it = 0;
  double chain = 0.0;                         // this CTA's chain (threads 0..3)
  for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++it) {
    const int64_t base = t * kTile;
    const int s = it & 1;
    const bool more = t + gridDim.x < ntiles;
    // stage s ^ 1 was last read one tile ago, before that tile's closing barrier
    if (threadIdx.x == 0 && more) issue(t + gridDim.x, s ^ 1);
    const bool stall = it == 0 && g_sixbit_stall_stage != 0;   // test switch: wait on the silent barrier
    const bool landed = stage_bar_wait(stall ? bar0 + 16u : bar0 + 8u * uint32_t(s), uint32_t(it >> 1) & 1u);
    if (__syncthreads_or(!landed)) {          // one verdict for the whole CTA
      if (threadIdx.x == 0) {
        if (err) atomicExch(err, int(kErrWaitTimeout));
        stage_bar_wait(bar0 + 8u * uint32_t(s), uint32_t(it >> 1) & 1u);
        if (more) stage_bar_wait(bar0 + 8u * uint32_t(s ^ 1), uint32_t((it + 1) >> 1) & 1u);
      }
      break;
    }
    const uint4* sv = reinterpret_cast<const uint4*>(gstage + size_t(s) * kGammaStage);
    float v[4] = {0.f, 0.f, 0.f, 0.f};          // lane sums S1, S0, Sd, So of this tile
    uint4 vi[kVecPerThread], vo[kVecPerThread], vd[kVecPerThread];
#pragma unroll
    for (int i = 0; i < kVecPerThread; ++i) {
      const int64_t idx = base + (int64_t(i) * kThreads + threadIdx.x) * 8;
      if (idx + 8 <= n) {
        const int o = i * kThreads + threadIdx.x;   // 16-byte group within the tile
        vi[i] = sv[o];
        vo[i] = sv[kTile / 8 + o];
        if (do_r2) vd[i] = sv[2 * (kTile / 8) + o];
      }
    }
#pragma unroll
    for (int i = 0; i < kVecPerThread; ++i) {
      const int64_t idx = base + (int64_t(i) * kThreads + threadIdx.x) * 8;
      if (idx >= n) continue;
      if (idx + 8 <= n) {
        const uint32_t* a = &vi[i].x;
        const uint32_t* b = &vo[i].x;
        const uint32_t* c = &vd[i].x;
        uint4 w;
        uint32_t* pw = &w.x;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float i0 = bf16lo(a[e]), i1 = bf16hi(a[e]);
          const float d0 = __fsub_rn(bf16lo(b[e]), i0), d1 = __fsub_rn(bf16hi(b[e]), i1);
          v[0] = __fadd_rn(__fadd_rn(v[0], fabsf(d0)), fabsf(d1));
          v[1] = __fadd_rn(__fadd_rn(v[1], fabsf(i0)), fabsf(i1));
          pw[e] = pack_bf16x2(d0, d1);         // D_new: one rounding of the fp32 difference
          if (do_r2) {
            const float e0 = __fsub_rn(bf16lo(pw[e]), bf16lo(c[e])), e1 = __fsub_rn(bf16hi(pw[e]), bf16hi(c[e]));
            v[2] = add_sq(add_sq(v[2], e0), e1);
            v[3] = add_sq(add_sq(v[3], bf16lo(c[e])), bf16hi(c[e]));
          }
        }
        if (do_delta) *reinterpret_cast<uint4*>(delta + idx) = w;
      } else {                                  // ragged tail (scalar, same element order)
        const int cnt = int(n - idx);
        for (int e = 0; e < cnt; ++e) {
          const float fi = bf16_to_f32(xin[idx + e]);
          const float d = __fsub_rn(bf16_to_f32(xout[idx + e]), fi);
          v[0] = __fadd_rn(v[0], fabsf(d));
          v[1] = __fadd_rn(v[1], fabsf(fi));
          const uint16_t dn = f32_to_bf16(d);
          if (do_r2) {
            const float fd = bf16_to_f32(delta[idx + e]);
            v[2] = add_sq(v[2], __fsub_rn(bf16_to_f32(dn), fd));
            v[3] = add_sq(v[3], fd);
          }
          if (do_delta) delta[idx + e] = dn;
        }
      }
    }
    tile_combine4(v, red, it, t + gridDim.x >= ntiles, chain);
    __syncthreads();                          // stage s read by every thread before it is refilled
  }
  double S[4];
  if (tiles_finish(ws, chains, chain, S)) gamma_publish(S, do_r2, computed, gamma_out, r2_out, tdc_state);
}

// a7 with the compressed update cache (an extension; layout in common.cuh):
// the same pass, but the previous update is read as E4M3 codes times its
// block scale, r2 compares the exact bf16 D_new with that cached value, and
// D_new is stored encoded.  Four consecutive threads hold one 32-element
// block (8 elements each): its maximum is two shuffles, and the first of the
// four reads the old scale byte and writes the new one (so its read comes
// before its own write).  n % 32 == 0.
// Stage of the compressed-cache pass: in, out (16 KB each), the cached codes
// (8 KB) and, for a whole tile, its 256 scale bytes (a partial last tile
// reads its few scale bytes directly: a bulk copy moves multiples of 16 B).
constexpr size_t kGammaMxStage = size_t(2) * kTile * 2 + kTile + kTile / 32;   // 41,216 bytes
constexpr size_t kGammaMxSmem = 2 * kGammaMxStage;
__global__ void __launch_bounds__(kThreads, kGammaCtasPerSm) gamma_mx_kernel(
    const uint16_t* __restrict__ xin, const uint16_t* __restrict__ xout, int64_t n, uint8_t* cache, float* gamma_out,
    float* r2_out, int32_t* tdc_state, const uint8_t* computed_ptr, GammaWs* ws, double* chains, int* err) {
  __shared__ TileRed red;
  __shared__ __align__(8) uint64_t sbar[3];   // two stages + one never signalled (test switch)
  extern __shared__ __align__(128) uint8_t gstage[];   // [2 stages][in | out | codes | scales]
  const bool computed = computed_ptr ? (*computed_ptr != 0) : true;
  const bool do_delta = computed && cache != nullptr;
  const bool do_r2 = do_delta && r2_out != nullptr && (tdc_state ? tdc_state[0] >= 1 : true);
  uint8_t* scales = cache ? cache + n : nullptr;
  const int lane = threadIdx.x & 31;
  const bool first = (lane & 3) == 0;
  const int64_t ntiles = cdiv(n, kTile);
  const uint32_t bar0 = uint32_t(__cvta_generic_to_shared(&sbar[0]));
  const uint32_t sbase = uint32_t(__cvta_generic_to_shared(gstage));
  auto issue = [&](int64_t t, int s) {       // tile t (n % 32 == 0: whole 32-element blocks) into stage s
    const int64_t base = t * kTile;
    const uint32_t el = uint32_t(n - base < kTile ? n - base : kTile);
    const bool whole = el == uint32_t(kTile);
    const uint32_t bar = bar0 + 8u * uint32_t(s), dst = sbase + uint32_t(s) * uint32_t(kGammaMxStage);
    stage_expect(bar, 4u * el + (do_r2 ? el + (whole ? el / 32u : 0u) : 0u));
    stage_copy(dst, xin + base, 2u * el, bar);
    stage_copy(dst + 2u * kTile, xout + base, 2u * el, bar);
    if (do_r2) {
      stage_copy(dst + 4u * kTile, cache + base, el, bar);
      if (whole) stage_copy(dst + 5u * kTile, scales + base / 32, el / 32u, bar);
    }
  };
  if (threadIdx.x == 0) {
    stage_bar_init(bar0);
    stage_bar_init(bar0 + 8u);
    stage_bar_init(bar0 + 16u);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    if (blockIdx.x < ntiles) issue(blockIdx.x, 0);
  }
  __syncthreads();
  int it = 0;
  double chain = 0.0;                         // this CTA's chain (threads 0..3)
  for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++it) {
    const int64_t base = t * kTile;
    const int s = it & 1;
    const bool more = t + gridDim.x < ntiles;
    if (threadIdx.x == 0 && more) issue(t + gridDim.x, s ^ 1);   // read one tile ago, before its closing barrier
    const bool stall = it == 0 && g_sixbit_stall_stage != 0;   // test switch: wait on the silent barrier
    const bool landed = stage_bar_wait(stall ? bar0 + 16u : bar0 + 8u * uint32_t(s), uint32_t(it >> 1) & 1u);
    if (__syncthreads_or(!landed)) {          // one verdict for the whole CTA
      if (threadIdx.x == 0) {
        if (err) atomicExch(err, int(kErrWaitTimeout));
        stage_bar_wait(bar0 + 8u * uint32_t(s), uint32_t(it >> 1) & 1u);
        if (more) stage_bar_wait(bar0 + 8u * uint32_t(s ^ 1), uint32_t((it + 1) >> 1) & 1u);
      }
      break;
    }
    const uint8_t* st = gstage + size_t(s) * kGammaMxStage;
    const bool whole = n - base >= kTile;
    float v[4] = {0.f, 0.f, 0.f, 0.f};          // lane sums S1, S0, Sd, So of this tile (missing elements add +0)
    uint4 vi[kVecPerThread], vo[kVecPerThread];
    uint2 vc[kVecPerThread];
    uint32_t vs[kVecPerThread];
#pragma unroll
    for (int i = 0; i < kVecPerThread; ++i) {
      const int o = i * kThreads + threadIdx.x;     // 8-element group within the tile
      const int64_t idx = base + int64_t(o) * 8;
      vi[i] = vo[i] = make_uint4(0, 0, 0, 0);
      vc[i] = make_uint2(0, 0);
      vs[i] = 0;
      if (idx < n) {                          // n % 32 == 0: whole 8-element groups
        vi[i] = reinterpret_cast<const uint4*>(st)[o];
        vo[i] = reinterpret_cast<const uint4*>(st + 2 * kTile)[o];
        if (do_r2) {
          vc[i] = reinterpret_cast<const uint2*>(st + 4 * kTile)[o];
          if (first) vs[i] = whole ? st[5 * kTile + o / 4] : scales[idx / 32];
        }
      }
    }
#pragma unroll
    for (int i = 0; i < kVecPerThread; ++i) {
      const int64_t idx = base + (int64_t(i) * kThreads + threadIdx.x) * 8;
      const bool valid = idx < n;               // uniform over each group of four threads
      const uint32_t* a = &vi[i].x;
      const uint32_t* b = &vo[i].x;
      uint32_t pw[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float i0 = bf16lo(a[e]), i1 = bf16hi(a[e]);
        const float d0 = __fsub_rn(bf16lo(b[e]), i0), d1 = __fsub_rn(bf16hi(b[e]), i1);
        v[0] = __fadd_rn(__fadd_rn(v[0], fabsf(d0)), fabsf(d1));
        v[1] = __fadd_rn(__fadd_rn(v[1], fabsf(i0)), fabsf(i1));
        pw[e] = pack_bf16x2(d0, d1);           // D_new: one rounding of the fp32 difference
      }
      if (do_r2) {
        const uint32_t sc = __shfl_sync(0xffffffffu, vs[i], lane & ~3);
        float c[8];
        mx_decode8(vc[i], exp2i(int(sc) - 127), c);
        if (valid) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float e0 = __fsub_rn(bf16lo(pw[e]), c[2 * e]), e1 = __fsub_rn(bf16hi(pw[e]), c[2 * e + 1]);
            v[2] = add_sq(add_sq(v[2], e0), e1);
            v[3] = add_sq(add_sq(v[3], c[2 * e]), c[2 * e + 1]);
          }
        }
      }
      if (do_delta) {
        float am = bf16x8_absmax(pw);
        am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
        am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
        const int k = mx_scale_exp(am);
        const float inv = exp2i(-k);
        float y[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          y[2 * e] = __fmul_rn(bf16lo(pw[e]), inv);
          y[2 * e + 1] = __fmul_rn(bf16hi(pw[e]), inv);
        }
        if (valid) {
          *reinterpret_cast<uint2*>(cache + idx) =
              make_uint2(e4m3x4(y[0], y[1], y[2], y[3]), e4m3x4(y[4], y[5], y[6], y[7]));
          if (first) scales[idx / 32] = uint8_t(k + 127);
        }
      }
    }
    tile_combine4(v, red, it, t + gridDim.x >= ntiles, chain);
    __syncthreads();                          // stage s read by every thread before it is refilled
  }
  double S[4];
  if (tiles_finish(ws, chains, chain, S)) gamma_publish(S, do_r2, computed, gamma_out, r2_out, tdc_state);
}

// Calibration diagnostic (DMPQ side, Figures 1 and 4): one pass over two
// tensors, {sum (a-b)^2, sum b^2, sum a*b, sum a^2}, each term rounded once
// (d = a - b, then d*d; b*b; a*b; a*a), summed by the fixed tree of the Gamma
// pass, so the four float64 sums do not depend on the grid.
template <typename T>
__device__ __forceinline__ void load8(const T* p, int64_t i, float (&v)[8]);
template <>
__device__ __forceinline__ void load8<uint16_t>(const uint16_t* p, int64_t i, float (&v)[8]) {
  const uint4 w = ldg_nc_v4(p + i);
  const uint32_t* pw = &w.x;
#pragma unroll
  for (int e = 0; e < 4; ++e) { v[2 * e] = bf16lo(pw[e]); v[2 * e + 1] = bf16hi(pw[e]); }
}
template <>
__device__ __forceinline__ void load8<float>(const float* p, int64_t i, float (&v)[8]) {
  const uint4 w0 = ldg_nc_v4(p + i), w1 = ldg_nc_v4(p + i + 4);
  v[0] = __uint_as_float(w0.x); v[1] = __uint_as_float(w0.y); v[2] = __uint_as_float(w0.z); v[3] = __uint_as_float(w0.w);
  v[4] = __uint_as_float(w1.x); v[5] = __uint_as_float(w1.y); v[6] = __uint_as_float(w1.z); v[7] = __uint_as_float(w1.w);
}

template <typename TA, typename TB>
__global__ void __launch_bounds__(kThreads, kGammaCtasPerSm) pair_stats_kernel(const TA* __restrict__ a,
                                                                               const TB* __restrict__ b, int64_t n,
                                                                               double* out, GammaWs* ws,
                                                                               double* chains) {
  __shared__ TileRed red;
  const int64_t ntiles = cdiv(n, kTile);
  int it = 0;
  double chain = 0.0;                         // this CTA's chain (threads 0..3)
  for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++it) {
    float v[4] = {0.f, 0.f, 0.f, 0.f};          // lane sums of (a-b)^2, b^2, a*b, a^2
#pragma unroll
    for (int i = 0; i < kVecPerThread; ++i) {
      const int64_t idx = t * kTile + (int64_t(i) * kThreads + threadIdx.x) * 8;
      if (idx >= n) continue;                   // n % 8 == 0: whole vectors only
      float va[8], vb[8];
      load8(a, idx, va);
      load8(b, idx, vb);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        v[0] = add_sq(v[0], __fsub_rn(va[e], vb[e]));
        v[1] = add_sq(v[1], vb[e]);
        v[2] = __fadd_rn(v[2], __fmul_rn(va[e], vb[e]));
        v[3] = add_sq(v[3], va[e]);
      }
    }
    tile_combine4(v, red, it, t + gridDim.x >= ntiles, chain);
  }
  double S[4];
  if (tiles_finish(ws, chains, chain, S))
#pragma unroll
    for (int i = 0; i < 4; ++i) out[i] = S[i];
}

// a8: p = f32(f32(alpha*Gamma) + beta); NVFP4 iff step > 0 and p < tau.
__global__ void dmpq_kernel(const float* __restrict__ gamma, const float* __restrict__ alpha,
                            const float* __restrict__ beta, const int32_t* __restrict__ layer_block,
                            int32_t n_layers, float tau, const int32_t* step, uint8_t* use_nvfp4, uint8_t* gates) {
  const int l = blockIdx.x * blockDim.x + threadIdx.x;
  if (l >= n_layers) return;
  const float p = __fadd_rn(__fmul_rn(alpha[l], gamma[layer_block[l]]), beta[l]);
  const uint8_t f = (*step > 0 && p < tau) ? 1 : 0;
  if (use_nvfp4) use_nvfp4[l] = f;
  if (gates) { gates[2 * l] = f; gates[2 * l + 1] = 1 - f; }
}

// a9: every CTA evaluates the (read-only) decision; CTA 0 publishes it; on a
// skip all CTAs write out = bf16(f32(in) + f32(delta)).  refresh_every > 0
// (a periodic-refresh PDR variant) forces a computed step whenever
// *step % refresh_every == 0.
__global__ void __launch_bounds__(kThreads) tdc_kernel(const uint16_t* __restrict__ xin, const uint16_t* __restrict__ delta,
                                                       int64_t n, const float* r2, float tau2, int32_t max_skip,
                                                       int32_t refresh_every, const int32_t* step,
                                                       const int32_t* tdc_state, uint8_t* compute_out,
                                                       uint16_t* __restrict__ out, uint8_t* gates, int32_t n_gates) {
  const bool refresh = refresh_every > 0 && (*step % refresh_every) == 0;
  const bool skip = !refresh && tdc_state[0] >= 2 && *r2 < tau2 && tdc_state[1] < max_skip;
  if (blockIdx.x == 0) {
    if (threadIdx.x == 0) *compute_out = skip ? 0 : 1;
    if (skip && gates)
      for (int i = threadIdx.x; i < n_gates; i += blockDim.x) gates[i] = 0;
  }
  if (!skip) return;
  const int64_t nvec = n / 8;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t v = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; v < nvec; v += stride) {
    const uint4 a = ldg_nc_v4(xin + v * 8), b = ldg_nc_v4(delta + v * 8);
    const uint32_t* pa = &a.x;
    const uint32_t* pb = &b.x;
    uint4 w;
    uint32_t* pw = &w.x;
#pragma unroll
    for (int e = 0; e < 4; ++e)
      pw[e] = pack_bf16x2(__fadd_rn(bf16lo(pa[e]), bf16lo(pb[e])), __fadd_rn(bf16hi(pa[e]), bf16hi(pb[e])));
    *reinterpret_cast<uint4*>(out + v * 8) = w;
  }
  if (blockIdx.x == 0)
    for (int64_t i = nvec * 8 + threadIdx.x; i < n; i += blockDim.x)
      out[i] = f32_to_bf16(__fadd_rn(bf16_to_f32(xin[i]), bf16_to_f32(delta[i])));
}

// LayerNorm without affine, one warp per row; float32 mean, then the
// centered second moment; y = (x - mean) / sqrt(var + eps) rounded to bf16.
__global__ void __launch_bounds__(kThreads) layernorm_kernel(const uint16_t* __restrict__ x, int64_t M, int64_t H, int64_t ldx,
                                                             float eps, uint16_t* __restrict__ y, int64_t ldy,
                                                             float* amax_out, float* row_amax_out, const uint8_t* pred) {
  if (pred && *pred == 0) return;
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * kThreads) >> 5;
  const int64_t nvec = H / 8;
  float tmax = 0.f;
  for (int64_t m = warp; m < M; m += nwarps) {
    const uint16_t* row = x + m * ldx;
    float s = 0.f;
    for (int64_t j = lane; j < nvec; j += 32) {
      const uint4 v = ldg_v4(row + j * 8);
      const uint32_t* p = &v.x;
#pragma unroll
      for (int e = 0; e < 4; ++e) s += bf16lo(p[e]) + bf16hi(p[e]);
    }
    const float mean = __fdiv_rn(warp_sum(s), float(H));
    float q = 0.f;
    for (int64_t j = lane; j < nvec; j += 32) {
      const uint4 v = ldg_v4(row + j * 8);
      const uint32_t* p = &v.x;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float a = bf16lo(p[e]) - mean, b = bf16hi(p[e]) - mean;
        q += a * a + b * b;
      }
    }
    const float var = __fdiv_rn(warp_sum(q), float(H));
    const float rstd = __fdiv_rn(1.f, __fsqrt_rn(var + eps));
    float rmax = 0.f;
    for (int64_t j = lane; j < nvec; j += 32) {
      const uint4 v = ldg_v4(row + j * 8);
      const uint32_t* p = &v.x;
      uint4 w;
      uint32_t* pw = &w.x;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        pw[e] = pack_bf16x2((bf16lo(p[e]) - mean) * rstd, (bf16hi(p[e]) - mean) * rstd);
        rmax = fmaxf(rmax, fmaxf(fabsf(bf16lo(pw[e])), fabsf(bf16hi(pw[e]))));
      }
      *reinterpret_cast<uint4*>(y + m * ldy + j * 8) = w;
    }
    rmax = warp_max(rmax);
    if (row_amax_out && lane == 0) row_amax_out[m] = rmax;
    tmax = fmaxf(tmax, rmax);
  }
  if (amax_out && lane == 0) atomic_max_nonneg(amax_out, tmax);
}

// a9 with the compressed update cache: the decision as tdc_kernel; a
// skipped block's output is bf16(in + E4M3(code) * 2^k).  n % 32 == 0.
__global__ void __launch_bounds__(kThreads) tdc_mx_kernel(const uint16_t* __restrict__ xin,
                                                          const uint8_t* __restrict__ cache, int64_t n, const float* r2,
                                                          float tau2, int32_t max_skip, int32_t refresh_every,
                                                          const int32_t* step, const int32_t* tdc_state,
                                                          uint8_t* compute_out, uint16_t* __restrict__ out,
                                                          uint8_t* gates, int32_t n_gates) {
  const bool refresh = refresh_every > 0 && (*step % refresh_every) == 0;
  const bool skip = !refresh && tdc_state[0] >= 2 && *r2 < tau2 && tdc_state[1] < max_skip;
  if (blockIdx.x == 0) {
    if (threadIdx.x == 0) *compute_out = skip ? 0 : 1;
    if (skip && gates)
      for (int i = threadIdx.x; i < n_gates; i += blockDim.x) gates[i] = 0;
  }
  if (!skip) return;
  const uint8_t* scales = cache + n;
  const int64_t nvec = n / 8;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t v = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; v < nvec; v += stride) {
    const uint4 a = ldg_nc_v4(xin + v * 8);
    float c[8];
    mx_decode8(*reinterpret_cast<const uint2*>(cache + v * 8), exp2i(int(scales[v / 4]) - 127), c);
    const uint32_t* pa = &a.x;
    uint4 w;
    uint32_t* pw = &w.x;
#pragma unroll
    for (int e = 0; e < 4; ++e)
      pw[e] = pack_bf16x2(__fadd_rn(bf16lo(pa[e]), c[2 * e]), __fadd_rn(bf16hi(pa[e]), c[2 * e + 1]));
    *reinterpret_cast<uint4*>(out + v * 8) = w;
  }
}

// LayerNorm that quantizes its own output for the next linear layer.  One
// warp per row, the row held in registers so x is read once: lane l holds
// the 16-element blocks l, l + 32, ... (NB per lane, 32 contiguous bytes
// each), so a lane owns whole NVFP4 blocks and computes each block's scale
// once.  float32 statistics in packed pairs (f32x2): mean = sum / H, var =
// sum (x - mean)^2 / H, y = bf16((x - mean) * (1 / sqrt(var + eps))).
// Outputs (each optional):
//   y              bf16 [M, ldy];
//   amax_out, row_amax_out  tensor / row |y| maxima;
//   NVFP4 (when nv): codes [M, H/2], scales (swizzled, rows padded to 128,
//                  pads zero) and g, by delayed scaling from `hist`
//                  (amax_t = headroom * the previous call's amax); lanes
//                  4j..4j+3 hold one 4-block scale word;
//   INT8 (when i8): digit planes [3][M][H/2] and row scales from the row's
//                  own amax (the exact per-token quantizer).
// hist (nullable) records this call's tensor amax for the next call.
// H % 16 == 0.
// Threads per CTA: rows of more than 4 blocks a lane need ~170 registers a
// thread, so 4-warp CTAs (3 resident per SM) keep more warps in flight than
// 8-warp ones (1 resident).
// Row prefetch: each warp owns kLnBufs row buffers in shared memory.  Lane 0
// copies the warp's next rows into them with bulk copies (the TMA engine,
// completing on one mbarrier per buffer), so a row's load is in flight while
// the previous row is normalized and encoded; the lanes read their blocks
// from shared memory.  A buffer is refilled only after every lane of the
// warp has read it.
template <int NB>
constexpr int kLnThreads = NB >= 6 ? 128 : 256;
constexpr int kLnBufs = 2;
constexpr uint32_t kLnSpinCap = 1u << 22;     // polls of a bounded row wait

__device__ __forceinline__ void ln_bar_init(uint32_t bar) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar));
}
__device__ __forceinline__ bool ln_bar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for a row buffer (every lane polls); false if the cap ran out.
__device__ __forceinline__ bool ln_bar_wait(uint32_t bar, uint32_t parity) {
  for (uint32_t i = 0; i < kLnSpinCap; ++i)
    if (ln_bar_try(bar, parity)) return true;
  return false;
}
// One row (bytes % 16 == 0, both addresses 16-byte aligned) into shared memory.
__device__ __forceinline__ void ln_row_copy(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

template <int NB, bool PF>
__global__ void __launch_bounds__(kLnThreads<NB>) ln_quant_kernel(const LnQuantCall a) {
  constexpr int LT = kLnThreads<NB>;
  if (a.pred && *a.pred == 0) return;
  extern __shared__ __align__(128) uint8_t ln_rows[];   // [LT / 32][kLnBufs][2 H] bytes
  __shared__ __align__(8) uint64_t ln_bar[LT / 32][kLnBufs + 1];   // + one never signalled (test switch)
  __shared__ uint32_t lut[256];
  __shared__ float red[LT / 32];
  const bool nv = a.codes != nullptr && (a.nv_pred == nullptr || *a.nv_pred != 0);
  const bool i8 = a.planes != nullptr && (a.i8_pred == nullptr || *a.i8_pred != 0);
  if (i8) {
    for (int i = threadIdx.x; i < 256; i += LT) lut[i] = digit_entry(int(int8_t(uint8_t(i))));
    __syncthreads();
  }
  const float amax_t = a.hist ? __fmul_rn(a.headroom, hist_prev(a.hist)) : 0.f;
  const float g = nvfp4_global_scale(amax_t);
  if (nv && blockIdx.x == 0 && threadIdx.x == 0) *a.g_out = g;
  // 1 / (S g) for every E4M3 scale a satfinite encode can give (codes
  // 0..126), computed once per CTA exactly as the per-block form would
  __shared__ float rtab[128];
  if (nv) {
    for (int i = threadIdx.x; i < 128; i += LT) {
      const float d = __fmul_rn(e4m3_decode(uint32_t(i)), g);
      rtab[i] = d != 0.f ? __frcp_rn(d) : 0.f;
    }
    __syncthreads();
  }
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t(blockIdx.x) * LT + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * LT) >> 5;
  const int64_t M = a.M, H = a.H, nblk = H / 16, kc4 = H / 16;
  const int64_t Mpad = nv ? cdiv(M, 128) * 128 : M;
  const int64_t plane_stride = M * (H / 2);
  const int wib = threadIdx.x >> 5;            // warp in CTA
  const uint32_t rbytes = uint32_t(H) * 2u;
  const uint32_t rbuf = uint32_t(__cvta_generic_to_shared(ln_rows)) + uint32_t(wib * kLnBufs) * rbytes;
  const uint32_t rbar = uint32_t(__cvta_generic_to_shared(&ln_bar[wib][0]));
  if (PF && lane == 0) {
#pragma unroll
    for (int j = 0; j <= kLnBufs; ++j) ln_bar_init(rbar + 8u * j);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
#pragma unroll
    for (int j = 0; j < kLnBufs; ++j)          // the warp's first rows
      if (warp + j * nwarps < M) ln_row_copy(rbuf + j * rbytes, a.x + (warp + j * nwarps) * a.ldx, rbytes, rbar + 8u * j);
  }
  if (PF) __syncwarp();
  float tmax = 0.f;
  int64_t k = 0;                               // rows < M come first in a warp's walk: k counts them
  for (int64_t m = warp; m < Mpad; m += nwarps, ++k) {
    if (m >= M) {                              // pad rows of the scale layout
#pragma unroll
      for (int i = 0; i < NB; ++i) {
        const int64_t b = int64_t(i) * 32 + lane;
        if (b < nblk && (lane & 3) == 0) *reinterpret_cast<uint32_t*>(a.sf + sf_offset(m, b, kc4)) = 0u;
      }
      continue;
    }
    uint4 v[NB][2];
    if constexpr (PF) {
      const int j = int(k % kLnBufs);
      const uint32_t par = uint32_t(k / kLnBufs) & 1u;
      const bool stall = k == 0 && g_sixbit_stall_stage != 0;   // test switch: wait on the silent barrier
      if (!__all_sync(0xffffffffu, ln_bar_wait(stall ? rbar + 8u * kLnBufs : rbar + 8u * j, par))) {
        // Give up: flag it, let the copies still in flight land (bounded), stop.
        if (lane == 0 && a.err) atomicExch(a.err, int(kErrWaitTimeout));
        for (int d = 1; d < kLnBufs; ++d)
          if (m + d * nwarps < M) ln_bar_wait(rbar + 8u * uint32_t((k + d) % kLnBufs), uint32_t((k + d) / kLnBufs) & 1u);
        ln_bar_wait(rbar + 8u * j, par);
        break;
      }
      const uint8_t* srow = ln_rows + size_t(wib * kLnBufs + j) * rbytes;
#pragma unroll
      for (int i = 0; i < NB; ++i) {
        const int64_t b = int64_t(i) * 32 + lane;
        if (b < nblk) {
          v[i][0] = *reinterpret_cast<const uint4*>(srow + b * 32);
          v[i][1] = *reinterpret_cast<const uint4*>(srow + b * 32 + 16);
        } else {
          v[i][0] = v[i][1] = make_uint4(0, 0, 0, 0);
        }
      }
      __syncwarp();                            // every lane has read buffer j
      if (lane == 0 && m + kLnBufs * nwarps < M) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        ln_row_copy(rbuf + j * rbytes, a.x + (m + kLnBufs * nwarps) * a.ldx, rbytes, rbar + 8u * j);
      }
    } else {
      const uint16_t* row = a.x + m * a.ldx;
#pragma unroll
      for (int i = 0; i < NB; ++i) {
        const int64_t b = int64_t(i) * 32 + lane;
        if (b < nblk) {
          v[i][0] = ldg_nc_v4(row + b * 16);
          v[i][1] = ldg_nc_v4(row + b * 16 + 8);
        } else {
          v[i][0] = v[i][1] = make_uint4(0, 0, 0, 0);
        }
      }
    }
    uint64_t s2 = 0;                           // (sum of even elements, sum of odd elements)
#pragma unroll
    for (int i = 0; i < NB; ++i)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t* p = &v[i][h].x;
#pragma unroll
        for (int e = 0; e < 4; ++e) s2 = f2_add(s2, f2_from_bf16x2(p[e]));
      }
    float sl, sh;
    f2_unpack(s2, sl, sh);
    const float mean = __fdiv_rn(warp_sum(__fadd_rn(sl, sh)), float(H));
    const uint64_t mean2 = f2_pack(mean, mean);
    uint64_t q2 = 0;
#pragma unroll
    for (int i = 0; i < NB; ++i) {
      if (int64_t(i) * 32 + lane >= nblk) continue;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t* p = &v[i][h].x;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint64_t d = f2_sub(f2_from_bf16x2(p[e]), mean2);
          q2 = f2_fma(d, d, q2);
        }
      }
    }
    float ql, qh;
    f2_unpack(q2, ql, qh);
    const float var = __fdiv_rn(warp_sum(__fadd_rn(ql, qh)), float(H));
    const float rstd = __fdiv_rn(1.f, __fsqrt_rn(__fadd_rn(var, a.eps)));
    const uint64_t rstd2 = f2_pack(rstd, rstd);
    float rmax = 0.f;
    float bmax[NB];                            // |y| max of each of the lane's blocks
#pragma unroll
    for (int i = 0; i < NB; ++i) {
      const int64_t b = int64_t(i) * 32 + lane;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t* p = &v[i][h].x;
#pragma unroll
        for (int e = 0; e < 4; ++e) p[e] = f2_to_bf16x2(f2_mul(f2_sub(f2_from_bf16x2(p[e]), mean2), rstd2));
      }
      if (b < nblk) {
        bmax[i] = fmaxf(bf16x8_absmax(&v[i][0].x), bf16x8_absmax(&v[i][1].x));
        rmax = fmaxf(rmax, bmax[i]);
        if (a.y) {
          uint4* yp = reinterpret_cast<uint4*>(a.y + m * a.ldy + b * 16);
          yp[0] = v[i][0];
          yp[1] = v[i][1];
        }
      } else {
        bmax[i] = 0.f;
        v[i][0] = v[i][1] = make_uint4(0, 0, 0, 0);
      }
    }
    rmax = warp_max(rmax);
    if (a.row_amax_out && lane == 0) a.row_amax_out[m] = rmax;
    tmax = fmaxf(tmax, rmax);
    if (i8) {
      const bool nz = rmax > 0.f;
      const float inv = nz ? __fdiv_rn(127.f, rmax) : 0.f;
      if (lane == 0) a.row_scale[m] = nz ? __fdiv_rn(rmax, 127.f) : 0.f;
#pragma unroll
      for (int i = 0; i < NB; ++i) {
        const int64_t b = int64_t(i) * 32 + lane;
        if (b >= nblk) continue;
        uint32_t qb[8], p0[2], p1[2], p2[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          int8_encode8<false>(&v[i][h].x, inv, qb);
          int8_planes8(qb, lut, p0[h], p1[h], p2[h]);
        }
        uint8_t* base = a.planes + m * (H / 2) + b * 8;
        *reinterpret_cast<uint2*>(base) = make_uint2(p0[0], p0[1]);
        *reinterpret_cast<uint2*>(base + plane_stride) = make_uint2(p1[0], p1[1]);
        *reinterpret_cast<uint2*>(base + 2 * plane_stride) = make_uint2(p2[0], p2[1]);
      }
    }
    if (nv) {
#pragma unroll
      for (int i = 0; i < NB; ++i) {
        if (i * 32 >= nblk) break;               // warp-uniform
        const int64_t b = int64_t(i) * 32 + lane;
        const uint32_t sb = e4m3_encode(amax_t == 0.f ? 0.f : __fdiv_rn(__fmul_rn(bmax[i], 448.f), amax_t));
        const float r = rtab[sb];
        const uint32_t w0 = nvfp4_codes8(&v[i][0].x, r), w1 = nvfp4_codes8(&v[i][1].x, r);
        uint32_t word = sb | (__shfl_down_sync(0xffffffffu, sb, 1) << 8);
        word |= __shfl_down_sync(0xffffffffu, word, 2) << 16;
        if (b < nblk) {
          *reinterpret_cast<uint2*>(a.codes + m * (H / 2) + b * 8) = make_uint2(w0, w1);
          if ((lane & 3) == 0) *reinterpret_cast<uint32_t*>(a.sf + sf_offset(m, b, kc4)) = word;
        }
      }
    }
  }
  if (a.amax_out || a.hist) {                // one atomic (and one fence) per CTA
    if (lane == 0) red[threadIdx.x >> 5] = tmax;
    __syncthreads();
    if (threadIdx.x == 0) {
      float cmax = 0.f;
      for (int w = 0; w < LT / 32; ++w) cmax = fmaxf(cmax, red[w]);
      if (a.amax_out) atomic_max_nonneg(a.amax_out, cmax);
      if (a.hist) hist_arrive(a.hist, cmax);
    }
  }
}

}  // namespace

// ---------------------------------------------------------------------------
// Scratch of a pass: the CTA counter, then 4 float64 chain sums per CTA.
constexpr size_t kWsHeader = 256;
constexpr size_t kWsBytes = kWsHeader + size_t(kChains) * 4 * sizeof(double);   // 8448, whatever n
size_t tiles_ws_bytes(int64_t) { return kWsBytes; }

// Scratch-free Gamma pass.  Some callers cannot give this library scratch
// memory: their device memory is entirely planned by another allocator, or
// they run where allocating is not allowed (a plugin's enqueue step, a
// latency-critical loop that cannot afford cudaMalloc's implicit device
// synchronization).  For them the pass keeps its CTA counter and chain sums
// in this fixed device array instead of caller scratch.  The array lives on
// every device that loads the library, until the process exits; its size
// does not depend on n, so the size limit is that of the regular pass.
constexpr int64_t kNoAllocMaxElems = int64_t(1) << 40;
static __device__ __align__(256) unsigned char g_gamma_scratch[kWsBytes];

namespace {
constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_scratch[kNoAllocMaxDevices] = {};

// Device address of the scratch array for the current device.  Host code may
// not use the array's name as a device pointer; the address is looked up
// once per device, with that device current, on the first call there.
void* noalloc_scratch_for_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_scratch[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_gamma_scratch) != cudaSuccess) return nullptr;
    g_noalloc_scratch[dev] = p;
  }
  return g_noalloc_scratch[dev];
}
}  // namespace

int64_t block_gamma_noalloc_max_elems() { return kNoAllocMaxElems; }

int launch_block_gamma_noalloc(const void* xin, const void* xout, int64_t n, void* delta, float* gamma_out,
                               float* r2_out, int32_t* tdc_state, const uint8_t* computed, int* err,
                               cudaStream_t s) {
  if (n > kNoAllocMaxElems) return kEShape;
  void* scratch = noalloc_scratch_for_current_device();
  if (!scratch) return kELaunch;
  // The array keeps the previous call's contents: the CTA counter must start at 0.
  if (cudaMemsetAsync(scratch, 0, 256, s) != cudaSuccess) return kELaunch;
  return launch_block_gamma(xin, xout, n, delta, gamma_out, r2_out, tdc_state, computed, scratch, err, s);
}

// One CTA per chain of the reduction tree: the grid is fixed by n alone.
int gamma_grid(int64_t n) {
  const int64_t tiles = cdiv(n, kTile);
  return int(tiles < kChains ? tiles : kChains);
}

size_t gamma_ws_bytes(int64_t n) { return tiles_ws_bytes(n); }

int launch_block_gamma(const void* xin, const void* xout, int64_t n, void* delta, float* gamma_out, float* r2_out,
                       int32_t* tdc_state, const uint8_t* computed, void* ws, int* err, cudaStream_t s) {
  GammaWs* w = static_cast<GammaWs*>(ws);
  double* chains = reinterpret_cast<double*>(static_cast<char*>(ws) + kWsHeader);
  // two tile stages: more than the default 48 KB of dynamic shared memory
  if (cudaFuncSetAttribute(gamma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kGammaSmem)) != cudaSuccess)
    return kELaunch;
  gamma_kernel<<<unsigned(gamma_grid(n)), kThreads, kGammaSmem, s>>>(
      static_cast<const uint16_t*>(xin), static_cast<const uint16_t*>(xout), n, static_cast<uint16_t*>(delta),
      gamma_out, r2_out, tdc_state, computed, w, chains, err);
  return cudaGetLastError() == cudaSuccess ? kOk : kELaunch;
}

int launch_block_gamma_mx(const void* xin, const void* xout, int64_t n, void* cache, float* gamma_out, float* r2_out,
                          int32_t* tdc_state, const uint8_t* computed, void* ws, int* err, cudaStream_t s) {
  GammaWs* w = static_cast<GammaWs*>(ws);
  double* chains = reinterpret_cast<double*>(static_cast<char*>(ws) + kWsHeader);
  if (cudaFuncSetAttribute(gamma_mx_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kGammaMxSmem)) !=
      cudaSuccess)
    return kELaunch;
  gamma_mx_kernel<<<unsigned(gamma_grid(n)), kThreads, kGammaMxSmem, s>>>(
      static_cast<const uint16_t*>(xin), static_cast<const uint16_t*>(xout), n, static_cast<uint8_t*>(cache),
      gamma_out, r2_out, tdc_state, computed, w, chains, err);
  return cudaGetLastError() == cudaSuccess ? kOk : kELaunch;
}

int launch_pair_stats(const void* a, int a_f32, const void* b, int b_f32, int64_t n, double* out, void* ws,
                      cudaStream_t s) {
  GammaWs* w = static_cast<GammaWs*>(ws);
  double* chains = reinterpret_cast<double*>(static_cast<char*>(ws) + kWsHeader);
  const unsigned grid = unsigned(gamma_grid(n));
  if (!a_f32 && !b_f32)
    pair_stats_kernel<uint16_t, uint16_t><<<grid, kThreads, 0, s>>>(static_cast<const uint16_t*>(a),
                                                                    static_cast<const uint16_t*>(b), n, out, w, chains);
  else if (!a_f32)
    pair_stats_kernel<uint16_t, float><<<grid, kThreads, 0, s>>>(static_cast<const uint16_t*>(a),
                                                                 static_cast<const float*>(b), n, out, w, chains);
  else if (!b_f32)
    pair_stats_kernel<float, uint16_t><<<grid, kThreads, 0, s>>>(static_cast<const float*>(a),
                                                                 static_cast<const uint16_t*>(b), n, out, w, chains);
  else
    pair_stats_kernel<float, float><<<grid, kThreads, 0, s>>>(static_cast<const float*>(a), static_cast<const float*>(b),
                                                              n, out, w, chains);
  return cudaGetLastError() == cudaSuccess ? kOk : kELaunch;
}

int launch_dmpq(const float* gamma, const float* alpha, const float* beta, const int32_t* layer_block,
                int32_t n_layers, float tau, const int32_t* step, uint8_t* use_nvfp4, uint8_t* gates, cudaStream_t s) {
  const int threads = 128;
  dmpq_kernel<<<unsigned(cdiv(n_layers, threads)), threads, 0, s>>>(gamma, alpha, beta, layer_block, n_layers, tau,
                                                                     step, use_nvfp4, gates);
  return cudaGetLastError() == cudaSuccess ? kOk : kELaunch;
}

int launch_tdc(const void* xin, const void* delta, int64_t n, const float* r2, float tau2, int32_t max_skip,
               int32_t refresh_every, const int32_t* step, const int32_t* tdc_state, uint8_t* compute_out, void* out,
               uint8_t* gates, int32_t n_gates, int num_sms, cudaStream_t s) {
  int64_t want = cdiv(n / 8 + 1, kThreads * 4);
  int64_t cap = int64_t(num_sms) * 8;
  const unsigned grid = unsigned(want < cap ? (want < 1 ? 1 : want) : cap);
  tdc_kernel<<<grid, kThreads, 0, s>>>(static_cast<const uint16_t*>(xin), static_cast<const uint16_t*>(delta), n, r2,
                                       tau2, max_skip, refresh_every, step, tdc_state, compute_out,
                                       static_cast<uint16_t*>(out), gates, n_gates);
  return cudaGetLastError() == cudaSuccess ? kOk : kELaunch;
}

int launch_tdc_mx(const void* xin, const void* cache, int64_t n, const float* r2, float tau2, int32_t max_skip,
                  int32_t refresh_every, const int32_t* step, const int32_t* tdc_state, uint8_t* compute_out,
                  void* out, uint8_t* gates, int32_t n_gates, int num_sms, cudaStream_t s) {
  int64_t want = cdiv(n / 8 + 1, kThreads * 4);
  int64_t cap = int64_t(num_sms) * 8;
  const unsigned grid = unsigned(want < cap ? (want < 1 ? 1 : want) : cap);
  tdc_mx_kernel<<<grid, kThreads, 0, s>>>(static_cast<const uint16_t*>(xin), static_cast<const uint8_t*>(cache), n, r2,
                                          tau2, max_skip, refresh_every, step, tdc_state, compute_out,
                                          static_cast<uint16_t*>(out), gates, n_gates);
  return cudaGetLastError() == cudaSuccess ? kOk : kELaunch;
}

// Persistent grid: as many CTAs as are resident at once, each walking rows,
// so the per-CTA tail (amax atomic, fence, history ticket) is paid once.
// With the row prefetch (PF), kLnBufs row buffers of 2 H bytes per warp of
// dynamic shared memory (at most 64 KB).  CTAs resident per SM, by H, found
// once under a lock.
template <int NB, bool PF>
void launch_lnq(const LnQuantCall& c, int64_t rows, int num_sms, cudaStream_t s) {
  static std::mutex mu;
  static int per_sm[kLnQuantMaxH / 16 + 1] = {};
  const size_t smem = PF ? size_t(kLnThreads<NB> / 32) * kLnBufs * size_t(c.H) * 2 : 0;
  int occ;
  {
    std::lock_guard<std::mutex> lock(mu);
    int& e = per_sm[c.H / 16];
    if (e == 0) {
      if (PF)
        cudaFuncSetAttribute(ln_quant_kernel<NB, PF>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(size_t(kLnThreads<NB> / 32) * kLnBufs * kLnQuantMaxH * 2));
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&e, ln_quant_kernel<NB, PF>, kLnThreads<NB>, smem) !=
              cudaSuccess ||
          e < 1)
        e = 1;
    }
    occ = e;
  }
  const int64_t want = cdiv(rows, kLnThreads<NB> / 32), cap = int64_t(num_sms) * occ;
  ln_quant_kernel<NB, PF><<<unsigned(want < cap ? (want < 1 ? 1 : want) : cap), kLnThreads<NB>, smem, s>>>(c);
}

// The prefetch is used where it measured faster (graph-timed on GB300 over
// rotated inputs larger than L2): with 8-warp CTAs (rows of up to 2048) when
// the bf16 output is written (1920: 22.5 -> 21.1 us, with NVFP4 as well
// 36.2 -> 32.6 us; quantized outputs alone 0.7 us slower with it), with
// 4-warp CTAs (rows of 2049-4096) when a quantized output is written (3072:
// NVFP4 79.7 -> 74.2 us, INT8 82.7 -> 78.7 us; bf16 alone 69.7 -> 80.2 us).
template <int NB>
void launch_lnq_pick(const LnQuantCall& c, int64_t rows, int num_sms, cudaStream_t s) {
  const bool quantized = c.codes != nullptr || c.planes != nullptr;
  const bool pf = kLnThreads<NB> == 256 ? c.y != nullptr : quantized;
  if (pf) launch_lnq<NB, true>(c, rows, num_sms, s);
  else launch_lnq<NB, false>(c, rows, num_sms, s);
}

int launch_ln_quant(const LnQuantCall& c, int num_sms, cudaStream_t s) {
  if (c.H % 16 != 0 || c.H > kLnQuantMaxH) return kEShape;
  if (c.amax_out && cudaMemsetAsync(c.amax_out, 0, sizeof(float), s) != cudaSuccess) return kELaunch;
  const int64_t per_lane = cdiv(c.H / 16, 32);         // 16-element blocks a lane holds
  const int64_t rows = c.codes ? cdiv(c.M, 128) * 128 : c.M;
  if (per_lane <= 1) launch_lnq_pick<1>(c, rows, num_sms, s);
  else if (per_lane <= 2) launch_lnq_pick<2>(c, rows, num_sms, s);
  else if (per_lane <= 4) launch_lnq_pick<4>(c, rows, num_sms, s);
  else if (per_lane <= 6) launch_lnq_pick<6>(c, rows, num_sms, s);
  else launch_lnq_pick<8>(c, rows, num_sms, s);
  return cudaGetLastError() == cudaSuccess ? kOk : kELaunch;
}

int launch_layernorm(const void* x, int64_t M, int64_t H, int64_t ldx, float eps, void* y, int64_t ldy,
                     float* amax_out, float* row_amax_out, const uint8_t* pred, int* err, int num_sms,
                     cudaStream_t s) {
  if (H % 16 == 0 && H <= kLnQuantMaxH) {      // the register-resident kernel, without quantized outputs
    LnQuantCall c = {};
    c.x = static_cast<const uint16_t*>(x); c.M = M; c.H = H; c.ldx = ldx; c.eps = eps;
    c.y = static_cast<uint16_t*>(y); c.ldy = ldy; c.amax_out = amax_out; c.row_amax_out = row_amax_out;
    c.pred = pred; c.err = err;
    return launch_ln_quant(c, num_sms, s);
  }
  if (amax_out && cudaMemsetAsync(amax_out, 0, sizeof(float), s) != cudaSuccess) return kELaunch;
  int64_t want = cdiv(M, kThreads / 32);
  int64_t cap = int64_t(num_sms) * 8;
  const unsigned grid = unsigned(want < cap ? (want < 1 ? 1 : want) : cap);
  layernorm_kernel<<<grid, kThreads, 0, s>>>(static_cast<const uint16_t*>(x), M, H, ldx, eps,
                                             static_cast<uint16_t*>(y), ldy, amax_out, row_amax_out, pred);
  return cudaGetLastError() == cudaSuccess ? kOk : kELaunch;
}

}  // namespace sixbit
