// Block-scaled FP4 GEMM on the sm_103a tensor cores (tcgen05), with the
// dequant / bias / GELU / residual epilogue fused.  Serves both linear
// layer types of 6Bit-Diffusion ("Abstract", mlsanity.com page; uniform
// W4A4 / W4A8 of Table 3, thelatestinai.com page):
//
//  mode 0, W4A4:  y = g_a g_w sum_k (E2M1 S)_a (E2M1 S)_w
//  mode 1, W4A8:  y = s_a[m] g_w sum_k q (E2M1 S)_w, with the INT8 code q
//                 given as three E2M1 digit planes, q = 64 a + 8 b + c.
//                 Each K step issues one MMA per plane with a constant
//                 E4M3 block scale (64, 8, 1) for A, so the tensor cores
//                 form q * w exactly and accumulate in fp32.  (sm_103a has
//                 no tcgen05 int8 kind, and its warp-level int8 MMA runs at
//                 ~150 TOP/s, far below the FP4 pipe.)
//
// Structure: persistent, warp-specialized CTA of 16 warps over 128 x 256
// output tiles, K in steps of KB bytes of codes per row (2*KB elements):
//   warps 0, 2  TMA producers (one lane each): the A code tile (or its three
//               digit planes) and the W code tile, KB-byte swizzle, into a
//               STAGES-deep shared-memory ring;
//   warp 3      TMA producer of the E4M3 scale atoms: with the code stages
//               (W4A8, CTA pairs) or, for W4A4 on one CTA, into a ring of
//               their own that runs ahead of the code stages;
//   warp 1      TMEM owner and MMA issuer: tcgen05.mma kind::mxf4nvf4
//               scale_vec::4X (128 x 256 x 64 per instruction, 256 x 256 on a
//               CTA pair) into the TMEM accumulator, tcgen05.commit to free
//               stages and publish tiles; the whole warp runs the loop and
//               lane 0 issues;
//   warps 4..7  scale warps, one per TMEM lane quarter: move each k-step's
//               scale atoms from shared memory into TMEM scale columns with
//               tcgen05.st, in the layout a replicating tcgen05.cp
//               (.32x128b.warpx4) produces;
//   warps 8..15 epilogue: two warps per TMEM lane quarter, 128 columns each.
//               They pull the whole accumulator into registers, release TMEM
//               at once (the next tile's MMAs start), then scale, add bias,
//               GELU (two special-function ops an element), add the residual
//               (a TMA-loaded tile) and write bf16 through 128-byte-swizzled
//               shared memory with TMA stores.  The QO instantiation can
//               instead encode the result as NVFP4 for the next layer
//               (delayed scaling) and report its exact amax.
// Only MMAs go through the tensor pipe's issue queue: on GB300 one thread
// issues about one tcgen05.mma/tcgen05.cp per 25 ns, so moving the three
// scale copies of each 128 x 256 x 64 MMA (66 ns of tensor work) to
// tcgen05.st from other warps takes the issue queue off the critical path.
// Registers: the CTA launches with 128 per thread; warpgroups 0-1 drop to
// 72 and the epilogue warpgroups rise to 184 (setmaxnreg), which adds up to
// exactly the launch allocation.  The host refuses to launch a build whose
// launch register count is not 128 (the rise would never be granted).
// Every mbarrier wait is bounded; on expiry the CTA records an error in the
// device error word, drains its own copies and MMAs, frees TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"

namespace sixbit {

// Test switch (set through sixbit_debug_stall_gemm): nonzero makes the MMA
// issuer of every GEMM launched afterwards wait on a barrier that is never
// signalled, so its bounded wait expires and the device-error path runs.
__device__ int g_sixbit_stall_mma = 0;

int set_gemm_stall(int on) {
  return cudaMemcpyToSymbol(g_sixbit_stall_mma, &on, sizeof(on)) == cudaSuccess ? kOk : kELaunch;
}

namespace {

constexpr int BM = 128;
constexpr int kThreads = 512;            // 4 warpgroups: control, scales, 2 x epilogue
constexpr int kLaunchRegs = 128;         // 65536 / kThreads
constexpr int kLowRegs = 72, kHighRegs = 184;
static_assert(2 * 128 * kLowRegs + 2 * 128 * kHighRegs == kThreads * kLaunchRegs, "register split");
constexpr uint32_t kSpinCap = 1u << 22;  // polls of a bounded mbarrier wait
constexpr uint32_t kTmemCols = 512;

#ifndef GEMM_PAIR
#define GEMM_PAIR true   // W4A8: CTA pairs with cta_group::2 MMAs (256 x 256 tiles; 5 stages fit instead of 4)
#endif
#ifndef W4A4_PAIR
#define W4A4_PAIR true   // W4A4: CTA pairs (each CTA streams half of W: ~145 instead of ~206 GB/s per SM)
#endif
#ifndef W4A8_NC
#define W4A8_NC 1
#define W4A8_STAGES (GEMM_PAIR ? 5 : 4)
#endif

template <int BN, int MODE, int STAGES, int KB, int NC, bool PAIR>
struct Cfg {
  static_assert(BN == 256, "epilogue assumes 256-column tiles");
  // PAIR: a cluster of two CTAs computes a 256 x BN tile with cta_group::2
  // MMAs; each CTA holds its own 128 rows of A and BN/2 rows of W.
  static constexpr int kTileM = PAIR ? 2 * BM : BM;
  static constexpr int kBRows = PAIR ? BN / 2 : BN;
  static_assert(KB == 64 || KB == 128, "K chunk of 64 or 128 bytes per row");
  static constexpr int kMmaK = KB / 32;                    // MMAs (K = 64 elements) per chunk
  static constexpr int kAtoms = kMmaK * NC;                // 512-byte scale atoms per 128 rows per stage
  static constexpr int kPlanes = MODE == 0 ? 1 : 3;
  static constexpr int kRT = BN / 128;                     // 128-row scale tiles of W per N tile
  static constexpr int kChunkA = BM * KB;                  // one chunk of one A plane
  static constexpr int kChunkB = kBRows * KB;
  static constexpr int kA = kChunkA * NC;                  // one A plane, all chunks of a stage
  static constexpr int kB = kChunkB * NC;
  static constexpr int kSFA = MODE == 0 ? 512 * kAtoms : 0;
  static constexpr int kSFB = 512 * kAtoms * kRT;
  static constexpr int offB = kPlanes * kA;
  static constexpr int offSFA = offB + kB;
  static constexpr int offSFB = offSFA + kSFA;
  // W4A4 on a single CTA keeps the scale atoms in a ring of their own
  // (kSfSlots slots of shared memory and TMEM, with their own barriers), so
  // the scale path can run ahead of the code tiles instead of landing with
  // them; the stages then hold the codes only.
  static constexpr bool kSfRing = MODE == 0 && !PAIR;
  static constexpr int kSfSlots = kSfRing ? 4 : STAGES;    // TMEM scale slots
  static constexpr int kStage = kSfRing ? offSFA : offSFB + kSFB;
  static constexpr int kSfSlotBytes = kSFA + kSFB;         // one ring slot: SFA atoms, then SFB atoms
  static constexpr int kRing = kSfRing ? kSfSlots * kSfSlotBytes : 0;
  static_assert(kStage % 1024 == 0 && kSfSlotBytes % 1024 == 0, "stages stay 1024-byte aligned");
  static constexpr uint32_t kTxA = kPlanes * kA;           // bytes landed per stage, by producer
  static constexpr uint32_t kTxB = kB;
  static constexpr uint32_t kTxS = kSFA + kSFB;
  // TMEM columns: accumulator [0, BN), then per-stage scale columns, then
  // the three constant digit-scale atoms (mode 1).  Each CTA of a pair holds
  // the scales of its own A rows and of all BN rows of W.
  static constexpr int kSfaCols = MODE == 0 ? 4 * kAtoms : 0;
  static constexpr int kSfStride = kSfaCols + 4 * kAtoms * kRT;
  static constexpr int kSfBase = BN;
  static constexpr int kConstCol = kSfBase + kSfSlots * kSfStride;
  static_assert(kConstCol + 12 <= int(kTmemCols), "TMEM budget");
  static constexpr int kStaging = 8 * 4096;               // per epilogue warp: 32 rows x 128 bytes of output
  static constexpr int kExtra = 1024;                      // barriers, TMEM address, abort flag
  static constexpr size_t kSmem = size_t(STAGES) * kStage + kRing + kStaging + kExtra + 1024;
  static_assert(kSmem <= 232448, "shared memory budget");
};

// ------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return uint32_t(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_try_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: false when the cap expired or another role aborted.  CL:
// the barrier also receives arrivals from the other CTA of a pair.
template <bool CL = false>
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  for (uint32_t i = 0; i < kSpinCap; ++i) {
    if (CL ? mbar_try_cluster(bar, parity) : mbar_try(bar, parity)) return true;
    if ((i & 255u) == 255u && abort_flag && *abort_flag) return false;
  }
  return false;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tm, int c0, int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* tm, int c0, int c1, int c2, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* tm, int c0, int c1, int c2, int c3,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* tm, uint32_t src, int c0, int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(tm)),
               "r"(c0), "r"(c1), "r"(src)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* tm) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// MMA and commit wrappers.  The MMA-issuing warp runs its loop with all 32
// lanes; one lane issues each instruction.  LANE0 puts that choice inside
// the asm as a predicate on %laneid (the warp never diverges); without it
// the caller branches on lane 0 around the call.  The two forms compile to
// different issue loops: the predicated one ran the W4A8 FFN-up GEMM 9%
// faster, the branch the W4A4 QKV and FFN-down GEMMs 3-4% faster (2B
// shapes, same results bit for bit).
#define SIXBIT_LANE0_PRED " .reg .pred e_;\n .reg .u32 l_;\n mov.u32 l_, %%laneid;\n setp.eq.u32 e_, l_, 0;\n"
// Commit of this thread's MMAs to a barrier of this CTA only.
template <bool PAIR, bool LANE0>
__device__ __forceinline__ void tc_commit_local(uint32_t bar) {
  if constexpr (PAIR && LANE0)
    asm volatile("{\n" SIXBIT_LANE0_PRED
                 " @e_ tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}" ::"r"(bar)
                 : "memory");
  else if constexpr (PAIR)
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
  else if constexpr (LANE0)
    asm volatile("{\n" SIXBIT_LANE0_PRED
                 " @e_ tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}" ::"r"(bar)
                 : "memory");
  else
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
template <bool PAIR, bool LANE0>
__device__ __forceinline__ void tc_mma_fp4(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                           uint32_t sfb, uint32_t accum) {
  if constexpr (PAIR && LANE0)
    asm volatile(
        "{\n .reg .pred p;\n" SIXBIT_LANE0_PRED " setp.ne.b32 p, %4, 0;\n"
        " @e_ tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n}" ::"r"(
            d),
        "l"(a), "l"(b), "r"(idesc), "r"(accum), "r"(sfa), "r"(sfb)
        : "memory");
  else if constexpr (PAIR)
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(accum), "r"(sfa), "r"(sfb)
        : "memory");
  else if constexpr (LANE0)
    asm volatile(
        "{\n .reg .pred p;\n" SIXBIT_LANE0_PRED " setp.ne.b32 p, %4, 0;\n"
        " @e_ tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n}" ::"r"(
            d),
        "l"(a), "l"(b), "r"(idesc), "r"(accum), "r"(sfa), "r"(sfb)
        : "memory");
  else
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(accum), "r"(sfa), "r"(sfb)
        : "memory");
}
// Commit of this thread's MMAs to a barrier; in a pair, to the barrier at the
// same offset in both CTAs.
template <bool PAIR, bool LANE0>
__device__ __forceinline__ void tc_commit_all(uint32_t bar) {
  if constexpr (PAIR && LANE0)
    asm volatile("{\n" SIXBIT_LANE0_PRED
                 " @e_ tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n}" ::"r"(
                     bar),
                 "h"(uint16_t(3))
                 : "memory");
  else if constexpr (PAIR)
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                     bar),
                 "h"(uint16_t(3))
                 : "memory");
  else if constexpr (LANE0)
    asm volatile("{\n" SIXBIT_LANE0_PRED
                 " @e_ tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}" ::"r"(bar)
                 : "memory");
  else
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
// Address of the same shared-memory object in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
// Arrival on a barrier of the other CTA of a pair.  The default semantics
// (release at CTA scope) keep the issuing thread's cost near 60 ns; the
// cluster-scope release form stalled the issuing thread for 280-440 ns.
// Callers order their tcgen05 work first (tcgen05.wait + fence).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ void st_cluster_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// Scale atoms into TMEM, laid out as tcgen05.cp .32x128b.warpx4 would: lane
// l of every lane quarter holds row l of each 512-byte atom (16 bytes, the
// scales of rows l, 32+l, 64+l, 96+l) in 4 consecutive columns.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, uint4 a, uint4 b, uint4 c, uint4 d) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w), "r"(c.x), "r"(c.y), "r"(c.z),
      "r"(c.w), "r"(d.x), "r"(d.y), "r"(d.z), "r"(d.w)
      : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, uint4 a, uint4 b) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(a.x),
               "r"(a.y), "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
               : "memory");
}
__device__ __forceinline__ void tmem_st4(uint32_t taddr, uint32_t w) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%1,%1,%1};" ::"r"(taddr), "r"(w) : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
template <int R>
__device__ __forceinline__ void regs_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(R)); }
template <int R>
__device__ __forceinline__ void regs_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(R)); }

// Shared-memory matrix descriptor, K-major, KB-byte swizzle: rows of KB
// bytes, 8-row groups 8*KB bytes apart (layout code 2 = 128B, 4 = 64B).
template <int KB>
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t saddr) {
  constexpr uint64_t layout = KB == 128 ? 2 : 4;
  return uint64_t((saddr & 0x3FFFFu) >> 4) | (uint64_t(1) << 16) | (uint64_t((8 * KB) >> 4) << 32) |
         (uint64_t(1) << 46) | (layout << 61);
}
// Instruction descriptor, kind::mxf4nvf4: A, B = E2M1, K-major, dense,
// UE4M3 scales, M = m (128, or 256 for a CTA pair), N = n.
__host__ __device__ constexpr uint32_t idesc_fp4(int m, int n) {
  return (1u << 7) | (1u << 10) | (uint32_t(n >> 3) << 17) | (uint32_t(m >> 4) << 24);
}

// tanh-form GELU, 0.5 x (1 + tanh(u)) with u = sqrt(2/pi) (x + 0.044715 x^3),
// written as x / (1 + 2^t), t = -2 u log2(e) = x (c1 + c2 x^2) (the same
// function), for two elements at a time: t on the packed f32x2 pipe, then
// the hardware approximations 2^t (ex2.approx) and 1 / (1 + 2^t)
// (rcp.approx), each accurate to about an fp32 unit in the last place.
// Both flush subnormals (.ftz): a subnormal 2^t adds nothing to 1 in fp32,
// and t is subnormal only where 2^t rounds to 1 anyway, so no result
// changes (the non-flushing exponential cost 6 us of the 2B FFN-up GEMM).
// Unlike 1 + tanh(u) this form has no cancellation for negative x, so the
// result keeps fp32 relative accuracy everywhere.  For t >= 128 (x below
// about -10) 2^t is +inf and the result is -0, the bf16 rounding of the
// exact value.  Against an exponent-flip seed with three Newton steps on
// the FMA pipe: identical bf16 outputs except one-ulp differences at
// rounding ties (3e-5 of the 2B FFN-up outputs) and -0 where that form's
// clamp of t at 126 left ~-1e-37; the W4A4 FFN-up ran 150.1 -> 127.6 us.
__device__ __forceinline__ void gelu_tanh2(float& x0, float& x1) {
  const uint64_t x = f2_pack(x0, x1);
  // c1 = -2 sqrt(2/pi) log2(e), c2 = 0.044715 c1
  const uint64_t t = f2_mul(x, f2_fma(f2_mul(x, x), f2_pack(-0.10294324f, -0.10294324f),
                                      f2_pack(-2.302208198f, -2.302208198f)));
  float t0, t1, e0, e1, d0, d1, r0, r1;
  f2_unpack(t, t0, t1);
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e0) : "f"(t0));
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e1) : "f"(t1));
  f2_unpack(f2_add(f2_pack(e0, e1), f2_pack(1.f, 1.f)), d0, d1);
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r0) : "f"(d0));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r1) : "f"(d1));
  f2_unpack(f2_mul(x, f2_pack(r0, r1)), x0, x1);
}

struct Params {
  int M, N, K, KT, MT, NT;
  const float* g_a;
  const float* row_scale;
  const float* g_w;
  const uint16_t* bias;
  const uint16_t* residual;
  int64_t ldr;
  void* y;
  int64_t ldy;
  int out_bf16, gelu;
  int chunked;               // 1: K chunk maps (one op per operand per stage); 0: 2-D maps, one chunk per stage
  const uint8_t* pred;
  int* err;
  // quantizing epilogue (q_hist != null), see GemmCall
  uint8_t* q_codes;
  uint8_t* q_sf;
  float* q_g;
  uint32_t* q_hist;
  float q_headroom;
  const uint8_t* q_pred;
};

// Which output tile each CTA pair (or CTA) computes.  The U pairs walk the
// tiles round-robin: pair u takes indices u, u + U, u + 2U, ..., index
// i = jU + u being its tile of round j, and the order of the indices is row
// order (row tile mt, then column tile nt), so the tiles of one round share
// their A rows and W columns in L2.
// With a half-width last column (`half`: W4A8 whose N % 256 == 128, run as
// N = 128 MMAs at half the MMA time), the round-robin alone gives the half
// tiles to a few pairs and leaves the last round's tiles to the first
// ntiles % U pairs at full cost.  Where the counts allow it (`bal`), each
// round still covers the same tiles, but within the round they go to the
// pairs so that the e = ntiles % U pairs with one tile more than the others
// take two half tiles, the next D - e pairs one (D = MT - e), and the rest
// none: every pair then has at most R = ntiles / U tiles' worth of MMAs
// instead of R + 1/2.  Half tile k (row k) goes to pair k, or to k - D for
// k >= D; the full tiles of a round go, in row order, to the pairs without
// a half tile in it.  D * NT >= U keeps a pair's two half tiles in
// different rounds.  Otherwise the half tiles of the last rows fill the
// last, partial round (`late`), and every other tile keeps its row-order
// place.
struct TileOrder {
  int MT, NT, U, ntiles, e, D, late;
  bool half, bal;
};

__host__ __device__ inline TileOrder make_tile_order(int MT, int NT, int U, bool half_col) {
  TileOrder o;
  o.MT = MT;
  o.NT = NT;
  o.U = U;
  o.ntiles = MT * NT;
  o.e = o.ntiles % U;
  o.D = MT - o.e;
  o.half = half_col && NT > 1;
  o.bal = o.half && MT >= 2 * o.e && o.D <= U && int64_t(o.D) * NT >= U;
  o.late = o.half && !o.bal && o.e <= MT ? o.e : 0;
  return o;
}

__host__ __device__ inline void tile_of(const TileOrder& o, int i, int& mt, int& nt) {
  if (o.bal) {
    const int j = i / o.U, u = i - j * o.U;
    const int lo = j * o.U, hi = lo + o.U < o.ntiles ? lo + o.U : o.ntiles;
    const int k_lo = lo / o.NT, k_hi = hi / o.NT;            // half tiles k with k NT + NT - 1 in [lo, hi)
    const int k1 = u < o.D ? u : -1, k2 = u < o.e ? u + o.D : -1;
    if (k1 >= k_lo && k1 < k_hi) { mt = k1; nt = o.NT - 1; return; }
    if (k2 >= k_lo && k2 < k_hi) { mt = k2; nt = o.NT - 1; return; }
    // pairs below u that take a half tile of this round
    const int a0 = k_lo, a1 = k_hi < (u < o.D ? u : o.D) ? k_hi : (u < o.D ? u : o.D);
    const int b0 = k_lo > o.D ? k_lo : o.D, b1 = k_hi < o.D + (u < o.e ? u : o.e) ? k_hi : o.D + (u < o.e ? u : o.e);
    const int below = (a1 > a0 ? a1 - a0 : 0) + (b1 > b0 ? b1 - b0 : 0);
    const int f = (lo - k_lo) + (u - below);                // full tile index, row order
    mt = f / (o.NT - 1);
    nt = f - mt * (o.NT - 1);
    return;
  }
  mt = i / o.NT;
  nt = i - mt * o.NT;
  if (o.late > 0) {
    const int first_late = o.ntiles - o.late, row0 = o.MT - o.late;
    if (i >= first_late) {
      mt = row0 + (i - first_late);
      nt = o.NT - 1;
    } else if (i >= row0 * o.NT) {             // the last rows without their half tiles
      const int j = i - row0 * o.NT;
      mt = row0 + j / (o.NT - 1);
      nt = j - (j / (o.NT - 1)) * (o.NT - 1);
    }
  }
}

template <int BN, int MODE, int STAGES, int KB, int NC, bool PAIR, bool QO>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_fp4_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmSFA, const __grid_constant__ CUtensorMap tmSFB,
                    const __grid_constant__ CUtensorMap tmY, const __grid_constant__ CUtensorMap tmR,
                    const Params p) {
  using C = Cfg<BN, MODE, STAGES, KB, NC, PAIR>;
  if (p.pred && *p.pred == 0) return;          // both CTAs of a pair read the same gate
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem + size_t(STAGES) * C::kStage;             // scale-atom ring (W4A4, one CTA)
  uint8_t* staging = ring + C::kRing;                            // 8 x 4 KB, 1024-byte aligned
  uint8_t* extra = staging + C::kStaging;
  // barriers: full[S] empty[S] sfready[R] tfull tempty drain resid[8] sffull[R] sfempty[R], R = kSfSlots
  constexpr int R = C::kSfSlots;
  uint64_t* bars = reinterpret_cast<uint64_t*>(extra);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 3 * R + 12);
  static_assert((2 * STAGES + 3 * R + 12) * 8 + 8 <= 512, "barriers, TMEM address and abort flag below the r table");
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? cluster_rank() : 0u;              // 0: the CTA that issues the MMAs
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * uint32_t(s); };
  auto empty_bar = [&](int s) { return bar0 + 8u * uint32_t(STAGES + s); };
  auto sfready_bar = [&](int s) { return bar0 + 8u * uint32_t(2 * STAGES + s); };
  const uint32_t tfull_bar = bar0 + 8u * uint32_t(2 * STAGES + R);
  const uint32_t tempty_bar = bar0 + 8u * uint32_t(2 * STAGES + R + 1);
  const uint32_t drain_bar = bar0 + 8u * uint32_t(2 * STAGES + R + 2);
  auto resid_bar = [&](int w) { return bar0 + 8u * uint32_t(2 * STAGES + R + 3 + w); };
  auto sffull_bar = [&](int s) { return bar0 + 8u * uint32_t(2 * STAGES + R + 11 + s); };   // ring only
  auto sfempty_bar = [&](int s) { return bar0 + 8u * uint32_t(2 * STAGES + 2 * R + 11 + s); };
  const uint32_t never_bar = bar0 + 8u * uint32_t(2 * STAGES + 3 * R + 11);   // initialised, never arrived on
  // Arrival on a barrier of the issuing CTA (rank 0): local, or across the pair.
  auto arrive_leader = [&](uint32_t bar) {
    if constexpr (PAIR) {
      if (rank == 0) mbar_arrive(bar);
      else mbar_arrive_remote(map_rank(bar, 0));
    } else {
      mbar_arrive(bar);
    }
  };
  constexpr int kCtas = PAIR ? 2 : 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), C::kSfRing ? 2 : 3);   // the A and W producers (and the scale producer)
      mbar_init(empty_bar(s), 1);
    }
    for (int s = 0; s < R; ++s) {
      mbar_init(sfready_bar(s), 4 * kCtas);    // one arrival per scale warp of the pair
      if (C::kSfRing) {
        mbar_init(sffull_bar(s), 1);           // the scale producer
        mbar_init(sfempty_bar(s), 1);          // the MMA commit of the k-step that read the slot
      }
    }
    mbar_init(tfull_bar, 1);
    mbar_init(tempty_bar, 8 * kCtas);          // one arrival per epilogue warp of the pair
    mbar_init(drain_bar, 1);
    for (int w = 0; w < 8; ++w) mbar_init(resid_bar(w), 1);
    mbar_init(never_bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    if (MODE == 0) prefetch_tmap(&tmSFA);
    prefetch_tmap(&tmSFB);
    if (p.out_bf16) prefetch_tmap(&tmY);
    if (p.out_bf16 && p.residual) prefetch_tmap(&tmR);
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      // one allocation for the pair: warp 1 of both CTAs takes part
      asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                   "r"(kTmemCols));
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
    } else {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                   "r"(kTmemCols));
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync();          // both CTAs' barriers and TMEM exist before any cross traffic
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int ntiles = p.MT * p.NT;
  // W4A8 with a half-width last column (N % 256 == 128, e.g. N = 1920): a
  // tile of that column runs as N = 128 MMAs, half the MMA work of a full
  // tile, and its W rows split 64 / 64 between the pair; make_tile_order
  // spreads those tiles over the pairs.
  const bool half_col = MODE == 1 && PAIR && p.N % BN == BN / 2;
  const TileOrder order = make_tile_order(p.MT, p.NT, int(gridDim.x) / kCtas, half_col);
  auto tile_at = [&](int tile, int& mt, int& nt) {
    if constexpr (MODE == 1 && PAIR) {
      tile_of(order, tile, mt, nt);
    } else {                                   // W4A4: plain row order
      mt = tile / p.NT;
      nt = tile - mt * p.NT;
    }
  };
  auto half_tile = [&](int nt) { return half_col && nt == p.NT - 1; };

  auto fail = [&]() {
    *abort_flag = 1;
    if constexpr (PAIR) st_cluster_u32(map_rank(smem_u32(const_cast<int*>(abort_flag)), rank ^ 1u), 1u);
    if (p.err) atomicExch(p.err, int(kErrWaitTimeout));
  };

  // ------------------------------------------------------------ MMA issuer
  // All 32 lanes of warp 1 (leader CTA) run this loop; lane 0 issues.  W4A8
  // predicates inside the asm, W4A4 branches around each call (see the
  // wrappers above).
  constexpr bool kPredIssue = MODE == 1;
  const bool issue_lane = lane == 0;
  auto mma_issuer = [&]() {
    constexpr uint32_t idesc_full = idesc_fp4(C::kTileM, BN);
    constexpr uint32_t idesc_half = idesc_fp4(C::kTileM, BN / 2);
    // Descriptors of stage 0; stage s adds s * kStage bytes (>> 4) to the start address field.
    const uint64_t adesc_s0 = desc_kmajor<KB>(smem_u32(smem));
    const uint64_t bdesc_s0 = desc_kmajor<KB>(smem_u32(smem + C::offB));
    int stage = 0, slot = 0;
    uint32_t phase = 0, sphase = 0, acc_phase = 0;
    bool ok = true;
    if (g_sixbit_stall_mma) {
      // Test switch: wait for an arrival that never comes, so the bounded wait
      // gives up and the abort path (error word, drain, TMEM release) runs.
      if (!mbar_wait<PAIR>(never_bar, 0, abort_flag)) { fail(); ok = false; }
    }
    for (int tile = blockIdx.x / kCtas; tile < ntiles && ok; tile += gridDim.x / kCtas) {
      int mt_, nt_;
      tile_at(tile, mt_, nt_);
      const uint32_t idesc = half_tile(nt_) ? idesc_half : idesc_full;
      // the epilogue warps (of both CTAs) have pulled the previous tile out of TMEM
      if (!mbar_wait<PAIR>(tempty_bar, acc_phase ^ 1u, abort_flag)) { fail(); ok = false; break; }
      tc_fence_after();
      for (int kt = 0; kt < p.KT; ++kt) {
        // the codes landed and the scale warps (of both CTAs) have written the k-step's scales
        if (C::kSfRing && !mbar_wait(full_bar(stage), phase, abort_flag)) { fail(); ok = false; break; }
        if (!mbar_wait<PAIR>(sfready_bar(slot), C::kSfRing ? sphase : phase, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t soff = uint64_t((stage * C::kStage) >> 4);
        const uint32_t sfa_t = tmem + uint32_t(C::kSfBase + slot * C::kSfStride);
        const uint32_t sfb_t = sfa_t + uint32_t(C::kSfaCols);
#pragma unroll
        for (int c = 0; c < NC; ++c) {
#pragma unroll
          for (int j = 0; j < C::kMmaK; ++j) {
            const int a = c * C::kMmaK + j;            // MMA index within the stage = scale atom index
            if ((kt * NC * C::kMmaK + a) * 64 >= p.K) continue;   // all 64 elements past K (zero fill)
            const uint64_t bdesc = bdesc_s0 + soff + uint64_t((c * C::kChunkB + 32 * j) >> 4);
            const uint32_t sfb = sfb_t + 4 * C::kRT * a;
            if (MODE == 0) {
              const uint64_t adesc = adesc_s0 + soff + uint64_t((c * C::kChunkA + 32 * j) >> 4);
              if (kPredIssue || issue_lane)
                tc_mma_fp4<PAIR, kPredIssue>(tmem, adesc, bdesc, idesc, sfa_t + 4 * a, sfb, (kt | a) != 0);
            } else {
#pragma unroll
              for (int pl = 0; pl < 3; ++pl) {
                const uint64_t adesc = adesc_s0 + soff + uint64_t((pl * C::kA + c * C::kChunkA + 32 * j) >> 4);
                if (kPredIssue || issue_lane)
                  tc_mma_fp4<PAIR, kPredIssue>(tmem, adesc, bdesc, idesc, tmem + C::kConstCol + 4 * pl, sfb,
                                               (kt | a | pl) != 0);
              }
            }
          }
        }
        if (kPredIssue || issue_lane) tc_commit_all<PAIR, kPredIssue>(empty_bar(stage));   // frees the stage in both CTAs
        if constexpr (C::kSfRing) {
          if (kPredIssue || issue_lane) tc_commit_all<PAIR, kPredIssue>(sfempty_bar(slot));   // frees the ring slot
          if (++slot == R) { slot = 0; sphase ^= 1u; }
        } else {
          slot = stage + 1 == STAGES ? 0 : stage + 1;
        }
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      if (kPredIssue || issue_lane) tc_commit_all<PAIR, kPredIssue>(tfull_bar);
      acc_phase ^= 1u;
    }
    // all MMAs issued by this warp's lane 0 complete before TMEM is released
    if (kPredIssue || issue_lane) tc_commit_local<PAIR, kPredIssue>(drain_bar);
    mbar_wait(drain_bar, 0, nullptr);
  };

  if (warp < 4) {
    // Warpgroup 0: the producer and MMA threads (warps 2-3 idle).  The
    // register drop is warpgroup-wide, so every lane executes it here.
    regs_dec<kLowRegs>();
    if ((warp == 0 || warp == 2 || warp == 3) && lane == 0) {
      // ---------------------------------------------------------- producers
      // warp 0 loads A (codes or the three digit planes), warp 2 loads W,
      // warp 3 the scale atoms: a single thread issues about one TMA op per
      // 75 ns plus ~150 ns per stage, which one producer for all four ops
      // of a stage could not keep ahead of the stage's MMAs.
      const int role = warp == 0 ? 0 : (warp == 2 ? 1 : 2);
      if (C::kSfRing && role == 2) {
        // the scale-atom ring: paced by its own free barrier, not the code stages'
        int slot = 0;
        uint32_t sphase = 0, issued = 0, last_par = 0;
        bool ok = true;
        for (int tile = blockIdx.x / kCtas; tile < ntiles && ok; tile += gridDim.x / kCtas) {
          const int mt = tile / p.NT, nt = tile - mt * p.NT;
          const int arow = mt * C::kTileM;
          for (int kt = 0; kt < p.KT; ++kt) {
            if (!mbar_wait(sfempty_bar(slot), sphase ^ 1u, abort_flag)) { fail(); ok = false; break; }
            uint8_t* rb = ring + size_t(slot) * C::kSfSlotBytes;
            const uint32_t fb = sffull_bar(slot);
            mbar_expect_tx(fb, C::kTxS);
            if (MODE == 0) tma_load_3d(smem_u32(rb), &tmSFA, 0, kt * C::kAtoms, arow / BM, fb);
            tma_load_3d(smem_u32(rb + C::kSFA), &tmSFB, 0, kt * C::kAtoms, nt * C::kRT, fb);
            issued |= 1u << slot;
            last_par = (last_par & ~(1u << slot)) | (sphase << slot);
            if (++slot == R) { slot = 0; sphase ^= 1u; }
          }
        }
        if (!ok) {   // let the copies already issued land before the CTA exits
          for (int s = 0; s < R; ++s)
            if (issued & (1u << s)) mbar_wait(sffull_bar(s), (last_par >> s) & 1u, nullptr);
        }
      } else {
      int stage = 0;
      uint32_t phase = 0, issued = 0, last_par = 0;
      bool ok = true;
      for (int tile = blockIdx.x / kCtas; tile < ntiles && ok; tile += gridDim.x / kCtas) {
        int mt, nt;
        tile_at(tile, mt, nt);
        const int arow = mt * C::kTileM + int(rank) * BM;          // this CTA's A rows
        const int brow = nt * BN + int(rank) * (half_tile(nt) ? C::kBRows / 2 : C::kBRows);   // this CTA's W rows
        for (int kt = 0; kt < p.KT; ++kt) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag)) { fail(); ok = false; break; }
          uint8_t* sb = smem + size_t(stage) * C::kStage;
          const uint32_t fb = full_bar(stage);
          if (role == 0) {
            mbar_expect_tx(fb, C::kTxA);
            if (p.chunked) {
              if (MODE == 0) tma_load_3d(smem_u32(sb), &tmA, 0, arow, kt * NC, fb);
              else tma_load_4d(smem_u32(sb), &tmA, 0, arow, kt * NC, 0, fb);   // all three planes
            } else if (MODE == 0) {
              tma_load_2d(smem_u32(sb), &tmA, kt * KB, arow, fb);
            } else {
#pragma unroll
              for (int pl = 0; pl < 3; ++pl) tma_load_3d(smem_u32(sb + pl * C::kA), &tmA, kt * KB, arow, pl, fb);
            }
          } else if (role == 1) {
            mbar_expect_tx(fb, C::kTxB);
            if (p.chunked) tma_load_3d(smem_u32(sb + C::offB), &tmB, 0, brow, kt * NC, fb);
            else tma_load_2d(smem_u32(sb + C::offB), &tmB, kt * KB, brow, fb);
          } else {
            mbar_expect_tx(fb, C::kTxS);
            if (MODE == 0) tma_load_3d(smem_u32(sb + C::offSFA), &tmSFA, 0, kt * C::kAtoms, arow / BM, fb);
            tma_load_3d(smem_u32(sb + C::offSFB), &tmSFB, 0, kt * C::kAtoms, nt * C::kRT, fb);
          }
          issued |= 1u << stage;
          last_par = (last_par & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) {   // let the copies already issued land before the CTA exits
        for (int s = 0; s < STAGES; ++s)
          if (issued & (1u << s)) mbar_wait(full_bar(s), (last_par >> s) & 1u, nullptr);
      }
      }
    } else if (warp == 1 && rank == 0) {
      mma_issuer();
    }
  } else if (warp < 8) {
    regs_dec<kLowRegs>();
    // ------------------------------------------------------------ scale warps
    // A slot's TMEM scale columns are free again once its next scales have
    // landed: their producer waited for the MMAs that read the slot (the
    // ring's free barrier, or the stage's empty barrier without the ring).
    const int q = warp & 3;
    const uint32_t lane_base = uint32_t(q * 32) << 16;
    if (MODE == 1) {
      // constant digit scales 64, 8, 1 (E4M3 0x68, 0x50, 0x38) for every row and K block
      const uint32_t cb = tmem + lane_base + uint32_t(C::kConstCol);
      tmem_st4(cb, 0x68686868u);
      tmem_st4(cb + 4, 0x50505050u);
      tmem_st4(cb + 8, 0x38383838u);
    }
    int slot = 0;                                // ring slot (the code stage when there is no ring)
    uint32_t phase = 0;
    bool ok = true;
    for (int tile = blockIdx.x / kCtas; tile < ntiles && ok; tile += gridDim.x / kCtas) {
      for (int kt = 0; kt < p.KT; ++kt) {
        // every lane waits (each acquires the landed bytes); the verdict is
        // made warp-uniform so the .sync.aligned stores below never diverge
        const bool landed = mbar_wait(C::kSfRing ? sffull_bar(slot) : full_bar(slot), phase, abort_flag);
        if (!__all_sync(0xffffffffu, landed)) {
          if (lane == 0) fail();
          ok = false;
          break;
        }
        const uint8_t* sfa_s = C::kSfRing ? ring + size_t(slot) * C::kSfSlotBytes
                                          : smem + size_t(slot) * C::kStage + C::offSFA;
        const uint8_t* sfb_s = C::kSfRing ? sfa_s + C::kSFA : smem + size_t(slot) * C::kStage + C::offSFB;
        const uint32_t sfa_t = tmem + lane_base + uint32_t(C::kSfBase + slot * C::kSfStride);
        const uint32_t sfb_t = sfa_t + uint32_t(C::kSfaCols);
        if (MODE == 0) {
          uint4 wa[C::kAtoms];
#pragma unroll
          for (int a = 0; a < C::kAtoms; ++a) wa[a] = *reinterpret_cast<const uint4*>(sfa_s + 512 * a + 16 * lane);
          if constexpr (C::kAtoms == 4) {
            tmem_st16(sfa_t, wa[0], wa[1], wa[2], wa[3]);
          } else {
            tmem_st8(sfa_t, wa[0], wa[1]);
          }
        }
#pragma unroll
        for (int g = 0; g < C::kAtoms / 2; ++g) {   // K steps 2g, 2g+1; row tiles 0, 1 of each
          const uint8_t* b0 = sfb_s + 16 * lane;
          const uint4 w00 = *reinterpret_cast<const uint4*>(b0 + 512 * (2 * g));
          const uint4 w01 = *reinterpret_cast<const uint4*>(b0 + 512 * (C::kAtoms + 2 * g));
          const uint4 w10 = *reinterpret_cast<const uint4*>(b0 + 512 * (2 * g + 1));
          const uint4 w11 = *reinterpret_cast<const uint4*>(b0 + 512 * (C::kAtoms + 2 * g + 1));
          tmem_st16(sfb_t + 16 * g, w00, w01, w10, w11);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive_leader(sfready_bar(slot));
        if (++slot == R) { slot = 0; phase ^= 1u; }
      }
    }
    tmem_st_wait();                              // nothing of this warp is in flight at teardown
  } else {
    regs_inc<kHighRegs>();
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                      // TMEM lane quarter this warp may access
    const int ew = warp - 8;                     // epilogue warp 0..7
    const int half = ew >> 2;                    // columns [128*half, 128*half + 128)
    // bf16 output leaves through this warp's staging block: 32 rows x 64
    // columns (128 bytes a row, 16-byte chunk j of row r at j ^ (r % 8), the
    // TMA 128-byte swizzle), written by one TMA store per 64 columns.
    uint8_t* stg = staging + ew * 4096;
    const uint32_t stg_s = smem_u32(stg);
    const uint32_t rbar = resid_bar(ew);
    uint32_t acc_phase = 0, r_phase = 0;
    bool r_pending = false;                      // a residual load issued and not yet seen landed
    bool ok = true;
    const float gw = *p.g_w;
    const float gscale = MODE == 0 ? __fmul_rn(*p.g_a, gw) : gw;
    // Quantizing epilogue: the bf16 result encoded as NVFP4 for the next
    // layer, with amax_t = headroom * the previous call's |y| amax (delayed
    // scaling); a lane holds 32 consecutive columns of one row, i.e. two
    // whole 16-element blocks.  Either way the lane tracks |bf16 y|'s max
    // over its rows < M for the history.
    const bool qo = QO && p.q_hist != nullptr;   // compiled out of the plain GEMM
    const bool q_nv = qo && p.q_codes != nullptr && (p.q_pred == nullptr || *p.q_pred != 0);
    const float q_amax_t = qo ? __fmul_rn(p.q_headroom, hist_prev(p.q_hist)) : 0.f;
    const float q_g = nvfp4_global_scale(q_amax_t);
    if (q_nv && blockIdx.x == 0 && ew == 0 && lane == 0) *p.q_g = q_g;
    const int q_mpad = ((p.M + 127) / 128) * 128;   // rows of the padded scale layout
    // 1 / (S g) for every E4M3 block scale S a satfinite encode can give
    // (codes 0..126), computed once per CTA exactly as the per-block form
    // would: the upper half of the barrier area holds it.
    float* const q_rtab = reinterpret_cast<float*>(extra + 512);
    if constexpr (QO) {
      if (q_nv) {
        const int i = ew * 32 + lane;
        if (i < 128) {
          const float d = __fmul_rn(e4m3_decode(uint32_t(i)), q_g);
          q_rtab[i] = d != 0.f ? __frcp_rn(d) : 0.f;
        }
        asm volatile("bar.sync 1, 256;" ::: "memory");   // the 8 epilogue warps of this CTA
      }
    }
    uint32_t q_run = 0;                          // |y| max as two bf16 halves
    for (int tile = blockIdx.x / kCtas; tile < ntiles && ok; tile += gridDim.x / kCtas) {
      int mt, nt;
      tile_at(tile, mt, nt);
      if (!__all_sync(0xffffffffu, mbar_wait(tfull_bar, acc_phase, abort_flag))) {   // warp-uniform verdict
        if (lane == 0) fail();
        break;
      }
      tc_fence_after();
      uint32_t r0[32], r1[32], r2[32], r3[32];
      const uint32_t taddr = tmem + uint32_t(half * 128) + (uint32_t(q * 32) << 16);
      __syncwarp();
      tmem_ld32(taddr, r0);
      tmem_ld32(taddr + 32, r1);
      tmem_ld32(taddr + 64, r2);
      tmem_ld32(taddr + 96, r3);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) arrive_leader(tempty_bar);  // TMEM is free: the next tile's MMAs may start
      acc_phase ^= 1u;
      const int m0 = mt * C::kTileM + int(rank) * BM + q * 32;   // first row of this warp's block
      const int m = m0 + lane;
      const int nbase = nt * BN + half * 128;
      if (q_nv) {
        const float scale = MODE == 0 ? gscale : (m < p.M ? __fmul_rn(p.row_scale[m], gw) : 0.f);
        const int64_t kc4 = p.N / 16;
        uint32_t sfw = 0;
        const uint64_t sc2 = f2_pack(scale, scale);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t* rc = c == 0 ? r0 : (c == 1 ? r1 : (c == 2 ? r2 : r3));
          const int n0 = nbase + 32 * c;
          if (n0 >= p.N) break;                  // N % 64 == 0: whole 64-column pairs
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; i += 2)
            f2_unpack(f2_mul(f2_pack(__uint_as_float(rc[i]), __uint_as_float(rc[i + 1])), sc2), v[i], v[i + 1]);
          if (p.bias) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint4 b = *reinterpret_cast<const uint4*>(p.bias + n0 + 8 * i);
              const uint32_t* pb = &b.x;
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                v[8 * i + 2 * e] = __fadd_rn(v[8 * i + 2 * e], bf16lo(pb[e]));
                v[8 * i + 2 * e + 1] = __fadd_rn(v[8 * i + 2 * e + 1], bf16hi(pb[e]));
              }
            }
          }
          if (p.gelu) {
#pragma unroll
            for (int i = 0; i < 32; i += 2) gelu_tanh2(v[i], v[i + 1]);
          }
          uint32_t pk[16];                       // the bf16 values the unfused path would store
#pragma unroll
          for (int j = 0; j < 16; ++j) pk[j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
          // block scales: S = E4M3((amax_b 448) / amax_t), r = 1 / (S g) from the table
          const float ba = fmaxf(bf16x8_absmax(pk), bf16x8_absmax(pk + 4));
          const float bb = fmaxf(bf16x8_absmax(pk + 8), bf16x8_absmax(pk + 12));
          const uint32_t sa = e4m3_encode(q_amax_t == 0.f ? 0.f : __fdiv_rn(__fmul_rn(ba, 448.f), q_amax_t));
          const uint32_t sb = e4m3_encode(q_amax_t == 0.f ? 0.f : __fdiv_rn(__fmul_rn(bb, 448.f), q_amax_t));
          const float ra = q_rtab[sa], rb = q_rtab[sb];
          if (m < p.M) {
            q_run = __vmaxu2(q_run, __float_as_uint(fmaxf(ba, bb)) >> 16);   // the chunk's |bf16 y| max
            uint4 w;
            w.x = nvfp4_codes8(pk, ra);
            w.y = nvfp4_codes8(pk + 4, ra);
            w.z = nvfp4_codes8(pk + 8, rb);
            w.w = nvfp4_codes8(pk + 12, rb);
            *reinterpret_cast<uint4*>(p.q_codes + int64_t(m) * (p.N / 2) + n0 / 2) = w;
          }
          sfw |= (sa | (sb << 8)) << (16 * (c & 1));
          if (c & 1) {                           // 4 blocks = one word of the swizzled layout
            if (m < q_mpad)
              *reinterpret_cast<uint32_t*>(p.q_sf + sf_offset(m, (n0 - 32) / 16, kc4)) = m < p.M ? sfw : 0u;
            sfw = 0;
          }
        }
      } else if (p.out_bf16) {
        const float scale = MODE == 0 ? gscale : (m < p.M ? __fmul_rn(p.row_scale[m], gw) : 0.f);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int n0 = nbase + 64 * k;
          if (n0 >= p.N) break;
          if (lane == 0) bulk_wait_read0();      // the previous store has read the block
          __syncwarp();
          if (p.residual) {
            if (lane == 0) {
              mbar_expect_tx(rbar, 4096);
              tma_load_2d(stg_s, &tmR, n0, m0, rbar);   // rows >= M and columns >= N read as 0
            }
            r_pending = true;
            if (!__all_sync(0xffffffffu, mbar_wait(rbar, r_phase, abort_flag))) {
              if (lane == 0) fail();
              ok = false;
              break;
            }
            r_pending = false;
            r_phase ^= 1u;
          }
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t* rc = k == 0 ? (h == 0 ? r0 : r1) : (h == 0 ? r2 : r3);
            const int nc = n0 + 32 * h;
            float v[32];                         // scale, bias (and residual) in f32x2 pairs
            const uint64_t sc2 = f2_pack(scale, scale);
#pragma unroll
            for (int i = 0; i < 32; i += 2)
              f2_unpack(f2_mul(f2_pack(__uint_as_float(rc[i]), __uint_as_float(rc[i + 1])), sc2), v[i], v[i + 1]);
            if (p.bias && nc < p.N) {
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                if (nc + 8 * i >= p.N) break;
                const uint4 b = *reinterpret_cast<const uint4*>(p.bias + nc + 8 * i);
                const uint32_t* pb = &b.x;
#pragma unroll
                for (int e = 0; e < 4; ++e)
                  f2_unpack(f2_add(f2_pack(v[8 * i + 2 * e], v[8 * i + 2 * e + 1]), f2_from_bf16x2(pb[e])),
                            v[8 * i + 2 * e], v[8 * i + 2 * e + 1]);
              }
            }
            if (p.gelu) {
#pragma unroll
              for (int i = 0; i < 32; i += 2) gelu_tanh2(v[i], v[i + 1]);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int j = 4 * h + i;           // 16-byte chunk of the 128-byte row
              uint4* slot = reinterpret_cast<uint4*>(stg + lane * 128 + ((j ^ (lane & 7)) << 4));
              if (p.residual) {
                const uint4 rr = *slot;
                const uint32_t* pr = &rr.x;
#pragma unroll
                for (int e = 0; e < 4; ++e)
                  f2_unpack(f2_add(f2_pack(v[8 * i + 2 * e], v[8 * i + 2 * e + 1]), f2_from_bf16x2(pr[e])),
                            v[8 * i + 2 * e], v[8 * i + 2 * e + 1]);
              }
              uint4 w;
              w.x = pack_bf16x2(v[8 * i + 0], v[8 * i + 1]);
              w.y = pack_bf16x2(v[8 * i + 2], v[8 * i + 3]);
              w.z = pack_bf16x2(v[8 * i + 4], v[8 * i + 5]);
              w.w = pack_bf16x2(v[8 * i + 6], v[8 * i + 7]);
              *slot = w;
              if (qo && m < p.M) {
                q_run = __vmaxu2(q_run, w.x & 0x7FFF7FFFu);
                q_run = __vmaxu2(q_run, w.y & 0x7FFF7FFFu);
                q_run = __vmaxu2(q_run, w.z & 0x7FFF7FFFu);
                q_run = __vmaxu2(q_run, w.w & 0x7FFF7FFFu);
              }
            }
          }
          fence_async_smem();                    // generic writes -> visible to the TMA store
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmY, stg_s, n0, m0);   // rows >= M and columns >= N are not written
            bulk_commit();
          }
        }
      } else {
        if (m >= p.M) continue;
        const float scale = MODE == 0 ? gscale : __fmul_rn(p.row_scale[m], gw);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t* rc = c == 0 ? r0 : (c == 1 ? r1 : (c == 2 ? r2 : r3));
          const int n0 = nbase + c * 32;
          if (n0 >= p.N) break;
          const int cols = (p.N - n0) < 32 ? (p.N - n0) : 32;   // 16 or 32 (N % 16 == 0)
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __fmul_rn(__uint_as_float(rc[i]), scale);
          if (p.bias) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              if (8 * i >= cols) break;
              const uint4 b = *reinterpret_cast<const uint4*>(p.bias + n0 + 8 * i);
              const uint32_t* pb = &b.x;
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                v[8 * i + 2 * e] = __fadd_rn(v[8 * i + 2 * e], bf16lo(pb[e]));
                v[8 * i + 2 * e + 1] = __fadd_rn(v[8 * i + 2 * e + 1], bf16hi(pb[e]));
              }
            }
          }
          if (p.gelu) {
#pragma unroll
            for (int i = 0; i < 32; i += 2) gelu_tanh2(v[i], v[i + 1]);
          }
          if (p.residual) {
            const uint16_t* rp = p.residual + int64_t(m) * p.ldr + n0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              if (8 * i >= cols) break;
              const uint4 b = *reinterpret_cast<const uint4*>(rp + 8 * i);
              const uint32_t* pb = &b.x;
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                v[8 * i + 2 * e] = __fadd_rn(v[8 * i + 2 * e], bf16lo(pb[e]));
                v[8 * i + 2 * e + 1] = __fadd_rn(v[8 * i + 2 * e + 1], bf16hi(pb[e]));
              }
            }
          }
          float* yp = static_cast<float*>(p.y) + int64_t(m) * p.ldy + n0;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (4 * i >= cols) break;
            *reinterpret_cast<float4*>(yp + 4 * i) = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
          }
        }
      }
    }
    if (r_pending) mbar_wait(rbar, r_phase, nullptr);   // an aborted tile's residual load has landed
    if (lane == 0) bulk_wait0();                 // this warp's output stores are complete
    if (qo) {
      const float a = warp_max(__uint_as_float(max(q_run & 0xFFFFu, q_run >> 16) << 16));
      if (lane == 0) hist_accumulate(p.q_hist, a);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (QO && threadIdx.x == 0 && p.q_hist) hist_arrive(p.q_hist);
  if constexpr (PAIR) cluster_sync();          // the leader's MMAs into this CTA's TMEM are complete
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR)
      asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
    else
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
  }
}

// ------------------------------------------------------------------ host
// Host-side lookups below are function-local statics: C++ initializes them
// once, and host threads calling the library at the same time wait for it.
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    return PFN_cuTensorMapEncodeTiled_v12000(nullptr);
  }();
  return fn;
}

bool make_map(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base, const uint64_t* dims,
              const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle sw) {
  auto fn = encode_fn();
  if (!fn) return false;
  uint32_t es[5] = {1, 1, 1, 1, 1};   // one per dimension, up to rank 5
  return fn(m, dt, rank, const_cast<void*>(base), dims, strides_bytes, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, int MODE, int STAGES, int KB, int NC, bool PAIR, bool QO>
int run(const GemmCall& c, int num_sms, cudaStream_t s) {
  using Cf = Cfg<BN, MODE, STAGES, KB, NC, PAIR>;
  constexpr CUtensorMapSwizzle kSw = KB == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  const int64_t kb = c.K / 2;                       // bytes of codes per row
  const int64_t natoms = c.K / 64;                  // 512-byte scale atoms per 128-row tile
  // Chunked maps view each row as K/2/KB chunks of KB bytes (chunk index is
  // the outer box dimension, so a box lands as NC consecutive [rows][KB]
  // tiles); this needs KB to divide K/2, else a chunk would run into the
  // next row instead of reading the zero fill.
  const bool chunked = kb % KB == 0;
  if (!chunked && NC != 1) return kEShape;
  const int64_t nch = kb / KB;
  CUtensorMap tA, tB, tSA, tSB;
  bool ok = true;
  if (MODE == 0) {
    if (chunked) {
      uint64_t d[3] = {uint64_t(KB), uint64_t(c.M), uint64_t(nch)}, st[2] = {uint64_t(kb), uint64_t(KB)};
      uint32_t b[3] = {uint32_t(KB), uint32_t(BM), uint32_t(NC)};
      ok &= make_map(&tA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, c.a, d, st, b, kSw);
    } else {
      uint64_t d[2] = {uint64_t(kb), uint64_t(c.M)}, st[1] = {uint64_t(kb)};
      uint32_t b[2] = {uint32_t(KB), uint32_t(BM)};
      ok &= make_map(&tA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, c.a, d, st, b, kSw);
    }
  } else {
    if (chunked) {
      uint64_t d[4] = {uint64_t(KB), uint64_t(c.M), uint64_t(nch), 3};
      uint64_t st[3] = {uint64_t(kb), uint64_t(KB), uint64_t(kb) * uint64_t(c.M)};
      uint32_t b[4] = {uint32_t(KB), uint32_t(BM), uint32_t(NC), 3};
      ok &= make_map(&tA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, c.a, d, st, b, kSw);
    } else {
      uint64_t d[3] = {uint64_t(kb), uint64_t(c.M), 3}, st[2] = {uint64_t(kb), uint64_t(kb) * uint64_t(c.M)};
      uint32_t b[3] = {uint32_t(KB), uint32_t(BM), 1};
      ok &= make_map(&tA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, c.a, d, st, b, kSw);
    }
  }
  if (chunked) {
    uint64_t d[3] = {uint64_t(KB), uint64_t(c.N), uint64_t(nch)}, st[2] = {uint64_t(kb), uint64_t(KB)};
    uint32_t b[3] = {uint32_t(KB), uint32_t(Cf::kBRows), uint32_t(NC)};
    ok &= make_map(&tB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, c.w, d, st, b, kSw);
  } else {
    uint64_t d[2] = {uint64_t(kb), uint64_t(c.N)}, st[1] = {uint64_t(kb)};
    uint32_t b[2] = {uint32_t(KB), uint32_t(Cf::kBRows)};
    ok &= make_map(&tB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, c.w, d, st, b, kSw);
  }
  {
    // scale atoms: [row tile][K step][128 x u32]; a box brings kAtoms K steps of one (A) or kRT (W) row tiles
    uint64_t d2[3] = {128, uint64_t(natoms), uint64_t(cdiv(c.N, 128))}, st2[2] = {512, uint64_t(natoms) * 512};
    uint32_t b2[3] = {128, uint32_t(Cf::kAtoms), uint32_t(Cf::kRT)};
    ok &= make_map(&tSB, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, c.w_sf, d2, st2, b2, CU_TENSOR_MAP_SWIZZLE_NONE);
    tSA = tSB;   // unused in mode 1
    if (MODE == 0) {
      uint64_t d3[3] = {128, uint64_t(natoms), uint64_t(cdiv(c.M, 128))};
      uint32_t b3[3] = {128, uint32_t(Cf::kAtoms), 1};
      ok &= make_map(&tSA, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, c.a_sf, d3, st2, b3, CU_TENSOR_MAP_SWIZZLE_NONE);
    }
  }
  // bf16 output (and residual) through 32-row x 64-column boxes, 128-byte swizzle
  CUtensorMap tY = tB, tR = tB;
  if (c.out_bf16) {
    uint64_t d[2] = {uint64_t(c.N), uint64_t(c.M)}, st[1] = {uint64_t(c.ldy) * 2};
    uint32_t b[2] = {64, 32};
    ok &= make_map(&tY, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, c.y, d, st, b, CU_TENSOR_MAP_SWIZZLE_128B);
    if (c.residual) {
      uint64_t dr[2] = {uint64_t(c.N), uint64_t(c.M)}, sr[1] = {uint64_t(c.ldr) * 2};
      ok &= make_map(&tR, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, c.residual, dr, sr, b, CU_TENSOR_MAP_SWIZZLE_128B);
    }
  }
  if (!ok) return kELaunch;
  Params p;
  p.M = int(c.M); p.N = int(c.N); p.K = int(c.K);
  p.KT = int(chunked ? cdiv(nch, NC) : cdiv(kb, KB));
  p.MT = int(cdiv(c.M, Cf::kTileM));
  p.NT = int(cdiv(c.N, BN));
  p.g_a = c.g_a; p.row_scale = c.row_scale; p.g_w = c.g_w;
  p.bias = static_cast<const uint16_t*>(c.bias);
  p.residual = static_cast<const uint16_t*>(c.residual);
  p.ldr = c.ldr; p.y = c.y; p.ldy = c.ldy; p.out_bf16 = c.out_bf16; p.gelu = c.gelu; p.pred = c.pred; p.err = c.err;
  p.chunked = chunked ? 1 : 0;
  p.q_codes = c.q_codes; p.q_sf = c.q_sf; p.q_g = c.q_g; p.q_hist = c.q_hist; p.q_headroom = c.q_headroom;
  p.q_pred = c.q_pred;

  auto kern = gemm_fp4_kernel<BN, MODE, STAGES, KB, NC, PAIR, QO>;
  static const bool attr_ok = [&] {
    // The register split (setmaxnreg) assumes exactly kLaunchRegs per thread
    // at launch; any other allocation would leave the epilogue's request
    // unsatisfiable, so such a build is refused here.
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess || fa.numRegs != kLaunchRegs) return false;
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(Cf::kSmem)) == cudaSuccess;
  }();
  if (!attr_ok) return kELaunch;
  const int tiles = p.MT * p.NT;
  constexpr int kCtas = PAIR ? 2 : 1;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCtas;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Cf::kSmem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // persistent grid: as many CTA pairs (or CTAs) as can be resident at once
  static const int resident = [&] {
    cfg.gridDim = dim3(kCtas * (num_sms / kCtas));
    int n = 0;
    if (PAIR && cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n > 0) return n;
    return num_sms / kCtas;
  }();
  const int units = tiles < resident ? tiles : resident;
  cfg.gridDim = dim3(kCtas * units);
  if (cudaLaunchKernelEx(&cfg, kern, tA, tB, tSA, tSB, tY, tR, p) != cudaSuccess) return kELaunch;
  return cudaGetLastError() == cudaSuccess ? kOk : kELaunch;
}

}  // namespace

int launch_gemm_fp4(const GemmCall& c, int num_sms, cudaStream_t s) {
  // W4A8 (three MMAs per K step) keeps 64-byte K steps: three planes of
  // 128-byte rows would leave room for only two stages.  K % 128 == 0:
  // chunked maps, one TMA op per operand; otherwise 2-D maps.
  const bool chunked = (c.K / 2) % 64 == 0;
  // W4A4: 128-byte K steps (a 128-byte box row per TMA row: 7-8% faster than
  // two 64-byte chunks); the K tail past K/2 bytes reads as zeros.
  // The quantizing epilogue is a separate instantiation: its code, even
  // when not taken, slowed the plain epilogue (the critical path of the
  // K = 1920 layers) by 5-10%.
  if (c.q_hist) {
    if (c.mode == 0) return run<256, 0, W4A4_PAIR ? 5 : 3, 128, 1, W4A4_PAIR, true>(c, num_sms, s);
    return chunked ? run<256, 1, W4A8_STAGES, 64, W4A8_NC, GEMM_PAIR, true>(c, num_sms, s)
                   : run<256, 1, W4A8_STAGES, 64, 1, GEMM_PAIR, true>(c, num_sms, s);
  }
  if (c.mode == 0) return run<256, 0, W4A4_PAIR ? 5 : 3, 128, 1, W4A4_PAIR, false>(c, num_sms, s);
  return chunked ? run<256, 1, W4A8_STAGES, 64, W4A8_NC, GEMM_PAIR, false>(c, num_sms, s)
                 : run<256, 1, W4A8_STAGES, 64, 1, GEMM_PAIR, false>(c, num_sms, s);
}

}  // namespace sixbit
