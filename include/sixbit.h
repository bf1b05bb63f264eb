/*
 * sixbit.h -- C ABI of the GB300 (sm_103a) hot path of 6Bit-Diffusion:
 * inference-time NVFP4/INT8 mixed-precision quantized linear layers for
 * video diffusion transformers, with the DMPQ precision predictor and the
 * Temporal Delta Cache (TDC).
 *
 * Method source: "6Bit-Diffusion: Inference-Time Mixed-Precision
 * Quantization for Video Diffusion Models" (arXiv 2603.18742) --
 * mlsanity.com page, "Abstract"; thelatestinai.com page, Figures 1-4 and
 * Tables 2-3.  Each entry point names the passage that defines it.
 *
 * Conventions for every call:
 *  - Pointers are DEVICE pointers owned by the caller unless stated.  The
 *    library never allocates or frees device memory; scratch ("ws") is
 *    caller memory of sixbit_workspace_size() bytes.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream) and never synchronizes the host, except
 *    sixbit_get_error().
 *  - bf16 tensors are raw 16-bit bf16 bit patterns, row-major; `ld*` is the
 *    row stride in elements.  Sizes are element counts.
 *  - `pred` (nullable) is a device byte: the launched kernels exit at once
 *    when *pred == 0.  This is how on-device DMPQ/TDC decisions gate work
 *    without a host round trip.
 *  - Return value: SIXBIT_OK, or a negative code for an argument the host
 *    can check (nothing is launched then), or SIXBIT_ELAUNCH when CUDA
 *    rejected a launch.  Device-side failures (a bounded wait that gave up)
 *    set a device error word read by sixbit_get_error().
 */
#ifndef SIXBIT_H
#define SIXBIT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* sixbit_stream_t;   /* same object as cudaStream_t */

enum {
  SIXBIT_OK = 0,
  SIXBIT_EINVAL = -1,   /* null pointer where one is required, bad enum, negative size */
  SIXBIT_ESHAPE = -2,   /* unsupported shape, e.g. K % 64 != 0 for NVFP4 operands */
  SIXBIT_EALIGN = -3,   /* pointer or stride not 16-byte aligned where TMA/vector loads need it */
  SIXBIT_ELAUNCH = -4,  /* CUDA launch or driver error */
  SIXBIT_EDEVICE = -5   /* returned by sixbit_get_error(): a device wait gave up */
};

/* Calls over M rows (amax, the activation quantizers, the linear layers, the
 * LayerNorms) return SIXBIT_OK at once when M == 0, before any check: no
 * pointer is used, so an empty tensor's NULL data pointer is accepted.
 * Calls over n elements (the Gamma passes, the pair sums, the TDC calls)
 * need n >= 1 and return SIXBIT_EINVAL for n <= 0: a block's update is
 * never empty, and an empty one has no defined Gamma. */
enum { SIXBIT_F32 = 0, SIXBIT_BF16 = 1 };          /* dtype / out_dtype */
enum { SIXBIT_EPI_GELU = 1 };                       /* epilogue flag bits */
enum { SIXBIT_QOUT_W4A4 = 0, SIXBIT_QOUT_W4A8 = 1 };  /* sixbit_qlinear_qout mode */

/* Library version string (static storage). */
const char* sixbit_version(void);

/* Bytes of the swizzled E4M3 scale-factor buffer of an NVFP4 operand with
 * `rows` rows and reduction length K: rows padded to 128, K/16 scale columns
 * padded to 4.  Byte of (row m, scale column c) sits at
 *   ((m/128)*(Kc4/4) + c/4)*512 + (m%32)*16 + ((m%128)/32)*4 + c%4
 * (the 128x4 atom layout the block-scaled tensor-core MMA reads). */
size_t sixbit_sf_bytes(int64_t rows, int64_t K);

/* Scratch bytes for sixbit_quantize_act_nvfp4(amax_in = NULL),
 * sixbit_quantize_weight_nvfp4 and sixbit_block_gamma over n = M*K elements.
 * The buffer must be zero-filled once before its first use; every call
 * leaves it ready for the next (calls sharing one buffer must not overlap). */
size_t sixbit_workspace_size(int64_t M, int64_t K);

/* a1 -- absolute maxima of a bf16 tensor [M, K] (row stride ldx).
 * amax_out (nullable): max |x| over the tensor (the NVFP4 tensor amax);
 * row_amax_out (nullable): max |x| per row, [M] (the per-token INT8 amax).
 * Source: NVFP4/INT8 activation quantization on the fly ("Abstract",
 * mlsanity.com page).  At least one output must be given. */
int sixbit_amax_bf16(const void* x, int64_t M, int64_t K, int64_t ldx,
                     float* amax_out, float* row_amax_out, sixbit_stream_t stream);

/* a2 -- NVFP4 activation quantization ("Abstract": NVFP4 for temporally
 * stable layers).  x bf16 [M, K], K % 64 == 0, ldx % 8 == 0.
 *   g = amax/2688 (1 if amax = 0); per 16-block S = E4M3(amax_b*448/amax);
 *   codes = E2M1(x * (1/(S*g))) (RNE, satfinite), +0 codes when S*g = 0.
 * amax_in (nullable): tensor amax from the producer; when NULL the call
 *   runs its own amax pass into `ws` (then ws must be non-NULL).
 * codes: [M, K/2] bytes, element 2j in the low nibble.
 * sf: sixbit_sf_bytes(M, K) bytes, swizzled; pad rows are written as 0.
 * g_out: [1] float, the dequantization tensor scale. */
int sixbit_quantize_act_nvfp4(const void* x, int64_t M, int64_t K, int64_t ldx,
                              const float* amax_in, uint8_t* codes, uint8_t* sf, float* g_out,
                              const uint8_t* pred, void* ws, sixbit_stream_t stream);

/* a4 -- NVFP4 weight quantization, offline, same rules as a2 on W [N, K]
 * (out x in, K contiguous).  dtype SIXBIT_F32 or SIXBIT_BF16.  Uses ws for
 * the tensor amax.  Source: "W4" weights of Table 2 / Table 3. */
int sixbit_quantize_weight_nvfp4(const void* w, int dtype, int64_t N, int64_t K,
                                 uint8_t* codes, uint8_t* sf, float* g_out,
                                 void* ws, sixbit_stream_t stream);

/* a3 -- per-token symmetric INT8 activation quantization ("Abstract": INT8
 * for volatile layers).  x bf16 [M, K], K % 64 == 0, K <= 16384.
 *   inv = 127/amax_m; q = clamp(rne(x*inv), -127, 127); s_m = amax_m/127;
 *   a zero row gives q = 0, s_m = 0.
 * row_amax_in (nullable): per-row amax from the producer.
 * q (nullable): int8 [M, K].
 * planes (nullable): the GEMM operand form of q, three E2M1 digit planes
 *   [3][M][K/2] bytes with q = 64*a + 8*b + c (plane 0 = a, 1 = b, 2 = c;
 *   each digit an integer in [-4, 4]); exact, no rounding.
 * row_scale: [M] float s_m.  At least one of q / planes must be given. */
int sixbit_quantize_act_int8(const void* x, int64_t M, int64_t K, int64_t ldx,
                             const float* row_amax_in, int8_t* q, uint8_t* planes,
                             float* row_scale, const uint8_t* pred, sixbit_stream_t stream);

/* The W4A8 operand form of plain INT8 activations, for callers that hold
 * per-token int8 codes from elsewhere (their own quantizer, a previous
 * layer): q int8 [M, K] (row stride ldq, ldq % 16 == 0), K % 64 == 0, ->
 * planes [3][M][K/2], the exact digit split q = 64a + 8b + c that
 * sixbit_quantize_act_int8 writes (digits in [-4, 4] as E2M1 codes, element
 * 2j in the low nibble).  Codes outside [-127, 127] (-128) are split
 * exactly too (a = -2, b = 0, c = 0).  With the row scales the caller already
 * has, sixbit_qlinear_w4a8 then runs on these planes.  One streaming pass:
 * 1 byte read and 1.5 bytes written per element. */
int sixbit_int8_digit_planes(const int8_t* q, int64_t M, int64_t K, int64_t ldq, uint8_t* planes,
                             sixbit_stream_t stream);

/* a5 -- W4A4 linear: y = g_a g_w sum_k (E2M1*S)_a (E2M1*S)_w + bias,
 * optional tanh-GELU, optional + residual; fp32 accumulation on tcgen05
 * block-scaled FP4 tensor cores.  Source: uniform W4A4 of Table 3, NVFP4
 * layers of the "Abstract".
 * A: codes [M, K/2], sf swizzled for M rows, g_a [1].  W: codes [N, K/2],
 * sf swizzled for N rows, g_w [1].  K % 64 == 0, N % 16 == 0.
 * bias (nullable) bf16 [N]; residual (nullable) bf16 [M, N] stride ldr;
 * epi: SIXBIT_EPI_GELU bit; out_dtype SIXBIT_F32 / SIXBIT_BF16;
 * y [M, N] stride ldy (ldy*elt % 16 == 0). */
int sixbit_qlinear_w4a4(const uint8_t* a_codes, const uint8_t* a_sf, const float* g_a,
                        int64_t M, int64_t K,
                        const uint8_t* w_codes, const uint8_t* w_sf, const float* g_w, int64_t N,
                        const void* bias, const void* residual, int64_t ldr, int epi,
                        int out_dtype, void* y, int64_t ldy,
                        const uint8_t* pred, sixbit_stream_t stream);

/* a6 -- W4A8 linear: y = s_a[m] g_w sum_k q (E2M1*S)_w + same epilogue.
 * Source: uniform W4A8 of Table 3, INT8 layers of the "Abstract".
 * The INT8 activations come as the digit planes of sixbit_quantize_act_int8
 * ([3][M][K/2]) plus row_scale [M]; the products q*w are exact and
 * accumulate in fp32 on the FP4 tensor cores (three digit MMAs per K step).
 * Weights, epilogue and constraints as sixbit_qlinear_w4a4. */
int sixbit_qlinear_w4a8(const uint8_t* a_planes, const float* row_scale, int64_t M, int64_t K,
                        const uint8_t* w_codes, const uint8_t* w_sf, const float* g_w, int64_t N,
                        const void* bias, const void* residual, int64_t ldr, int epi,
                        int out_dtype, void* y, int64_t ldy,
                        const uint8_t* pred, sixbit_stream_t stream);

/* a7 -- one pass over a block's input/output (Figure 2: Gamma; Figure 4:
 * update Delta and its relative L2 change).  in, out: bf16 [n] (whole block
 * tensor).  Always: gamma_out[0] = ||out-in||_1/||in||_1 (0 if ||in|| = 0).
 * computed (nullable; NULL = computed): the TDC byte of this step, 1 if
 * the block ran, 0 if TDC skipped it.  When computed and delta != NULL:
 * delta (bf16 [n], in: previous update, out: bf16(f32(out)-f32(in))) is
 * replaced in place, and if tdc_state[0] >= 1 (or tdc_state is NULL and
 * r2_out is given) the relative change
 * r2_out[0] = ||D_new-D_old||^2/||D_old||^2 (+inf if ||D_old|| = 0) is
 * written.  tdc_state (nullable) int32[2] = {fresh_count, consec}:
 * computed -> {fresh+1, 0}; skipped -> {fresh, consec+1}.
 * Reduction (a reading: the pages fix no precision): float32 terms
 * (d = out - in, |d|, |in|; e = D_new - D_old, e*e, D_old*D_old, each rounded
 * once), summed by one fixed tree -- 8192-element tiles; in a tile, lane t
 * of 256 adds elements j*2048 + 8t + e (j < 4, e < 8) in order in float32;
 * lanes combine by a butterfly within each 32 (t^16, ..., t^1), then the 8
 * group sums by halving; tile sums are added in float64 into 256 chains
 * (tile k to chain k % 256, in order) and the chain sums are halved;
 * Gamma = f32(S1/S0), r2 = f32(Sd/So).  The result depends only on the
 * input, never on the GPU.  ws: sixbit_workspace_size(n, 1) bytes (a
 * 256-byte header and 4 doubles a chain: 8448 bytes whatever n).  Tiles
 * are staged through shared memory by bulk copies; a bounded wait for one
 * that gives up sets the device error word (sixbit_get_error). */
int sixbit_block_gamma(const void* in, const void* out, int64_t n, void* delta,
                       float* gamma_out, float* r2_out, int32_t* tdc_state,
                       const uint8_t* computed, void* ws, sixbit_stream_t stream);

/* Scratch-free variant of sixbit_block_gamma.  The paper has no counterpart:
 * this exists for callers that cannot hand the library scratch memory --
 * applications whose device memory is fully planned by another allocator,
 * or code running where allocation is not allowed (a plugin's enqueue step,
 * a latency-critical loop that cannot take cudaMalloc's implicit device
 * synchronization).  Same arguments and results as sixbit_block_gamma
 * without `ws`; n <= SIXBIT_NOALLOC_GAMMA_MAX_ELEMS (the limit of
 * sixbit_block_gamma), else SIXBIT_ESHAPE and nothing is launched.  The
 * scratch is a fixed 8448-byte device array inside the library (the same
 * layout as `ws`) that every device loading the library holds until the
 * process exits.  The first call on a device looks up that array's device
 * address (with the device current), so make that first call before any
 * stream capture.  Every call clears the array's counter (an async memset on
 * `stream`) and then reuses it, so calls whose kernels overlap on the GPU --
 * on different streams, or on different host threads -- race and must be
 * avoided.  Allocates no device memory. */
#define SIXBIT_NOALLOC_GAMMA_MAX_ELEMS (((int64_t)1) << 40)
int sixbit_block_gamma_noalloc(const void* in, const void* out, int64_t n, void* delta,
                               float* gamma_out, float* r2_out, int32_t* tdc_state,
                               const uint8_t* computed, sixbit_stream_t stream);

/* DMPQ calibration diagnostic (Figure 1: per-layer relative L2 quantization
 * error; Figure 4: updates compared by cosine similarity and relative L2).
 * One pass over two tensors of n elements (a_dtype, b_dtype: SIXBIT_BF16 or
 * SIXBIT_F32; n % 8 == 0; 16-byte aligned):
 *   out[0..3] = float64 {sum (a-b)^2, sum b^2, sum a*b, sum a^2}
 * so ||a-b||/||b|| = sqrt(out[0]/out[1]) and cos = out[2]/sqrt(out[3]*out[1]).
 * Each term is rounded once in float32 (d = a - b, then d*d; b*b; a*b;
 * a*a) and the sums follow the fixed tree of sixbit_block_gamma, so the
 * result depends only on the input.  ws: sixbit_workspace_size(n, 1) bytes
 * of scratch; out: 4 device doubles. */
int sixbit_pair_stats(const void* a, int a_dtype, const void* b, int b_dtype, int64_t n,
                      double* out, void* ws, sixbit_stream_t stream);

/* a8 -- DMPQ assignment (Figure 3: per-layer line E_rel = alpha*Gamma_{t-1}
 * + beta; "Abstract": NVFP4 for stable layers).  For each layer l:
 *   p = f32(f32(alpha[l]*gamma[layer_block[l]]) + beta[l]);
 *   use_nvfp4[l] = (*step > 0) && (p < tau)      (tie -> INT8)
 * gates (nullable) uint8 [n_layers][2] = {use_nvfp4, !use_nvfp4}: the
 * `pred` bytes of the layer's NVFP4 and INT8 kernels.  step: device int32. */
int sixbit_dmpq_assign(const float* gamma, const float* alpha, const float* beta,
                       const int32_t* layer_block, int32_t n_layers, float tau,
                       const int32_t* step, uint8_t* use_nvfp4, uint8_t* gates,
                       sixbit_stream_t stream);

/* a9 -- TDC decision and reuse (Figure 2: skip from the updates of the two
 * preceding steps; "Abstract": skip invariant blocks).
 *   refresh = refresh_every > 0 && *step % refresh_every == 0
 *   skip = !refresh && tdc_state[0] >= 2 && r2[0] < f32(tau_tdc^2)
 *          && tdc_state[1] < max_skip
 * compute_out[0] = !skip.  If skip: out = bf16(f32(in) + f32(delta)) over n
 * elements and gates[0..n_gates) are cleared (so the block's kernels exit).
 * The counters are advanced by sixbit_block_gamma, not here.
 * max_skip > 1 and refresh_every > 0 are the PDR variants (Table 3 names
 * "PDR" without defining it): consecutive reuses allowed, and a forced
 * computed step every refresh_every steps.  refresh_every = 0: off (then
 * step may be NULL); step: device int32, the denoising step index. */
int sixbit_tdc_decide_and_apply(const void* in, const void* delta, int64_t n, const float* r2,
                                float tau_tdc, int32_t max_skip, int32_t refresh_every,
                                const int32_t* step, const int32_t* tdc_state,
                                uint8_t* compute_out, void* out, uint8_t* gates, int32_t n_gates,
                                sixbit_stream_t stream);

/* ---- Compressed update cache (an extension, not from the pages: Figure 2
 * reuses a block's update, the pages do not say how it is stored).  One bf16
 * update per block is 2 B/element (2-9 GB for the pages' models); this
 * cache stores it as E4M3 codes with one power-of-two scale per 32
 * consecutive elements, 1.03 B/element:
 *   k_b = the smallest integer with max|D| over block b <= 448 * 2^k_b,
 *         clamped to [-127, 127] (-127 for a zero block);
 *   code_i = E4M3(D_i * 2^-k_b) (round to nearest even, saturating);
 *   cached value = E4M3(code_i) * 2^k_b.
 * Layout: n code bytes, then n/32 scale bytes (k_b + 127).  Element type and
 * block size are those of OCP MXFP8 (E4M3); its shared-exponent rule can
 * clip a block's largest element, this one does not.  n % 32 == 0. */

/* Bytes of a compressed cache for n elements (0 if n <= 0 or n % 32 != 0). */
size_t sixbit_mxcache_bytes(int64_t n);

/* a7 with the compressed cache: as sixbit_block_gamma, with `cache`
 * (sixbit_mxcache_bytes(n), 16-byte aligned, nullable) in place of delta.
 * r2 compares the exact D_new = bf16(f32(out)-f32(in)) with the cached value
 * of the previous update; a computed block stores D_new encoded.
 * ws: sixbit_workspace_size(n, 1) bytes. */
int sixbit_block_gamma_mxcache(const void* in, const void* out, int64_t n, void* cache,
                               float* gamma_out, float* r2_out, int32_t* tdc_state,
                               const uint8_t* computed, void* ws, sixbit_stream_t stream);

/* a9 with the compressed cache: the decision of sixbit_tdc_decide_and_apply;
 * a skipped block's output is bf16(f32(in) + cached value). */
int sixbit_tdc_decide_and_apply_mxcache(const void* in, const void* cache, int64_t n, const float* r2,
                                        float tau_tdc, int32_t max_skip, int32_t refresh_every,
                                        const int32_t* step, const int32_t* tdc_state,
                                        uint8_t* compute_out, void* out, uint8_t* gates, int32_t n_gates,
                                        sixbit_stream_t stream);

/* Block harness: LayerNorm without affine over rows of H, eps given,
 * fp32 statistics, bf16 out.  Optional side outputs for the next quantizer:
 * amax_out (tensor max |y|, zeroed by the call) and row_amax_out [M].
 * Rows may be staged through shared memory by bulk copies; a bounded wait
 * for one that gives up sets the device error word (sixbit_get_error). */
int sixbit_layernorm_bf16(const void* x, int64_t M, int64_t H, int64_t ldx, float eps,
                          void* y, int64_t ldy, float* amax_out, float* row_amax_out,
                          const uint8_t* pred, sixbit_stream_t stream);

/* ---- Quantizing producers (an extension, not from the pages): the next
 * linear layer's activation quantization fused into the kernel that
 * produces the activation, which removes the bf16 write and re-read of it.
 *
 * Delayed scaling.  A one-pass producer cannot know the tensor amax of what
 * it produces, so its NVFP4 output uses amax_t = headroom * (the exact
 * tensor amax of its previous call's output), read from `amax_hist`, and
 * records this call's exact amax there for the next call.  amax_hist:
 * device uint32[4], 16-byte aligned, one per producing layer, zeroed by the
 * caller before the first call and then owned by the library (previous
 * amax, running amax, CTA ticket; the call's last CTA rolls it over, so no
 * other kernel is needed).  Calls that share one amax_hist must be ordered
 * on one stream.  With a zero history every NVFP4 code is 0 (amax_t = 0).
 * With a power-of-two headroom and an unchanged amax the codes equal those
 * of sixbit_quantize_act_nvfp4 with the true amax (S halves, g doubles);
 * an amax that grew past headroom * previous saturates the largest blocks.
 * INT8 outputs need no history: a row-owning producer knows the row amax.
 * Results equal: the bf16 value the unfused producer would store, then the
 * quantizer of a2 (NVFP4 with amax_in = headroom * previous amax) or a3. */

/* LayerNorm (as sixbit_layernorm_bf16) that also quantizes its output.
 * Outputs, each optional, at least one given:
 *   y        bf16 [M, ldy];
 *   NVFP4    codes [M, H/2], sf (sixbit_sf_bytes(M, H)), g_out[0], by delayed
 *            scaling from amax_hist (required with codes); written when
 *            nv_pred is NULL or *nv_pred != 0;
 *   INT8     planes [3][M][H/2] and row_scale [M] as sixbit_quantize_act_int8
 *            with the row's own amax; written when i8_pred is NULL or
 *            *i8_pred != 0.
 * amax_hist (nullable without codes) records |y|'s tensor amax.
 * H % 16 == 0, H <= 4096, and H % 64 == 0 with codes or planes. */
int sixbit_layernorm_quant(const void* x, int64_t M, int64_t H, int64_t ldx, float eps,
                           void* y, int64_t ldy,
                           uint8_t* codes, uint8_t* sf, float* g_out, uint32_t* amax_hist, float headroom,
                           const uint8_t* nv_pred,
                           uint8_t* planes, float* row_scale, const uint8_t* i8_pred,
                           const uint8_t* pred, sixbit_stream_t stream);

/* Linear layer with a quantizing epilogue: the product and epilogue of
 * sixbit_qlinear_w4a4 (mode SIXBIT_QOUT_W4A4: a = codes, a_sf, g_a) or
 * sixbit_qlinear_w4a8 (mode SIXBIT_QOUT_W4A8: a = digit planes, row_scale),
 * bias and SIXBIT_EPI_GELU allowed, no residual, a bf16 result.  When q_pred
 * is NULL or *q_pred != 0 the result leaves as NVFP4 for the next layer --
 * q_codes [M, N/2], q_sf (sixbit_sf_bytes(M, N)), q_g[0], delayed scaling from
 * amax_hist -- and y is not written; otherwise it leaves as bf16 y [M, ldy]
 * (for an INT8 next layer).  amax_hist records |y|'s amax either way.
 * N % 64 == 0 (the next layer's K).
 * q_codes, q_sf, q_g may all be NULL: then y is always written and the call
 * is the plain linear layer with an exact amax side output -- after it,
 * amax_hist[0] holds max |y| as a float (a next quantizer's amax_in, which
 * then skips its own amax pass); N % 16 == 0 suffices. */
int sixbit_qlinear_qout(int mode, const uint8_t* a, const uint8_t* a_sf, const float* g_a,
                        const float* row_scale, int64_t M, int64_t K,
                        const uint8_t* w_codes, const uint8_t* w_sf, const float* g_w, int64_t N,
                        const void* bias, int epi, void* y, int64_t ldy,
                        uint8_t* q_codes, uint8_t* q_sf, float* q_g, uint32_t* amax_hist, float headroom,
                        const uint8_t* q_pred, const uint8_t* pred, sixbit_stream_t stream);

/* Test switch of the failure path (no counterpart in the pages).  on != 0:
 * every linear-layer launch on the current device that follows makes its
 * MMA-issuing thread wait on a barrier nothing signals, so that bounded wait
 * expires (after its normal poll cap): the kernel records SIXBIT_EDEVICE in
 * the device error word, tells its other roles to stop, waits for its own
 * copies and MMAs in flight, frees its tensor memory and exits, leaving the
 * output undefined.  on = 0 restores normal operation.  Synchronous (a
 * copy to a device variable); allocates nothing.  For tests of the
 * sixbit_get_error() contract only. */
int sixbit_debug_stall_gemm(int on);

/* Test switch of the same kind for the kernels that stage their inputs
 * through shared memory with bulk copies (no counterpart in the pages):
 * the LayerNorm producers in their row-prefetch form (sixbit_layernorm_bf16
 * with rows of up to 2048, sixbit_layernorm_quant writing a bf16 output
 * with rows of up to 2048 or a quantized output with longer rows) and the
 * Gamma passes (sixbit_block_gamma, its scratch-free and compressed-cache
 * forms).  on != 0: each warp (LayerNorm) or CTA (Gamma) waits for its first
 * row or tile on a barrier nothing signals; the bounded wait expires, the
 * kernel records SIXBIT_EDEVICE, waits for its own copies in flight and
 * stops, leaving the outputs undefined (a Gamma pass still completes its
 * CTA count, so the scratch stays consistent).  on = 0 restores normal
 * operation.  Synchronous; allocates nothing.  For tests of the
 * sixbit_get_error() contract only. */
int sixbit_debug_stall_staging(int on);

/* Synchronizes `stream`, returns SIXBIT_EDEVICE if a device wait gave up
 * since the last call (and clears the word), else the stream's CUDA status
 * mapped to SIXBIT_OK / SIXBIT_ELAUNCH. */
int sixbit_get_error(sixbit_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* SIXBIT_H */
