// Host-side launchers of the sixbit kernels (internal to the library).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace sixbit {

int launch_amax(const void* x, int dtype, int64_t M, int64_t K, int64_t ldx, float* amax_out, float* row_amax_out,
                const uint8_t* pred, int num_sms, cudaStream_t s);
int launch_nvfp4_quant(const void* x, int dtype, int64_t M, int64_t K, int64_t ldx, const float* amax,
                       uint8_t* codes, uint8_t* sf, float* g_out, const uint8_t* pred, int num_sms, cudaStream_t s);
int launch_int8_planes(const int8_t* q, int64_t M, int64_t K, int64_t ldq, uint8_t* planes, int num_sms,
                       cudaStream_t s);
int launch_int8_quant(const void* x, int64_t M, int64_t K, int64_t ldx, const float* row_amax_in, int8_t* q,
                      uint8_t* planes, float* row_scale, const uint8_t* pred, int num_sms, cudaStream_t s);

size_t gamma_ws_bytes(int64_t n);
int launch_block_gamma(const void* xin, const void* xout, int64_t n, void* delta, float* gamma_out, float* r2_out,
                       int32_t* tdc_state, const uint8_t* computed, void* ws, int* err, cudaStream_t s);
int64_t block_gamma_noalloc_max_elems();
int launch_block_gamma_noalloc(const void* xin, const void* xout, int64_t n, void* delta, float* gamma_out,
                               float* r2_out, int32_t* tdc_state, const uint8_t* computed, int* err,
                               cudaStream_t s);
// The compressed update cache (E4M3 + power-of-two scale per 32 elements; n % 32 == 0).
int launch_block_gamma_mx(const void* xin, const void* xout, int64_t n, void* cache, float* gamma_out, float* r2_out,
                          int32_t* tdc_state, const uint8_t* computed, void* ws, int* err, cudaStream_t s);
int launch_tdc_mx(const void* xin, const void* cache, int64_t n, const float* r2, float tau2, int32_t max_skip,
                  int32_t refresh_every, const int32_t* step, const int32_t* tdc_state, uint8_t* compute_out,
                  void* out, uint8_t* gates, int32_t n_gates, int num_sms, cudaStream_t s);
int launch_pair_stats(const void* a, int a_f32, const void* b, int b_f32, int64_t n, double* out, void* ws,
                      cudaStream_t s);
int launch_dmpq(const float* gamma, const float* alpha, const float* beta, const int32_t* layer_block,
                int32_t n_layers, float tau, const int32_t* step, uint8_t* use_nvfp4, uint8_t* gates, cudaStream_t s);
int launch_tdc(const void* xin, const void* delta, int64_t n, const float* r2, float tau2, int32_t max_skip,
               int32_t refresh_every, const int32_t* step,
               const int32_t* tdc_state, uint8_t* compute_out, void* out, uint8_t* gates, int32_t n_gates,
               int num_sms, cudaStream_t s);
int launch_layernorm(const void* x, int64_t M, int64_t H, int64_t ldx, float eps, void* y, int64_t ldy,
                     float* amax_out, float* row_amax_out, const uint8_t* pred, int* err, int num_sms, cudaStream_t s);

// LayerNorm that also quantizes its output (NVFP4 by delayed scaling, INT8
// exact per row); every output pointer is optional.  H % 16 == 0 and
// H <= kLnQuantMaxH; NVFP4 / INT8 outputs need H % 64 == 0.
constexpr int64_t kLnQuantMaxH = 4096;
struct LnQuantCall {
  const uint16_t* x;
  int64_t M, H, ldx;
  float eps;
  uint16_t* y;
  int64_t ldy;
  float* amax_out;
  float* row_amax_out;
  uint8_t* codes;
  uint8_t* sf;
  float* g_out;
  uint32_t* hist;
  float headroom;
  const uint8_t* nv_pred;
  uint8_t* planes;
  float* row_scale;
  const uint8_t* i8_pred;
  const uint8_t* pred;
  int* err;                  // device error word: set when a bounded row wait gives up
};
int launch_ln_quant(const LnQuantCall& c, int num_sms, cudaStream_t s);

// Block-scaled FP4 GEMM on tcgen05.  mode 0: W4A4 (A = NVFP4 codes + scales),
// mode 1: W4A8 (A = three E2M1 digit planes of the INT8 codes + row scales).
struct GemmCall {
  int mode;
  const uint8_t* a;          // codes [M, K/2] or planes [3][M][K/2]
  const uint8_t* a_sf;       // mode 0: swizzled scales of A
  const float* g_a;          // mode 0
  const float* row_scale;    // mode 1
  const uint8_t* w;          // [N, K/2]
  const uint8_t* w_sf;       // swizzled scales of W
  const float* g_w;
  int64_t M, N, K;
  const void* bias;          // bf16 [N] or null
  const void* residual;      // bf16 [M, ldr] or null
  int64_t ldr;
  int gelu;
  int out_bf16;
  void* y;
  int64_t ldy;
  const uint8_t* pred;
  int* err;                  // device error word
  // Quantizing epilogue (q_hist != null): the bf16 result is also encoded as
  // NVFP4 for the next layer by delayed scaling.  When q_codes is set and
  // q_pred is null or *q_pred != 0 the codes [M, N/2], swizzled scales and g
  // are written and y is not; otherwise y is written.  The history records
  // |y|'s amax either way (with q_codes null: an exact amax side output).
  uint8_t* q_codes;
  uint8_t* q_sf;
  float* q_g;
  uint32_t* q_hist;
  float q_headroom;
  const uint8_t* q_pred;
};
int launch_gemm_fp4(const GemmCall& c, int num_sms, cudaStream_t s);
// Test switch of the GEMM's abort path (see sixbit_debug_stall_gemm).
int set_gemm_stall(int on);
// Test switch of the staged producers' abort paths (see sixbit_debug_stall_staging).
int set_stage_stall(int on);

}  // namespace sixbit
