// C ABI of the sixbit library: argument checks on the host, then launches.
// Nothing here allocates device memory.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/sixbit.h"
#include "common.cuh"
#include "kernels.h"

using namespace sixbit;

// Device error word, set by bounded waits that gave up (see sixbit_get_error).
__device__ int g_sixbit_error = 0;

namespace {

constexpr int kMaxDevices = 64;
struct DeviceInfo {
  int num_sms;
  int* err;
};
std::mutex g_dev_mu;
DeviceInfo g_dev[kMaxDevices] = {};

// Per-device setup with the device current: SM count and the device address
// of the error word (host code must not take the address of a __device__
// variable directly).  Filled once per device under a lock, so host threads
// calling the library at the same time see a complete entry.
int device_setup(int* num_sms, int** err) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return kELaunch;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (d.num_sms == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return kELaunch;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_sixbit_error) != cudaSuccess) return kELaunch;
    d.err = static_cast<int*>(p);
    d.num_sms = n;
  }
  *num_sms = d.num_sms;
  if (err) *err = d.err;
  return kOk;
}

// Scratch layout: [0, 4) CTA counter of the Gamma pass (and of the pair
// statistics), [64, 68) tensor amax, [256, 8448) the 4 float64 sums of each
// of the 256 reduction chains of those passes.
constexpr size_t kWsAmaxOffset = 64;

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline cudaStream_t cs(sixbit_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

}  // namespace

extern "C" {

const char* sixbit_version(void) { return "sixbit 0.1 (sm_103a)"; }

size_t sixbit_sf_bytes(int64_t rows, int64_t K) {
  if (rows < 0 || K < 0) return 0;
  const int64_t kc4 = cdiv(K / 16, 4) * 4;
  return size_t(cdiv(rows, 128) * 128 * kc4);
}

size_t sixbit_workspace_size(int64_t M, int64_t K) {
  if (M < 0 || K < 0) return 0;
  const size_t g = gamma_ws_bytes(M * K);
  return g < 512 ? 512 : g;
}

int sixbit_amax_bf16(const void* x, int64_t M, int64_t K, int64_t ldx, float* amax_out, float* row_amax_out,
                     sixbit_stream_t stream) {
  if (M == 0) return kOk;                 // empty: nothing to do, pointers unused
  if (!x || (!amax_out && !row_amax_out) || M < 0 || K < 0 || ldx < K) return kEInval;
  if (K % 8 != 0 || ldx % 8 != 0) return kEShape;
  if (!aligned16(x)) return kEAlign;
  int sms;
  if (device_setup(&sms, nullptr) != kOk) return kELaunch;
  return launch_amax(x, SIXBIT_BF16, M, K, ldx, amax_out, row_amax_out, nullptr, sms, cs(stream));
}

int sixbit_quantize_act_nvfp4(const void* x, int64_t M, int64_t K, int64_t ldx, const float* amax_in, uint8_t* codes,
                              uint8_t* sf, float* g_out, const uint8_t* pred, void* ws, sixbit_stream_t stream) {
  if (M == 0) return kOk;                 // empty: nothing to do, pointers unused
  if (!x || !codes || !sf || !g_out || M < 0 || K <= 0 || ldx < K) return kEInval;
  if (!amax_in && !ws) return kEInval;
  if (K % 64 != 0 || ldx % 8 != 0) return kEShape;
  if (!aligned16(x) || !aligned16(codes) || !aligned16(sf)) return kEAlign;
  int sms;
  if (device_setup(&sms, nullptr) != kOk) return kELaunch;
  const float* amax = amax_in;
  if (!amax) {
    float* wamax = reinterpret_cast<float*>(static_cast<char*>(ws) + kWsAmaxOffset);
    int rc = launch_amax(x, SIXBIT_BF16, M, K, ldx, wamax, nullptr, pred, sms, cs(stream));
    if (rc != kOk) return rc;
    amax = wamax;
  }
  return launch_nvfp4_quant(x, SIXBIT_BF16, M, K, ldx, amax, codes, sf, g_out, pred, sms, cs(stream));
}

int sixbit_quantize_weight_nvfp4(const void* w, int dtype, int64_t N, int64_t K, uint8_t* codes, uint8_t* sf,
                                 float* g_out, void* ws, sixbit_stream_t stream) {
  if (!w || !codes || !sf || !g_out || !ws || N <= 0 || K <= 0) return kEInval;
  if (dtype != SIXBIT_F32 && dtype != SIXBIT_BF16) return kEInval;
  if (K % 64 != 0) return kEShape;
  if (!aligned16(w) || !aligned16(codes) || !aligned16(sf)) return kEAlign;
  int sms;
  if (device_setup(&sms, nullptr) != kOk) return kELaunch;
  float* wamax = reinterpret_cast<float*>(static_cast<char*>(ws) + kWsAmaxOffset);
  int rc = launch_amax(w, dtype, N, K, K, wamax, nullptr, nullptr, sms, cs(stream));
  if (rc != kOk) return rc;
  return launch_nvfp4_quant(w, dtype, N, K, K, wamax, codes, sf, g_out, nullptr, sms, cs(stream));
}

int sixbit_quantize_act_int8(const void* x, int64_t M, int64_t K, int64_t ldx, const float* row_amax_in, int8_t* q,
                             uint8_t* planes, float* row_scale, const uint8_t* pred, sixbit_stream_t stream) {
  if (M == 0) return kOk;                 // empty: nothing to do, pointers unused
  if (!x || !row_scale || (!q && !planes) || M < 0 || K <= 0 || ldx < K) return kEInval;
  if (K % 64 != 0 || K > 16384 || ldx % 8 != 0) return kEShape;
  if (!aligned16(x) || (q && !aligned16(q)) || (planes && !aligned16(planes))) return kEAlign;
  int sms;
  if (device_setup(&sms, nullptr) != kOk) return kELaunch;
  return launch_int8_quant(x, M, K, ldx, row_amax_in, q, planes, row_scale, pred, sms, cs(stream));
}

int sixbit_int8_digit_planes(const int8_t* q, int64_t M, int64_t K, int64_t ldq, uint8_t* planes,
                             sixbit_stream_t stream) {
  if (M == 0) return kOk;                 // empty: nothing to do, pointers unused
  if (!q || !planes || M < 0 || K <= 0 || ldq < K) return kEInval;
  if (K % 64 != 0 || ldq % 16 != 0) return kEShape;
  if (!aligned16(q) || !aligned16(planes)) return kEAlign;
  int sms;
  if (device_setup(&sms, nullptr) != kOk) return kELaunch;
  return launch_int8_planes(q, M, K, ldq, planes, sms, cs(stream));
}

static int check_gemm(const uint8_t* a, const uint8_t* w, const uint8_t* w_sf, const float* g_w, int64_t M, int64_t K,
                      int64_t N, const void* bias, const void* residual, int64_t ldr, int out_dtype, void* y,
                      int64_t ldy) {
  if (!a || !w || !w_sf || !g_w || !y || M < 0 || K <= 0 || N <= 0) return kEInval;
  if (out_dtype != SIXBIT_F32 && out_dtype != SIXBIT_BF16) return kEInval;
  if (K % 64 != 0 || N % 16 != 0 || ldy < N || (residual && ldr < N)) return kEShape;
  if (M > (int64_t(1) << 30) || N > (int64_t(1) << 30) || K > (int64_t(1) << 20)) return kEShape;
  if (!aligned16(a) || !aligned16(w) || !aligned16(w_sf) || !aligned16(y)) return kEAlign;
  if ((out_dtype == SIXBIT_F32 ? ldy % 4 : ldy % 8) != 0) return kEAlign;
  if (bias && !aligned16(bias)) return kEAlign;
  if (residual && (!aligned16(residual) || ldr % 8 != 0)) return kEAlign;
  return kOk;
}

int sixbit_qlinear_w4a4(const uint8_t* a_codes, const uint8_t* a_sf, const float* g_a, int64_t M, int64_t K,
                        const uint8_t* w_codes, const uint8_t* w_sf, const float* g_w, int64_t N, const void* bias,
                        const void* residual, int64_t ldr, int epi, int out_dtype, void* y, int64_t ldy,
                        const uint8_t* pred, sixbit_stream_t stream) {
  if (M == 0) return kOk;                 // empty: nothing to do, pointers unused
  int rc = check_gemm(a_codes, w_codes, w_sf, g_w, M, K, N, bias, residual, ldr, out_dtype, y, ldy);
  if (rc != kOk) return rc;
  if (!a_sf || !g_a) return kEInval;
  if (!aligned16(a_sf)) return kEAlign;
  int sms;
  int* err;
  if (device_setup(&sms, &err) != kOk) return kELaunch;
  GemmCall c{0, a_codes, a_sf, g_a, nullptr, w_codes, w_sf, g_w, M, N, K, bias, residual, ldr,
             (epi & SIXBIT_EPI_GELU) ? 1 : 0, out_dtype == SIXBIT_BF16 ? 1 : 0, y, ldy, pred, err};
  return launch_gemm_fp4(c, sms, cs(stream));
}

int sixbit_qlinear_w4a8(const uint8_t* a_planes, const float* row_scale, int64_t M, int64_t K, const uint8_t* w_codes,
                        const uint8_t* w_sf, const float* g_w, int64_t N, const void* bias, const void* residual,
                        int64_t ldr, int epi, int out_dtype, void* y, int64_t ldy, const uint8_t* pred,
                        sixbit_stream_t stream) {
  if (M == 0) return kOk;                 // empty: nothing to do, pointers unused
  int rc = check_gemm(a_planes, w_codes, w_sf, g_w, M, K, N, bias, residual, ldr, out_dtype, y, ldy);
  if (rc != kOk) return rc;
  if (!row_scale) return kEInval;
  int sms;
  int* err;
  if (device_setup(&sms, &err) != kOk) return kELaunch;
  GemmCall c{1, a_planes, nullptr, nullptr, row_scale, w_codes, w_sf, g_w, M, N, K, bias, residual, ldr,
             (epi & SIXBIT_EPI_GELU) ? 1 : 0, out_dtype == SIXBIT_BF16 ? 1 : 0, y, ldy, pred, err};
  return launch_gemm_fp4(c, sms, cs(stream));
}

int sixbit_qlinear_qout(int mode, const uint8_t* a, const uint8_t* a_sf, const float* g_a, const float* row_scale,
                        int64_t M, int64_t K, const uint8_t* w_codes, const uint8_t* w_sf, const float* g_w, int64_t N,
                        const void* bias, int epi, void* y, int64_t ldy, uint8_t* q_codes, uint8_t* q_sf, float* q_g,
                        uint32_t* amax_hist, float headroom, const uint8_t* q_pred, const uint8_t* pred,
                        sixbit_stream_t stream) {
  if (M == 0) return kOk;                 // empty: nothing to do, pointers unused
  if (mode != SIXBIT_QOUT_W4A4 && mode != SIXBIT_QOUT_W4A8) return kEInval;
  int rc = check_gemm(a, w_codes, w_sf, g_w, M, K, N, bias, nullptr, 0, SIXBIT_BF16, y, ldy);
  if (rc != kOk) return rc;
  if (mode == SIXBIT_QOUT_W4A4 ? (!a_sf || !g_a) : !row_scale) return kEInval;
  const bool q_any = q_codes || q_sf || q_g;
  if (q_any && !(q_codes && q_sf && q_g)) return kEInval;        // the NVFP4 outputs come together
  if (!amax_hist || !(headroom > 0.f) || headroom > 3.0e38f) return kEInval;
  if (q_any && N % 64 != 0) return kEShape;
  if ((a_sf && !aligned16(a_sf)) || (q_any && (!aligned16(q_codes) || !aligned16(q_sf))) || !aligned16(amax_hist))
    return kEAlign;
  int sms;
  int* err;
  if (device_setup(&sms, &err) != kOk) return kELaunch;
  GemmCall c{mode == SIXBIT_QOUT_W4A4 ? 0 : 1, a, mode == SIXBIT_QOUT_W4A4 ? a_sf : nullptr,
             mode == SIXBIT_QOUT_W4A4 ? g_a : nullptr, mode == SIXBIT_QOUT_W4A4 ? nullptr : row_scale, w_codes, w_sf,
             g_w, M, N, K, bias, nullptr, 0, (epi & SIXBIT_EPI_GELU) ? 1 : 0, 1, y, ldy, pred, err,
             q_codes, q_sf, q_g, amax_hist, headroom, q_pred};
  return launch_gemm_fp4(c, sms, cs(stream));
}

int sixbit_block_gamma(const void* in, const void* out, int64_t n, void* delta, float* gamma_out, float* r2_out,
                       int32_t* tdc_state, const uint8_t* computed, void* ws, sixbit_stream_t stream) {
  if (!in || !out || !gamma_out || !ws || n <= 0) return kEInval;
  if (n > (int64_t(1) << 40)) return kEShape;
  if (!aligned16(in) || !aligned16(out) || (delta && !aligned16(delta)) || !aligned16(ws)) return kEAlign;
  int sms;
  int* err;
  if (device_setup(&sms, &err) != kOk) return kELaunch;
  return launch_block_gamma(in, out, n, delta, gamma_out, r2_out, tdc_state, computed, ws, err, cs(stream));
}

int sixbit_block_gamma_noalloc(const void* in, const void* out, int64_t n, void* delta, float* gamma_out,
                               float* r2_out, int32_t* tdc_state, const uint8_t* computed, sixbit_stream_t stream) {
  if (!in || !out || !gamma_out || n <= 0) return kEInval;
  if (n > block_gamma_noalloc_max_elems()) return kEShape;
  if (!aligned16(in) || !aligned16(out) || (delta && !aligned16(delta))) return kEAlign;
  int sms;
  int* err;
  if (device_setup(&sms, &err) != kOk) return kELaunch;
  return launch_block_gamma_noalloc(in, out, n, delta, gamma_out, r2_out, tdc_state, computed, err, cs(stream));
}

int sixbit_pair_stats(const void* a, int a_dtype, const void* b, int b_dtype, int64_t n, double* out, void* ws,
                      sixbit_stream_t stream) {
  if (!a || !b || !out || !ws || n <= 0) return kEInval;
  if ((a_dtype != SIXBIT_BF16 && a_dtype != SIXBIT_F32) || (b_dtype != SIXBIT_BF16 && b_dtype != SIXBIT_F32))
    return kEInval;
  if (n % 8 != 0) return kEShape;
  if (!aligned16(a) || !aligned16(b) || !aligned16(ws) || (reinterpret_cast<uintptr_t>(out) & 7u)) return kEAlign;
  int sms;
  if (device_setup(&sms, nullptr) != kOk) return kELaunch;
  return launch_pair_stats(a, a_dtype == SIXBIT_F32, b, b_dtype == SIXBIT_F32, n, out, ws, cs(stream));
}

int sixbit_dmpq_assign(const float* gamma, const float* alpha, const float* beta, const int32_t* layer_block,
                       int32_t n_layers, float tau, const int32_t* step, uint8_t* use_nvfp4, uint8_t* gates,
                       sixbit_stream_t stream) {
  if (!gamma || !alpha || !beta || !layer_block || !step || (!use_nvfp4 && !gates) || n_layers <= 0) return kEInval;
  return launch_dmpq(gamma, alpha, beta, layer_block, n_layers, tau, step, use_nvfp4, gates, cs(stream));
}

int sixbit_tdc_decide_and_apply(const void* in, const void* delta, int64_t n, const float* r2, float tau_tdc,
                                int32_t max_skip, int32_t refresh_every, const int32_t* step,
                                const int32_t* tdc_state, uint8_t* compute_out, void* out, uint8_t* gates,
                                int32_t n_gates, sixbit_stream_t stream) {
  if (!in || !delta || !r2 || !tdc_state || !compute_out || !out || n <= 0 || (gates && n_gates < 0)) return kEInval;
  if (refresh_every < 0 || (refresh_every > 0 && !step)) return kEInval;
  if (!aligned16(in) || !aligned16(delta) || !aligned16(out)) return kEAlign;
  int sms;
  if (device_setup(&sms, nullptr) != kOk) return kELaunch;
  const float tau2 = tau_tdc * tau_tdc;   // float32 product, round to nearest
  return launch_tdc(in, delta, n, r2, tau2, max_skip, refresh_every, step, tdc_state, compute_out, out, gates,
                    gates ? n_gates : 0, sms, cs(stream));
}

size_t sixbit_mxcache_bytes(int64_t n) {
  if (n <= 0 || n % 32 != 0) return 0;
  return size_t(n + n / 32);
}

int sixbit_block_gamma_mxcache(const void* in, const void* out, int64_t n, void* cache, float* gamma_out,
                               float* r2_out, int32_t* tdc_state, const uint8_t* computed, void* ws,
                               sixbit_stream_t stream) {
  if (!in || !out || !gamma_out || !ws || n <= 0) return kEInval;
  if (n % 32 != 0 || n > (int64_t(1) << 40)) return kEShape;
  if (!aligned16(in) || !aligned16(out) || (cache && !aligned16(cache)) || !aligned16(ws)) return kEAlign;
  int sms;
  int* err;
  if (device_setup(&sms, &err) != kOk) return kELaunch;
  return launch_block_gamma_mx(in, out, n, cache, gamma_out, r2_out, tdc_state, computed, ws, err, cs(stream));
}

int sixbit_tdc_decide_and_apply_mxcache(const void* in, const void* cache, int64_t n, const float* r2, float tau_tdc,
                                        int32_t max_skip, int32_t refresh_every, const int32_t* step,
                                        const int32_t* tdc_state, uint8_t* compute_out, void* out, uint8_t* gates,
                                        int32_t n_gates, sixbit_stream_t stream) {
  if (!in || !cache || !r2 || !tdc_state || !compute_out || !out || n <= 0 || (gates && n_gates < 0)) return kEInval;
  if (refresh_every < 0 || (refresh_every > 0 && !step)) return kEInval;
  if (n % 32 != 0) return kEShape;
  if (!aligned16(in) || !aligned16(cache) || !aligned16(out)) return kEAlign;
  int sms;
  if (device_setup(&sms, nullptr) != kOk) return kELaunch;
  const float tau2 = tau_tdc * tau_tdc;   // float32 product, round to nearest
  return launch_tdc_mx(in, cache, n, r2, tau2, max_skip, refresh_every, step, tdc_state, compute_out, out, gates,
                       gates ? n_gates : 0, sms, cs(stream));
}

int sixbit_layernorm_bf16(const void* x, int64_t M, int64_t H, int64_t ldx, float eps, void* y, int64_t ldy,
                          float* amax_out, float* row_amax_out, const uint8_t* pred, sixbit_stream_t stream) {
  if (M == 0) return kOk;                 // empty: nothing to do, pointers unused
  if (!x || !y || M < 0 || H <= 0 || ldx < H || ldy < H) return kEInval;
  if (H % 8 != 0 || ldx % 8 != 0 || ldy % 8 != 0) return kEShape;
  if (!aligned16(x) || !aligned16(y)) return kEAlign;
  int sms;
  int* err;
  if (device_setup(&sms, &err) != kOk) return kELaunch;
  return launch_layernorm(x, M, H, ldx, eps, y, ldy, amax_out, row_amax_out, pred, err, sms, cs(stream));
}

int sixbit_layernorm_quant(const void* x, int64_t M, int64_t H, int64_t ldx, float eps, void* y, int64_t ldy,
                           uint8_t* codes, uint8_t* sf, float* g_out, uint32_t* amax_hist, float headroom,
                           const uint8_t* nv_pred, uint8_t* planes, float* row_scale, const uint8_t* i8_pred,
                           const uint8_t* pred, sixbit_stream_t stream) {
  if (M == 0) return kOk;                 // empty: nothing to do, pointers unused
  if (!x || M < 0 || H <= 0 || ldx < H || (y && ldy < H)) return kEInval;
  if (!y && !codes && !planes) return kEInval;
  if (codes && (!sf || !g_out || !amax_hist)) return kEInval;
  if (planes && !row_scale) return kEInval;
  if (amax_hist && (!(headroom > 0.f) || headroom > 3.0e38f)) return kEInval;
  if (H % 16 != 0 || H > kLnQuantMaxH || ldx % 8 != 0 || (y && ldy % 8 != 0)) return kEShape;
  if ((codes || planes) && H % 64 != 0) return kEShape;
  if (M > (int64_t(1) << 30)) return kEShape;
  if (!aligned16(x) || (y && !aligned16(y)) || (codes && (!aligned16(codes) || !aligned16(sf))) ||
      (planes && !aligned16(planes)) || (amax_hist && !aligned16(amax_hist)))
    return kEAlign;
  int sms;
  int* err;
  if (device_setup(&sms, &err) != kOk) return kELaunch;
  LnQuantCall c = {};
  c.x = static_cast<const uint16_t*>(x); c.M = M; c.H = H; c.ldx = ldx; c.eps = eps;
  c.y = static_cast<uint16_t*>(y); c.ldy = ldy;
  c.codes = codes; c.sf = sf; c.g_out = g_out; c.hist = amax_hist; c.headroom = headroom; c.nv_pred = nv_pred;
  c.planes = planes; c.row_scale = row_scale; c.i8_pred = i8_pred; c.pred = pred; c.err = err;
  return launch_ln_quant(c, sms, cs(stream));
}

int sixbit_debug_stall_gemm(int on) {
  int sms;
  if (device_setup(&sms, nullptr) != kOk) return kELaunch;
  return set_gemm_stall(on ? 1 : 0);
}

int sixbit_debug_stall_staging(int on) {
  int sms;
  if (device_setup(&sms, nullptr) != kOk) return kELaunch;
  return set_stage_stall(on ? 1 : 0);
}

int sixbit_get_error(sixbit_stream_t stream) {
  if (cudaStreamSynchronize(cs(stream)) != cudaSuccess) return kELaunch;
  int sms;
  int* err;
  if (device_setup(&sms, &err) != kOk) return kELaunch;
  int v = 0;
  if (cudaMemcpy(&v, err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return kELaunch;
  if (v != 0) {
    const int zero = 0;
    cudaMemcpy(err, &zero, sizeof(int), cudaMemcpyHostToDevice);
    return kEDevice;
  }
  return kOk;
}

}  // extern "C"
