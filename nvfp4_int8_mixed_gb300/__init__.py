"""Python binding of the sixbit C ABI (include/sixbit.h) for GB300.

Thin argument marshalling over ctypes: torch supplies device memory and the
current stream; every step of the path runs in the library's CUDA kernels.
There is no fallback: if the library is missing or no CUDA device is present,
the calls raise.

Build the library first:  python -m nvfp4_int8_mixed_gb300.build
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib6bit.so")

OK, EINVAL, ESHAPE, EALIGN, ELAUNCH, EDEVICE = 0, -1, -2, -3, -4, -5
_ERR_NAMES = {EINVAL: "invalid argument", ESHAPE: "unsupported shape", EALIGN: "misaligned pointer or stride",
              ELAUNCH: "CUDA launch error", EDEVICE: "device wait gave up"}
F32, BF16 = 0, 1
EPI_GELU = 1

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_INT = ctypes.c_int
_F = ctypes.c_float

_SIGS = {
    "sixbit_version": ([], ctypes.c_char_p),
    "sixbit_sf_bytes": ([_I64, _I64], ctypes.c_size_t),
    "sixbit_workspace_size": ([_I64, _I64], ctypes.c_size_t),
    "sixbit_amax_bf16": ([_P, _I64, _I64, _I64, _P, _P, _P], _INT),
    "sixbit_quantize_act_nvfp4": ([_P, _I64, _I64, _I64, _P, _P, _P, _P, _P, _P, _P], _INT),
    "sixbit_quantize_weight_nvfp4": ([_P, _INT, _I64, _I64, _P, _P, _P, _P, _P], _INT),
    "sixbit_quantize_act_int8": ([_P, _I64, _I64, _I64, _P, _P, _P, _P, _P, _P], _INT),
    "sixbit_qlinear_w4a4": ([_P, _P, _P, _I64, _I64, _P, _P, _P, _I64, _P, _P, _I64, _INT, _INT, _P, _I64, _P, _P], _INT),
    "sixbit_qlinear_w4a8": ([_P, _P, _I64, _I64, _P, _P, _P, _I64, _P, _P, _I64, _INT, _INT, _P, _I64, _P, _P], _INT),
    "sixbit_block_gamma": ([_P, _P, _I64, _P, _P, _P, _P, _P, _P, _P], _INT),
    "sixbit_block_gamma_noalloc": ([_P, _P, _I64, _P, _P, _P, _P, _P, _P], _INT),
    "sixbit_dmpq_assign": ([_P, _P, _P, _P, _I32, _F, _P, _P, _P, _P], _INT),
    "sixbit_pair_stats": ([_P, _I32, _P, _I32, _I64, _P, _P, _P], _INT),
    "sixbit_tdc_decide_and_apply": ([_P, _P, _I64, _P, _F, _I32, _I32, _P, _P, _P, _P, _P, _I32, _P], _INT),
    "sixbit_layernorm_bf16": ([_P, _I64, _I64, _I64, _F, _P, _I64, _P, _P, _P, _P], _INT),
    "sixbit_mxcache_bytes": ([_I64], ctypes.c_size_t),
    "sixbit_block_gamma_mxcache": ([_P, _P, _I64, _P, _P, _P, _P, _P, _P, _P], _INT),
    "sixbit_tdc_decide_and_apply_mxcache": ([_P, _P, _I64, _P, _F, _I32, _I32, _P, _P, _P, _P, _P, _I32, _P],
                                            _INT),
    "sixbit_layernorm_quant": ([_P, _I64, _I64, _I64, _F, _P, _I64, _P, _P, _P, _P, _F, _P, _P, _P, _P, _P, _P],
                               _INT),
    "sixbit_qlinear_qout": ([_INT, _P, _P, _P, _P, _I64, _I64, _P, _P, _P, _I64, _P, _INT, _P, _I64, _P, _P, _P, _P,
                             _F, _P, _P, _P], _INT),
    "sixbit_debug_stall_gemm": ([_INT], _INT),
    "sixbit_debug_stall_staging": ([_INT], _INT),
    "sixbit_int8_digit_planes": ([_P, _I64, _I64, _I64, _P, _P], _INT),
    "sixbit_get_error": ([_P], _INT),
}

_lib = None


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"sixbit CUDA library not found at {LIB_PATH}; "
                               "build it with: python -m nvfp4_int8_mixed_gb300.build")
        L = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGS.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


class SixbitError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn} failed: {_ERR_NAMES.get(code, code)} ({code})")
        self.code = code


def _check(fn, rc):
    if rc != OK:
        raise SixbitError(fn, rc)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("sixbit works on CUDA tensors only")


def sf_bytes(rows: int, K: int) -> int:
    return int(lib().sixbit_sf_bytes(rows, K))


_ws_cache: dict = {}


def workspace(nbytes: int, device=None) -> torch.Tensor:
    """Zero-initialised scratch shared by calls on one device (grown on demand)."""
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)
    t = _ws_cache.get(dev)
    if t is None or t.numel() < nbytes:
        t = torch.zeros(max(nbytes, 1 << 16), dtype=torch.uint8, device=dev)
        _ws_cache[dev] = t
    return t


def _ws_for(n_elems: int):
    return workspace(int(lib().sixbit_workspace_size(n_elems, 1)))


# --------------------------------------------------------------- quantizers
def amax(x: torch.Tensor, tensor=True, rows=False):
    """a1: (tensor amax [1] or None, row amax [M] or None) of a bf16 [M, K] view."""
    _need_cuda(x)
    M, K = x.shape
    ta = torch.empty(1, dtype=torch.float32, device=x.device) if tensor else None
    ra = torch.empty(M, dtype=torch.float32, device=x.device) if rows else None
    _check("sixbit_amax_bf16", lib().sixbit_amax_bf16(_ptr(x), M, K, x.stride(0), _ptr(ta), _ptr(ra), _stream()))
    return ta, ra


def quantize_act_nvfp4(x: torch.Tensor, amax_in=None, pred=None, out=None):
    """a2: bf16 [M, K] (row stride may exceed K) -> (codes [M, K/2] u8, sf u8 (swizzled), g [1] f32)."""
    _need_cuda(x)
    M, K = x.shape
    if out is None:
        codes = torch.empty((M, K // 2), dtype=torch.uint8, device=x.device)
        sf = torch.empty(sf_bytes(M, K), dtype=torch.uint8, device=x.device)
        g = torch.empty(1, dtype=torch.float32, device=x.device)
    else:
        codes, sf, g = out
    ws = None if amax_in is not None else _ws_for(0)
    _check("sixbit_quantize_act_nvfp4",
           lib().sixbit_quantize_act_nvfp4(_ptr(x), M, K, x.stride(0), _ptr(amax_in), _ptr(codes), _ptr(sf), _ptr(g),
                                           _ptr(pred), _ptr(ws), _stream()))
    return codes, sf, g


def quantize_weight_nvfp4(w: torch.Tensor):
    """a4: f32 or bf16 [N, K] contiguous -> (codes, sf (swizzled), g)."""
    _need_cuda(w)
    w = w.contiguous()
    N, K = w.shape
    dt = {torch.float32: F32, torch.bfloat16: BF16}[w.dtype]
    codes = torch.empty((N, K // 2), dtype=torch.uint8, device=w.device)
    sf = torch.empty(sf_bytes(N, K), dtype=torch.uint8, device=w.device)
    g = torch.empty(1, dtype=torch.float32, device=w.device)
    _check("sixbit_quantize_weight_nvfp4",
           lib().sixbit_quantize_weight_nvfp4(_ptr(w), dt, N, K, _ptr(codes), _ptr(sf), _ptr(g), _ptr(_ws_for(0)),
                                              _stream()))
    return codes, sf, g


def quantize_act_int8(x: torch.Tensor, row_amax=None, want_q=True, want_planes=True, pred=None, out=None):
    """a3: bf16 [M, K] -> (q int8 [M, K] or None, planes u8 [3, M, K/2] or None, row_scale f32 [M])."""
    _need_cuda(x)
    M, K = x.shape
    if out is None:
        q = torch.empty((M, K), dtype=torch.int8, device=x.device) if want_q else None
        planes = torch.empty((3, M, K // 2), dtype=torch.uint8, device=x.device) if want_planes else None
        s = torch.empty(M, dtype=torch.float32, device=x.device)
    else:
        q, planes, s = out
    _check("sixbit_quantize_act_int8",
           lib().sixbit_quantize_act_int8(_ptr(x), M, K, x.stride(0), _ptr(row_amax), _ptr(q), _ptr(planes), _ptr(s),
                                          _ptr(pred), _stream()))
    return q, planes, s


# --------------------------------------------------------------- GEMMs
def int8_digit_planes(q: torch.Tensor, out=None):
    """Plain int8 codes [M, K] -> the W4A8 operand planes u8 [3, M, K/2] (exact digit split)."""
    _need_cuda(q)
    M, K = q.shape
    planes = torch.empty((3, M, K // 2), dtype=torch.uint8, device=q.device) if out is None else out
    _check("sixbit_int8_digit_planes",
           lib().sixbit_int8_digit_planes(_ptr(q), M, K, q.stride(0), _ptr(planes), _stream()))
    return planes


def _out(M, N, dtype, device, out):
    if out is not None:
        return out
    return torch.empty((M, N), dtype=dtype, device=device)


def qlinear_w4a4(a_codes, a_sf, g_a, w_codes, w_sf, g_w, bias=None, residual=None, gelu=False,
                 out_dtype=torch.bfloat16, out=None, pred=None):
    """a5: y [M, N] = W4A4 product with fused epilogue."""
    _need_cuda(a_codes, w_codes)
    M, K = a_codes.shape[0], a_codes.shape[1] * 2
    N = w_codes.shape[0]
    y = _out(M, N, out_dtype, a_codes.device, out)
    _check("sixbit_qlinear_w4a4",
           lib().sixbit_qlinear_w4a4(_ptr(a_codes), _ptr(a_sf), _ptr(g_a), M, K, _ptr(w_codes), _ptr(w_sf), _ptr(g_w),
                                     N, _ptr(bias), _ptr(residual), residual.stride(0) if residual is not None else 0,
                                     EPI_GELU if gelu else 0, BF16 if y.dtype == torch.bfloat16 else F32, _ptr(y),
                                     y.stride(0), _ptr(pred), _stream()))
    return y


def qlinear_w4a8(planes, row_scale, w_codes, w_sf, g_w, bias=None, residual=None, gelu=False,
                 out_dtype=torch.bfloat16, out=None, pred=None):
    """a6: y [M, N] = W4A8 product (INT8 activations as digit planes) with fused epilogue."""
    _need_cuda(planes, w_codes)
    M, K = planes.shape[1], planes.shape[2] * 2
    N = w_codes.shape[0]
    y = _out(M, N, out_dtype, planes.device, out)
    _check("sixbit_qlinear_w4a8",
           lib().sixbit_qlinear_w4a8(_ptr(planes), _ptr(row_scale), M, K, _ptr(w_codes), _ptr(w_sf), _ptr(g_w), N,
                                     _ptr(bias), _ptr(residual), residual.stride(0) if residual is not None else 0,
                                     EPI_GELU if gelu else 0, BF16 if y.dtype == torch.bfloat16 else F32, _ptr(y),
                                     y.stride(0), _ptr(pred), _stream()))
    return y


def amax_hist_value(h: torch.Tensor) -> torch.Tensor:
    """The float32 view of a history row's first word: the amax its producer's
    last call recorded (an amax_in for the quantizers)."""
    return h[0:1].view(torch.float32)


def amax_history(n: int = 1, device=None) -> torch.Tensor:
    """Zeroed delayed-scaling histories for n quantizing producers: uint32 [n, 4]
    (16-byte rows), handed to layernorm_quant / qlinear_qout one row per layer."""
    dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
    return torch.zeros((n, 4), dtype=torch.int32, device=dev)


def qlinear_qout(mode: str, a, w_codes, w_sf, g_w, q_codes, q_sf, q_g, amax_hist, a_sf=None, g_a=None,
                 row_scale=None, bias=None, gelu=False, headroom=2.0, y=None, q_pred=None, pred=None):
    """Linear layer whose epilogue quantizes its bf16 result to NVFP4 for the
    next layer by delayed scaling (y written instead when *q_pred == 0).
    mode "w4a4": a = codes [M, K/2] with a_sf, g_a; "w4a8": a = digit planes
    [3, M, K/2] with row_scale.  q_codes, q_sf, q_g all None: y is written
    and amax_hist[0] receives max |y| (float bits), an exact amax side output
    for the next quantizer (amax_hist_value(h) views it as float32).
    Returns y (bf16 [M, N]; allocated if None)."""
    w4a4 = mode == "w4a4"
    _need_cuda(a, w_codes)
    M, K = (a.shape[0], a.shape[1] * 2) if w4a4 else (a.shape[1], a.shape[2] * 2)
    N = w_codes.shape[0]
    y = _out(M, N, torch.bfloat16, a.device, y)
    _check("sixbit_qlinear_qout",
           lib().sixbit_qlinear_qout(0 if w4a4 else 1, _ptr(a), _ptr(a_sf), _ptr(g_a), _ptr(row_scale), M, K,
                                     _ptr(w_codes), _ptr(w_sf), _ptr(g_w), N, _ptr(bias), EPI_GELU if gelu else 0,
                                     _ptr(y), y.stride(0), _ptr(q_codes), _ptr(q_sf), _ptr(q_g), _ptr(amax_hist),
                                     float(headroom), _ptr(q_pred), _ptr(pred), _stream()))
    return y


# --------------------------------------------------------------- block ops
def mxcache(n: int, device=None) -> torch.Tensor:
    """A zeroed compressed update cache for n elements (uint8, codes then scales)."""
    nb = int(lib().sixbit_mxcache_bytes(n))
    if nb == 0:
        raise ValueError("the compressed cache needs n > 0 and n % 32 == 0")
    dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
    return torch.zeros(nb, dtype=torch.uint8, device=dev)


def block_gamma(xin, xout, delta=None, gamma_out=None, r2_out=None, tdc_state=None, computed=None, ws=None):
    """a7: Gamma (and Delta in place, r2, TDC counters). Returns (gamma [1], r2 [1]).
    delta: the bf16 update, or a uint8 compressed cache (mxcache).  ws: scratch
    of sixbit_workspace_size(n, 1) bytes, zeroed before its first use (default:
    the device's shared scratch; a pass running on another stream at the same
    time as other library calls needs its own)."""
    _need_cuda(xin, xout)
    n = xin.numel()
    dev = xin.device
    g = gamma_out if gamma_out is not None else torch.empty(1, dtype=torch.float32, device=dev)
    r2 = r2_out if r2_out is not None else torch.full((1,), float("nan"), dtype=torch.float32, device=dev)
    name = "sixbit_block_gamma_mxcache" if delta is not None and delta.dtype == torch.uint8 else "sixbit_block_gamma"
    _check(name, getattr(lib(), name)(_ptr(xin), _ptr(xout), n, _ptr(delta), _ptr(g), _ptr(r2), _ptr(tdc_state),
                                      _ptr(computed), _ptr(ws if ws is not None else _ws_for(n)), _stream()))
    return g, r2


def pair_stats(a, b, out=None):
    """Calibration diagnostic: float64 device tensor [4] = {sum (a-b)^2,
    sum b^2, sum a*b, sum a^2} over two same-size bf16/fp32 tensors."""
    _need_cuda(a, b)
    if a.numel() != b.numel():
        raise ValueError("pair_stats: size mismatch")
    dt = {torch.bfloat16: BF16, torch.float32: F32}
    if a.dtype not in dt or b.dtype not in dt:
        raise ValueError("pair_stats: bf16 or fp32 tensors")
    a, b = a.contiguous(), b.contiguous()
    n = a.numel()
    o = out if out is not None else torch.empty(4, dtype=torch.float64, device=a.device)
    _check("sixbit_pair_stats", lib().sixbit_pair_stats(_ptr(a), dt[a.dtype], _ptr(b), dt[b.dtype], n, _ptr(o),
                                                        _ptr(_ws_for(n)), _stream()))
    return o


def dmpq_assign(gamma, alpha, beta, layer_block, tau: float, step, use_nvfp4=None, gates=None):
    """a8: uint8 flags per layer (1 = NVFP4); optional gates [n_layers, 2]."""
    n = alpha.numel()
    f = use_nvfp4 if use_nvfp4 is not None else torch.empty(n, dtype=torch.uint8, device=alpha.device)
    _check("sixbit_dmpq_assign",
           lib().sixbit_dmpq_assign(_ptr(gamma), _ptr(alpha), _ptr(beta), _ptr(layer_block), n, float(tau), _ptr(step),
                                    _ptr(f), _ptr(gates), _stream()))
    return f


def tdc_decide_and_apply(xin, delta, r2, tau_tdc: float, max_skip: int, tdc_state, compute_out, out, gates=None,
                         refresh_every: int = 0, step=None):
    """a9: compute_out[0] = 1 if the block must run; on a skip out = in + Delta.
    refresh_every > 0 (with step, a device int32) forces a computed step every
    refresh_every steps.  delta: the bf16 update, or a uint8 compressed cache."""
    n = xin.numel()
    name = "sixbit_tdc_decide_and_apply_mxcache" if delta.dtype == torch.uint8 else "sixbit_tdc_decide_and_apply"
    _check(name, getattr(lib(), name)(_ptr(xin), _ptr(delta), n, _ptr(r2), float(tau_tdc), int(max_skip),
                                      int(refresh_every), _ptr(step), _ptr(tdc_state), _ptr(compute_out),
                                      _ptr(out), _ptr(gates), gates.numel() if gates is not None else 0,
                                      _stream()))
    return compute_out


def layernorm(x, eps=1e-5, out=None, amax_out=None, row_amax_out=None, pred=None):
    M, H = x.shape
    y = out if out is not None else torch.empty((M, H), dtype=torch.bfloat16, device=x.device)
    _check("sixbit_layernorm_bf16",
           lib().sixbit_layernorm_bf16(_ptr(x), M, H, x.stride(0), float(eps), _ptr(y), y.stride(0), _ptr(amax_out),
                                       _ptr(row_amax_out), _ptr(pred), _stream()))
    return y


def layernorm_quant(x, eps=1e-5, y=None, nvfp4=None, amax_hist=None, headroom=2.0, nv_pred=None, int8=None,
                    i8_pred=None, pred=None):
    """LayerNorm that quantizes its output for the next linear layer.
    nvfp4 = (codes [M, H/2], sf, g) by delayed scaling from amax_hist;
    int8 = (planes [3, M, H/2], row_scale [M]) exact per row; y bf16 [M, H]
    (optional).  Each quantized output is written when its gate is None or
    nonzero."""
    M, H = x.shape
    codes, sf, g = nvfp4 if nvfp4 is not None else (None, None, None)
    planes, rs = int8 if int8 is not None else (None, None)
    _check("sixbit_layernorm_quant",
           lib().sixbit_layernorm_quant(_ptr(x), M, H, x.stride(0), float(eps), _ptr(y),
                                        y.stride(0) if y is not None else 0, _ptr(codes), _ptr(sf), _ptr(g),
                                        _ptr(amax_hist), float(headroom), _ptr(nv_pred), _ptr(planes), _ptr(rs),
                                        _ptr(i8_pred), _ptr(pred), _stream()))
    return y


def get_error():
    """Synchronize the current stream and raise if a device wait gave up."""
    _check("sixbit_get_error", lib().sixbit_get_error(_stream()))
