"""The C-ABI library loads without a GPU, exports every symbol the header
declares, and rejects bad arguments on the host before any CUDA call."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sixbit.h")


@pytest.fixture(scope="module")
def lib():
    import nvfp4_int8_mixed_gb300 as sb
    if not os.path.exists(sb.LIB_PATH):
        from nvfp4_int8_mixed_gb300 import build
        build.build()
    return sb.lib()


def declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(sixbit_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = declared()
    assert len(names) >= 14
    for n in names:
        assert hasattr(lib, n), n


def test_binding_covers_header():
    import nvfp4_int8_mixed_gb300 as sb
    assert set(declared()) == set(sb._SIGS)


def _prototypes():
    """{name: [argument type text, ...]} of every declaration in the header."""
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    out = {}
    for name, args in re.findall(r"\b(sixbit_[a-z0-9_]+)\s*\(([^)]*)\)\s*;", src):
        args = " ".join(args.split())
        out[name] = [] if args in ("", "void") else [a.strip() for a in args.split(",")]
    return out


def _kind(decl):
    """ctypes type an argument declaration must be marshalled as."""
    if "*" in decl or decl.startswith("sixbit_stream_t"):
        return ctypes.c_void_p
    for ctype, kind in (("int64_t", ctypes.c_int64), ("int32_t", ctypes.c_int32), ("float", ctypes.c_float),
                        ("int", ctypes.c_int)):
        if re.match(rf"(const\s+)?{ctype}\b", decl):
            return kind
    raise AssertionError(f"unclassified argument: {decl}")


def test_binding_signatures_match_header():
    """Every ctypes signature has the header's argument count and kinds, in
    order (a drifted signature would only misbehave on a GPU)."""
    import nvfp4_int8_mixed_gb300 as sb
    protos = _prototypes()
    assert set(protos) == set(sb._SIGS)
    for name, decls in protos.items():
        want = [_kind(d) for d in decls]
        got = sb._SIGS[name][0]
        assert len(got) == len(want), (name, len(got), len(want))
        for i, (g, w) in enumerate(zip(got, want)):
            assert g is w, (name, i, decls[i], g, w)


def test_host_helpers(lib):
    assert lib.sixbit_version().startswith(b"sixbit")
    assert lib.sixbit_sf_bytes(256, 256) == 256 * 16
    assert lib.sixbit_sf_bytes(200, 1920) == 256 * 120        # rows padded to 128
    assert lib.sixbit_sf_bytes(1, 64) == 128 * 4
    # Gamma pass scratch: a 256-byte header, then 4 doubles for each of the
    # 256 reduction chains, whatever the size
    assert lib.sixbit_workspace_size(17776, 1920) == 256 + 256 * 4 * 8
    assert lib.sixbit_workspace_size(1, 64) == 8448
    assert lib.sixbit_workspace_size(1 << 27, 1) == 8448


def test_argument_errors_before_launch(lib):
    import nvfp4_int8_mixed_gb300 as sb
    P = ctypes.c_void_p
    fake = P(1 << 20)       # never dereferenced: checks fail first
    # null input
    assert lib.sixbit_quantize_act_nvfp4(None, 16, 64, 64, fake, fake, fake, fake, None, None, None) == sb.EINVAL
    # K not a multiple of 64
    assert lib.sixbit_quantize_act_nvfp4(fake, 16, 96, 96, fake, fake, fake, fake, None, None, None) == sb.ESHAPE
    # misaligned codes pointer
    assert lib.sixbit_quantize_act_nvfp4(fake, 16, 64, 64, fake, P((1 << 20) + 4), fake, fake, None, None,
                                         None) == sb.EALIGN
    # INT8: neither q nor planes
    assert lib.sixbit_quantize_act_int8(fake, 4, 64, 64, None, None, None, fake, None, None) == sb.EINVAL
    assert lib.sixbit_quantize_act_int8(fake, 4, 32768, 32768, None, fake, None, fake, None, None) == sb.ESHAPE
    # GEMM: N not a multiple of 16, bad dtype, ldy < N
    args = lambda N, dt, ldy: (fake, fake, fake, 128, 256, fake, fake, fake, N, None, None, 0, 0, dt, fake, ldy,
                               None, None)
    assert lib.sixbit_qlinear_w4a4(*args(40, sb.BF16, 40)) == sb.ESHAPE
    assert lib.sixbit_qlinear_w4a4(*args(64, 7, 64)) == sb.EINVAL
    assert lib.sixbit_qlinear_w4a4(*args(64, sb.BF16, 32)) == sb.ESHAPE
    assert lib.sixbit_qlinear_w4a8(fake, None, 128, 256, fake, fake, fake, 64, None, None, 0, 0, sb.F32, fake, 64,
                                   None, None) == sb.EINVAL
    assert lib.sixbit_block_gamma(fake, fake, 0, None, fake, None, None, None, fake, None) == sb.EINVAL
    assert lib.sixbit_dmpq_assign(fake, fake, fake, fake, 0, ctypes.c_float(0.1), fake, fake, None, None) == sb.EINVAL
    assert lib.sixbit_tdc_decide_and_apply(fake, fake, 16, fake, ctypes.c_float(0.05), 1, 0, None, None, fake, fake,
                                           None, 0, None) == sb.EINVAL
    # a periodic refresh needs the step counter
    assert lib.sixbit_tdc_decide_and_apply(fake, fake, 16, fake, ctypes.c_float(0.05), 1, 3, None, fake, fake, fake,
                                           None, 0, None) == sb.EINVAL
    assert lib.sixbit_layernorm_bf16(fake, 4, 20, 20, ctypes.c_float(1e-5), fake, 20, None, None, None,
                                     None) == sb.ESHAPE


def test_mxcache_argument_errors(lib):
    import nvfp4_int8_mixed_gb300 as sb
    P = ctypes.c_void_p
    fake = P(1 << 20)
    assert lib.sixbit_mxcache_bytes(64) == 66 and lib.sixbit_mxcache_bytes(33) == 0 and lib.sixbit_mxcache_bytes(0) == 0
    assert lib.sixbit_block_gamma_mxcache(fake, fake, 48, fake, fake, None, None, None, fake, None) == sb.ESHAPE
    assert lib.sixbit_block_gamma_mxcache(fake, fake, 64, P((1 << 20) + 8), fake, None, None, None, fake,
                                          None) == sb.EALIGN
    assert lib.sixbit_tdc_decide_and_apply_mxcache(fake, None, 64, fake, ctypes.c_float(0.05), 1, 0, None, fake,
                                                   fake, fake, None, 0, None) == sb.EINVAL
    assert lib.sixbit_tdc_decide_and_apply_mxcache(fake, fake, 40, fake, ctypes.c_float(0.05), 1, 0, None, fake,
                                                   fake, fake, None, 0, None) == sb.ESHAPE


def test_quantizing_producer_argument_errors(lib):
    import nvfp4_int8_mixed_gb300 as sb
    P = ctypes.c_void_p
    fake = P(1 << 20)
    f = ctypes.c_float
    eps = f(1e-5)

    def ln(M=4, H=128, y=fake, codes=fake, sf=fake, g=fake, hist=fake, head=2.0, planes=None, rs=None):
        return lib.sixbit_layernorm_quant(fake, M, H, H, eps, y, H, codes, sf, g, hist, f(head), None, planes, rs,
                                          None, None, None)
    assert ln(hist=None) == sb.EINVAL                 # NVFP4 output needs a history
    assert ln(head=0.0) == sb.EINVAL
    assert ln(head=float("nan")) == sb.EINVAL
    assert ln(y=None, codes=None) == sb.EINVAL        # no output at all
    assert ln(codes=None, planes=fake) == sb.EINVAL   # planes without row scales
    assert ln(H=96) == sb.ESHAPE                      # quantized outputs need H % 64 == 0
    assert ln(H=8192) == sb.ESHAPE                    # row must fit the registers
    assert ln(hist=P((1 << 20) + 4)) == sb.EALIGN

    def qo(mode=0, N=128, hist=fake, head=2.0, a_sf=fake, rs=None):
        return lib.sixbit_qlinear_qout(mode, fake, a_sf, fake, rs, 128, 256, fake, fake, fake, N, None, 0, fake, N,
                                       fake, fake, fake, hist, f(head), None, None, None)
    assert qo(mode=7) == sb.EINVAL
    assert qo(N=80) == sb.ESHAPE                      # the next layer's K: N % 64 == 0
    assert qo(hist=None) == sb.EINVAL
    assert qo(head=-1.0) == sb.EINVAL
    assert qo(mode=1, a_sf=None) == sb.EINVAL         # W4A8 needs the row scales
    # the NVFP4 outputs come together (all three, or none for the amax side output)
    assert lib.sixbit_qlinear_qout(0, fake, fake, fake, None, 128, 256, fake, fake, fake, 128, None, 0, fake, 128,
                                   fake, None, fake, fake, f(2.0), None, None, None) == sb.EINVAL
    assert qo(hist=P((1 << 20) + 8)) == sb.EALIGN


def test_empty_row_count_is_a_no_op(lib):
    """Calls over M rows return SIXBIT_OK for M == 0 before any check or
    device call: an empty tensor's NULL data pointer is accepted, so these
    run on a machine without a GPU."""
    import nvfp4_int8_mixed_gb300 as sb
    f = ctypes.c_float
    assert lib.sixbit_amax_bf16(None, 0, 64, 64, None, None, None) == sb.OK
    assert lib.sixbit_quantize_act_nvfp4(None, 0, 64, 64, None, None, None, None, None, None, None) == sb.OK
    assert lib.sixbit_quantize_act_int8(None, 0, 64, 64, None, None, None, None, None, None) == sb.OK
    assert lib.sixbit_int8_digit_planes(None, 0, 64, 64, None, None) == sb.OK
    assert lib.sixbit_qlinear_w4a4(None, None, None, 0, 256, None, None, None, 128, None, None, 0, 0, sb.BF16, None,
                                   128, None, None) == sb.OK
    assert lib.sixbit_qlinear_w4a8(None, None, 0, 256, None, None, None, 128, None, None, 0, 0, sb.BF16, None, 128,
                                   None, None) == sb.OK
    assert lib.sixbit_qlinear_qout(0, None, None, None, None, 0, 256, None, None, None, 128, None, 0, None, 128, None,
                                   None, None, None, f(2.0), None, None, None) == sb.OK
    assert lib.sixbit_layernorm_bf16(None, 0, 128, 128, f(1e-5), None, 128, None, None, None, None) == sb.OK
    assert lib.sixbit_layernorm_quant(None, 0, 128, 128, f(1e-5), None, 128, None, None, None, None, f(2.0), None,
                                      None, None, None, None, None) == sb.OK
    # a negative row count is still an error
    assert lib.sixbit_amax_bf16(None, -1, 64, 64, None, None, None) == sb.EINVAL
    # the element-count calls have no empty form: n = 0 is rejected
    assert lib.sixbit_block_gamma(None, None, 0, None, None, None, None, None, None, None) == sb.EINVAL
    assert lib.sixbit_pair_stats(None, 0, None, 0, 0, None, None, None) == sb.EINVAL
