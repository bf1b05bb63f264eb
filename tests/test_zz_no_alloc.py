"""The scratch-free Gamma pass (sixbit_block_gamma_noalloc) against the
regular one (sixbit_block_gamma), through the C ABI.

The variant exists for callers that cannot give the library scratch memory
(device memory fully planned by another allocator, or code where allocating
is not allowed); it keeps its scratch in a fixed array inside the library.
Two calls in a row check that the array's leftover contents from one call do
not leak into the next.
"""
import ctypes

import numpy as np
import pytest
import torch

import synthetic
from tests.helpers import dev_bf16, host, host_bf16_bits

pytestmark = pytest.mark.gpu


def _call(fn, *args):
    import nvfp4_int8_mixed_gb300 as sb
    rc = getattr(sb.lib(), fn)(*args)
    assert rc == sb.OK, (fn, rc)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("trim", [0, 3])
def test_noalloc_matches_workspace_version_on_two_calls(trim):
    import nvfp4_int8_mixed_gb300 as sb
    M, H = 3000, 1920                                   # 5.76M elements: 703 tiles, the last one partial
    pairs = [synthetic.gamma_pair(31, M, H), synthetic.gamma_pair(32, M, H, scale=0.08)]
    start = dev_bf16(pairs[0]["delta_prev"])
    d_ref, d_new = start.clone(), start.clone()
    st_ref = torch.tensor([1, 0], dtype=torch.int32, device="cuda")
    st_new = st_ref.clone()
    n = M * H - trim                                    # trim = 3: a tail that is not a whole 8-element vector
    ws = sb.workspace(int(sb.lib().sixbit_workspace_size(n, 1)))
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for p in pairs:
        xin, xout = dev_bf16(p["xin"]), dev_bf16(p["xout"])
        g_ref = torch.full((1,), -1.0, device="cuda")
        r_ref = torch.full((1,), -1.0, device="cuda")
        g_new = torch.full((1,), -1.0, device="cuda")
        r_new = torch.full((1,), -1.0, device="cuda")
        _call("sixbit_block_gamma", _p(xin), _p(xout), n, _p(d_ref), _p(g_ref), _p(r_ref), _p(st_ref), None, _p(ws),
              stream)
        _call("sixbit_block_gamma_noalloc", _p(xin), _p(xout), n, _p(d_new), _p(g_new), _p(r_new), _p(st_new), None,
              stream)
        torch.cuda.synchronize()
        gr, gn = host(g_ref)[0], host(g_new)[0]
        rr, rn = host(r_ref)[0], host(r_new)[0]
        assert gr > 0 and rr > 0
        assert gn == gr and rn == rr                    # the same reduction tree: bit-identical
        assert np.array_equal(host_bf16_bits(d_new), host_bf16_bits(d_ref))
        assert host(st_new).tolist() == host(st_ref).tolist()


def test_noalloc_rejects_sizes_beyond_its_limit():
    import nvfp4_int8_mixed_gb300 as sb
    x = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    g = torch.zeros(1, device="cuda")
    too_big = (1 << 40) + 1                             # SIXBIT_NOALLOC_GAMMA_MAX_ELEMS + 1: rejected before any launch
    rc = sb.lib().sixbit_block_gamma_noalloc(_p(x), _p(x), too_big, None, _p(g), None, None, None, None)
    assert rc == sb.ESHAPE
