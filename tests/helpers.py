"""Shared helpers of the GPU parity tests (host <-> device marshalling only)."""
import numpy as np
import torch


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host_bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def rel_err_max(got, ref) -> float:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-30))


def bf16_ulp(x) -> np.ndarray:
    """Spacing of bf16 values at |x| (8 significant bits): 2^(floor(log2|x|) - 7)."""
    a = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(e - 7), 0.0)


def assert_gemm_close(got, ref, out_dtype, tol=1e-3):
    """fp32 outputs: max |y - r| <= tol * max |r| (normwise-max relative error).
    bf16 outputs: the device and the oracle each round to bf16, so two values
    that agree to within tol can still round one bf16 ulp apart; each element
    may additionally differ by one ulp of the oracle's value."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    scale = max(np.max(np.abs(ref)), 1e-30)
    lim = tol * scale + (bf16_ulp(ref) if out_dtype == "bf16" else 0.0)
    bad = np.abs(got - ref) > lim
    assert not bad.any(), f"{bad.sum()} elements off; max rel err {rel_err_max(got, ref):.3e}"
