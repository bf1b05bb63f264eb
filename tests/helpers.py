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


def assert_gemm_close(got, ref, out_dtype, tol=1e-3):
    """fp32 outputs: max |y - r| <= tol * max |r| (normwise-max relative error).
    bf16 outputs additionally allow one bf16 rounding (2^-8 relative) per element."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    scale = max(np.max(np.abs(ref)), 1e-30)
    lim = tol * scale + (2.0 ** -8 * np.abs(ref) if out_dtype == "bf16" else 0.0)
    bad = np.abs(got - ref) > lim
    assert not bad.any(), f"{bad.sum()} elements off; max rel err {rel_err_max(got, ref):.3e}"
