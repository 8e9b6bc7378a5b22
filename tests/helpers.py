"""Shared test helpers: tolerances, error measures, device handling."""
import numpy as np
import torch

# Tolerances stated for the path: max relative error <= 2e-2 for outputs of
# bf16-input computations, <= 1e-5 for fp32 paths.
TOL_BF16 = 2e-2
TOL_F32 = 1e-5


def max_rel_err(got, ref) -> float:
    """max_i |g_i - r_i| / max(|r_i|, rms(r)): elementwise relative error, floored at
    the reference's root-mean-square so that near-zero entries do not dominate."""
    g = np.asarray(got, dtype=np.float64).ravel()
    r = np.asarray(ref, dtype=np.float64).ravel()
    if r.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(r * r)))
    den = np.maximum(np.abs(r), rms if rms > 0 else 1.0)
    return float(np.max(np.abs(g - r) / den))


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float64).numpy()


def bits_equal(a: torch.Tensor, b: torch.Tensor) -> bool:
    # a fresh dense copy: .contiguous() keeps the stride of a size-1 dimension,
    # which a byte view does not accept
    a = torch.empty_like(a, device="cpu", memory_format=torch.contiguous_format).copy_(a.detach())
    b = torch.empty_like(b, device="cpu", memory_format=torch.contiguous_format).copy_(b.detach())
    if a.shape != b.shape or a.dtype != b.dtype:
        return False
    return bool(torch.equal(a.view(torch.uint8), b.view(torch.uint8)))


def cuda(t: torch.Tensor) -> torch.Tensor:
    return t.to("cuda").contiguous()
