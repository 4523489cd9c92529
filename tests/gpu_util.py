"""Helpers shared by the GPU tests: host<->device copies of bf16 bit patterns
and the parity metrics.  Holds none of the sharded-Linear arithmetic."""
import numpy as np

BF16_TOL = 5e-3   # max|d| / max|y_ref| for bf16 outputs
FP32_TOL = 1e-5   # same, fp32-output mode


def dev(b16):
    """numpy uint16 (bf16 bits) -> contiguous torch bf16 CUDA tensor."""
    import torch
    a = np.ascontiguousarray(b16, dtype=np.uint16).view(np.int16)
    return torch.from_numpy(a).cuda().view(torch.bfloat16)


def host_f64(t):
    """torch CUDA tensor (bf16 / fp32) -> float64 numpy (exact widening)."""
    import torch
    return t.detach().to(torch.float32).cpu().numpy().astype(np.float64)


def host_bits(t):
    """torch bf16 CUDA tensor -> numpy uint16 bit patterns."""
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def empty(shape, f32=False):
    import torch
    return torch.empty(shape, dtype=torch.float32 if f32 else torch.bfloat16, device="cuda")


def poisoned(shape, f32=False):
    """Output buffer pre-filled with NaN so that unwritten elements show up."""
    import torch
    return torch.full(shape, float("nan"), dtype=torch.float32 if f32 else torch.bfloat16, device="cuda")


def rel_err(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if not np.all(np.isfinite(got)):
        return float("inf")
    scale = np.max(np.abs(ref)) if ref.size else 0.0
    if scale == 0.0:
        return float(np.max(np.abs(got))) if got.size else 0.0
    return float(np.max(np.abs(got - ref)) / scale)


def assert_close(got, ref, f32=False, what=""):
    tol = FP32_TOL if f32 else BF16_TOL
    e = rel_err(got, ref)
    assert e <= tol, f"{what}: max|d|/max|ref| = {e:.3e} > {tol:.0e}"
