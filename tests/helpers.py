"""Shared helpers for the tests: moving bf16 bit patterns between numpy and
torch, and the parity metrics.  No attention arithmetic lives here."""
import numpy as np

MAX_ABS_TOL = 2e-2      # element-wise bound, GPU (bf16 out) vs fp64 oracle
REL_RMS_TOL = 5e-3      # ||gpu - ref||_2 / ||ref||_2 over one call's output


def to_dev(bits_u16, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits_u16).view(np.int16)).view(torch.bfloat16).to(device)


def from_dev(t) -> np.ndarray:
    """bf16 CUDA tensor -> float64 numpy (exact widening)."""
    import torch
    u = t.detach().view(torch.int16).cpu().numpy().view(np.uint16)
    return (u.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bits_from_dev(t) -> np.ndarray:
    import torch
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def i32_dev(a, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def parity(gpu: np.ndarray, ref: np.ndarray):
    diff = gpu - ref
    max_abs = float(np.max(np.abs(diff))) if diff.size else 0.0
    den = float(np.sqrt(np.sum(ref * ref)))
    rel_rms = float(np.sqrt(np.sum(diff * diff)) / den) if den > 0 else 0.0
    return max_abs, rel_rms


def assert_parity(gpu, ref, what=""):
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite values in GPU output"
    max_abs, rel_rms = parity(gpu, ref)
    assert max_abs <= MAX_ABS_TOL and rel_rms <= REL_RMS_TOL, \
        f"{what}: max_abs={max_abs:.3e} (tol {MAX_ABS_TOL}), rel_rms={rel_rms:.3e} (tol {REL_RMS_TOL})"
    return max_abs, rel_rms
