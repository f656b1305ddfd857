"""Tolerances and comparison helpers for the GPU-vs-oracle parity tests.

Tolerances (bf16 inputs, fp32 accumulation, bf16 output): max |dO| <= 2e-2,
mean |dO| <= 2e-3 over all compared elements, |dLSE| <= 1e-3 absolute.
"""
import numpy as np
import pytest

MAX_ABS_O = 2e-2
MEAN_ABS_O = 2e-3
MAX_ABS_LSE = 1e-3


def compare(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    """o_gpu / lse_gpu: torch tensors (any device); o_ref / lse_ref: fp64 numpy."""
    o = o_gpu.float().cpu().numpy().astype(np.float64)
    lse = lse_gpu.float().cpu().numpy().astype(np.float64)
    assert o.shape == o_ref.shape and lse.shape == lse_ref.shape, what
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse)), f"{what}: non-finite output"
    do = np.abs(o - o_ref)
    dl = np.abs(lse - lse_ref)
    msg = f"{what}: max|dO|={do.max():.3e} mean|dO|={do.mean():.3e} max|dLSE|={dl.max():.3e}"
    assert do.max() <= MAX_ABS_O and do.mean() <= MEAN_ABS_O and dl.max() <= MAX_ABS_LSE, msg
    return do.max(), do.mean(), dl.max()


def require_gpu():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    major, minor = torch.cuda.get_device_capability()
    if (major, minor) != (10, 3):
        pytest.skip(f"kernels are built for sm_103a, device is sm_{major}{minor}")
    from exact_attention_29_gb300 import build

    build.build()
