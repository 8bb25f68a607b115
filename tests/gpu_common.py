"""Shared helpers for the GPU parity tests (all of them call the library through its C ABI)."""
import numpy as np
import pytest
import torch

import exact_io_aware_08_gb300 as fa
from exact_io_aware_08_gb300 import build as fabuild

# Tolerances: O max-abs <= 1e-2, lse max-abs <= 1e-3, dQ/dK/dV max-abs relative to the
# tensor's largest reference magnitude <= 2e-2 (bf16 inputs and outputs, fp32 accumulation).
O_TOL = 1e-2
LSE_TOL = 1e-3
GRAD_REL_TOL = 2e-2


def require_gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    fabuild.build()
    fa.load_library()


def cuda(t):
    return t.to("cuda", non_blocking=False).contiguous()


def poisoned(shape, dtype):
    """Output buffer pre-filled with NaN so an element the kernel never writes is caught."""
    return torch.full(shape, float("nan"), dtype=dtype, device="cuda")


def max_abs(a, b):
    a = a.detach().to("cpu", torch.float64).numpy() if isinstance(a, torch.Tensor) else a
    return float(np.max(np.abs(np.asarray(a, dtype=np.float64) - np.asarray(b, dtype=np.float64)))) \
        if np.size(b) else 0.0


def assert_lse_close(lse_gpu, lse_ref, tol=LSE_TOL):
    g = lse_gpu.detach().to("cpu", torch.float64).numpy()
    r = np.asarray(lse_ref, dtype=np.float64)
    fin = np.isfinite(r)
    assert (np.isfinite(g) == fin).all(), "lse finiteness differs from the oracle"
    assert (g[~fin] == r[~fin]).all()
    if fin.any():
        err = np.max(np.abs(g[fin] - r[fin]))
        assert err <= tol, f"lse max-abs error {err:.3e} > {tol}"


def assert_o_close(o_gpu, o_ref, tol=O_TOL):
    g = o_gpu.detach().to("cpu", torch.float64).numpy()
    assert np.isfinite(g).all(), "non-finite output"
    err = max_abs(g, o_ref)
    assert err <= tol, f"O max-abs error {err:.3e} > {tol}"


def assert_grad_close(g_gpu, g_ref, name, tol=GRAD_REL_TOL):
    g = g_gpu.detach().to("cpu", torch.float64).numpy()
    assert np.isfinite(g).all(), f"non-finite {name}"
    r = np.asarray(g_ref, dtype=np.float64)
    scale = max(np.max(np.abs(r)), 1e-30) if r.size else 1.0
    err = max_abs(g, r) / scale
    assert err <= tol, f"{name} relative max-abs error {err:.3e} > {tol}"
