"""Shared pieces of the GPU parity tests: tolerances and comparisons.

Tolerances (floating point, bf16 inputs, fp32 accumulation, bf16 output):
O max-abs 2e-2 and mean-abs 2e-3, LSE abs 1e-3 against the float64 oracle.
Integer/byte work (the page gather) is compared bit for bit.
"""

import numpy as np
import pytest
import torch

O_MAX_ABS = 2e-2
O_MEAN_ABS = 2e-3
LSE_ABS = 1e-3


def f64(t):
    """bf16/fp32 tensor -> float64 numpy, exactly."""
    return t.detach().to(torch.float32).cpu().numpy().astype(np.float64)


def assert_o_close(o_gpu, o_ref, what=""):
    got = f64(o_gpu) if isinstance(o_gpu, torch.Tensor) else o_gpu
    assert got.shape == o_ref.shape, (got.shape, o_ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite O"
    diff = np.abs(got - o_ref)
    mx, mean = float(diff.max(initial=0.0)), float(diff.mean()) if diff.size else 0.0
    assert mx <= O_MAX_ABS and mean <= O_MEAN_ABS, f"{what}: O max-abs {mx:.3e} mean-abs {mean:.3e}"
    return mx, mean


def assert_lse_close(lse_gpu, lse_ref, what=""):
    got = f64(lse_gpu) if isinstance(lse_gpu, torch.Tensor) else lse_gpu
    assert got.shape == lse_ref.shape, (got.shape, lse_ref.shape)
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(got), fin), f"{what}: LSE finiteness differs"
    assert np.all(got[~fin] == lse_ref[~fin]), f"{what}: -inf rows differ"
    diff = np.abs(got[fin] - lse_ref[fin])
    mx = float(diff.max(initial=0.0))
    assert mx <= LSE_ABS, f"{what}: LSE max-abs {mx:.3e}"
    return mx


@pytest.fixture(scope="session")
def fa():
    """The loaded library (built on first use); CUDA must be present."""
    import exact_tiled_attention_fwd_gb300 as F
    from exact_tiled_attention_fwd_gb300 import _build

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    _build.build()
    F.load()
    return F
