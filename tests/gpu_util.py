"""Shared helpers of the GPU parity tests: tolerances and the elementwise
allclose check against the fp64 oracle."""
import numpy as np
import pytest
import torch

# fp32 inputs run on TF32 tensor cores: the pages' stricter tolerance
# (atol 1e-3, rtol 1e-2).  bf16/fp16 against the fp64 oracle: 2e-2 / 2e-2.
TOL = {torch.float32: (1e-3, 1e-2), torch.bfloat16: (2e-2, 2e-2), torch.float16: (2e-2, 2e-2)}


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def assert_close(got, want, dtype, what="", tol=None):
    g = got.detach().to(torch.float64).cpu().numpy() if isinstance(got, torch.Tensor) else np.asarray(got)
    want = np.asarray(want, dtype=np.float64)
    assert g.shape == want.shape, (g.shape, want.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    atol, rtol = TOL[dtype] if tol is None else tol
    err = np.abs(g - want)
    bound = atol + rtol * np.abs(want)
    ratio = err / bound
    bad = ratio > 1.0
    if bad.any():
        idx = np.unravel_index(ratio.argmax(), ratio.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements outside atol={atol} rtol={rtol}; "
            f"max abs err {err.max():.3g}; worst at {idx}: got {g[idx]:.6g} want {want[idx]:.6g}")
    return float(err.max())


def tf32_round(t):
    """fp32 values rounded to TF32 (10 fraction bits, nearest, ties to even):
    the operands the TF32 tensor-core products see after the rounding copy."""
    b = t.detach().float().contiguous().view(torch.int32).to(torch.int64) & 0xFFFFFFFF
    b = (b + 0x0FFF + ((b >> 13) & 1)) & 0xFFFFE000
    b = torch.where(b >= 2 ** 31, b - 2 ** 32, b).to(torch.int32)
    return b.view(torch.float32).reshape(t.shape)
