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


# fp32 comparisons held to the derived TF32 bound (tests/tf32_bound.py):
# (what, elements beyond the fp32 atol/rtol pair, elements, worst
# error / bound), printed at the end of the session by conftest.py.
TF32_RECORDS = []
# at most this share of an fp32 output may lie beyond atol 1e-3 / rtol 1e-2
# (the worst case measured: 2.3%, keys whose norms grow to scores near 100)
MAX_BEYOND_FRACTION = 0.05


def assert_within_tf32(got, want, bound, what=""):
    """fp32 parity against the fp64 oracle on the stored inputs: every element
    within the derived TF32 error bound.  Also counts the elements beyond the
    fp32 tolerance pair (atol 1e-3, rtol 1e-2), which TF32 products alone can
    miss where few keys or large scores leave the rounding unaveraged."""
    g = got.detach().to(torch.float64).cpu().numpy() if isinstance(got, torch.Tensor) else np.asarray(got)
    want = np.asarray(want, dtype=np.float64)
    bound = np.asarray(bound, dtype=np.float64)
    assert g.shape == want.shape == bound.shape, (g.shape, want.shape, bound.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    err = np.abs(g - want)
    atol, rtol = TOL[torch.float32]
    beyond = int((err > atol + rtol * np.abs(want)).sum())
    ratio = err / bound
    TF32_RECORDS.append((what, beyond, err.size, float(ratio.max()) if ratio.size else 0.0))
    bad = ratio > 1.0
    if bad.any():
        idx = np.unravel_index(ratio.argmax(), ratio.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements beyond the TF32 bound; worst at {idx}: "
            f"got {g[idx]:.6g} want {want[idx]:.6g} bound {bound[idx]:.3g}")
    # The bound is a worst case and grows loose where scores are large; a
    # second check: TF32 rounding leaves only a few elements beyond the
    # fp32 tolerance pair, while a wrong mask, index or term moves most of them.
    assert beyond <= MAX_BEYOND_FRACTION * err.size, \
        f"{what}: {beyond} of {err.size} elements beyond atol {atol} / rtol {rtol}"
    return beyond


def with_ramp(v, amplitude=16.0):
    """v [B, H, S_kv, D] plus a ramp over key positions (0 .. amplitude).
    With N(0, 1) values an output row averages thousands of them and sits
    near 0, inside the half-precision atol, so a key range left out or
    counted twice could pass; with the ramp every output depends on which
    keys were included (one 128-key tile dropped from the rows next to the
    diagonal at S = 4096 puts a quarter of their elements beyond the
    tolerance)."""
    S_kv = v.shape[2]
    ramp = amplitude * torch.arange(S_kv, dtype=torch.float32) / S_kv
    return (v.float() + ramp[None, None, :, None]).to(v.dtype)
