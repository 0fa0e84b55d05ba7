"""Pins for the ULP arithmetic of the reduced-precision study: the pages'
worked example (tests/golden/precision.txt) and the spacing of stored values
measured directly (numpy's spacing for fp16/fp32, the gap to the next bf16
bit pattern).  CPU only."""
import os

import numpy as np
import pytest
import torch

from layer_attn_fwd_gb300 import ulp

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "precision.txt")


def _golden():
    rows = []
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            rows.append(line.split())
    return rows


def test_pages_worked_example():
    rows = _golden()
    assert len(rows) == 4
    for r in rows:
        if r[0] == "ulp":
            assert ulp.ulp(float(r[2]), r[1]) == float(r[3])
        elif r[0] == "rel":
            got = float(r[3]) * ulp.ulp(float(r[2]), r[1]) / float(r[2])
            assert round(got, len(r[4].split(".")[1])) == float(r[4])
        elif r[0] == "ulps_of_rtol":
            got = float(r[3]) * float(r[2]) / ulp.ulp(float(r[2]), r[1])
            assert round(got, 3) == float(r[4])
        else:
            raise AssertionError(r)


@pytest.mark.parametrize("fmt,np_t", [("f16", np.float16), ("f32", np.float32)])
def test_matches_numpy_spacing(fmt, np_t):
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.standard_normal(2000) * 10.0 ** rng.integers(-6, 4, 2000),
                        [1.0, 2.0, 0.5, 60000.0 if fmt == "f16" else 3.0e38, 6.2e-5, 1e-7]])
    x = x.astype(np_t)
    x = x[x != 0]
    assert np.array_equal(ulp.ulp(x.astype(np.float64), fmt), np.abs(np.spacing(np.abs(x))).astype(np.float64))
    if fmt == "f16":  # the largest finite value (numpy's spacing there runs into infinity)
        assert ulp.ulp(65504.0, fmt) == 32.0


def test_matches_next_bf16_pattern():
    g = torch.Generator().manual_seed(6)
    x = (torch.randn(4000, generator=g) * torch.exp2(torch.randint(-20, 20, (4000,), generator=g).float()))
    x = x.to(torch.bfloat16).abs()
    x = x[x > 0]
    nxt = (x.view(torch.int16) + 1).view(torch.bfloat16)
    gap = (nxt.double() - x.double()).numpy()
    assert np.array_equal(ulp.ulp(x.double().numpy(), "bf16"), gap)


def test_unit_roundoff_is_half_an_ulp_at_one():
    for fmt in ("bf16", "f16", "tf32", "f32"):
        assert ulp.unit_roundoff(fmt) == ulp.ulp(1.0, fmt) / 2
    assert ulp.unit_roundoff("bf16") == 2.0 ** -8 and ulp.unit_roundoff("f16") == 2.0 ** -11
