"""Reduced precision (bf16, fp16) element by element against the fp64 oracle.

The half-precision path rounds twice: P (kept in fp32 until then, up to 2^8
with the lazy rescale) to the operand type before the PV product, and the
fp32 output to its storage type.  So every element must satisfy

  |o - r| <= 0.5 ulp(r) + u * sum_j p_j |v_j| + (fp16) 2^-25 sum_j |v_j| / l
             + slack * (sum_j p_j |v_j| + |r|)

with p the oracle's normalised probabilities, u the unit roundoff of the
operand type (2^-8 bf16, 2^-11 fp16), the fp16 term for probabilities in the
subnormal range (absolute rounding 2^-25, l >= 1 with the row maximum's
weight 1) and a slack of 2^-12 for the fp32 score, exponential and
accumulation arithmetic.  A kernel that rounded anything else to half
precision, or rounded P twice, fails it.

With LA_PRECISION_REPORT set to a file name, the study of the pages'
reduced-precision analysis ("Shape-Aware Attention", section Challenges we
ran into: bf16's worst element 2 ULP against a 1% tolerance of 1.389 ULP) is
written there as JSON: per format, the largest error in ULPs among elements
with |r| >= 1 and how many elements miss atol 1e-3 / rtol 1e-2."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from gpu_util import need_gpu
from precision_bound import SLACK, rounding_bound
from layer_attn_fwd_gb300 import api, build, inputs, ulp

pytestmark = pytest.mark.gpu

FMT = {torch.bfloat16: "bf16", torch.float16: "f16"}
_study = {}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    need_gpu()
    build.build()
    api.load()
    yield
    path = os.environ.get("LA_PRECISION_REPORT")
    if path and _study:
        with open(path, "w") as f:
            json.dump(_study, f, indent=1)


_bound = rounding_bound


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "f16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_error_within_the_two_roundings(dtype, D, causal):
    B, H, S = 1, 4, 256
    fmt = FMT[dtype]
    st = _study.setdefault(fmt, {"elements": 0, "max_ulps_at_ge1": 0.0, "n_ge1": 0, "n_over_1ulp_at_ge1": 0,
                                 "n_fail_1e-3_1e-2": 0, "worst_bound_ratio": 0.0})
    for seed in range(4):
        q, k, v = inputs.attn_inputs(B, H, S, S, D, dtype, seed=100 + seed)
        o = api.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal)
        assert api.get_last_error() == api.LA_OK
        g = o.double().cpu().numpy()
        r = oracle.attn(q, k, v, causal=causal)
        P = oracle.attn_probs(q, k, causal=causal)
        err = np.abs(g - r)
        ratio = err / _bound(r, g, P, v.double().numpy(), fmt)
        worst = np.unravel_index(ratio.argmax(), ratio.shape)
        assert ratio.max() <= 1.0, (f"seed {seed}: error {err[worst]:.3g} at {worst} (got {g[worst]:.6g}, "
                                    f"want {r[worst]:.6g}) is {ratio.max():.3f} of the rounding bound")
        big = np.abs(r) >= 1.0
        u = ulp.in_ulps(err, r, fmt)
        st["elements"] += int(err.size)
        st["n_ge1"] += int(big.sum())
        st["max_ulps_at_ge1"] = max(st["max_ulps_at_ge1"], float(u[big].max()) if big.any() else 0.0)
        st["n_over_1ulp_at_ge1"] += int((u[big] > 1.0).sum())
        st["n_fail_1e-3_1e-2"] += int((err > 1e-3 + 1e-2 * np.abs(r)).sum())
        st["worst_bound_ratio"] = max(st["worst_bound_ratio"], float(ratio.max()))
