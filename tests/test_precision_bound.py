"""CPU check of the half-precision rounding bound used by the GPU precision
study: a float64 emulation of the path's arithmetic (P rounded to the
operand type, output rounded once) stays inside it, and the same emulation
with P biased by 0.4% (one extra bf16 rounding step's worth) breaks it on
causal cases.  CPU only."""
import numpy as np
import pytest
import torch

import oracle
from layer_attn_fwd_gb300 import inputs
from precision_bound import rounding_bound

FMT = {torch.bfloat16: "bf16", torch.float16: "f16"}


def _round(x, dtype):
    return torch.as_tensor(x, dtype=torch.float32).to(dtype).double().numpy()


def _emulate(q, k, v, causal, dtype, p_bias=1.0):
    qd, kd, vd = (t.double().numpy() for t in (q, k, v))
    D, S = qd.shape[-1], kd.shape[2]
    s = np.einsum("bhid,bhjd->bhij", qd, kd) / np.sqrt(D)
    if causal:
        s = np.where(np.tril(np.ones((qd.shape[2], S), bool)), s, -np.inf)
    pu = np.exp(s - s.max(-1, keepdims=True))
    l = pu.sum(-1, keepdims=True)
    return _round(np.einsum("bhij,bhjd->bhid", _round(pu, dtype) * p_bias, vd) / l, dtype)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "f16"])
@pytest.mark.parametrize("causal", [False, True])
def test_emulated_path_inside_biased_outside(dtype, causal):
    q, k, v = inputs.attn_inputs(1, 2, 128, 128, 64, dtype, seed=150)
    r = oracle.attn(q, k, v, causal=causal)
    P = oracle.attn_probs(q, k, causal=causal)
    vd = v.double().numpy()
    g = _emulate(q, k, v, causal, dtype)
    assert (np.abs(g - r) / rounding_bound(r, g, P, vd, FMT[dtype])).max() < 1.0
    if causal or dtype == torch.float16:
        gb = _emulate(q, k, v, causal, dtype, p_bias=1.004)
        assert (np.abs(gb - r) / rounding_bound(r, gb, P, vd, FMT[dtype])).max() > 1.0
