"""CPU checks of the fp32 (TF32) error bound in tests/tf32_bound.py against a
model of the TF32 arithmetic: operands truncated to TF32 (the worst rounding
the copy into shared memory may apply), products and sums in fp32, P rounded
to TF32 to nearest.  The modelled error must stay within the bound on every
element, on ordinary inputs and on the hard cases of the parity tests (scores
near 100 and 300, rows with a single visible key, growing key norms); and a
bound missing its input-rounding term must fail on the large scores, so
these checks can fail."""
import numpy as np
import pytest
import torch

import oracle
import tf32_bound as tb
from layer_attn_fwd_gb300 import inputs


def _bits(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32)).view(np.uint32)


def tf32_trunc(x):
    return (_bits(x) & np.uint32(0xFFFFE000)).view(np.float32)


def tf32_nearest_away(x):
    return ((_bits(x) + np.uint32(0x1000)) & np.uint32(0xFFFFE000)).view(np.float32)


def model_attn(q, k, v, scale, causal=False, kv_len=None):
    """TF32 attention as the fp32 path computes it (fp32 everywhere else)."""
    q, k, v = (tf32_trunc(t) for t in (q, k, v))
    B, H, S_q, D = q.shape
    S_kv = k.shape[2]
    o = np.zeros((B, H, S_q, D), dtype=np.float32)
    off = S_kv - S_q
    for b in range(B):
        lim = S_kv if kv_len is None else min(int(kv_len[b]), S_kv)
        for h in range(H):
            s = (q[b, h] @ k[b, h].T).astype(np.float32) * np.float32(scale)
            j = np.arange(S_kv)[None, :]
            vis = j < lim
            if causal:
                vis = vis & (j <= np.arange(S_q)[:, None] + off)
            s = np.where(vis, s, -np.inf).astype(np.float32)
            m = np.max(s, axis=1, keepdims=True)
            m = np.where(np.isfinite(m), m, 0).astype(np.float32)
            p = np.exp(s - m).astype(np.float32)
            l = p.sum(axis=1, keepdims=True, dtype=np.float32)
            pv = (tf32_nearest_away(p) @ v[b, h]).astype(np.float32)
            o[b, h] = np.where(l > 0, pv / np.where(l > 0, l, 1), 0)
    return o.astype(np.float64)


CASES = [
    # (name, B, H, S_q, S_kv, D, causal, q multiplier, kv_len)
    ("plain", 1, 2, 96, 96, 64, False, 1.0, None),
    ("causal", 1, 2, 96, 96, 64, True, 1.0, None),
    ("d128", 1, 1, 64, 80, 128, True, 1.0, None),
    ("scores~300", 1, 2, 64, 64, 64, False, 300.0, None),
    ("few keys", 2, 2, 64, 64, 64, True, 1.0, [1, 7]),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_attention_model_within_bound(case):
    name, B, H, S_q, S_kv, D, causal, mul, kl = case
    q, k, v = inputs.attn_inputs(B, H, S_q, S_kv, D, torch.float32, seed=500 + len(name))
    q = q * mul
    kv_len = None if kl is None else np.array(kl, dtype=np.int32)
    scale = 1.0 / D ** 0.5
    want = oracle.attn(q, k, v, causal=causal, scale=scale, kv_len=kv_len)
    P = oracle.attn_probs(q, k, causal=causal, scale=scale, kv_len=kv_len)
    got = model_attn(q.numpy(), k.numpy(), v.numpy(), scale, causal, kv_len)
    bound = tb.attn_bound(q.numpy(), k.numpy(), v.numpy(), P, want, scale)
    err = np.abs(got - want)
    assert np.all(err <= bound), f"{name}: worst err/bound {np.max(err / bound):.3f}"


def test_growing_key_norms_within_bound():
    """Key norms growing along the sequence (scores up to ~100), scale 0.5."""
    B, H, S, D = 1, 2, 200, 64
    q, k, v = inputs.attn_inputs(B, H, S, S, D, torch.float32, seed=511)
    k = k * (1.0 + torch.arange(S, dtype=torch.float32) / 64.0)[None, None, :, None]
    want = oracle.attn(q, k, v, causal=True, scale=0.5)
    P = oracle.attn_probs(q, k, causal=True, scale=0.5)
    got = model_attn(q.numpy(), k.numpy(), v.numpy(), 0.5, True)
    bound = tb.attn_bound(q.numpy(), k.numpy(), v.numpy(), P, want, 0.5)
    assert np.all(np.abs(got - want) <= bound)


def test_bound_without_input_rounding_fails_on_large_scores():
    """A planted mistake: the bound with its input-rounding term dropped does
    not cover the modelled error at scores ~300."""
    q, k, v = inputs.attn_inputs(1, 2, 64, 64, 64, torch.float32, seed=512)
    q = q * 300.0
    want = oracle.attn(q, k, v, scale=0.125)
    P = oracle.attn_probs(q, k, scale=0.125)
    got = model_attn(q.numpy(), k.numpy(), v.numpy(), 0.125)
    saved = tb.U_IN
    try:
        tb.U_IN = 0.0
        bound = tb.attn_bound(q.numpy(), k.numpy(), v.numpy(), P, want, 0.125)
    finally:
        tb.U_IN = saved
    assert np.any(np.abs(got - want) > bound)


def test_gemm_model_within_bound_and_planted_mistake():
    x, W, _ = inputs.layer_inputs(2, 50, 384, torch.float32, seed=513)
    x = x.numpy().reshape(-1, 384)
    W = W.numpy()
    exact = x.astype(np.float64) @ W.astype(np.float64)
    got = (tf32_trunc(x) @ tf32_trunc(W)).astype(np.float64)
    err = np.abs(got - exact)
    assert np.all(err <= tb.gemm_bound(x, W))
    # without the operand rounding the bound is far too small
    assert np.any(err > (384 + 2) * tb.U_ACC * (np.abs(x) @ np.abs(W)) + tb.TINY)


def test_sublayer_model_within_bound():
    """Projection then attention (errors of q, k, v carried into the attention
    bound): the modelled sublayer stays within the composed bound."""
    B, S, dm, H = 1, 64, 128, 2
    x, W, b = inputs.layer_inputs(B, S, dm, torch.float32, seed=514, bias="normal")
    xn, Wn, bn = x.numpy(), W.numpy(), b.numpy()
    y = (tf32_trunc(xn.reshape(-1, dm)) @ tf32_trunc(Wn)).astype(np.float32) + bn
    y = y.reshape(B, S, 3 * dm)
    qg, kg, vg = (tb._heads(y.astype(np.float64), H, i) for i in range(3))
    D = dm // H
    got = tb.merged(model_attn(qg.astype(np.float32), kg.astype(np.float32), vg.astype(np.float32), D ** -0.5))
    q, k, v = oracle.qkv_proj(x, W, b, H)
    want = oracle.layer_attn(x, W, b, H)
    P = oracle.attn_probs(q, k)
    dq, dk, dv = tb.qkv_bounds(xn, Wn, H)
    bound = tb.merged(tb.attn_bound(q, k, v, P, oracle.attn(q, k, v), D ** -0.5, dq, dk, dv))
    assert np.all(np.abs(got - want) <= bound)
