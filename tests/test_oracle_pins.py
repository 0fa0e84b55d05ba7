"""Pins for the fp64 CPU oracle: closed forms, invariants, brute force and a
library routine for the special case.  None of these re-types the oracle's
formula; each would fail on a dropped term, a wrong sign or index, or a
transposed operand somewhere in it.  CPU only.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from layer_attn_fwd_gb300 import inputs


def _np(t):
    return t.double().numpy()


def _sdpa64(q, k, v, causal, kv_len=None, scale=None):
    """torch CPU float64 SDPA with an explicit boolean mask (causal rows aligned
    to the end of the key range, keys >= kv_len[b] masked)."""
    q, k, v = (torch.as_tensor(_np(t) if isinstance(t, torch.Tensor) else t) for t in (q, k, v))
    B, H, S_q, D = q.shape
    S_kv = k.shape[2]
    i = torch.arange(S_q)[:, None] + (S_kv - S_q)
    j = torch.arange(S_kv)[None, :]
    mask = torch.ones(B, 1, S_q, S_kv, dtype=torch.bool)
    if causal:
        mask &= (j <= i)[None, None]
    if kv_len is not None:
        mask &= (j[None] < torch.as_tensor(kv_len).view(B, 1, 1))[:, None]
    o = F.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=scale)
    return o.numpy(), mask.expand(B, H, S_q, S_kv).any(-1).numpy()


# --------------------------------------------------------------------------
# widening of stored values
# --------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_widen_every_16bit_pattern(dtype):
    bits = torch.arange(0, 65536, dtype=torch.int32).to(torch.int16)
    t = bits.view(dtype)
    got = oracle.widen(t)
    want = t.to(torch.float64).numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def test_widen_f32_exact():
    t = torch.tensor([0.0, -0.0, 1.0, 3.0e38, 1.0e-45, -2.5, float("inf")], dtype=torch.float32)
    assert np.array_equal(oracle.widen(t), t.double().numpy())


# --------------------------------------------------------------------------
# closed forms
# --------------------------------------------------------------------------
def test_zero_queries_give_mean_of_values():
    q, k, v = inputs.attn_inputs(2, 3, 37, 37, 16, seed=1)
    q = torch.zeros_like(q)
    o = oracle.attn(q, k, v, causal=False)
    assert np.allclose(o, _np(v).mean(axis=2, keepdims=True), atol=1e-13, rtol=0)
    # causal: prefix mean
    oc = oracle.attn(q, k, v, causal=True)
    pref = np.cumsum(_np(v), axis=2) / np.arange(1, 38)[None, None, :, None]
    assert np.allclose(oc, pref, atol=1e-13, rtol=0)


def test_zero_queries_with_padding_give_mean_of_valid_values():
    q, k, v = inputs.attn_inputs(4, 2, 9, 20, 8, seed=2)
    q = torch.zeros_like(q)
    kv_len = torch.tensor([20, 15, 1, 7], dtype=torch.int32)
    o = oracle.attn(q, k, v, kv_len=kv_len)
    for b in range(4):
        L = int(kv_len[b])
        want = _np(v)[b, :, :L].mean(axis=1)
        assert np.allclose(o[b], want[:, None, :], atol=1e-13, rtol=0)


def test_single_key_returns_its_value():
    q, k, v = inputs.attn_inputs(2, 2, 11, 1, 32, seed=3)
    o = oracle.attn(q, k, v, causal=False)
    assert np.array_equal(o, np.broadcast_to(_np(v), o.shape))
    # causal, rows aligned to the end: only the last query row sees the key
    oc = oracle.attn(q, k, v, causal=True)
    assert np.array_equal(oc[:, :, -1:], _np(v))
    assert np.array_equal(oc[:, :, :-1], np.zeros_like(oc[:, :, :-1]))


def test_constant_values_are_returned_unchanged():
    q, k, v = inputs.attn_inputs(1, 2, 13, 29, 8, seed=4)
    c = torch.randn(1, 2, 1, 8, generator=torch.Generator().manual_seed(5))
    v = c.expand_as(v).contiguous()
    for causal in (False, True):
        o = oracle.attn(q, k, v, causal=causal)
        assert np.allclose(o, np.broadcast_to(_np(c), o.shape), atol=1e-14, rtol=1e-14)


def test_two_keys_logistic_weight():
    from scipy.special import expit
    q, k, v = inputs.attn_inputs(2, 2, 5, 2, 16, seed=6)
    scale = 0.3
    o = oracle.attn(q, k, v, scale=scale)
    s = scale * np.einsum("bhid,bhjd->bhij", _np(q), _np(k))
    w0 = expit(s[..., 0] - s[..., 1])[..., None]
    want = w0 * _np(v)[:, :, 0:1, :] + (1 - w0) * _np(v)[:, :, 1:2, :]
    assert np.allclose(o, want, atol=1e-14, rtol=1e-12)


def test_causal_first_row_is_first_value():
    q, k, v = inputs.attn_inputs(2, 3, 10, 10, 8, seed=7)
    o = oracle.attn(q, k, v, causal=True)
    assert np.array_equal(o[:, :, 0, :], _np(v)[:, :, 0, :])


def test_no_valid_key_gives_zero_row():
    q, k, v = inputs.attn_inputs(2, 1, 4, 6, 8, seed=8)
    o = oracle.attn(q, k, v, kv_len=torch.tensor([0, 6], dtype=torch.int32))
    assert np.array_equal(o[0], np.zeros_like(o[0]))
    assert np.abs(o[1]).sum() > 0
    # S_kv = 0: every row is empty
    k0, v0 = k[:, :, :0].contiguous(), v[:, :, :0].contiguous()
    assert np.array_equal(oracle.attn(q, k0, v0), np.zeros((2, 1, 4, 8)))


def test_large_score_limit_selects_argmax_value():
    q, k, v = inputs.attn_inputs(1, 2, 16, 24, 16, seed=9)
    q = q * 1.0e5  # scores up to ~1e6: exp overflows unless the max is subtracted
    o = oracle.attn(q, k, v, scale=1.0)
    s = np.einsum("bhid,bhjd->bhij", _np(q), _np(k))
    arg = s.argmax(-1)
    srt = np.sort(s, axis=-1)
    assert (srt[..., -1] - srt[..., -2]).min() > 50  # one-hot to far below 1e-20
    want = np.take_along_axis(_np(v), arg[..., None], axis=2)
    assert np.allclose(o, want, atol=1e-15, rtol=0)


# --------------------------------------------------------------------------
# invariants
# --------------------------------------------------------------------------
def test_probability_rows_sum_to_one_and_respect_mask():
    q, k, v = inputs.attn_inputs(2, 2, 7, 12, 8, seed=10)
    kv_len = torch.tensor([12, 9], dtype=torch.int32)
    p = oracle.attn_probs(q, k, causal=True, kv_len=kv_len)
    assert np.allclose(p.sum(-1), 1.0, atol=1e-14)
    i = np.arange(7)[:, None] + 5
    j = np.arange(12)[None, :]
    for b in range(2):
        allowed = (j <= i) & (j < int(kv_len[b]))
        assert np.all(p[b][:, ~allowed] == 0.0)
        assert np.all(p[b][:, allowed] > 0.0)
    # P v reproduces the output
    o = oracle.attn(q, k, v, causal=True, kv_len=kv_len)
    assert np.allclose(np.einsum("bhij,bhjd->bhid", p, _np(v)), o, atol=1e-14)


def test_key_permutation_invariance_and_query_equivariance():
    q, k, v = inputs.attn_inputs(2, 2, 9, 17, 8, seed=11)
    o = oracle.attn(q, k, v)
    perm = torch.randperm(17, generator=torch.Generator().manual_seed(12))
    o2 = oracle.attn(q, k[:, :, perm].contiguous(), v[:, :, perm].contiguous())
    assert np.allclose(o, o2, atol=1e-14, rtol=0)
    pq = torch.randperm(9, generator=torch.Generator().manual_seed(13))
    o3 = oracle.attn(q[:, :, pq].contiguous(), k, v)
    assert np.allclose(o3, o[:, :, pq.numpy()], atol=1e-15, rtol=0)


def test_key_shift_invariance():
    q, k, v = inputs.attn_inputs(2, 2, 11, 11, 8, seed=14)
    c = torch.randn(1, 1, 1, 8, generator=torch.Generator().manual_seed(15), dtype=torch.float64)
    for causal in (False, True):
        o = oracle.attn(q.double(), k.double(), v.double(), causal=causal)
        o2 = oracle.attn(q.double(), (k.double() + c).contiguous(), v.double(), causal=causal)
        assert np.allclose(o, o2, atol=1e-13, rtol=0)


def test_linearity_in_values():
    q, k, v1 = inputs.attn_inputs(1, 2, 8, 14, 8, seed=16)
    _, _, v2 = inputs.attn_inputs(1, 2, 8, 14, 8, seed=17)
    a, b = 0.75, -2.5
    v = (a * v1.double() + b * v2.double()).contiguous()
    for causal in (False, True):
        o = oracle.attn(q.double(), k.double(), v, causal=causal)
        want = a * oracle.attn(q, k, v1, causal=causal) + b * oracle.attn(q, k, v2, causal=causal)
        assert np.allclose(o, want, atol=1e-13, rtol=0)


def test_padding_equals_truncated_keys():
    q, k, v = inputs.attn_inputs(3, 2, 6, 16, 8, seed=18)
    kv_len = torch.tensor([16, 11, 3], dtype=torch.int32)
    o = oracle.attn(q, k, v, kv_len=kv_len)
    for b in range(3):
        L = int(kv_len[b])
        ob = oracle.attn(q[b:b + 1], k[b:b + 1, :, :L].contiguous(), v[b:b + 1, :, :L].contiguous())
        assert np.allclose(o[b:b + 1], ob, atol=1e-15, rtol=0)


# --------------------------------------------------------------------------
# brute force and the library routine
# --------------------------------------------------------------------------
def test_brute_force_high_precision_no_max_subtraction():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 40
    q, k, v = inputs.attn_inputs(1, 2, 5, 6, 4, seed=19)
    scale = 0.5
    for causal in (False, True):
        o = oracle.attn(q, k, v, causal=causal, scale=scale)
        qn, kn, vn = _np(q), _np(k), _np(v)
        for h in range(2):
            for i in range(5):
                lim = i + 1 + 1 if causal else 6  # S_kv - S_q = 1
                w = [mpmath.exp(scale * mpmath.fsum(mpmath.mpf(float(qn[0, h, i, d])) * float(kn[0, h, j, d])
                                                    for d in range(4))) for j in range(lim)]
                Z = mpmath.fsum(w)
                for d in range(4):
                    ref = mpmath.fsum(w[j] * float(vn[0, h, j, d]) for j in range(lim)) / Z
                    assert abs(float(ref) - o[0, h, i, d]) <= 1e-14 * (1 + abs(float(ref)))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(1, 1, 1, 1, 8), (2, 2, 16, 16, 8), (1, 3, 5, 13, 16),
                                   (2, 1, 13, 5, 4), (1, 2, 33, 70, 64)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_matches_torch_float64_sdpa(shape, causal, dtype):
    B, H, S_q, S_kv, D = shape
    q, k, v = inputs.attn_inputs(B, H, S_q, S_kv, D, dtype=dtype, seed=20 + S_kv)
    kv_len = torch.randint(1, S_kv + 1, (B,), generator=torch.Generator().manual_seed(21)).to(torch.int32)
    for kl in (None, kv_len):
        o = oracle.attn(q, k, v, causal=causal, kv_len=kl)
        ref, has_key = _sdpa64(q, k, v, causal, kl)
        assert np.allclose(o[has_key], ref[has_key], atol=1e-12, rtol=1e-12)
        assert np.all(o[~has_key] == 0.0)


# --------------------------------------------------------------------------
# the reformulations the GPU path relies on: online softmax, split-KV, chunking
# --------------------------------------------------------------------------
@pytest.mark.parametrize("block", [1, 3, 16, 128])
def test_online_softmax_equals_definition(block):
    q, k, v = inputs.attn_inputs(2, 2, 19, 45, 8, seed=22)
    kv_len = torch.tensor([45, 30], dtype=torch.int32)
    for causal in (False, True):
        o = oracle.attn(q, k, v, causal=causal, kv_len=kv_len)
        o2 = oracle.attn_online(q, k, v, block, causal=causal, kv_len=kv_len)
        assert np.allclose(o, o2, atol=1e-14, rtol=1e-13)


@pytest.mark.parametrize("n_split", [1, 2, 3, 7, 60])
def test_split_kv_merge_equals_definition(n_split):
    q, k, v = inputs.attn_inputs(2, 2, 13, 41, 8, seed=23)
    kv_len = torch.tensor([41, 20], dtype=torch.int32)
    for causal in (False, True):
        o = oracle.attn(q, k, v, causal=causal, kv_len=kv_len)
        o2 = oracle.attn_split(q, k, v, n_split, causal=causal, kv_len=kv_len)
        assert np.allclose(o, o2, atol=1e-14, rtol=1e-13)


@pytest.mark.parametrize("chunk", [1, 4, 7, 30, 64])
def test_chunked_equals_unchunked(chunk):
    q, k, v = inputs.attn_inputs(2, 2, 30, 30, 8, seed=24)
    for causal in (True, False):
        o = oracle.attn_chunked(q, k, v, chunk, causal=causal)
        if causal:
            want = oracle.attn(q, k, v, causal=True)
            assert np.allclose(o, want, atol=1e-14, rtol=1e-13)
        else:
            # non-causal windows see only the cache so far: window c attends keys < its end
            for s0, L in inputs.chunk_bounds(30, chunk):
                w = oracle.attn(q[:, :, s0:s0 + L].contiguous(), k[:, :, :s0 + L].contiguous(),
                                v[:, :, :s0 + L].contiguous())
                assert np.allclose(o[:, :, s0:s0 + L], w, atol=1e-14, rtol=1e-13)


def test_rows_match_full_output():
    q, k, v = inputs.attn_inputs(2, 3, 40, 40, 16, dtype=torch.bfloat16, seed=25)
    rows = inputs.sample_rows(2, 3, 40, n=25, seed=26, forced=(0, 39))
    full = oracle.attn(q, k, v, causal=True)
    got = oracle.attn_rows(q, k, v, rows, causal=True)
    r = rows.numpy()
    assert np.array_equal(got, full[r[:, 0], r[:, 1], r[:, 2]])
    assert {0, 39} <= set(r[:, 2].tolist())


# --------------------------------------------------------------------------
# fused projection and the sublayer
# --------------------------------------------------------------------------
def test_qkv_proj_head_split_by_construction():
    B, S, dm, H = 2, 5, 24, 3
    x, _, _ = inputs.layer_inputs(B, S, dm, seed=27)
    eye = torch.eye(dm, dtype=torch.float64)
    W = torch.cat([eye, 2 * eye, 3 * eye], dim=1)
    bias = torch.arange(3 * dm, dtype=torch.float64)
    q, k, v = oracle.qkv_proj(x.double(), W, bias, H, q_scale=0.5)
    D = dm // H
    xs = _np(x).reshape(B, S, H, D).transpose(0, 2, 1, 3)
    bs = bias.numpy().reshape(3, H, D)
    assert np.allclose(q, 0.5 * (xs + bs[0][None, :, None, :]), atol=1e-13)
    assert np.allclose(k, 2 * xs + bs[1][None, :, None, :], atol=1e-13)
    assert np.allclose(v, 3 * xs + bs[2][None, :, None, :], atol=1e-13)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_qkv_proj_matches_matmul(dtype):
    B, S, dm, H = 2, 7, 32, 2
    x, W, b = inputs.layer_inputs(B, S, dm, dtype=dtype, seed=28, bias="normal")
    q, k, v = oracle.qkv_proj(x, W, b, H)
    y = _np(x).reshape(B * S, dm) @ _np(W) + _np(b)
    D = dm // H
    y = y.reshape(B, S, 3, H, D).transpose(2, 0, 3, 1, 4)
    for got, want in zip((q, k, v), y):
        assert np.allclose(got, want, atol=1e-12, rtol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_layer_attn_matches_library_pipeline(causal):
    B, S, dm, H = 2, 9, 32, 4
    x, W, b = inputs.layer_inputs(B, S, dm, seed=29, bias="normal")
    kv_len = torch.tensor([9, 6], dtype=torch.int32)
    o = oracle.layer_attn(x, W, b, H, causal=causal, kv_len=kv_len)
    D = dm // H
    y = torch.from_numpy(_np(x).reshape(B * S, dm) @ _np(W) + _np(b)).reshape(B, S, 3, H, D)
    q, k, v = (y[:, :, t].transpose(1, 2).contiguous() for t in range(3))
    ref, _ = _sdpa64(q, k, v, causal, kv_len)
    ref = ref.transpose(0, 2, 1, 3).reshape(B, S, dm)
    assert np.allclose(o, ref, atol=1e-12, rtol=1e-12)


# --------------------------------------------------------------------------
# output projection and the sublayer with it
# --------------------------------------------------------------------------
def test_out_proj_cyclic_shift_moves_columns_one_way():
    """Wo[i, (i+1) % d] = 1 sends column i of a to column i+1 of y; a transposed
    weight would send it to column i-1."""
    M, d = 5, 12
    a = torch.randn(M, d, generator=torch.Generator().manual_seed(60), dtype=torch.float64)
    W = torch.zeros(d, d, dtype=torch.float64)
    W[torch.arange(d), (torch.arange(d) + 1) % d] = 1.0
    bias = torch.arange(d, dtype=torch.float64)
    y = oracle.out_proj(a, W, bias)
    want = np.roll(a.numpy(), 1, axis=1) + bias.numpy()
    assert np.array_equal(y, want)


def test_out_proj_small_integers_exact_by_brute_force():
    """Small integers: every product and sum is exact in fp64, so the result
    must equal plain integer arithmetic bit for bit (non-square, with bias)."""
    g = torch.Generator().manual_seed(61)
    M, d_in, d_out = 4, 6, 5
    a = torch.randint(-4, 5, (M, d_in), generator=g).to(torch.float32)
    W = torch.randint(-4, 5, (d_in, d_out), generator=g).to(torch.float32)
    b = torch.randint(-9, 10, (d_out,), generator=g).to(torch.float32)
    y = oracle.out_proj(a, W, b)
    ai, Wi, bi = a.int().tolist(), W.int().tolist(), b.int().tolist()
    for r in range(M):
        for n in range(d_out):
            assert y[r, n] == sum(ai[r][c] * Wi[c][n] for c in range(d_in)) + bi[n]


def test_out_proj_zero_weight_gives_bias():
    a = torch.randn(3, 4, 8, dtype=torch.float64)
    b = torch.linspace(-1, 1, 8, dtype=torch.float64)
    y = oracle.out_proj(a, torch.zeros(8, 8, dtype=torch.float64), b)
    assert y.shape == (3, 4, 8)
    assert np.array_equal(y, np.broadcast_to(b.numpy(), (3, 4, 8)))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_out_proj_matches_matmul(dtype):
    Wo, bo = inputs.out_proj_inputs(32, dtype=dtype, seed=62, bias="normal")
    a = torch.randn(2, 7, 32, generator=torch.Generator().manual_seed(63)).to(dtype)
    y = oracle.out_proj(a, Wo, bo)
    want = _np(a).reshape(14, 32) @ _np(Wo) + _np(bo)
    assert np.allclose(y.reshape(14, 32), want, atol=1e-12, rtol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_layer_attn_out_matches_library_pipeline(causal):
    """Projection, torch float64 SDPA, head merge, then a float64 matmul with
    Wo: the oracle's sublayer with its output projection must agree."""
    B, S, dm, H = 2, 9, 32, 4
    x, W, b = inputs.layer_inputs(B, S, dm, seed=64, bias="normal")
    Wo, bo = inputs.out_proj_inputs(dm, seed=65, bias="normal")
    kv_len = torch.tensor([9, 5], dtype=torch.int32)
    y = oracle.layer_attn_out(x, W, b, Wo, bo, H, causal=causal, kv_len=kv_len)
    D = dm // H
    p = torch.from_numpy(_np(x).reshape(B * S, dm) @ _np(W) + _np(b)).reshape(B, S, 3, H, D)
    q, k, v = (p[:, :, t].transpose(1, 2).contiguous() for t in range(3))
    o, _ = _sdpa64(q, k, v, causal, kv_len)
    o = o.transpose(0, 2, 1, 3).reshape(B * S, dm)
    want = (o @ _np(Wo) + _np(bo)).reshape(B, S, dm)
    assert np.allclose(y, want, atol=1e-12, rtol=1e-12)


def test_layer_attn_out_identity_weight_is_layer_attn():
    B, S, dm, H = 1, 6, 16, 2
    x, W, b = inputs.layer_inputs(B, S, dm, seed=66, bias="normal")
    eye = torch.eye(dm, dtype=torch.float32)
    y = oracle.layer_attn_out(x, W, b, eye, None, H, causal=True)
    assert np.array_equal(y, oracle.layer_attn(x, W, b, H, causal=True))


# --------------------------------------------------------------------------
# LayerNorm and the pre-norm block
# --------------------------------------------------------------------------
def test_layernorm_closed_form_row():
    """x = [1, 2, 3, 4]: mean 2.5, biased variance 1.25, so with eps = 0 the
    normalised row is [-3, -1, 1, 3] / sqrt(5); then gamma and beta per column."""
    x = torch.tensor([[1.0, 2.0, 3.0, 4.0]], dtype=torch.float64)
    g = torch.tensor([1.0, 2.0, 3.0, 4.0], dtype=torch.float64)
    b = torch.tensor([10.0, 20.0, 30.0, 40.0], dtype=torch.float64)
    y = oracle.layernorm(x, g, b, eps=0.0)
    want = np.array([-3.0, -1.0, 1.0, 3.0]) / math.sqrt(5.0) * g.numpy() + b.numpy()
    assert np.allclose(y[0], want, atol=1e-14, rtol=0)


def test_layernorm_moments_with_eps():
    """gamma = 1, beta = 0: every row has mean 0 and mean square var/(var+eps)."""
    g = torch.Generator().manual_seed(67)
    x = 3.0 + 2.0 * torch.randn(6, 96, generator=g, dtype=torch.float64)
    eps = 0.1
    y = oracle.layernorm(x, torch.ones(96, dtype=torch.float64), torch.zeros(96, dtype=torch.float64), eps=eps)
    var = x.var(dim=1, unbiased=False).numpy()
    assert np.allclose(y.mean(axis=1), 0.0, atol=1e-13)
    assert np.allclose((y * y).mean(axis=1), var / (var + eps), atol=1e-13, rtol=0)


def test_layernorm_affine_invariance():
    """With eps = 0, LN(a x + c) = sign(a) LN(x) for a row-wise shift c."""
    g = torch.Generator().manual_seed(68)
    x = torch.randn(5, 64, generator=g, dtype=torch.float64)
    gam = torch.randn(64, generator=g, dtype=torch.float64)
    bet = torch.randn(64, generator=g, dtype=torch.float64)
    base = oracle.layernorm(x, gam, bet, eps=0.0)
    c = torch.randn(5, 1, generator=g, dtype=torch.float64) * 10
    assert np.allclose(oracle.layernorm(7.5 * x + c, gam, bet, eps=0.0), base, atol=1e-12)
    flipped = oracle.layernorm(-2.0 * x + c, gam, bet, eps=0.0)
    assert np.allclose(flipped - bet.numpy(), -(base - bet.numpy()), atol=1e-12)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_layernorm_matches_torch_float64(dtype):
    g = torch.Generator().manual_seed(69)
    x = (1.5 + torch.randn(2, 7, 128, generator=g)).to(dtype)
    gam = (1.0 + 0.1 * torch.randn(128, generator=g)).to(dtype)
    bet = (0.1 * torch.randn(128, generator=g)).to(dtype)
    want = F.layer_norm(x.double(), (128,), gam.double(), bet.double(), eps=1e-5).numpy()
    assert np.allclose(oracle.layernorm(x, gam, bet, eps=1e-5), want, atol=1e-12, rtol=1e-12)


@pytest.mark.parametrize("with_out", [False, True])
def test_layer_attn_ln_matches_library_pipeline(with_out):
    """torch float64 layer_norm, then the oracle's sublayer pipeline in
    torch (projection, SDPA, merge) and the output projection."""
    B, S, dm, H = 2, 9, 32, 4
    x, W, b = inputs.layer_inputs(B, S, dm, seed=70, bias="normal")
    gam, bet = inputs.ln_inputs(dm, seed=71)
    Wo, bo = inputs.out_proj_inputs(dm, seed=72, bias="normal") if with_out else (None, None)
    kv_len = torch.tensor([9, 4], dtype=torch.int32)
    y = oracle.layer_attn_ln(x, gam, bet, W, b, Wo, bo, H, causal=True, kv_len=kv_len, eps=1e-5)
    xn = F.layer_norm(x.double(), (dm,), gam.double(), bet.double(), eps=1e-5).numpy()
    D = dm // H
    p = torch.from_numpy(xn.reshape(B * S, dm) @ _np(W) + _np(b)).reshape(B, S, 3, H, D)
    q, k, v = (p[:, :, t].transpose(1, 2).contiguous() for t in range(3))
    o, _ = _sdpa64(q, k, v, True, kv_len)
    o = o.transpose(0, 2, 1, 3).reshape(B * S, dm)
    want = (o @ _np(Wo) + _np(bo)) if with_out else o
    assert np.allclose(y, want.reshape(B, S, dm), atol=1e-12, rtol=1e-12)
