"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds no attention arithmetic: it only draws random tensors with
the shapes and distributions of the workloads (N(0,1) activations, N(0, 1/d)
projection weights, a key-padding pattern, sampled query rows) from
``torch.Generator`` seeds on the CPU, so that the CUDA path and the CPU oracle
see identical stored bits.  Half-precision inputs are drawn in fp32 and
rounded to nearest-even by ``Tensor.to``.
"""
from __future__ import annotations

import torch


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def attn_inputs(B, H, S_q, S_kv, D, dtype=torch.float32, seed=0):
    """q [B,H,S_q,D], k and v [B,H,S_kv,D], i.i.d. N(0,1), cast to dtype."""
    g = _gen(seed)
    q = torch.randn(B, H, S_q, D, generator=g, dtype=torch.float32)
    k = torch.randn(B, H, S_kv, D, generator=g, dtype=torch.float32)
    v = torch.randn(B, H, S_kv, D, generator=g, dtype=torch.float32)
    return q.to(dtype), k.to(dtype), v.to(dtype)


def layer_inputs(B, S, d_model, dtype=torch.float32, seed=0, bias="zero"):
    """x [B,S,d] ~ N(0,1); Wqkv [d,3d] ~ N(0,1/d); bqkv [3d] zero or N(0,1/4)."""
    g = _gen(seed)
    x = torch.randn(B, S, d_model, generator=g, dtype=torch.float32)
    W = torch.randn(d_model, 3 * d_model, generator=g, dtype=torch.float32) / (d_model ** 0.5)
    if bias == "zero":
        b = torch.zeros(3 * d_model, dtype=torch.float32)
    elif bias == "normal":
        b = 0.5 * torch.randn(3 * d_model, generator=g, dtype=torch.float32)
    else:
        raise ValueError(bias)
    return x.to(dtype), W.to(dtype), b.to(dtype)


def out_proj_inputs(d_model, dtype=torch.float32, seed=0, bias="zero"):
    """Output projection weight Wo [d,d] ~ N(0,1/d) and bias bo [d], zero or
    N(0,1/4)."""
    g = _gen(seed)
    Wo = torch.randn(d_model, d_model, generator=g, dtype=torch.float32) / (d_model ** 0.5)
    if bias == "zero":
        bo = torch.zeros(d_model, dtype=torch.float32)
    elif bias == "normal":
        bo = 0.5 * torch.randn(d_model, generator=g, dtype=torch.float32)
    else:
        raise ValueError(bias)
    return Wo.to(dtype), bo.to(dtype)


def ln_inputs(d_model, dtype=torch.float32, seed=0):
    """LayerNorm gain gamma [d] ~ 1 + N(0, 0.1^2) and shift beta [d] ~ N(0, 0.1^2)."""
    g = _gen(seed)
    gamma = 1.0 + 0.1 * torch.randn(d_model, generator=g, dtype=torch.float32)
    beta = 0.1 * torch.randn(d_model, generator=g, dtype=torch.float32)
    return gamma.to(dtype), beta.to(dtype)


def padding_kv_len(B, S_kv):
    """Key-padding pattern: the first half of the batch keeps 75% of its keys
    (the last quarter is padding); the second half keeps all of them."""
    kv = torch.full((B,), S_kv, dtype=torch.int32)
    kv[: B // 2] = S_kv - S_kv // 4
    return kv


def sample_rows(B, H, S, n=256, seed=1234, forced=()):
    """n query rows (b, h, i) drawn uniformly with a seed; positions listed in
    `forced` (chunk boundaries, the last row) are always included, each with a
    seeded (b, h).  Returns an int64 tensor [n, 3]."""
    g = _gen(seed)
    forced = [int(i) for i in forced if 0 <= int(i) < S]
    m = max(n - len(forced), 0)
    b = torch.randint(0, B, (n,), generator=g)
    h = torch.randint(0, H, (n,), generator=g)
    i = torch.randint(0, S, (m,), generator=g)
    i = torch.cat([torch.tensor(forced, dtype=torch.int64), i])[:n]
    return torch.stack([b[: len(i)], h[: len(i)], i], dim=1).to(torch.int64)


def chunk_bounds(S, chunk):
    """[(start, length)] of consecutive windows of `chunk` positions over S."""
    return [(s, min(chunk, S - s)) for s in range(0, S, chunk)]
