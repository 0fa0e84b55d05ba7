"""Chunked long-context mode on the GPU through the C ABI: window by window
against a growing cache equals unchunked attention and the oracle."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close, need_gpu, with_ramp
from layer_attn_fwd_gb300 import api, build, inputs

pytestmark = pytest.mark.gpu


def _id(x):
    names = {torch.float32: "f32", torch.bfloat16: "bf16", torch.float16: "f16"}
    return names.get(x, str(x))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    need_gpu()
    build.build()
    api.load()


def _run_chunked(q, k, v, chunk, causal=True, S_max=None):
    B, H, S, D = q.shape
    cache = api.KVCache(B, H, S_max or S, D, q.dtype)
    outs = []
    for s0, L in inputs.chunk_bounds(S, chunk):
        sl = slice(s0, s0 + L)
        outs.append(api.attn_chunked(q[:, :, sl].contiguous(), k[:, :, sl].contiguous(),
                                     v[:, :, sl].contiguous(), cache, causal=causal))
        assert cache.len == s0 + L
    assert api.get_last_error() == api.LA_OK
    return torch.cat(outs, dim=2)


@pytest.mark.parametrize("dtype,D", [(torch.bfloat16, 64), (torch.float32, 64), (torch.float16, 128)], ids=lambda p: _id(p) if not isinstance(p, int) else str(p))
def test_chunked_small(dtype, D):
    B, H, S, C = 2, 2, 1000, 256
    q, k, v = inputs.attn_inputs(B, H, S, S, D, dtype, seed=51)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    o = _run_chunked(qd, kd, vd, C, S_max=S + 24)
    want = oracle.attn(q, k, v, causal=True)
    assert_close(o, want, dtype, "chunked vs oracle")
    o_full = api.attn_fwd(qd, kd, vd, causal=True)
    assert_close(o, o_full.double().cpu().numpy(), dtype, "chunked vs unchunked")
    # the step-by-step oracle agrees too
    assert_close(o, oracle.attn_chunked(q, k, v, C), dtype, "chunked oracle")


def test_chunked_fp32_cache_holds_v_transposed():
    """fp32: each window's values are appended to the cache transposed (V^T
    [B, H, D, S_max]), including windows that start off a 16-byte boundary
    (250-row windows), and the attention reads them from there: the cache
    equals V^T bit for bit and the output matches the oracle."""
    B, H, S, D, C = 2, 3, 1000, 64, 250
    q, k, v = inputs.attn_inputs(B, H, S, S, D, torch.float32, seed=53)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    cache = api.KVCache(B, H, S + 3, D, torch.float32)
    assert cache.c.S_max == 1004 and tuple(cache.v.shape) == (B, H, D, 1004)
    outs = []
    for s0, L in inputs.chunk_bounds(S, C):
        sl = slice(s0, s0 + L)
        outs.append(api.attn_chunked(qd[:, :, sl].contiguous(), kd[:, :, sl].contiguous(),
                                     vd[:, :, sl].contiguous(), cache, causal=True))
    assert api.get_last_error() == api.LA_OK
    assert torch.equal(cache.v[:, :, :, :S].cpu(), v.transpose(2, 3))
    assert torch.equal(cache.k[:, :, :S].cpu(), k)
    assert_close(torch.cat(outs, dim=2), oracle.attn(q, k, v, causal=True), torch.float32, "fp32 chunked, V^T cache")


def test_chunk_of_one_row():
    q, k, v = inputs.attn_inputs(1, 2, 40, 40, 64, torch.bfloat16, seed=52)
    o = _run_chunked(q.cuda(), k.cuda(), v.cuda(), 1)
    assert_close(o, oracle.attn(q, k, v, causal=True), torch.bfloat16, "chunk 1")


def test_chunked_100k_sampled_rows():
    """bf16 causal B=2 H=16 S=100000 D=64, windows of 4096 (the last 1696),
    checked on 256 seeded rows including the window boundaries and the last row."""
    B, H, S, D, C = 2, 16, 100000, 64, 4096
    q, k, v = inputs.attn_inputs(B, H, S, S, D, torch.bfloat16, seed=61)
    o = _run_chunked(q.cuda(), k.cuda(), v.cuda(), C).cpu()
    rows = inputs.sample_rows(B, H, S, n=256, seed=1234, forced=(0, 4095, 4096, 98303, 98304, 99999))
    want = oracle.attn_rows(q, k, v, rows, causal=True)
    r = rows.numpy()
    assert_close(o[r[:, 0], r[:, 1], r[:, 2]], want, torch.bfloat16, "100k sampled rows")


def test_chunked_100k_ramp_values_sampled_rows():
    """The 100k-token chunked run with a ramp over key positions added to the
    values (gpu_util.with_ramp): a window that missed part of the cache, or
    saw a key twice, moves its rows far beyond the tolerance.  256 seeded
    rows including the window boundaries and the last row."""
    B, H, S, D, C = 2, 16, 100000, 64, 4096
    q, k, v = inputs.attn_inputs(B, H, S, S, D, torch.bfloat16, seed=62)
    v = with_ramp(v)
    o = _run_chunked(q.cuda(), k.cuda(), v.cuda(), C).cpu()
    rows = inputs.sample_rows(B, H, S, n=256, seed=1235, forced=(0, 4095, 4096, 98303, 98304, 99999))
    want = oracle.attn_rows(q, k, v, rows, causal=True)
    r = rows.numpy()
    assert_close(o[r[:, 0], r[:, 1], r[:, 2]], want, torch.bfloat16, "100k sampled rows, ramp values")


@pytest.mark.parametrize("dtype,D", [(torch.bfloat16, 64), (torch.float16, 128), (torch.float32, 64)],
                         ids=lambda p: _id(p) if not isinstance(p, int) else str(p))
def test_cache_holds_exactly_the_appended_rows(dtype, D):
    """After windows of uneven length (the last one ragged) the cache holds
    every appended key row, bit for bit, at its position for every (batch,
    head) pair, V likewise (fp32: transposed), and the rows past the
    cache's length keep what was there before (a sentinel)."""
    B, H, S, S_max = 3, 5, 700, 760
    q, k, v = inputs.attn_inputs(B, H, S, S, D, dtype, seed=63)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    cache = api.KVCache(B, H, S_max, D, dtype)
    cache.k.fill_(7.0)
    cache.v.fill_(7.0)
    for s0, L in ((0, 256), (256, 1), (257, 300), (557, 143)):
        sl = slice(s0, s0 + L)
        api.attn_chunked(qd[:, :, sl].contiguous(), kd[:, :, sl].contiguous(), vd[:, :, sl].contiguous(), cache)
        assert cache.len == s0 + L
    assert api.get_last_error() == api.LA_OK
    ck, cv = cache.k.cpu(), cache.v.cpu()
    assert torch.equal(ck[:, :, :S], k)
    assert bool((ck[:, :, S:] == 7.0).all())
    if dtype == torch.float32:
        assert torch.equal(cv[:, :, :, :S], v.transpose(2, 3))
        assert bool((cv[:, :, :, S:] == 7.0).all())
    else:
        assert torch.equal(cv[:, :, :S], v)
        assert bool((cv[:, :, S:] == 7.0).all())
