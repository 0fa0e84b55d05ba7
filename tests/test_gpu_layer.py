"""Fused Q/K/V projection and the attention sublayer on the GPU through the
C ABI, against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close, need_gpu, tf32_round
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


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16], ids=_id)
@pytest.mark.parametrize("dm,H", [(256, 4), (256, 2), (384, 6)])
def test_qkv_proj(dtype, dm, H):
    B, S = 2, 201
    x, W, b = inputs.layer_inputs(B, S, dm, dtype, seed=41, bias="normal")
    q, k, v = api.qkv_proj(x.cuda(), W.cuda(), b.cuda(), H, q_scale=0.5)
    assert api.get_last_error() == api.LA_OK
    # fp32 runs on TF32 tensor cores: a K-long dot product of TF32-rounded
    # operands can miss 1e-3 at K = 384 on its own, so fp32 is checked on the
    # operands the tensor cores see (the sublayer tests check fp32 end to end)
    xr, Wr = (x, W) if dtype != torch.float32 else (tf32_round(x), tf32_round(W))
    wq, wk, wv = oracle.qkv_proj(xr, Wr, b, H, q_scale=0.5)
    for got, want, n in ((q, wq, "q"), (k, wk, "k"), (v, wv, "v")):
        assert_close(got, want, dtype, n)


def test_qkv_proj_no_bias():
    x, W, _ = inputs.layer_inputs(1, 130, 128, torch.bfloat16, seed=42)
    q, k, v = api.qkv_proj(x.cuda(), W.cuda(), None, 2)
    wq, wk, wv = oracle.qkv_proj(x, W, None, 2)
    for got, want in ((q, wq), (k, wk), (v, wv)):
        assert_close(got, want, torch.bfloat16)


def test_layer_fp32_b8_s512_d512():
    """The attention sublayer workload: fp32 x [8,512,512], Wqkv ~ N(0,1/512), zero bias, H=8."""
    x, W, b = inputs.layer_inputs(8, 512, 512, torch.float32, seed=43)
    o = api.layer_attn(x.cuda(), W.cuda(), b.cuda(), 8)
    assert api.get_last_error() == api.LA_OK
    assert_close(o, oracle.layer_attn(x, W, b, 8), torch.float32, "layer")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=_id)
@pytest.mark.parametrize("causal", [False, True])
def test_layer_small(dtype, causal):
    B, S, dm, H = 3, 150, 256, 2
    x, W, b = inputs.layer_inputs(B, S, dm, dtype, seed=44, bias="normal")
    kv_len = torch.tensor([150, 100, 7], dtype=torch.int32)
    o = api.layer_attn(x.cuda(), W.cuda(), b.cuda(), H, causal=causal, kv_len=kv_len.cuda())
    assert api.get_last_error() == api.LA_OK
    assert_close(o, oracle.layer_attn(x, W, b, H, causal=causal, kv_len=kv_len), dtype, "layer small")
