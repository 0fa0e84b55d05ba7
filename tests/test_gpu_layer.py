"""Fused Q/K/V projection and the attention sublayer on the GPU through the
C ABI, against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import numpy as np

import tf32_bound as tb
from gpu_util import assert_close, assert_within_tf32, need_gpu
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
    wq, wk, wv = oracle.qkv_proj(x, W, b, H, q_scale=0.5)
    if dtype == torch.float32:
        # TF32 products: a K-long dot product of TF32-rounded operands can miss
        # 1e-3 at K = 384 on its own; held to the derived TF32 bound
        bounds = tb.qkv_bounds(x.numpy(), W.numpy(), H, q_scale=0.5)
        bb = tb._heads(np.broadcast_to(2.0 ** -23 * np.abs(b.numpy()), (B, S, 3 * dm)), H, 0)
        for got, want, bnd, n in zip((q, k, v), (wq, wk, wv), bounds, "qkv"):
            assert_within_tf32(got, want, bnd + bb, f"qkv_proj {n} d={dm} H={H}")
    else:
        for got, want, n in ((q, wq, "q"), (k, wk, "k"), (v, wv, "v")):
            assert_close(got, want, dtype, n)


def test_qkv_proj_no_bias():
    x, W, _ = inputs.layer_inputs(1, 130, 128, torch.bfloat16, seed=42)
    q, k, v = api.qkv_proj(x.cuda(), W.cuda(), None, 2)
    wq, wk, wv = oracle.qkv_proj(x, W, None, 2)
    for got, want in ((q, wq), (k, wk), (v, wv)):
        assert_close(got, want, torch.bfloat16)


@pytest.mark.parametrize("seed", range(8))
def test_layer_fp32_b8_s512_d512(seed):
    """The attention sublayer workload: fp32 x [8,512,512], Wqkv ~ N(0,1/512), zero bias, H=8; 8 seeds."""
    x, W, b = inputs.layer_inputs(8, 512, 512, torch.float32, seed=43 + 100 * seed)
    o = api.layer_attn(x.cuda(), W.cuda(), b.cuda(), 8)
    assert api.get_last_error() == api.LA_OK
    assert_close(o, oracle.layer_attn(x, W, b, 8), torch.float32, "layer")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16], ids=_id)
@pytest.mark.parametrize("causal", [False, True])
def test_layer_small(dtype, causal):
    B, S, dm, H = 3, 150, 256, 2
    x, W, b = inputs.layer_inputs(B, S, dm, dtype, seed=44, bias="normal")
    kv_len = torch.tensor([150, 100, 7], dtype=torch.int32)
    o = api.layer_attn(x.cuda(), W.cuda(), b.cuda(), H, causal=causal, kv_len=kv_len.cuda())
    assert api.get_last_error() == api.LA_OK
    assert_close(o, oracle.layer_attn(x, W, b, H, causal=causal, kv_len=kv_len), dtype, "layer small")


# --------------------------------------------------------------------------
# output projection and the sublayer with it
# --------------------------------------------------------------------------
def _act(M, dm, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    return (0.5 * torch.randn(M, dm, generator=g)).to(dtype)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16], ids=_id)
@pytest.mark.parametrize("M,dm", [(300, 512), (4096, 512), (129, 192), (1000, 1024)])
def test_out_proj(dtype, M, dm):
    """Ragged row counts (a partial last 128-row tile) and widths that are and
    are not multiples of the tile width."""
    a = _act(M, dm, dtype, 70 + dm)
    Wo, bo = inputs.out_proj_inputs(dm, dtype, seed=71, bias="normal")
    y = api.out_proj(a.cuda(), Wo.cuda(), bo.cuda())
    assert api.get_last_error() == api.LA_OK
    want = oracle.out_proj(a, Wo, bo)
    if dtype == torch.float32:  # TF32 products: the derived bound (see test_qkv_proj)
        bound = tb.gemm_bound(a.numpy(), Wo.numpy()) + 2.0 ** -23 * np.abs(bo.numpy())
        assert_within_tf32(y, want, bound, f"out_proj M={M} d={dm}")
    else:
        assert_close(y, want, dtype, "out_proj")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=_id)
def test_out_proj_wide_tiles_sampled_rows(dtype):
    """M = 8192, d = 1024: enough tiles that the wide tile (fp32 192, bf16 256
    columns) is chosen; 256 sampled rows against the oracle."""
    M, dm = 8192, 1024
    a = _act(M, dm, dtype, 72)
    Wo, _ = inputs.out_proj_inputs(dm, dtype, seed=73)
    y = api.out_proj(a.cuda(), Wo.cuda(), None).cpu()
    assert api.get_last_error() == api.LA_OK
    rows = torch.randperm(M, generator=torch.Generator().manual_seed(74))[:256]
    rows[:2] = torch.tensor([0, M - 1])
    want = oracle.out_proj(a[rows], Wo)
    if dtype == torch.float32:
        assert_within_tf32(y[rows], want, tb.gemm_bound(a[rows].numpy(), Wo.numpy()), "out_proj wide")
    else:
        assert_close(y[rows], want, dtype, "out_proj wide")


def test_layer_out_fp32_b8_s512_d512():
    """The sublayer workload with its output projection: fp32 x [8,512,512],
    Wqkv and Wo ~ N(0,1/512), zero biases, H=8."""
    x, W, b = inputs.layer_inputs(8, 512, 512, torch.float32, seed=75)
    Wo, bo = inputs.out_proj_inputs(512, torch.float32, seed=76)
    y = api.layer_attn_out(x.cuda(), W.cuda(), b.cuda(), Wo.cuda(), bo.cuda(), 8)
    assert api.get_last_error() == api.LA_OK
    assert_close(y, oracle.layer_attn_out(x, W, b, Wo, bo, 8), torch.float32, "layer+out")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16], ids=_id)
@pytest.mark.parametrize("causal", [False, True])
def test_layer_out_small(dtype, causal):
    B, S, dm, H = 3, 150, 256, 2
    x, W, b = inputs.layer_inputs(B, S, dm, dtype, seed=77, bias="normal")
    Wo, bo = inputs.out_proj_inputs(dm, dtype, seed=78, bias="normal")
    kv_len = torch.tensor([150, 100, 7], dtype=torch.int32)
    y = api.layer_attn_out(x.cuda(), W.cuda(), b.cuda(), Wo.cuda(), bo.cuda(), H, causal=causal,
                           kv_len=kv_len.cuda())
    assert api.get_last_error() == api.LA_OK
    want = oracle.layer_attn_out(x, W, b, Wo, bo, H, causal=causal, kv_len=kv_len)
    if dtype == torch.float32:
        # three TF32 contractions in a row (projection, attention, output
        # projection); with only 7 visible keys in one batch entry the output
        # repeats single rows of v, so the TF32 rounding is not averaged away
        # and can pass 1e-3 on its own: held to the composed TF32 bound
        bound = tb.sublayer_bound(x, W, b, H, causal=causal, kv_len=kv_len, Wo=Wo, bo=bo)
        assert_within_tf32(y, want, bound, f"layer+out small causal={causal}")
    else:
        assert_close(y, want, dtype, "layer+out small")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=_id)
def test_layer_out_equals_separate_calls(dtype):
    """The one-call sublayer equals la_layer_attn then la_out_proj bit for bit
    (same kernels, same stored intermediate), also when a second call with
    another Wo follows at once on the same workspace."""
    B, S, dm, H = 2, 384, 512, 8
    x, W, b = (t.cuda() for t in inputs.layer_inputs(B, S, dm, dtype, seed=79, bias="normal"))
    Wo1, bo1 = (t.cuda() for t in inputs.out_proj_inputs(dm, dtype, seed=80, bias="normal"))
    Wo2, bo2 = (t.cuda() for t in inputs.out_proj_inputs(dm, dtype, seed=81, bias="normal"))
    ws = torch.empty(api.workspace_size(api.LA_OP_LAYER_ATTN_OUT, B, H, S, S, dm // H, dtype), dtype=torch.uint8,
                     device="cuda")
    y1 = api.layer_attn_out(x, W, b, Wo1, bo1, H, workspace=ws)
    y2 = api.layer_attn_out(x, W, b, Wo2, bo2, H, workspace=ws)
    o = api.layer_attn(x, W, b, H)
    assert api.get_last_error() == api.LA_OK
    assert torch.equal(y1, api.out_proj(o, Wo1, bo1))
    assert torch.equal(y2, api.out_proj(o, Wo2, bo2))


def test_layer_f16_b8_s512_d512():
    """The sublayer workload in fp16 end to end (x, weights, q/k/v, output)."""
    x, W, b = inputs.layer_inputs(8, 512, 512, torch.float16, seed=83)
    o = api.layer_attn(x.cuda(), W.cuda(), b.cuda(), 8)
    assert api.get_last_error() == api.LA_OK
    assert_close(o, oracle.layer_attn(x, W, b, 8), torch.float16, "layer f16")


def test_layer_bf16_b8_s512_d512_wide_projection_tile():
    """bf16 sublayer at B=8 S=512 d=512: the projection takes the 256-column
    tile here (the small cases above take the 128-column one)."""
    x, W, b = inputs.layer_inputs(8, 512, 512, torch.bfloat16, seed=82, bias="normal")
    o = api.layer_attn(x.cuda(), W.cuda(), b.cuda(), 8, causal=True)
    assert api.get_last_error() == api.LA_OK
    assert_close(o, oracle.layer_attn(x, W, b, 8, causal=True), torch.bfloat16, "layer bf16 wide")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=_id)
@pytest.mark.parametrize("form", ["sublayer", "with_out", "prenorm"])
def test_prepared_weights_equal_unprepared(dtype, form):
    """Weights prepared once (la_prepare_weight: fp32 transposed, half
    precision copied) give the unprepared calls' results bit for bit."""
    B, S, dm, H = 2, 300, 512, 8
    x, W, b = (t.cuda() for t in inputs.layer_inputs(B, S, dm, dtype, seed=84, bias="normal"))
    Wo, bo = (t.cuda() for t in inputs.out_proj_inputs(dm, dtype, seed=85, bias="normal"))
    gam, bet = (t.cuda() for t in inputs.ln_inputs(dm, dtype, seed=86))
    Wp, Wop = api.prepare_weight(W), api.prepare_weight(Wo)
    if dtype == torch.float32:
        assert torch.equal(Wp, W.t()) and torch.equal(Wop, Wo.t())
    else:
        assert torch.equal(Wp, W) and torch.equal(Wop, Wo)
    if form == "sublayer":
        want = api.layer_attn(x, W, b, H, causal=True)
        got = api.layer_attn_prepared(x, Wp, b, H, causal=True)
    elif form == "with_out":
        want = api.layer_attn_out(x, W, b, Wo, bo, H, causal=True)
        got = api.layer_attn_prepared(x, Wp, b, H, Wo_p=Wop, bo=bo, causal=True)
    else:
        want = api.layer_attn_ln(x, gam, bet, W, b, Wo, bo, H, causal=True)
        got = api.layer_attn_prepared(x, Wp, b, H, gamma=gam, beta=bet, Wo_p=Wop, bo=bo, causal=True)
    assert api.get_last_error() == api.LA_OK
    assert torch.equal(got, want)
