"""LayerNorm and the pre-norm attention block on the GPU through the C ABI,
against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import tf32_bound as tb
from gpu_util import assert_close, assert_within_tf32, need_gpu
from layer_attn_fwd_gb300 import api, build, inputs, ulp

pytestmark = pytest.mark.gpu

FMT = {torch.float32: "f32", torch.bfloat16: "bf16", torch.float16: "f16"}


def _id(x):
    return {torch.float32: "f32", torch.bfloat16: "bf16", torch.float16: "f16"}.get(x, str(x))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    need_gpu()
    build.build()
    api.load()


def _rows(M, d, dtype, seed, mean=3.0, std=2.0):
    g = torch.Generator().manual_seed(seed)
    return (mean + std * torch.randn(M, d, generator=g)).to(dtype)


def _check_ln(y, want, dtype, what):
    """Output rounding (half an ulp of the output type) plus the fp32
    statistics: sums of at most 4096 values, per lane then across the warp,
    ~1e-5 relative."""
    g = y.double().cpu().numpy()
    err = np.abs(g - want)
    bound = 0.5 * ulp.ulp(want, FMT[dtype]) + 1e-5 * (1.0 + np.abs(want))
    worst = np.unravel_index((err / bound).argmax(), err.shape)
    assert (err <= bound).all(), f"{what}: error {err[worst]:.3g} at {worst} over bound {bound[worst]:.3g}"


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16], ids=_id)
@pytest.mark.parametrize("M,d", [(1, 64), (300, 512), (4096, 512), (77, 1024), (33, 2048), (9, 4096)])
def test_layernorm(dtype, M, d):
    """Rows with mean 3 and deviation 2 (the statistics must not lose the
    small deviations to the mean), per-column gamma and beta.  Rows of up to
    512 fp32 / 1024 half values are held in registers, longer ones take the
    three-pass form."""
    x = _rows(M, d, dtype, 110 + d)
    gam, bet = inputs.ln_inputs(d, dtype, seed=111)
    y = api.layernorm(x.cuda(), gam.cuda(), bet.cuda(), eps=1e-5)
    assert api.get_last_error() == api.LA_OK
    _check_ln(y, oracle.layernorm(x, gam, bet, eps=1e-5), dtype, "layernorm")


def test_layernorm_in_place_and_large_eps():
    x = _rows(129, 256, torch.float32, 112, mean=-1.0, std=0.05)
    gam, bet = inputs.ln_inputs(256, seed=113)
    xd = x.cuda()
    api.layernorm(xd, gam.cuda(), bet.cuda(), eps=0.01, out=xd)
    assert api.get_last_error() == api.LA_OK
    _check_ln(xd, oracle.layernorm(x, gam, bet, eps=0.01), torch.float32, "in place")


@pytest.mark.parametrize("with_out", [False, True])
def test_block_fp32_b8_s512_d512(with_out):
    """The pre-norm block on the sublayer workload: fp32 x [8,512,512] with
    mean 3, LayerNorm, Wqkv, attention, (Wo)."""
    x, W, b = inputs.layer_inputs(8, 512, 512, torch.float32, seed=114)
    x = x + 3.0
    gam, bet = inputs.ln_inputs(512, seed=115)
    Wo, bo = inputs.out_proj_inputs(512, seed=116, bias="normal") if with_out else (None, None)
    dev = [None if t is None else t.cuda() for t in (x, gam, bet, W, b, Wo, bo)]
    y = api.layer_attn_ln(*dev, 8)
    assert api.get_last_error() == api.LA_OK
    assert_close(y, oracle.layer_attn_ln(x, gam, bet, W, b, Wo, bo, 8), torch.float32, "block")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16], ids=_id)
@pytest.mark.parametrize("causal", [False, True])
def test_block_small(dtype, causal):
    """Ragged rows and key padding down to 7 visible keys."""
    B, S, dm, H = 3, 150, 256, 2
    x, W, b = inputs.layer_inputs(B, S, dm, dtype, seed=117, bias="normal")
    gam, bet = inputs.ln_inputs(dm, dtype, seed=118)
    Wo, bo = inputs.out_proj_inputs(dm, dtype, seed=119, bias="normal")
    kv_len = torch.tensor([150, 100, 7], dtype=torch.int32)
    y = api.layer_attn_ln(x.cuda(), gam.cuda(), bet.cuda(), W.cuda(), b.cuda(), Wo.cuda(), bo.cuda(), H,
                          causal=causal, kv_len=kv_len.cuda())
    assert api.get_last_error() == api.LA_OK
    want = oracle.layer_attn_ln(x, gam, bet, W, b, Wo, bo, H, causal=causal, kv_len=kv_len)
    if dtype == torch.float32:
        # three TF32 contractions in a row after the LayerNorm, rows with 7
        # visible keys: held to the composed TF32 bound
        xhat = oracle.layernorm(x, gam, bet)
        bound = tb.sublayer_bound(xhat, W, b, H, causal=causal, kv_len=kv_len, Wo=Wo, bo=bo,
                                  dx=tb.layernorm_error(xhat))
        assert_within_tf32(y, want, bound, f"block small causal={causal}")
    else:
        assert_close(y, want, dtype, "block small")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=_id)
def test_block_equals_separate_calls_and_replays(dtype):
    """la_layer_attn_ln (LayerNorm fused into the projection) equals
    la_layernorm then la_layer_attn_out (bit for bit in half precision), and
    a CUDA-graph replay of it equals the direct call."""
    B, S, dm, H = 2, 384, 512, 8
    x, W, b = (t.cuda() for t in inputs.layer_inputs(B, S, dm, dtype, seed=120, bias="normal"))
    gam, bet = (t.cuda() for t in inputs.ln_inputs(dm, dtype, seed=121))
    Wo, bo = (t.cuda() for t in inputs.out_proj_inputs(dm, dtype, seed=122, bias="normal"))
    y = api.layer_attn_ln(x, gam, bet, W, b, Wo, bo, H, causal=True)
    sep = api.layer_attn_out(api.layernorm(x, gam, bet), W, b, Wo, bo, H, causal=True)
    if dtype == torch.float32:
        # the fused LayerNorm rounds x^ to TF32 itself (to nearest, ties
        # away), where the separate path leaves that to the copy into shared
        # memory: both are held to the block's TF32 bound against the oracle
        xc, gc, bc, Wc, bqc, Woc, boc = (t.cpu() for t in (x, gam, bet, W, b, Wo, bo))
        want = oracle.layer_attn_ln(xc, gc, bc, Wc, bqc, Woc, boc, H, causal=True)
        xhat = oracle.layernorm(xc, gc, bc)
        bound = tb.sublayer_bound(xhat, Wc, bqc, H, causal=True, Wo=Woc, bo=boc, dx=tb.layernorm_error(xhat))
        assert_within_tf32(y, want, bound, "fused LayerNorm block")
        assert_within_tf32(sep, want, bound, "separate LayerNorm then block")
    else:
        # half precision: the fused normalisation is the LayerNorm kernel's
        # arithmetic and rounding, so the results agree bit for bit
        assert torch.equal(y, sep)
    ws = torch.empty(api.workspace_size(api.LA_OP_LAYER_ATTN_LN, B, H, S, S, dm // H, dtype), dtype=torch.uint8,
                     device="cuda")
    yg = torch.empty_like(x)
    g = api.Graph(lambda: api.layer_attn_ln(x, gam, bet, W, b, Wo, bo, H, causal=True, out=yg, workspace=ws))
    yg.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert api.get_last_error() == api.LA_OK
    assert torch.equal(yg, y)
