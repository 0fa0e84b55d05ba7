"""A seeded sweep of random attention problems on the GPU through the C ABI,
element by element against the fp64 oracle: element type, head size, batch,
heads, query and key lengths (1 to 900, ragged), causal or not, with or
without key padding (lengths from 0 to past the end).  The sizes span the
one-CTA-per-item and the persistent forms and split key ranges."""
import numpy as np
import pytest
import torch

import oracle
import tf32_bound as tb
from gpu_util import assert_close, assert_within_tf32, need_gpu
from layer_attn_fwd_gb300 import api, build, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    need_gpu()
    build.build()
    api.load()


def _case(seed):
    r = np.random.default_rng(1000 + seed)
    dtype = [torch.float32, torch.bfloat16, torch.float16][int(r.integers(3))]
    D = int(r.choice([64, 128]))
    B = int(r.integers(1, 5))
    # fp32 is held to its TF32 bound, which needs the probabilities: fewer heads
    H = int(r.integers(1, 7 if dtype == torch.float32 else 49))
    S_q, S_kv = int(r.integers(1, 701)), int(r.integers(1, 901))
    causal = bool(r.integers(2))
    kv_len = torch.tensor(r.integers(0, S_kv + 50, size=B), dtype=torch.int32) if r.integers(3) == 0 else None
    return dtype, D, B, H, S_q, S_kv, causal, kv_len


@pytest.mark.parametrize("seed", range(24))
def test_random_problem(seed):
    dtype, D, B, H, S_q, S_kv, causal, kv_len = _case(seed)
    what = f"seed {seed}: {dtype} D={D} B={B} H={H} S_q={S_q} S_kv={S_kv} causal={causal} kv_len={kv_len}"
    q, k, v = inputs.attn_inputs(B, H, S_q, S_kv, D, dtype, seed=2000 + seed)
    kl = kv_len.cuda() if kv_len is not None else None
    o = api.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, kv_len=kl)
    assert api.get_last_error() == api.LA_OK, what
    kn = kv_len.numpy() if kv_len is not None else None
    want = oracle.attn(q, k, v, causal=causal, kv_len=kn)
    if dtype == torch.float32:
        P = oracle.attn_probs(q, k, causal=causal, kv_len=kn)
        assert_within_tf32(o, want, tb.attn_bound(q.numpy(), k.numpy(), v.numpy(), P, want, D ** -0.5), what)
    else:
        assert_close(o, want, dtype, what)


def _layer_case(seed):
    r = np.random.default_rng(3000 + seed)
    dtype = [torch.float32, torch.bfloat16, torch.float16][int(r.integers(3))]
    D = int(r.choice([64, 128]))
    H = int(r.integers(1, (512 if dtype == torch.float32 else 1024) // D + 1))
    B, S = int(r.integers(1, 5)), int(r.integers(1, 601))
    causal = bool(r.integers(2))
    kv_len = torch.tensor(r.integers(0, S + 20, size=B), dtype=torch.int32) if r.integers(3) == 0 else None
    bias = "normal" if r.integers(2) else "zero"
    prepared = bool(r.integers(2))
    return dtype, D, H, B, S, causal, kv_len, bias, prepared


@pytest.mark.parametrize("seed", range(12))
def test_random_sublayer(seed):
    """The projection and attention sublayer on random shapes (d_model = H x D
    up to 512 for fp32, 1024 for half precision), on per-call or prepared
    weights, every output element against the fp64 oracle (fp32 held to the
    composed TF32 bound of the projection and the attention: rows with few
    visible keys do not average the TF32 roundings away)."""
    dtype, D, H, B, S, causal, kv_len, bias, prepared = _layer_case(seed)
    dm = H * D
    what = f"seed {seed}: {dtype} B={B} S={S} d={dm} H={H} causal={causal} kv_len={kv_len} bias={bias} prepared={prepared}"
    x, W, b = inputs.layer_inputs(B, S, dm, dtype, seed=4000 + seed, bias=bias)
    xd, Wd, bd = x.cuda(), W.cuda(), b.cuda()
    kl = kv_len.cuda() if kv_len is not None else None
    if prepared:
        o = api.layer_attn_prepared(xd, api.prepare_weight(Wd), bd, H, causal=causal, kv_len=kl)
    else:
        o = api.layer_attn(xd, Wd, bd, H, causal=causal, kv_len=kl)
    assert api.get_last_error() == api.LA_OK, what
    kn = kv_len.numpy() if kv_len is not None else None
    want = oracle.layer_attn(x, W, b, H, causal=causal, kv_len=kn)
    if dtype == torch.float32:
        assert_within_tf32(o, want, tb.sublayer_bound(x, W, b, H, causal=causal, kv_len=kn), what)
    else:
        assert_close(o, want, dtype, what)


def _chunked_case(seed):
    r = np.random.default_rng(5000 + seed)
    dtype = [torch.float32, torch.bfloat16, torch.float16][int(r.integers(3))]
    D = int(r.choice([64, 128]))
    B, H, S = int(r.integers(1, 4)), int(r.integers(1, 17)), int(r.integers(1, 1501))
    chunk = int(r.integers(max(1, S // 100), 701))
    # fp32 is held to the TF32 bound of causal attention over the whole
    # sequence, which the windows reproduce only when causal
    causal = True if dtype == torch.float32 else bool(r.integers(2))
    return dtype, D, B, H, S, chunk, causal


@pytest.mark.parametrize("seed", range(8))
def test_random_chunked(seed):
    """The chunked mode on random shapes and window lengths (the last window
    ragged), causal or not, every output element against the window-by-window
    fp64 oracle; the cache holds the appended keys bit for bit."""
    dtype, D, B, H, S, chunk, causal = _chunked_case(seed)
    what = f"seed {seed}: {dtype} D={D} B={B} H={H} S={S} chunk={chunk} causal={causal}"
    q, k, v = inputs.attn_inputs(B, H, S, S, D, dtype, seed=6000 + seed)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    cache = api.KVCache(B, H, S, D, dtype)
    outs = []
    for s0, L in inputs.chunk_bounds(S, chunk):
        sl = slice(s0, s0 + L)
        outs.append(api.attn_chunked(qd[:, :, sl].contiguous(), kd[:, :, sl].contiguous(),
                                     vd[:, :, sl].contiguous(), cache, causal=causal))
    assert api.get_last_error() == api.LA_OK, what
    o = torch.cat(outs, dim=2)
    assert torch.equal(cache.k[:, :, :S].cpu(), k), what
    want = oracle.attn_chunked(q, k, v, chunk, causal=causal)
    if dtype == torch.float32:
        P = oracle.attn_probs(q, k, causal=True)
        assert_within_tf32(o, want, tb.attn_bound(q.numpy(), k.numpy(), v.numpy(), P, want, D ** -0.5), what)
    else:
        assert_close(o, want, dtype, what)


def _block_case(seed):
    r = np.random.default_rng(7000 + seed)
    dtype = [torch.float32, torch.bfloat16, torch.float16][int(r.integers(3))]
    D = int(r.choice([64, 128]))
    H = int(r.integers(1, 768 // D + 1))
    B, S = int(r.integers(1, 4)), int(r.integers(1, 401))
    causal = bool(r.integers(2))
    kv_len = torch.tensor(r.integers(0, S + 20, size=B), dtype=torch.int32) if r.integers(3) == 0 else None
    prepared = bool(r.integers(2))
    return dtype, D, H, B, S, causal, kv_len, prepared


@pytest.mark.parametrize("seed", range(8))
def test_random_prenorm_block(seed):
    """The pre-norm block (LayerNorm fused into the projection, attention,
    output projection) on random shapes, on per-call or prepared weights,
    every output element against the fp64 oracle (fp32 held to the composed
    TF32 bound of the LayerNorm and the three contractions)."""
    dtype, D, H, B, S, causal, kv_len, prepared = _block_case(seed)
    dm = H * D
    what = f"seed {seed}: {dtype} B={B} S={S} d={dm} H={H} causal={causal} kv_len={kv_len} prepared={prepared}"
    x, W, b = inputs.layer_inputs(B, S, dm, dtype, seed=8000 + seed, bias="normal")
    gam, bet = inputs.ln_inputs(dm, dtype, seed=8100 + seed)
    Wo, bo = inputs.out_proj_inputs(dm, dtype, seed=8200 + seed, bias="normal")
    dev = [t.cuda() for t in (x, gam, bet, W, b, Wo, bo)]
    kl = kv_len.cuda() if kv_len is not None else None
    if prepared:
        y = api.layer_attn_prepared(dev[0], api.prepare_weight(dev[3]), dev[4], H, gamma=dev[1], beta=dev[2],
                                    Wo_p=api.prepare_weight(dev[5]), bo=dev[6], causal=causal, kv_len=kl)
    else:
        y = api.layer_attn_ln(dev[0], dev[1], dev[2], dev[3], dev[4], dev[5], dev[6], H, causal=causal, kv_len=kl)
    assert api.get_last_error() == api.LA_OK, what
    kn = kv_len.numpy() if kv_len is not None else None
    want = oracle.layer_attn_ln(x, gam, bet, W, b, Wo, bo, H, causal=causal, kv_len=kn)
    if dtype == torch.float32:
        xhat = oracle.layernorm(x, gam, bet)
        bound = tb.sublayer_bound(xhat, W, b, H, causal=causal, kv_len=kn, Wo=Wo, bo=bo, dx=tb.layernorm_error(xhat))
        assert_within_tf32(y, want, bound, what)
    else:
        assert_close(y, want, dtype, what)
