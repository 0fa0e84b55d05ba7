"""Attention forward on the GPU through the C ABI, element by element against
the fp64 oracle on identical seeded inputs."""
import numpy as np
import pytest
import torch

import oracle
import tf32_bound as tb
from gpu_util import TOL, assert_close, assert_within_tf32, need_gpu, with_ramp
from layer_attn_fwd_gb300 import api, build, inputs

pytestmark = pytest.mark.gpu


def _id(x):
    names = {torch.float32: "f32", torch.bfloat16: "bf16", torch.float16: "f16"}
    return names.get(x, str(x))

DTYPES = [torch.float32, torch.bfloat16, torch.float16]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    need_gpu()
    build.build()
    api.load()


def _gpu_attn(q, k, v, causal, kv_len=None, split=True, scale=None):
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    kl = kv_len.cuda() if kv_len is not None else None
    if split:
        ws = None  # the binding sizes the workspace with la_workspace_size: splits allowed
    else:       # only what an fp32 call must have (V transposed): no room for split partials
        B, H, _, D = q.shape
        n = api.fp32_vt_bytes(B, H, k.shape[2], D) if q.dtype == torch.float32 else 0
        ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    o = api.attn_fwd(qd, kd, vd, causal=causal, scale=scale, kv_len=kl, workspace=ws)
    assert api.get_last_error() == api.LA_OK
    return o


def test_c1_seed_sweep():
    """fp32, non-causal, B=1 H=2 S=128 D=64 over 40 seeds."""
    for seed in range(40):
        q, k, v = inputs.attn_inputs(1, 2, 128, 128, 64, torch.float32, seed=seed)
        o = _gpu_attn(q, k, v, False)
        assert_close(o, oracle.attn(q, k, v), torch.float32, f"seed {seed}")


SHAPES = [(2, 3, 300, 300), (1, 2, 77, 519), (1, 1, 519, 77), (2, 2, 1, 1), (1, 2, 1, 700), (3, 1, 256, 256)]


@pytest.mark.parametrize("dtype", DTYPES, ids=_id)
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SHAPES)
def test_shapes(dtype, D, causal, shape):
    B, H, S_q, S_kv = shape
    q, k, v = inputs.attn_inputs(B, H, S_q, S_kv, D, dtype, seed=S_q * 7 + S_kv + D)
    o = _gpu_attn(q, k, v, causal)
    assert_close(o, oracle.attn(q, k, v, causal=causal), dtype, f"{shape} D={D} causal={causal}")


@pytest.mark.parametrize("dtype", DTYPES, ids=_id)
@pytest.mark.parametrize("causal", [False, True])
def test_key_padding(dtype, causal):
    B, H, S, D = 5, 2, 333, 64
    q, k, v = inputs.attn_inputs(B, H, S, S, D, dtype, seed=11)
    kv_len = torch.tensor([333, 250, 0, 1, 1000], dtype=torch.int32)  # 1000 clamps to S
    o = _gpu_attn(q, k, v, causal, kv_len=kv_len)
    want = oracle.attn(q, k, v, causal=causal, kv_len=kv_len)
    assert_close(o, want, dtype, "padding")
    assert torch.count_nonzero(o[2]).item() == 0  # no visible key -> zero rows


@pytest.mark.parametrize("dtype,D", [(torch.bfloat16, 128), (torch.float16, 64), (torch.float32, 64),
                                     (torch.float32, 128)], ids=lambda p: _id(p) if not isinstance(p, int) else str(p))
@pytest.mark.parametrize("causal", [False, True])
def test_split_kv_equals_unsplit(dtype, D, causal):
    B, H, S_q, S_kv = 1, 2, 256, 4096 + 77
    assert api.workspace_size(api.LA_OP_ATTN_FWD, B, H, S_q, S_kv, D, dtype) > 0  # the plan splits
    q, k, v = inputs.attn_inputs(B, H, S_q, S_kv, D, dtype, seed=12)
    o_split = _gpu_attn(q, k, v, causal, split=True)
    o_one = _gpu_attn(q, k, v, causal, split=False)
    want = oracle.attn(q, k, v, causal=causal)
    assert_close(o_split, want, dtype, "split")
    assert_close(o_one, want, dtype, "unsplit")
    assert_close(o_split, o_one.double().cpu().numpy(), dtype, "split vs unsplit")


def test_scale_parameter():
    q, k, v = inputs.attn_inputs(2, 2, 200, 200, 64, torch.bfloat16, seed=13)
    for scale in (0.01, 0.3):
        o = _gpu_attn(q, k, v, True, scale=scale)
        assert_close(o, oracle.attn(q, k, v, causal=True, scale=scale), torch.bfloat16, f"scale {scale}")


@pytest.mark.parametrize("dtype", DTYPES, ids=_id)
@pytest.mark.parametrize("causal", [False, True])
def test_growing_scores_rescale(dtype, causal):
    """Keys whose norm grows along the sequence: row maxima rise tile after
    tile, so the running max moves (and O is rescaled) for some rows of a warp
    and not for others."""
    B, H, S, D = 2, 2, 700, 64
    q, k, v = inputs.attn_inputs(B, H, S, S, D, torch.float32, seed=18)
    k = k * (1.0 + torch.arange(S, dtype=torch.float32) / 64.0)[None, None, :, None]
    q, k, v = (t.to(dtype) for t in (q, k, v))
    o = _gpu_attn(q, k, v, causal, scale=0.5)
    want = oracle.attn(q, k, v, causal=causal, scale=0.5)
    if dtype == torch.float32:
        # Scores here reach ~100: TF32 inputs alone move them by ~0.05, beyond
        # any 1e-3 tolerance; held to the derived TF32 bound instead.
        P = oracle.attn_probs(q, k, causal=causal, scale=0.5)
        assert_within_tf32(o, want, tb.attn_bound(q.numpy(), k.numpy(), v.numpy(), P, want, 0.5),
                           f"growing scores causal={causal}")
    else:
        assert_close(o, want, dtype, "growing scores")


def test_repeat_runs_bitwise_identical():
    q, k, v = inputs.attn_inputs(2, 4, 1000, 1000, 128, torch.bfloat16, seed=14)
    a = _gpu_attn(q, k, v, True)
    b = _gpu_attn(q, k, v, True)
    assert torch.equal(a, b)


@pytest.mark.parametrize("dtype", DTYPES, ids=_id)
def test_empty_sizes(dtype):
    """S_q = 0 is a no-op; S_kv = 0 gives zero rows (fp32 too, which then
    needs no V transpose and builds no tensor map)."""
    q, k, v = inputs.attn_inputs(2, 2, 0, 50, 64, dtype, seed=15)
    o = _gpu_attn(q, k, v, False)
    assert o.shape == (2, 2, 0, 64)
    q, k, v = inputs.attn_inputs(2, 2, 40, 0, 64, dtype, seed=16)
    qd = q.cuda()
    o = torch.full_like(qd, float("nan"))
    api.attn_fwd(qd, k.cuda(), v.cuda(), out=o)  # the workspace la_workspace_size asks for (fp32: none for V)
    assert api.get_last_error() == api.LA_OK
    assert torch.count_nonzero(o).item() == 0


def test_large_scores_no_overflow():
    q, k, v = inputs.attn_inputs(1, 2, 256, 256, 64, torch.float32, seed=17)
    q = q * 300.0
    o = _gpu_attn(q, k, v, False)
    # scores ~ 300: held to the TF32 bound (see test_growing_scores_rescale)
    want = oracle.attn(q, k, v)
    P = oracle.attn_probs(q, k)
    assert_within_tf32(o, want, tb.attn_bound(q.numpy(), k.numpy(), v.numpy(), P, want, 0.125), "large scores")


def _sampled(o, rows):
    r = rows.numpy()
    return o[r[:, 0], r[:, 1], r[:, 2]]


# The workloads over 8 seeds each (inputs and sampled rows both seeded).
WORKLOAD_SEEDS = range(8)


@pytest.mark.parametrize("padded", [False, True])
@pytest.mark.parametrize("seed", WORKLOAD_SEEDS)
def test_workload_fp32_causal_2048(padded, seed):
    """fp32 causal B=8 H=8 S=2048 D=64 (and the padded variant), 512 sampled rows."""
    B, H, S, D = 8, 8, 2048, 64
    q, k, v = inputs.attn_inputs(B, H, S, S, D, torch.float32, seed=21 + 100 * seed)
    kv_len = inputs.padding_kv_len(B, S) if padded else None
    o = _gpu_attn(q, k, v, True, kv_len=kv_len).cpu()
    rows = inputs.sample_rows(B, H, S, n=512, seed=22 + 100 * seed, forced=(0, 127, 128, 1535, 1536, 2047))
    want = oracle.attn_rows(q, k, v, rows, causal=True, kv_len=kv_len)
    assert_close(_sampled(o, rows), want, torch.float32, f"fp32 causal 2048, seed {seed}")


@pytest.mark.parametrize("padded", [False, True])
def test_workload_fp32_causal_2048_every_row(padded):
    """fp32 causal B=8 H=8 S=2048 D=64 (and the padded variant), one seed,
    every output element against the oracle (held to the TF32 bound, with the
    elements beyond atol 1e-3 / rtol 1e-2 counted)."""
    B, H, S, D = 8, 8, 2048, 64
    q, k, v = inputs.attn_inputs(B, H, S, S, D, torch.float32, seed=25)
    kv_len = inputs.padding_kv_len(B, S) if padded else None
    o = _gpu_attn(q, k, v, True, kv_len=kv_len).cpu()
    want = oracle.attn(q, k, v, causal=True, kv_len=kv_len)
    bound = np.empty_like(want)
    for b in range(B):  # the weights of one batch entry at a time (8 x 2048 x 2048)
        sl = slice(b, b + 1)
        kl = None if kv_len is None else kv_len[sl]
        P = oracle.attn_probs(q[sl], k[sl], causal=True, kv_len=kl)
        bound[sl] = tb.attn_bound(q[sl].numpy(), k[sl].numpy(), v[sl].numpy(), P, want[sl], D ** -0.5)
        del P
    assert_within_tf32(o, want, bound, f"fp32 causal 2048 every row, padded={padded}")


def test_workload_bf16_causal_4096_every_row():
    """bf16 causal B=4 H=16 S=4096 D=128, one seed, every output element."""
    B, H, S, D = 4, 16, 4096, 128
    q, k, v = inputs.attn_inputs(B, H, S, S, D, torch.bfloat16, seed=35)
    o = _gpu_attn(q, k, v, True).cpu()
    assert_close(o, oracle.attn(q, k, v, causal=True), torch.bfloat16, "bf16 causal 4096 every row")


def test_workload_bf16_causal_4096_ramp_values_every_row():
    """The bf16 workload with a ramp over key positions added to the values
    (gpu_util.with_ramp), so that a key tile left out or counted twice fails
    the tolerance: every output element."""
    B, H, S, D = 4, 16, 4096, 128
    q, k, v = inputs.attn_inputs(B, H, S, S, D, torch.bfloat16, seed=36)
    v = with_ramp(v)
    o = _gpu_attn(q, k, v, True).cpu()
    assert_close(o, oracle.attn(q, k, v, causal=True), torch.bfloat16, "bf16 causal 4096 ramp values")


@pytest.mark.parametrize("seed", range(2))
def test_workload_f16_causal_4096(seed):
    """The same workload in fp16 (the fp16 configuration), 256 sampled rows."""
    B, H, S, D = 4, 16, 4096, 128
    q, k, v = inputs.attn_inputs(B, H, S, S, D, torch.float16, seed=41 + 100 * seed)
    o = _gpu_attn(q, k, v, True).cpu()
    rows = inputs.sample_rows(B, H, S, n=256, seed=42 + 100 * seed, forced=(0, 255, 256, 4095))
    want = oracle.attn_rows(q, k, v, rows, causal=True)
    assert_close(_sampled(o, rows), want, torch.float16, f"f16 causal 4096, seed {seed}")


@pytest.mark.parametrize("seed", WORKLOAD_SEEDS)
def test_workload_bf16_causal_4096(seed):
    """bf16 causal B=4 H=16 S=4096 D=128, 256 sampled rows."""
    B, H, S, D = 4, 16, 4096, 128
    q, k, v = inputs.attn_inputs(B, H, S, S, D, torch.bfloat16, seed=31 + 100 * seed)
    o = _gpu_attn(q, k, v, True).cpu()
    rows = inputs.sample_rows(B, H, S, n=256, seed=32 + 100 * seed, forced=(0, 255, 256, 4095))
    want = oracle.attn_rows(q, k, v, rows, causal=True)
    assert_close(_sampled(o, rows), want, torch.bfloat16, f"bf16 causal 4096, seed {seed}")


@pytest.mark.parametrize("D,S_q,S_kv", [(64, 128, 128), (64, 200, 100), (64, 77, 1), (128, 64, 64), (128, 100, 37)])
def test_fp32_one_key_tile_transposes_v_in_kernel(D, S_q, S_kv):
    """fp32 calls of one key tile and one CTA per item transpose V inside
    the attention kernel (no V^T pre-pass): bit for bit what the pre-pass
    path computes (the same inputs as one call of more items than SMs, which
    takes the persistent form and the pre-pass), and within the TF32 bound
    of the oracle.  Ragged key counts leave zero-filled rows in the tile."""
    B, H = 2, 80
    q, k, v = inputs.attn_inputs(B, H, S_q, S_kv, D, torch.float32, seed=131 + D + S_kv)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    whole = api.attn_fwd(qd, kd, vd, causal=True)  # 160 items or more: persistent form, V^T pre-pass
    halves = torch.cat([api.attn_fwd(qd[b:b + 1], kd[b:b + 1], vd[b:b + 1], causal=True) for b in range(B)])
    assert api.get_last_error() == api.LA_OK
    assert torch.equal(whole, halves)
    want = oracle.attn(q, k, v, causal=True)
    P = oracle.attn_probs(q, k, causal=True)
    assert_within_tf32(halves, want, tb.attn_bound(q.numpy(), k.numpy(), v.numpy(), P, want, D ** -0.5),
                       f"in-kernel V transpose D={D} S_kv={S_kv}")


def _vt_given(q, k, v, causal):
    """The same attention with V^T handed to the kernel: one window of the
    chunked mode, whose fp32 cache keeps V transposed."""
    B, H, S, D = q.shape
    cache = api.KVCache(B, H, S, D, torch.float32)
    return api.attn_chunked(q, k, v, cache, causal=causal)


@pytest.mark.parametrize("D,S,causal,padded", [(64, 512, True, False), (64, 300, False, True),
                                               (128, 256, True, False), (128, 200, False, False)])
def test_fp32_persistent_pre_pass_equals_vt_given(D, S, causal, padded):
    """fp32 calls in the persistent form (more items than SMs; the epilogue
    stores each row directly): the V^T pre-pass result equals, bit for bit,
    the result with V^T handed in (one window of the chunked mode, whose
    fp32 cache keeps V transposed), and both stay within the TF32 bound of
    the oracle.  Several key tiles per item, ragged tails, key padding."""
    B, H = 2, 80
    q, k, v = inputs.attn_inputs(B, H, S, S, D, torch.float32, seed=141 + D + S)
    kv_len = torch.tensor([S, S // 2 + 3], dtype=torch.int32) if padded else None
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    kl = kv_len.cuda() if padded else None
    o = api.attn_fwd(qd, kd, vd, causal=causal, kv_len=kl)
    assert api.get_last_error() == api.LA_OK
    if not padded:
        ref = _vt_given(qd, kd, vd, causal)
        assert api.get_last_error() == api.LA_OK
        assert torch.equal(o, ref)
    kln = kv_len.numpy() if padded else None
    want = oracle.attn(q, k, v, causal=causal, kv_len=kln)
    P = oracle.attn_probs(q, k, causal=causal, kv_len=kln)
    assert_within_tf32(o, want, tb.attn_bound(q.numpy(), k.numpy(), v.numpy(), P, want, D ** -0.5),
                       f"persistent fp32 D={D} S={S}")
