"""The largest shapes the library accepts, on the GPU through the C ABI,
element by element against the fp64 oracle: the most (batch, head) pairs an
attention call takes (B*H = 65535; one more is refused, tests/test_abi.py),
and a wide model through the fused projection (d_model = 4096, 32 heads of
128)."""
import numpy as np
import pytest
import torch

import oracle
import tf32_bound as tb
from gpu_util import assert_close, assert_within_tf32, need_gpu, with_ramp
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


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=_id)
def test_most_batch_head_pairs(dtype):
    """B*H = 65535 heads of 24 rows (a ragged 128-row tile), causal, with key
    padding that leaves some batches one key: every output element."""
    B, H, S, D = 5, 13107, 24, 64
    assert B * H == 65535
    q, k, v = inputs.attn_inputs(B, H, S, S, D, dtype, seed=71)
    kv_len = torch.tensor([24, 7, 1, 24, 13], dtype=torch.int32)
    o = api.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True, kv_len=kv_len.cuda())
    assert api.get_last_error() == api.LA_OK
    want = oracle.attn(q, k, v, causal=True, kv_len=kv_len.numpy())
    if dtype == torch.float32:
        P = oracle.attn_probs(q, k, causal=True, kv_len=kv_len.numpy())
        bound = tb.attn_bound(q.numpy(), k.numpy(), v.numpy(), P, want, D ** -0.5)
        assert_within_tf32(o, want, bound, "B*H = 65535")
    else:
        assert_close(o, want, dtype, "B*H = 65535")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=_id)
def test_qkv_proj_wide_model(dtype):
    """d_model = 4096 (K = 4096 per dot product, 12288 output columns), 200
    rows (a full and a partial 128-row tile), non-zero bias."""
    B, S, dm, H = 1, 200, 4096, 32
    x, W, b = inputs.layer_inputs(B, S, dm, dtype, seed=72, bias="normal")
    q, k, v = api.qkv_proj(x.cuda(), W.cuda(), b.cuda(), H)
    assert api.get_last_error() == api.LA_OK
    wq, wk, wv = oracle.qkv_proj(x, W, b, H)
    if dtype == torch.float32:
        bounds = tb.qkv_bounds(x.numpy(), W.numpy(), H)
        bb = tb._heads(np.broadcast_to(2.0 ** -23 * np.abs(b.numpy()), (B, S, 3 * dm)), H, 0)
        for got, want, bnd, n in zip((q, k, v), (wq, wk, wv), bounds, "qkv"):
            assert_within_tf32(got, want, bnd + bb, f"qkv_proj {n} d=4096")
    else:
        for got, want, n in ((q, wq, "q"), (k, wk, "k"), (v, wv, "v")):
            assert_close(got, want, dtype, f"qkv_proj {n} d=4096")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=_id)
def test_long_key_range_one_call(dtype):
    """256 queries against 500,000 keys in one call (3907 key tiles, split
    across CTAs and merged by the combine kernel), causal rows aligned to the
    end with key padding on one head: every output element.  The values
    carry a ramp over key positions (0 to 4), so that every output depends
    on which keys were included: a split left out or counted twice moves it
    far beyond the tolerance."""
    B, H, S_q, S_kv, D = 2, 1, 256, 500_000, 64
    q, k, v = inputs.attn_inputs(B, H, S_q, S_kv, D, dtype, seed=73)
    v = with_ramp(v, 4.0)
    kv_len = torch.tensor([S_kv, 333_333], dtype=torch.int32)
    o = api.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True, kv_len=kv_len.cuda())
    assert api.get_last_error() == api.LA_OK
    want = oracle.attn(q, k, v, causal=True, kv_len=kv_len.numpy())
    if dtype == torch.float32:
        P = oracle.attn_probs(q, k, causal=True, kv_len=kv_len.numpy())
        bound = tb.attn_bound(q.numpy(), k.numpy(), v.numpy(), P, want, D ** -0.5)
        assert_within_tf32(o, want, bound, "S_kv = 500000")
    else:
        assert_close(o, want, dtype, "S_kv = 500000")
