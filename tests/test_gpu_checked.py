"""The checked build (liblayerattn_checked.so: every global store of the
attention, merge and projection kernels checked against its buffer's extent)
on representative calls of every entry point and kernel form: no check may
fire (LA_OK) and results match the fp64 oracle.  A test hook that declares
an output one row short shows a check firing: the row is skipped, the call
reports LA_ERR_INTERNAL, nothing faults."""
import pytest
import torch

import oracle
import tf32_bound as tb
from gpu_util import assert_close, assert_within_tf32, need_gpu
from layer_attn_fwd_gb300 import api, build, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _checked_lib():
    need_gpu()
    build.build()
    api.load(api.CHECKED_LIB_PATH, reload=True)
    assert api.is_checked_build()
    yield
    api.load(api.LIB_PATH, reload=True)
    assert not api.is_checked_build()


def _attn(q, k, v, **kw):
    o = api.attn_fwd(q.cuda(), k.cuda(), v.cuda(), **kw)
    assert api.get_last_error() == api.LA_OK
    return o


@pytest.mark.parametrize("dtype,D,causal", [(torch.float32, 64, False), (torch.float32, 128, True),
                                            (torch.bfloat16, 128, True), (torch.float16, 64, False)])
def test_single_and_persistent_forms(dtype, D, causal):
    """B=1 H=2 S=300 (one CTA per item) and B=4 H=40 S=512 (the persistent form).
    fp32 is held to the derived TF32 bound on the stored inputs: early causal
    rows average two or three keys, where input rounding alone can reach
    1e-3."""
    for (B, H, S), seed in (((1, 2, 300), 130), ((4, 40, 512), 131)):
        q, k, v = inputs.attn_inputs(B, H, S, S, D, dtype, seed=seed)
        o = _attn(q, k, v, causal=causal)
        want = oracle.attn(q, k, v, causal=causal)
        if dtype == torch.float32:
            P = oracle.attn_probs(q, k, causal=causal)
            bound = tb.attn_bound(q.numpy(), k.numpy(), v.numpy(), P, want, D ** -0.5)
            assert_within_tf32(o, want, bound, f"checked {B}x{H}x{S} D={D}")
        else:
            assert_close(o, want, dtype, f"{B}x{H}x{S}")


def test_split_partials_and_merge():
    """A long key range on few heads: split partials, then the merge kernel."""
    B, H, S_q, S_kv, D = 1, 4, 256, 8192, 64
    q, k, v = inputs.attn_inputs(B, H, S_q, S_kv, D, torch.bfloat16, seed=132)
    assert api.workspace_size(api.LA_OP_ATTN_FWD, B, H, S_q, S_kv, D, torch.bfloat16) > 0
    o = _attn(q, k, v).cpu()
    rows = inputs.sample_rows(B, H, S_q, n=64, seed=133, forced=(0, 255))
    r = rows.numpy()
    assert_close(o[r[:, 0], r[:, 1], r[:, 2]], oracle.attn_rows(q, k, v, rows), torch.bfloat16, "split")


def test_chunked_windows():
    B, H, S, D, C = 1, 2, 2500, 64, 1024
    q, k, v = inputs.attn_inputs(B, H, S, S, D, torch.bfloat16, seed=134)
    cache = api.KVCache(B, H, S, D, torch.bfloat16)
    outs = []
    for s0, L in inputs.chunk_bounds(S, C):
        sl = slice(s0, s0 + L)
        outs.append(api.attn_chunked(q[:, :, sl].contiguous().cuda(), k[:, :, sl].contiguous().cuda(),
                                     v[:, :, sl].contiguous().cuda(), cache, causal=True))
    assert api.get_last_error() == api.LA_OK
    assert_close(torch.cat(outs, dim=2), oracle.attn(q, k, v, causal=True), torch.bfloat16, "chunked")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_prenorm_block_with_output_projection(dtype):
    """LayerNorm, projection (fp32: V written transposed), attention with
    heads merged, output projection (row-major)."""
    B, S, dm, H = 2, 200, 256, 2
    x, W, b = inputs.layer_inputs(B, S, dm, dtype, seed=135, bias="normal")
    g, be = inputs.ln_inputs(dm, dtype, seed=136)
    Wo, bo = inputs.out_proj_inputs(dm, dtype, seed=137, bias="normal")
    y = api.layer_attn_ln(*(t.cuda() for t in (x, g, be, W, b, Wo, bo)), H)
    assert api.get_last_error() == api.LA_OK
    assert_close(y, oracle.layer_attn_ln(x, g, be, W, b, Wo, bo, H), dtype, "block")


def test_a_check_fires_without_a_fault():
    """The output declared one row short: that row (the last head's last
    query) keeps its old contents, every other row is right, the call reports
    LA_ERR_INTERNAL, and the next call is clean."""
    B, H, S, D = 1, 2, 128, 64
    q, k, v = inputs.attn_inputs(B, H, S, S, D, torch.bfloat16, seed=138)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o = torch.full_like(qd, 7.0)
    api.debug_shrink_output_extent(1)
    api.attn_fwd(qd, kd, vd, out=o)
    assert api.get_last_error() == api.LA_ERR_INTERNAL
    oc = o.cpu()
    assert torch.all(oc[B - 1, H - 1, S - 1] == 7.0)
    want = oracle.attn(q, k, v)
    assert_close(oc[:, :, :S - 1], want[:, :, :S - 1], torch.bfloat16, "other rows")
    assert_close(oc[:, :H - 1], want[:, :H - 1], torch.bfloat16, "other heads")
    o2 = api.attn_fwd(qd, kd, vd)
    assert api.get_last_error() == api.LA_OK
    assert_close(o2, want, torch.bfloat16, "next call")
