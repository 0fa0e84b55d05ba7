"""CUDA-graph capture and replay of library calls: persistent attention
launches (work tickets), the sublayer with its output projection and the
small-shape case, each replay checked against a direct call and the oracle."""
import pytest
import torch

import oracle
from gpu_util import assert_close, need_gpu
from layer_attn_fwd_gb300 import api, build, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    need_gpu()
    build.build()
    api.load()


def test_graph_replays_persistent_attention_with_new_inputs():
    """bf16 B=2 H=80 S=512: 160 work items, so the persistent form with its
    ticket counter runs; six replays, new inputs copied in before each."""
    B, H, S, D = 2, 80, 512, 64
    dtype = torch.bfloat16
    q, k, v = (t.cuda() for t in inputs.attn_inputs(B, H, S, S, D, dtype, seed=90))
    o = torch.empty_like(q)
    g = api.Graph(lambda: api.attn_fwd(q, k, v, causal=True, out=o))
    for rep in range(6):
        qh, kh, vh = inputs.attn_inputs(B, H, S, S, D, dtype, seed=91 + rep)
        q.copy_(qh)
        k.copy_(kh)
        v.copy_(vh)
        g.replay()
        direct = api.attn_fwd(q, k, v, causal=True)
        torch.cuda.synchronize()
        assert api.get_last_error() == api.LA_OK
        assert torch.equal(o, direct), f"replay {rep}"
        if rep in (0, 5):
            assert_close(o, oracle.attn(qh, kh, vh, causal=True), dtype, f"replay {rep}")


def test_graph_replays_interleaved_with_direct_persistent_calls():
    """Direct persistent launches (each with a workspace of its own, under
    a ticket tag of its own) between replays of a captured one (the same tag
    on every replay): every launch hands out each item once."""
    B, H, S, D = 4, 40, 512, 128
    dtype = torch.bfloat16
    q, k, v = (t.cuda() for t in inputs.attn_inputs(B, H, S, S, D, dtype, seed=97))
    o = torch.empty_like(q)
    ref = api.attn_fwd(q, k, v)
    g = api.Graph(lambda: api.attn_fwd(q, k, v, out=o))
    for rep in range(70):
        if rep % 3 == 0:
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(o, ref), f"replay {rep}"
        else:
            assert torch.equal(api.attn_fwd(q, k, v), ref), f"direct {rep}"
    assert api.get_last_error() == api.LA_OK
    assert_close(ref, oracle.attn(q.cpu(), k.cpu(), v.cpu()), dtype, "reference")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_graph_replays_sublayer_with_output_projection(dtype):
    B, S, dm, H = 8, 512, 512, 8
    x, W, b = (t.cuda() for t in inputs.layer_inputs(B, S, dm, dtype, seed=92, bias="normal"))
    Wo, bo = (t.cuda() for t in inputs.out_proj_inputs(dm, dtype, seed=93, bias="normal"))
    ws = torch.empty(api.workspace_size(api.LA_OP_LAYER_ATTN_OUT, B, H, S, S, dm // H, dtype), dtype=torch.uint8,
                     device="cuda")
    y = torch.empty_like(x)
    g = api.Graph(lambda: api.layer_attn_out(x, W, b, Wo, bo, H, out=y, workspace=ws))
    want = api.layer_attn_out(x, W, b, Wo, bo, H)
    for _ in range(3):
        y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y, want)
    assert api.get_last_error() == api.LA_OK


def test_graph_small_shape_fp32():
    """The small case, fp32 B=1 H=2 S=128 D=64 (V transposed first, then one
    CTA per head): replayed against the oracle."""
    B, H, S, D = 1, 2, 128, 64
    q, k, v = inputs.attn_inputs(B, H, S, S, D, torch.float32, seed=94)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    o = torch.empty_like(qd)
    ws = torch.empty(api.workspace_size(api.LA_OP_ATTN_FWD, B, H, S, S, D, torch.float32), dtype=torch.uint8,
                     device="cuda")
    g = api.Graph(lambda: api.attn_fwd(qd, kd, vd, out=o, workspace=ws))
    for _ in range(3):
        o.zero_()
        g.replay()
    torch.cuda.synchronize()
    assert api.get_last_error() == api.LA_OK
    assert_close(o, oracle.attn(q, k, v), torch.float32, "small graph")
