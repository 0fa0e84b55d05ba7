"""Failure detection on the GPU without a fault: a load that is never issued
makes the kernel's bounded waits run out; the status comes back as
LA_ERR_TIMEOUT, the context stays usable and the next call is correct."""
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


def test_bounded_wait_reports_timeout_and_context_survives():
    q, k, v = inputs.attn_inputs(1, 1, 128, 128, 64, torch.bfloat16, seed=71)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    assert api.get_last_error() == api.LA_OK
    api.debug_inject_timeout(1)
    api.attn_fwd(qd, kd, vd, causal=False)   # launches; its loads are never issued
    assert api.get_last_error() == api.LA_ERR_TIMEOUT
    assert api.get_last_error() == api.LA_OK  # the word was cleared
    o = api.attn_fwd(qd, kd, vd, causal=False)
    assert api.get_last_error() == api.LA_OK
    assert_close(o, oracle.attn(q, k, v), torch.bfloat16, "after timeout")


def test_withdrawn_request_does_nothing():
    q, k, v = inputs.attn_inputs(1, 1, 64, 64, 64, torch.bfloat16, seed=72)
    api.debug_inject_timeout(1)
    api.debug_inject_timeout(0)
    o = api.attn_fwd(q.cuda(), k.cuda(), v.cuda())
    assert api.get_last_error() == api.LA_OK
    assert_close(o, oracle.attn(q, k, v), torch.bfloat16)


def test_timeout_in_persistent_form_then_correct_launches():
    """The same on a launch with more work items than SMs (the persistent
    form): every CTA still draws its tickets to the end, so the launches
    after the timed-out one (reusing the same workspace, hence the same
    ticket words) hand out each item exactly once."""
    B, H, S, D = 2, 80, 512, 64  # 320 items
    q, k, v = inputs.attn_inputs(B, H, S, S, D, torch.bfloat16, seed=73)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    assert api.get_last_error() == api.LA_OK
    ws = torch.empty(api.workspace_size(api.LA_OP_ATTN_FWD, B, H, S, S, D, torch.bfloat16), dtype=torch.uint8,
                     device="cuda")
    api.debug_inject_timeout(1)
    api.attn_fwd(qd, kd, vd, causal=True, workspace=ws)
    assert api.get_last_error() == api.LA_ERR_TIMEOUT
    want = oracle.attn(q, k, v, causal=True)
    for i in range(66):
        o = api.attn_fwd(qd, kd, vd, causal=True, workspace=ws)
        if i in (0, 1, 65):
            assert api.get_last_error() == api.LA_OK
            assert_close(o, want, torch.bfloat16, f"launch {i} after timeout")
    assert api.get_last_error() == api.LA_OK
