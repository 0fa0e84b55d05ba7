"""The persistent form of the attention kernel (launches with more work items
than SMs): items handed out by ticket, barrier phases and the key/value ring
carried from item to item, inactive items skipped by every role, split
partials, and the ticket counter's slots reused across many launches.  Each
case is compared with the fp64 oracle on identical seeded inputs."""
import pytest
import torch

import oracle
from gpu_util import assert_close, need_gpu
from layer_attn_fwd_gb300 import api, build, inputs

pytestmark = pytest.mark.gpu

SMS = 152  # a launch with more items than this runs the persistent form


@pytest.fixture(scope="module", autouse=True)
def _lib():
    need_gpu()
    build.build()
    api.load()


def _items(B, H, S_q, dtype, D):
    rows = 128 if (dtype == torch.float32 and D == 128) else 256  # query rows per item
    return B * H * ((S_q + rows - 1) // rows)


def _run(q, k, v, causal, kv_len=None, workspace=None):
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    kl = kv_len.cuda() if kv_len is not None else None
    o = api.attn_fwd(qd, kd, vd, causal=causal, kv_len=kl, workspace=workspace)
    assert api.get_last_error() == api.LA_OK
    return o


CASES = [(torch.float32, 64), (torch.float32, 128), (torch.bfloat16, 128), (torch.float16, 64)]


@pytest.mark.parametrize("dtype,D", CASES, ids=lambda p: str(p).replace("torch.", ""))
@pytest.mark.parametrize("causal", [False, True])
def test_many_items_every_row(dtype, D, causal):
    """B=4 H=40 S=512 (320 or 640 items, two to five per CTA), every row."""
    B, H, S = 4, 40, 512
    assert _items(B, H, S, dtype, D) > SMS
    q, k, v = inputs.attn_inputs(B, H, S, S, D, dtype, seed=41 + D)
    o = _run(q, k, v, causal)
    assert_close(o, oracle.attn(q, k, v, causal=causal), dtype, f"persistent {dtype} D={D}")


@pytest.mark.parametrize("dtype,D", [(torch.float32, 64), (torch.bfloat16, 128)],
                         ids=lambda p: str(p).replace("torch.", ""))
def test_inactive_items_between_active_ones(dtype, D):
    """Key padding with empty batches: some items have no visible key at all
    (zero rows, no loads, no MMAs), between items that do."""
    B, H, S = 8, 20, 512
    assert _items(B, H, S, dtype, D) > SMS
    q, k, v = inputs.attn_inputs(B, H, S, S, D, dtype, seed=43)
    kv_len = torch.tensor([512, 0, 1, 300, 0, 129, 512, 0], dtype=torch.int32)
    o = _run(q, k, v, True, kv_len=kv_len)
    assert_close(o, oracle.attn(q, k, v, causal=True, kv_len=kv_len), dtype, "inactive items")
    for b in (1, 4, 7):
        assert torch.count_nonzero(o[b]).item() == 0


def test_persistent_with_split_partials():
    """B=1 H=40 S_q=1024 S_kv=8192 bf16: more items than SMs and a split key
    range; sampled rows against the oracle and against the unsplit launch."""
    B, H, S_q, S_kv, D = 1, 40, 1024, 8192, 64
    dtype = torch.bfloat16
    assert api.workspace_size(api.LA_OP_ATTN_FWD, B, H, S_q, S_kv, D, dtype) > 0  # the plan splits
    q, k, v = inputs.attn_inputs(B, H, S_q, S_kv, D, dtype, seed=44)
    o_split = _run(q, k, v, False).cpu()
    o_one = _run(q, k, v, False, workspace=torch.empty(0, dtype=torch.uint8, device="cuda")).cpu()
    rows = inputs.sample_rows(B, H, S_q, n=256, seed=45, forced=(0, 255, 256, 1023))
    r = rows.numpy()
    want = oracle.attn_rows(q, k, v, rows, causal=False)
    assert_close(o_split[r[:, 0], r[:, 1], r[:, 2]], want, dtype, "split")
    assert_close(o_one[r[:, 0], r[:, 1], r[:, 2]], want, dtype, "unsplit")


def test_ticket_slots_reused_across_launches():
    """70 persistent launches (the ticket counter has 64 slots, taken in
    turn): every launch must hand out each item exactly once."""
    B, H, S, D = 2, 80, 512, 64
    dtype = torch.bfloat16
    assert _items(B, H, S, dtype, D) > SMS
    q, k, v = inputs.attn_inputs(B, H, S, S, D, dtype, seed=46)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    first = api.attn_fwd(qd, kd, vd, causal=True)
    outs = [api.attn_fwd(qd, kd, vd, causal=True) for _ in range(70)]
    assert api.get_last_error() == api.LA_OK
    for i, o in enumerate(outs):
        assert torch.equal(o, first), f"launch {i}"
    assert_close(first, oracle.attn(q, k, v, causal=True), dtype, "reference launch")
