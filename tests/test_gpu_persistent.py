"""The persistent form of the attention kernel (launches with more work items
than SMs): items handed out by ticket, barrier phases and the key/value ring
carried from item to item, inactive items skipped by every role, split
partials, the ticket words in the workspace reused across many launches, and
launches on two streams at the same time (each with its own workspace).
Each case is compared with the fp64 oracle on identical seeded inputs."""
import pytest
import torch

import oracle
import tf32_bound as tb
from gpu_util import assert_close, assert_within_tf32, need_gpu, with_ramp
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


def test_ticket_words_reused_across_launches():
    """70 persistent launches on one workspace (its ticket words reused, each
    launch under a tag of its own): every launch must hand out each item
    exactly once."""
    B, H, S, D = 2, 80, 512, 64
    dtype = torch.bfloat16
    assert _items(B, H, S, dtype, D) > SMS
    q, k, v = inputs.attn_inputs(B, H, S, S, D, dtype, seed=46)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    ws = torch.empty(api.workspace_size(api.LA_OP_ATTN_FWD, B, H, S, S, D, dtype), dtype=torch.uint8, device="cuda")
    first = api.attn_fwd(qd, kd, vd, causal=True, workspace=ws)
    outs = [api.attn_fwd(qd, kd, vd, causal=True, workspace=ws) for _ in range(70)]
    assert api.get_last_error() == api.LA_OK
    for i, o in enumerate(outs):
        assert torch.equal(o, first), f"launch {i}"
    assert_close(first, oracle.attn(q, k, v, causal=True), dtype, "reference launch")


def test_fresh_workspace_with_garbage_ticket_words():
    """A workspace whose first bytes hold leftovers (here: every byte 0xA5,
    and the tag pattern of other launches) needs no clearing: the launch
    claims the words under its own tag."""
    B, H, S, D = 2, 80, 512, 64
    dtype = torch.bfloat16
    q, k, v = inputs.attn_inputs(B, H, S, S, D, dtype, seed=47)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    n = api.workspace_size(api.LA_OP_ATTN_FWD, B, H, S, S, D, dtype)
    want = oracle.attn(q, k, v, causal=True)
    for fill in (0xA5, 0x01, 0xFF):
        ws = torch.full((n,), fill, dtype=torch.uint8, device="cuda")
        o = api.attn_fwd(qd, kd, vd, causal=True, workspace=ws)
        assert api.get_last_error() == api.LA_OK
        assert_close(o, want, dtype, f"workspace filled with {fill:#x}")


@pytest.mark.parametrize("dtype,D", [(torch.bfloat16, 64), (torch.float32, 64)],
                         ids=lambda p: str(p).replace("torch.", ""))
def test_two_streams_at_once(dtype, D):
    """Persistent launches on two streams with no ordering between them, each
    stream with its own workspace (hence its own ticket words), 24 launches
    each, interleaved: every output must equal its stream's first and the
    oracle.  With a ticket counter shared between the streams, items would be
    taken by the wrong launch and rows left unwritten."""
    B, H, S = 2, 80, 512
    assert _items(B, H, S, dtype, D) > SMS
    ins = [inputs.attn_inputs(B, H, S, S, D, dtype, seed=48 + i) for i in range(2)]
    dev = [tuple(t.cuda() for t in x) for x in ins]
    n = api.workspace_size(api.LA_OP_ATTN_FWD, B, H, S, S, D, dtype)
    streams = [torch.cuda.Stream() for _ in range(2)]
    wss = [torch.empty(n, dtype=torch.uint8, device="cuda") for _ in range(2)]
    outs = [[], []]
    torch.cuda.synchronize()
    for it in range(24):
        for i in range(2):
            o = torch.full_like(dev[i][0], float("nan"))
            with torch.cuda.stream(streams[i]):
                api.attn_fwd(*dev[i], causal=True, out=o, workspace=wss[i], stream=streams[i])
            outs[i].append(o)
    torch.cuda.synchronize()
    assert api.get_last_error() == api.LA_OK
    for i in range(2):
        for j, o in enumerate(outs[i]):
            assert torch.equal(o, outs[i][0]), f"stream {i} launch {j}"
        want = oracle.attn(*ins[i], causal=True)
        if dtype == torch.float32:  # early causal rows: the TF32 bound
            q, k, v = (t.numpy() for t in ins[i])
            P = oracle.attn_probs(*ins[i][:2], causal=True)
            assert_within_tf32(outs[i][0], want, tb.attn_bound(q, k, v, P, want, D ** -0.5), f"two streams {i}")
        else:
            assert_close(outs[i][0], want, dtype, f"stream {i}")


@pytest.mark.parametrize("D,S_kv", [(64, 50_000), (128, 24_000)], ids=["D64", "D128"])
def test_causal_items_in_head_groups(D, S_kv):
    """Causal items are numbered by groups of (b, h) pairs whose keys and
    values fill about 32 MB, heaviest first within a group.  bf16 B=1 H=11
    S_q=4096 with S_kv keys of 12.8 / 12.3 MB a pair: groups of two pairs,
    the last one short, 176 or more items in the persistent form.  Values
    carry a ramp over key positions, so an item run twice, skipped or given
    another head's keys moves its rows far beyond the tolerance.  Every head's
    first and last rows of each of several query blocks, and 179 seeded rows."""
    B, H, S_q = 1, 11, 4096
    assert (32 << 20) // (S_kv * D * 2 * 2) == 2  # pairs per group
    assert _items(B, H, S_q, torch.bfloat16, D) > SMS
    q, k, v = inputs.attn_inputs(B, H, S_q, S_kv, D, torch.bfloat16, seed=47 + D)
    v = with_ramp(v, 4.0)
    o = _run(q, k, v, causal=True).cpu()
    edges = [(0, h, i) for h in range(H) for i in (0, 255, 256, 2047, 2048, 3840, 4095)]
    rows = torch.cat([torch.tensor(edges, dtype=torch.int64), inputs.sample_rows(B, H, S_q, n=179, seed=1240 + D)])
    want = oracle.attn_rows(q, k, v, rows, causal=True)
    r = rows.numpy()
    assert_close(o[r[:, 0], r[:, 1], r[:, 2]], want, torch.bfloat16, f"head groups D={D}")
