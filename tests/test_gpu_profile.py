"""Per-launch device timing (la_profile_start / la_profile_stop): every
launch of the library bracketed by CUDA events on its stream, names and
times in launch order; launches past the record limit are not recorded and
do not disturb the recorded ones."""
import pytest
import torch

from gpu_util import need_gpu
from layer_attn_fwd_gb300 import api, build, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    need_gpu()
    build.build()
    api.load()


def test_records_each_launch_in_order():
    q, k, v = (t.cuda() for t in inputs.attn_inputs(1, 4, 256, 8192, 64, torch.bfloat16, seed=140))
    ws = torch.empty(api.workspace_size(api.LA_OP_ATTN_FWD, 1, 4, 256, 8192, 64, torch.bfloat16),
                     dtype=torch.uint8, device="cuda")
    api.attn_fwd(q, k, v, workspace=ws)  # first-call set-up outside the records
    torch.cuda.synchronize()
    with api.Profile() as p:
        api.attn_fwd(q, k, v, workspace=ws)  # splits the key range: attention, then the merge
        x, W, b = (t.cuda() for t in inputs.layer_inputs(1, 128, 128, torch.float32, seed=141))
        api.layer_attn(x, W, b, 2)           # fp32: weight transpose, projection, attention
    assert api.get_last_error() == api.LA_OK
    names = [n for n, _ in p.records]
    assert names == ["attn_fwd_kernel", "combine_kernel", "transpose32_kernel", "qkv_proj_kernel",
                     "attn_fwd_kernel"], names
    assert all(0.0 < ms < 100.0 for _, ms in p.records), p.records


def test_launches_past_the_limit_leave_records_alone():
    q, k, v = (t.cuda() for t in inputs.attn_inputs(1, 2, 128, 128, 64, torch.bfloat16, seed=142))
    api.attn_fwd(q, k, v)
    torch.cuda.synchronize()
    with api.Profile(max_launches=2) as p:
        for _ in range(2):
            api.attn_fwd(q, k, v)
        big_q, big_k, big_v = (t.cuda() for t in inputs.attn_inputs(8, 16, 4096, 4096, 64, torch.bfloat16, seed=143))
        for _ in range(3):  # not recorded: these must not stretch the second record
            api.attn_fwd(big_q, big_k, big_v, causal=True)
    assert len(p.records) == 2
    assert all(ms < 0.5 for _, ms in p.records), p.records  # a small launch each, not the long ones after
