"""The attention entry point that allocates nothing (la_attn_fwd_noalloc).

Some callers cannot allocate device memory -- a plugin interface that passes
only input and output tensors, a service that fixes its device memory at
start-up, a latency-critical loop that must not call cudaMalloc -- so this
entry keeps its scratch in a static device array inside the library.  Its
output must match the workspace-taking la_attn_fwd within the parity
tolerance, on two calls in a row (the array keeps the previous call's
contents), and it must refuse a call whose scratch exceeds the array.
This file is collected last; it runs alone or after the rest of the suite.
"""
import ctypes

import pytest
import torch

from gpu_util import TOL, assert_close, need_gpu
from layer_attn_fwd_gb300 import api, build, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    need_gpu()
    build.build()
    api.load()


def _noalloc(lib, q, k, v, o, causal, dt):
    B, H, S_q, D = q.shape
    return lib.la_attn_fwd_noalloc(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
                                   ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(o.data_ptr()), B, H, S_q,
                                   k.shape[2], D, int(causal), 1.0 / D ** 0.5, None, dt,
                                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


# (dtype, B, H, S_q, S_kv, D, causal): the first case splits the key range
# (partials in the static array); the fp32 case keeps V transposed there.
CASES = [(torch.bfloat16, 1, 2, 256, 4173, 128, True), (torch.float16, 2, 2, 300, 300, 64, False),
         (torch.float32, 1, 2, 300, 700, 64, True)]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{str(c[0]).split('.')[-1]}-{c[3]}x{c[4]}-D{c[5]}")
def test_noalloc_matches_workspace_entry(case):
    dt, B, H, S_q, S_kv, D, causal = case
    lib = api.load()
    q, k, v = (t.cuda() for t in inputs.attn_inputs(B, H, S_q, S_kv, D, dt, seed=81))
    ref = api.attn_fwd(q, k, v, causal=causal)
    assert api.get_last_error() == api.LA_OK
    for call in range(2):  # two calls in a row share the static scratch
        o = torch.full_like(q, float("nan"))
        st = _noalloc(lib, q, k, v, o, causal, api._DT[dt])
        assert st == api.LA_OK, api.status_string(st)
        assert api.get_last_error() == api.LA_OK
        assert_close(o, ref.double().cpu().numpy(), dt, f"call {call + 1}")


@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16], ids=lambda d: str(d).split(".")[-1])
def test_noalloc_without_keys_writes_zero_rows(dt):
    """S_kv = 0: every row is a zero row, for fp32 as well (no V to transpose)."""
    lib = api.load()
    q = torch.randn(1, 2, 40, 64, device="cuda").to(dt)
    kv = torch.empty(1, 2, 0, 64, device="cuda", dtype=dt)
    o = torch.full_like(q, float("nan"))
    assert _noalloc(lib, q, kv, kv, o, False, api._DT[dt]) == api.LA_OK
    assert api.get_last_error() == api.LA_OK
    assert torch.count_nonzero(o).item() == 0


def test_noalloc_refuses_scratch_beyond_its_array():
    lib = api.load()
    # fp32 with V transposed needs 8*8*64*2048*4 = 32 MiB > 16 MiB: refused before any launch
    q = torch.zeros(8, 8, 2048, 64, device="cuda")
    o = torch.full_like(q, 7.0)
    st = _noalloc(lib, q, q, q, o, True, api.LA_F32)
    assert st == api.LA_ERR_WORKSPACE
    assert torch.all(o == 7.0)
