"""The C ABI on a machine without a GPU: the library builds, loads, exports
every entry point declared in include/layerattn.h, and rejects invalid calls
on the host before touching any device.  No compute call is made here."""
import ctypes
import os
import re

import pytest

from layer_attn_fwd_gb300 import api, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "layerattn.h")

# plausible, 256-byte aligned addresses that validation must reject before use
FAKE = ctypes.c_void_p(0x7f0000000000)


@pytest.fixture(scope="module")
def lib():
    build.build()
    return api.load()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(la_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert {"la_qkv_proj", "la_attn_fwd", "la_attn_chunked", "la_layer_attn", "la_workspace_size",
            "la_get_last_error", "la_status_string"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_debug_hook_validates_mode(lib):
    assert lib.la_debug_inject_timeout(7) == api.LA_ERR_INVALID
    assert lib.la_debug_inject_timeout(0) == api.LA_OK


def test_status_strings(lib):
    for s in range(7):
        assert api.status_string(s).startswith("LA_")
    assert "unknown" in api.status_string(99)


def _attn(lib, q=FAKE, k=FAKE, v=FAKE, o=FAKE, B=1, H=1, S_q=16, S_kv=16, D=64, causal=0, scale=0.125,
          kv_len=None, dt=api.LA_BF16, ws=None, ws_bytes=0):
    return lib.la_attn_fwd(q, k, v, o, B, H, S_q, S_kv, D, causal, scale, kv_len, dt, ws, ws_bytes, None)


def test_fp32_attention_needs_workspace(lib):
    assert _attn(lib, dt=api.LA_F32) == api.LA_ERR_WORKSPACE
    assert _attn(lib, dt=api.LA_F32, ws=FAKE, ws_bytes=api.fp32_vt_bytes(1, 1, 16, 64) - 1) == api.LA_ERR_WORKSPACE


def test_attn_fwd_rejects_bad_arguments(lib):
    assert _attn(lib, q=None) == api.LA_ERR_INVALID
    assert _attn(lib, o=None) == api.LA_ERR_INVALID
    assert _attn(lib, B=0) == api.LA_ERR_INVALID
    assert _attn(lib, H=-1) == api.LA_ERR_INVALID
    assert _attn(lib, S_q=-1) == api.LA_ERR_INVALID
    assert _attn(lib, S_kv=-5) == api.LA_ERR_INVALID
    assert _attn(lib, scale=0.0) == api.LA_ERR_INVALID
    assert _attn(lib, scale=-1.0) == api.LA_ERR_INVALID
    assert _attn(lib, scale=float("inf")) == api.LA_ERR_INVALID
    assert _attn(lib, scale=float("nan")) == api.LA_ERR_INVALID
    assert _attn(lib, dt=7) == api.LA_ERR_INVALID
    assert _attn(lib, q=ctypes.c_void_p(0x7f0000000008)) == api.LA_ERR_INVALID   # not 16-byte aligned
    assert _attn(lib, kv_len=ctypes.c_void_p(0x7f0000000002)) == api.LA_ERR_INVALID
    assert _attn(lib, D=96) == api.LA_ERR_UNSUPPORTED
    assert _attn(lib, D=32) == api.LA_ERR_UNSUPPORTED
    assert _attn(lib, B=300, H=300) == api.LA_ERR_UNSUPPORTED                     # B*H > grid limit


def test_qkv_proj_rejects_bad_arguments(lib):
    def call(x=FAKE, W=FAKE, b=None, B=2, S=8, dm=128, H=2, qs=1.0, dt=api.LA_F32):
        return lib.la_qkv_proj(x, W, b, FAKE, FAKE, FAKE, B, S, dm, H, qs, dt, None, 0, None)
    assert call(x=None) == api.LA_ERR_INVALID
    assert call(dm=129, H=2) == api.LA_ERR_INVALID        # d_model not a multiple of H
    assert call(dm=192, H=2) == api.LA_ERR_UNSUPPORTED    # D = 96
    assert call(S=-1) == api.LA_ERR_INVALID
    assert call(qs=float("nan")) == api.LA_ERR_INVALID
    assert call(b=ctypes.c_void_p(0x7f0000000001)) == api.LA_ERR_INVALID
    assert call() == api.LA_ERR_WORKSPACE                 # fp32 transposes the weight into ws


def test_layer_attn_checks_workspace_before_launch(lib):
    need = api.workspace_size(api.LA_OP_LAYER_ATTN, 8, 8, 512, 512, 64, api.torch.float32)
    assert need >= 3 * 8 * 512 * 512 * 4
    st = lib.la_layer_attn(FAKE, FAKE, None, FAKE, 8, 512, 512, 8, 0, None, api.LA_F32, FAKE, 3 * 8 * 512 * 512 * 4 - 1,
                           None)
    assert st == api.LA_ERR_WORKSPACE
    st = lib.la_layer_attn(FAKE, FAKE, None, FAKE, 8, 512, 512, 8, 0, None, api.LA_F32, None, need, None)
    assert st == api.LA_ERR_INVALID


def test_chunked_rejects_overflowing_cache_and_keeps_len(lib):
    c = api.la_kv_cache(0x7f0000000000, 0x7f0000100000, 2, 16, 64, 100, 90, api.LA_BF16)
    st = lib.la_attn_chunked(FAKE, FAKE, FAKE, ctypes.byref(c), FAKE, 11, 1, 0.125, None, 0, None)
    assert st == api.LA_ERR_INVALID
    assert c.len == 90
    c.D = 80
    st = lib.la_attn_chunked(FAKE, FAKE, FAKE, ctypes.byref(c), FAKE, 5, 1, 0.125, None, 0, None)
    assert st == api.LA_ERR_UNSUPPORTED
    assert c.len == 90


def test_chunked_fp32_cache_needs_s_max_multiple_of_4(lib):
    """An fp32 cache keeps V transposed, rows S_max long: S_max must keep
    each row 16-byte aligned; the refusal comes before any launch and leaves
    len unchanged."""
    c = api.la_kv_cache(0x7f0000000000, 0x7f0000100000, 2, 16, 64, 102, 40, api.LA_F32)
    st = lib.la_attn_chunked(FAKE, FAKE, FAKE, ctypes.byref(c), FAKE, 8, 1, 0.125, None, 0, None)
    assert st == api.LA_ERR_INVALID
    assert c.len == 40


def test_workspace_sizes(lib):
    bad = ctypes.c_size_t(-1).value
    assert lib.la_workspace_size(api.LA_OP_ATTN_FWD, 1, 1, 16, 16, 96, api.LA_BF16) == bad
    assert lib.la_workspace_size(9, 1, 1, 16, 16, 64, api.LA_BF16) == bad
    assert lib.la_workspace_size(api.LA_OP_LAYER_ATTN, 1, 1, 16, 32, 64, api.LA_BF16) == bad
    # short key ranges never split; half precision needs only the 256 bytes of
    # the persistent scheduling's ticket words
    assert lib.la_workspace_size(api.LA_OP_ATTN_FWD, 8, 8, 512, 512, 64, api.LA_BF16) == 256
    # fp32 also holds V transposed for the TF32 tensor cores
    assert lib.la_workspace_size(api.LA_OP_ATTN_FWD, 8, 8, 512, 512, 64, api.LA_F32) == \
        api.fp32_vt_bytes(8, 8, 512, 64) + 256
    assert lib.la_workspace_size(api.LA_OP_QKV_PROJ, 8, 8, 512, 512, 64, api.LA_F32) == 3 * 512 * 512 * 4
    assert lib.la_workspace_size(api.LA_OP_QKV_PROJ, 8, 8, 512, 512, 64, api.LA_BF16) == 0
    # the chunked mode needs no V^T scratch: an fp32 cache holds V transposed
    assert lib.la_workspace_size(api.LA_OP_ATTN_CHUNKED, 8, 8, 512, 512, 64, api.LA_F32) == 256
    # the 100k-token chunked case: partials stay far below the cache itself
    n = lib.la_workspace_size(api.LA_OP_ATTN_CHUNKED, 2, 16, 4096, 100000, 64, api.LA_BF16)
    assert n != bad and n < 2 * 16 * 100000 * 64 * 2 * 4
    # one long row range on a small grid splits, and asks for room for it
    n = lib.la_workspace_size(api.LA_OP_ATTN_FWD, 1, 1, 256, 8192, 128, api.LA_BF16)
    assert n >= 2 * 256 * 128 * 4


def test_out_proj_rejects_bad_arguments(lib):
    def call(a=FAKE, W=FAKE, b=None, y=FAKE, M=64, dm=512, dt=api.LA_BF16, ws=None, nb=0):
        return lib.la_out_proj(a, W, b, y, M, dm, dt, ws, nb, None)
    assert call(a=None) == api.LA_ERR_INVALID
    assert call(y=None) == api.LA_ERR_INVALID
    assert call(M=-1) == api.LA_ERR_INVALID
    assert call(dm=0) == api.LA_ERR_INVALID
    assert call(dt=5) == api.LA_ERR_INVALID
    assert call(dm=96) == api.LA_ERR_UNSUPPORTED           # not a multiple of 64
    assert call(a=ctypes.c_void_p(0x7f0000000004)) == api.LA_ERR_INVALID
    assert call(b=ctypes.c_void_p(0x7f0000000002)) == api.LA_ERR_INVALID
    assert call(dt=api.LA_F32) == api.LA_ERR_WORKSPACE     # fp32 transposes Wo into ws
    assert call(dt=api.LA_F32, ws=FAKE, nb=512 * 512 * 4 - 1) == api.LA_ERR_WORKSPACE
    assert call(M=0, dt=api.LA_F32) == api.LA_OK           # empty: nothing to do, nothing launched


def test_layer_attn_out_checks_workspace_before_launch(lib):
    need = api.workspace_size(api.LA_OP_LAYER_ATTN_OUT, 8, 8, 512, 512, 64, api.torch.float32)
    base = api.workspace_size(api.LA_OP_LAYER_ATTN, 8, 8, 512, 512, 64, api.torch.float32)
    assert need == base + 8 * 512 * 512 * 4 + 512 * 512 * 4     # + merged output + Wo^T
    # the last 256 bytes of `need` hold the attention's ticket words, which a
    # call can do without; one byte short of the rest is refused
    def call(ws=FAKE, nb=need - 256 - 1, Wo=FAKE):
        return lib.la_layer_attn_out(FAKE, FAKE, None, Wo, None, FAKE, 8, 512, 512, 8, 0, None, api.LA_F32, ws, nb,
                                     None)
    assert call() == api.LA_ERR_WORKSPACE
    assert call(ws=None, nb=need) == api.LA_ERR_INVALID
    assert call(Wo=None, nb=need) == api.LA_ERR_INVALID


def test_out_proj_workspace_sizes(lib):
    assert lib.la_workspace_size(api.LA_OP_OUT_PROJ, 1, 8, 4096, 4096, 64, api.LA_F32) == 512 * 512 * 4
    assert lib.la_workspace_size(api.LA_OP_OUT_PROJ, 1, 8, 4096, 4096, 64, api.LA_BF16) == 0
    bf = lib.la_workspace_size(api.LA_OP_LAYER_ATTN_OUT, 8, 8, 512, 512, 64, api.LA_BF16)
    assert bf == lib.la_workspace_size(api.LA_OP_LAYER_ATTN, 8, 8, 512, 512, 64, api.LA_BF16) + 8 * 512 * 512 * 2


def test_layernorm_rejects_bad_arguments(lib):
    def call(x=FAKE, g=FAKE, b=FAKE, y=FAKE, M=16, d=512, eps=1e-5, dt=api.LA_F32):
        return lib.la_layernorm(x, g, b, y, M, d, eps, dt, None)
    assert call(x=None) == api.LA_ERR_INVALID
    assert call(g=None) == api.LA_ERR_INVALID
    assert call(b=None) == api.LA_ERR_INVALID
    assert call(M=-1) == api.LA_ERR_INVALID
    assert call(eps=-1.0) == api.LA_ERR_INVALID
    assert call(eps=float("nan")) == api.LA_ERR_INVALID
    assert call(dt=9) == api.LA_ERR_INVALID
    assert call(d=96) == api.LA_ERR_UNSUPPORTED
    assert call(g=ctypes.c_void_p(0x7f0000000008)) == api.LA_ERR_INVALID
    assert call(M=0) == api.LA_OK


def test_layer_attn_ln_checks_arguments_before_launch(lib):
    need = api.workspace_size(api.LA_OP_LAYER_ATTN_LN, 8, 8, 512, 512, 64, api.torch.float32)
    assert need == api.workspace_size(api.LA_OP_LAYER_ATTN_OUT, 8, 8, 512, 512, 64, api.torch.float32) \
        + 8 * 512 * 8                                             # + the row statistics (mean, rstd)
    def call(g=FAKE, eps=1e-5, Wo=FAKE, bo=None, nb=need - 256 - 1):  # short of all but the ticket words
        return lib.la_layer_attn_ln(FAKE, g, FAKE, eps, FAKE, None, Wo, bo, FAKE, 8, 512, 512, 8, 0, None,
                                    api.LA_F32, FAKE, nb, None)
    assert call() == api.LA_ERR_WORKSPACE
    assert call(g=None, nb=need) == api.LA_ERR_INVALID
    assert call(eps=-0.5, nb=need) == api.LA_ERR_INVALID
    assert call(Wo=None, bo=FAKE, nb=need) == api.LA_ERR_INVALID   # a bias without a weight


def test_checked_build_exports_and_identifies_itself(lib):
    """liblayerattn_checked.so (bounds checks on every global store) exports
    the same entry points; each library says which it is."""
    checked = ctypes.CDLL(build.LIB_CHECKED)
    for n in _declared():
        assert hasattr(checked, n), n
    checked.la_is_checked_build.restype = ctypes.c_int
    assert checked.la_is_checked_build() == 1
    assert lib.la_is_checked_build() == 0
    assert lib.la_debug_shrink_output_extent(3) == api.LA_ERR_INVALID
    assert lib.la_debug_shrink_output_extent(0) == api.LA_OK
