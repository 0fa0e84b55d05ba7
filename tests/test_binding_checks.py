"""The Python binding checks every operand's shape and element type before
anything touches a device (the C ABI takes plain pointers and cannot see a
tensor's size).  CPU only: wrong operands raise TypeError/ValueError naming
the operand; right ones get as far as the device check."""
import pytest
import torch

from layer_attn_fwd_gb300 import api

F32, BF16 = torch.float32, torch.bfloat16


def _t(*shape, dtype=F32):
    return torch.zeros(*shape, dtype=dtype)


def test_attn_fwd_operands():
    q, k, v = _t(1, 2, 8, 64), _t(1, 2, 16, 64), _t(1, 2, 16, 64)
    with pytest.raises(ValueError, match="v: shape"):
        api.attn_fwd(q, k, _t(1, 2, 15, 64))
    with pytest.raises(TypeError, match="k: dtype"):
        api.attn_fwd(q, _t(1, 2, 16, 64, dtype=BF16), v)
    with pytest.raises(TypeError, match="kv_len: dtype"):
        api.attn_fwd(q, k, v, kv_len=torch.zeros(1, dtype=torch.int64))
    with pytest.raises(ValueError, match="kv_len: shape"):
        api.attn_fwd(q, k, v, kv_len=torch.zeros(2, dtype=torch.int32))
    with pytest.raises(ValueError, match="out: shape"):
        api.attn_fwd(q, k, v, out=_t(1, 2, 16, 64))
    with pytest.raises(ValueError, match="CUDA"):
        api.attn_fwd(q, k, v)
    with pytest.raises(ValueError, match="v: shape"):
        api.attn_fwd_noalloc(q, k, _t(1, 2, 16, 32))


def test_projection_operands():
    x = _t(2, 8, 128)
    with pytest.raises(ValueError, match="Wqkv: shape"):
        api.qkv_proj(x, _t(128, 256), None, 2)
    with pytest.raises(TypeError, match="Wqkv: dtype"):
        api.qkv_proj(x, _t(128, 384, dtype=BF16), None, 2)
    with pytest.raises(ValueError, match="bqkv: shape"):
        api.qkv_proj(x, _t(128, 384), _t(128), 2)
    with pytest.raises(ValueError, match="CUDA"):
        api.qkv_proj(x, _t(128, 384), _t(384), 2)
    with pytest.raises(ValueError, match="Wo: shape"):
        api.out_proj(_t(16, 128), _t(128, 64))
    with pytest.raises(TypeError, match="bo: dtype"):
        api.out_proj(_t(16, 128), _t(128, 128), _t(128, dtype=BF16))


def test_sublayer_operands():
    x, W = _t(2, 8, 128), _t(128, 384)
    with pytest.raises(ValueError, match="Wqkv: shape"):
        api.layer_attn(x, _t(384, 128), None, 2)
    with pytest.raises(ValueError, match="out: shape"):
        api.layer_attn(x, W, None, 2, out=_t(2, 8, 64))
    with pytest.raises(ValueError, match="Wo: shape"):
        api.layer_attn_out(x, W, None, _t(128, 127), None, 2)
    with pytest.raises(ValueError, match="gamma: shape"):
        api.layer_attn_ln(x, _t(64), _t(128), W, None, None, None, 2)
    with pytest.raises(TypeError, match="beta: dtype"):
        api.layer_attn_ln(x, _t(128), _t(128, dtype=BF16), W, None, None, None, 2)
    with pytest.raises(ValueError, match="gamma: shape"):
        api.layernorm(_t(4, 128), _t(127), _t(128))
    with pytest.raises(ValueError, match="CUDA"):
        api.layernorm(_t(4, 128), _t(128), _t(128))


def test_chunked_operands_match_the_cache():
    cache = api.KVCache(1, 2, 64, 64, F32, device="cpu")
    q = _t(1, 2, 16, 64)
    with pytest.raises(ValueError, match="k_chunk: shape"):
        api.attn_chunked(q, _t(1, 2, 8, 64), _t(1, 2, 16, 64), cache)
    with pytest.raises(TypeError, match="q_chunk: dtype"):
        api.attn_chunked(q.to(BF16), _t(1, 2, 16, 64), _t(1, 2, 16, 64), cache)
    with pytest.raises(ValueError, match="q_chunk: shape"):
        api.attn_chunked(_t(1, 3, 16, 64), _t(1, 2, 16, 64), _t(1, 2, 16, 64), cache)
