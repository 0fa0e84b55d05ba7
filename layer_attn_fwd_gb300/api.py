"""Thin ctypes binding of liblayerattn.so (declared in include/layerattn.h).

Argument marshalling only: every step of the computation runs in the CUDA
library.  Tensors are torch CUDA tensors (PyTorch supplies device memory and
streams); calls go onto ``torch.cuda.current_stream()``.  Workspaces are
allocated here with torch when the caller passes none; the library itself
never allocates.  A missing library raises ``RuntimeError``; there is no CPU
or PyTorch fallback.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "liblayerattn.so")
# the same library with bounds checks on every global store (see layerattn.h)
CHECKED_LIB_PATH = os.path.join(_PKG, "_build", "liblayerattn_checked.so")

LA_OK, LA_ERR_INVALID, LA_ERR_UNSUPPORTED, LA_ERR_WORKSPACE, LA_ERR_CUDA, LA_ERR_TIMEOUT, LA_ERR_INTERNAL = range(7)
LA_F32, LA_BF16, LA_F16 = 0, 1, 2
(LA_OP_ATTN_FWD, LA_OP_ATTN_CHUNKED, LA_OP_LAYER_ATTN, LA_OP_QKV_PROJ, LA_OP_OUT_PROJ, LA_OP_LAYER_ATTN_OUT,
 LA_OP_LAYER_ATTN_LN) = range(7)

_DT = {torch.float32: LA_F32, torch.bfloat16: LA_BF16, torch.float16: LA_F16}

_lock = threading.Lock()
_lib = None


class LayerAttnError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


class la_kv_cache(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("B", ctypes.c_int), ("H", ctypes.c_int),
                ("D", ctypes.c_int), ("S_max", ctypes.c_int), ("len", ctypes.c_int), ("dtype", ctypes.c_int)]


def load(path: str | None = None, reload: bool = False):
    """Load the library (once; with reload, switch to `path`, e.g.
    CHECKED_LIB_PATH).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None and not reload:
            return _lib
        path = path or LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(f"liblayerattn.so not built ({path}); run layer_attn_fwd_gb300.build.build()")
        lib = ctypes.CDLL(path)
        P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.la_qkv_proj.argtypes = [P, P, P, P, P, P, I, I, I, I, F, I, P, Z, P]
        lib.la_attn_fwd.argtypes = [P, P, P, P, I, I, I, I, I, I, F, P, I, P, Z, P]
        lib.la_attn_fwd_noalloc.argtypes = [P, P, P, P, I, I, I, I, I, I, F, P, I, P]
        lib.la_attn_fwd_noalloc.restype = I
        lib.la_attn_chunked.argtypes = [P, P, P, ctypes.POINTER(la_kv_cache), P, I, I, F, P, Z, P]
        lib.la_layer_attn.argtypes = [P, P, P, P, I, I, I, I, I, P, I, P, Z, P]
        lib.la_out_proj.argtypes = [P, P, P, P, I, I, I, P, Z, P]
        lib.la_layer_attn_out.argtypes = [P, P, P, P, P, P, I, I, I, I, I, P, I, P, Z, P]
        lib.la_layernorm.argtypes = [P, P, P, P, I, I, F, I, P]
        lib.la_layer_attn_ln.argtypes = [P, P, P, F, P, P, P, P, P, I, I, I, I, I, P, I, P, Z, P]
        lib.la_workspace_size.argtypes = [I, I, I, I, I, I, I]
        lib.la_workspace_size.restype = Z
        lib.la_get_last_error.argtypes = [P]
        lib.la_last_error_detail.argtypes = []
        lib.la_last_error_detail.restype = ctypes.c_uint32
        lib.la_debug_inject_timeout.argtypes = [I]
        lib.la_debug_inject_timeout.restype = I
        lib.la_debug_shrink_output_extent.argtypes = [I]
        lib.la_debug_shrink_output_extent.restype = I
        lib.la_is_checked_build.argtypes = []
        lib.la_is_checked_build.restype = I
        lib.la_prepare_weight.argtypes = [P, P, I, I, I, P]
        lib.la_prepare_weight.restype = I
        lib.la_layer_attn_prepared.argtypes = [P, P, P, F, P, P, P, P, P, I, I, I, I, I, P, I, P, Z, P]
        lib.la_layer_attn_prepared.restype = I
        lib.la_profile_start.argtypes = [I]
        lib.la_profile_start.restype = I
        lib.la_profile_stop.argtypes = [ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_float), I]
        lib.la_profile_stop.restype = I
        lib.la_status_string.argtypes = [I]
        lib.la_status_string.restype = ctypes.c_char_p
        for name in ("la_qkv_proj", "la_attn_fwd", "la_attn_chunked", "la_layer_attn", "la_out_proj",
                     "la_layer_attn_out", "la_layernorm", "la_layer_attn_ln", "la_get_last_error"):
            getattr(lib, name).restype = I
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().la_status_string(int(status)).decode()


def _check(status, where):
    if status != LA_OK:
        raise LayerAttnError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dt(t):
    try:
        return _DT[t.dtype]
    except KeyError:
        raise TypeError(f"unsupported dtype {t.dtype}") from None


def _spec(t, name, shape=None, dtype=None):
    """t: a tensor of exactly `shape` and `dtype` (None: not checked).  The
    library takes plain pointers and cannot see a tensor's size, so every
    entry point checks each operand's shape and type here, before anything
    touches a device: a short weight or a wider element type would make a
    kernel read past a buffer."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")


def _spec_opt(t, name, shape, dtype):
    if t is not None:
        _spec(t, name, shape, dtype)


def _kvlen_spec(kv_len, B):
    if kv_len is not None:
        _spec(kv_len, "kv_len", (B,), torch.int32)


def _need(t, name, dev=True):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if dev and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def workspace_size(op, B, H, S_q, S_kv, D, dtype) -> int:
    n = load().la_workspace_size(int(op), B, H, S_q, S_kv, D, _DT[dtype])
    if n == ctypes.c_size_t(-1).value:
        raise ValueError("workspace_size: invalid arguments")
    return int(n)


def _workspace(nbytes, device, ws):
    if ws is not None:
        return ws
    if nbytes == 0:
        return None
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def qkv_proj(x, Wqkv, bqkv, H, q_scale=1.0, out=None, workspace=None, stream=None):
    """x [B,S,d], Wqkv [d,3d], bqkv [3d] or None -> q, k, v [B,H,S,D]."""
    _spec(x, "x")
    if x.dim() != 3:
        raise ValueError("x must be [B, S, d_model]")
    B, S, dm = x.shape
    D = dm // H if H > 0 else 0
    _spec(Wqkv, "Wqkv", (dm, 3 * dm), x.dtype)
    _spec_opt(bqkv, "bqkv", (3 * dm,), x.dtype)
    if out is not None:
        for t, n in zip(out, "qkv"):
            _spec(t, n, (B, H, S, D), x.dtype)
    for t, n in ((x, "x"), (Wqkv, "Wqkv")):
        _need(t, n)
    if bqkv is not None:
        _need(bqkv, "bqkv")
    if out is None:
        out = tuple(torch.empty(B, H, S, D, dtype=x.dtype, device=x.device) for _ in range(3))
    q, k, v = out
    if workspace is None and D in (64, 128) and x.dtype in _DT:
        workspace = _workspace(workspace_size(LA_OP_QKV_PROJ, B, H, S, S, D, x.dtype), x.device, None)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().la_qkv_proj(_ptr(x), _ptr(Wqkv), _ptr(bqkv), _ptr(q), _ptr(k), _ptr(v), B, S, dm, H,
                              float(q_scale), _dt(x), _ptr(workspace), nbytes, _stream(stream)), "la_qkv_proj")
    return q, k, v


def fp32_vt_bytes(B, H, S_kv, D):
    """Workspace an fp32 attention call needs at least (V transposed for the
    TF32 tensor cores): B*H*D*round_up(S_kv, 4)*4 rounded up to 256."""
    n = B * H * D * ((S_kv + 3) // 4 * 4) * 4
    return (n + 255) // 256 * 256


def _attn_spec(q, k, v, kv_len, out):
    _spec(q, "q")
    if q.dim() != 4:
        raise ValueError("q must be [B, H, S_q, D]")
    B, H, S_q, D = q.shape
    _spec(k, "k", None, q.dtype)
    if k.dim() != 4:
        raise ValueError("k must be [B, H, S_kv, D]")
    S_kv = k.shape[2]
    _spec(k, "k", (B, H, S_kv, D), q.dtype)
    _spec(v, "v", (B, H, S_kv, D), q.dtype)
    _kvlen_spec(kv_len, B)
    _spec_opt(out, "out", (B, H, S_q, D), q.dtype)
    return B, H, S_q, D, S_kv


def attn_fwd(q, k, v, causal=False, scale=None, kv_len=None, out=None, workspace=None, stream=None):
    """softmax(scale q k^T) v: q [B,H,S_q,D], k/v [B,H,S_kv,D] -> [B,H,S_q,D]."""
    B, H, S_q, D, S_kv = _attn_spec(q, k, v, kv_len, out)
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    if kv_len is not None:
        _need(kv_len, "kv_len")
    o = torch.empty_like(q) if out is None else out
    if workspace is None and D in (64, 128) and q.dtype in _DT:
        workspace = _workspace(workspace_size(LA_OP_ATTN_FWD, B, H, S_q, S_kv, D, q.dtype), q.device, None)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().la_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, H, S_q, S_kv, D, int(bool(causal)), scale,
                              _ptr(kv_len), _dt(q), _ptr(workspace), nbytes, _stream(stream)), "la_attn_fwd")
    return o


def attn_fwd_noalloc(q, k, v, causal=False, scale=None, kv_len=None, out=None, stream=None):
    """attn_fwd for callers that cannot allocate: the library's own static
    16 MiB device scratch stands in for the workspace (see layerattn.h)."""
    B, H, S_q, D, S_kv = _attn_spec(q, k, v, kv_len, out)
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n)
    if kv_len is not None:
        _need(kv_len, "kv_len")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    o = torch.empty_like(q) if out is None else out
    _check(load().la_attn_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, H, S_q, S_kv, D, int(bool(causal)),
                                      scale, _ptr(kv_len), _dt(q), _stream(stream)), "la_attn_fwd_noalloc")
    return o


class KVCache:
    """Caller-owned growing key/value cache for the chunked mode: k
    [B,H,S_max,D]; v the same for bf16/fp16 and transposed, [B,H,D,S_max],
    for fp32 (S_max then rounded up to a multiple of 4)."""

    def __init__(self, B, H, S_max, D, dtype, device="cuda"):
        if dtype == torch.float32:
            S_max = (S_max + 3) // 4 * 4
        self.k = torch.empty(B, H, S_max, D, dtype=dtype, device=device)
        if dtype == torch.float32:
            self.v = torch.empty(B, H, D, S_max, dtype=dtype, device=device)
        else:
            self.v = torch.empty(B, H, S_max, D, dtype=dtype, device=device)
        self.c = la_kv_cache(self.k.data_ptr(), self.v.data_ptr(), B, H, D, S_max, 0, _DT[dtype])

    @property
    def len(self):
        return self.c.len

    def reset(self):
        self.c.len = 0


def attn_chunked(q_chunk, k_chunk, v_chunk, cache: KVCache, causal=True, scale=None, out=None, workspace=None,
                 stream=None):
    """Append this window's k/v to the cache, then attend q_chunk to the cache."""
    c = cache.c
    dtype = cache.k.dtype
    _spec(q_chunk, "q_chunk", None, dtype)
    if q_chunk.dim() != 4:
        raise ValueError("q_chunk must be [B, H, chunk, D]")
    shape = (c.B, c.H, q_chunk.shape[2], c.D)
    for t, n in ((q_chunk, "q_chunk"), (k_chunk, "k_chunk"), (v_chunk, "v_chunk")):
        _spec(t, n, shape, dtype)
    _spec_opt(out, "out", shape, dtype)
    for t, n in ((q_chunk, "q_chunk"), (k_chunk, "k_chunk"), (v_chunk, "v_chunk")):
        _need(t, n)
    B, H, C, D = q_chunk.shape
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    o = torch.empty_like(q_chunk) if out is None else out
    if workspace is None:
        workspace = _workspace(workspace_size(LA_OP_ATTN_CHUNKED, B, H, C, cache.c.S_max, D, q_chunk.dtype),
                               q_chunk.device, None)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().la_attn_chunked(_ptr(q_chunk), _ptr(k_chunk), _ptr(v_chunk), ctypes.byref(cache.c), _ptr(o), C,
                                  int(bool(causal)), scale, _ptr(workspace), nbytes, _stream(stream)),
           "la_attn_chunked")
    return o


def _layer_spec(x, Wqkv, bqkv, H, kv_len, out):
    _spec(x, "x")
    if x.dim() != 3:
        raise ValueError("x must be [B, S, d_model]")
    B, S, dm = x.shape
    _spec(Wqkv, "Wqkv", (dm, 3 * dm), x.dtype)
    _spec_opt(bqkv, "bqkv", (3 * dm,), x.dtype)
    _kvlen_spec(kv_len, B)
    _spec_opt(out, "out", (B, S, dm), x.dtype)
    return B, S, dm, (dm // H if H > 0 else 0)


def layer_attn(x, Wqkv, bqkv, H, causal=False, kv_len=None, out=None, workspace=None, stream=None):
    """Projection + per-head attention + head merge: x [B,S,d] -> [B,S,d]."""
    B, S, dm, D = _layer_spec(x, Wqkv, bqkv, H, kv_len, out)
    _need(x, "x")
    o = torch.empty_like(x) if out is None else out
    if workspace is None:
        workspace = _workspace(workspace_size(LA_OP_LAYER_ATTN, B, H, S, S, D, x.dtype), x.device, None)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().la_layer_attn(_ptr(x), _ptr(Wqkv), _ptr(bqkv), _ptr(o), B, S, dm, H, int(bool(causal)),
                                _ptr(kv_len), _dt(x), _ptr(workspace), nbytes, _stream(stream)), "la_layer_attn")
    return o


def out_proj(a, Wo, bo=None, out=None, workspace=None, stream=None):
    """a [..., d] (row-major), Wo [d, d], bo [d] or None -> a Wo + bo."""
    _spec(a, "a")
    dm = a.shape[-1] if a.dim() > 0 else 0
    _spec(Wo, "Wo", (dm, dm), a.dtype)
    _spec_opt(bo, "bo", (dm,), a.dtype)
    _spec_opt(out, "out", tuple(a.shape), a.dtype)
    for t, n in ((a, "a"), (Wo, "Wo")):
        _need(t, n)
    if bo is not None:
        _need(bo, "bo")
    M = a.numel() // dm if dm > 0 else 0
    y = torch.empty_like(a) if out is None else out
    if workspace is None and dm % 64 == 0 and dm > 0 and a.dtype in _DT:
        workspace = _workspace(workspace_size(LA_OP_OUT_PROJ, 1, dm // 64, M, M, 64, a.dtype), a.device, None)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().la_out_proj(_ptr(a), _ptr(Wo), _ptr(bo), _ptr(y), M, dm, _dt(a), _ptr(workspace), nbytes,
                              _stream(stream)), "la_out_proj")
    return y


def layer_attn_out(x, Wqkv, bqkv, Wo, bo, H, causal=False, kv_len=None, out=None, workspace=None, stream=None):
    """The sublayer with its output projection: x [B,S,d] -> [B,S,d]."""
    B, S, dm, D = _layer_spec(x, Wqkv, bqkv, H, kv_len, out)
    _spec(Wo, "Wo", (dm, dm), x.dtype)
    _spec_opt(bo, "bo", (dm,), x.dtype)
    _need(x, "x")
    y = torch.empty_like(x) if out is None else out
    if workspace is None:
        workspace = _workspace(workspace_size(LA_OP_LAYER_ATTN_OUT, B, H, S, S, D, x.dtype), x.device, None)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().la_layer_attn_out(_ptr(x), _ptr(Wqkv), _ptr(bqkv), _ptr(Wo), _ptr(bo), _ptr(y), B, S, dm, H,
                                    int(bool(causal)), _ptr(kv_len), _dt(x), _ptr(workspace), nbytes,
                                    _stream(stream)), "la_layer_attn_out")
    return y


def layernorm(x, gamma, beta, eps=1e-5, out=None, stream=None):
    """LayerNorm over the last dimension of x (rows of d, d a multiple of 64)."""
    _spec(x, "x")
    d = x.shape[-1] if x.dim() > 0 else 0
    _spec(gamma, "gamma", (d,), x.dtype)
    _spec(beta, "beta", (d,), x.dtype)
    _spec_opt(out, "out", tuple(x.shape), x.dtype)
    for t, n in ((x, "x"), (gamma, "gamma"), (beta, "beta")):
        _need(t, n)
    M = x.numel() // d if d > 0 else 0
    y = torch.empty_like(x) if out is None else out
    _check(load().la_layernorm(_ptr(x), _ptr(gamma), _ptr(beta), _ptr(y), M, d, float(eps), _dt(x),
                               _stream(stream)), "la_layernorm")
    return y


def layer_attn_ln(x, gamma, beta, Wqkv, bqkv, Wo, bo, H, causal=False, kv_len=None, eps=1e-5, out=None,
                  workspace=None, stream=None):
    """The pre-norm attention block: LayerNorm, the sublayer and (Wo not None)
    the output projection: x [B,S,d] -> [B,S,d]."""
    B, S, dm, D = _layer_spec(x, Wqkv, bqkv, H, kv_len, out)
    _spec(gamma, "gamma", (dm,), x.dtype)
    _spec(beta, "beta", (dm,), x.dtype)
    _spec_opt(Wo, "Wo", (dm, dm), x.dtype)
    _spec_opt(bo, "bo", (dm,), x.dtype)
    _need(x, "x")
    y = torch.empty_like(x) if out is None else out
    if workspace is None:
        workspace = _workspace(workspace_size(LA_OP_LAYER_ATTN_LN, B, H, S, S, D, x.dtype), x.device, None)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().la_layer_attn_ln(_ptr(x), _ptr(gamma), _ptr(beta), float(eps), _ptr(Wqkv), _ptr(bqkv), _ptr(Wo),
                                   _ptr(bo), _ptr(y), B, S, dm, H, int(bool(causal)), _ptr(kv_len), _dt(x),
                                   _ptr(workspace), nbytes, _stream(stream)), "la_layer_attn_ln")
    return y


def prepare_weight(W, out=None, stream=None):
    """A projection weight W [rows, cols] in the layout the projection
    kernels read (fp32: W^T [cols, rows]; bf16/fp16: a copy), prepared once
    for layer_attn_prepared."""
    _spec(W, "W")
    if W.dim() != 2:
        raise ValueError("W must be [rows, cols]")
    _need(W, "W")
    rows, cols = W.shape
    shape = (cols, rows) if W.dtype == torch.float32 else (rows, cols)
    _spec_opt(out, "out", shape, W.dtype)
    Wp = torch.empty(shape, dtype=W.dtype, device=W.device) if out is None else out
    _check(load().la_prepare_weight(_ptr(W), _ptr(Wp), rows, cols, _dt(W), _stream(stream)), "la_prepare_weight")
    return Wp


def layer_attn_prepared(x, Wqkv_p, bqkv, H, gamma=None, beta=None, Wo_p=None, bo=None, causal=False, kv_len=None,
                        eps=1e-5, out=None, workspace=None, stream=None):
    """The block of layer_attn_ln on prepared weights (prepare_weight): with
    or without the LayerNorm (gamma, beta) and the output projection (Wo_p,
    bo).  x [B,S,d] -> [B,S,d]."""
    _spec(x, "x")
    if x.dim() != 3:
        raise ValueError("x must be [B, S, d_model]")
    B, S, dm = x.shape
    D = dm // H if H > 0 else 0
    wshape = (3 * dm, dm) if x.dtype == torch.float32 else (dm, 3 * dm)
    _spec(Wqkv_p, "Wqkv_p", wshape, x.dtype)
    _spec_opt(bqkv, "bqkv", (3 * dm,), x.dtype)
    _spec_opt(gamma, "gamma", (dm,), x.dtype)
    _spec_opt(beta, "beta", (dm,), x.dtype)
    _spec_opt(Wo_p, "Wo_p", (dm, dm), x.dtype)
    _spec_opt(bo, "bo", (dm,), x.dtype)
    _kvlen_spec(kv_len, B)
    _spec_opt(out, "out", (B, S, dm), x.dtype)
    _need(x, "x")
    y = torch.empty_like(x) if out is None else out
    if workspace is None:
        workspace = _workspace(workspace_size(LA_OP_LAYER_ATTN_LN, B, H, S, S, D, x.dtype), x.device, None)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().la_layer_attn_prepared(_ptr(x), _ptr(gamma), _ptr(beta), float(eps), _ptr(Wqkv_p), _ptr(bqkv),
                                         _ptr(Wo_p), _ptr(bo), _ptr(y), B, S, dm, H, int(bool(causal)),
                                         _ptr(kv_len), _dt(x), _ptr(workspace), nbytes, _stream(stream)),
           "la_layer_attn_prepared")
    return y


class Graph:
    """Library calls captured once and replayed as one CUDA graph.

    ``fn()`` issues library calls (any of the functions above) on fixed device
    tensors, workspaces included; a replay re-runs the same kernels on the
    same addresses, reading whatever the inputs hold at that time.  Replaying
    saves the host work of every call (argument checks, tensor-map encoding,
    launches): the regime of small shapes, where that work outlasts the
    kernels.  ``fn`` runs once before the capture, so that first-call set-up
    (kernel attributes, device symbol lookups) happens outside it.  Do not
    replay one Graph on two streams at the same time.
    """

    def __init__(self, fn, stream=None):
        self.graph = torch.cuda.CUDAGraph()
        self.stream = stream if stream is not None else torch.cuda.Stream()
        self.stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(self.stream):
            fn()
        self.stream.synchronize()
        with torch.cuda.graph(self.graph, stream=self.stream):
            fn()

    def replay(self):
        self.graph.replay()


class Profile:
    """Per-launch device times of the library's kernels (CUDA events on each
    launch's stream; see la_profile_start in layerattn.h):

        with api.Profile() as p:
            ...library calls...
        p.records  # [(kernel name, ms), ...] in launch order
    """

    def __init__(self, max_launches=4096):
        self.max = int(max_launches)
        self.records = []

    def __enter__(self):
        _check(load().la_profile_start(self.max), "la_profile_start")
        return self

    def __exit__(self, *exc):
        names = (ctypes.c_char_p * self.max)()
        ms = (ctypes.c_float * self.max)()
        n = load().la_profile_stop(names, ms, self.max)
        if n < 0:
            raise RuntimeError("la_profile_stop: a CUDA call failed")
        self.records = [(names[i].decode(), float(ms[i])) for i in range(n)]
        return False

    def by_kernel(self):
        """{kernel name: [ms of each launch]}."""
        out = {}
        for name, ms in self.records:
            out.setdefault(name, []).append(ms)
        return out


def last_error_detail() -> int:
    """Raw device error word seen by the latest get_last_error()."""
    return int(load().la_last_error_detail())


def is_checked_build() -> bool:
    """True when the loaded library is the checked build."""
    return bool(load().la_is_checked_build())


def debug_shrink_output_extent(mode=1):
    """Test hook: the next attention launch declares its output one row short,
    so the checked build skips that row and reports LA_ERR_INTERNAL."""
    _check(load().la_debug_shrink_output_extent(int(mode)), "la_debug_shrink_output_extent")


def debug_inject_timeout(mode=1):
    """Test hook: the next attention launch skips its loads so its bounded
    waits run out and get_last_error() reports LA_ERR_TIMEOUT."""
    _check(load().la_debug_inject_timeout(int(mode)), "la_debug_inject_timeout")


def get_last_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error status."""
    return int(load().la_get_last_error(_stream(stream)))
