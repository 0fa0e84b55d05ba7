"""Test infrastructure only: the fp64 CPU oracle for the attention sublayer.

Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline leg may import this package.  It shares no code with the CUDA
library: the arithmetic lives in ``attn_oracle.c`` (plain C, fp64, OpenMP over
output rows), compiled on first use with gcc; this module only marshals
buffers and returns numpy float64 arrays.

Inputs may be torch CPU tensors or numpy arrays of dtype float64, float32,
bfloat16 (torch only) or float16; the oracle widens the stored values to fp64
exactly and never rounds.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

F64, F32, BF16, F16 = 0, 1, 2, 3


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (fp contraction off, so x86 and Arm agree)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_SO)
            and os.path.getmtime(_SO) >= os.path.getmtime(_SRC)):
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fopenmp", "-fPIC",
           "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P, I, LL, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong, ctypes.c_double
            lib.oracle_attn.argtypes = [P, P, P, I, P, I, I, LL, LL, I, I, D, P]
            lib.oracle_attn_rows.argtypes = [P, P, P, I, I, I, LL, LL, I, I, D, P, P, LL, P]
            lib.oracle_attn_probs.argtypes = [P, P, I, P, I, I, LL, LL, I, I, D, P]
            lib.oracle_attn_online.argtypes = [P, P, P, I, P, I, I, LL, LL, I, I, D, P, LL]
            lib.oracle_attn_split.argtypes = [P, P, P, I, P, I, I, LL, LL, I, I, D, P, I]
            lib.oracle_attn_chunked.argtypes = [P, P, P, I, P, I, I, LL, I, I, D, LL]
            lib.oracle_qkv_proj.argtypes = [P, P, P, I, P, P, P, I, LL, I, I, D]
            lib.oracle_layer_attn.argtypes = [P, P, P, I, P, I, LL, I, I, I, P]
            lib.oracle_out_proj.argtypes = [P, I, P, P, I, P, LL, I, I]
            lib.oracle_layer_attn_out.argtypes = [P, P, P, P, P, I, P, I, LL, I, I, I, P]
            lib.oracle_layernorm.argtypes = [P, I, P, P, I, P, LL, I, D]
            lib.oracle_layer_attn_ln.argtypes = [P, P, P, D, P, P, P, P, I, P, I, LL, I, I, I, P]
            lib.oracle_widen.argtypes = [P, I, LL]
            lib.oracle_widen.restype = D
            lib.oracle_num_threads.restype = I
            lib.oracle_set_num_threads.argtypes = [I]
            lib.oracle_set_num_threads.restype = None
            _lib = lib
    return _lib


def _as_buffer(t):
    """Return (numpy array holding the stored bits, dtype code)."""
    try:
        import torch
    except ImportError:  # pragma: no cover
        torch = None
    if torch is not None and isinstance(t, torch.Tensor):
        t = t.detach().cpu().contiguous()
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy().view(np.uint16), BF16
        if t.dtype == torch.float16:
            return t.view(torch.int16).numpy().view(np.uint16), F16
        if t.dtype == torch.float32:
            return t.numpy(), F32
        if t.dtype == torch.float64:
            return t.numpy(), F64
        raise TypeError(f"oracle: unsupported dtype {t.dtype}")
    a = np.ascontiguousarray(t)
    if a.dtype == np.float64:
        return a, F64
    if a.dtype == np.float32:
        return a, F32
    if a.dtype == np.float16:
        return a.view(np.uint16), F16
    raise TypeError(f"oracle: unsupported dtype {a.dtype}")


def _same_type(*ts):
    bufs = [_as_buffer(t) for t in ts]
    codes = {c for _, c in bufs}
    if len(codes) != 1:
        raise TypeError("oracle: all inputs must share one element type")
    return [b for b, _ in bufs], codes.pop()


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _kvlen(kv_len, B):
    if kv_len is None:
        return None
    a = np.ascontiguousarray(np.asarray(kv_len.cpu() if hasattr(kv_len, "cpu") else kv_len,
                                        dtype=np.int32))
    if a.shape != (B,):
        raise ValueError("oracle: kv_len must have shape [B]")
    return a


def _check(rc, name):
    if rc != 0:
        raise RuntimeError(f"oracle: {name} failed (rc={rc})")


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """Threads of later oracle calls (n < 1: all the host's cores again)."""
    _load().oracle_set_num_threads(int(n))


def attn(q, k, v, causal=False, scale=None, kv_len=None):
    """softmax(scale q k^T) v per (b, h); q [B,H,S_q,D], k/v [B,H,S_kv,D]."""
    (qb, kb, vb), dt = _same_type(q, k, v)
    B, H, S_q, D = qb.shape
    S_kv = kb.shape[2]
    assert kb.shape == (B, H, S_kv, D) and vb.shape == kb.shape
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    kl = _kvlen(kv_len, B)
    o = np.zeros((B, H, S_q, D), dtype=np.float64)
    _check(_load().oracle_attn(_ptr(qb), _ptr(kb), _ptr(vb), dt, _ptr(o), B, H, S_q, S_kv, D,
                               int(bool(causal)), scale, _ptr(kl)), "attn")
    return o


def attn_rows(q, k, v, rows, causal=False, scale=None, kv_len=None):
    """Selected output rows; rows is an int array [n, 3] of (b, h, i)."""
    (qb, kb, vb), dt = _same_type(q, k, v)
    B, H, S_q, D = qb.shape
    S_kv = kb.shape[2]
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    kl = _kvlen(kv_len, B)
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    out = np.zeros((r.shape[0], D), dtype=np.float64)
    _check(_load().oracle_attn_rows(_ptr(qb), _ptr(kb), _ptr(vb), dt, B, H, S_q, S_kv, D,
                                    int(bool(causal)), scale, _ptr(kl), _ptr(r), r.shape[0],
                                    _ptr(out)), "attn_rows")
    return out


def attn_probs(q, k, causal=False, scale=None, kv_len=None):
    """P = softmax(scale q k^T) with masked entries 0: [B,H,S_q,S_kv]."""
    (qb, kb), dt = _same_type(q, k)
    B, H, S_q, D = qb.shape
    S_kv = kb.shape[2]
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    kl = _kvlen(kv_len, B)
    p = np.zeros((B, H, S_q, S_kv), dtype=np.float64)
    _check(_load().oracle_attn_probs(_ptr(qb), _ptr(kb), dt, _ptr(p), B, H, S_q, S_kv, D,
                                     int(bool(causal)), scale, _ptr(kl)), "attn_probs")
    return p


def attn_online(q, k, v, block, causal=False, scale=None, kv_len=None):
    """Online-softmax formulation over key blocks of `block` keys."""
    (qb, kb, vb), dt = _same_type(q, k, v)
    B, H, S_q, D = qb.shape
    S_kv = kb.shape[2]
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    kl = _kvlen(kv_len, B)
    o = np.zeros((B, H, S_q, D), dtype=np.float64)
    _check(_load().oracle_attn_online(_ptr(qb), _ptr(kb), _ptr(vb), dt, _ptr(o), B, H, S_q, S_kv,
                                      D, int(bool(causal)), scale, _ptr(kl), int(block)),
           "attn_online")
    return o


def attn_split(q, k, v, n_split, causal=False, scale=None, kv_len=None):
    """Split-KV partials merged by log-sum-exp."""
    (qb, kb, vb), dt = _same_type(q, k, v)
    B, H, S_q, D = qb.shape
    S_kv = kb.shape[2]
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    kl = _kvlen(kv_len, B)
    o = np.zeros((B, H, S_q, D), dtype=np.float64)
    _check(_load().oracle_attn_split(_ptr(qb), _ptr(kb), _ptr(vb), dt, _ptr(o), B, H, S_q, S_kv,
                                     D, int(bool(causal)), scale, _ptr(kl), int(n_split)),
           "attn_split")
    return o


def attn_chunked(q, k, v, chunk, causal=True, scale=None):
    """Window-by-window attention against a growing cache; q/k/v [B,H,S,D]."""
    (qb, kb, vb), dt = _same_type(q, k, v)
    B, H, S, D = qb.shape
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    o = np.zeros((B, H, S, D), dtype=np.float64)
    _check(_load().oracle_attn_chunked(_ptr(qb), _ptr(kb), _ptr(vb), dt, _ptr(o), B, H, S, D,
                                       int(bool(causal)), scale, int(chunk)), "attn_chunked")
    return o


def qkv_proj(x, W, bias, H, q_scale=1.0):
    """x [B,S,d], W [d,3d], bias [3d] or None -> (q, k, v) head-major fp64."""
    if bias is None:
        (xb, wb), dt = _same_type(x, W)
        bb = None
    else:
        (xb, wb, bb), dt = _same_type(x, W, bias)
    B, S, dm = xb.shape
    assert wb.shape == (dm, 3 * dm)
    D = dm // H
    q = np.zeros((B, H, S, D)); k = np.zeros_like(q); v = np.zeros_like(q)
    _check(_load().oracle_qkv_proj(_ptr(xb), _ptr(wb), _ptr(bb), dt, _ptr(q), _ptr(k), _ptr(v),
                                   B, S, dm, H, float(q_scale)), "qkv_proj")
    return q, k, v


def layer_attn(x, W, bias, H, causal=False, kv_len=None):
    """Projection, per-head attention (scale 1/sqrt(D)), heads merged: [B,S,d]."""
    if bias is None:
        (xb, wb), dt = _same_type(x, W)
        bb = None
    else:
        (xb, wb, bb), dt = _same_type(x, W, bias)
    B, S, dm = xb.shape
    kl = _kvlen(kv_len, B)
    o = np.zeros((B, S, dm))
    _check(_load().oracle_layer_attn(_ptr(xb), _ptr(wb), _ptr(bb), dt, _ptr(o), B, S, dm, H,
                                     int(bool(causal)), _ptr(kl)), "layer_attn")
    return o


def out_proj(a, W, bias=None):
    """a [..., d_in] (any supported type), W [d_in, d_out], bias [d_out] or
    None -> a W + bias in fp64, shape [..., d_out]."""
    ab, dta = _as_buffer(a)
    if bias is None:
        (wb,), dtw = _same_type(W)
        bb = None
    else:
        (wb, bb), dtw = _same_type(W, bias)
    d_in, d_out = wb.shape
    if ab.shape[-1] != d_in:
        raise ValueError("oracle: a and W disagree on d_in")
    M = ab.size // d_in
    y = np.zeros(ab.shape[:-1] + (d_out,), dtype=np.float64)
    _check(_load().oracle_out_proj(_ptr(ab), dta, _ptr(wb), _ptr(bb), dtw, _ptr(y), M, d_in, d_out),
           "out_proj")
    return y


def layer_attn_out(x, W, bias, Wo, bo, H, causal=False, kv_len=None):
    """layer_attn followed by the output projection (d -> d): [B,S,d]."""
    ts = [x, W, Wo] + ([] if bias is None else [bias]) + ([] if bo is None else [bo])
    _, dt = _same_type(*ts)
    xb, wb, wob = (_as_buffer(t)[0] for t in (x, W, Wo))
    bb = None if bias is None else _as_buffer(bias)[0]
    bob = None if bo is None else _as_buffer(bo)[0]
    B, S, dm = xb.shape
    assert wob.shape == (dm, dm)
    kl = _kvlen(kv_len, B)
    y = np.zeros((B, S, dm))
    _check(_load().oracle_layer_attn_out(_ptr(xb), _ptr(wb), _ptr(bb), _ptr(wob), _ptr(bob), dt, _ptr(y),
                                         B, S, dm, H, int(bool(causal)), _ptr(kl)), "layer_attn_out")
    return y


def layernorm(x, gamma, beta, eps=1e-5):
    """LayerNorm over the last dimension of x (any supported type; gamma and
    beta [d] share one type): fp64, biased variance."""
    xb, dtx = _as_buffer(x)
    (gb, bb), dtg = _same_type(gamma, beta)
    d = xb.shape[-1]
    if gb.shape != (d,) or bb.shape != (d,):
        raise ValueError("oracle: gamma and beta must have shape [d]")
    M = xb.size // d
    y = np.zeros(xb.shape, dtype=np.float64)
    _check(_load().oracle_layernorm(_ptr(xb), dtx, _ptr(gb), _ptr(bb), dtg, _ptr(y), M, d, float(eps)),
           "layernorm")
    return y


def layer_attn_ln(x, gamma, beta, W, bias, Wo, bo, H, causal=False, kv_len=None, eps=1e-5):
    """The pre-norm block: LayerNorm, the sublayer, then (Wo given) the
    output projection: [B,S,d]."""
    ts = [x, gamma, beta, W] + [t for t in (bias, Wo, bo) if t is not None]
    _, dt = _same_type(*ts)
    xb, gb, btb, wb = (_as_buffer(t)[0] for t in (x, gamma, beta, W))
    bb, wob, bob = (None if t is None else _as_buffer(t)[0] for t in (bias, Wo, bo))
    B, S, dm = xb.shape
    kl = _kvlen(kv_len, B)
    y = np.zeros((B, S, dm))
    _check(_load().oracle_layer_attn_ln(_ptr(xb), _ptr(gb), _ptr(btb), float(eps), _ptr(wb), _ptr(bb), _ptr(wob),
                                        _ptr(bob), dt, _ptr(y), B, S, dm, H, int(bool(causal)), _ptr(kl)),
           "layer_attn_ln")
    return y


def widen(t):
    """The oracle's own fp64 reading of every stored element (flattened)."""
    buf, dt = _as_buffer(t)
    flat = buf.reshape(-1)
    lib = _load()
    return np.array([lib.oracle_widen(_ptr(flat), dt, i) for i in range(flat.size)])
