"""The per-element error bound of the fp32 path, which runs its products on
the TF32 tensor cores (shared by the fp32 GPU parity tests and checked on the
CPU against a model of that arithmetic in tests/test_tf32_bound.py).

Where the arithmetic rounds, relative to the exact (fp64) result:
  - every fp32 operand of a product (q, k, v; x and the weights) is rounded to
    TF32 by the copy into shared memory.  The rounding mode of that copy is
    not documented, so one TF32 ulp is allowed (U_IN = 2^-10, truncation);
  - P is rounded to TF32 to nearest by the kernel (U_P = 2^-11);
  - the tensor cores accumulate in fp32 (allowing a truncating accumulator,
    U_ACC = 2^-23 per addition; n additions cost at most n U_ACC of the sum
    of magnitudes);
  - the softmax arithmetic (scale * log2 e, the exponent argument, the exp2
    unit) perturbs each score by a few fp32 ulps of its magnitude.

Attention, one row: with w_j the exact weights, o the exact output and E_j a
bound on the perturbation of score j (from the rounded q and k, from any
error q and k already carry, and from the softmax arithmetic), the weights
move to w_j exp(d_j - dbar) with |d_j| <= E_j, so to first order
  |do_c| <= sum_j w_j E_j |v_jc - o_c| <= sum_j w_j E_j (|v_jc| + |o_c|),
times exp(2 max E) for the higher orders.  Rounding P and V adds
(U_P + U_IN) sum_j w_j |v_jc|, an error dv the values already carry adds
sum_j w_j dv_jc, and the fp32 sums of P V and of the row sum add
2 (n + 8) U_ACC sum_j w_j |v_jc|.

A product y = a W (+ b): |dy| <= (2 U_IN + U_IN^2 + (K + 2) U_ACC) |a| |W|
+ (1 + U_IN) da |W| for an error da already in a.
"""
import numpy as np

U_IN = 2.0 ** -10
U_P = 2.0 ** -11
U_ACC = 2.0 ** -23
U_SM = 2.0 ** -20      # softmax arithmetic, relative to the score magnitudes
TINY = 1e-7            # absolute floor (fp32 resolution of values near 0)


def gemm_bound(a, w, da=None):
    """Bound on |(a W)_gpu - (a W)_exact| for a [..., K], w [K, N] (float64
    arrays of the stored values); da: elementwise bound of an error a carries."""
    aa = np.abs(np.asarray(a, dtype=np.float64))
    aw = np.abs(np.asarray(w, dtype=np.float64))
    K = aw.shape[0]
    b = (2 * U_IN + U_IN ** 2 + (K + 2) * U_ACC) * (aa @ aw)
    if da is not None:
        b = b + (1 + U_IN) * (np.asarray(da) @ aw)
    return b + TINY


def _heads(y, H, which):
    """[B, S, 3d] (or [B, S, d] with which=None) -> [B, H, S, D] of block `which`."""
    B, S, n = y.shape
    d = n // 3 if which is not None else n
    blk = y[..., which * d:(which + 1) * d] if which is not None else y
    return np.ascontiguousarray(blk.reshape(B, S, H, d // H).transpose(0, 2, 1, 3))


def qkv_bounds(x, W, H, q_scale=1.0, dx=None):
    """Bounds of the projection's q, k, v [B, H, S, D] (x [B, S, d], W [d, 3d])."""
    y = gemm_bound(x, W, dx)
    bq, bk, bv = (_heads(y, H, i) for i in range(3))
    return bq * abs(q_scale), bk, bv


def attn_bound(q, k, v, P, o, scale, dq=None, dk=None, dv=None):
    """Bound on |o_gpu - o_exact| per element, [B, H, S_q, D].  q, k, v, o:
    exact (float64) values, P: the exact weights [B, H, S_q, S_kv] (0 where
    masked); dq, dk, dv: elementwise bounds of errors the inputs already carry
    (the projection's), or None."""
    q, k, v, o = (np.asarray(t, dtype=np.float64) for t in (q, k, v, o))
    B, H, S_q, D = q.shape
    S_kv = k.shape[2]
    out = np.empty_like(o)
    c_in = 2 * U_IN + U_IN ** 2 + (D + 2) * U_ACC
    c_v = U_IN + U_P + 2 * (S_kv + 8) * U_ACC
    for b in range(B):
        for h in range(H):
            aq, ak, av = np.abs(q[b, h]), np.abs(k[b, h]), np.abs(v[b, h])
            p = P[b, h]
            s = np.abs(scale * (q[b, h] @ k[b, h].T))
            smax = np.max(np.where(p > 0, s, 0.0), axis=1, keepdims=True)
            E = scale * c_in * (aq @ ak.T) + U_SM * (s + smax + 1.0)
            if dq is not None:
                E = E + scale * (1 + U_IN) * (dq[b, h] @ ak.T + aq @ dk[b, h].T + dq[b, h] @ dk[b, h].T)
            Emax = np.max(np.where(p > 0, E, 0.0), axis=1, keepdims=True)
            pe = p * E
            ao = np.abs(o[b, h])
            t1 = np.exp(2.0 * Emax) * (pe @ av + pe.sum(axis=1, keepdims=True) * ao)
            t2 = c_v * (p @ av)
            if dv is not None:
                t2 = t2 + (1 + U_IN + U_P) * (p @ dv[b, h])
            out[b, h] = t1 + t2 + U_SM * ao + TINY
    return out


def merged(t):
    """[B, H, S, D] -> heads merged [B, S, H*D] (the sublayer's output layout)."""
    B, H, S, D = t.shape
    return np.ascontiguousarray(t.transpose(0, 2, 1, 3).reshape(B, S, H * D))


def _f64(t):
    if t is None:
        return None
    if hasattr(t, "detach"):
        t = t.detach().cpu().double().numpy()
    return np.asarray(t, dtype=np.float64)


def sublayer_bound(x, W, b, H, causal=False, kv_len=None, Wo=None, bo=None, dx=None):
    """Bound of the fp32 sublayer (projection, attention, heads merged) on
    x [B, S, d], or with Wo of its output projection y = o Wo + bo: the
    projection's errors carried into the attention bound, the attention's
    into the output projection's.  Exact intermediate values come from the
    oracle (widened to fp64, so x may be an exact fp64 LayerNorm output)."""
    import oracle
    x, W, b, Wo, bo = (_f64(t) for t in (x, W, b, Wo, bo))
    q, k, v = oracle.qkv_proj(x, W, b, H)
    D = q.shape[-1]
    scale = D ** -0.5
    P = oracle.attn_probs(q, k, causal=causal, scale=scale, kv_len=kv_len)
    o = oracle.attn(q, k, v, causal=causal, scale=scale, kv_len=kv_len)
    dq, dk, dv = qkv_bounds(x, W, H, dx=dx)
    if b is not None:  # the fp32 bias add rounds once more
        db = 2.0 ** -23 * np.abs(b)
        dq, dk, dv = (d + _heads(np.broadcast_to(db, x.shape[:2] + db.shape), H, i) for i, d in enumerate((dq, dk, dv)))
    bo_att = merged(attn_bound(q, k, v, P, o, scale, dq, dk, dv))
    if Wo is None:
        return bo_att
    y_b = gemm_bound(merged(o), Wo, da=bo_att)
    if bo is not None:
        y_b = y_b + 2.0 ** -23 * np.abs(bo)
    return y_b


def layernorm_error(xhat):
    """Bound of the fp32 LayerNorm's error on its exact output x^ (mean,
    variance and the normalisation in fp32: a few fp32 ulps of |x^| + 1)."""
    return 2.0 ** -19 * (np.abs(np.asarray(xhat)) + 1.0)
