"""Algorithmic work and traffic of the attention sublayer (measurement only).

FLOPs count the useful arithmetic of the method, never the work a kernel
wastes: attention is 4 * D multiply-adds-as-FLOPs per (query, valid key) pair
per head (2 D for q.k, 2 D for p.v), summed over the pairs the mask keeps;
the fused projection is 2 * rows * d_model * 3 d_model.

The layer model of "Shape-Aware Attention" (section How we built it: the
FLOP count 8BSd^2 + 4BS^2d + 4BSdf, the Amdahl ceiling and the arithmetic
intensity table) is reproduced by layer_model_* so that its printed worked
example pins this arithmetic.
"""
from __future__ import annotations


def attn_pairs(B, S_q, S_kv, causal, kv_len=None):
    """Number of (query, key) pairs the mask keeps, summed over the batch.
    Causal rows are aligned to the end of the key range."""
    off = S_kv - S_q
    total = 0
    for b in range(B):
        L = S_kv if kv_len is None else min(int(kv_len[b]), S_kv)
        if not causal:
            total += S_q * max(L, 0)
            continue
        # row i sees keys j <= i + off and j < L
        for_rows = 0
        # rows where i + off + 1 < L see i + off + 1 keys (if positive)
        i_split = min(max(L - off - 1, 0), S_q)        # rows i < i_split: limit i+off+1
        i_lo = min(max(-off, 0), S_q)                  # rows i < i_lo see nothing
        if i_split > i_lo:
            a, z = i_lo + off + 1, i_split - 1 + off + 1
            for_rows += (a + z) * (i_split - i_lo) // 2
        for_rows += (S_q - max(i_split, i_lo)) * max(L, 0) if S_q > max(i_split, i_lo) else 0
        total += for_rows
    return total


def attn_flops(B, H, S_q, S_kv, D, causal, kv_len=None):
    return 4 * H * D * attn_pairs(B, S_q, S_kv, causal, kv_len)


def proj_flops(B, S, d_model):
    return 2 * B * S * d_model * 3 * d_model


def out_proj_flops(B, S, d_model):
    """The output projection y = o Wo + bo, Wo [d, d]."""
    return 2 * B * S * d_model * d_model


def attn_min_bytes(B, H, S_q, S_kv, D, in_bytes, out_bytes):
    """Compulsory HBM traffic: read q, k, v once, write o once."""
    return B * H * D * (S_q * in_bytes + 2 * S_kv * in_bytes + S_q * out_bytes)


def proj_min_bytes(B, S, d_model, in_bytes, out_bytes, bias=True):
    w = 3 * d_model * d_model * in_bytes + (3 * d_model * in_bytes if bias else 0)
    return B * S * d_model * in_bytes + w + 3 * B * S * d_model * out_bytes


# --- the pages' layer model ---------------------------------------------------
def layer_model_flops(B, S, d, f):
    """Per-layer FLOPs: projections (Q, K, V, output), attention, FFN."""
    return {"proj": 8 * B * S * d * d, "attn": 4 * B * S * S * d, "ffn": 4 * B * S * d * f}


def layer_model_bytes(B, S, d, f, H, fused, elem=4):
    """Bytes of the layer as reconstructed from the intensity table: weights
    (4d^2 + 2df) plus 30 activation-sized tensors; the unfused chain also moves
    the [B,H,S,S] score matrix three times (write, softmax read+write ... read)."""
    base = (4 * d * d + 2 * d * f) * elem + 30 * B * S * d * elem
    return base if fused else base + 3 * B * H * S * S * elem


def layer_model_intensity(B, S, d, f, H, fused):
    fl = sum(layer_model_flops(B, S, d, f).values())
    return fl / layer_model_bytes(B, S, d, f, H, fused)
