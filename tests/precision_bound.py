"""The per-element error bound of the half-precision attention path (shared
by the GPU precision study and its CPU check).

The path rounds twice: P (fp32 until then) to the operand type before the
PV product, and the fp32 output to its storage type.  With r the oracle's
value, g the computed one, p the oracle's normalised probabilities and v the
values:

  |g - r| <= 0.5 max(ulp(r), ulp(g)) + u * sum_j p_j |v_j|
             + (fp16) 2^-25 * sum_{j visible} |v_j|
             + SLACK * (sum_j p_j |v_j| + |r|)

u the unit roundoff of the operand type (2^-8 bf16, 2^-11 fp16), the fp16
term for probabilities in the subnormal range (absolute rounding 2^-25; the
row maximum's weight is at least 1), SLACK for the fp32 score, exponential
and accumulation arithmetic."""
import numpy as np

from layer_attn_fwd_gb300 import ulp

SLACK = 2.0 ** -12


def rounding_bound(r, g, P, v, fmt):
    """r, g [B,H,S_q,D]; P [B,H,S_q,S_kv] normalised; v [B,H,S_kv,D] (float64)."""
    av = np.abs(v)
    ep = np.einsum("bhij,bhjd->bhid", P, av)                 # sum_j p_j |v_j|
    b = 0.5 * np.maximum(ulp.ulp(r, fmt), ulp.ulp(g, fmt)) + ulp.unit_roundoff(fmt) * ep
    if fmt == "f16":
        b += 2.0 ** -25 * np.einsum("bhij,bhjd->bhid", (P > 0).astype(np.float64), av)
    return b + SLACK * (ep + np.abs(r))
