"""Pins for the measurement arithmetic: the pages' worked example
(tests/golden/layer_model.txt) and brute-force pair counts.  CPU only."""
import os

import numpy as np
import pytest

from layer_attn_fwd_gb300 import flops

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "layer_model.txt")


def _golden():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                key, *vals = line.split()
                rows.append((key, [float(v) for v in vals]))
    return rows


def test_golden_layer_model():
    B, d, f, H = 8, 512, 2048, 8
    seen = set()
    for key, vals in _golden():
        seen.add(key)
        if key == "attn_share":
            S, want = vals
            fl = flops.layer_model_flops(B, int(S), d, f)
            assert round(fl["attn"] / sum(fl.values()), 3) == want
        elif key == "amdahl":
            S, want = vals
            fl = flops.layer_model_flops(B, int(S), d, f)
            share = fl["attn"] / sum(fl.values())
            assert round(1 / (1 - share), 3) == want
        elif key == "runtime_share":
            speedup, want = vals
            # the page prints the whole percent, truncated (40.6% -> "40%")
            assert int(100 * (1 - 1 / speedup)) == round(100 * want)
        elif key == "intensity":
            S, ref, fused = vals
            assert round(flops.layer_model_intensity(B, int(S), d, f, H, fused=False), 1) == ref
            assert round(flops.layer_model_intensity(B, int(S), d, f, H, fused=True), 1) == fused
        elif key == "ridge":
            peak, bw, want = vals
            assert round(peak / bw, 1) == want
    assert seen == {"attn_share", "amdahl", "runtime_share", "intensity", "ridge"}


def _brute_pairs(B, S_q, S_kv, causal, kv_len):
    i = np.arange(S_q)[:, None] + (S_kv - S_q)
    j = np.arange(S_kv)[None, :]
    n = 0
    for b in range(B):
        m = np.ones((S_q, S_kv), dtype=bool)
        if causal:
            m &= j <= i
        if kv_len is not None:
            m &= j < kv_len[b]
        n += int(m.sum())
    return n


@pytest.mark.parametrize("S_q,S_kv", [(1, 1), (5, 5), (7, 3), (3, 9), (128, 128), (100, 357), (0, 4), (4, 0)])
@pytest.mark.parametrize("causal", [False, True])
def test_pairs_brute_force(S_q, S_kv, causal):
    for kv_len in (None, [S_kv, max(S_kv - 2, 0), 0, S_kv // 2]):
        B = 4
        assert flops.attn_pairs(B, S_q, S_kv, causal, kv_len) == _brute_pairs(B, S_q, S_kv, causal, kv_len)


def test_workload_flop_counts():
    # causal S=2048: 2048*2049/2 pairs per (b, h)
    assert flops.attn_pairs(1, 2048, 2048, True) == 2_098_176
    # last quarter of keys padded for half the batch
    assert flops.attn_pairs(2, 2048, 2048, True, [1536, 2048]) == 1_966_848 + 2_098_176
    assert flops.proj_flops(8, 512, 512) == 6_442_450_944
    assert flops.attn_flops(8, 8, 512, 512, 64, False) == 4_294_967_296
