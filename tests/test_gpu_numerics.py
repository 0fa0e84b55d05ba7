"""Device numeric helpers of the softmax, checked on the GPU against fp64
references: the FMA-pipe exp2 polynomial and the MUFU exp2."""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

from gpu_util import need_gpu

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.fixture(scope="module")
def probe():
    need_gpu()
    src = os.path.join(HERE, "gpu_probe", "la_probe.cu")
    out = os.path.join(HERE, "gpu_probe", "_build", "la_probe.so")
    os.makedirs(os.path.dirname(out), exist_ok=True)
    subprocess.run(["nvcc", "-shared", "-Xcompiler", "-fPIC", "-O3", "-std=c++17",
                    "-gencode", "arch=compute_103a,code=sm_103a",
                    "-I", os.path.join(ROOT, "layer_attn_fwd_gb300", "csrc"), "-I", os.path.join(ROOT, "include"),
                    src, "-o", out], check=True)
    lib = ctypes.CDLL(out)
    lib.probe_ex2.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int]
    return lib


def test_ex2_polynomial_error_bound(probe):
    x = torch.cat([torch.linspace(-130.0, 64.0, 1_000_003), torch.tensor([float("-inf"), 0.0, -0.5, 0.5, 8.0]),
                   torch.randn(100_000) * 10]).float()
    xd = x.cuda()
    poly = torch.empty_like(xd)
    mufu = torch.empty_like(xd)
    assert probe.probe_ex2(xd.data_ptr(), poly.data_ptr(), mufu.data_ptr(), xd.numel()) == 0
    xs = x.double().numpy()
    ref = np.exp2(xs)
    p = poly.double().cpu().numpy()
    m = mufu.double().cpu().numpy()
    normal = xs >= -125.0
    rel = np.abs(p[normal] - ref[normal]) / ref[normal]
    assert rel.max() < 8e-5, rel.max()          # the fitted bound is 7.5e-5 (plus fp32 rounding)
    assert np.all(p[~normal] == 0.0)             # below the range (and -inf): exactly 0
    ok = xs > -126.0
    relm = np.abs(m[ok] - ref[ok]) / ref[ok]
    assert relm.max() < 1e-6, relm.max()         # the MUFU exp2 the other lanes use
    assert m[np.isneginf(xs)][0] == 0.0
