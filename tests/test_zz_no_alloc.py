"""The allocation-free forward (moe_nvfp4_forward_noalloc) against the regular one.

moe_nvfp4_forward_noalloc serves callers that may not allocate device memory:
it runs the W4A4 forward on a scratch array the library reserves on each
device (64 MiB), so the caller passes only inputs and outputs.  This file is
named to be collected last, so a run that stops at the first failure has run
every other test first.  Two calls in a row with different shapes check that
whatever the first call leaves in the shared scratch does not leak into the
second; each is compared with moe_nvfp4_forward on a caller-owned workspace
within the suite's output tolerance (relative L2 <= 1e-2).
"""
import numpy as np
import pytest
import torch

import nvfp4_token_routed_gb300 as M
from nvfp4_token_routed_gb300 import workloads as W

pytestmark = pytest.mark.gpu

SHAPES = [
    W.TINY_RELU2,
    W.Workload("swiglu_T300_H512_I256_E4_K2", 300, 512, 256, 4, 2, "swiglu"),
]


def _setup(wl):
    dev = "cuda"
    x = W.make_x(wl).to(dev)
    w1, w2 = W.make_weights(wl)
    ids, wts = W.make_routing(wl)
    w = M.prepare_weights(w1.to(dev), w2.to(dev), wl.act)
    codes, sf, scale = M.quantize_tokens(x)
    return w, codes, sf, scale, ids.to(dev), wts.to(dev)


def _rel_l2(a, b):
    a = a.float()
    b = b.float()
    return float((a - b).norm() / b.norm().clamp_min(1e-30))


def test_noalloc_forward_matches_forward_two_calls_in_a_row():
    runs = []
    for wl in SHAPES:
        w, codes, sf, scale, ids, wts = _setup(wl)
        ref = M.forward(w, codes, sf, scale, ids, wts)
        out = torch.full((wl.T, wl.H), float("nan"), dtype=torch.bfloat16, device="cuda")
        runs.append((wl, w, codes, sf, scale, ids, wts, ref, out))
    torch.cuda.synchronize()
    # two allocation-free calls back to back on the same stream
    for wl, w, codes, sf, scale, ids, wts, ref, out in runs:
        M.moe_nvfp4_forward_noalloc(w.dims, w, codes, sf, scale, ids, wts, out)
    torch.cuda.synchronize()
    for wl, w, codes, sf, scale, ids, wts, ref, out in runs:
        assert torch.isfinite(out.float()).all(), wl.name
        assert _rel_l2(out, ref) <= 1e-2, wl.name


def test_noalloc_rejects_problems_beyond_its_scratch():
    wl = W.SWIGLU_E64
    d = M.dims(wl.E, wl.H, wl.I, wl.act)
    T = 4096
    assert M.moe_nvfp4_workspace_bytes(d, T, wl.K) > 64 << 20
    w = M.PreparedWeights(wl.E, wl.H, wl.I, wl.act)
    dev = "cuda"
    codes = torch.zeros(T, wl.H // 2, dtype=torch.uint8, device=dev)
    sf = torch.zeros(T, wl.H // 16, dtype=torch.uint8, device=dev)
    scale = torch.zeros(T, dtype=torch.float32, device=dev)
    ids = torch.zeros(T, wl.K, dtype=torch.int32, device=dev)
    wts = torch.zeros(T, wl.K, dtype=torch.float32, device=dev)
    out = torch.zeros(T, wl.H, dtype=torch.bfloat16, device=dev)
    with pytest.raises(M.MoeError) as ei:
        M.moe_nvfp4_forward_noalloc(d, w, codes, sf, scale, ids, wts, out)
    assert ei.value.code == 4  # MOE_ERR_WORKSPACE_TOO_SMALL
    assert not out.any()
