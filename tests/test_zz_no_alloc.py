"""The allocation-free forward (moe_nvfp4_forward_noalloc) against the regular one.

moe_nvfp4_forward_noalloc serves callers that may not allocate device memory
(a plugin inside a framework that owns every allocation, code under a locked or
budgeted allocator, an embedded runtime with memory fixed at start-up): it runs
the W4A4 forward on a scratch array the library reserves on each device
(64 MiB), so the caller passes only inputs and outputs.  This file is named to
be collected last, so a run that stops at the first failure has run every other
test first.

It runs exactly the kernels of moe_nvfp4_forward, and every step of the path is
deterministic, so its output must be bitwise that of moe_nvfp4_forward on a
caller-owned workspace.  The calls run back to back on the shared scratch, in
both orders of a one-launch shape (few routes per expert: FC1, the FC2-input
requant and FC2 in one persistent launch, with per-tile counters in the
scratch) and a three-launch shape, so each path also starts on whatever the
other path left in the scratch.
"""
import pytest
import torch

import nvfp4_token_routed_gb300 as M
from nvfp4_token_routed_gb300 import workloads as W

pytestmark = pytest.mark.gpu

ONE_LAUNCH = W.TINY_RELU2                                                      # 32 routes, E=8
THREE_LAUNCH = W.Workload("swiglu_T300_H512_I256_E4_K2", 300, 512, 256, 4, 2, "swiglu")  # 600


def _setup(wl):
    dev = "cuda"
    x = W.make_x(wl).to(dev)
    w1, w2 = W.make_weights(wl)
    ids, wts = W.make_routing(wl)
    w = M.prepare_weights(w1.to(dev), w2.to(dev), wl.act)
    codes, sf, scale = M.quantize_tokens(x)
    return w, codes, sf, scale, ids.to(dev), wts.to(dev)


def test_the_two_shapes_take_the_two_paths():
    count = M.moe_nvfp4_forward_kernel_count
    one = count(M.dims(ONE_LAUNCH.E, ONE_LAUNCH.H, ONE_LAUNCH.I, ONE_LAUNCH.act),
                ONE_LAUNCH.T, ONE_LAUNCH.K)
    three = count(M.dims(THREE_LAUNCH.E, THREE_LAUNCH.H, THREE_LAUNCH.I, THREE_LAUNCH.act),
                  THREE_LAUNCH.T, THREE_LAUNCH.K)
    assert one == 1 + 1 + 1 and three == 2 + 3 + 1


@pytest.mark.parametrize("order", [(ONE_LAUNCH, THREE_LAUNCH), (THREE_LAUNCH, ONE_LAUNCH)],
                         ids=["one_then_three", "three_then_one"])
def test_noalloc_forward_is_bitwise_the_forward_on_calls_in_a_row(order):
    runs = []
    for wl in order:
        w, codes, sf, scale, ids, wts = _setup(wl)
        ref = M.forward(w, codes, sf, scale, ids, wts)
        outs = [torch.full((wl.T, wl.H), float("nan"), dtype=torch.bfloat16, device="cuda")
                for _ in range(2)]
        runs.append((wl, w, codes, sf, scale, ids, wts, ref, outs))
    torch.cuda.synchronize()
    # the sequence twice, back to back on one stream: every call starts on the
    # scratch the previous call (the other shape) left behind
    for rep in range(2):
        for wl, w, codes, sf, scale, ids, wts, ref, outs in runs:
            M.moe_nvfp4_forward_noalloc(w.dims, w, codes, sf, scale, ids, wts, outs[rep])
    torch.cuda.synchronize()
    for wl, w, codes, sf, scale, ids, wts, ref, outs in runs:
        for out in outs:
            assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), wl.name


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
