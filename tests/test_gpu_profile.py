"""The profiling hooks on the GPU: the stage events the library records between
its kernels (moe_nvfp4_profile_events) and the grouped GEMM launches' spans by
the GPU's global timer (moe_nvfp4_profile_spans)."""
import pytest
import torch

import nvfp4_token_routed_gb300 as M
from nvfp4_token_routed_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"
U64_MAX = -1  # all ones: the atomic minimum's starting value, read as int64


def _layer(wl):
    w1, w2 = W.make_weights(wl)
    w = M.prepare_weights(w1.to(DEV), w2.to(DEV), wl.act)
    x = W.make_x(wl).to(DEV)
    ids, wts = W.make_routing(wl)
    return w, x, ids.to(DEV), wts.to(DEV)


def _profiled(w, x, ids, wts):
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    for e in marks:  # created and recorded once by torch; the library records them again
        e.record()
    torch.cuda.synchronize()
    span = torch.tensor([U64_MAX, 0, U64_MAX, 0], dtype=torch.int64, device=DEV)
    codes, sf, scale = M.quantize_tokens(x)
    M.moe_nvfp4_profile_events(marks)
    M.moe_nvfp4_profile_spans(span)
    try:
        out = M.forward(w, codes, sf, scale, ids, wts)
        torch.cuda.synchronize()
    finally:
        M.moe_nvfp4_profile_events([])
        M.moe_nvfp4_profile_spans(None)
    stages_ns = [marks[j].elapsed_time(marks[j + 1]) * 1e6 for j in range(5)]
    return out, span.tolist(), stages_ns


def test_three_launch_spans_and_stage_events():
    """1024 routes over 64 experts: FC1, the requant and FC2 are three launches.
    FC1 ends before FC2 starts (FC2 reads the requantized rows), and each
    launch's span lies within the event interval around it."""
    w, x, ids, wts = _layer(W.SWIGLU_E64)
    out, s, st = _profiled(w, x, ids, wts)
    assert 0 < s[0] < s[1] <= s[2] < s[3]
    assert all(v >= 0 for v in st)
    slack = 2000  # ns: the global timer's update interval
    assert s[1] - s[0] <= st[1] + slack      # FC1 within the FC1 stage
    assert s[3] - s[2] <= st[3] + slack      # FC2 within the FC2 stage
    # the hooks change nothing in the results
    codes, sf, scale = M.quantize_tokens(x)
    plain = M.forward(w, codes, sf, scale, ids, wts)
    assert torch.equal(out.view(torch.int16), plain.view(torch.int16))


def test_one_launch_spans():
    """A few routes: FC1, the requant and FC2 run as one launch, whose span is
    folded into the FC1 slots; the FC2 slots keep their starting values and the
    requant and FC2 stages are empty."""
    wl = W.SWIGLU_E64.with_T(4)
    w, x, ids, wts = _layer(wl)
    out, s, st = _profiled(w, x, ids, wts)
    assert 0 < s[0] < s[1]
    assert s[2] == U64_MAX and s[3] == 0
    assert s[1] - s[0] <= st[1] + 2000
