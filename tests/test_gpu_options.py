"""The *_ex forwards: int64 expert ids and clamped SwiGLU ([FI] "Tensor and
numerical contract": signed int32/int64 ids; the clamp caps the gate above the
limit and clips up symmetrically).

Bars: int64 ids give bitwise the outputs of the same int32 ids, and an int64
value outside the int32 range counts as an invalid id (flagged, slot ignored);
clamped SwiGLU matches the oracle's clamped forward (relative L2 <= 1e-2, FC2
input codes within one E2M1 step in <= 0.1% of elements) on the W4A4 paths (one
launch and three launches) and on W4A16, and stays batch invariant.
"""
import numpy as np
import pytest
import torch

import nvfp4_token_routed_gb300 as M
from nvfp4_token_routed_gb300 import workloads as W
from oracle import oracle as O

from helpers import bf16_np, rel_l2, signed_step, to_np_u16, unpack_codes

pytestmark = pytest.mark.gpu
DEV = "cuda"

CASES = {
    # 160 routes over 32 experts: the one-launch FC1 -> FC2 path
    "fused": W.Workload("swiglu_T40_H512_I512_E32_K4", 40, 512, 512, 32, 4, "swiglu"),
    # 600 routes over 4 experts: three launches, two to three token tiles per expert
    "separate": W.Workload("swiglu_T300_H512_I256_E4_K2", 300, 512, 256, 4, 2, "swiglu"),
    # 1024 routes over 64 experts: three launches, 16-row tiles read by route
    "wide": W.Workload("swiglu_T256_H512_I1024_E64_K4", 256, 512, 1024, 64, 4, "swiglu"),
}
LIMIT = 0.05


def _inputs(wl):
    x = W.make_x(wl)
    w1, w2 = W.make_weights(wl)
    ids, wts = W.make_routing(wl)
    return x, w1, w2, ids, wts


@pytest.mark.parametrize("name", list(CASES))
def test_int64_ids_match_int32_and_flag_out_of_range(name):
    wl = CASES[name]
    x, w1, w2, ids, wts = _inputs(wl)
    w = M.prepare_weights(w1.to(DEV), w2.to(DEV), wl.act)
    c, s, sc = M.quantize_tokens(x.to(DEV))
    ids32, wd = ids.to(DEV), wts.to(DEV)
    ref = M.forward(w, c, s, sc, ids32, wd)
    got = M.forward_ex(w, c, s, sc, ids32.long(), wd)
    got16 = M.forward_w4a16_ex(w, x.to(DEV), ids32.long(), wd)
    ref16 = M.forward_w4a16(w, x.to(DEV), ids32, wd)
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
    assert torch.equal(got16.view(torch.int16), ref16.view(torch.int16))
    # values beyond int32 are invalid ids, not their low 32 bits
    bad64 = ids32.long().clone()
    bad64[0, 0] = (1 << 40) + int(bad64[0, 0])
    bad64[1, 1] = -(1 << 35)
    empty = ids32.clone()
    empty[0, 0] = -1
    empty[1, 1] = -1
    ws = M.workspace(w, wl.T, wl.K)
    got = M.forward_ex(w, c, s, sc, bad64, wd, ws=ws)
    assert M.moe_nvfp4_read_status(ws) == 7  # MOE_ERR_BAD_EXPERT_ID
    ref = M.forward(w, c, s, sc, empty, wd)
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("name", list(CASES))
def test_clamped_swiglu_matches_the_oracle(name):
    wl = CASES[name]
    x, w1, w2, ids, wts = _inputs(wl)
    Wt = O.Weights(to_np_u16(w1), to_np_u16(w2))
    xc, xsf, xs = O.quantize_tokens(to_np_u16(x))
    ref = O.forward_w4a4(Wt, xc, xsf, xs, ids.numpy(), wts.numpy(), wl.E, wl.H, wl.I, wl.act,
                         limit=LIMIT)
    plain = O.forward_w4a4(Wt, xc, xsf, xs, ids.numpy(), wts.numpy(), wl.E, wl.H, wl.I, wl.act)
    assert rel_l2(bf16_np(ref["out"]), bf16_np(plain["out"])) > 0.05  # the clamp matters here

    w = M.prepare_weights(w1.to(DEV), w2.to(DEV), wl.act)
    c, s, sc = M.quantize_tokens(x.to(DEV))
    ws = M.workspace(w, wl.T, wl.K)
    out = M.forward_ex(w, c, s, sc, ids.to(DEV), wts.to(DEV), swiglu_limit=LIMIT, ws=ws)
    torch.cuda.synchronize()
    assert M.moe_nvfp4_read_status(ws) == 0
    assert rel_l2(bf16_np(to_np_u16(out)), bf16_np(ref["out"])) <= 1e-2
    L = M.moe_nvfp4_workspace_layout(w.dims, wl.T, wl.K)
    Ip = M.padded(wl.I)
    inv = M.ws_view(ws, L, "inv", torch.int32, (wl.T * wl.K,)).cpu().numpy()
    g_fc2 = M.ws_view(ws, L, "fc2q_codes", torch.uint8, (L["rows_cap"], Ip // 2)).cpu().numpy()
    valid = inv >= 0
    steps = signed_step(unpack_codes(g_fc2[inv[valid]][:, : wl.I // 2]),
                        unpack_codes(ref["fc2c"][ref["inv"][valid]]))
    assert steps.max() <= 1 and (steps > 0).mean() <= 1e-3

    ref16 = O.forward_w4a16(Wt, to_np_u16(x), ids.numpy(), wts.numpy(), wl.E, wl.H, wl.I, wl.act,
                            limit=LIMIT)
    out16 = M.forward_w4a16_ex(w, x.to(DEV), ids.to(DEV), wts.to(DEV), swiglu_limit=LIMIT)
    torch.cuda.synchronize()
    assert rel_l2(bf16_np(to_np_u16(out16)), bf16_np(ref16["out"])) <= 1e-2


def test_clamped_swiglu_batch_invariance_and_argument_checks():
    wl = CASES["separate"]
    x, w1, w2, ids, wts = _inputs(wl)
    w = M.prepare_weights(w1.to(DEV), w2.to(DEV), wl.act)
    xd, idd, wd = x.to(DEV), ids.to(DEV), wts.to(DEV)
    c, s, sc = M.quantize_tokens(xd)
    full = M.forward_ex(w, c, s, sc, idd, wd, swiglu_limit=LIMIT)
    sel = torch.randperm(wl.T, generator=torch.Generator().manual_seed(4))[:9].to(DEV)
    c2, s2, sc2 = M.quantize_tokens(xd[sel])
    part = M.forward_ex(w, c2, s2, sc2, idd[sel], wd[sel], swiglu_limit=LIMIT)
    torch.cuda.synchronize()
    assert torch.equal(part.view(torch.int16), full[sel].view(torch.int16))
    # a clamp on squared ReLU, a negative or NaN limit, an unknown id width: rejected
    wr = M.prepare_weights(w1[:, :256].contiguous().to(DEV), w2.to(DEV), "relu2")
    with pytest.raises(M.MoeError):
        M.forward_ex(wr, c, s, sc, idd, wd, swiglu_limit=1.0)
    for lim in (-1.0, float("nan")):
        with pytest.raises(M.MoeError):
            M.forward_ex(w, c, s, sc, idd, wd, swiglu_limit=lim)
    ws = M.workspace(w, wl.T, wl.K)
    out = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(M.MoeError):
        M.moe_nvfp4_forward_ex(w.dims, w, c, s, sc, idd, wd, out, ws, M.moe_forward_opts(2, 0.0))
