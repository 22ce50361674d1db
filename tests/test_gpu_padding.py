"""Non-256-aligned shapes (Megatron-LM PR #8262, "Why CuTe DSL": hidden sizes are
padded to 256, 2688 -> 2816; "What is tested": non-aligned shapes exercise the
padding).  The library stores H and I zero-padded to multiples of 256; the
oracle runs on the unpadded shapes.  Bars: quantized tokens and prepared weights
bit-exact on the real region and zero in the padding; outputs within relative
L2 1e-2 of the oracle; per-token outputs bitwise batch invariant.
"""
import numpy as np
import pytest
import torch

import nvfp4_token_routed_gb300 as M
from nvfp4_token_routed_gb300 import workloads as W
from oracle import oracle as O

from helpers import bf16_np, rel_l2, to_np_u16, unswizzle

pytestmark = pytest.mark.gpu
DEV = "cuda"

CASES = {
    # H -> 512, I -> 256: padding in both dimensions, a single 128-row FC2 tile pair
    "relu2_H320_I192": W.Workload("relu2_T40_H320_I192_E8_K2", 40, 320, 192, 8, 2, "relu2"),
    "swiglu_H320_I192": W.Workload("swiglu_T40_H320_I192_E8_K2", 40, 320, 192, 8, 2, "swiglu"),
    # the pages' example hidden size 2688 -> 2816, I 1856 -> 2048
    "swiglu_H2688_I1856": W.Workload("swiglu_T48_H2688_I1856_E16_K4", 48, 2688, 1856, 16, 4,
                                     "swiglu", x_dist="normal"),
}


def stored_rows_padded(I, Ip, act):
    """Canonical FC1 row held at each stored row of the padded layout, -1 for padding."""
    if act != "swiglu":
        r = np.arange(Ip)
        return np.where(r < I, r, -1)
    ir = np.arange(2 * Ip)
    b = ir // 64
    half, f = b % 2, (b // 2) * 64 + ir % 64
    return np.where(f < I, half * I + f, -1)


_cache = {}


def _setup(name):
    if name not in _cache:
        wl = CASES[name]
        x = W.make_x(wl)
        w1, w2 = W.make_weights(wl)
        ids, wts = W.make_routing(wl)
        Wt = O.Weights(to_np_u16(w1), to_np_u16(w2))
        xc, xsf, xs = O.quantize_tokens(to_np_u16(x))
        ref = O.forward_w4a4(Wt, xc, xsf, xs, ids.numpy(), wts.numpy(), wl.E, wl.H, wl.I, wl.act)
        ref16 = O.forward_w4a16(Wt, to_np_u16(x), ids.numpy(), wts.numpy(), wl.E, wl.H, wl.I,
                                wl.act)
        _cache[name] = (wl, x, w1, w2, ids, wts, Wt, (xc, xsf, xs), ref, ref16)
    return _cache[name]


@pytest.mark.parametrize("name", list(CASES))
def test_padded_quantization_and_weights(name):
    wl, x, w1, w2, ids, wts, Wt, (xc, xsf, xs), _, _ = _setup(name)
    H, I, Hp, Ip = wl.H, wl.I, M.padded(wl.H), M.padded(wl.I)
    codes, sf, scale = M.quantize_tokens(x.to(DEV))
    codes, sf = codes.cpu().numpy(), sf.cpu().numpy()
    assert codes.shape == (wl.T, Hp // 2) and sf.shape == (wl.T, Hp // 16)
    assert np.array_equal(codes[:, : H // 2], xc) and not codes[:, H // 2:].any()
    assert np.array_equal(sf[:, : H // 16], xsf) and not sf[:, H // 16:].any()
    assert np.array_equal(scale.cpu().numpy(), xs)

    w = M.prepare_weights(w1.to(DEV), w2.to(DEV), wl.act)
    torch.cuda.synchronize()
    assert np.array_equal(w.fc1_alpha.cpu().numpy(), Wt.a1)
    assert np.array_equal(w.fc2_alpha.cpu().numpy(), Wt.a2)
    src = stored_rows_padded(I, Ip, wl.act)
    real = src >= 0
    g1 = w.fc1_codes.cpu().numpy()
    s1 = w.fc1_sf.cpu().numpy().reshape(wl.E, -1)
    g2 = w.fc2_codes.cpu().numpy()
    s2 = w.fc2_sf.cpu().numpy().reshape(wl.E, -1)
    for e in range(wl.E):
        assert np.array_equal(g1[e][real, : H // 2], Wt.w1c[e][src[real]])
        assert not g1[e][real, H // 2:].any() and not g1[e][~real].any()
        lin = unswizzle(s1[e], np.arange(len(src)), Hp // 16)
        assert np.array_equal(lin[real, : H // 16], Wt.w1sf[e][src[real]])
        assert not lin[real, H // 16:].any() and not lin[~real].any()
        assert np.array_equal(g2[e][:H, : I // 2], Wt.w2c[e])
        assert not g2[e][:H, I // 2:].any() and not g2[e][H:].any()
        lin2 = unswizzle(s2[e], np.arange(Hp), Ip // 16)
        assert np.array_equal(lin2[:H, : I // 16], Wt.w2sf[e])
        assert not lin2[:H, I // 16:].any() and not lin2[H:].any()


@pytest.mark.parametrize("name", list(CASES))
def test_padded_forward_matches_the_unpadded_oracle(name):
    wl, x, w1, w2, ids, wts, _, _, ref, ref16 = _setup(name)
    w = M.prepare_weights(w1.to(DEV), w2.to(DEV), wl.act)
    codes, sf, scale = M.quantize_tokens(x.to(DEV))
    ws = M.workspace(w, wl.T, wl.K)
    out = M.forward(w, codes, sf, scale, ids.to(DEV), wts.to(DEV), ws=ws)
    torch.cuda.synchronize()
    assert M.moe_nvfp4_read_status(ws) == 0
    assert out.shape == (wl.T, wl.H)
    got = to_np_u16(out)
    assert rel_l2(bf16_np(got), bf16_np(ref["out"])) <= 1e-2

    ws16 = M.workspace(w, wl.T, wl.K, w4a16=True)
    out16 = M.forward_w4a16(w, x.to(DEV), ids.to(DEV), wts.to(DEV), ws=ws16)
    torch.cuda.synchronize()
    assert M.moe_nvfp4_read_status(ws16) == 0
    assert rel_l2(bf16_np(to_np_u16(out16)), bf16_np(ref16["out"])) <= 1e-2


@pytest.mark.parametrize("name", ["swiglu_H320_I192", "swiglu_H2688_I1856"])
def test_padded_batch_invariance(name):
    wl, x, w1, w2, ids, wts, *_ = _setup(name)
    w = M.prepare_weights(w1.to(DEV), w2.to(DEV), wl.act)
    xd, idd, wd = x.to(DEV), ids.to(DEV), wts.to(DEV)
    codes, sf, scale = M.quantize_tokens(xd)
    full = M.forward(w, codes, sf, scale, idd, wd)
    full16 = M.forward_w4a16(w, xd, idd, wd)
    g = torch.Generator().manual_seed(5)
    for n in (1, 7):
        sel = torch.randperm(wl.T, generator=g)[:n].to(DEV)
        c, s, sc = M.quantize_tokens(xd[sel])
        part = M.forward(w, c, s, sc, idd[sel], wd[sel])
        part16 = M.forward_w4a16(w, xd[sel], idd[sel], wd[sel])
        torch.cuda.synchronize()
        assert torch.equal(part.view(torch.int16), full[sel].view(torch.int16))
        assert torch.equal(part16.view(torch.int16), full16[sel].view(torch.int16))
