"""GPU parity of every stage against the CPU oracle, through the C ABI.

Bars: token/weight quantization and the routing permutation bit-exact; FC2-input
requantized codes at most one E2M1 step apart in at most 0.1% of elements,
block scales at most one E4M3 code apart in at most 0.1% of blocks, s2 within
1e-5 relative; final output relative L2 <= 1e-2.
"""
import numpy as np
import pytest
import torch

import nvfp4_token_routed_gb300 as M
from nvfp4_token_routed_gb300 import workloads as W
from oracle import oracle as O

from helpers import (TILE_ROWS, OracleRun, bf16_np, check_scaled_f16_rows, rel_l2, signed_step,
                     stored_fc1_rows, to_np_u16, unpack_codes, unswizzle)

pytestmark = pytest.mark.gpu

CASES = {
    "tiny_relu2": W.TINY_RELU2,
    "swiglu_ragged": W.Workload("swiglu_T300_H512_I256_E4_K2", 300, 512, 256, 4, 2, "swiglu"),
    "relu2_zipf": W.Workload("relu2_T200_H768_I512_E16_K4_zipf", 200, 768, 512, 16, 4, "relu2",
                             x_dist="logspread", routing="zipf", empty_experts=2),
    "swiglu_e64": W.SWIGLU_E64,
    # few routes per expert: FC1, the FC2-input requant and FC2 run as one launch
    "swiglu_fused": W.Workload("swiglu_T40_H512_I512_E32_K4", 40, 512, 512, 32, 4, "swiglu"),
    "relu2_fused": W.Workload("relu2_T24_H768_I512_E64_K6", 24, 768, 512, 64, 6, "relu2",
                              x_dist="logspread"),
}


def _inputs(wl):
    x = W.make_x(wl)
    w1, w2 = W.make_weights(wl)
    ids, wts = W.make_routing(wl)
    return x, w1, w2, ids, wts


class GpuForward:
    def __init__(self, wl, x, w1, w2, ids, wts):
        dev = "cuda"
        self.wl = wl
        self.w = M.prepare_weights(w1.to(dev), w2.to(dev), wl.act)
        self.codes, self.sf, self.scale = M.quantize_tokens(x.to(dev))
        self.ids = ids.to(dev)
        self.wts = wts.to(dev)
        self.ws = M.workspace(self.w, wl.T, wl.K)
        self.L = M.moe_nvfp4_workspace_layout(self.w.dims, wl.T, wl.K)
        self.out = M.forward(self.w, self.codes, self.sf, self.scale, self.ids, self.wts, ws=self.ws)
        torch.cuda.synchronize()
        self.status = M.moe_nvfp4_read_status(self.ws)

    def view(self, name, dtype, shape):
        return M.ws_view(self.ws, self.L, name, dtype, shape).cpu().numpy()


_cache = {}


def _run(name):
    if name not in _cache:
        wl = CASES[name]
        x, w1, w2, ids, wts = _inputs(wl)
        _cache[name] = (wl, GpuForward(wl, x, w1, w2, ids, wts), OracleRun(wl, x, w1, w2, ids, wts))
    return _cache[name]


def _rows_map(g, o):
    """GPU permuted row of each oracle compact position q."""
    E = g.wl.E
    counts = o.res["counts"]
    start = np.concatenate([[0], np.cumsum(counts)[:-1]])
    row0 = g.view("group_row0", torch.int32, (E,))
    q_expert = np.repeat(np.arange(E), counts)
    q = np.arange(counts.sum())
    return row0[q_expert] + (q - start[q_expert])


@pytest.mark.parametrize("name", list(CASES))
def test_token_quant_bit_exact(name):
    wl, g, o = _run(name)
    assert np.array_equal(g.codes.cpu().numpy(), o.xc)
    assert np.array_equal(g.sf.cpu().numpy(), o.xsf)
    assert np.array_equal(g.scale.cpu().numpy().view(np.uint32), o.xs.view(np.uint32))


@pytest.mark.parametrize("name", list(CASES))
def test_weight_prep_bit_exact(name):
    wl, g, o = _run(name)
    E, H, I, N1 = wl.E, wl.H, wl.I, wl.N1
    rows = stored_fc1_rows(N1, I, wl.act)
    c1 = g.w.fc1_codes.cpu().numpy()
    assert np.array_equal(c1, o.W.w1c[:, rows, :])
    s1 = g.w.fc1_sf.cpu().numpy().reshape(E, -1)
    for e in range(E):
        assert np.array_equal(unswizzle(s1[e], np.arange(N1), H // 16), o.W.w1sf[e][rows])
    assert np.array_equal(g.w.fc1_alpha.cpu().numpy().view(np.uint32), o.W.a1.view(np.uint32))
    assert np.array_equal(g.w.fc2_codes.cpu().numpy(), o.W.w2c)
    s2 = g.w.fc2_sf.cpu().numpy().reshape(E, -1)
    for e in range(E):
        assert np.array_equal(unswizzle(s2[e], np.arange(H), I // 16), o.W.w2sf[e])
    assert np.array_equal(g.w.fc2_alpha.cpu().numpy().view(np.uint32), o.W.a2.view(np.uint32))


@pytest.mark.parametrize("name", list(CASES))
def test_routing_permutation_bit_exact(name):
    wl, g, o = _run(name)
    E, TK = wl.E, wl.T * wl.K
    counts = g.view("counts", torch.int32, (E,))
    assert np.array_equal(counts, o.res["counts"])
    row0 = g.view("group_row0", torch.int32, (E,))
    tiles = np.ceil(counts / TILE_ROWS).astype(np.int64)
    assert np.array_equal(row0, TILE_ROWS * np.concatenate([[0], np.cumsum(tiles)[:-1]]))
    status = g.view("status", torch.int32, (16,))
    assert status[1] == tiles.sum()
    assert status[3] == min(TILE_ROWS, counts.max())
    rmap = _rows_map(g, o)
    perm = g.view("perm", torch.int32, (g.L["rows_cap"],))
    assert np.array_equal(perm[rmap], o.res["perm"])
    inv = g.view("inv", torch.int32, (TK,))
    want = np.full(TK, -1, np.int64)
    want[o.res["perm"]] = rmap
    assert np.array_equal(inv, want)
    assert g.status == 0


@pytest.mark.parametrize("name", list(CASES))
def test_permuted_token_rows_are_the_quantized_rows(name):
    wl, g, o = _run(name)
    rmap = _rows_map(g, o)
    t = o.res["perm"] // wl.K
    rc = g.L["rows_cap"]
    xq = g.view("xq_codes", torch.uint8, (rc, wl.H // 2))
    assert np.array_equal(xq[rmap], o.xc[t])
    xs = g.view("xq_scale", torch.float32, (rc,))
    assert np.array_equal(xs[rmap].view(np.uint32), o.xs[t].view(np.uint32))
    sfp = g.view("xq_sf", torch.uint8, (rc * wl.H // 16,))
    assert np.array_equal(unswizzle(sfp, rmap, wl.H // 16), o.xsf[t])


@pytest.mark.parametrize("name", list(CASES))
def test_fc2_input_requant_within_bounds(name):
    wl, g, o = _run(name)
    rmap = _rows_map(g, o)
    rc, I = g.L["rows_cap"], wl.I
    act = g.view("act", torch.float32, (rc, I))[rmap]
    assert rel_l2(act, o.res["act"]) < 1e-5
    s2 = g.view("fc2q_scale", torch.float32, (rc,))[rmap]
    ref = o.res["s2"]
    assert np.all(np.abs(s2 - ref) <= 1e-5 * np.abs(ref))
    sfg = unswizzle(g.view("fc2q_sf", torch.uint8, (rc * I // 16,)), rmap, I // 16)
    sfo = o.res["fc2sf"]
    d_sf = np.abs(sfg.astype(np.int64) - sfo.astype(np.int64))
    assert d_sf.max() <= 1 and (d_sf > 0).mean() <= 1e-3
    cg = unpack_codes(g.view("fc2q_codes", torch.uint8, (rc, I // 2))[rmap])
    co = unpack_codes(o.res["fc2c"])
    steps = signed_step(cg, co)
    assert steps.max() <= 1 and (steps > 0).mean() <= 1e-3, (steps.max(), (steps > 0).mean())


@pytest.mark.parametrize("name", list(CASES))
def test_route_rows_and_output_rel_l2(name):
    wl, g, o = _run(name)
    rmap = _rows_map(g, o)
    route = g.view("route", torch.int16, (g.L["rows_cap"], wl.H))[rmap].view(np.uint16)
    assert rel_l2(bf16_np(route), bf16_np(o.res["route"])) <= 1e-2
    out = g.out.cpu().view(torch.int16).numpy().view(np.uint16)
    assert rel_l2(bf16_np(out), bf16_np(o.res["out"])) <= 1e-2


# ----------------------------------------------------------------------------- W4A16

class GpuForward16:
    def __init__(self, wl, x, w1, w2, ids, wts):
        dev = "cuda"
        self.wl = wl
        self.w = M.prepare_weights(w1.to(dev), w2.to(dev), wl.act)
        self.ws = M.workspace(self.w, wl.T, wl.K, w4a16=True)
        self.L = M.moe_nvfp4_workspace_layout(self.w.dims, wl.T, wl.K, w4a16=True)
        self.out = M.forward_w4a16(self.w, x.to(dev), ids.to(dev), wts.to(dev), ws=self.ws)
        torch.cuda.synchronize()
        self.status = M.moe_nvfp4_read_status(self.ws)

    def view(self, name, dtype, shape):
        return M.ws_view(self.ws, self.L, name, dtype, shape).cpu().numpy()


_cache16 = {}


def _run16(name):
    if name not in _cache16:
        wl = CASES[name]
        x, w1, w2, ids, wts = _inputs(wl)
        _cache16[name] = (wl, GpuForward16(wl, x, w1, w2, ids, wts),
                          OracleRun(wl, x, w1, w2, ids, wts, w4a16=True), x)
    return _cache16[name]


@pytest.mark.parametrize("name", list(CASES))
def test_w4a16_permuted_rows_and_routing(name):
    wl, g, o, x = _run16(name)
    assert g.status == 0
    counts = g.view("counts", torch.int32, (wl.E,))
    assert np.array_equal(counts, o.res["counts"])
    rmap = _rows_map(g, o)
    perm = g.view("perm", torch.int32, (g.L["rows_cap"],))
    assert np.array_equal(perm[rmap], o.res["perm"])
    # the FC1 GEMM's f16 token rows
    xp = g.view("x_perm", torch.int16, (g.L["rows_cap"], wl.H))[rmap]
    rs = g.view("xq_scale", torch.float32, (g.L["rows_cap"],))[rmap]
    check_scaled_f16_rows(xp, rs, bf16_np(to_np_u16(x)[o.res["perm"] // wl.K]))


@pytest.mark.parametrize("name", list(CASES))
def test_w4a16_handoff_route_rows_and_output(name):
    wl, g, o, x = _run16(name)
    rmap = _rows_map(g, o)
    act = g.view("act_bf16", torch.int16, (g.L["rows_cap"], wl.I))[rmap].view(np.uint16)
    a_g, a_o = bf16_np(act), bf16_np(o.res["act"])
    assert rel_l2(a_g, a_o) <= 4e-3
    # bf16 rounding of an fp32-accumulated vs an fp64 value: one bf16 step apart
    # at most, except where cancellation leaves a value near zero (at most 0.1%)
    step = np.abs(a_g.view(np.int32) - a_o.view(np.int32)) >> 16
    assert (step > 1).mean() <= 1e-3
    # the FC2 GEMM's f16 rows: the handoff rows, scaled
    a16 = g.view("act_f16", torch.int16, (g.L["rows_cap"], wl.I))[rmap]
    ars = g.view("act_scale", torch.float32, (g.L["rows_cap"],))[rmap]
    check_scaled_f16_rows(a16, ars, a_g)
    route = g.view("route", torch.int16, (g.L["rows_cap"], wl.H))[rmap].view(np.uint16)
    assert rel_l2(bf16_np(route), bf16_np(o.res["route"])) <= 1e-2
    out = g.out.cpu().view(torch.int16).numpy().view(np.uint16)
    assert rel_l2(bf16_np(out), bf16_np(o.res["out"])) <= 1e-2
