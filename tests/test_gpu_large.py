"""Full-size workloads on the GPU, checked against the oracle on what it can
afford: every token's quantization and the whole routing permutation bit-exact,
and, for a seeded sample of tokens, the prepared weights of the experts they
use (bit-exact) and their final outputs (relative L2 <= 1e-2).  The GPU runs
the full batch in the same launch configuration bench.py times.
"""
import gc

import numpy as np
import pytest
import torch

import nvfp4_token_routed_gb300 as M
from nvfp4_token_routed_gb300 import workloads as W
from oracle import oracle as O

from helpers import TILE_ROWS, bf16_np, rel_l2, stored_fc1_rows, to_np_u16

pytestmark = pytest.mark.gpu
DEV = "cuda"

LARGE = {
    "mid_zipf_T2048": W.MID_ZIPF,
    "dsv3_T1": W.DSV3_LIKE.with_T(1),
    "dsv3_T4096": W.DSV3_LIKE.with_T(4096),
    "e384_T4096": W.PAGES_E384.with_T(4096),
}


@pytest.mark.parametrize("name", list(LARGE))
def test_full_size_workload(name):
    wl = LARGE[name]
    x = W.make_x(wl, device=DEV)
    w1, w2 = W.make_weights(wl, device=DEV)
    ids, wts = W.make_routing(wl, device=DEV)
    w = M.prepare_weights(w1, w2, wl.act)
    codes, sf, scale = M.quantize_tokens(x)
    ws = M.workspace(w, wl.T, wl.K)
    out = M.forward(w, codes, sf, scale, ids, wts, ws=ws)
    torch.cuda.synchronize()
    assert M.moe_nvfp4_read_status(ws) == 0

    # every token's quantization
    oc, osf, os_ = O.quantize_tokens(to_np_u16(x))
    assert np.array_equal(codes.cpu().numpy(), oc)
    assert np.array_equal(sf.cpu().numpy(), osf)
    assert np.array_equal(scale.cpu().numpy(), os_)

    # the whole routing permutation
    idsn = ids.cpu().numpy()
    counts, perm, inv = O.route(idsn, wl.E)
    L = M.moe_nvfp4_workspace_layout(w.dims, wl.T, wl.K)
    gcounts = M.ws_view(ws, L, "counts", torch.int32, (wl.E,)).cpu().numpy()
    assert np.array_equal(gcounts, counts)
    row0 = M.ws_view(ws, L, "group_row0", torch.int32, (wl.E,)).cpu().numpy()
    tiles = -(-counts // TILE_ROWS)
    assert np.array_equal(row0, TILE_ROWS * np.concatenate([[0], np.cumsum(tiles)[:-1]]))
    start = np.concatenate([[0], np.cumsum(counts)[:-1]])
    qe = np.repeat(np.arange(wl.E), counts)
    rmap = row0[qe] + (np.arange(perm.size) - start[qe])
    gperm = M.ws_view(ws, L, "perm", torch.int32, (L["rows_cap"],)).cpu().numpy()
    assert np.array_equal(gperm[rmap], perm)

    # a seeded sample of tokens through the oracle, with only the experts they use
    g = np.random.default_rng(7)
    sample = np.sort(g.choice(wl.T, size=min(4, wl.T), replace=False))
    s_ids = idsn[sample]
    used = np.unique(s_ids[s_ids >= 0])
    idx = torch.as_tensor(used, device=DEV)
    sw1 = to_np_u16(w1.index_select(0, idx))
    sw2 = to_np_u16(w2.index_select(0, idx))
    Wt = O.Weights(sw1, sw2)
    rows = stored_fc1_rows(wl.N1, wl.I, wl.act)
    g1 = w.fc1_codes.index_select(0, idx).cpu().numpy()
    assert np.array_equal(g1, Wt.w1c[:, rows])
    assert np.array_equal(w.fc1_alpha[idx].cpu().numpy(), Wt.a1)
    assert np.array_equal(w.fc2_codes.index_select(0, idx).cpu().numpy(), Wt.w2c)
    assert np.array_equal(w.fc2_alpha[idx].cpu().numpy(), Wt.a2)
    remap = np.full(wl.E, -1, np.int32)
    remap[used] = np.arange(used.size, dtype=np.int32)
    sub = np.where(s_ids >= 0, remap[np.clip(s_ids, 0, None)], -1).astype(np.int32)
    res = O.forward_w4a4(Wt, oc[sample], osf[sample], os_[sample], sub,
                         wts.cpu().numpy()[sample], used.size, wl.H, wl.I, wl.act)
    got = out[torch.as_tensor(sample, device=DEV)].cpu().view(torch.int16).numpy().view(np.uint16)
    assert rel_l2(bf16_np(got), bf16_np(res["out"])) <= 1e-2

    del x, w1, w2, w, ws, out, codes, sf, scale
    gc.collect()
    torch.cuda.empty_cache()


LARGE16 = {
    "e384_T1024_w4a16": W.PAGES_E384.with_T(1024),
    "dsv3_T128_w4a16": W.DSV3_LIKE.with_T(128),
}


@pytest.mark.parametrize("name", list(LARGE16))
def test_full_size_workload_w4a16(name):
    wl = LARGE16[name]
    x = W.make_x(wl, device=DEV)
    w1, w2 = W.make_weights(wl, device=DEV)
    ids, wts = W.make_routing(wl, device=DEV)
    w = M.prepare_weights(w1, w2, wl.act)
    ws = M.workspace(w, wl.T, wl.K, w4a16=True)
    out = M.forward_w4a16(w, x, ids, wts, ws=ws)
    torch.cuda.synchronize()
    assert M.moe_nvfp4_read_status(ws) == 0
    idsn = ids.cpu().numpy()
    g = np.random.default_rng(11)
    sample = np.sort(g.choice(wl.T, size=min(4, wl.T), replace=False))
    s_ids = idsn[sample]
    used = np.unique(s_ids[s_ids >= 0])
    idx = torch.as_tensor(used, device=DEV)
    Wt = O.Weights(to_np_u16(w1.index_select(0, idx)), to_np_u16(w2.index_select(0, idx)))
    remap = np.full(wl.E, -1, np.int32)
    remap[used] = np.arange(used.size, dtype=np.int32)
    sub = np.where(s_ids >= 0, remap[np.clip(s_ids, 0, None)], -1).astype(np.int32)
    xs = to_np_u16(x)[sample]
    res = O.forward_w4a16(Wt, xs, sub, wts.cpu().numpy()[sample], used.size, wl.H, wl.I, wl.act)
    got = out[torch.as_tensor(sample, device=DEV)].cpu().view(torch.int16).numpy().view(np.uint16)
    assert rel_l2(bf16_np(got), bf16_np(res["out"])) <= 1e-2
    del x, w1, w2, w, ws, out
    gc.collect()
    torch.cuda.empty_cache()
