"""Full-size workloads on the GPU, checked against the oracle on what it can
afford.  The GPU runs the whole batch in the launch configuration bench.py
times; the oracle checks every token's quantization and the whole routing
permutation bit-exact, and, for a seeded sample of tokens (32, or every token
of a smaller batch), the prepared weights of the experts they use (bit-exact),
their FC2-input requantization (the pages' bound), their per-route rows and
their final outputs (relative L2 <= 1e-2).

The sweep points are those of the mid-scale Zipf layer (T=2048), the
H7168/I2048/E256 top-8 SwiGLU layer (T in {1, 16, 128, 512, 4096}; W4A16 at
128 and 4096) and the
pages' benchmark shape H7168/I3072/E384 top-6 (W4A4 at T in {512, 1024, 4096},
W4A16 at T in {512, 1024, 4096}).  Each layer's weights are drawn and prepared
once for all its sweep points.
"""
import gc
import types

import numpy as np
import pytest
import torch

import nvfp4_token_routed_gb300 as M
from nvfp4_token_routed_gb300 import workloads as W
from oracle import oracle as O

from helpers import (TILE_ROWS, bf16_np, rel_l2, signed_step, stored_fc1_rows,
                     to_np_u16, unpack_codes, unswizzle)

pytestmark = pytest.mark.gpu
DEV = "cuda"
SAMPLE = 32

# (layer, T, variant); cases of one layer are adjacent so its weights are drawn once
CASES = [(W.MID_ZIPF, 2048, "w4a4")]
CASES += [(W.DSV3_LIKE, T, "w4a4") for T in (1, 16, 128, 512, 4096)]
CASES += [(W.DSV3_LIKE, T, "w4a16") for T in (128, 4096)]   # 4096: 128-token tiles in halves
CASES += [(W.PAGES_E384, T, "w4a4") for T in (512, 1024, 4096)]
CASES += [(W.PAGES_E384, T, "w4a16") for T in (512, 1024, 4096)]


class Layer:
    """One layer's BF16 weights on the device, the GPU-prepared weights and the
    oracle's preparation of the experts used so far (prepared in batches, each
    expert once)."""

    def __init__(self, wl):
        self.wl = wl
        self.w1, self.w2 = W.make_weights(wl, device=DEV)
        self.w = M.prepare_weights(self.w1, self.w2, wl.act)
        torch.cuda.synchronize()
        self.prep = {}      # expert -> (w1c, w1sf, a1, w2c, w2sf, a2)
        self.checked = set()

    def oracle_weights(self, used):
        todo = [int(e) for e in used if int(e) not in self.prep]
        for i in range(0, len(todo), 16):
            batch = todo[i:i + 16]
            idx = torch.as_tensor(batch, device=DEV)
            c1, f1, a1 = O.prepare_fc(to_np_u16(self.w1.index_select(0, idx)))
            c2, f2, a2 = O.prepare_fc(to_np_u16(self.w2.index_select(0, idx)))
            for j, e in enumerate(batch):
                self.prep[e] = (c1[j], f1[j], a1[j], c2[j], f2[j], a2[j])
        p = [self.prep[int(e)] for e in used]
        return types.SimpleNamespace(**{k: np.stack([q[i] for q in p])
                                        for i, k in enumerate(("w1c", "w1sf", "a1", "w2c", "w2sf",
                                                               "a2"))})

    def check_prepared(self, used, Wt):
        """The GPU-prepared codes and alphas of experts not yet compared."""
        new = [i for i, e in enumerate(used) if int(e) not in self.checked]
        if not new:
            return
        wl = self.wl
        idx = torch.as_tensor(used[new], device=DEV)
        rows = stored_fc1_rows(wl.N1, wl.I, wl.act)
        assert np.array_equal(self.w.fc1_codes.index_select(0, idx).cpu().numpy(),
                              Wt.w1c[new][:, rows])
        assert np.array_equal(self.w.fc1_alpha[idx].cpu().numpy(), Wt.a1[new])
        assert np.array_equal(self.w.fc2_codes.index_select(0, idx).cpu().numpy(), Wt.w2c[new])
        assert np.array_equal(self.w.fc2_alpha[idx].cpu().numpy(), Wt.a2[new])
        self.checked.update(int(e) for e in used[new])


_layer = {}


def layer_of(wl):
    if wl.name not in _layer:
        _layer.clear()
        gc.collect()
        torch.cuda.empty_cache()
        _layer[wl.name] = Layer(wl)
    return _layer[wl.name]


def _sample(T, seed):
    g = np.random.default_rng(seed)
    return np.sort(g.choice(T, size=min(SAMPLE, T), replace=False))


def _sub_problem(idsn, sample, E):
    """The sample's ids renumbered over the experts it uses."""
    s_ids = idsn[sample]
    used = np.unique(s_ids[(s_ids >= 0) & (s_ids < E)])
    remap = np.full(E, -1, np.int32)
    remap[used] = np.arange(used.size, dtype=np.int32)
    sub = np.where(s_ids >= 0, remap[np.clip(s_ids, 0, None)], -1).astype(np.int32)
    return used, sub


def _check_routing(ws, L, idsn, E):
    counts, perm, inv = O.route(idsn, E)
    gcounts = M.ws_view(ws, L, "counts", torch.int32, (E,)).cpu().numpy()
    assert np.array_equal(gcounts, counts)
    row0 = M.ws_view(ws, L, "group_row0", torch.int32, (E,)).cpu().numpy()
    tiles = -(-counts // TILE_ROWS)
    assert np.array_equal(row0, TILE_ROWS * np.concatenate([[0], np.cumsum(tiles)[:-1]]))
    start = np.concatenate([[0], np.cumsum(counts)[:-1]])
    qe = np.repeat(np.arange(E), counts)
    rmap = row0[qe] + (np.arange(perm.size) - start[qe])
    gperm = M.ws_view(ws, L, "perm", torch.int32, (L["rows_cap"],)).cpu().numpy()
    assert np.array_equal(gperm[rmap], perm)
    ginv = M.ws_view(ws, L, "inv", torch.int32, (idsn.size,)).cpu().numpy()
    want = np.full(idsn.size, -1, np.int64)
    want[perm] = rmap
    assert np.array_equal(ginv, want)
    return ginv


def _sample_rows(ginv, res, sample, K):
    """GPU permuted rows and oracle sub-problem rows of the sample's routes."""
    gi = ginv.reshape(-1, K)[sample].ravel()
    oi = res["inv"]
    keep = oi >= 0
    assert np.array_equal(keep, gi >= 0)
    return gi[keep], oi[keep]


@pytest.mark.parametrize("wl,T,variant", CASES,
                         ids=[f"{wl.name}-T{T}-{v}" for wl, T, v in CASES])
def test_full_size_workload(wl, T, variant):
    wl = wl.with_T(T)
    lay = layer_of(W.ALL[wl.name.split("@")[0]])
    x = W.make_x(wl, device=DEV)
    ids, wts = W.make_routing(wl, device=DEV)
    w16 = variant == "w4a16"
    ws = M.workspace(lay.w, wl.T, wl.K, w4a16=w16)
    L = M.moe_nvfp4_workspace_layout(lay.w.dims, wl.T, wl.K, w16)
    if w16:
        out = M.forward_w4a16(lay.w, x, ids, wts, ws=ws)
    else:
        codes, sf, scale = M.quantize_tokens(x)
        out = M.forward(lay.w, codes, sf, scale, ids, wts, ws=ws)
    torch.cuda.synchronize()
    assert M.moe_nvfp4_read_status(ws) == 0
    idsn = ids.cpu().numpy()
    wtn = wts.cpu().numpy()
    xn = to_np_u16(x)

    if not w16:  # every token's quantization
        oc, osf, os_ = O.quantize_tokens(xn)
        assert np.array_equal(codes.cpu().numpy(), oc)
        assert np.array_equal(sf.cpu().numpy(), osf)
        assert np.array_equal(scale.cpu().numpy(), os_)
    ginv = _check_routing(ws, L, idsn, wl.E)     # the whole routing permutation

    # a seeded sample of tokens through the oracle, with only the experts they use
    sample = _sample(wl.T, seed=7 + T)
    used, sub = _sub_problem(idsn, sample, wl.E)
    Wt = lay.oracle_weights(used)
    lay.check_prepared(used, Wt)
    if w16:
        res = O.forward_w4a16(Wt, xn[sample], sub, wtn[sample], used.size, wl.H, wl.I, wl.act)
    else:
        res = O.forward_w4a4(Wt, oc[sample], osf[sample], os_[sample], sub, wtn[sample],
                             used.size, wl.H, wl.I, wl.act)
    gp, op = _sample_rows(ginv, res, sample, wl.K)
    Hp, Ip = M.padded(wl.H), M.padded(wl.I)
    rc = L["rows_cap"]
    route = M.ws_view(ws, L, "route", torch.int16, (rc, Hp))
    route = route[torch.as_tensor(gp, device=DEV)].cpu().numpy().view(np.uint16)[:, :wl.H]
    assert rel_l2(bf16_np(route), bf16_np(res["route"][op])) <= 1e-2
    if not w16:
        # FC2-input requant of the sample's routes within the pages' bound
        idx = torch.as_tensor(gp, device=DEV)
        s2 = M.ws_view(ws, L, "fc2q_scale", torch.float32, (rc,))[idx].cpu().numpy()
        assert np.all(np.abs(s2 - res["s2"][op]) <= 1e-5 * np.abs(res["s2"][op]))
        cg = unpack_codes(M.ws_view(ws, L, "fc2q_codes", torch.uint8, (rc, Ip // 2))[idx]
                          .cpu().numpy())[:, :wl.I]
        steps = signed_step(cg, unpack_codes(res["fc2c"][op]))
        assert steps.max() <= 1 and (steps > 0).mean() <= 1e-3, (steps.max(), (steps > 0).mean())
        plane = M.ws_view(ws, L, "fc2q_sf", torch.uint8, (rc * Ip // 16,)).cpu().numpy()
        sfg = unswizzle(plane, gp, Ip // 16)[:, :wl.I // 16]
        d_sf = np.abs(sfg.astype(np.int64) - res["fc2sf"][op].astype(np.int64))
        assert d_sf.max() <= 1 and (d_sf > 0).mean() <= 1e-3
    else:
        # the bf16 handoff of the sample's routes
        act = M.ws_view(ws, L, "act_bf16", torch.int16, (rc, Ip))
        act = act[torch.as_tensor(gp, device=DEV)].cpu().numpy().view(np.uint16)
        act = act[:, :wl.I]
        assert rel_l2(bf16_np(act), bf16_np(res["act"][op])) <= 1e-2
    got = out[torch.as_tensor(sample, device=DEV)].cpu().view(torch.int16).numpy().view(np.uint16)
    assert rel_l2(bf16_np(got), bf16_np(res["out"])) <= 1e-2
    for i in range(sample.size):  # and token by token
        assert rel_l2(bf16_np(got[i]), bf16_np(res["out"][i])) <= 2e-2

    del x, ws, out
    if not w16:
        del codes, sf, scale
    torch.cuda.empty_cache()


def test_release_large_layers():
    """Not a check: frees the last layer's device memory for the tests after this file."""
    _layer.clear()
    gc.collect()
    torch.cuda.empty_cache()
