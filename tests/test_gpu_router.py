"""The plain top-K router on the GPU against the oracle (Megatron-LM PR #8262,
"Performance": plain top-k routing).  Bars: expert ids bit-exact (the decision
is a comparison of the same fp32 logits on both sides), scores within 2e-6
relative of the oracle's fp64 softmax, per-token results batch invariant.
"""
import numpy as np
import pytest
import torch

import nvfp4_token_routed_gb300 as M
from oracle import oracle as O

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _logits(T, E, kind, seed):
    g = np.random.default_rng(seed)
    if kind == "normal":
        return g.standard_normal((T, E)).astype(np.float32)
    if kind == "ties":      # few distinct values: many exact ties
        return g.integers(-3, 4, size=(T, E)).astype(np.float32)
    if kind == "extreme":   # -inf entries, huge spreads, equal rows
        x = (g.standard_normal((T, E)) * 50).astype(np.float32)
        x[:, ::7] = -np.inf
        x[0, :] = 1.0
        x[1, :] = -np.inf
        return x
    raise ValueError(kind)


@pytest.mark.parametrize("E,K", [(8, 2), (64, 8), (256, 8), (384, 6), (1000, 32), (33, 32)])
@pytest.mark.parametrize("kind", ["normal", "ties", "extreme"])
def test_router_matches_the_oracle(E, K, kind):
    T = 257
    lg = _logits(T, E, kind, seed=E * 7 + K)
    ref_ids, ref_w = O.route_topk(lg, K)
    ids, w = M.route_topk(torch.from_numpy(lg).to(DEV), K)
    torch.cuda.synchronize()
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    got = w.cpu().numpy()
    finite = np.isfinite(ref_w)
    assert np.array_equal(finite, np.isfinite(got))
    assert np.allclose(got[finite], ref_w[finite], rtol=2e-6, atol=1e-12)


def test_router_batch_invariance_and_feeds_the_layer():
    T, E, K = 300, 64, 8
    lg = torch.from_numpy(_logits(T, E, "normal", seed=1)).to(DEV)
    ids, w = M.route_topk(lg, K)
    sel = torch.randperm(T, generator=torch.Generator().manual_seed(2))[:17].to(DEV)
    ids2, w2 = M.route_topk(lg[sel], K)
    torch.cuda.synchronize()
    assert torch.equal(ids2, ids[sel]) and torch.equal(w2.view(torch.int32), w[sel].view(torch.int32))
    # the router output drives the expert layer directly
    from nvfp4_token_routed_gb300 import workloads as W
    wl = W.Workload("swiglu_T300_H256_I256_E64_K8", T, 256, 256, E, K, "swiglu")
    w1, w2_ = W.make_weights(wl, device=DEV)
    x = W.make_x(wl, device=DEV)
    pw = M.prepare_weights(w1, w2_, wl.act)
    c, s, sc = M.quantize_tokens(x)
    ws = M.workspace(pw, T, K)
    out = M.forward(pw, c, s, sc, ids, w, ws=ws)
    torch.cuda.synchronize()
    assert M.moe_nvfp4_read_status(ws) == 0 and torch.isfinite(out.float()).all()
