"""CUDA-graph capture and bitwise replay (Megatron-LM PR #8262, "What is tested",
CUDA-graph capture and bitwise replay; layer level: graph replay follows new
inputs and refreshed weights).

The whole step -- token quantization and the W4A4 forward, or the W4A16
forward -- is captured once.  Replays must equal eager calls bit for bit after
new inputs are copied into the captured buffers and after the weights are
refreshed in place.
"""
import pytest
import torch

import nvfp4_token_routed_gb300 as M
from nvfp4_token_routed_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"

WL = W.Workload("swiglu_T96_H512_I256_E16_K4", 96, 512, 256, 16, 4, "swiglu")


def _inputs(seed):
    wl = WL
    x = W.make_x(wl, device=DEV, seed=seed + 1)
    ids, wts = W.make_routing(wl, device=DEV, seed=seed + 4)
    return x, ids, wts


def _weights(seed):
    return W.make_weights(WL, device=DEV, seed=seed)


def _same(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("w4a16", [False, True])
def test_graph_replay_is_bitwise_and_follows_inputs_and_refits(w4a16):
    wl = WL
    w1, w2 = _weights(100)
    w = M.prepare_weights(w1, w2, wl.act)
    x, ids, wts = _inputs(200)
    # captured buffers
    gx, gids, gwts = x.clone(), ids.clone(), wts.clone()
    Hp = M.padded(wl.H)
    codes = torch.empty(wl.T, Hp // 2, dtype=torch.uint8, device=DEV)
    sf = torch.empty(wl.T, Hp // 16, dtype=torch.uint8, device=DEV)
    scale = torch.empty(wl.T, dtype=torch.float32, device=DEV)
    out = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device=DEV)
    ws = M.workspace(w, wl.T, wl.K, w4a16=w4a16)
    stream = torch.cuda.Stream()

    def step():
        if w4a16:
            M.moe_nvfp4_forward_w4a16(w.dims, w, gx, gids, gwts, out, ws, stream)
        else:
            M.moe_nvfp4_quantize_tokens(gx, codes, sf, scale, stream)
            M.moe_nvfp4_forward(w.dims, w, codes, sf, scale, gids, gwts, out, ws, stream)

    def eager(xe, ide, wte):
        if w4a16:
            return M.forward_w4a16(w, xe, ide, wte)
        c, s_, sc = M.quantize_tokens(xe)
        return M.forward(w, c, s_, sc, ide, wte)

    with torch.cuda.stream(stream):
        step()  # the device check runs outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
    torch.cuda.synchronize()

    # 1. replay == eager on the captured inputs, and replays repeat bit for bit
    g.replay()
    torch.cuda.synchronize()
    ref = eager(x, ids, wts)
    torch.cuda.synchronize()
    assert _same(out, ref)
    first = out.clone()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert _same(out, first)

    # 2. new inputs copied into the captured buffers
    x2, ids2, wts2 = _inputs(300)
    gx.copy_(x2)
    gids.copy_(ids2)
    gwts.copy_(wts2)
    g.replay()
    torch.cuda.synchronize()
    assert _same(out, eager(x2, ids2, wts2))
    assert not _same(out, first)

    # 3. weights refreshed in place (same addresses) after a refit
    v1, v2 = _weights(400)
    M.prepare_weights(v1, v2, wl.act, out=w)
    g.replay()
    torch.cuda.synchronize()
    after = out.clone()
    assert _same(after, eager(x2, ids2, wts2))
    w_fresh = M.prepare_weights(v1, v2, wl.act)
    if w4a16:
        fresh = M.forward_w4a16(w_fresh, x2, ids2, wts2)
    else:
        c, s_, sc = M.quantize_tokens(x2)
        fresh = M.forward(w_fresh, c, s_, sc, ids2, wts2)
    torch.cuda.synchronize()
    assert _same(after, fresh)
    assert M.moe_nvfp4_read_status(ws) == 0
