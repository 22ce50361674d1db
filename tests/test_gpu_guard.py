"""Guards on the GPU: no kernel writes past the end of its output or workspace
buffers (canary bytes after every buffer), and the in-kernel failure detection
works (a bounded wait that can never be satisfied gives up, records a timeout
and leaves the context usable; nothing traps or hangs).
"""
import time

import pytest
import torch

import nvfp4_token_routed_gb300 as M
from nvfp4_token_routed_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"
CANARY = 0xA5
PAD = 4096


def _with_tail(n_bytes):
    """A uint8 buffer of n_bytes followed by PAD canary bytes."""
    b = torch.full((n_bytes + PAD,), CANARY, dtype=torch.uint8, device=DEV)
    return b


def _tail_intact(b, n_bytes):
    return bool((b[n_bytes:] == CANARY).all())


@pytest.mark.parametrize("wl", [
    W.Workload("swiglu_T40_H320_I192_E32_K4", 40, 320, 192, 32, 4, "swiglu"),   # one launch, padded
    W.Workload("relu2_T300_H512_I256_E4_K2", 300, 512, 256, 4, 2, "relu2"),     # three launches
], ids=lambda w: w.name)
def test_no_writes_past_any_buffer(wl):
    x = W.make_x(wl, device=DEV)
    w1, w2 = W.make_weights(wl, device=DEV)
    ids, wts = W.make_routing(wl, device=DEV)
    w = M.prepare_weights(w1, w2, wl.act)
    Hp = M.padded(wl.H)
    T, H, K = wl.T, wl.H, wl.K
    # quantized tokens
    nc, ns, nsc = T * Hp // 2, T * Hp // 16, T * 4
    bc, bs, bsc = _with_tail(nc), _with_tail(ns), _with_tail(nsc)
    codes, sf = bc[:nc].view(T, Hp // 2), bs[:ns].view(T, Hp // 16)
    scale = bsc[:nsc].view(torch.float32)
    M.moe_nvfp4_quantize_tokens(x, codes, sf, scale)
    # W4A4 and W4A16 forwards into canary-guarded output and workspace
    for w4a16 in (False, True):
        nws = M.moe_nvfp4_workspace_bytes(w.dims, T, K, w4a16)
        bws = _with_tail(nws)
        ws = bws[:nws]
        nout = T * H * 2
        bout = _with_tail(nout)
        out = bout[:nout].view(torch.bfloat16).view(T, H)
        if w4a16:
            M.moe_nvfp4_forward_w4a16(w.dims, w, x, ids, wts, out, ws)
        else:
            M.moe_nvfp4_forward(w.dims, w, codes, sf, scale, ids, wts, out, ws)
        torch.cuda.synchronize()
        assert M.moe_nvfp4_read_status(ws) == 0
        assert _tail_intact(bws, nws), "workspace overrun"
        assert _tail_intact(bout, nout), "output overrun"
    for b, n in ((bc, nc), (bs, ns), (bsc, nsc)):
        assert _tail_intact(b, n), "quantized-token overrun"


def test_bounded_waits_time_out_and_leave_the_context_usable():
    ws = torch.empty(1 << 16, dtype=torch.uint8, device=DEV)
    t0 = time.time()
    M.moe_nvfp4_selftest_wait_timeout(ws)
    assert M.moe_nvfp4_read_status(ws) == 8  # MOE_ERR_DEVICE_TIMEOUT
    dt = time.time() - t0
    assert 3.0 < dt < 30.0, dt  # two waits of about 2 s each
    # the context still works: a forward afterwards is correct and error-free
    wl = W.TINY_RELU2
    x = W.make_x(wl, device=DEV)
    w1, w2 = W.make_weights(wl, device=DEV)
    ids, wts = W.make_routing(wl, device=DEV)
    w = M.prepare_weights(w1, w2, wl.act)
    c, s, sc = M.quantize_tokens(x)
    ws2 = M.workspace(w, wl.T, wl.K)
    out = M.forward(w, c, s, sc, ids, wts, ws=ws2)
    torch.cuda.synchronize()
    assert M.moe_nvfp4_read_status(ws2) == 0 and torch.isfinite(out.float()).all()
