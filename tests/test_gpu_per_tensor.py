"""Per-tensor NVFP4 x NVFP4 recipe on the GPU (Megatron-LM PR #8262, "How to
extend", "Per-tensor NVFP4 x NVFP4"): static calibrated FC1 / FC2 input scales,
folded into the alphas; weight codes and block scales unchanged.

Bars: static token quantization and the folded alphas bit-exact against the
oracle, weight codes and scales identical to the per-token preparation, FC2
input codes at most one E2M1 step apart in at most 0.1% of elements, output
relative L2 <= 1e-2 against the oracle's per-tensor forward, per-token outputs
bitwise batch invariant.
"""
import numpy as np
import pytest
import torch

import nvfp4_token_routed_gb300 as M
from nvfp4_token_routed_gb300 import workloads as W
from oracle import oracle as O

from helpers import TILE_ROWS, bf16_np, rel_l2, signed_step, to_np_u16, unpack_codes

pytestmark = pytest.mark.gpu
DEV = "cuda"

CASES = {
    "relu2_tiny": W.TINY_RELU2,
    "swiglu_ragged": W.Workload("swiglu_T300_H512_I256_E4_K2", 300, 512, 256, 4, 2, "swiglu"),
    "relu2_padded": W.Workload("relu2_T64_H320_I192_E8_K2", 64, 320, 192, 8, 2, "relu2"),
}


def _calibrate(wl, x, w1, w2, ids, wts):
    """Static scales as a calibration pass would set them: 2688 / amax of the
    FC1 inputs and of the activated FC1 rows over the batch (fp32)."""
    a1 = np.float32(np.float32(2688.0) / np.float32(x.float().abs().max().item()))
    Wt = O.Weights(to_np_u16(w1), to_np_u16(w2))
    xc, xsf, xs = O.quantize_tokens(to_np_u16(x))
    ref = O.forward_w4a4(Wt, xc, xsf, xs, ids.numpy(), wts.numpy(), wl.E, wl.H, wl.I, wl.act)
    a2 = np.float32(np.float32(2688.0) / np.float32(np.abs(ref["act"]).max()))
    return a1, a2


@pytest.mark.parametrize("name", list(CASES))
def test_per_tensor_matches_the_oracle(name):
    wl = CASES[name]
    x = W.make_x(wl)
    w1, w2 = W.make_weights(wl)
    ids, wts = W.make_routing(wl)
    a1, a2 = _calibrate(wl, x, w1, w2, ids, wts)
    Wpt = O.WeightsPerTensor(to_np_u16(w1), to_np_u16(w2), a1, a2)
    xc, xsf = O.quantize_tokens_static(to_np_u16(x), a1)
    ref = O.forward_w4a4_per_tensor(Wpt, xc, xsf, a2, ids.numpy(), wts.numpy(), wl.E, wl.H, wl.I,
                                    wl.act)

    d_a1 = torch.tensor([a1], dtype=torch.float32, device=DEV)
    d_a2 = torch.tensor([a2], dtype=torch.float32, device=DEV)
    w = M.prepare_weights_per_tensor(w1.to(DEV), w2.to(DEV), wl.act, d_a1, d_a2)
    w_tok = M.prepare_weights(w1.to(DEV), w2.to(DEV), wl.act)
    codes, sf = M.quantize_tokens_static(x.to(DEV), d_a1)
    ws = M.workspace(w, wl.T, wl.K)
    out = M.forward_per_tensor(w, codes, sf, d_a2, ids.to(DEV), wts.to(DEV), ws=ws)
    torch.cuda.synchronize()
    assert M.moe_nvfp4_read_status(ws) == 0

    # alphas folded, codes and block scales those of the per-token preparation
    assert np.array_equal(w.fc1_alpha.cpu().numpy(), Wpt.a1)
    assert np.array_equal(w.fc2_alpha.cpu().numpy(), Wpt.a2)
    for a, b in [(w.fc1_codes, w_tok.fc1_codes), (w.fc1_sf, w_tok.fc1_sf),
                 (w.fc2_codes, w_tok.fc2_codes), (w.fc2_sf, w_tok.fc2_sf)]:
        assert torch.equal(a, b)
    # static token quantization, bit-exact on the real columns, zero padding
    H = wl.H
    g_codes, g_sf = codes.cpu().numpy(), sf.cpu().numpy()
    assert np.array_equal(g_codes[:, : H // 2], xc) and not g_codes[:, H // 2:].any()
    assert np.array_equal(g_sf[:, : H // 16], xsf) and not g_sf[:, H // 16:].any()

    # FC2 input: static requant codes within one step in <= 0.1% of elements
    L = M.moe_nvfp4_workspace_layout(w.dims, wl.T, wl.K)
    Ip = M.padded(wl.I)
    inv = M.ws_view(ws, L, "inv", torch.int32, (wl.T * wl.K,)).cpu().numpy()
    g_fc2 = M.ws_view(ws, L, "fc2q_codes", torch.uint8, (L["rows_cap"], Ip // 2)).cpu().numpy()
    q_of_route = ref["inv"]
    valid = inv >= 0
    got_rows = g_fc2[inv[valid]][:, : wl.I // 2]
    ref_rows = ref["fc2c"][q_of_route[valid]]
    steps = signed_step(unpack_codes(got_rows), unpack_codes(ref_rows))
    assert steps.max() <= 1 and (steps > 0).mean() <= 1e-3
    s2 = M.ws_view(ws, L, "fc2q_scale", torch.float32, (L["rows_cap"],)).cpu().numpy()
    assert np.all(s2[inv[valid]] == 1.0)

    got = bf16_np(to_np_u16(out))
    assert rel_l2(got, bf16_np(ref["out"])) <= 1e-2


def test_per_tensor_batch_invariance():
    wl = CASES["swiglu_ragged"]
    x = W.make_x(wl, device=DEV)
    w1, w2 = W.make_weights(wl, device=DEV)
    ids, wts = W.make_routing(wl, device=DEV)
    d_a1 = torch.tensor([2688.0 / x.float().abs().max().item()], dtype=torch.float32, device=DEV)
    d_a2 = torch.tensor([64.0], dtype=torch.float32, device=DEV)
    w = M.prepare_weights_per_tensor(w1, w2, wl.act, d_a1, d_a2)
    codes, sf = M.quantize_tokens_static(x, d_a1)
    full = M.forward_per_tensor(w, codes, sf, d_a2, ids, wts)
    g = torch.Generator().manual_seed(9)
    for n in (1, 7, 128):
        sel = torch.randperm(wl.T, generator=g)[:n].to(DEV)
        c, s = M.quantize_tokens_static(x[sel], d_a1)
        part = M.forward_per_tensor(w, c, s, d_a2, ids[sel], wts[sel])
        torch.cuda.synchronize()
        assert torch.equal(part.view(torch.int16), full[sel].view(torch.int16))
