"""GPU edge cases, batch invariance and the hand-worked fixtures, through the C ABI.

Batch invariance is the pages' protocol (Megatron-LM PR #8262, "What is
tested", batch invariance): a target batch's per-token outputs are bitwise
identical alone and inside batches of 193 and 1024 tokens whose co-batched
tokens are 100x larger and routed to the same experts; plus subsets T in
{1, 7, 128} of a 128-token master set in shuffled orders.
"""
import json
import os

import numpy as np
import pytest
import torch

import nvfp4_token_routed_gb300 as M
from nvfp4_token_routed_gb300 import workloads as W
from oracle import oracle as O

from helpers import OracleRun, bf16_np, rel_l2, to_np_u16

pytestmark = pytest.mark.gpu
DEV = "cuda"
GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _fwd(w, x, ids, wts):
    codes, sf, scale = M.quantize_tokens(x)
    return M.forward(w, codes, sf, scale, ids, wts)


@pytest.fixture(scope="module")
def e64():
    wl = W.SWIGLU_E64
    w1, w2 = W.make_weights(wl)
    w = M.prepare_weights(w1.to(DEV), w2.to(DEV), wl.act)
    x = W.make_x(wl).to(DEV)
    ids, wts = W.make_routing(wl)
    return wl, w, x, ids.to(DEV), wts.to(DEV)


def test_batch_invariance_subsets_and_shuffles(e64):
    wl, w, x, ids, wts = e64
    full = _fwd(w, x, ids, wts)
    g = torch.Generator().manual_seed(W.BASE_SEED + 5)
    for T in (1, 7, 128):
        for _ in range(3):
            sel = torch.randperm(wl.T, generator=g)[:T].to(DEV)
            out = _fwd(w, x[sel].contiguous(), ids[sel].contiguous(), wts[sel].contiguous())
            assert torch.equal(out.view(torch.int16), full[sel].view(torch.int16)), T


def test_batch_invariance_pages_protocol(e64):
    """Target batch alone vs inside 193- and 1024-token batches of 100x larger
    tokens routed to the same experts."""
    wl, w, x, ids, wts = e64
    tgt = slice(0, 7)
    alone = _fwd(w, x[tgt].contiguous(), ids[tgt].contiguous(), wts[tgt].contiguous())
    g = torch.Generator(device=DEV).manual_seed(W.BASE_SEED + 6)
    for total in (193, 1024):
        n_other = total - 7
        big = (torch.randn(n_other, wl.H, generator=g, device=DEV) * 100.0).to(torch.bfloat16)
        rep = torch.arange(n_other, device=DEV) % 7           # same experts as the targets
        xb = torch.cat([big[: n_other // 2], x[tgt], big[n_other // 2:]])
        ib = torch.cat([ids[tgt][rep][: n_other // 2], ids[tgt], ids[tgt][rep][n_other // 2:]])
        wb = torch.cat([wts[tgt][rep][: n_other // 2], wts[tgt], wts[tgt][rep][n_other // 2:]])
        out = _fwd(w, xb.contiguous(), ib.contiguous(), wb.contiguous())
        got = out[n_other // 2: n_other // 2 + 7]
        assert torch.equal(got.view(torch.int16), alone.view(torch.int16)), total


def test_repeat_is_bitwise_deterministic(e64):
    wl, w, x, ids, wts = e64
    a = _fwd(w, x, ids, wts)
    b = _fwd(w, x, ids, wts)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_empty_slots_invalid_ids_and_zero_tokens():
    wl = W.Workload("edge_relu2_T40_H256_I512_E8_K3", 40, 256, 512, 8, 3, "relu2")
    x = W.make_x(wl)
    x[5] = 0.0                       # an all-zero token
    w1, w2 = W.make_weights(wl)
    w1[3] = 0.0                      # an all-zero expert (alpha 0)
    ids, wts = W.make_routing(wl)
    ids[0, :] = -1                   # a token with no route -> zero output
    ids[1, 1] = -1                   # one empty slot
    ids[2, 0] = wl.E + 3             # invalid id: slot ignored, status flagged
    ids[3, 2] = -7
    o_ids = ids.clone()
    o_ids[2, 0] = -1
    o_ids[3, 2] = -1
    w = M.prepare_weights(w1.to(DEV), w2.to(DEV), wl.act)
    codes, sf, scale = M.quantize_tokens(x.to(DEV))
    ws = M.workspace(w, wl.T, wl.K)
    out = M.forward(w, codes, sf, scale, ids.to(DEV), wts.to(DEV), ws=ws)
    assert M.moe_nvfp4_read_status(ws) == 7          # MOE_ERR_BAD_EXPERT_ID
    o = OracleRun(wl, x, w1, w2, o_ids, wts)
    got = out.cpu().view(torch.int16).numpy().view(np.uint16)
    assert not bf16_np(got[0]).any()
    assert rel_l2(bf16_np(got), bf16_np(o.res["out"])) <= 1e-2
    assert np.array_equal(codes[5].cpu().numpy(), np.zeros(wl.H // 2, np.uint8))
    assert scale[5].item() == 0.0
    assert w.fc1_alpha[3].item() == 0.0
    # the next forward on the same workspace clears the flag
    M.forward(w, codes, sf, scale, o_ids.to(DEV), wts.to(DEV), ws=ws)
    assert M.moe_nvfp4_read_status(ws) == 0


def test_t_zero_is_a_noop_and_t_one_works():
    wl = W.TINY_RELU2
    w1, w2 = W.make_weights(wl)
    w = M.prepare_weights(w1.to(DEV), w2.to(DEV), wl.act)
    ws = M.workspace(w, 1, wl.K)
    z = torch.empty(0, wl.K, dtype=torch.int32, device=DEV)
    out0 = torch.empty(0, wl.H, dtype=torch.bfloat16, device=DEV)
    M.moe_nvfp4_forward(w.dims, w, torch.empty(0, wl.H // 2, dtype=torch.uint8, device=DEV),
                        torch.empty(0, wl.H // 16, dtype=torch.uint8, device=DEV),
                        torch.empty(0, dtype=torch.float32, device=DEV), z,
                        torch.empty(0, wl.K, device=DEV), out0, ws)
    x = W.make_x(wl)[:1]
    ids, wts = W.make_routing(wl)
    out = _fwd(w, x.to(DEV), ids[:1].to(DEV), wts[:1].to(DEV))
    o = OracleRun(wl.with_T(1), x, w1, w2, ids[:1], wts[:1])
    assert rel_l2(bf16_np(out.cpu().view(torch.int16).numpy().view(np.uint16)),
                  bf16_np(o.res["out"])) <= 1e-2


def test_host_validation_launches_nothing():
    wl = W.TINY_RELU2
    w = M.PreparedWeights(wl.E, wl.H, wl.I, wl.act)
    codes = torch.zeros(4, wl.H // 2, dtype=torch.uint8, device=DEV)
    sf = torch.zeros(4, wl.H // 16, dtype=torch.uint8, device=DEV)
    scale = torch.zeros(4, device=DEV)
    ids = torch.zeros(4, wl.K, dtype=torch.int32, device=DEV)
    wts = torch.zeros(4, wl.K, device=DEV)
    out = torch.full((4, wl.H), 3.0, dtype=torch.bfloat16, device=DEV)
    small = torch.zeros(64, dtype=torch.uint8, device=DEV)
    with pytest.raises(M.MoeError) as ei:
        M.moe_nvfp4_forward(w.dims, w, codes, sf, scale, ids, wts, out, small)
    assert ei.value.code == 4
    bad = M.dims(wl.E, 200, wl.I, wl.act)
    ws = M.workspace(w, 4, wl.K)
    with pytest.raises(M.MoeError) as ei:
        M.moe_nvfp4_forward(bad, w, codes, sf, scale, ids, wts, out, ws)
    assert ei.value.code == 2
    torch.cuda.synchronize()
    assert (out.float() == 3.0).all()


def test_hand_worked_fixtures_on_gpu():
    """The golden round trips, each padded with zeros to H = 256 (zeros change
    neither the row amax nor the fixture's blocks)."""
    with open(os.path.join(GOLD, "quant_roundtrips.json")) as f:
        cases = json.load(f)["cases"]
    H = 256
    x = torch.zeros(len(cases), H, dtype=torch.float32)
    for i, c in enumerate(cases):
        x[i, : len(c["row"])] = torch.tensor(c["row"])
    codes, sf, scale = M.quantize_tokens(x.to(torch.bfloat16).to(DEV))
    codes, sf = codes.cpu().numpy(), sf.cpu().numpy()
    for i, c in enumerate(cases):
        n = len(c["codes"])
        assert list(codes[i, :n]) == c["codes"], c["name"]
        assert list(sf[i, : len(c["sf"])]) == c["sf"], c["name"]
        assert not codes[i, n:].any() and not sf[i, len(c["sf"]):].any()


def test_every_bf16_value_in_range_encodes_like_the_oracle():
    """All bf16 values in [-6, 6]: each 16-block holds a 6.0 pin (so enc = 448,
    block scale 448, r = 1) and 15 probe values, so the codes are E2M1(v)."""
    u = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    v = O.bf16_to_f32(u)
    v = v[np.isfinite(v) & (np.abs(v) <= 6.0)]
    n_blocks = (v.size + 14) // 15
    probe = np.zeros(n_blocks * 15, np.float32)
    probe[: v.size] = v
    blocks = np.concatenate([np.full((n_blocks, 1), 6.0, np.float32), probe.reshape(-1, 15)], 1)
    rows = blocks.reshape(-1)
    H = 256
    pad = (-rows.size) % H
    rows = np.concatenate([rows, np.zeros(pad, np.float32)]).reshape(-1, H)
    rows[:, 0] = 6.0                                   # every row's amax is 6
    xb = torch.from_numpy(rows).to(torch.bfloat16)
    codes, sf, scale = M.quantize_tokens(xb.to(DEV))
    oc, osf, os_ = O.quantize_tokens(to_np_u16(xb))
    assert np.array_equal(codes.cpu().numpy(), oc)
    assert np.array_equal(sf.cpu().numpy(), osf)
    assert np.array_equal(scale.cpu().numpy(), os_)


def test_prepare_refreshes_in_place():
    """Re-running prepare into the same buffers keeps the addresses and tracks new weights."""
    wl = W.TINY_RELU2
    w1, w2 = W.make_weights(wl)
    w = M.prepare_weights(w1.to(DEV), w2.to(DEV), wl.act)
    ptrs = [t.data_ptr() for t in (w.fc1_codes, w.fc1_sf, w.fc2_codes, w.fc2_sf)]
    w1b = (w1.float() * -0.5).to(torch.bfloat16)
    M.prepare_weights(w1b.to(DEV), w2.to(DEV), wl.act, out=w)
    assert ptrs == [t.data_ptr() for t in (w.fc1_codes, w.fc1_sf, w.fc2_codes, w.fc2_sf)]
    oc, osf, oa = O.prepare_fc(to_np_u16(w1b))
    assert np.array_equal(w.fc1_alpha.cpu().numpy(), oa)
    assert np.array_equal(w.fc1_codes.cpu().numpy(), oc)


def test_w4a16_batch_invariance(e64):
    wl, w, x, ids, wts = e64
    full = M.forward_w4a16(w, x, ids, wts)
    g = torch.Generator().manual_seed(W.BASE_SEED + 7)
    for T in (1, 7, 128):
        sel = torch.randperm(wl.T, generator=g)[:T].to(DEV)
        out = M.forward_w4a16(w, x[sel].contiguous(), ids[sel].contiguous(), wts[sel].contiguous())
        assert torch.equal(out.view(torch.int16), full[sel].view(torch.int16)), T
    # inside a 1024-token batch of 100x larger tokens routed to the same experts
    tgt = slice(0, 7)
    alone = M.forward_w4a16(w, x[tgt].contiguous(), ids[tgt].contiguous(), wts[tgt].contiguous())
    gd = torch.Generator(device=DEV).manual_seed(W.BASE_SEED + 8)
    big = (torch.randn(1017, wl.H, generator=gd, device=DEV) * 100.0).to(torch.bfloat16)
    rep = torch.arange(1017, device=DEV) % 7
    xb = torch.cat([x[tgt], big]).contiguous()
    ib = torch.cat([ids[tgt], ids[tgt][rep]]).contiguous()
    wb = torch.cat([wts[tgt], wts[tgt][rep]]).contiguous()
    out = M.forward_w4a16(w, xb, ib, wb)
    assert torch.equal(out[:7].view(torch.int16), alone.view(torch.int16))


def test_w4a16_token_rows_of_any_magnitude():
    """The W4A16 GEMMs carry each bf16 row as f16 times a power of two: rows far
    outside f16's range (1e-12, 1e6 and 1e15 in magnitude), a zero row and a
    row spanning 2^40 of dynamic range meet the oracle's fp64 expert like
    ordinary rows, and a row's output does not depend on its neighbours."""
    wl = W.Workload("swiglu_T8_H256_I256_E4_K2", 8, 256, 256, 4, 2, "swiglu")
    w1, w2 = W.make_weights(wl)
    w = M.prepare_weights(w1.to(DEV), w2.to(DEV), wl.act)
    x = W.make_x(wl).float()
    scale = torch.tensor([1.0, 1e-12, 1e6, 1e15, 0.0, 1.0, 3e-5, 1.0]).unsqueeze(1)
    x = x * scale
    x[5, ::2] *= 2.0 ** -40                        # a row spanning 2^40
    x = x.to(torch.bfloat16)
    ids, wts = W.make_routing(wl)
    out = M.forward_w4a16(w, x.to(DEV), ids.to(DEV), wts.to(DEV))
    torch.cuda.synchronize()
    Wt = O.Weights(to_np_u16(w1), to_np_u16(w2))
    ref = O.forward_w4a16(Wt, to_np_u16(x), ids.numpy(), wts.numpy(), wl.E, wl.H, wl.I, wl.act)
    got = bf16_np(to_np_u16(out.cpu()))
    want = bf16_np(ref["out"])
    for t in range(wl.T):
        if t == 4:
            assert not got[t].any()                # a zero row gives a zero output
            continue
        assert np.isfinite(got[t]).all(), t
        assert rel_l2(got[t], want[t]) <= 2e-2, t
    # each token alone gives its row of the batch, bit for bit
    for t in range(wl.T):
        one = M.forward_w4a16(w, x[t:t + 1].to(DEV), ids[t:t + 1].to(DEV), wts[t:t + 1].to(DEV))
        assert torch.equal(one.view(torch.int16), out[t:t + 1].view(torch.int16)), t
