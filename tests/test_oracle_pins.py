"""Pins of the CPU oracle against what the pages and the mathematics fix.

Nothing here reruns the oracle's own formula: each check uses an independent
route (the printed grid, a library conversion, hand-worked values, invariants,
brute force, an unquantized fp64 MoE).
"""
import json
import os

import numpy as np
import pytest
import torch

from oracle import oracle as O
from nvfp4_token_routed_gb300 import workloads as W

GOLD = os.path.join(os.path.dirname(__file__), "golden")
GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def bf16_bits_of(values):
    t = torch.tensor(values, dtype=torch.float32).to(torch.bfloat16)
    assert torch.equal(t.float(), torch.tensor(values, dtype=torch.float32)), "not bf16-exact"
    return t.view(torch.int16).numpy().view(np.uint16)


# --------------------------------------------------------------------------- formats

def test_e2m1_decode_is_the_printed_grid():
    for code in range(16):
        mag = GRID[code & 7]
        assert O.e2m1_decode(code) == (-mag if code & 8 else mag)


def _nearest_grid_ties_even(v):
    """Brute force: nearest of the 8 grid magnitudes, ties to the even code index."""
    a = abs(float(v))
    best, bestd = None, None
    for i, g in enumerate(GRID):
        dd = abs(a - g)
        if bestd is None or dd < bestd or (dd == bestd and i % 2 == 0):
            best, bestd = i, dd
    if a > 6.0:
        best = 7
    return best | (8 if np.signbit(v) else 0)


def test_e2m1_encode_matches_bruteforce_nearest():
    rng = np.random.default_rng(0)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    near = np.concatenate([mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(9))])
    grid = np.array(GRID, np.float32)
    vals = np.concatenate([near, -near, grid, -grid, np.linspace(-8, 8, 4001, dtype=np.float32),
                           rng.uniform(-8, 8, 20000).astype(np.float32),
                           np.array([7.0, 100.0, -1e30, 6.0000005], np.float32)])
    got = O.e2m1_encode(vals)
    want = np.array([_nearest_grid_ties_even(v) for v in vals], np.uint8)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(vals[i], got[i], want[i]) for i in bad[:10]]


def test_e2m1_tie_table_from_the_reading():
    # ties to even: 0.25->0, 0.75->1.0, 1.25->1.0, 1.75->2, 2.5->2, 3.5->4, 5->4, >5 -> 6
    ins = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 5.01, 9.0], np.float32)
    want = [0, 2, 2, 4, 4, 6, 6, 7, 7]
    assert list(O.e2m1_encode(ins)) == want


def test_e4m3_matches_torch_float8_e4m3fn():
    rng = np.random.default_rng(1)
    codes = np.arange(0, 0x7F, dtype=np.uint8)            # every finite non-negative E4M3
    vals = O.e4m3_decode(codes).astype(np.float32)
    mids = ((vals[1:].astype(np.float64) + vals[:-1]) / 2).astype(np.float32)
    probe = np.concatenate([vals, mids, np.nextafter(mids, np.float32(0)),
                            np.nextafter(mids, np.float32(1000)),
                            rng.uniform(0, 448, 50000).astype(np.float32),
                            np.exp(rng.uniform(np.log(2.0 ** -12), np.log(448), 50000)).astype(np.float32)])
    probe = probe[probe <= 448.0]
    got = O.e4m3_encode(probe)
    want = torch.from_numpy(probe).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(probe[i], got[i], want[i]) for i in bad[:10]]
    # decode agrees with torch's e4m3fn -> float conversion for every finite code
    allc = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    tdec = torch.from_numpy(allc).view(torch.float8_e4m3fn).float().numpy()
    assert np.array_equal(O.e4m3_decode(allc), tdec.astype(np.float64))


def test_e4m3_max_is_448_and_saturates():
    assert O.e4m3_decode(np.array([0x7E], np.uint8))[0] == 448.0
    assert list(O.e4m3_encode(np.array([448.0, 449.0, 470.0, 1e6, 3e38], np.float32))) == [0x7E] * 5
    assert O.e4m3_decode(np.array([0x01], np.uint8))[0] == 2.0 ** -9     # smallest subnormal
    assert O.e4m3_decode(np.array([0x08], np.uint8))[0] == 2.0 ** -6     # smallest normal


def test_recipe_constant_is_one_over_448x6():
    c = O.recipe_c()
    assert c.dtype == np.float32
    # the binary32 nearest to 1/2688: within half an ulp of the exact value
    ulp = np.spacing(np.float32(1.0 / 2688.0))
    assert abs(float(c) - 1.0 / 2688.0) <= ulp / 2


def test_f64_to_bf16_matches_torch_for_float32_inputs():
    rng = np.random.default_rng(2)
    v = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.uniform(-30, 30, 20000),
                        [0.0, -0.0, 1.0, 3.140625, 1.00390625, 1.01171875]]).astype(np.float32)
    got = O.f64_to_bf16(v.astype(np.float64))
    want = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)


# --------------------------------------------------------------------------- quantizers

def _load_cases():
    with open(os.path.join(GOLD, "quant_roundtrips.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _load_cases(), ids=lambda c: c["name"])
def test_hand_worked_round_trips(case):
    bits = bf16_bits_of(case["row"]).reshape(1, -1)
    codes, sf, s = O.quantize_tokens(bits)
    assert list(sf[0]) == case["sf"]
    assert list(codes[0]) == case["codes"]
    amax = case["amax"]
    if amax == 0:
        assert s[0] == 0.0
    else:
        # the per-token decode scale is amax/(448*6), to within one binary32 rounding step
        assert abs(float(s[0]) - amax / 2688.0) <= 2 * np.spacing(np.float32(amax / 2688.0))


def test_power_of_two_scaling_invariance():
    """Scaling a token by 2^m leaves codes and block scales unchanged and scales s by 2^m."""
    x = W.make_x(W.TINY_RELU2)
    bits = W.bf16_bits(x)
    c0, f0, s0 = O.quantize_tokens(bits)
    for m in (-7, -1, 3, 9):
        xs = (x.float() * 2.0 ** m).to(torch.bfloat16)
        c1, f1, s1 = O.quantize_tokens(W.bf16_bits(xs))
        assert np.array_equal(c0, c1) and np.array_equal(f0, f1)
        assert np.array_equal(s1, (s0 * np.float32(2.0 ** m)).astype(np.float32))


def test_dequant_error_within_half_step_of_block_scale():
    """|x - deq| <= half an E2M1 step (1 for |q| in [4,6]) times the block scale, times s."""
    x = W.make_x(W.TINY_RELU2)
    codes, sf, s = O.quantize_tokens(W.bf16_bits(x))
    deq = O.dequant(codes, sf) * s[:, None].astype(np.float64)
    xf = x.float().numpy().astype(np.float64)
    bs = np.repeat(O.e4m3_decode(sf).reshape(sf.shape), 16, axis=1) * s[:, None]
    # largest E2M1 gap is 2 (between 4 and 6) -> half-gap 1; plus the scale's own rounding
    assert np.all(np.abs(xf - deq) <= 1.0 * bs * 1.0001 + 1e-30)


def test_weight_prep_alpha_and_codes():
    """An expert whose amax is 6 gets w_scale 448 and alpha 1/448; its codes are the grid."""
    row = np.array(GRID + [-g for g in GRID], np.float32)      # 16 values, amax 6
    w = torch.from_numpy(np.tile(row, (1, 4, 2))).to(torch.bfloat16)  # [1, 4, 32]
    codes, sf, alpha = O.prepare_fc(W.bf16_bits(w))
    assert alpha[0] == np.float32(1.0) / np.float32(448.0)
    assert np.all(sf == 0x7E)
    want = [c | (8 if i >= 8 else 0) for i, c in enumerate(list(range(8)) * 2)]
    want_bytes = [want[2 * j] | (want[2 * j + 1] << 4) for j in range(8)]
    assert list(codes[0, 0, :8]) == want_bytes


def test_weight_prep_zero_expert():
    w = torch.zeros(2, 4, 32, dtype=torch.bfloat16)
    w[1, 2, 5] = 1.0
    codes, sf, alpha = O.prepare_fc(W.bf16_bits(w))
    assert alpha[0] == 0 and not codes[0].any() and not sf[0].any()
    assert alpha[1] == np.float32(1.0) / (np.float32(2688.0) / np.float32(1.0))


def test_swizzled_plane_size_and_bijection():
    """P = round_up(N,128)*round_up(D/16,4) (Tensor and numerical contract) and every
    (row, scale column) lands on its own byte."""
    for N, c16 in [(128, 16), (256, 448 // 1), (300, 20), (4096, 128)]:
        lin = np.arange(N * c16, dtype=np.int64)
        offs = np.array([O.sf_swizzle_offset(r, j, c16) for r in range(N) for j in range(c16)])
        P = (N + 127) // 128 * 128 * ((c16 + 3) // 4 * 4)
        assert offs.min() >= 0 and offs.max() < P
        assert np.unique(offs).size == lin.size
        # each 512-byte atom holds 128 rows x 4 consecutive scale columns of one row block
        r = np.arange(N).repeat(c16)
        j = np.tile(np.arange(c16), N)
        assert np.array_equal(offs // 512, (r // 128) * ((c16 + 3) // 4) + j // 4)


# --------------------------------------------------------------------------- routing

def test_route_matches_numpy_stable_argsort():
    rng = np.random.default_rng(3)
    for T, K, E in [(16, 2, 8), (37, 6, 20), (128, 8, 64)]:
        ids = rng.integers(-1, E, size=(T, K)).astype(np.int32)
        ids[0, 0] = E + 5          # invalid id -> empty slot
        counts, perm, inv = O.route(ids, E)
        flat = ids.ravel()
        valid = (flat >= 0) & (flat < E)
        order = np.argsort(np.where(valid, flat, E + 10), kind="stable")[: valid.sum()]
        assert np.array_equal(perm, order.astype(np.int32))
        assert np.array_equal(counts, np.bincount(flat[valid], minlength=E).astype(np.int32))
        assert np.all(inv[~valid] == -1)
        assert np.array_equal(inv[perm], np.arange(perm.size))


# --------------------------------------------------------------------------- forward

def _tiny(act="relu2", T=16, H=256, I=512, E=8, K=2, seed=0):
    wl = W.Workload(f"t_{act}", T, H, I, E, K, act)
    x = W.make_x(wl, seed=seed + 11)
    w1, w2 = W.make_weights(wl, seed=seed + 20)
    ids, wts = W.make_routing(wl, seed=seed + 30)
    return wl, x, w1, w2, ids.numpy(), wts.numpy()


def test_forward_equals_dense_bruteforce_exactly():
    for act in ("relu2", "swiglu"):
        wl, x, w1, w2, ids, wts = _tiny(act, I=256 if act == "swiglu" else 512)
        Wt = O.Weights(W.bf16_bits(w1), W.bf16_bits(w2))
        xc, xsf, xs = O.quantize_tokens(W.bf16_bits(x))
        routed = O.forward_w4a4(Wt, xc, xsf, xs, ids, wts, wl.E, wl.H, wl.I, act)
        dense = O.dense_w4a4(Wt, xc, xsf, xs, ids, wts, wl.E, wl.H, wl.I, act)
        assert np.array_equal(routed["out"], dense)


def test_finalize_top1_unit_weight_is_the_route_row():
    rng = np.random.default_rng(4)
    T, K, H = 5, 3, 32
    rows = torch.randn(T, H).to(torch.bfloat16)
    inv = -np.ones(T * K, np.int32)
    w = np.zeros(T * K, np.float32)
    for t in range(T):
        k = rng.integers(0, K)
        inv[t * K + k] = t
        w[t * K + k] = 1.0
    out = O.finalize(W.bf16_bits(rows), inv, w, T, K)
    assert np.array_equal(out, W.bf16_bits(rows))


def _unquantized_moe(x, w1, w2, ids, wts, act, I):
    xf = x.double().numpy()
    out = np.zeros_like(xf)
    for t in range(xf.shape[0]):
        for k in range(ids.shape[1]):
            e = ids[t, k]
            y = w1[e].double().numpy() @ xf[t]
            if act == "relu2":
                a = np.maximum(y, 0) ** 2
            else:
                g, u = y[:I], y[I:]
                a = g / (1 + np.exp(-g)) * u
            out[t] += wts[t, k] * (w2[e].double().numpy() @ a)
    return out


@pytest.mark.parametrize("act", ["relu2", "swiglu"])
def test_sanity_against_unquantized_fp64_moe(act):
    """The pages' accuracy bound for the NVFP4 MoE against an unquantized one:
    per-token cosine mean > 0.97 and min > 0.95 (What is tested)."""
    wl, x, w1, w2, ids, wts = _tiny(act, I=256 if act == "swiglu" else 512)
    Wt = O.Weights(W.bf16_bits(w1), W.bf16_bits(w2))
    xc, xsf, xs = O.quantize_tokens(W.bf16_bits(x))
    got = O.bf16_to_f32(O.forward_w4a4(Wt, xc, xsf, xs, ids, wts, wl.E, wl.H, wl.I, act)["out"])
    ref = _unquantized_moe(x, w1, w2, ids, wts, act, wl.I)
    cos = (got * ref).sum(1) / np.linalg.norm(got, axis=1) / np.linalg.norm(ref, axis=1)
    assert cos.mean() > 0.97 and cos.min() > 0.95, cos
    # the W4A16 variant keeps activations in bf16: tighter
    got16 = O.bf16_to_f32(O.forward_w4a16(Wt, W.bf16_bits(x), ids, wts, wl.E, wl.H, wl.I, act)["out"])
    cos16 = (got16 * ref).sum(1) / np.linalg.norm(got16, axis=1) / np.linalg.norm(ref, axis=1)
    assert cos16.min() > cos.min() - 1e-3 and cos16.mean() > 0.98


def _f32_alpha(w_bf16_expert):
    """alpha = 1 / w_scale with w_scale = 2688 / amax, each one binary32 operation,
    written here with numpy scalars (How to extend: alpha = 1 / w_scale)."""
    amax = np.float32(np.abs(w_bf16_expert.float().numpy()).max())
    return np.float32(np.float32(1.0) / np.float32(np.float32(2688.0) / amax))


def _bf16_of(a):
    """Nearest bf16 of fp64 values, through torch's float32 -> bfloat16 conversion."""
    t = torch.from_numpy(np.asarray(a, np.float64).astype(np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _mismatches_within_one_ulp(got_u16, want_u16):
    """Count of differing bf16 elements; fails if any differs by more than one ulp."""
    g = got_u16.astype(np.int64)
    w = want_u16.astype(np.int64)
    sg = np.where(g & 0x8000, -(g & 0x7FFF), g & 0x7FFF)
    sw = np.where(w & 0x8000, -(w & 0x7FFF), w & 0x7FFF)
    assert np.abs(sg - sw).max(initial=0) <= 1
    return int((g != w).sum())


@pytest.mark.parametrize("act", ["relu2", "swiglu"])
def test_w4a16_expert_matches_a_direct_dequantized_matmul(act):
    """W4A16 compute order (Tensor and numerical contract): FC1 over the bf16 token
    row with weights decoded from the oracle's codes and scales, times alpha1;
    activation; a bf16 handoff; FC2 over the handoff times alpha2; bf16 route
    rows.  Computed here with numpy from the bf16 weights' own amax, so a dropped
    or doubled alpha1 / alpha2, or an FC2 fed with the unrounded activation,
    moves hundreds of elements."""
    wl, x, w1, w2, ids, wts = _tiny(act, I=256 if act == "swiglu" else 512)
    Wt = O.Weights(W.bf16_bits(w1), W.bf16_bits(w2))
    res = O.forward_w4a16(Wt, W.bf16_bits(x), ids, wts, wl.E, wl.H, wl.I, act)
    xf = x.float().numpy().astype(np.float64)          # bf16 values, exact
    act_miss = route_miss = n_act = n_route = 0
    for q in range(res["R"]):
        r = int(res["perm"][q]); t, e = r // wl.K, int(ids[r // wl.K, r % wl.K])
        a1, a2 = _f32_alpha(w1[e]), _f32_alpha(w2[e])
        assert a1 == Wt.a1[e] and a2 == Wt.a2[e]
        y = (O.dequant(Wt.w1c[e], Wt.w1sf[e]) @ xf[t]) * np.float64(a1)
        if act == "relu2":
            a = np.maximum(y, 0) ** 2
        else:
            g, u = y[: wl.I], y[wl.I:]
            a = g / (1 + np.exp(-g)) * u
        a_h = _bf16_of(a)                                  # the handoff
        act_miss += _mismatches_within_one_ulp(res["act"][q], a_h)
        n_act += a_h.size
        z = (O.dequant(Wt.w2c[e], Wt.w2sf[e]) @ O.bf16_to_f32(a_h).astype(np.float64))
        route = _bf16_of(z * np.float64(a2))
        route_miss += _mismatches_within_one_ulp(res["route"][q], route)
        n_route += route.size
    # only values within rounding-order noise of a bf16 midpoint may round apart
    assert act_miss <= 2 and route_miss <= 2, (act_miss, n_act, route_miss, n_route)


def test_swiglu_gate_up_split():
    """up rows zero -> output 0; gate rows zero -> output 0; swapping the halves
    changes the output (canonical FC1 = [gate; up], Tensor and numerical contract)."""
    wl, x, w1, w2, ids, wts = _tiny("swiglu", T=4, I=128, E=4, K=1)
    xc, xsf, xs = O.quantize_tokens(W.bf16_bits(x))
    I = wl.I

    def run(w1m):
        Wt = O.Weights(W.bf16_bits(w1m), W.bf16_bits(w2))
        return O.forward_w4a4(Wt, xc, xsf, xs, ids, wts, wl.E, wl.H, I, "swiglu")["out"]

    up0 = w1.clone()
    up0[:, I:] = 0
    assert not O.bf16_to_f32(run(up0)).any()
    g0 = w1.clone()
    g0[:, :I] = 0
    assert not O.bf16_to_f32(run(g0)).any()
    sw = torch.cat([w1[:, I:], w1[:, :I]], dim=1)
    assert not np.array_equal(run(sw), run(w1))
    # and silu(g)*u, not g*silu(u): with the gate forced negative-large, output ~ 0
    neg = w1.clone()
    neg[:, :I] = 0
    neg[:, :I, 0] = -100.0
    xpos = torch.zeros_like(x)
    xpos[:, 0] = 1.0
    xc2, xsf2, xs2 = O.quantize_tokens(W.bf16_bits(xpos))
    Wt = O.Weights(W.bf16_bits(neg), W.bf16_bits(w2))
    out = O.forward_w4a4(Wt, xc2, xsf2, xs2, ids, wts, wl.E, wl.H, I, "swiglu")["out"]
    assert np.abs(O.bf16_to_f32(out)).max() < 1e-20


def test_relu2_output_scales_by_four_to_the_m():
    """Squared ReLU: scaling tokens by 2^m scales each route row (and output) by 4^m exactly."""
    wl, x, w1, w2, ids, wts = _tiny("relu2", T=6)
    Wt = O.Weights(W.bf16_bits(w1), W.bf16_bits(w2))
    r0 = O.forward_w4a4(Wt, *O.quantize_tokens(W.bf16_bits(x)), ids, wts, wl.E, wl.H, wl.I, "relu2")
    x2 = (x.float() * 4.0).to(torch.bfloat16)
    r1 = O.forward_w4a4(Wt, *O.quantize_tokens(W.bf16_bits(x2)), ids, wts, wl.E, wl.H, wl.I, "relu2")
    assert np.array_equal(O.bf16_to_f32(r1["route"]), O.bf16_to_f32(r0["route"]) * 16.0)
    assert np.array_equal(r1["fc2c"], r0["fc2c"]) and np.array_equal(r1["fc2sf"], r0["fc2sf"])


# --------------------------------------------------------------------------- per-tensor recipe
# Megatron-LM PR #8262, "How to extend", "Per-tensor NVFP4 x NVFP4": static FC1 /
# FC2 input scales (encode scales, like w_scale), folded into the alphas.

def test_static_quantization_with_the_tokens_own_scale_is_per_token():
    """A row quantized with the static scale fl(2688/amax) of its own amax gets
    exactly the per-token codes and block scales."""
    x = W.make_x(W.TINY_RELU2)
    bits = W.bf16_bits(x)
    c_pt, f_pt, s_pt = O.quantize_tokens(bits)
    for t in range(4):
        amax = np.float32(np.abs(x[t].float().numpy()).max())
        a1 = np.float32(np.float32(2688.0) / amax)
        c, f = O.quantize_tokens_static(bits[t:t + 1], a1)
        assert np.array_equal(c[0], c_pt[t]) and np.array_equal(f[0], f_pt[t])


def test_static_quantization_scales_against_the_values():
    """x * 2^m quantized with a1 * 2^-m gives the same codes and block scales."""
    x = W.make_x(W.TINY_RELU2)
    c0, f0 = O.quantize_tokens_static(W.bf16_bits(x), np.float32(64.0))
    for m in (-3, 2, 5):
        xs = (x.float() * 2.0 ** m).to(torch.bfloat16)
        c1, f1 = O.quantize_tokens_static(W.bf16_bits(xs), np.float32(64.0 * 2.0 ** -m))
        assert np.array_equal(c0, c1) and np.array_equal(f0, f1)


def test_static_quantization_saturates():
    """A static scale far too large clips: block scales 448 (0x7E) and codes +-6,
    so the dequantized magnitude is 6 * 448 / a1 whatever the input."""
    row = np.array([1.0, -1.0, 2.0, -3.0] * 4, np.float32)
    c, f = O.quantize_tokens_static(bf16_bits_of(row)[None, :], np.float32(1e6))
    assert f[0, 0] == 0x7E
    deq = O.dequant(c, f)[0]
    assert np.all(np.abs(deq) == 6.0 * 448.0)


def test_per_tensor_alpha_folds_the_input_scale():
    """alpha = fl(1/fl(w_scale * a)); an amax-6 expert has w_scale 448, so with
    a = 2 the alpha is fl(1/896); a zero expert keeps alpha 0."""
    row = np.array(GRID + [-g for g in GRID], np.float32)
    w = torch.from_numpy(np.tile(row, (2, 4, 2))).to(torch.bfloat16)
    w[1] = 0
    alpha = O.alpha_per_tensor(W.bf16_bits(w), np.float32(2.0))
    assert alpha[0] == np.float32(1.0) / np.float32(896.0) and alpha[1] == 0.0


def test_per_tensor_forward_matches_a_direct_dequantized_matmul():
    """Per-tensor FC1 rows and route rows against numpy: weights dequantized from
    the oracle codes over w_scale, tokens dequantized over a1 (no row scales),
    FC2 input dequantized over a2.  A missing or doubled a1/a2 factor moves every
    value by that factor."""
    wl, x, w1, w2, ids, wts = _tiny("relu2", I=512)
    a1, a2 = np.float32(8.0), np.float32(0.25)
    Wt = O.WeightsPerTensor(W.bf16_bits(w1), W.bf16_bits(w2), a1, a2)
    xc, xsf = O.quantize_tokens_static(W.bf16_bits(x), a1)
    res = O.forward_w4a4_per_tensor(Wt, xc, xsf, a2, ids, wts, wl.E, wl.H, wl.I, "relu2")
    # independent numpy composition
    w1f, w2f = w1.float().numpy().astype(np.float64), w2.float().numpy().astype(np.float64)
    xq = O.dequant(xc, xsf) / np.float64(a1)                        # tokens as the MMA sees them
    for q in range(min(res["R"], 12)):
        r = int(res["perm"][q]); t, e = r // wl.K, int(ids[r // wl.K, r % wl.K])
        amax1 = np.float32(np.abs(w1f[e]).max())
        ws1 = np.float32(np.float32(2688.0) / amax1)
        c1, f1, _ = O.prepare_fc(W.bf16_bits(w1[e:e + 1]))
        w1q = O.dequant(c1[0], f1[0]) / np.float64(ws1)
        y = w1q @ xq[t]
        a = np.maximum(y, 0) ** 2
        assert np.allclose(res["act"][q], a, rtol=1e-5, atol=1e-6 * np.abs(a).max())
        fq = O.dequant(res["fc2c"][q:q + 1], res["fc2sf"][q:q + 1])[0] / np.float64(a2)
        amax2 = np.float32(np.abs(w2f[e]).max())
        ws2 = np.float32(np.float32(2688.0) / amax2)
        c2, f2, _ = O.prepare_fc(W.bf16_bits(w2[e:e + 1]))
        w2q = O.dequant(c2[0], f2[0]) / np.float64(ws2)
        route = w2q @ fq
        got = O.bf16_to_f32(res["route"][q]).astype(np.float64)
        assert np.allclose(got, route, rtol=1e-2, atol=1e-2 * np.abs(route).max())


# --------------------------------------------------------------------------- router

def test_router_topk_matches_a_stable_sort_and_the_softmax_closed_form():
    """ids = the K largest logits (descending; equal logits to the lower id, as a
    stable sort of -logits gives them); scores = exp(l - l_max) / sum over the
    selected, which is the full softmax renormalised over the selected K."""
    g = np.random.default_rng(3)
    T, E, K = 64, 96, 6
    lg = g.standard_normal((T, E)).astype(np.float32)
    lg[5, 10] = lg[5, 3] = lg[5].max() + 1.0            # an exact tie at the top
    lg[7, :] = 0.5                                       # all equal
    ids, w = O.route_topk(lg, K)
    ref_ids = np.argsort(-lg, axis=1, kind="stable")[:, :K]
    assert np.array_equal(ids, ref_ids)
    assert ids[5, 0] == 3 and ids[5, 1] == 10 and list(ids[7]) == list(range(K))
    full = np.exp(lg.astype(np.float64) - lg.max(axis=1, keepdims=True))
    full /= full.sum(axis=1, keepdims=True)
    sel = np.take_along_axis(full, ref_ids, axis=1)
    assert np.allclose(w, sel / sel.sum(axis=1, keepdims=True), rtol=1e-6, atol=0)
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-6)
    assert np.all(np.diff(w, axis=1) <= 0)
    # top-1 always scores exactly 1
    assert np.all(O.route_topk(lg, 1)[1] == 1.0)


# --------------------------------------------------------------------------- clamped SwiGLU

def test_clamped_swiglu_caps_the_gate_and_clips_up():
    """act = silu(min(g, L)) * clip(u, -L, L) on the FC1 outputs g, u (computed here
    with numpy from the dequantized operands); a limit above every |g|, |u| is
    no clamp at all."""
    wl, x, w1, w2, ids, wts = _tiny("swiglu", I=256)
    Wt = O.Weights(W.bf16_bits(w1), W.bf16_bits(w2))
    xc, xsf, xs = O.quantize_tokens(W.bf16_bits(x))
    plain = O.forward_w4a4(Wt, xc, xsf, xs, ids, wts, wl.E, wl.H, wl.I, "swiglu")
    huge = O.forward_w4a4(Wt, xc, xsf, xs, ids, wts, wl.E, wl.H, wl.I, "swiglu", limit=1e30)
    assert np.array_equal(plain["out"], huge["out"]) and np.array_equal(plain["act"], huge["act"])
    L = 0.05
    res = O.forward_w4a4(Wt, xc, xsf, xs, ids, wts, wl.E, wl.H, wl.I, "swiglu", limit=L)
    xq = O.dequant(xc, xsf) * xs[:, None].astype(np.float64)
    clamped_any = False
    for q in range(res["R"]):
        r = int(res["perm"][q]); t, e = r // wl.K, int(ids[r // wl.K, r % wl.K])
        w1q = O.dequant(Wt.w1c[e], Wt.w1sf[e]) * np.float64(Wt.a1[e])
        y = w1q @ xq[t]
        g, u = y[: wl.I], y[wl.I:]
        clamped_any |= bool((g > L).any() or (np.abs(u) > L).any())
        gc, uc = np.minimum(g, L), np.clip(u, -L, L)
        ref = gc / (1 + np.exp(-gc)) * uc
        assert np.allclose(res["act"][q], ref, rtol=1e-5, atol=1e-7 * L * L)
    assert clamped_any
