"""Test-side helpers: layout maps, comparisons and the oracle runs of a workload.

Nothing here is product code and nothing here computes the layer: the layer's
expected values come from the oracle package only.
"""
import numpy as np
import torch

from oracle import oracle as O
from nvfp4_token_routed_gb300 import workloads as W


TILE_ROWS = 128  # each expert group of the permuted buffers starts at a multiple of this


def sf_offsets(rows, c16):
    """Byte offsets of (row, scale column) in a 128x4-swizzled plane (vectorised)."""
    r = np.asarray(rows, np.int64)[:, None]
    j = np.arange(c16, dtype=np.int64)[None, :]
    return ((r // 128) * (c16 // 4) + j // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + (j % 4)


def unswizzle(plane, rows, c16):
    """Linear [len(rows), c16] scale bytes read from a swizzled plane."""
    plane = np.asarray(plane, np.uint8).ravel()
    return plane[sf_offsets(rows, c16)]


def stored_fc1_rows(N1, I, act):
    """Canonical FC1 row held at each stored row (stored order interleaves 64-row
    [gate | up] blocks for SwiGLU; identity for squared ReLU)."""
    ir = np.arange(N1)
    if act != "swiglu":
        return ir
    b = ir // 64
    return (b % 2) * I + (b // 2) * 64 + ir % 64


def signed_step(codes_a, codes_b):
    """Distance in E2M1 grid steps between unpacked 4-bit codes (-0 == +0)."""
    def sidx(c):
        m = (c & 7).astype(np.int64)
        return np.where(c & 8, -m, m)
    return np.abs(sidx(codes_a) - sidx(codes_b))


def unpack_codes(packed):
    packed = np.asarray(packed, np.uint8)
    return np.stack([packed & 15, packed >> 4], axis=-1).reshape(*packed.shape[:-1], -1)


def check_scaled_f16_rows(f16_rows, scales, want):
    """The W4A16 GEMMs' f16 operand rows: each row of `want` (bf16 values as
    float) times 2^-k, with its largest magnitude in [2^14, 2^15) and 2^k in
    `scales`; exact down to f16's normal range, within half an f16 subnormal
    step below it."""
    got16 = np.asarray(f16_rows).view(np.float16).astype(np.float64)
    rs = np.asarray(scales, np.float64)
    want = np.asarray(want, np.float64)
    amax = np.abs(want).max(axis=1)
    k = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - 14, 0.0)
    assert np.array_equal(rs, 2.0 ** k)
    assert np.all(np.abs(want / rs[:, None]).max(axis=1) < 2.0 ** 15)
    got = got16 * rs[:, None]
    normal = np.abs(want) >= rs[:, None] * 2.0 ** -14
    assert np.array_equal(got[normal], want[normal])
    tol = np.broadcast_to(rs[:, None] * 2.0 ** -25, want.shape)
    assert np.all(np.abs(got - want)[~normal] <= tol[~normal])


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


def to_np_u16(t):
    return W.bf16_bits(t)


def bf16_np(u16):
    return O.bf16_to_f32(u16)


class OracleRun:
    """Oracle results for one workload's inputs (inputs given as torch CPU tensors)."""

    def __init__(self, wl, x, w1, w2, ids, wts, w4a16=False):
        self.wl = wl
        self.W = O.Weights(to_np_u16(w1), to_np_u16(w2))
        self.ids = ids.cpu().numpy().astype(np.int32)
        self.wts = wts.cpu().numpy().astype(np.float32)
        if w4a16:
            self.res = O.forward_w4a16(self.W, to_np_u16(x), self.ids, self.wts, wl.E, wl.H, wl.I,
                                       wl.act)
        else:
            self.xc, self.xsf, self.xs = O.quantize_tokens(to_np_u16(x))
            self.res = O.forward_w4a4(self.W, self.xc, self.xsf, self.xs, self.ids, self.wts,
                                      wl.E, wl.H, wl.I, wl.act)
