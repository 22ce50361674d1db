"""ctypes binding of the C oracle (moe_oracle.c).

TEST INFRASTRUCTURE.  Only the test suite, the package smoke check and the
benchmark's CPU-baseline leg may import this module.  Arrays are numpy; bf16
values travel as uint16 bit patterns.  Nothing here touches a GPU or the CUDA
library, and nothing here is shared with it.
"""
import ctypes as C
import os

import numpy as np

from . import build as _build

_lib = None


class Dims(C.Structure):
    _fields_ = [("E", C.c_int64), ("H", C.c_int64), ("I", C.c_int64), ("act", C.c_int32),
                ("limit", C.c_double)]


def _p(a):
    return a.ctypes.data_as(C.c_void_p)


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        _lib = C.CDLL(path)
        L = _lib
        L.orc_e2m1_decode.restype = C.c_double
        L.orc_e2m1_decode.argtypes = [C.c_uint8]
        L.orc_e2m1_encode.restype = C.c_uint8
        L.orc_e2m1_encode.argtypes = [C.c_float]
        L.orc_e4m3_decode.restype = C.c_double
        L.orc_e4m3_decode.argtypes = [C.c_uint8]
        L.orc_e4m3_encode.restype = C.c_uint8
        L.orc_e4m3_encode.argtypes = [C.c_float]
        L.orc_recipe_c.restype = C.c_float
        L.orc_f64_to_bf16.restype = C.c_uint16
        L.orc_f64_to_bf16.argtypes = [C.c_double]
        L.orc_sf_swizzle_offset.restype = C.c_int64
        L.orc_sf_swizzle_offset.argtypes = [C.c_int64, C.c_int64, C.c_int64]
        L.orc_route.restype = C.c_int64
        L.orc_forward_w4a4.restype = C.c_int64
        L.orc_forward_w4a16.restype = C.c_int64
        L.orc_forward_w4a4_per_tensor.restype = C.c_int64
        L.orc_num_threads.restype = C.c_int
        L.orc_quantize_row_per_token_f32.restype = C.c_float
        for name in ["orc_e2m1_encode_n", "orc_e4m3_encode_n", "orc_e4m3_decode_n",
                     "orc_f64_to_bf16_n", "orc_sf_to_swizzled", "orc_quantize_row",
                     "orc_quantize_tokens", "orc_prepare_fc", "orc_finalize", "orc_dense_w4a4",
                     "orc_route", "orc_forward_w4a4", "orc_forward_w4a16",
                     "orc_quantize_row_per_token_f32", "orc_quantize_tokens_static",
                     "orc_alpha_per_tensor", "orc_forward_w4a4_per_tensor", "orc_route_topk"]:
            getattr(L, name).argtypes = None
    return _lib


def num_threads():
    return int(lib().orc_num_threads())


def recipe_c():
    return np.float32(lib().orc_recipe_c())


# ----------------------------------------------------------------------------- formats

def e2m1_decode(code):
    return lib().orc_e2m1_decode(int(code))


def e2m1_encode(v):
    v = np.ascontiguousarray(v, dtype=np.float32).ravel()
    out = np.empty(v.size, np.uint8)
    lib().orc_e2m1_encode_n(_p(v), C.c_int64(v.size), _p(out))
    return out


def e4m3_encode(v):
    v = np.ascontiguousarray(v, dtype=np.float32).ravel()
    out = np.empty(v.size, np.uint8)
    lib().orc_e4m3_encode_n(_p(v), C.c_int64(v.size), _p(out))
    return out


def e4m3_decode(b):
    b = np.ascontiguousarray(b, dtype=np.uint8).ravel()
    out = np.empty(b.size, np.float64)
    lib().orc_e4m3_decode_n(_p(b), C.c_int64(b.size), _p(out))
    return out


def f64_to_bf16(v):
    v = np.ascontiguousarray(v, dtype=np.float64).ravel()
    out = np.empty(v.size, np.uint16)
    lib().orc_f64_to_bf16_n(_p(v), C.c_int64(v.size), _p(out))
    return out


def bf16_to_f32(u16):
    u16 = np.ascontiguousarray(u16, dtype=np.uint16)
    return (u16.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits(x):
    """Round float values to bf16 (nearest even) through the oracle's rounding."""
    x = np.asarray(x, dtype=np.float64)
    return f64_to_bf16(x).reshape(x.shape)


# ----------------------------------------------------------------------------- quantizers

def quantize_row(v, enc):
    v = np.ascontiguousarray(v, dtype=np.float32)
    D = v.size
    codes = np.empty(D // 2, np.uint8)
    sf = np.empty(D // 16, np.uint8)
    lib().orc_quantize_row(_p(v), C.c_int64(D), C.c_float(enc), _p(codes), _p(sf))
    return codes, sf


def quantize_row_per_token(v):
    v = np.ascontiguousarray(v, dtype=np.float32)
    D = v.size
    codes = np.empty(D // 2, np.uint8)
    sf = np.empty(D // 16, np.uint8)
    s = lib().orc_quantize_row_per_token_f32(_p(v), C.c_int64(D), _p(codes), _p(sf))
    return codes, sf, np.float32(s)


def quantize_tokens(x_bf16):
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    T, H = x.shape
    codes = np.empty((T, H // 2), np.uint8)
    sf = np.empty((T, H // 16), np.uint8)
    s = np.empty(T, np.float32)
    lib().orc_quantize_tokens(C.c_int64(T), C.c_int64(H), _p(x), _p(codes), _p(sf), _p(s))
    return codes, sf, s


def quantize_tokens_static(x_bf16, a1):
    """Per-tensor recipe: every row quantized with the static encode scale a1 (R12)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    T, H = x.shape
    codes = np.empty((T, H // 2), np.uint8)
    sf = np.empty((T, H // 16), np.uint8)
    lib().orc_quantize_tokens_static(C.c_int64(T), C.c_int64(H), _p(x), C.c_float(a1), _p(codes),
                                     _p(sf))
    return codes, sf


def alpha_per_tensor(w_bf16, a):
    """Per-tensor alphas fl(1/fl(w_scale*a)) of one BF16 FC stack [E][N][D] (R12)."""
    w = np.ascontiguousarray(w_bf16, dtype=np.uint16)
    E, N, D = w.shape
    alpha = np.empty(E, np.float32)
    lib().orc_alpha_per_tensor(C.c_int64(E), C.c_int64(N), C.c_int64(D), _p(w), C.c_float(a),
                               _p(alpha))
    return alpha


def prepare_fc(w_bf16):
    """BF16 [E][N][D] (canonical rows) -> codes [E][N][D/2], linear sf [E][N][D/16], alpha [E]."""
    w = np.ascontiguousarray(w_bf16, dtype=np.uint16)
    E, N, D = w.shape
    codes = np.empty((E, N, D // 2), np.uint8)
    sf = np.empty((E, N, D // 16), np.uint8)
    alpha = np.empty(E, np.float32)
    lib().orc_prepare_fc(C.c_int64(E), C.c_int64(N), C.c_int64(D), _p(w), _p(codes), _p(sf),
                         _p(alpha))
    return codes, sf, alpha


def sf_swizzle_offset(r, j, ncols16):
    return lib().orc_sf_swizzle_offset(int(r), int(j), int(ncols16))


def sf_to_swizzled(lin):
    """Linear [N][D/16] scale plane -> swizzled plane of round_up(N,128)*round_up(D/16,4) bytes."""
    lin = np.ascontiguousarray(lin, dtype=np.uint8)
    N, c16 = lin.shape
    P = (N + 127) // 128 * 128 * ((c16 + 3) // 4 * 4)
    out = np.empty(P, np.uint8)
    lib().orc_sf_to_swizzled(C.c_int64(N), C.c_int64(c16), _p(lin), _p(out))
    return out


# ----------------------------------------------------------------------------- routing + forward

def route_topk(logits, K):
    """Plain top-K router (R14): ids int32 [T][K] (descending, ties to the lower
    id) and fp32 softmax scores over the selected logits."""
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = lg.shape
    if not 1 <= K <= E:
        raise ValueError(f"top-K router needs 1 <= K <= E, got K={K}, E={E}")
    ids = np.empty((T, K), np.int32)
    w = np.empty((T, K), np.float32)
    lib().orc_route_topk(C.c_int64(T), C.c_int64(E), C.c_int64(K), _p(lg), _p(ids), _p(w))
    return ids, w


def route(ids, E):
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T, K = ids.shape
    counts = np.empty(E, np.int32)
    perm = np.empty(T * K, np.int32)
    inv = np.empty(T * K, np.int32)
    R = lib().orc_route(C.c_int64(T), C.c_int64(K), C.c_int64(E), _p(ids), _p(counts), _p(perm),
                        _p(inv))
    return counts, perm[:R].copy(), inv


def finalize(route_rows, inv, w, T, K):
    route_rows = np.ascontiguousarray(route_rows, dtype=np.uint16)
    inv = np.ascontiguousarray(inv, dtype=np.int32)
    w = np.ascontiguousarray(w, dtype=np.float32)
    H = route_rows.shape[1]
    out = np.empty((T, H), np.uint16)
    lib().orc_finalize(C.c_int64(T), C.c_int64(K), C.c_int64(H), _p(route_rows), _p(inv), _p(w),
                       _p(out))
    return out


class Weights:
    """Oracle-prepared weights in canonical row order with linear scales."""

    def __init__(self, w1_bf16, w2_bf16):
        self.w1c, self.w1sf, self.a1 = prepare_fc(w1_bf16)
        self.w2c, self.w2sf, self.a2 = prepare_fc(w2_bf16)


def _dims(E, H, I, act, limit=0.0):
    return Dims(E, H, I, 1 if act == "swiglu" else 0, float(limit))


def forward_w4a4(W, xc, xsf, xs, ids, w, E, H, I, act, limit=0.0):
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    w = np.ascontiguousarray(w, dtype=np.float32)
    T, K = ids.shape
    TK = T * K
    d = _dims(E, H, I, act, limit)
    counts = np.empty(E, np.int32)
    perm = np.empty(TK, np.int32)
    inv = np.empty(TK, np.int32)
    act_rows = np.empty((TK, I), np.float32)
    fc2c = np.empty((TK, I // 2), np.uint8)
    fc2sf = np.empty((TK, I // 16), np.uint8)
    s2 = np.empty(TK, np.float32)
    routes = np.empty((TK, H), np.uint16)
    out = np.empty((T, H), np.uint16)
    xc = np.ascontiguousarray(xc, np.uint8)
    xsf = np.ascontiguousarray(xsf, np.uint8)
    xs = np.ascontiguousarray(xs, np.float32)
    R = lib().orc_forward_w4a4(C.byref(d), C.c_int64(T), C.c_int64(K), _p(W.w1c), _p(W.w1sf),
                               _p(W.a1), _p(W.w2c), _p(W.w2sf), _p(W.a2), _p(xc), _p(xsf),
                               _p(xs), _p(ids), _p(w), _p(counts), _p(perm), _p(inv),
                               _p(act_rows), _p(fc2c), _p(fc2sf), _p(s2), _p(routes), _p(out))
    return dict(R=R, counts=counts, perm=perm[:R].copy(), inv=inv, act=act_rows[:R],
                fc2c=fc2c[:R], fc2sf=fc2sf[:R], s2=s2[:R], route=routes[:R], out=out)


def forward_w4a4_per_tensor(W, xc, xsf, a2_static, ids, w, E, H, I, act):
    """Per-tensor W4A4 forward (R12): W holds the per-tensor alphas (a1/a2 folded),
    tokens come from quantize_tokens_static, the FC2 input uses a2_static."""
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    w = np.ascontiguousarray(w, dtype=np.float32)
    T, K = ids.shape
    TK = T * K
    d = _dims(E, H, I, act)
    counts = np.empty(E, np.int32)
    perm = np.empty(TK, np.int32)
    inv = np.empty(TK, np.int32)
    act_rows = np.empty((TK, I), np.float32)
    fc2c = np.empty((TK, I // 2), np.uint8)
    fc2sf = np.empty((TK, I // 16), np.uint8)
    routes = np.empty((TK, H), np.uint16)
    out = np.empty((T, H), np.uint16)
    xc = np.ascontiguousarray(xc, np.uint8)
    xsf = np.ascontiguousarray(xsf, np.uint8)
    R = lib().orc_forward_w4a4_per_tensor(
        C.byref(d), C.c_int64(T), C.c_int64(K), _p(W.w1c), _p(W.w1sf), _p(W.a1), _p(W.w2c),
        _p(W.w2sf), _p(W.a2), _p(xc), _p(xsf), C.c_float(a2_static), _p(ids), _p(w), _p(counts),
        _p(perm), _p(inv), _p(act_rows), _p(fc2c), _p(fc2sf), _p(routes), _p(out))
    return dict(R=R, counts=counts, perm=perm[:R].copy(), inv=inv, act=act_rows[:R],
                fc2c=fc2c[:R], fc2sf=fc2sf[:R], route=routes[:R], out=out)


class WeightsPerTensor:
    """Oracle-prepared weights of the per-tensor recipe: per-token codes and
    scales, alphas with the static input scales folded in (R12)."""

    def __init__(self, w1_bf16, w2_bf16, a1, a2):
        self.w1c, self.w1sf, _ = prepare_fc(w1_bf16)
        self.w2c, self.w2sf, _ = prepare_fc(w2_bf16)
        self.a1 = alpha_per_tensor(w1_bf16, a1)
        self.a2 = alpha_per_tensor(w2_bf16, a2)


def forward_w4a16(W, x_bf16, ids, w, E, H, I, act, limit=0.0):
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    w = np.ascontiguousarray(w, dtype=np.float32)
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    T, K = ids.shape
    TK = T * K
    d = _dims(E, H, I, act, limit)
    counts = np.empty(E, np.int32)
    perm = np.empty(TK, np.int32)
    inv = np.empty(TK, np.int32)
    act_rows = np.empty((TK, I), np.uint16)
    routes = np.empty((TK, H), np.uint16)
    out = np.empty((T, H), np.uint16)
    R = lib().orc_forward_w4a16(C.byref(d), C.c_int64(T), C.c_int64(K), _p(W.w1c), _p(W.w1sf),
                                _p(W.a1), _p(W.w2c), _p(W.w2sf), _p(W.a2), _p(x), _p(ids), _p(w),
                                _p(counts), _p(perm), _p(inv), _p(act_rows), _p(routes), _p(out))
    return dict(R=R, counts=counts, perm=perm[:R].copy(), inv=inv, act=act_rows[:R],
                route=routes[:R], out=out)


def dense_w4a4(W, xc, xsf, xs, ids, w, E, H, I, act):
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    w = np.ascontiguousarray(w, dtype=np.float32)
    T, K = ids.shape
    d = _dims(E, H, I, act)
    out = np.empty((T, H), np.uint16)
    xc = np.ascontiguousarray(xc, np.uint8)
    xsf = np.ascontiguousarray(xsf, np.uint8)
    xs = np.ascontiguousarray(xs, np.float32)
    lib().orc_dense_w4a4(C.byref(d), C.c_int64(T), C.c_int64(K), _p(W.w1c), _p(W.w1sf), _p(W.a1),
                         _p(W.w2c), _p(W.w2sf), _p(W.a2), _p(xc), _p(xsf), _p(xs), _p(ids), _p(w),
                         _p(out))
    return out


def dequant(codes, sf):
    """Decode NVFP4 rows (codes [..., D/2], linear sf [..., D/16]) to float64 [..., D]."""
    codes = np.asarray(codes, np.uint8)
    lo = codes & 15
    hi = codes >> 4
    q = np.stack([lo, hi], axis=-1).reshape(*codes.shape[:-1], codes.shape[-1] * 2)
    mag = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float64)
    v = mag[q & 7] * np.where(q & 8, -1.0, 1.0)
    s = e4m3_decode(np.asarray(sf, np.uint8)).reshape(np.asarray(sf).shape)
    return v * np.repeat(s, 16, axis=-1)
