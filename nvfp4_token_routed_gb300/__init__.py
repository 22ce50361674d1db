"""nvfp4_token_routed_gb300 -- Python binding of libmoe_nvfp4.so.

A single-GPU routed mixture-of-experts expert layer in NVFP4 for GB300
(sm_103a).  Every stage runs in the library's own CUDA kernels; this module
only marshals torch tensors (device memory + the current stream) into the C
ABI declared in include/moe_nvfp4.h.  The functions named moe_nvfp4_* mirror
the C entry points one to one; the lower-case helpers allocate buffers.

There is no CPU fallback: if the compiled library is missing, importing the
binding's entry points raises.
"""
import ctypes as C
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_nvfp4.so")

ACT = {"relu2": 0, "swiglu": 1}

STATUS = {
    0: "ok", 1: "invalid argument", 2: "unsupported shape", 3: "misaligned pointer",
    4: "workspace too small", 5: "unsupported device", 6: "CUDA error",
    7: "bad expert id", 8: "device wait timeout",
}


class MoeError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)} ({code})")


class moe_dims(C.Structure):
    _fields_ = [("E", C.c_int32), ("H", C.c_int32), ("I", C.c_int32), ("act", C.c_int32)]


class moe_nvfp4_weights(C.Structure):
    _fields_ = [("fc1_codes", C.c_void_p), ("fc1_sf", C.c_void_p), ("fc1_alpha", C.c_void_p),
                ("fc2_codes", C.c_void_p), ("fc2_sf", C.c_void_p), ("fc2_alpha", C.c_void_p)]


_LAYOUT_FIELDS = ["total", "rows_cap", "status", "counts", "group_row0", "tiles",
                  "chunk_counts", "chunk_prefix", "inv", "perm", "xq_codes", "xq_sf",
                  "xq_scale", "act", "fc2q_codes", "fc2q_sf", "fc2q_scale", "x_perm", "act_bf16",
                  "route", "tile_sync", "act_f16", "act_scale"]


class moe_forward_opts(C.Structure):
    _fields_ = [("ids_int64", C.c_int32), ("swiglu_limit", C.c_float)]


class moe_ws_layout(C.Structure):
    _fields_ = [(n, C.c_int64 if n == "rows_cap" else C.c_size_t) for n in _LAYOUT_FIELDS]


_lib = None


def lib():
    """Load libmoe_nvfp4.so (built by nvfp4_token_routed_gb300.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: run `python -m nvfp4_token_routed_gb300.build`")
        L = C.CDLL(LIB_PATH)
        vp, i32, sz = C.c_void_p, C.c_int32, C.c_size_t
        L.moe_nvfp4_abi_version.restype = i32
        L.moe_nvfp4_status_string.restype = C.c_char_p
        L.moe_nvfp4_status_string.argtypes = [C.c_int]
        L.moe_nvfp4_weight_sizes.argtypes = [C.POINTER(moe_dims), C.POINTER(C.c_size_t)]
        L.moe_nvfp4_prepare_weights.argtypes = [C.POINTER(moe_dims), vp, vp,
                                                C.POINTER(moe_nvfp4_weights), vp]
        L.moe_nvfp4_quantize_tokens.argtypes = [i32, i32, vp, vp, vp, vp, vp]
        L.moe_nvfp4_workspace_bytes.restype = sz
        L.moe_nvfp4_workspace_bytes.argtypes = [C.POINTER(moe_dims), i32, i32, i32]
        L.moe_nvfp4_forward_kernel_count.restype = i32
        L.moe_nvfp4_forward_kernel_count.argtypes = [C.POINTER(moe_dims), i32, i32, i32]
        L.moe_nvfp4_workspace_layout.argtypes = [C.POINTER(moe_dims), i32, i32, i32,
                                                 C.POINTER(moe_ws_layout)]
        L.moe_nvfp4_forward.argtypes = [C.POINTER(moe_dims), C.POINTER(moe_nvfp4_weights), i32,
                                        i32, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.moe_nvfp4_forward_w4a16.argtypes = [C.POINTER(moe_dims), C.POINTER(moe_nvfp4_weights),
                                              i32, i32, vp, vp, vp, vp, vp, sz, vp]
        L.moe_nvfp4_read_status.argtypes = [vp, vp]
        L.moe_nvfp4_forward_noalloc.argtypes = [C.POINTER(moe_dims), C.POINTER(moe_nvfp4_weights),
                                                i32, i32, vp, vp, vp, vp, vp, vp, vp]
        L.moe_nvfp4_profile_events.argtypes = [C.POINTER(C.c_void_p), i32]
        L.moe_nvfp4_profile_spans.argtypes = [vp]
        L.moe_nvfp4_prepare_weights_per_tensor.argtypes = [
            C.POINTER(moe_dims), vp, vp, vp, vp, C.POINTER(moe_nvfp4_weights), vp]
        L.moe_nvfp4_quantize_tokens_static.argtypes = [i32, i32, vp, vp, vp, vp, vp]
        L.moe_nvfp4_forward_per_tensor.argtypes = [C.POINTER(moe_dims),
                                                   C.POINTER(moe_nvfp4_weights), i32, i32, vp, vp,
                                                   vp, vp, vp, vp, vp, sz, vp]
        L.moe_nvfp4_route_topk.argtypes = [i32, i32, i32, vp, vp, vp, vp]
        L.moe_nvfp4_selftest_wait_timeout.argtypes = [vp, sz, vp]
        L.moe_nvfp4_forward_ex.argtypes = [C.POINTER(moe_dims), C.POINTER(moe_nvfp4_weights), i32,
                                           i32, vp, vp, vp, vp, vp, vp, vp, sz,
                                           C.POINTER(moe_forward_opts), vp]
        L.moe_nvfp4_forward_w4a16_ex.argtypes = [C.POINTER(moe_dims),
                                                 C.POINTER(moe_nvfp4_weights), i32, i32, vp, vp,
                                                 vp, vp, vp, sz, C.POINTER(moe_forward_opts), vp]
        for f in ["moe_nvfp4_selftest_wait_timeout",
                  "moe_nvfp4_route_topk", "moe_nvfp4_forward_ex", "moe_nvfp4_forward_w4a16_ex",
                  "moe_nvfp4_prepare_weights_per_tensor", "moe_nvfp4_quantize_tokens_static",
                  "moe_nvfp4_forward_per_tensor",
                  "moe_nvfp4_weight_sizes", "moe_nvfp4_prepare_weights",
                  "moe_nvfp4_quantize_tokens", "moe_nvfp4_workspace_layout", "moe_nvfp4_forward",
                  "moe_nvfp4_forward_w4a16", "moe_nvfp4_read_status", "moe_nvfp4_profile_events",
                  "moe_nvfp4_profile_spans", "moe_nvfp4_forward_noalloc"]:
            getattr(L, f).restype = C.c_int
        _lib = L
    return _lib


def _check(code, where):
    if code != 0:
        raise MoeError(code, where)


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("all tensors must be CUDA tensors (no CPU path exists)")
        if t is not None and not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


def padded(n):
    """The stored size of a hidden or intermediate dimension: n rounded up to 256."""
    return (n + 255) // 256 * 256


def dims(E, H, I, act):
    return moe_dims(E, H, I, ACT[act] if isinstance(act, str) else int(act))


# ------------------------------------------------------------------ one-to-one C entry points

def moe_nvfp4_abi_version():
    return lib().moe_nvfp4_abi_version()


def moe_nvfp4_status_string(code):
    return lib().moe_nvfp4_status_string(code).decode()


def moe_nvfp4_weight_sizes(d):
    out = (C.c_size_t * 6)()
    _check(lib().moe_nvfp4_weight_sizes(C.byref(d), out), "moe_nvfp4_weight_sizes")
    return list(out)


def moe_nvfp4_prepare_weights(d, fc1_bf16, fc2_bf16, w, stream=None):
    _need_cuda(fc1_bf16, fc2_bf16)
    _check(lib().moe_nvfp4_prepare_weights(C.byref(d), _ptr(fc1_bf16), _ptr(fc2_bf16),
                                           C.byref(w.c), _stream(stream)),
           "moe_nvfp4_prepare_weights")


def moe_nvfp4_quantize_tokens(x_bf16, codes, sf, scale, stream=None):
    _need_cuda(x_bf16, codes, sf, scale)
    T, H = x_bf16.shape
    _check(lib().moe_nvfp4_quantize_tokens(T, H, _ptr(x_bf16), _ptr(codes), _ptr(sf),
                                           _ptr(scale), _stream(stream)),
           "moe_nvfp4_quantize_tokens")


def moe_nvfp4_prepare_weights_per_tensor(d, fc1_bf16, fc2_bf16, a1_scale, a2_scale, w,
                                         stream=None):
    _need_cuda(fc1_bf16, fc2_bf16, a1_scale, a2_scale)
    _check(lib().moe_nvfp4_prepare_weights_per_tensor(
        C.byref(d), _ptr(fc1_bf16), _ptr(fc2_bf16), _ptr(a1_scale), _ptr(a2_scale), C.byref(w.c),
        _stream(stream)), "moe_nvfp4_prepare_weights_per_tensor")


def moe_nvfp4_quantize_tokens_static(x_bf16, a1_scale, codes, sf, stream=None):
    _need_cuda(x_bf16, a1_scale, codes, sf)
    T, H = x_bf16.shape
    _check(lib().moe_nvfp4_quantize_tokens_static(T, H, _ptr(x_bf16), _ptr(a1_scale), _ptr(codes),
                                                  _ptr(sf), _stream(stream)),
           "moe_nvfp4_quantize_tokens_static")


def moe_nvfp4_forward_per_tensor(d, w, codes, sf, a2_scale, topk_ids, topk_w, out, ws,
                                 stream=None):
    _need_cuda(codes, sf, a2_scale, topk_ids, topk_w, out, ws)
    T, K = topk_ids.shape
    _check(lib().moe_nvfp4_forward_per_tensor(C.byref(d), C.byref(w.c), T, K, _ptr(codes),
                                              _ptr(sf), _ptr(a2_scale), _ptr(topk_ids),
                                              _ptr(topk_w), _ptr(out), _ptr(ws),
                                              ws.numel() * ws.element_size(), _stream(stream)),
           "moe_nvfp4_forward_per_tensor")


def moe_nvfp4_selftest_wait_timeout(ws, stream=None):
    _need_cuda(ws)
    _check(lib().moe_nvfp4_selftest_wait_timeout(_ptr(ws), ws.numel() * ws.element_size(),
                                                 _stream(stream)),
           "moe_nvfp4_selftest_wait_timeout")


def moe_nvfp4_route_topk(logits, topk_ids, topk_w, stream=None):
    _need_cuda(logits, topk_ids, topk_w)
    T, E = logits.shape
    K = topk_ids.shape[1]
    _check(lib().moe_nvfp4_route_topk(T, E, K, _ptr(logits), _ptr(topk_ids), _ptr(topk_w),
                                      _stream(stream)), "moe_nvfp4_route_topk")


def moe_nvfp4_workspace_bytes(d, T_max, K, w4a16=False):
    return int(lib().moe_nvfp4_workspace_bytes(C.byref(d), T_max, K, int(bool(w4a16))))


def moe_nvfp4_forward_kernel_count(d, T, K, w4a16=False):
    return int(lib().moe_nvfp4_forward_kernel_count(C.byref(d), T, K, int(bool(w4a16))))


def moe_nvfp4_workspace_layout(d, T, K, w4a16=False):
    L = moe_ws_layout()
    _check(lib().moe_nvfp4_workspace_layout(C.byref(d), T, K, int(bool(w4a16)), C.byref(L)),
           "moe_nvfp4_workspace_layout")
    return {n: int(getattr(L, n)) for n in _LAYOUT_FIELDS}


def moe_nvfp4_forward(d, w, codes, sf, scale, topk_ids, topk_w, out, ws, stream=None):
    _need_cuda(codes, sf, scale, topk_ids, topk_w, out, ws)
    T, K = topk_ids.shape
    _check(lib().moe_nvfp4_forward(C.byref(d), C.byref(w.c), T, K, _ptr(codes), _ptr(sf),
                                   _ptr(scale), _ptr(topk_ids), _ptr(topk_w), _ptr(out), _ptr(ws),
                                   ws.numel() * ws.element_size(), _stream(stream)),
           "moe_nvfp4_forward")


def moe_nvfp4_forward_ex(d, w, codes, sf, scale, topk_ids, topk_w, out, ws, opts, stream=None):
    """opts: moe_forward_opts (int64 ids are taken from topk_ids' dtype)."""
    _need_cuda(codes, sf, scale, topk_ids, topk_w, out, ws)
    T, K = topk_ids.shape
    _check(lib().moe_nvfp4_forward_ex(C.byref(d), C.byref(w.c), T, K, _ptr(codes), _ptr(sf),
                                      _ptr(scale), _ptr(topk_ids), _ptr(topk_w), _ptr(out),
                                      _ptr(ws), ws.numel() * ws.element_size(), C.byref(opts),
                                      _stream(stream)), "moe_nvfp4_forward_ex")


def moe_nvfp4_forward_w4a16_ex(d, w, x_bf16, topk_ids, topk_w, out, ws, opts, stream=None):
    _need_cuda(x_bf16, topk_ids, topk_w, out, ws)
    T, K = topk_ids.shape
    _check(lib().moe_nvfp4_forward_w4a16_ex(C.byref(d), C.byref(w.c), T, K, _ptr(x_bf16),
                                            _ptr(topk_ids), _ptr(topk_w), _ptr(out), _ptr(ws),
                                            ws.numel() * ws.element_size(), C.byref(opts),
                                            _stream(stream)), "moe_nvfp4_forward_w4a16_ex")


def moe_nvfp4_forward_w4a16(d, w, x_bf16, topk_ids, topk_w, out, ws, stream=None):
    _need_cuda(x_bf16, topk_ids, topk_w, out, ws)
    T, K = topk_ids.shape
    _check(lib().moe_nvfp4_forward_w4a16(C.byref(d), C.byref(w.c), T, K, _ptr(x_bf16),
                                         _ptr(topk_ids), _ptr(topk_w), _ptr(out), _ptr(ws),
                                         ws.numel() * ws.element_size(), _stream(stream)),
           "moe_nvfp4_forward_w4a16")


def moe_nvfp4_forward_noalloc(d, w, codes, sf, scale, topk_ids, topk_w, out, stream=None):
    """The W4A4 forward on the library's own 64 MiB device scratch array, for
    callers that cannot allocate device memory (see include/moe_nvfp4.h)."""
    _need_cuda(codes, sf, scale, topk_ids, topk_w, out)
    T, K = topk_ids.shape
    _check(lib().moe_nvfp4_forward_noalloc(C.byref(d), C.byref(w.c), T, K, _ptr(codes), _ptr(sf),
                                           _ptr(scale), _ptr(topk_ids), _ptr(topk_w), _ptr(out),
                                           _stream(stream)),
           "moe_nvfp4_forward_noalloc")


def moe_nvfp4_read_status(ws, stream=None):
    """Device-reported status code of the last forward on `ws` (syncs the stream)."""
    return int(lib().moe_nvfp4_read_status(_ptr(ws), _stream(stream)))


def moe_nvfp4_profile_events(events):
    """Register torch.cuda.Event objects (already recorded once) as stage markers."""
    if not events:
        _check(lib().moe_nvfp4_profile_events(None, 0), "moe_nvfp4_profile_events")
        return
    arr = (C.c_void_p * len(events))(*[e.cuda_event for e in events])
    _check(lib().moe_nvfp4_profile_events(arr, len(events)), "moe_nvfp4_profile_events")


def moe_nvfp4_profile_spans(spans):
    """Register a CUDA int64 tensor of 4 elements (or None to unregister) that
    the grouped GEMM launches fold their %globaltimer spans into: [0]/[1] the
    FC1 (or one-launch) launch's earliest CTA start / latest CTA end, [2]/[3]
    the FC2 launch's.  Reset [0], [2] to the maximum and [1], [3] to 0 first."""
    if spans is not None and (not spans.is_cuda or spans.dtype != torch.int64
                              or spans.numel() < 4 or not spans.is_contiguous()):
        raise ValueError("spans: a contiguous CUDA int64 tensor of 4 elements")
    _check(lib().moe_nvfp4_profile_spans(None if spans is None else _ptr(spans)),
           "moe_nvfp4_profile_spans")


# ------------------------------------------------------------------ allocating helpers

class PreparedWeights:
    """Device buffers of the prepared NVFP4 weights (layouts in include/moe_nvfp4.h)."""

    def __init__(self, E, H, I, act, device="cuda"):
        self.dims = dims(E, H, I, act)
        self.E, self.H, self.I, self.act = E, H, I, act
        sizes = moe_nvfp4_weight_sizes(self.dims)
        Hp, Ip = padded(H), padded(I)
        N1 = 2 * Ip if act == "swiglu" else Ip
        self.fc1_codes = torch.empty(E, N1, Hp // 2, dtype=torch.uint8, device=device)
        self.fc1_sf = torch.empty(sizes[1], dtype=torch.uint8, device=device)
        self.fc1_alpha = torch.empty(E, dtype=torch.float32, device=device)
        self.fc2_codes = torch.empty(E, Hp, Ip // 2, dtype=torch.uint8, device=device)
        self.fc2_sf = torch.empty(sizes[4], dtype=torch.uint8, device=device)
        self.fc2_alpha = torch.empty(E, dtype=torch.float32, device=device)
        assert self.fc1_codes.numel() == sizes[0] and self.fc2_codes.numel() == sizes[3]
        self.c = moe_nvfp4_weights(*[t.data_ptr() for t in (
            self.fc1_codes, self.fc1_sf, self.fc1_alpha, self.fc2_codes, self.fc2_sf,
            self.fc2_alpha)])

    def nbytes(self):
        return sum(t.numel() * t.element_size() for t in (
            self.fc1_codes, self.fc1_sf, self.fc1_alpha, self.fc2_codes, self.fc2_sf,
            self.fc2_alpha))


def prepare_weights(fc1_bf16, fc2_bf16, act, out=None, stream=None):
    """Quantize BF16 stacks fc1 [E,N1,H] ([gate; up] for SwiGLU) and fc2 [E,H,I]."""
    E, N1, H = fc1_bf16.shape
    I = fc2_bf16.shape[2]
    w = out if out is not None else PreparedWeights(E, H, I, act, device=fc1_bf16.device)
    moe_nvfp4_prepare_weights(w.dims, fc1_bf16, fc2_bf16, w, stream)
    return w


def quantize_tokens(x_bf16, stream=None):
    T, H = x_bf16.shape
    dev = x_bf16.device
    Hp = padded(H)  # rows are zero-padded to Hp columns
    codes = torch.empty(T, Hp // 2, dtype=torch.uint8, device=dev)
    sf = torch.empty(T, Hp // 16, dtype=torch.uint8, device=dev)
    scale = torch.empty(T, dtype=torch.float32, device=dev)
    moe_nvfp4_quantize_tokens(x_bf16, codes, sf, scale, stream)
    return codes, sf, scale


def prepare_weights_per_tensor(fc1_bf16, fc2_bf16, act, a1_scale, a2_scale, out=None,
                               stream=None):
    """Per-tensor recipe weights: codes/scales as prepare_weights, alphas with the
    static device scalars a1_scale / a2_scale folded in."""
    E, N1, H = fc1_bf16.shape
    I = fc2_bf16.shape[2]
    w = out if out is not None else PreparedWeights(E, H, I, act, device=fc1_bf16.device)
    moe_nvfp4_prepare_weights_per_tensor(w.dims, fc1_bf16, fc2_bf16, a1_scale, a2_scale, w, stream)
    return w


def quantize_tokens_static(x_bf16, a1_scale, stream=None):
    T, H = x_bf16.shape
    Hp = padded(H)
    codes = torch.empty(T, Hp // 2, dtype=torch.uint8, device=x_bf16.device)
    sf = torch.empty(T, Hp // 16, dtype=torch.uint8, device=x_bf16.device)
    moe_nvfp4_quantize_tokens_static(x_bf16, a1_scale, codes, sf, stream)
    return codes, sf


def forward_per_tensor(w, codes, sf, a2_scale, topk_ids, topk_w, ws=None, out=None, stream=None):
    T, K = topk_ids.shape
    if ws is None:
        ws = workspace(w, T, K, device=codes.device)
    if out is None:
        out = torch.empty(T, w.H, dtype=torch.bfloat16, device=codes.device)
    moe_nvfp4_forward_per_tensor(w.dims, w, codes, sf, a2_scale, topk_ids, topk_w, out, ws, stream)
    return out


def route_topk(logits, K, stream=None):
    """Plain top-K router: fp32 logits [T,E] -> (int32 ids [T,K], fp32 scores [T,K])."""
    T = logits.shape[0]
    ids = torch.empty(T, K, dtype=torch.int32, device=logits.device)
    w = torch.empty(T, K, dtype=torch.float32, device=logits.device)
    moe_nvfp4_route_topk(logits, ids, w, stream)
    return ids, w


def workspace(w, T_max, K, w4a16=False, device="cuda"):
    n = moe_nvfp4_workspace_bytes(w.dims, T_max, K, w4a16)
    if n == 0:
        raise MoeError(2, "moe_nvfp4_workspace_bytes")
    return torch.empty(n, dtype=torch.uint8, device=device)


def forward(w, codes, sf, scale, topk_ids, topk_w, ws=None, out=None, stream=None):
    T, K = topk_ids.shape
    if ws is None:
        ws = workspace(w, T, K, device=codes.device)
    if out is None:
        out = torch.empty(T, w.H, dtype=torch.bfloat16, device=codes.device)
    moe_nvfp4_forward(w.dims, w, codes, sf, scale, topk_ids, topk_w, out, ws, stream)
    return out


def forward_opts(topk_ids, swiglu_limit=0.0):
    """Options for the *_ex calls: int64 ids follow from the tensor's dtype."""
    return moe_forward_opts(1 if topk_ids.dtype == torch.int64 else 0, float(swiglu_limit))


def forward_ex(w, codes, sf, scale, topk_ids, topk_w, swiglu_limit=0.0, ws=None, out=None,
               stream=None):
    T, K = topk_ids.shape
    if ws is None:
        ws = workspace(w, T, K, device=codes.device)
    if out is None:
        out = torch.empty(T, w.H, dtype=torch.bfloat16, device=codes.device)
    moe_nvfp4_forward_ex(w.dims, w, codes, sf, scale, topk_ids, topk_w, out, ws,
                         forward_opts(topk_ids, swiglu_limit), stream)
    return out


def forward_w4a16_ex(w, x_bf16, topk_ids, topk_w, swiglu_limit=0.0, ws=None, out=None,
                     stream=None):
    T, K = topk_ids.shape
    if ws is None:
        ws = workspace(w, T, K, w4a16=True, device=x_bf16.device)
    if out is None:
        out = torch.empty(T, w.H, dtype=torch.bfloat16, device=x_bf16.device)
    moe_nvfp4_forward_w4a16_ex(w.dims, w, x_bf16, topk_ids, topk_w, out, ws,
                               forward_opts(topk_ids, swiglu_limit), stream)
    return out


def forward_w4a16(w, x_bf16, topk_ids, topk_w, ws=None, out=None, stream=None):
    T, K = topk_ids.shape
    if ws is None:
        ws = workspace(w, T, K, w4a16=True, device=x_bf16.device)
    if out is None:
        out = torch.empty(T, w.H, dtype=torch.bfloat16, device=x_bf16.device)
    moe_nvfp4_forward_w4a16(w.dims, w, x_bf16, topk_ids, topk_w, out, ws, stream)
    return out


def ws_view(ws, layout, name, dtype, shape):
    """A typed view of one workspace region (offsets from moe_nvfp4_workspace_layout)."""
    off = layout[name]
    n = 1
    for s in shape:
        n *= s
    nbytes = n * torch.empty((), dtype=dtype).element_size()
    return ws[off:off + nbytes].view(dtype).view(*shape)
