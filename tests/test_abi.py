"""The C ABI without a GPU: the library loads, exports every entry point that
include/moe_nvfp4.h declares, and its host-side logic (sizes, workspace layout,
argument validation) answers before any CUDA call."""
import ctypes as C
import os
import re
import subprocess

import pytest

import nvfp4_token_routed_gb300 as M

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_nvfp4.h")


def _declared():
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_nvfp4_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from nvfp4_token_routed_gb300 import build
    build.build()
    return M.lib()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 12, names
    out = subprocess.run(["nm", "-D", "--defined-only", M.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (\w+)", out))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        assert hasattr(lib, n)


def test_abi_version_and_status_strings(lib):
    assert M.moe_nvfp4_abi_version() == 3
    for code in range(9):
        assert M.moe_nvfp4_status_string(code)
    assert M.moe_nvfp4_status_string(5).startswith("unsupported device")


def test_weight_sizes_match_the_contract(lib):
    d = M.dims(8, 256, 512, "swiglu")
    sz = M.moe_nvfp4_weight_sizes(d)
    # FC1 [E, 2I, H/2] codes, P = round_up(N,128)*round_up(D/16,4) scale bytes per expert
    assert sz == [8 * 1024 * 128, 8 * 1024 * 16, 32, 8 * 256 * 256, 8 * 256 * 32, 32]
    d2 = M.dims(8, 256, 512, "relu2")
    assert M.moe_nvfp4_weight_sizes(d2)[0] == 8 * 512 * 128


def test_non_aligned_shapes_are_stored_padded_to_256(lib):
    # H = 320 -> Hp = 512, I = 192 -> Ip = 256; SwiGLU pads each half: N1p = 512
    d = M.dims(8, 320, 192, "swiglu")
    assert M.moe_nvfp4_weight_sizes(d) == [8 * 512 * 256, 8 * 512 * 32, 32, 8 * 512 * 128,
                                           8 * 512 * 16, 32]
    d = M.dims(8, 2688, 1856, "relu2")   # 2688 -> 2816 (the pages' example), 1856 -> 2048
    assert M.moe_nvfp4_weight_sizes(d)[0] == 8 * 2048 * 1408
    assert M.moe_nvfp4_weight_sizes(d)[3] == 8 * 2816 * 1024
    L = M.moe_nvfp4_workspace_layout(d, 4, 2, False)
    assert L["fc2q_codes"] - L["act"] >= L["rows_cap"] * 2048 * 4
    assert M.padded(2688) == 2816 and M.padded(256) == 256 and M.padded(64) == 256


@pytest.mark.parametrize("act", ["relu2", "swiglu"])
@pytest.mark.parametrize("w4a16", [False, True])
def test_workspace_layout_is_aligned_disjoint_and_monotone(lib, act, w4a16):
    d = M.dims(64, 2048, 1024, act)
    prev = 0
    for T in (1, 7, 128, 1000):
        L = M.moe_nvfp4_workspace_layout(d, T, 8, w4a16)
        assert L["total"] == M.moe_nvfp4_workspace_bytes(d, T, 8, w4a16)
        assert L["total"] >= prev
        prev = L["total"]
        offs = sorted(v for k, v in L.items() if k not in ("total", "rows_cap") and (v or k == "status"))
        assert all(o % 256 == 0 for o in offs)
        assert len(set(offs)) == len(offs)
        TK = T * 8
        assert L["rows_cap"] % 128 == 0 and L["rows_cap"] >= TK + min(64, TK) * 127
        used = (("x_perm", "xq_scale", "act_bf16", "act_f16", "act_scale") if w4a16
                else ("xq_codes", "xq_scale", "act", "fc2q_codes"))
        unused = (("xq_codes", "act", "fc2q_codes") if w4a16
                  else ("x_perm", "act_bf16", "act_f16", "act_scale"))
        assert all(L[k] > 0 for k in used) and all(L[k] == 0 for k in unused)


def test_invalid_shapes_are_rejected_on_the_host(lib):
    for E, H, I in [(0, 256, 256), (2000, 256, 256), (8, 200, 256), (8, 256, 300), (8, 32, 256),
                    (8, 256, 65600)]:
        d = M.dims(E, H, I, "relu2")
        assert M.moe_nvfp4_workspace_bytes(d, 4, 2) == 0
        with pytest.raises(M.MoeError) as ei:
            M.moe_nvfp4_weight_sizes(d)
        assert ei.value.code == 2
    d = M.dims(8, 256, 256, "relu2")
    assert M.moe_nvfp4_workspace_bytes(d, 4, 9) == 0       # K > E
    assert M.moe_nvfp4_workspace_bytes(d, -1, 2) == 0
    bad_act = M.moe_dims(8, 256, 256, 7)
    with pytest.raises(M.MoeError) as ei:
        M.moe_nvfp4_weight_sizes(bad_act)
    assert ei.value.code == 1


class _FakeWeights:
    """Non-null, aligned, never-dereferenced pointers: validation must answer
    before anything touches them."""

    def __init__(self, dims):
        self.dims = dims
        self.c = M.moe_nvfp4_weights(*([4096] * 6))


def test_forward_validation_without_a_gpu(lib):
    L = lib
    d = M.dims(8, 256, 512, "relu2")
    w = _FakeWeights(d)
    vp = C.c_void_p
    # T == 0 is a no-op that succeeds without touching the device
    rc = L.moe_nvfp4_forward(C.byref(d), C.byref(w.c), 0, 2, vp(4096), vp(4096), vp(4096),
                             vp(4096), vp(4096), vp(4096), vp(4096), 1 << 20, None)
    assert rc == 0
    # missing pointers
    rc = L.moe_nvfp4_forward(C.byref(d), C.byref(w.c), 4, 2, None, vp(4096), vp(4096),
                             vp(4096), vp(4096), vp(4096), vp(4096), 1 << 30, None)
    assert rc == 1
    # misaligned workspace
    rc = L.moe_nvfp4_forward(C.byref(d), C.byref(w.c), 4, 2, vp(4096), vp(4096), vp(4096),
                             vp(4096), vp(4096), vp(4096), vp(4096 + 8), 1 << 30, None)
    assert rc == 3
    # workspace too small
    rc = L.moe_nvfp4_forward(C.byref(d), C.byref(w.c), 4, 2, vp(4096), vp(4096), vp(4096),
                             vp(4096), vp(4096), vp(4096), vp(4096), 64, None)
    assert rc == 4
    # unsupported top-k
    rc = L.moe_nvfp4_forward(C.byref(d), C.byref(w.c), 4, 33, vp(4096), vp(4096), vp(4096),
                             vp(4096), vp(4096), vp(4096), vp(4096), 1 << 30, None)
    assert rc == 2
    # misaligned weights
    wbad = M.moe_nvfp4_weights(4096 + 4, 4096, 4096, 4096, 4096, 4096)
    rc = L.moe_nvfp4_forward(C.byref(d), C.byref(wbad), 4, 2, vp(4096), vp(4096), vp(4096),
                             vp(4096), vp(4096), vp(4096), vp(4096), 1 << 30, None)
    assert rc == 3
    # quantize: bad H, T == 0
    assert L.moe_nvfp4_quantize_tokens(4, 100, vp(4096), vp(4096), vp(4096), vp(4096), None) == 2
    assert L.moe_nvfp4_quantize_tokens(0, 256, None, None, None, None, None) == 0
    # the allocation-free forward rejects a problem beyond its scratch before any CUDA call
    big = M.dims(64, 2048, 1024, "swiglu")
    wb = _FakeWeights(big)
    rc = L.moe_nvfp4_forward_noalloc(C.byref(big), C.byref(wb.c), 4096, 8, vp(4096), vp(4096),
                                     vp(4096), vp(4096), vp(4096), vp(4096), None)
    assert rc == 4
    # ... and reports a bad shape with the status moe_nvfp4_forward gives it
    for T, K, want in ((4, 0, 1), (-1, 2, 1), (4, 33, 2)):
        args = (C.byref(d), C.byref(w.c), T, K, vp(4096), vp(4096), vp(4096), vp(4096),
                vp(4096), vp(4096))
        assert L.moe_nvfp4_forward(*args, vp(4096), 1 << 30, None) == want
        assert L.moe_nvfp4_forward_noalloc(*args, None) == want
    bad_act = M.moe_dims(8, 256, 512, 7)
    assert L.moe_nvfp4_forward_noalloc(C.byref(bad_act), C.byref(w.c), 4, 2, vp(4096), vp(4096),
                                       vp(4096), vp(4096), vp(4096), vp(4096), None) == 1


def test_profile_events_argument_checks(lib):
    assert lib.moe_nvfp4_profile_events(None, 0) == 0
    assert lib.moe_nvfp4_profile_events(None, 9) == 1
    assert lib.moe_nvfp4_profile_events(None, -1) == 1


def test_profile_spans_argument_checks(lib):
    import ctypes as C
    assert lib.moe_nvfp4_profile_spans(C.c_void_p(4100)) == 3  # MOE_ERR_MISALIGNED
    assert lib.moe_nvfp4_profile_spans(None) == 0


def test_binding_rejects_cpu_tensors():
    import torch
    w = _FakeWeights(M.dims(8, 256, 512, "relu2"))
    x = torch.zeros(4, 256, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        M.moe_nvfp4_forward_w4a16(w.dims, w, x, torch.zeros(4, 2, dtype=torch.int32),
                                  torch.zeros(4, 2), torch.zeros(4, 256, dtype=torch.bfloat16),
                                  torch.zeros(1024, dtype=torch.uint8))


def test_forward_kernel_count(lib):
    """Launches of one forward call: routing and gather (one kernel up to 32
    routes, two up to 2048, four beyond), GEMMs (W4A4: one launch when
    T*K <= min(2048, 8E), else FC1, requant, FC2; W4A16: FC1, the f16 FC2
    operand, FC2), finalize."""
    e64 = M.dims(64, 2048, 1024, "swiglu")
    e256 = M.dims(256, 7168, 2048, "relu2")
    count = M.moe_nvfp4_forward_kernel_count
    assert count(e64, 128, 8) == 2 + 3 + 1              # 1024 routes > 8 per expert
    assert count(e64, 128, 8, True) == 2 + 3 + 1
    assert count(e64, 64, 8) == 2 + 1 + 1               # 512 routes = 8 per expert: one launch
    assert count(e256, 1, 8) == 1 + 1 + 1               # 8 routes: rows gathered by the routing block
    assert count(e256, 4, 8) == 1 + 1 + 1               # 32 routes
    assert count(e256, 5, 8) == 2 + 1 + 1               # 40 routes: separate gather
    assert count(e256, 256, 8) == 2 + 1 + 1             # 2048 routes
    assert count(e256, 257, 8) == 4 + 3 + 1             # 2056 routes: three routing kernels
    assert count(e256, 4096, 8, True) == 4 + 3 + 1
    assert count(e256, 0, 8) == 0
    assert count(e256, 4, 0) == -1 and count(e256, 4, 33) == -1 and count(e256, -1, 8) == -1
