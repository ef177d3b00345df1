"""Host-side checks of the C ABI (no GPU): the library loads, exports every
symbol include/muon.h declares, sizes workspaces, and rejects bad arguments
with the documented status before touching the device.

Every call here fails argument checking before any CUDA call, so fake device
addresses are never dereferenced (these tests are also safe on a GPU machine).
"""

import ctypes
import os
import re

import pytest

from newton_schulz_08_gb300 import muon

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(muon.LIB_PATH):
        from newton_schulz_08_gb300 import build
        build.build()
    return muon.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "muon.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:[A-Za-z_][\w\s\*]*?)\b([a-z_0-9]+)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "defined")))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert set(names) == set(muon.EXPORTS), names
    for n in names:
        assert hasattr(L, n), n


def test_plan_cache_clear_is_host_only(L):
    # drops host memory only: callable with no GPU and no prepared call
    muon.muon_plan_cache_clear()
    muon.muon_plan_cache_clear()


def test_status_strings(L):
    for code in range(-8, 2):
        assert muon.muon_status_str(code)
    assert muon.muon_status_str(-99) == "unknown status"


def desc(param=0x100000, grad=0x200000, buf=0x300000, rows=4, cols=8, dtype=muon.MUON_BF16, reserved=0):
    return muon.muon_mat_desc(param, grad, buf, rows, cols, dtype, reserved)


def call_step(L, descs, ns_steps=5, ws=0x40000000, ws_bytes=1 << 40, nesterov=1, n=None):
    arr = (muon.muon_mat_desc * max(len(descs), 1))(*descs)
    return L.muon_step(arr, len(descs) if n is None else n, 0.02, 0.95, nesterov, ns_steps,
                       ctypes.c_void_p(ws), ws_bytes, None)


def test_workspace_size_single(L):
    # layout of one 128 x 512 matrix: 256 B header, 4 partial sums (32 rows
    # per block) padded to 1 KiB, a 32 B table entry padded to 1 KiB, then two
    # X buffers (128 x 512 bf16) and A, B (128 x 128 bf16), each 1 KiB aligned
    assert muon.muon_workspace_size([(128, 512)]) == 2048 + 2 * 131072 + 2 * 32768
    assert muon.muon_workspace_size([(512, 128)]) > 0
    assert muon.ns5_workspace_size(1, 128, 512) == muon.muon_workspace_size([(128, 512)])


def test_workspace_size_grows_and_classes(L):
    a = muon.muon_workspace_size([(768, 768)] * 4)
    b = muon.muon_workspace_size([(768, 768)] * 8)
    assert b > a > 0
    # a tall matrix and its transpose share one shape class
    assert muon.muon_workspace_size([(3072, 768), (768, 3072)]) == muon.muon_workspace_size([(768, 3072)] * 2)
    assert muon.ns5_bank_workspace_size([(64, 32), (32, 64)]) == muon.ns5_workspace_size(2, 32, 64)


def test_workspace_size_invalid(L):
    assert muon.muon_workspace_size([]) == 0
    assert muon.muon_workspace_size([(0, 5)]) == 0
    assert muon.muon_workspace_size([(5, -1)]) == 0
    assert muon.ns5_workspace_size(0, 4, 4) == 0
    assert muon.ns5_workspace_size(2, 1 << 32, 4) == 0


def test_layout(L):
    lay = muon.ns5_workspace_layout(3, 300, 100)  # tall: X is 100 x 300
    assert lay["m"] == 100 and lay["n"] == 300
    assert lay["ldx"] == 304 and lay["lda"] == 104
    assert lay["x_offset"][0] % 1024 == 0 and lay["x_offset"][1] - lay["x_offset"][0] >= 3 * 100 * 304 * 2
    assert lay["b_offset"] - lay["a_offset"] >= 3 * 100 * 104 * 2


def test_empty_inputs_are_noops(L):
    assert call_step(L, [], n=0) == muon.MUON_OK
    assert L.ns5(None, 0, None, 0, 4, 4, 5, None, 0, None) == muon.MUON_OK


@pytest.mark.parametrize("case,code", [
    ("null_param", muon.MUON_ERR_INVALID_ARG),
    ("null_grad", muon.MUON_ERR_INVALID_ARG),
    ("zero_rows", muon.MUON_ERR_INVALID_ARG),
    ("neg_cols", muon.MUON_ERR_INVALID_ARG),
    ("bad_dtype", muon.MUON_ERR_INVALID_ARG),
    ("reserved", muon.MUON_ERR_INVALID_ARG),
    ("neg_steps", muon.MUON_ERR_INVALID_ARG),
    ("bad_nesterov", muon.MUON_ERR_INVALID_ARG),
    ("neg_n", muon.MUON_ERR_INVALID_ARG),
    ("misaligned_param", muon.MUON_ERR_MISALIGNED),
    ("misaligned_grad", muon.MUON_ERR_MISALIGNED),
    ("misaligned_ws", muon.MUON_ERR_MISALIGNED),
    ("null_ws", muon.MUON_ERR_INVALID_ARG),
    ("ws_small", muon.MUON_ERR_WORKSPACE_TOO_SMALL),
    ("alias_param_buf", muon.MUON_ERR_ALIASING),
    ("alias_grad_param", muon.MUON_ERR_ALIASING),
    ("alias_across", muon.MUON_ERR_ALIASING),
    ("alias_ws", muon.MUON_ERR_ALIASING),
    ("too_large", muon.MUON_ERR_TOO_LARGE),
])
def test_step_argument_errors(L, case, code):
    d = desc()
    kw = {}
    descs = [d]
    if case == "null_param":
        descs = [desc(param=0)]
    elif case == "null_grad":
        descs = [desc(grad=0)]
    elif case == "zero_rows":
        descs = [desc(rows=0)]
    elif case == "neg_cols":
        descs = [desc(cols=-3)]
    elif case == "bad_dtype":
        descs = [desc(dtype=7)]
    elif case == "reserved":
        descs = [desc(reserved=1)]
    elif case == "neg_steps":
        kw["ns_steps"] = -1
    elif case == "bad_nesterov":
        kw["nesterov"] = 2
    elif case == "neg_n":
        kw["n"] = -1
    elif case == "misaligned_param":
        descs = [desc(param=0x100004)]
    elif case == "misaligned_grad":
        descs = [desc(grad=0x200008)]
    elif case == "misaligned_ws":
        kw["ws"] = 0x40000010
    elif case == "null_ws":
        kw["ws"] = 0
    elif case == "ws_small":
        kw["ws_bytes"] = 1024
    elif case == "alias_param_buf":
        descs = [desc(buf=0x100000 + 64)]
    elif case == "alias_grad_param":
        descs = [desc(grad=0x100000 + 16)]
    elif case == "alias_across":
        descs = [desc(), desc(param=0x500000, grad=0x600000, buf=0x300000)]
    elif case == "alias_ws":
        kw["ws"] = 0x100000 - 256
    elif case == "too_large":
        descs = [desc(rows=1 << 31)]
    assert call_step(L, descs, **kw) == code


def test_shared_read_only_grad_is_allowed_before_device(L):
    # two matrices may read the same gradient; with a too-small workspace the
    # call stops at the workspace check, after the aliasing check passed
    descs = [desc(), desc(param=0x500000, buf=0x600000)]
    assert call_step(L, descs, ws_bytes=16) == muon.MUON_ERR_WORKSPACE_TOO_SMALL


def test_ns5_argument_errors(L):
    f = L.ns5
    big = 1 << 40
    assert f(None, 0, ctypes.c_void_p(0x1000), 1, 4, 4, 5, ctypes.c_void_p(0x40000000), big, None) == muon.MUON_ERR_INVALID_ARG
    assert f(ctypes.c_void_p(0x1000), 3, ctypes.c_void_p(0x2000), 1, 4, 4, 5, ctypes.c_void_p(0x40000000), big, None) == muon.MUON_ERR_INVALID_ARG
    assert f(ctypes.c_void_p(0x1002), 0, ctypes.c_void_p(0x2000), 1, 4, 4, 5, ctypes.c_void_p(0x40000000), big, None) == muon.MUON_ERR_MISALIGNED
    # G and O overlap
    assert f(ctypes.c_void_p(0x1000), 0, ctypes.c_void_p(0x1010), 1, 4, 4, 5, ctypes.c_void_p(0x40000000), big, None) == muon.MUON_ERR_ALIASING
    assert f(ctypes.c_void_p(0x1000), 0, ctypes.c_void_p(0x2000), 1, 4, 4, -2, ctypes.c_void_p(0x40000000), big, None) == muon.MUON_ERR_INVALID_ARG
    assert f(ctypes.c_void_p(0x1000), 0, ctypes.c_void_p(0x2000), 1, 4, 4, 5, ctypes.c_void_p(0x40000000), 8, None) == muon.MUON_ERR_WORKSPACE_TOO_SMALL
    assert f(ctypes.c_void_p(0x1000), 0, ctypes.c_void_p(0x2000), -1, 4, 4, 5, ctypes.c_void_p(0x40000000), big, None) == muon.MUON_ERR_INVALID_ARG


def test_set_debug_keys(L):
    assert L.muon_set_debug(b"no_such_key", 1) == -1
    assert L.muon_set_debug(b"wait_budget_cycles", 4000000000) == 0
    assert L.muon_set_debug(b"inject_stall", 0) == 0
    assert L.muon_set_debug(b"record_kernel_events", 0) == 0


# ------------------------------------------------------------------ fp8_mm
FX, FW, FO, FXQ, FWQ, FWS = (0x7F0000000000 + k * 0x10000000 for k in range(6))


def fp8_call(L, M=256, N=256, K=256, x_s=0.01, w_s=0.02, x=FX, w=FW, out=FO, xq=FXQ, wq=FWQ, ws=FWS, wsb=256):
    c = ctypes.c_void_p
    return L.fp8_mm(c(x), c(w), x_s, w_s, c(out), c(xq), c(wq), M, N, K, c(ws), wsb, None)


@pytest.mark.parametrize("kw,code", [
    (dict(K=24), "INVALID_ARG"), (dict(K=0), "INVALID_ARG"), (dict(N=12), "INVALID_ARG"),
    (dict(M=-1), "INVALID_ARG"), (dict(x=0), "INVALID_ARG"), (dict(wq=0), "INVALID_ARG"),
    (dict(ws=0), "INVALID_ARG"), (dict(x_s=0.0), "INVALID_ARG"), (dict(w_s=-1.0), "INVALID_ARG"),
    (dict(x_s=float("inf")), "INVALID_ARG"), (dict(w_s=float("nan")), "INVALID_ARG"),
    (dict(x=FX + 8), "MISALIGNED"), (dict(xq=FXQ + 4), "MISALIGNED"), (dict(ws=FWS + 16), "MISALIGNED"),
    (dict(wsb=128), "WORKSPACE_TOO_SMALL"), (dict(M=1 << 31), "TOO_LARGE"),
    (dict(out=FX + 256), "ALIASING"), (dict(wq=FXQ + 4096), "ALIASING"), (dict(ws=FO), "ALIASING"),
])
def test_fp8_mm_argument_errors(L, kw, code):
    """Every case is rejected before any CUDA call (fake device addresses)."""
    assert fp8_call(L, **kw) == getattr(muon, "MUON_ERR_" + code)


def test_fp8_mm_empty_is_a_no_op(L):
    assert fp8_call(L, M=0) == muon.MUON_OK
    assert fp8_call(L, N=0, x=0) == muon.MUON_OK


def test_fp8_mm_binding_rejects_bad_tensors():
    """Argument checks of the binding, before any library call."""
    import torch
    x = torch.zeros((4, 16), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        muon.fp8_mm(x, x, 1.0, 1.0)  # not CUDA tensors
    with pytest.raises(ValueError):
        muon.fp8_mm(x.float(), x, 1.0, 1.0)  # not bfloat16


def test_ns5_bank_binding_checks_outs():
    import torch
    G = [torch.zeros((4, 8)), torch.zeros((8, 4))]
    with pytest.raises(ValueError):
        muon.ns5_bank(G, 5, outs=[torch.zeros((4, 8), dtype=torch.bfloat16)])  # one out for two G
    with pytest.raises(ValueError):
        muon.ns5_bank(G, 5, outs=[torch.zeros((4, 8), dtype=torch.bfloat16), torch.zeros((4, 8), dtype=torch.bfloat16)])
    with pytest.raises(ValueError):
        muon.ns5_bank([torch.zeros(8)], 5)  # not 2-D


def test_fp8_backward_workspace_size(L):
    assert muon.fp8_mm_backward_workspace_size(0, 16, 16) == 256
    assert muon.fp8_mm_backward_workspace_size(17, 16, 16) == 0
    assert muon.fp8_mm_backward_workspace_size(-16, 16, 16) == 0
    # status word, then the transposed copies of g_f8 (N x M), x_f8 (K x M)
    # and w_f8 (K x N), 1 KiB aligned; 36 output tiles of grad_w split twice
    M, N, K = 65536, 3072, 768
    size = muon.fp8_mm_backward_workspace_size(M, N, K)
    copies = 1024 + N * M + K * M + K * N
    assert size == copies + 2 * N * K * 4
    # enough output tiles: no partial sums
    assert muon.fp8_mm_backward_workspace_size(256, 4096, 4096) == 1024 + 4096 * 256 * 2 + 4096 * 4096


@pytest.mark.parametrize("case,code", [
    ("ragged_m", muon.MUON_ERR_INVALID_ARG),
    ("neg_k", muon.MUON_ERR_INVALID_ARG),
    ("null_g", muon.MUON_ERR_INVALID_ARG),
    ("zero_scale", muon.MUON_ERR_INVALID_ARG),
    ("nan_scale", muon.MUON_ERR_INVALID_ARG),
    ("misaligned_out", muon.MUON_ERR_MISALIGNED),
    ("misaligned_ws", muon.MUON_ERR_MISALIGNED),
    ("ws_small", muon.MUON_ERR_WORKSPACE_TOO_SMALL),
    ("alias_out_in", muon.MUON_ERR_ALIASING),
    ("alias_ws", muon.MUON_ERR_ALIASING),
])
def test_fp8_backward_argument_errors(L, case, code):
    M, N, K = 64, 32, 48
    a = dict(g=0x1000000, x=0x2000000, w=0x3000000, gx=0x4000000, gw=0x5000000, gq=0x6000000,
             xs=1.0, ws_=1.0, gs=1.0, M=M, N=N, K=K, wsp=0x8000000,
             wsb=muon.fp8_mm_backward_workspace_size(M, N, K))
    if case == "ragged_m":
        a["M"] = 60
    elif case == "neg_k":
        a["K"] = -16
    elif case == "null_g":
        a["g"] = 0
    elif case == "zero_scale":
        a["gs"] = 0.0
    elif case == "nan_scale":
        a["xs"] = float("nan")
    elif case == "misaligned_out":
        a["gx"] += 8
    elif case == "misaligned_ws":
        a["wsp"] += 16
    elif case == "ws_small":
        a["wsb"] -= 1
    elif case == "alias_out_in":
        a["gx"] = a["g"] + 64
    elif case == "alias_ws":
        a["gw"] = a["wsp"] + 256
    vp = ctypes.c_void_p
    st = L.fp8_mm_backward(vp(a["g"]), vp(a["x"]), vp(a["w"]), a["xs"], a["ws_"], a["gs"], vp(a["gx"]), vp(a["gw"]),
                           vp(a["gq"]), a["M"], a["N"], a["K"], vp(a["wsp"]), a["wsb"], None)
    assert st == code


def test_debug_build_exports_and_release_reports_no_checks(L):
    import ctypes
    D = muon.load(muon.DEBUG_LIB_PATH)
    for n in declared_functions():
        assert hasattr(D, n), n
    n = ctypes.c_longlong(-5)
    assert L.muon_debug_check_failures(n) == -1 and n.value == 0  # release: no checks
    assert L.muon_debug_check_failures(None) == -1
