"""ctypes binding of libmuon.so (include/muon.h): argument marshalling only.

Every step of the Muon update runs inside the library's CUDA kernels; this
module turns torch tensors into device pointers and the current torch stream
into a cudaStream_t, allocates the workspace with torch when the caller does
not pass one, and raises ``MuonError`` on a non-OK status.  It loads the
library on first use and fails loudly if it has not been built.
"""

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libmuon.so")
#: the same library with device-side checks (tests and debugging)
DEBUG_LIB_PATH = os.path.join(_PKG, "lib", "libmuon_debug.so")

MUON_OK = 0
MUON_WARN_NONFINITE = 1
MUON_ERR_INVALID_ARG = -1
MUON_ERR_MISALIGNED = -2
MUON_ERR_ALIASING = -3
MUON_ERR_WORKSPACE_TOO_SMALL = -4
MUON_ERR_CUDA = -5
MUON_ERR_DEVICE_TIMEOUT = -6
MUON_ERR_UNSUPPORTED_DEVICE = -7
MUON_ERR_TOO_LARGE = -8
MUON_ERR_SCRATCH_LIMIT = -9
MUON_BF16 = 0
MUON_F32 = 1

#: every symbol include/muon.h declares
EXPORTS = ["muon_workspace_size", "muon_step", "ns5_workspace_size", "ns5", "ns5_bank",
           "ns5_bank_workspace_size", "muon_device_status", "muon_status_str",
           "ns5_workspace_layout", "muon_set_debug", "muon_kernel_times", "ns5_noalloc", "ns5_noalloc_status",
           "muon_partition", "adam_step", "fp8_mm", "muon_plan_cache_clear",
           "fp8_mm_backward", "fp8_mm_backward_workspace_size", "muon_debug_check_failures"]

#: bytes of the static device scratch ns5_noalloc uses (MUON_NOALLOC_SCRATCH_BYTES)
NOALLOC_SCRATCH_BYTES = 64 << 20

#: kernel kinds reported by muon_kernel_times
KERNEL_KINDS = ["momentum_cast", "normalise", "gram", "poly", "update", "apply", "update_apply", "fp8_quantize",
                "fp8_mm", "fp8_transpose", "fp8_mm_bwd", "fp8_reduce"]


class MuonError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {muon_status_str(status)} (status {status})")


class muon_mat_desc(ctypes.Structure):
    _fields_ = [("param", ctypes.c_void_p), ("grad", ctypes.c_void_p), ("buf", ctypes.c_void_p),
                ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("grad_dtype", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class muon_ws_layout(ctypes.Structure):
    _fields_ = [("x_offset", ctypes.c_size_t * 2), ("a_offset", ctypes.c_size_t),
                ("b_offset", ctypes.c_size_t), ("ldx", ctypes.c_int64), ("lda", ctypes.c_int64),
                ("m", ctypes.c_int64), ("n", ctypes.c_int64)]


class adam_tensor_desc(ctypes.Structure):
    _fields_ = [("param", ctypes.c_void_p), ("grad", ctypes.c_void_p), ("exp_avg", ctypes.c_void_p),
                ("exp_avg_sq", ctypes.c_void_p), ("numel", ctypes.c_int64),
                ("grad_dtype", ctypes.c_int32), ("reserved", ctypes.c_int32)]


_lib = None


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        _lib = load(LIB_PATH)
    return _lib


def load(path):
    """A ctypes handle on the library at `path` with every entry point's
    signature declared (the release library, or the debug build)."""
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           "`python -m newton_schulz_08_gb300.build` (or __graft_entry__.build())")
    L = ctypes.CDLL(path)
    c_int, c_i64, c_sz, c_vp, c_f = ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_float
    P = ctypes.POINTER
    L.muon_workspace_size.argtypes = [P(muon_mat_desc), c_int]
    L.muon_workspace_size.restype = c_sz
    L.muon_step.argtypes = [P(muon_mat_desc), c_int, c_f, c_f, c_int, c_int, c_vp, c_sz, c_vp]
    L.muon_step.restype = c_int
    L.ns5_workspace_size.argtypes = [c_int, c_i64, c_i64]
    L.ns5_workspace_size.restype = c_sz
    L.ns5.argtypes = [c_vp, c_int, c_vp, c_int, c_i64, c_i64, c_int, c_vp, c_sz, c_vp]
    L.ns5.restype = c_int
    L.ns5_bank.argtypes = [P(c_vp), P(ctypes.c_int32), P(c_vp), P(c_i64), P(c_i64), c_int, c_int,
                           c_vp, c_sz, c_vp]
    L.ns5_bank.restype = c_int
    L.ns5_bank_workspace_size.argtypes = [P(c_i64), P(c_i64), c_int]
    L.ns5_bank_workspace_size.restype = c_sz
    L.muon_device_status.argtypes = [c_vp, c_vp]
    L.muon_device_status.restype = c_int
    L.muon_status_str.argtypes = [c_int]
    L.muon_status_str.restype = ctypes.c_char_p
    L.ns5_workspace_layout.argtypes = [c_int, c_i64, c_i64, P(muon_ws_layout)]
    L.ns5_workspace_layout.restype = c_int
    L.muon_set_debug.argtypes = [ctypes.c_char_p, ctypes.c_longlong]
    L.muon_set_debug.restype = c_int
    L.muon_kernel_times.argtypes = [P(ctypes.c_double), P(c_int), c_int]
    L.muon_kernel_times.restype = c_int
    L.ns5_noalloc.argtypes = [c_vp, c_int, c_vp, c_int, c_i64, c_i64, c_int, c_vp]
    L.ns5_noalloc.restype = c_int
    L.ns5_noalloc_status.argtypes = [c_vp]
    L.ns5_noalloc_status.restype = c_int
    L.muon_partition.argtypes = [P(c_i64), P(c_i64), c_int, c_int, P(c_int)]
    L.muon_partition.restype = c_int
    L.adam_step.argtypes = [P(adam_tensor_desc), c_int, c_f, c_f, c_f, c_f, c_f, c_int, c_int, c_vp]
    L.adam_step.restype = c_int
    L.fp8_mm.argtypes = [c_vp, c_vp, c_f, c_f, c_vp, c_vp, c_vp, c_i64, c_i64, c_i64, c_vp, c_sz, c_vp]
    L.fp8_mm.restype = c_int
    L.fp8_mm_backward_workspace_size.argtypes = [c_i64, c_i64, c_i64]
    L.fp8_mm_backward_workspace_size.restype = c_sz
    L.fp8_mm_backward.argtypes = [c_vp, c_vp, c_vp, c_f, c_f, c_f, c_vp, c_vp, c_vp, c_i64, c_i64, c_i64, c_vp,
                                  c_sz, c_vp]
    L.fp8_mm_backward.restype = c_int
    L.muon_plan_cache_clear.argtypes = []
    L.muon_plan_cache_clear.restype = None
    L.muon_debug_check_failures.argtypes = [P(ctypes.c_longlong)]
    L.muon_debug_check_failures.restype = c_int
    return L


def muon_status_str(status):
    return lib().muon_status_str(int(status)).decode()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(status, where, ok=(MUON_OK,)):
    if status not in ok:
        raise MuonError(status, where)
    return status


def _device_of(tensors, what):
    """The one CUDA device all `tensors` live on (raises otherwise).  The
    library works on the current device with device pointers, so a CPU
    tensor or a tensor of another GPU must never reach it."""
    dev = None
    for t in tensors:
        if not t.is_cuda:
            raise ValueError(f"{what}: every tensor must be a CUDA tensor")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"{what}: tensors are on {dev} and {t.device}; all must share one device")
    return dev


def _dtype_code(t):
    if t.dtype == torch.bfloat16:
        return MUON_BF16
    if t.dtype == torch.float32:
        return MUON_F32
    raise TypeError(f"unsupported dtype {t.dtype} (bfloat16 or float32)")


def _descs(params, grads, bufs):
    n = len(params)
    if len(grads) != n or len(bufs) != n:
        raise ValueError("params, grads and bufs must have the same length")
    arr = (muon_mat_desc * max(n, 1))()
    for i, (p, g, b) in enumerate(zip(params, grads, bufs)):
        if p.dim() != 2 or g.shape != p.shape or b.shape != p.shape:
            raise ValueError(f"matrix {i}: param, grad and buf must be 2-D of one shape")
        if p.dtype != torch.float32 or b.dtype != torch.float32:
            raise TypeError(f"matrix {i}: param and buf must be float32")
        if not (p.is_contiguous() and g.is_contiguous() and b.is_contiguous()):
            raise ValueError(f"matrix {i}: tensors must be contiguous")
        arr[i] = muon_mat_desc(p.data_ptr(), g.data_ptr(), b.data_ptr(), p.shape[0], p.shape[1],
                               _dtype_code(g), 0)
    return arr, n


def muon_workspace_size(shapes):
    """Workspace bytes for a bank given as a list of (rows, cols)."""
    n = len(shapes)
    arr = (muon_mat_desc * max(n, 1))()
    for i, (r, c) in enumerate(shapes):
        arr[i] = muon_mat_desc(0, 0, 0, r, c, MUON_BF16, 0)
    return lib().muon_workspace_size(arr, n)


def new_workspace(nbytes, device=None):
    device = device or torch.device("cuda", torch.cuda.current_device())
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def muon_step(params, grads, bufs, lr=0.02, momentum=0.95, nesterov=True, ns_steps=5,
              workspace=None, stream=None):
    """One Muon step over a bank (lists of 2-D CUDA tensors), in place."""
    arr, n = _descs(params, grads, bufs)
    if n == 0:
        return workspace
    dev = _device_of(list(params) + list(grads) + list(bufs) + ([workspace] if workspace is not None else []),
                     "muon_step")
    with torch.cuda.device(dev):
        if workspace is None:
            workspace = new_workspace(lib().muon_workspace_size(arr, n), dev)
        st = lib().muon_step(arr, n, float(lr), float(momentum), int(bool(nesterov)), int(ns_steps),
                             ctypes.c_void_p(workspace.data_ptr()), workspace.numel(), _stream(stream))
    _check(st, "muon_step")
    return workspace


class StepGraph:
    """One muon_step recorded in a CUDA graph for fixed tensors, scalars and
    workspace; replay() runs the step's launches (momentum pass, normalise,
    the Newton-Schulz launches) with one host call.  The recording itself
    runs nothing: params and bufs are first changed by the first replay.
    The graph holds the tensors' addresses, so they must stay alive and in
    place; a change of lr, momentum or ns_steps needs a new StepGraph.
    Kernel-event recording (muon_set_debug "record_kernel_events") must be
    off while recording."""

    def __init__(self, params, grads, bufs, lr=0.02, momentum=0.95, nesterov=True, ns_steps=5, workspace=None):
        self.tensors = (list(params), list(grads), list(bufs))
        arr, n = _descs(*self.tensors)
        if n == 0:
            raise ValueError("StepGraph needs at least one matrix")
        dev = _device_of(self.tensors[0] + self.tensors[1] + self.tensors[2]
                         + ([workspace] if workspace is not None else []), "StepGraph")
        with torch.cuda.device(dev):
            if workspace is None:
                workspace = new_workspace(lib().muon_workspace_size(arr, n), dev)
            self.workspace = workspace
            self.stream = torch.cuda.Stream(dev)
            self.graph = torch.cuda.CUDAGraph()
            self.stream.wait_stream(torch.cuda.current_stream(dev))
            # relaxed: the first call of a bank also sets kernel attributes and
            # queries occupancy, which are not stream work
            with torch.cuda.graph(self.graph, stream=self.stream, capture_error_mode="relaxed"):
                muon_step(params, grads, bufs, lr=lr, momentum=momentum, nesterov=nesterov, ns_steps=ns_steps,
                          workspace=workspace, stream=self.stream)

    def replay(self):
        """Runs the recorded step (on the graph's stream, ordered after the
        current stream's work so far; the current stream waits for it)."""
        cur = torch.cuda.current_stream(self.stream.device)
        self.stream.wait_stream(cur)
        with torch.cuda.stream(self.stream):
            self.graph.replay()
        cur.wait_stream(self.stream)


def ns5_workspace_size(batch, rows, cols):
    return lib().ns5_workspace_size(int(batch), int(rows), int(cols))


def ns5(G, ns_steps=5, out=None, workspace=None, stream=None):
    """zeropower_via_newtonschulz5 on a (batch x) rows x cols CUDA tensor -> bf16."""
    squeeze = G.dim() == 2
    G3 = G.unsqueeze(0) if squeeze else G
    if G3.dim() != 3 or not G3.is_contiguous():
        raise ValueError("G must be a contiguous 2-D or 3-D tensor")
    batch, rows, cols = G3.shape
    if out is None:
        out = torch.empty(G3.shape, dtype=torch.bfloat16, device=G.device)
    if out.shape != G3.shape or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError("out must be a contiguous bfloat16 tensor shaped like G")
    dev = _device_of([G3, out] + ([workspace] if workspace is not None else []), "ns5")
    with torch.cuda.device(dev):
        if workspace is None:
            workspace = new_workspace(ns5_workspace_size(batch, rows, cols) if batch else 256, dev)
        st = lib().ns5(ctypes.c_void_p(G3.data_ptr()), _dtype_code(G3), ctypes.c_void_p(out.data_ptr()),
                       batch, rows, cols, int(ns_steps), ctypes.c_void_p(workspace.data_ptr()),
                       workspace.numel(), _stream(stream))
    _check(st, "ns5")
    return out[0] if squeeze else out


def ns5_bank_workspace_size(shapes):
    n = len(shapes)
    rows = (ctypes.c_int64 * max(n, 1))(*[s[0] for s in shapes])
    cols = (ctypes.c_int64 * max(n, 1))(*[s[1] for s in shapes])
    return lib().ns5_bank_workspace_size(rows, cols, n)


def ns5_bank(Gs, ns_steps=5, outs=None, workspace=None, stream=None):
    """Newton-Schulz on a list of differently shaped 2-D CUDA tensors -> bf16 list."""
    n = len(Gs)
    if outs is None:
        outs = [torch.empty(g.shape, dtype=torch.bfloat16, device=g.device) for g in Gs]
    if len(outs) != n:
        raise ValueError("outs must have one tensor per G")
    for g, o in zip(Gs, outs):
        if (g.dim() != 2 or not g.is_contiguous() or o.shape != g.shape or o.dtype != torch.bfloat16
                or not o.is_contiguous()):
            raise ValueError("each G must be 2-D contiguous with a contiguous bf16 out of the same shape")
    if n == 0:
        return outs
    dev = _device_of(list(Gs) + list(outs) + ([workspace] if workspace is not None else []), "ns5_bank")
    gp = (ctypes.c_void_p * max(n, 1))(*[g.data_ptr() for g in Gs])
    op = (ctypes.c_void_p * max(n, 1))(*[o.data_ptr() for o in outs])
    dt = (ctypes.c_int32 * max(n, 1))(*[_dtype_code(g) for g in Gs])
    rows = (ctypes.c_int64 * max(n, 1))(*[g.shape[0] for g in Gs])
    cols = (ctypes.c_int64 * max(n, 1))(*[g.shape[1] for g in Gs])
    with torch.cuda.device(dev):
        if workspace is None:
            workspace = new_workspace(lib().ns5_bank_workspace_size(rows, cols, n), dev)
        st = lib().ns5_bank(gp, dt, op, rows, cols, n, int(ns_steps),
                            ctypes.c_void_p(workspace.data_ptr()), workspace.numel(), _stream(stream))
    _check(st, "ns5_bank")
    return outs


def muon_device_status(workspace, stream=None):
    """Synchronise and read the workspace's device status word (an int code)."""
    return lib().muon_device_status(ctypes.c_void_p(workspace.data_ptr()), _stream(stream))


def ns5_workspace_layout(batch, rows, cols):
    out = muon_ws_layout()
    _check(lib().ns5_workspace_layout(int(batch), int(rows), int(cols), ctypes.byref(out)),
           "ns5_workspace_layout")
    return {"x_offset": (out.x_offset[0], out.x_offset[1]), "a_offset": out.a_offset,
            "b_offset": out.b_offset, "ldx": out.ldx, "lda": out.lda, "m": out.m, "n": out.n}


def muon_plan_cache_clear():
    """Drop the library's prepared calls (host memory only)."""
    lib().muon_plan_cache_clear()


def muon_set_debug(key, value):
    if lib().muon_set_debug(key.encode(), int(value)) != 0:
        raise KeyError(key)


def muon_kernel_times():
    """{kind: (total_ms, launches)} for launches recorded since the last call."""
    n = len(KERNEL_KINDS)
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_int * n)()
    if lib().muon_kernel_times(ms, cnt, n) != 0:
        raise RuntimeError("muon_kernel_times failed")
    return {k: (ms[i], cnt[i]) for i, k in enumerate(KERNEL_KINDS)}


def ns5_noalloc(G, ns_steps=5, out=None, stream=None):
    """ns5 without a workspace: the library's own static device scratch is
    used (for callers that may not allocate device memory; see include/muon.h).
    Only `out` is allocated here when the caller does not pass one."""
    squeeze = G.dim() == 2
    G3 = G.unsqueeze(0) if squeeze else G
    if G3.dim() != 3 or not G3.is_contiguous():
        raise ValueError("G must be a contiguous 2-D or 3-D tensor")
    batch, rows, cols = G3.shape
    if out is None:
        out = torch.empty(G3.shape, dtype=torch.bfloat16, device=G.device)
    if out.shape != G3.shape or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError("out must be a contiguous bfloat16 tensor shaped like G")
    dev = _device_of([G3, out], "ns5_noalloc")
    # the library's scratch array and the default stream are the current
    # device's: make G's device current for the call
    with torch.cuda.device(dev):
        st = lib().ns5_noalloc(ctypes.c_void_p(G3.data_ptr()), _dtype_code(G3),
                               ctypes.c_void_p(out.data_ptr()), batch, rows, cols, int(ns_steps),
                               _stream(stream))
    _check(st, "ns5_noalloc")
    return out[0] if squeeze else out


def ns5_noalloc_status(stream=None, device=None):
    """Device status of the last ns5_noalloc call on `device` (default: the
    current one), read after synchronising `stream`: MUON_OK,
    MUON_WARN_NONFINITE or MUON_ERR_DEVICE_TIMEOUT (see include/muon.h)."""
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        return lib().ns5_noalloc_status(_stream(stream))


def partition(shapes, world):
    """Owner rank of each matrix of a bank of (rows, cols) shapes when the
    step runs on `world` processes: heaviest Newton-Schulz work first, each
    matrix to the least-loaded rank (muon_partition; host only)."""
    n = len(shapes)
    rows = (ctypes.c_int64 * max(n, 1))(*[int(r) for r, _ in shapes])
    cols = (ctypes.c_int64 * max(n, 1))(*[int(c) for _, c in shapes])
    owner = (ctypes.c_int * max(n, 1))()
    _check(lib().muon_partition(rows, cols, n, int(world), owner), "muon_partition")
    return [owner[i] for i in range(n)]


def adam_step(params, grads, exp_avgs, exp_avg_sqs, step, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8,
              weight_decay=0.0, cautious=True, stream=None):
    """Adam step with cautious weight decay over lists of CUDA tensors, in
    place (fp32 params and moments; bf16 or fp32 grads).  See adam_step in
    include/muon.h for the arithmetic."""
    n = len(params)
    if not (len(grads) == len(exp_avgs) == len(exp_avg_sqs) == n):
        raise ValueError("params, grads, exp_avgs, exp_avg_sqs must have the same length")
    arr = (adam_tensor_desc * max(n, 1))()
    for i, (p, g, m, v) in enumerate(zip(params, grads, exp_avgs, exp_avg_sqs)):
        for t in (p, m, v):
            if t.dtype != torch.float32 or not t.is_contiguous() or not t.is_cuda:
                raise ValueError("params and moments must be contiguous float32 CUDA tensors")
        if not (p.numel() == g.numel() == m.numel() == v.numel()) or not g.is_contiguous():
            raise ValueError("tensor sizes differ or a gradient is not contiguous")
        arr[i] = adam_tensor_desc(p.data_ptr(), g.data_ptr(), m.data_ptr(), v.data_ptr(), p.numel(),
                                  _dtype_code(g), 0)
    if n == 0:
        return
    dev = _device_of(list(params) + list(grads) + list(exp_avgs) + list(exp_avg_sqs), "adam_step")
    with torch.cuda.device(dev):
        st = lib().adam_step(arr, n, float(lr), float(beta1), float(beta2), float(eps), float(weight_decay),
                             int(step), int(bool(cautious)), _stream(stream))
    _check(st, "adam_step")


def fp8_mm(x, w, x_s, w_s, out=None, x_f8=None, w_f8=None, workspace=None, stream=None):
    """FP8 scaled product of bf16 CUDA tensors x (M x K) and w (N x K):
    returns (out, x_f8, w_f8), out = bf16(x_s w_s (x_f8 . w_f8^T)) with
    x_f8 = E4M3(bf16(x / x_s)), w_f8 = E4M3(bf16(w / w_s)) as float8_e4m3fn
    tensors.  See fp8_mm in include/muon.h."""
    for t in (x, w):
        if t.dim() != 2 or t.dtype != torch.bfloat16 or not t.is_contiguous() or not t.is_cuda:
            raise ValueError("x and w must be contiguous 2-D bfloat16 CUDA tensors")
    M, K = x.shape
    N = w.shape[0]
    if w.shape[1] != K:
        raise ValueError("x and w must have the same number of columns")
    dev = x.device
    out = torch.empty((M, N), dtype=torch.bfloat16, device=dev) if out is None else out
    x_f8 = torch.empty((M, K), dtype=torch.uint8, device=dev) if x_f8 is None else x_f8
    w_f8 = torch.empty((N, K), dtype=torch.uint8, device=dev) if w_f8 is None else w_f8
    # the library writes exactly these sizes: check the caller's buffers
    if out.shape != (M, N) or out.dtype != torch.bfloat16 or not out.is_contiguous() or out.device != dev:
        raise ValueError("out must be a contiguous M x N bfloat16 tensor on x's device")
    for t, shape in ((x_f8, (M, K)), (w_f8, (N, K))):
        if (t.shape != shape or t.element_size() != 1 or not t.is_contiguous() or t.device != dev
                or t.dtype not in (torch.uint8, torch.float8_e4m3fn)):
            raise ValueError("x_f8 / w_f8 must be contiguous one-byte (uint8 or float8_e4m3fn) tensors "
                             "shaped like x / w, on x's device")
    x_f8, w_f8 = x_f8.view(torch.uint8), w_f8.view(torch.uint8)
    if w.device != dev:
        raise ValueError("x and w must be on the same device")
    _device_of([x, w, out, x_f8, w_f8] + ([workspace] if workspace is not None else []), "fp8_mm")
    with torch.cuda.device(dev):
        if workspace is None:
            workspace = new_workspace(256, dev)
        st = lib().fp8_mm(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(w.data_ptr()), float(x_s), float(w_s),
                          ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(x_f8.data_ptr()),
                          ctypes.c_void_p(w_f8.data_ptr()), M, N, K, ctypes.c_void_p(workspace.data_ptr()),
                          workspace.numel(), _stream(stream))
    _check(st, "fp8_mm")
    return out, x_f8.view(torch.float8_e4m3fn), w_f8.view(torch.float8_e4m3fn)


def fp8_mm_backward_workspace_size(M, N, K):
    return lib().fp8_mm_backward_workspace_size(int(M), int(N), int(K))


def fp8_mm_backward(g, x_f8, w_f8, x_s, w_s, grad_s, grad_x=None, grad_w=None, g_f8=None, workspace=None,
                    stream=None):
    """Backward of the FP8 scaled product: g (M x N bf16) and the forward's
    x_f8 (M x K) and w_f8 (N x K) E4M3 codes -> (grad_x, grad_w, g_f8):
    grad_x = bf16(grad_s w_s (g_f8 . w_f8)), grad_w = bf16(grad_s x_s
    (g_f8^T . x_f8)), g_f8 = E5M2(bf16(g / grad_s)) as a float8_e5m2 tensor.
    See fp8_mm_backward in include/muon.h."""
    if g.dim() != 2 or g.dtype != torch.bfloat16 or not g.is_contiguous():
        raise ValueError("g must be a contiguous 2-D bfloat16 CUDA tensor")
    M, N = g.shape
    for t, shape in ((x_f8, None), (w_f8, None)):
        if t.dim() != 2 or t.element_size() != 1 or not t.is_contiguous():
            raise ValueError("x_f8 / w_f8 must be contiguous 2-D one-byte tensors")
    K = x_f8.shape[1]
    if x_f8.shape != (M, K) or w_f8.shape != (N, K):
        raise ValueError("x_f8 must be M x K and w_f8 N x K for g of M x N")
    dev = _device_of([g, x_f8, w_f8] + [t for t in (grad_x, grad_w, g_f8, workspace) if t is not None],
                     "fp8_mm_backward")
    grad_x = torch.empty((M, K), dtype=torch.bfloat16, device=dev) if grad_x is None else grad_x
    grad_w = torch.empty((N, K), dtype=torch.bfloat16, device=dev) if grad_w is None else grad_w
    g_f8 = torch.empty((M, N), dtype=torch.uint8, device=dev) if g_f8 is None else g_f8
    for t, shape in ((grad_x, (M, K)), (grad_w, (N, K))):
        if t.shape != shape or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError("grad_x / grad_w must be contiguous bfloat16 tensors of M x K / N x K")
    if (g_f8.shape != (M, N) or g_f8.element_size() != 1 or not g_f8.is_contiguous()
            or g_f8.dtype not in (torch.uint8, torch.float8_e5m2)):
        raise ValueError("g_f8 must be a contiguous M x N one-byte tensor (uint8 or float8_e5m2)")
    g_f8 = g_f8.view(torch.uint8)
    with torch.cuda.device(dev):
        if workspace is None:
            workspace = new_workspace(fp8_mm_backward_workspace_size(M, N, K), dev)
        st = lib().fp8_mm_backward(ctypes.c_void_p(g.data_ptr()), ctypes.c_void_p(x_f8.data_ptr()),
                                   ctypes.c_void_p(w_f8.data_ptr()), float(x_s), float(w_s), float(grad_s),
                                   ctypes.c_void_p(grad_x.data_ptr()), ctypes.c_void_p(grad_w.data_ptr()),
                                   ctypes.c_void_p(g_f8.data_ptr()), M, N, K, ctypes.c_void_p(workspace.data_ptr()),
                                   workspace.numel(), _stream(stream))
    _check(st, "fp8_mm_backward")
    return grad_x, grad_w, g_f8.view(torch.float8_e5m2)
