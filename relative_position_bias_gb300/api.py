"""ctypes binding of libdera_relpos (argument marshalling only).

Every step of the computation runs in the library's CUDA kernels; this module
only checks that tensor shapes agree with the sizes it passes, takes data
pointers and the current CUDA stream from PyTorch, and turns error codes
into exceptions.  There is no fallback: if the library is missing or a call
fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdera_relpos.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "dera_relpos.h")

DERA_F16, DERA_BF16, DERA_F32 = 0, 1, 2
_DTYPE_CODE = {torch.float16: DERA_F16, torch.bfloat16: DERA_BF16, torch.float32: DERA_F32}
STATUS_NAMES = {0: "DERA_OK", 1: "DERA_ERR_NULL", 2: "DERA_ERR_SHAPE", 3: "DERA_ERR_DTYPE",
                4: "DERA_ERR_HEAD_DIM", 5: "DERA_ERR_ALIGN", 6: "DERA_ERR_DEVICE", 7: "DERA_ERR_TIMEOUT",
                8: "DERA_ERR_CUDA", 9: "DERA_ERR_SCRATCH"}

_lib = None
_lock = threading.Lock()
_workspaces: dict = {}    # (device index, stream handle) -> uint8 scratch reused by the calls on that stream


class DeraError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load (once) the in-tree shared library and declare its signatures."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is missing: build it with `python -m relative_position_bias_gb300.build`")
        lib = ctypes.CDLL(p)
        vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        lib.dera_relpos_project.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, vp]
        lib.dera_relpos_project.restype = i
        sz = ctypes.c_size_t
        lib.dera_relpos_attention.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, i, i, vp, sz, vp]
        lib.dera_relpos_attention.restype = i
        lib.dera_relpos_fused.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp, sz, vp]
        lib.dera_relpos_fused.restype = i
        lib.dera_relpos_workspace_size.argtypes = [i, i, i, i, ctypes.POINTER(sz)]
        lib.dera_relpos_workspace_size.restype = i
        lib.dera_status_string.argtypes = [i]
        lib.dera_status_string.restype = ctypes.c_char_p
        lib.dera_relpos_device_status.argtypes = [ctypes.POINTER(i), i]
        lib.dera_relpos_device_status.restype = i
        lib.dera_relpos_selftest_wait_timeout.argtypes = [ctypes.c_longlong, vp]
        lib.dera_relpos_selftest_wait_timeout.restype = i
        lib.dera_relpos_abi_version.argtypes = []
        lib.dera_relpos_abi_version.restype = i
        lib.dera_relpos_fused_lse.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp, sz, vp]
        lib.dera_relpos_fused_lse.restype = i
        lib.dera_relpos_backward_workspace_size.argtypes = [i, i, i, i, ctypes.POINTER(sz)]
        lib.dera_relpos_backward_workspace_size.restype = i
        lib.dera_relpos_fused_backward.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f,
                                                   i, i, i, vp, sz, vp]
        lib.dera_relpos_fused_backward.restype = i
        _lib = lib
        return lib


def declared_entry_points() -> list[str]:
    """Function names declared in include/dera_relpos.h."""
    with open(HEADER) as fh:
        text = fh.read()
    pat = r"^\s*DERA_API\s+(?:const\s+char\s*\*|dera_status|int)\s+(dera_\w+)\s*\("
    return sorted(set(re.findall(pat, text, re.M)))


def _check(status: int) -> None:
    if status != 0:
        msg = load_library().dera_status_string(status).decode()
        raise DeraError(status, msg)


def _code(t: torch.dtype) -> int:
    if t not in _DTYPE_CODE:
        raise TypeError(f"unsupported dtype {t}")
    return _DTYPE_CODE[t]


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(device: torch.device, stream) -> int | None:
    if stream is not None:
        return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    if device.type != "cuda":
        return None
    return torch.cuda.current_stream(device).cuda_stream


def workspace_size(BH: int, H: int, W: int, head_dim: int = 64) -> int:
    """Scratch bytes the attention entries use for this size on the current device (0 if none)."""
    n = ctypes.c_size_t(0)
    _check(load_library().dera_relpos_workspace_size(BH, H, W, head_dim, ctypes.byref(n)))
    return n.value


def _workspace(device: torch.device, BH: int, H: int, W: int, d: int, workspace, stream_handle):
    """(pointer, bytes) of the scratch for one call: the caller's tensor, none, or a cached buffer.

    The cached buffer is kept per (device, stream): calls on one stream are ordered by it, and
    calls on different streams, which may overlap on the GPU, never share scratch.  A buffer used
    on a stream other than the one current at its allocation is recorded on that stream, so the
    allocator does not hand its memory out again before that stream's work is done."""
    if workspace is False or device.type != "cuda" or BH == 0:
        return None, 0
    if isinstance(workspace, torch.Tensor):
        return workspace.data_ptr(), workspace.numel() * workspace.element_size()
    with torch.cuda.device(device):
        need = workspace_size(BH, H, W, d)
    if need == 0:
        return None, 0
    idx = device.index if device.index is not None else torch.cuda.current_device()
    key = (idx, int(stream_handle or 0))
    with _lock:
        buf = _workspaces.get(key)
        if buf is None or buf.numel() < need:
            buf = torch.empty(need, dtype=torch.uint8, device=device)
            if int(stream_handle or 0) != torch.cuda.current_stream(device).cuda_stream:
                buf.record_stream(torch.cuda.ExternalStream(int(stream_handle or 0), device=device))
            _workspaces[key] = buf
    return buf.data_ptr(), buf.numel()


def _expect(t: torch.Tensor, shape: tuple, name: str) -> None:
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def project(q: torch.Tensor, rel_pos_h: torch.Tensor, rel_pos_w: torch.Tensor, H: int, W: int,
            bias_dtype: torch.dtype = torch.float32, rel_h: torch.Tensor | None = None,
            rel_w: torch.Tensor | None = None, stream=None):
    """``rel_h [BH,N,H]``, ``rel_w [BH,N,W]`` via ``dera_relpos_project``."""
    BH, N, d = q.shape
    if rel_h is None:
        rel_h = torch.empty((BH, N, H), dtype=bias_dtype, device=q.device)
    if rel_w is None:
        rel_w = torch.empty((BH, N, W), dtype=bias_dtype, device=q.device)
    _expect(q, (BH, H * W, d), "q")
    _expect(rel_pos_h, (2 * H - 1, d), "rel_pos_h")
    _expect(rel_pos_w, (2 * W - 1, d), "rel_pos_w")
    _expect(rel_h, (BH, N, H), "rel_h")
    _expect(rel_w, (BH, N, W), "rel_w")
    if rel_h.dtype != rel_w.dtype:
        raise TypeError("rel_h and rel_w must share a dtype")
    lib = load_library()
    _check(lib.dera_relpos_project(_ptr(q), _ptr(rel_pos_h), _ptr(rel_pos_w), _ptr(rel_h), _ptr(rel_w), BH, H, W,
                                   d, _code(q.dtype), _code(rel_h.dtype), _stream(q.device, stream)))
    return rel_h, rel_w


def attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, rel_h: torch.Tensor, rel_w: torch.Tensor,
              H: int, W: int, scale: float | None = None, out_dtype: torch.dtype | None = None,
              out: torch.Tensor | None = None, stream=None, workspace=None) -> torch.Tensor:
    """Attention with a compact bias via ``dera_relpos_attention``.

    ``workspace``: None = a cached scratch buffer per (device, stream), False = no scratch (one
    CTA per unit), or a caller-owned uint8 tensor, which no other call in flight may use."""
    BH, N, d = q.shape
    scale = d ** -0.5 if scale is None else scale
    if out is None:
        out = torch.empty((BH, N, d), dtype=out_dtype or q.dtype, device=q.device)
    for t, name in ((q, "q"), (k, "k"), (v, "v"), (out, "out")):
        _expect(t, (BH, H * W, d), name)
    _expect(rel_h, (BH, N, H), "rel_h")
    _expect(rel_w, (BH, N, W), "rel_w")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share a dtype")
    if rel_h.dtype != rel_w.dtype:
        raise TypeError("rel_h and rel_w must share a dtype")
    lib = load_library()
    st = _stream(q.device, stream)
    ws, ws_bytes = _workspace(q.device, BH, H, W, d, workspace, st)
    _check(lib.dera_relpos_attention(_ptr(q), _ptr(k), _ptr(v), _ptr(rel_h), _ptr(rel_w), _ptr(out), BH, H, W, d,
                                     float(scale), _code(q.dtype), _code(rel_h.dtype), _code(out.dtype), ws,
                                     ws_bytes, st))
    return out


def fused(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, rel_pos_h: torch.Tensor, rel_pos_w: torch.Tensor,
          H: int, W: int, scale: float | None = None, out_dtype: torch.dtype | None = None,
          out: torch.Tensor | None = None, stream=None, workspace=None) -> torch.Tensor:
    """Projection + attention in one kernel via ``dera_relpos_fused`` (``workspace`` as in :func:`attention`)."""
    BH, N, d = q.shape
    scale = d ** -0.5 if scale is None else scale
    if out is None:
        out = torch.empty((BH, N, d), dtype=out_dtype or q.dtype, device=q.device)
    for t, name in ((q, "q"), (k, "k"), (v, "v"), (out, "out")):
        _expect(t, (BH, H * W, d), name)
    _expect(rel_pos_h, (2 * H - 1, d), "rel_pos_h")
    _expect(rel_pos_w, (2 * W - 1, d), "rel_pos_w")
    for t in (k, v, rel_pos_h, rel_pos_w):
        if t.dtype != q.dtype:
            raise TypeError("q, k, v and the tables must share a dtype")
    lib = load_library()
    st = _stream(q.device, stream)
    ws, ws_bytes = _workspace(q.device, BH, H, W, d, workspace, st)
    _check(lib.dera_relpos_fused(_ptr(q), _ptr(k), _ptr(v), _ptr(rel_pos_h), _ptr(rel_pos_w), _ptr(out), BH, H, W,
                                 d, float(scale), _code(q.dtype), _code(out.dtype), ws, ws_bytes, st))
    return out


def fused_lse(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, rel_pos_h: torch.Tensor, rel_pos_w: torch.Tensor,
              H: int, W: int, scale: float | None = None, out_dtype: torch.dtype | None = None, stream=None,
              workspace=None) -> tuple[torch.Tensor, torch.Tensor]:
    """Training forward via ``dera_relpos_fused_lse``: ``(out, lse)``, lse [BH, N] fp32 (base 2)."""
    BH, N, d = q.shape
    scale = d ** -0.5 if scale is None else scale
    out = torch.empty((BH, N, d), dtype=out_dtype or q.dtype, device=q.device)
    lse = torch.empty((BH, N), dtype=torch.float32, device=q.device)
    for t, name in ((q, "q"), (k, "k"), (v, "v")):
        _expect(t, (BH, H * W, d), name)
    _expect(rel_pos_h, (2 * H - 1, d), "rel_pos_h")
    _expect(rel_pos_w, (2 * W - 1, d), "rel_pos_w")
    for t in (k, v, rel_pos_h, rel_pos_w):
        if t.dtype != q.dtype:
            raise TypeError("q, k, v and the tables must share a dtype")
    lib = load_library()
    st = _stream(q.device, stream)
    ws, ws_bytes = _workspace(q.device, BH, H, W, d, workspace, st)
    _check(lib.dera_relpos_fused_lse(_ptr(q), _ptr(k), _ptr(v), _ptr(rel_pos_h), _ptr(rel_pos_w), _ptr(out), _ptr(lse),
                                     BH, H, W, d, float(scale), _code(q.dtype), _code(out.dtype), ws, ws_bytes, st))
    return out, lse


def backward_workspace_size(BH: int, H: int, W: int, head_dim: int = 64) -> int:
    """Scratch bytes of :func:`fused_backward` for this size."""
    n = ctypes.c_size_t(0)
    _check(load_library().dera_relpos_backward_workspace_size(BH, H, W, head_dim, ctypes.byref(n)))
    return n.value


def fused_backward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, rel_pos_h: torch.Tensor,
                   rel_pos_w: torch.Tensor, out: torch.Tensor, lse: torch.Tensor, dout: torch.Tensor, H: int, W: int,
                   scale: float | None = None, grad_dtype: torch.dtype | None = None, stream=None,
                   workspace: torch.Tensor | None = None):
    """Gradients of :func:`fused` via ``dera_relpos_fused_backward``:
    ``(dq, dk, dv, drel_pos_h, drel_pos_w)``; dq, dk, dv in ``grad_dtype`` (default fp32), the
    table gradients fp32.  ``out`` and ``lse`` come from :func:`fused_lse`."""
    BH, N, d = q.shape
    scale = d ** -0.5 if scale is None else scale
    gd = grad_dtype or torch.float32
    for t, name in ((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout")):
        _expect(t, (BH, H * W, d), name)
    _expect(lse, (BH, H * W), "lse")
    _expect(rel_pos_h, (2 * H - 1, d), "rel_pos_h")
    _expect(rel_pos_w, (2 * W - 1, d), "rel_pos_w")
    for t in (k, v, rel_pos_h, rel_pos_w, dout):
        if t.dtype != q.dtype:
            raise TypeError("q, k, v, dout and the tables must share a dtype")
    if lse.dtype != torch.float32:
        raise TypeError("lse must be float32")
    dq = torch.empty((BH, N, d), dtype=gd, device=q.device)
    dk = torch.empty_like(dq)
    dv = torch.empty_like(dq)
    dth = torch.empty((2 * H - 1, d), dtype=torch.float32, device=q.device)
    dtw = torch.empty((2 * W - 1, d), dtype=torch.float32, device=q.device)
    lib = load_library()
    st = _stream(q.device, stream)
    if workspace is None:
        with torch.cuda.device(q.device):
            need = backward_workspace_size(BH, H, W, d)
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
        if int(st or 0) != torch.cuda.current_stream(q.device).cuda_stream:
            # freed when this call returns: the allocator must not hand it out again before
            # the kernels on that stream are done with it
            workspace.record_stream(torch.cuda.ExternalStream(int(st or 0), device=q.device))
    _check(lib.dera_relpos_fused_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(rel_pos_h), _ptr(rel_pos_w), _ptr(out),
                                          _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dth), _ptr(dtw),
                                          BH, H, W, d, float(scale), _code(q.dtype), _code(out.dtype), _code(gd),
                                          workspace.data_ptr(), workspace.numel() * workspace.element_size(), st))
    return dq, dk, dv, dth, dtw


def device_status(reset: bool = True) -> int:
    """The device status word (0 or DERA_ERR_TIMEOUT); synchronises the device."""
    st = ctypes.c_int(0)
    _check(load_library().dera_relpos_device_status(ctypes.byref(st), 1 if reset else 0))
    return st.value


def selftest_wait_timeout(budget_cycles: int = 1_000_000, stream=None) -> None:
    """Launch the bounded-wait self-test kernel (its wait can never succeed)."""
    dev = torch.device("cuda", torch.cuda.current_device())
    _check(load_library().dera_relpos_selftest_wait_timeout(int(budget_cycles), _stream(dev, stream)))
