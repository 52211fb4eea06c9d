"""Python binding of the C ABI in include/falcon.h (ctypes; argument marshalling only).

Every function here forwards to ``_build/libfalcon.so``; all arithmetic runs in
the library's CUDA kernels. There is no fallback: if the library has not been
built (``weight_linear_attention_gb300.build.build()``) or cannot be loaded,
every call raises.

PyTorch is used only to hand over device pointers and the current CUDA stream.
"""

from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

FALCON_1, FALCON_1A, FALCON_2, FALCON_2A, FALCON_3, FALCON_3A = 1, 2, 3, 4, 5, 6
FALCON_F32, FALCON_BF16 = 0, 1
FALCON_OK = 0
FALCON_ERR_INVALID_ARG = 1
FALCON_ERR_UNSUPPORTED = 2
FALCON_ERR_MISALIGNED = 3
FALCON_ERR_CUDA = 4
FALCON_ERR_DEVICE_TIMEOUT = 5

VARIANTS = {"falcon1": FALCON_1, "falcon1a": FALCON_1A, "falcon2": FALCON_2, "falcon2a": FALCON_2A,
            "falcon3": FALCON_3, "falcon3a": FALCON_3A}


class FalconDims(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int64),
        ("heads", ctypes.c_int64),
        ("seqlen", ctypes.c_int64),
        ("dk", ctypes.c_int64),
        ("dv", ctypes.c_int64),
        ("window", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("pos", ctypes.c_int64),
        ("eps", ctypes.c_float),
        ("eps_gamma", ctypes.c_float),
    ]


assert ctypes.sizeof(FalconDims) == 64

_lock = threading.Lock()
_lib = None

EXPORTED = ("falcon_fwd", "falcon_workspace_bytes", "falcon_fwd_static", "falcon_tail_bytes",
            "falcon_status_string", "falcon_device_status", "falcon_kernel_for", "falcon_abi_version",
            "falcon_bwd", "falcon_bwd_workspace_bytes")
STATIC_WORKSPACE_BYTES = 16 << 20


class FalconError(RuntimeError):
    def __init__(self, status: int, what: str = "falcon_fwd"):
        self.status = status
        super().__init__(f"{what} failed with status {status}: {status_string(status)}")


def lib_path() -> str:
    return _build.LIB


def load(path: str | None = None):
    """Load the C-ABI library (raises if it is missing)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or _build.LIB
        if not os.path.exists(p):
            raise RuntimeError(f"CUDA library not built: {p} (run weight_linear_attention_gb300.build.build())")
        lib = ctypes.CDLL(p)
        vp = ctypes.c_void_p
        lib.falcon_fwd.restype = ctypes.c_int
        lib.falcon_fwd.argtypes = [ctypes.c_int, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                   ctypes.POINTER(FalconDims), ctypes.c_int, vp, ctypes.c_size_t, vp]
        lib.falcon_fwd_static.restype = ctypes.c_int
        lib.falcon_fwd_static.argtypes = [ctypes.c_int, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                          ctypes.POINTER(FalconDims), ctypes.c_int, vp]
        lib.falcon_workspace_bytes.restype = ctypes.c_size_t
        lib.falcon_workspace_bytes.argtypes = [ctypes.c_int, ctypes.POINTER(FalconDims), ctypes.c_int]
        lib.falcon_tail_bytes.restype = ctypes.c_size_t
        lib.falcon_tail_bytes.argtypes = [ctypes.POINTER(FalconDims)]
        lib.falcon_status_string.restype = ctypes.c_char_p
        lib.falcon_status_string.argtypes = [ctypes.c_int]
        lib.falcon_device_status.restype = ctypes.c_int
        lib.falcon_device_status.argtypes = [vp]
        lib.falcon_kernel_for.restype = ctypes.c_int
        lib.falcon_kernel_for.argtypes = [ctypes.c_int, ctypes.POINTER(FalconDims), ctypes.c_int]
        lib.falcon_abi_version.restype = ctypes.c_int
        lib.falcon_abi_version.argtypes = []
        lib.falcon_bwd.restype = ctypes.c_int
        lib.falcon_bwd.argtypes = [ctypes.c_int] + [vp] * 16 + [ctypes.POINTER(FalconDims), ctypes.c_int, vp,
                                                                ctypes.c_size_t, vp]
        lib.falcon_bwd_workspace_bytes.restype = ctypes.c_size_t
        lib.falcon_bwd_workspace_bytes.argtypes = [ctypes.c_int, ctypes.POINTER(FalconDims), ctypes.c_int]
        if path is None:
            _lib = lib
        return lib


def make_dims(batch, heads, seqlen, dk, dv, *, window=1, dtype=FALCON_BF16, pos=0, eps=1e-6,
              eps_gamma=1e-6) -> FalconDims:
    return FalconDims(int(batch), int(heads), int(seqlen), int(dk), int(dv), int(window), int(dtype), int(pos),
                      float(eps), float(eps_gamma))


def status_string(status: int) -> str:
    return load().falcon_status_string(int(status)).decode()


def falcon_tail_bytes(dims: FalconDims) -> int:
    return int(load().falcon_tail_bytes(ctypes.byref(dims)))


def falcon_workspace_bytes(variant: int, dims: FalconDims, chunk: int) -> int:
    return int(load().falcon_workspace_bytes(int(variant), ctypes.byref(dims), int(chunk)))


def falcon_kernel_for(variant: int, dims: FalconDims, chunk: int) -> int:
    return int(load().falcon_kernel_for(int(variant), ctypes.byref(dims), int(chunk)))


def falcon_device_status(stream=None) -> int:
    return int(load().falcon_device_status(_stream_handle(stream)))


def falcon_abi_version() -> int:
    return int(load().falcon_abi_version())


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream_handle(stream):
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def falcon_fwd(variant, q, k, v, beta, lam, S0, tail, out, S_final, tail_out, dims: FalconDims, chunk: int,
               workspace=None, workspace_bytes=None, stream=None) -> int:
    """The C entry point with the same argument order; tensors or raw device pointers. Returns the status.

    ``workspace_bytes`` defaults to the size of a tensor workspace (0 for a raw pointer)."""
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None or isinstance(workspace, int) else \
            workspace.numel() * workspace.element_size()
    return int(load().falcon_fwd(int(variant), _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(lam), _ptr(S0),
                                 _ptr(tail), _ptr(out), _ptr(S_final), _ptr(tail_out), ctypes.byref(dims),
                                 int(chunk), _ptr(workspace), int(workspace_bytes), _stream_handle(stream)))


def falcon_fwd_static(variant, q, k, v, beta, lam, S0, tail, out, S_final, tail_out, dims: FalconDims, chunk: int,
                      stream=None) -> int:
    """The no-allocation C entry point (the library's own fixed scratch); returns the status."""
    return int(load().falcon_fwd_static(int(variant), _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(lam), _ptr(S0),
                                        _ptr(tail), _ptr(out), _ptr(S_final), _ptr(tail_out), ctypes.byref(dims),
                                        int(chunk), _stream_handle(stream)))


def falcon_bwd(variant, q, k, v, beta, lam, S0, tail, dout, dS_final, dq, dk, dv, dbeta, dlam, dS0, dtail,
               dims: FalconDims, chunk: int, workspace=None, workspace_bytes=None, stream=None) -> int:
    """The C entry point falcon_bwd with the same argument order; tensors or raw device pointers."""
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None or isinstance(workspace, int) else \
            workspace.numel() * workspace.element_size()
    return int(load().falcon_bwd(int(variant), _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(lam), _ptr(S0),
                                 _ptr(tail), _ptr(dout), _ptr(dS_final), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dbeta),
                                 _ptr(dlam), _ptr(dS0), _ptr(dtail), ctypes.byref(dims), int(chunk),
                                 _ptr(workspace), int(workspace_bytes), _stream_handle(stream)))


def falcon_bwd_workspace_bytes(variant: int, dims: FalconDims, chunk: int) -> int:
    return int(load().falcon_bwd_workspace_bytes(int(variant), ctypes.byref(dims), int(chunk)))


def backward(variant, q, k, v, beta, lam, dout, S0=None, dS_final=None, tail=None, *, pos=0, chunk=64, eps=1e-6,
             eps_gamma=1e-6, want_dS0=True, stream=None):
    """Allocate fp32 gradients and a workspace with torch on q's device and call falcon_bwd; raises
    FalconError on a nonzero status. Returns a dict dq, dk, dv, dbeta, dlam, dS0 (None unless
    want_dS0), dtail (None unless pos > 0)."""
    import torch

    if isinstance(variant, str):
        variant = VARIANTS[variant]
    B, H, T, dk_ = q.shape
    dv_ = v.shape[-1]
    dt = FALCON_BF16 if q.dtype == torch.bfloat16 else FALCON_F32
    dims = make_dims(B, H, T, dk_, dv_, dtype=dt, pos=pos, eps=eps, eps_gamma=eps_gamma)
    f32 = dict(dtype=torch.float32, device=q.device)
    g = {"dq": torch.empty((B, H, T, dk_), **f32), "dk": torch.empty((B, H, T, dk_), **f32),
         "dv": torch.empty((B, H, T, dv_), **f32), "dbeta": torch.empty((B, H, T), **f32),
         "dlam": torch.empty((B, H, T), **f32),
         "dS0": torch.empty((B, H, dk_, dv_), **f32) if want_dS0 else None,
         "dtail": torch.empty((B, H, dk_), **f32) if pos > 0 else None}
    n = falcon_bwd_workspace_bytes(variant, dims, chunk)
    ws = torch.empty(n, dtype=torch.uint8, device=q.device) if n > 0 else None
    st = falcon_bwd(variant, q, k, v, beta, lam, S0, tail, dout, dS_final, g["dq"], g["dk"], g["dv"], g["dbeta"],
                    g["dlam"], g["dS0"], g["dtail"], dims, chunk, ws, stream=stream)
    if st != FALCON_OK:
        raise FalconError(st, "falcon_bwd")
    return g


def workspace_for(variant, dims: FalconDims, chunk: int, device):
    """A workspace tensor sized for falcon_fwd's split path, or None when no path needs one."""
    import torch

    n = falcon_workspace_bytes(variant, dims, chunk)
    return torch.empty(n, dtype=torch.uint8, device=device) if n > 0 else None


def forward(variant, q, k, v, beta, lam, S0=None, tail=None, *, pos=0, window=1, chunk=64, eps=1e-6,
            eps_gamma=1e-6, want_state=True, want_tail=True, split=True, stream=None):
    """Allocate outputs with torch on q's device and call falcon_fwd; raises FalconError on a nonzero status.

    Returns (out, S_final or None, tail_out or None). tail/tail_out are flat byte-sized
    buffers in q's dtype, laid out per (b,h) as keys[window][dk] then vals[window-1][dv].
    ``split=True`` hands falcon_fwd a workspace whenever a path can use one; ``False`` runs the
    single-pass kernels.
    """
    import torch

    if isinstance(variant, str):
        variant = VARIANTS[variant]
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    dt = FALCON_BF16 if q.dtype == torch.bfloat16 else FALCON_F32
    dims = make_dims(B, H, T, dk, dv, window=window, dtype=dt, pos=pos, eps=eps, eps_gamma=eps_gamma)
    out = torch.empty((B, H, T, dv), dtype=q.dtype, device=q.device)
    S_final = torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device) if want_state else None
    tail_out = None
    if want_tail:
        n = falcon_tail_bytes(dims) // q.element_size()
        tail_out = torch.empty(n, dtype=q.dtype, device=q.device)
    ws = workspace_for(variant, dims, chunk, q.device) if split else None
    st = falcon_fwd(variant, q, k, v, beta, lam, S0, tail, out, S_final, tail_out, dims, chunk, ws, stream=stream)
    if st != FALCON_OK:
        raise FalconError(st)
    return out, S_final, tail_out


def split_tail(tail_flat, B, H, W, dk, dv):
    """View a flat tail buffer as (keys [B,H,W,dk], vals [B,H,W-1,dv])."""
    per = W * dk + (W - 1) * dv
    t = tail_flat.view(B, H, per)
    return t[..., : W * dk].reshape(B, H, W, dk), t[..., W * dk:].reshape(B, H, W - 1, dv)


def join_tail(keys, vals):
    """Pack (keys [B,H,W,dk], vals [B,H,W-1,dv]) into the flat tail layout."""
    import torch

    B, H = keys.shape[:2]
    return torch.cat([keys.reshape(B, H, -1), vals.reshape(B, H, -1)], dim=-1).reshape(-1).contiguous()
