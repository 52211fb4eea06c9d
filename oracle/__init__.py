"""CPU oracle for the Falcon fast-weight forward pass (fp64, token by token).

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package. The product path (the
CUDA library and its Python binding) never imports, links or runs it, and it
shares no code with that path.

The arithmetic lives in ``falcon_ref.c`` (plain C, fp64, no -ffast-math); this
module compiles it with gcc and marshals numpy arrays to it. Every input is
converted exactly to fp64 first, so bf16/fp32 input rounding is not counted as
an error of the path under test.

Every function here is pinned by ``tests/test_oracle.py`` against closed forms,
hand-worked examples, a library eigensolver, autograd gradient steps of the
stated objectives and a brute-force masked-parallel solve.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "falcon_ref.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libfalcon_ref.so")

FALCON_1, FALCON_1A, FALCON_2, FALCON_2A, FALCON_3, FALCON_3A = 1, 2, 3, 4, 5, 6

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile falcon_ref.c into a shared library (gcc, -O2, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", "-ffp-contract=off",
             "-o", tmp, _SRC, "-lpthread", "-lm"],
            check=True,
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            dp = ctypes.POINTER(ctypes.c_double)
            i64 = ctypes.c_int64
            lib.falcon_ref_fwd.restype = ctypes.c_int
            lib.falcon_ref_fwd.argtypes = [
                ctypes.c_int, i64, i64, i64, i64, i64, ctypes.c_int, i64,
                dp, dp, dp, dp, dp, dp, dp, dp,
                ctypes.c_double, ctypes.c_double,
                dp, dp, dp, dp, ctypes.c_int,
            ]
            lib.falcon_ref_lambda_max.restype = ctypes.c_double
            lib.falcon_ref_lambda_max.argtypes = [ctypes.c_int, dp]
            _lib = lib
    return _lib


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor: exact widening to fp64
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    if a is None:
        return ctypes.POINTER(ctypes.c_double)()
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def lambda_max(g) -> float:
    """Largest eigenvalue of a small symmetric matrix, by the oracle's Jacobi sweep."""
    g = _f64(g)
    n = g.shape[0]
    assert g.shape == (n, n)
    return float(_load().falcon_ref_lambda_max(n, _ptr(g)))


def falcon_ref_fwd(variant, q, k, v, beta, lam, S0=None, tail=None, *, pos=0, window=1,
                   eps=1e-6, eps_gamma=1e-6, nthreads=None):
    """Run the fp64 recurrence.

    q, k: [B,H,T,dk]; v: [B,H,T,dv]; beta: [B,H,T] (Falcon-2, 2A: [B,H,T,dv]);
    lam: [B,H,T]; S0: [B,H,dk,dv] or None; tail: (keys [B,H,W,dk] holding
    k_{pos-W+1..pos}, vals [B,H,W-1,dv] holding v_{pos-W+2..pos}) or None iff
    pos == 0. Returns (out [B,H,T,dv], S_final [B,H,dk,dv], (tail_keys, tail_vals))
    as fp64 numpy arrays, the tail describing position pos + T.
    """
    q, k, v, beta, lam, S0 = (_f64(a) for a in (q, k, v, beta, lam, S0))
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    W = int(window)
    tk = tv = None
    if tail is not None:
        tk, tv = _f64(tail[0]), _f64(tail[1])
        assert tk.shape == (B, H, W, dk), tk.shape
        assert tv.shape == (B, H, W - 1, dv), tv.shape
    assert k.shape == (B, H, T, dk) and v.shape == (B, H, T, dv)
    assert lam.shape == (B, H, T)
    if variant in (FALCON_2, FALCON_2A):
        assert beta.shape == (B, H, T, dv)
    else:
        assert beta.shape == (B, H, T)
    if S0 is not None:
        assert S0.shape == (B, H, dk, dv)
    out = np.zeros((B, H, T, dv))
    S = np.zeros((B, H, dk, dv))
    tko = np.zeros((B, H, W, dk))
    tvo = np.zeros((B, H, max(W - 1, 0), dv))
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    rc = _load().falcon_ref_fwd(
        int(variant), B, H, T, dk, dv, W, int(pos),
        _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(lam), _ptr(S0), _ptr(tk), _ptr(tv),
        float(eps), float(eps_gamma),
        _ptr(out), _ptr(S), _ptr(tko), _ptr(tvo), int(nthreads),
    )
    if rc != 0:
        raise ValueError(f"falcon_ref_fwd rejected its arguments (code {rc})")
    return out, S, (tko, tvo)
