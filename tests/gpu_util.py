"""Helpers for the GPU parity tests: run the CUDA path and the oracle on the same inputs."""

from __future__ import annotations

import numpy as np
import torch

import oracle
from weight_linear_attention_gb300 import falcon as F

TOL_F32 = 1e-4   # max|gpu - ref| / max|ref|, fp32 inputs
TOL_BF16 = 2e-2  # max|gpu - ref| / RMS(ref), bf16 inputs with fp32 state


def bf16_half_ulp(x):
    """Largest error of rounding x to the nearest bf16 (8 significant bits): 2^(e-8), x in [2^e, 2^(e+1))."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(e - 8), 0.0)


def rel_err(gpu, ref, dtype, quantized_bf16=False) -> float:
    """fp32: max|gpu-ref| / max|ref|.  bf16: max|gpu-ref| / RMS(ref); when the GPU value is
    itself a bf16 output, each element's final-rounding half-ulp is subtracted first, so the
    bound measures the computation and not the output format."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    diff = np.abs(gpu - ref)
    if quantized_bf16:
        diff = np.maximum(diff - bf16_half_ulp(ref), 0.0)
    diff = diff.max()
    if dtype == torch.float32:
        den = np.abs(ref).max()
    else:
        den = np.sqrt(np.mean(ref * ref))
    if den == 0:
        return float(diff)
    return float(diff / den)


def tol(dtype) -> float:
    return TOL_F32 if dtype == torch.float32 else TOL_BF16


def run_gpu(variant, inp, *, pos=0, window=1, chunk=64, S0=None, tail=None, eps=1e-6, eps_gamma=1e-6,
            dev="cuda", split=True):
    """inp: dict of CPU tensors q,k,v,beta,lam. Returns CPU tensors (out, S_final, tail_flat).
    split=True passes a workspace (the split path where one exists); False runs the single-pass kernels."""
    g = {n: inp[n].to(dev).contiguous() for n in ("q", "k", "v", "beta", "lam")}
    S0d = S0.to(dev).contiguous() if S0 is not None else None
    taild = tail.to(dev).contiguous() if tail is not None else None
    out, S, t = F.forward(variant, g["q"], g["k"], g["v"], g["beta"], g["lam"], S0d, taild, pos=pos,
                          window=window, chunk=chunk, eps=eps, eps_gamma=eps_gamma, split=split)
    torch.cuda.synchronize()
    assert F.falcon_device_status() == F.FALCON_OK
    return out.cpu(), S.cpu(), t.cpu()


def run_oracle(variant, inp, *, pos=0, window=1, S0=None, tail=None, eps=1e-6, eps_gamma=1e-6):
    """tail: (keys, vals) fp64 arrays from an earlier oracle call, or None."""
    return oracle.falcon_ref_fwd(variant, inp["q"], inp["k"], inp["v"], inp["beta"], inp["lam"], S0, tail,
                                 pos=pos, window=window, eps=eps, eps_gamma=eps_gamma)


def slice_inputs(inp, t0, t1):
    return {n: inp[n][:, :, t0:t1].contiguous() for n in ("q", "k", "v", "beta", "lam")}
