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


def bf16_round(x):
    """Round fp64 values to the nearest bf16 (ties to even), returned as fp64."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64)).to(torch.float32).to(torch.bfloat16)
    return t.double().numpy()


def bf16_spacing(x):
    """Distance from a bf16 value to the next one away from zero: 2^(e-7) for |x| in [2^e, 2^(e+1))."""
    return 2.0 * bf16_half_ulp(x)


def rounded_check(gpu, ref, bound=TOL_BF16):
    """The second bf16 check, with no allowance subtracted: every output against the oracle's output
    rounded to bf16, max|gpu - bf16(ref)| / RMS(ref) <= bound, over the outputs whose bf16 spacing is
    within the bound (there a correctly rounded result one spacing off, from a tiny computation error
    near a rounding boundary, still meets it; beyond it no computation but the exact one could); and
    RMS(gpu - ref) / RMS(ref) <= bound over all outputs. Returns (max error, share of outputs left
    out, RMS error)."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0, 0.0, 0.0
    rms = np.sqrt(np.mean(ref * ref))
    if rms == 0:
        return float(np.abs(gpu - ref).max()), 0.0, 0.0
    rr = bf16_round(ref)
    keep = bf16_spacing(rr) <= bound * rms
    err = float(np.abs(gpu - rr)[keep].max() / rms) if keep.any() else 0.0
    rms_err = float(np.sqrt(np.mean((gpu - ref) ** 2)) / rms)
    return err, float(1.0 - keep.mean()), rms_err


def tol(dtype) -> float:
    return TOL_F32 if dtype == torch.float32 else TOL_BF16


def check(name, gpu, ref, dtype, bound=None):
    """Parity of one output tensor against the oracle. fp32: max|gpu - ref| / max|ref|. bf16: both
    the bound with each output's rounding half-ulp excluded and, with no allowance, the bound against
    the oracle rounded to bf16 (rounded_check). Prints the figures; returns the first."""
    quant = hasattr(gpu, "dtype") and gpu.dtype == torch.bfloat16
    g = gpu.float().numpy() if hasattr(gpu, "numpy") else np.asarray(gpu)
    e = rel_err(g, ref, dtype, quantized_bf16=quant)
    raw = rel_err(g, ref, dtype)
    b = tol(dtype) if bound is None else bound
    msg = f"PARITY {name}: err {e:.3e} (raw {raw:.3e}) bound {b:.1e}"
    ok = np.isfinite(e) and e <= b
    if quant:
        e2, out, rms = rounded_check(g, ref, b)
        msg += f"; vs bf16(ref) {e2:.3e} ({100 * out:.3f}% of outputs beyond the bf16 spacing bound), rms {rms:.3e}"
        ok = ok and e2 <= b and rms <= b
    print(msg)
    assert ok, msg
    return e


def run_gpu(variant, inp, *, pos=0, window=1, chunk=64, S0=None, tail=None, eps=1e-6, eps_gamma=1e-6,
            dev="cuda", split=True):
    """inp: dict of CPU tensors q,k,v,beta,lam. Returns CPU tensors (out, S_final, tail_flat).
    split=True passes a workspace whenever a path uses one (the scan path); False runs without."""
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
