"""Seeded synthetic inputs for the Falcon forward pass.

This module draws random numbers and shapes them; it holds none of the
method's arithmetic, so the CUDA path's tests and the oracle's tests can both
use it. Workloads stand in for the pages' ~130M-parameter language models
(12 heads of width 64, sequence length 1,024 and longer; "Fast Weight Attention
for Continual Learning", paperlayer summary §5 and agihunt explainer "Results"):
no dataset or trained weight is available, so inputs are drawn, not read.

Recipe (every workload, seed 0 unless a caller passes another):
  generator = torch.Generator("cpu").manual_seed(seed); draws in this order,
  each N(0, 1) in fp32 of the full tensor shape:
    q [B,H,T,dk], k [B,H,T,dk], v [B,H,T,dv],
    beta logits [B,H,T] (Falcon-2, 2A: [B,H,T,dv]), lambda logits [B,H,T],
    then S0 [B,H,dk,dv] only when the workload asks for a nonzero initial state.
  q and k: RMSNorm over the feature axis (no gain, eps 1e-6; the pages' blocks
  use QK-RMSNorm upstream of the fast-memory update), then cast to the dtype.
  v: cast to the dtype directly. beta = sigmoid(logit); lambda = sigmoid(logit +
  shift) or a constant. beta and lambda stay fp32. S0 = N(0,1)/sqrt(dk) in fp32,
  so that the first reads S0^T q have the values' unit scale.
  A workload that starts after pos0 > 0 earlier tokens (window 1) also draws, last, the pending key
  k_pos0 [B,H,1,dk] (RMS-normed like k), which is its tail.
"""

from __future__ import annotations

from dataclasses import dataclass, field, replace

import torch

VARIANT_IDS = {"falcon1": 1, "falcon1a": 2, "falcon2": 3, "falcon2a": 4, "falcon3": 5, "falcon3a": 6}


@dataclass(frozen=True)
class Workload:
    name: str
    variant: str          # falcon1 | falcon1a | falcon2 | falcon2a | falcon3 | falcon3a
    batch: int
    heads: int
    seqlen: int           # tokens per call (per segment for segmented workloads)
    dk: int
    dv: int
    dtype: str            # "f32" | "bf16"
    chunk: int
    window: int = 1
    lam_shift: float | None = None   # lambda = sigmoid(N(0,1) + shift)
    lam_const: float | None = None   # lambda = constant
    beta_scale: float = 1.0          # beta = beta_scale * sigmoid(N(0,1))
    eps: float = 1e-6
    eps_gamma: float = 1e-6
    segments: int = 1                # the sequence is `segments` calls of `seqlen` tokens
    nonzero_s0: bool = False
    pos0: int = 0                    # tokens consumed before the first call (needs a tail; window 1)
    backward: bool = False           # a backward pass (falcon_bwd) rather than a forward one
    extra: dict = field(default_factory=dict)

    @property
    def variant_id(self) -> int:
        return VARIANT_IDS[self.variant]

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def total_tokens(self) -> int:
        return self.batch * self.seqlen * self.segments

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five workloads: (1) tiny fp32 Falcon-1; (2) Falcon-1 at the 130M shape;
# (3) Falcon-1A at that shape with stronger ridge; (4) Falcon-2 with per-channel
# gains at length 2048; (5) Falcon-3 window 4 at length 16384 as two segments.
WORKLOADS = {
    "f1_tiny_fp32": Workload("f1_tiny_fp32", "falcon1", 1, 2, 64, 16, 16, "f32", 16, lam_const=0.01),
    "f1_b8h12t1024_bf16": Workload("f1_b8h12t1024_bf16", "falcon1", 8, 12, 1024, 64, 64, "bf16", 64,
                                   lam_shift=-4.0),
    "f1a_b8h12t1024_bf16": Workload("f1a_b8h12t1024_bf16", "falcon1a", 8, 12, 1024, 64, 64, "bf16", 64,
                                    lam_shift=-3.0),
    "f2_b8h12t2048_bf16": Workload("f2_b8h12t2048_bf16", "falcon2", 8, 12, 2048, 64, 64, "bf16", 64,
                                   lam_const=0.01),
    "f3w4_b2h12t16384_bf16": Workload("f3w4_b2h12t16384_bf16", "falcon3", 2, 12, 8192, 64, 64, "bf16", 32,
                                      window=4, lam_shift=-2.0, segments=2),
    # the inner-product variants at the Falcon-2 and Falcon-3 shapes
    "f2a_b8h12t2048_bf16": Workload("f2a_b8h12t2048_bf16", "falcon2a", 8, 12, 2048, 64, 64, "bf16", 64,
                                    lam_const=0.01),
    "f3aw4_b2h12t16384_bf16": Workload("f3aw4_b2h12t16384_bf16", "falcon3a", 2, 12, 8192, 64, 64, "bf16", 32,
                                       window=4, lam_shift=-2.0, segments=2),
    # the backward pass of Falcon-1 and 1A at the 130M shape (output and final-state adjoints drawn too)
    "f1_bwd_b8h12t1024_bf16": Workload("f1_bwd_b8h12t1024_bf16", "falcon1", 8, 12, 1024, 64, 64, "bf16", 64,
                                       lam_shift=-4.0, backward=True),
    "f1a_bwd_b8h12t1024_bf16": Workload("f1a_bwd_b8h12t1024_bf16", "falcon1a", 8, 12, 1024, 64, 64, "bf16", 64,
                                        lam_shift=-3.0, backward=True),
    # one decoding step of 256 sequences (12 heads of 64) after 1024 tokens: the recurrent form
    "f1_decode_b256h12_bf16": Workload("f1_decode_b256h12_bf16", "falcon1", 256, 12, 1, 64, 64, "bf16", 64,
                                       lam_shift=-4.0, nonzero_s0=True, pos0=1024),
}

HEADLINE = "f1_b8h12t1024_bf16"


def make_adjoints(w: Workload, seed: int = 0, seqlen: int | None = None, batch: int | None = None) -> dict:
    """Adjoints for a backward pass: dout [B,H,T,dv] in the workload dtype (unit normal) and
    dS_final [B,H,dk,dv] fp32 (normal, scaled by 1/sqrt(dk) like S0). Drawn from their own seed stream."""
    B = w.batch if batch is None else batch
    T = (w.seqlen * w.segments) if seqlen is None else seqlen
    g = torch.Generator("cpu").manual_seed(1_000_003 + seed)
    dout = torch.randn(B, w.heads, T, w.dv, generator=g).to(w.torch_dtype)
    dS = (torch.randn(B, w.heads, w.dk, w.dv, generator=g) / w.dk ** 0.5).float()
    return {"dout": dout, "dS_final": dS}


def _rmsnorm(x: torch.Tensor, eps: float = 1e-6) -> torch.Tensor:
    return x * torch.rsqrt(x.pow(2).mean(dim=-1, keepdim=True) + eps)


def make_inputs(w: Workload, seed: int = 0, seqlen: int | None = None, batch: int | None = None) -> dict:
    """Draw one workload's inputs on the CPU.

    The full sequence (segments * seqlen tokens) is drawn at once; a segmented
    workload is split by the caller. ``seqlen``/``batch`` override the shape
    (for reduced parity cases that keep the workload's distributions).
    """
    B = w.batch if batch is None else batch
    T = (w.seqlen * w.segments) if seqlen is None else seqlen
    H, dk, dv = w.heads, w.dk, w.dv
    g = torch.Generator("cpu").manual_seed(seed)
    q = torch.randn(B, H, T, dk, generator=g)
    k = torch.randn(B, H, T, dk, generator=g)
    v = torch.randn(B, H, T, dv, generator=g)
    bshape = (B, H, T, dv) if w.variant in ("falcon2", "falcon2a") else (B, H, T)
    beta_logit = torch.randn(*bshape, generator=g)
    lam_logit = torch.randn(B, H, T, generator=g)
    S0 = torch.randn(B, H, dk, dv, generator=g) / dk ** 0.5 if w.nonzero_s0 else None
    assert w.pos0 == 0 or w.window == 1, "a starting tail is drawn for window 1 only"
    tail_k = torch.randn(B, H, 1, dk, generator=g) if w.pos0 > 0 else None
    dt = w.torch_dtype
    out = {
        "q": _rmsnorm(q).to(dt),
        "k": _rmsnorm(k).to(dt),
        "v": v.to(dt),
        "beta": (w.beta_scale * torch.sigmoid(beta_logit)).float().contiguous(),
        "lam": (torch.full((B, H, T), float(w.lam_const)) if w.lam_const is not None
                else torch.sigmoid(lam_logit + float(w.lam_shift))).float().contiguous(),
        "S0": S0,
        "tail": _rmsnorm(tail_k).to(dt).reshape(-1).contiguous() if tail_k is not None else None,
    }
    return out
