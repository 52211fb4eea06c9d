"""GPU parity of the single-token kernel (T = 1 per call, Falcon-1, 1A, 2, 2A with d = 64) against the
fp64 oracle: fresh starts, continuations from a tail and a nonzero state, the state updated in place,
and a run of consecutive steps that must equal one call over the same tokens."""

import numpy as np
import pytest
import torch

from tests.gpu_util import check, rel_err, run_oracle, slice_inputs, tol
from weight_linear_attention_gb300 import falcon as F
from weight_linear_attention_gb300 import inputs as I

pytestmark = pytest.mark.gpu

NAMES = {1: "falcon1", 2: "falcon1a", 3: "falcon2", 4: "falcon2a"}


def _inputs(variant, dtype, seqlen, batch=3, seed=21):
    w = I.WORKLOADS[I.HEADLINE].with_(variant=NAMES[variant], dtype=dtype, nonzero_s0=True, heads=5)
    return w, I.make_inputs(w, seed=seed, seqlen=seqlen, batch=batch)


def _check(name, got, ref, dtype):
    check(name, got, ref, dtype)


def _step(variant, inp, t, dims_pos, S, tail, dt, inplace=False):
    """One falcon_fwd call on token t; returns (out, S_final, tail_out) on the device."""
    B, H, _, dk = inp["q"].shape
    x = {n: inp[n][:, :, t:t + 1].contiguous().cuda() for n in ("q", "k", "v", "beta", "lam")}
    out = torch.empty_like(x["v"])
    S_final = S if inplace else torch.empty(B, H, dk, dk, dtype=torch.float32, device="cuda")
    tail_out = torch.empty(B * H * dk, dtype=dt, device="cuda")
    d = F.make_dims(B, H, 1, dk, dk, dtype=F.FALCON_BF16 if dt == torch.bfloat16 else F.FALCON_F32, pos=dims_pos)
    assert F.falcon_kernel_for(variant, d, 64) == 4
    st = F.falcon_fwd(variant, x["q"], x["k"], x["v"], x["beta"], x["lam"], S, tail, out, S_final, tail_out, d, 64)
    assert st == F.FALCON_OK
    return out, S_final, tail_out


@pytest.mark.parametrize("variant", [1, 2, 3, 4])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_single_step_fresh_and_continued(variant, dtype):
    w, inp = _inputs(variant, dtype, seqlen=40)
    dt = w.torch_dtype
    S0 = inp["S0"]
    # fresh start (pos = 0, no tail): x_1 = 0, so the state is unchanged and o = S0^T q
    out, S1, t1 = _step(variant, inp, 0, 0, S0.cuda(), None, dt)
    torch.cuda.synchronize()
    ro, rS, rt = run_oracle(variant, slice_inputs(inp, 0, 1), S0=S0)
    _check("out", out.cpu(), ro, dt)
    _check("S", S1.cpu(), rS, dt)
    np.testing.assert_array_equal(t1.view(3, 5, 1, 64).double().cpu().numpy(), rt[0])
    # continuation at pos = 37 from the oracle's own state and tail after 37 tokens
    po, pS, pt = run_oracle(variant, slice_inputs(inp, 0, 37), S0=S0)
    S37 = torch.from_numpy(pS).float()
    tail = torch.from_numpy(pt[0]).to(dt).reshape(-1)
    out, S38, _ = _step(variant, inp, 37, 37, S37.cuda(), tail.cuda(), dt)
    torch.cuda.synchronize()
    ro, rS, _ = run_oracle(variant, slice_inputs(inp, 37, 38), S0=S37.double(), tail=(pt[0], pt[1]), pos=37)
    _check("out", out.cpu(), ro, dt)
    _check("S", S38.cpu(), rS, dt)
    assert F.falcon_device_status() == F.FALCON_OK


@pytest.mark.parametrize("variant", [1, 2, 3, 4])
def test_consecutive_steps_in_place_match_one_call(variant):
    """24 single-token calls, the state updated in place and the tail carried, equal the oracle over the
    24 tokens (the decode loop of a server)."""
    w, inp = _inputs(variant, "bf16", seqlen=24, batch=2)
    dt = w.torch_dtype
    S = inp["S0"].cuda().contiguous()
    tail, outs = None, []
    for t in range(24):
        o, S, tail_out = _step(variant, inp, t, t, S, tail, dt, inplace=True)
        outs.append(o)
        tail = tail_out
    torch.cuda.synchronize()
    assert F.falcon_device_status() == F.FALCON_OK
    ro, rS, _ = run_oracle(variant, inp, S0=inp["S0"])
    _check("out", torch.cat([o.cpu() for o in outs], dim=2), ro, dt)
    _check("S", S.cpu(), rS, dt)


def test_clamp_stress_single_token():
    """beta = 1.5, lambda = 1000: alpha = 1 - eps_gamma, gamma = eps_gamma."""
    w, inp = _inputs(1, "f32", seqlen=3, batch=1)
    inp["beta"] = torch.full_like(inp["beta"], 1.5)
    inp["lam"] = torch.full_like(inp["lam"], 1000.0)
    po, pS, pt = run_oracle(1, slice_inputs(inp, 0, 2), S0=inp["S0"])
    S2 = torch.from_numpy(pS).float()
    tail = torch.from_numpy(pt[0]).float().reshape(-1)
    out, S3, _ = _step(1, inp, 2, 2, S2.cuda(), tail.cuda(), torch.float32)
    torch.cuda.synchronize()
    ro, rS, _ = run_oracle(1, slice_inputs(inp, 2, 3), S0=S2.double(), tail=(pt[0], pt[1]), pos=2)
    _check("out", out.cpu(), ro, torch.float32)
    _check("S", S3.cpu(), rS, torch.float32)
