"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle, element by element.

Tolerances (per output tensor, out and S_final separately):
  fp32 inputs: max|gpu - ref| / max|ref| <= 1e-4
  bf16 inputs: max|gpu - ref| / RMS(ref) <= 2e-2
The oracle always runs on its own outputs (its own S_final and tail for a second
segment); no oracle input comes from the GPU.
"""

import numpy as np
import pytest
import torch

from tests.gpu_util import check, run_gpu, run_oracle, slice_inputs
from weight_linear_attention_gb300 import falcon as F
from weight_linear_attention_gb300 import inputs as I

pytestmark = pytest.mark.gpu

F1, F1A, F2, F3 = 1, 2, 3, 5
HEAD = I.HEADLINE


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weight_linear_attention_gb300 import build

    build.build()
    F.load()


def _check(name, gpu, ref, dtype, bound=None):
    return check(name, gpu, ref, dtype, bound)


def _parity(w: I.Workload, inp, *, chunk=None, S0=None, name=""):
    """GPU against the oracle on `inp`; a workload that starts after pos0 tokens starts from its drawn
    state and tail."""
    chunk = chunk or w.chunk
    pos, tail0, rtail0 = 0, None, None
    if w.pos0 > 0 and inp.get("tail") is not None:
        B, H, _, dk = inp["q"].shape
        pos, tail0 = w.pos0, inp["tail"][: B * H * dk]
        rtail0 = (tail0.view(B, H, 1, dk).double().numpy(), np.zeros((B, H, 0, inp["v"].shape[-1])))
        if S0 is None and inp.get("S0") is not None:
            S0 = inp["S0"][:B]
    out, S, tail = run_gpu(w.variant_id, inp, window=w.window, chunk=chunk, S0=S0, tail=tail0, pos=pos, eps=w.eps,
                           eps_gamma=w.eps_gamma)
    r_out, r_S, r_tail = run_oracle(w.variant_id, inp, window=w.window, S0=S0, tail=rtail0, pos=pos, eps=w.eps,
                                    eps_gamma=w.eps_gamma)
    _check(f"{name} out", out, r_out, w.torch_dtype)
    _check(f"{name} S_final", S, r_S, torch.float32 if w.dtype == "f32" else w.torch_dtype)
    B, H, T, dk = inp["q"].shape
    tk, tv = F.split_tail(tail, B, H, w.window, dk, inp["v"].shape[-1])
    np.testing.assert_array_equal(tk.double().numpy(), r_tail[0])
    np.testing.assert_array_equal(tv.double().numpy(), r_tail[1])


# ------------------------------------------------------------------ the five workloads

@pytest.mark.parametrize("wname", list(I.WORKLOADS))
def test_workload_reduced(wname):
    """Each workload's distributions at a size spanning several chunks plus a ragged tail."""
    w = I.WORKLOADS[wname]
    T = 3 * w.chunk + 7
    inp = I.make_inputs(w, seed=1, seqlen=T, batch=1)
    _parity(w, inp, name=wname)


@pytest.mark.parametrize("wname", [n for n in I.WORKLOADS if I.WORKLOADS[n].segments == 1])
def test_workload_full_size(wname):
    """Full workload size, same launch configuration as the benchmark."""
    w = I.WORKLOADS[wname]
    inp = I.make_inputs(w, seed=0)
    _parity(w, inp, name=wname)


@pytest.mark.parametrize("wname", ["f3w4_b2h12t16384_bf16", "f3aw4_b2h12t16384_bf16"])
def test_falcon3_two_segments_full_size(wname):
    """Falcon-3 / 3A, window 4, 2 x 12 x 16384 run as two 8192-token segments carrying S and the tail
    (the launch configuration the benchmark times)."""
    w = I.WORKLOADS[wname]
    V = w.variant_id
    inp = I.make_inputs(w, seed=0)
    Ts = w.seqlen
    a, b = slice_inputs(inp, 0, Ts), slice_inputs(inp, Ts, 2 * Ts)
    o1, S1, t1 = run_gpu(V, a, window=4, chunk=w.chunk)
    S1d = S1.clone()
    o2, S2, t2 = run_gpu(V, b, window=4, chunk=w.chunk, pos=Ts, S0=S1d, tail=t1)
    ro1, rS1, rt1 = run_oracle(V, a, window=4)
    ro2, rS2, rt2 = run_oracle(V, b, window=4, pos=Ts, S0=rS1, tail=rt1)
    _check("seg1 out", o1, ro1, torch.bfloat16)
    _check("seg1 S", S1, rS1, torch.bfloat16)
    _check("seg2 out", o2, ro2, torch.bfloat16)
    _check("seg2 S", S2, rS2, torch.bfloat16)
    B, H = 2, 12
    tk, tv = F.split_tail(t2, B, H, 4, 64, 64)
    np.testing.assert_array_equal(tk.double().numpy(), rt2[0])
    np.testing.assert_array_equal(tv.double().numpy(), rt2[1])
    # and the oracle's own split equals its unsplit run (exact continuation)
    ro_full, rS_full, _ = run_oracle(V, inp, window=4)
    np.testing.assert_allclose(np.concatenate([ro1, ro2], axis=2), ro_full, rtol=0, atol=1e-9)
    np.testing.assert_allclose(rS2, rS_full, rtol=0, atol=1e-9)


# ------------------------------------------------------------------ edge cases

@pytest.mark.parametrize("variant", [F1, F1A, F2, F3])
@pytest.mark.parametrize("chunk", [16, 32, 64])
def test_chunk_size_invariance(variant, chunk):
    W = 4 if variant == F3 else 1
    if variant == F3 and chunk * W > 128:
        pytest.skip("chunk*window > 128 is unsupported")
    w = I.WORKLOADS[HEAD].with_(variant={1: "falcon1", 2: "falcon1a", 3: "falcon2", 5: "falcon3"}[variant],
                                window=W, chunk=chunk)
    inp = I.make_inputs(w, seed=2, seqlen=200, batch=1)
    _parity(w, inp, name=f"v{variant} C{chunk}")



@pytest.mark.parametrize("variant", [F1, F1A, F2, F3])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_nonzero_initial_state(variant, dtype):
    W = 3 if variant == F3 else 1
    name = {1: "falcon1", 2: "falcon1a", 3: "falcon2", 5: "falcon3"}[variant]
    w = I.WORKLOADS[HEAD].with_(variant=name, window=W, chunk=32, dtype=dtype, nonzero_s0=True)
    inp = I.make_inputs(w, seed=3, seqlen=150, batch=2)
    _parity(w, inp, S0=inp["S0"], name=f"v{variant} {dtype} S0")


@pytest.mark.parametrize("variant", [F1, F1A])
def test_S_final_may_alias_S0(variant):
    w = I.WORKLOADS[HEAD].with_(variant="falcon1" if variant == F1 else "falcon1a", nonzero_s0=True)
    inp = I.make_inputs(w, seed=4, seqlen=130, batch=2)
    dev = {n: inp[n].cuda() for n in ("q", "k", "v", "beta", "lam")}
    S = inp["S0"].cuda().contiguous()
    out = torch.empty_like(dev["v"])
    d = F.make_dims(2, 12, 130, 64, 64, dtype=F.FALCON_BF16)
    st = F.falcon_fwd(variant, dev["q"], dev["k"], dev["v"], dev["beta"], dev["lam"], S, None, out, S, None, d, 64)
    assert st == 0
    torch.cuda.synchronize()
    r_out, r_S, _ = run_oracle(variant, inp, S0=inp["S0"])
    _check("out", out.cpu(), r_out, torch.bfloat16)
    _check("S", S.cpu(), r_S, torch.bfloat16)


@pytest.mark.parametrize("variant", [F1, F1A, F2, F3])
def test_clamp_stress(variant):
    """beta = 1.5, lambda = 1000: alpha hits 1 - eps_gamma on every step, gamma = eps_gamma."""
    W = 2 if variant == F3 else 1
    name = {1: "falcon1", 2: "falcon1a", 3: "falcon2", 5: "falcon3"}[variant]
    w = I.WORKLOADS[HEAD].with_(variant=name, window=W, chunk=32, lam_const=1000.0, lam_shift=None)
    inp = I.make_inputs(w, seed=5, seqlen=100, batch=1)
    inp["beta"] = torch.full_like(inp["beta"], 1.5)
    _parity(w, inp, name=f"clamp v{variant}")


def test_falcon2_mixed_decay_columns():
    """Falcon-2 with lambda = 1000 and per-column gains alternating 1.5 (clamped: strong decay) and 1e-3
    (weak decay): in one chunk some columns take the factored exponentials, the others do not."""
    w = I.WORKLOADS[HEAD].with_(variant="falcon2", chunk=64, lam_const=1000.0, lam_shift=None)
    inp = I.make_inputs(w, seed=11, seqlen=200, batch=1)
    b = torch.full_like(inp["beta"], 1e-3)
    b[..., 0::2] = 1.5
    inp["beta"] = b
    _parity(w, inp, name="falcon2 mixed columns")


@pytest.mark.parametrize("variant", [F1, F1A, F2, F3])
def test_zero_keys_with_zero_denominator(variant):
    """lambda = eps = 0 and some all-zero keys: eta = 0 there (no NaN)."""
    W = 2 if variant == F3 else 1
    name = {1: "falcon1", 2: "falcon1a", 3: "falcon2", 5: "falcon3"}[variant]
    w = I.WORKLOADS[HEAD].with_(variant=name, window=W, chunk=16, lam_const=0.0, lam_shift=None, dtype="f32",
                                eps=0.0)
    inp = I.make_inputs(w, seed=6, seqlen=70, batch=1)
    inp["k"][:, :, 10:14] = 0.0
    inp["k"][:, :, 40] = 0.0
    _parity(w, inp, name=f"zero-key v{variant}")


@pytest.mark.parametrize("T", [0, 1, 2, 63, 64, 65, 129])
def test_ragged_and_tiny_lengths(T):
    w = I.WORKLOADS[HEAD]
    inp = I.make_inputs(w, seed=7, seqlen=max(T, 1), batch=1)
    if T == 0:
        inp = slice_inputs(inp, 0, 0)
    _parity(w, inp, name=f"T={T}")


@pytest.mark.parametrize("variant,W,split", [(F1, 1, 1), (F1, 1, 100), (F1A, 1, 64), (F2, 1, 37),
                                             (F3, 4, 2), (F3, 4, 3), (F3, 4, 50), (F3, 2, 64)])
def test_segment_continuation(variant, W, split):
    """Two calls carrying S_final and the tail equal one call (and the oracle on the same split)."""
    name = {1: "falcon1", 2: "falcon1a", 3: "falcon2", 5: "falcon3"}[variant]
    w = I.WORKLOADS[HEAD].with_(variant=name, window=W, chunk=32)
    T = 160
    inp = I.make_inputs(w, seed=8, seqlen=T, batch=1)
    a, b = slice_inputs(inp, 0, split), slice_inputs(inp, split, T)
    o1, S1, t1 = run_gpu(variant, a, window=W, chunk=32)
    o2, S2, t2 = run_gpu(variant, b, window=W, chunk=32, pos=split, S0=S1, tail=t1)
    ro, rS, rt = run_oracle(variant, inp, window=W)
    _check("out", torch.cat([o1, o2], dim=2), ro, torch.bfloat16)
    _check("S", S2, rS, torch.bfloat16)
    tk, tv = F.split_tail(t2, 1, 12, W, 64, 64)
    np.testing.assert_array_equal(tk.double().numpy(), rt[0])
    np.testing.assert_array_equal(tv.double().numpy(), rt[1])


@pytest.mark.parametrize("dk,dv", [(16, 16), (32, 32), (128, 128), (64, 32), (32, 128)])
@pytest.mark.parametrize("variant", [F1, F2, F3])
def test_other_head_sizes(dk, dv, variant):
    W = 2 if variant == F3 else 1
    name = {1: "falcon1", 2: "falcon1a", 3: "falcon2", 5: "falcon3"}[variant]
    w = I.WORKLOADS[HEAD].with_(variant=name, window=W, chunk=32, dk=dk, dv=dv, heads=3)
    inp = I.make_inputs(w, seed=9, seqlen=100, batch=2)
    _parity(w, inp, name=f"dk{dk} dv{dv} v{variant}")


@pytest.mark.parametrize("variant", [F1, F1A, F2, F3])
def test_fp32_inputs_tight_tolerance(variant):
    W = 3 if variant == F3 else 1
    name = {1: "falcon1", 2: "falcon1a", 3: "falcon2", 5: "falcon3"}[variant]
    w = I.WORKLOADS["f1_tiny_fp32"].with_(variant=name, window=W, heads=4)
    inp = I.make_inputs(w, seed=10, seqlen=90, batch=2)
    _parity(w, inp, name=f"fp32 v{variant}")


def test_rejects_bad_call_without_touching_outputs():
    w = I.WORKLOADS[HEAD]
    inp = I.make_inputs(w, seed=11, seqlen=64, batch=1)
    dev = {n: inp[n].cuda() for n in ("q", "k", "v", "beta", "lam")}
    out = torch.full_like(dev["v"], 7.0)
    d = F.make_dims(1, 12, 64, 64, 64, dtype=F.FALCON_BF16, pos=5)  # pos > 0 but no tail
    st = F.falcon_fwd(F1, dev["q"], dev["k"], dev["v"], dev["beta"], dev["lam"], None, None, out, None, None, d, 64)
    assert st == F.FALCON_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)


# ------------------------------------------------------------------ inner-product variants 2A and 3A

F2A, F3A = 4, 6
_IP = {F2A: "falcon2a", F3A: "falcon3a"}


@pytest.mark.parametrize("variant,W", [(F2A, 1), (F3A, 2), (F3A, 4)])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("chunk", [16, 32])
def test_inner_product_variants(variant, W, dtype, chunk):
    """Falcon-2A and 3A from a nonzero state, several chunks and a ragged tail."""
    w = I.WORKLOADS[HEAD].with_(variant=_IP[variant], window=W, chunk=chunk, dtype=dtype, nonzero_s0=True,
                                heads=4)
    inp = I.make_inputs(w, seed=31, seqlen=3 * chunk + 11, batch=2)
    _parity(w, inp, S0=inp["S0"], name=f"v{variant} W{W} {dtype} C{chunk}")


@pytest.mark.parametrize("variant,W", [(F2A, 1), (F3A, 3)])
def test_inner_product_clamp_stress(variant, W):
    """beta = 1.5, lambda = 1000: alpha = 1 - eps_gamma on every step (strong decay in every chunk)."""
    w = I.WORKLOADS[HEAD].with_(variant=_IP[variant], window=W, chunk=32, lam_const=1000.0, lam_shift=None)
    inp = I.make_inputs(w, seed=32, seqlen=100, batch=1)
    inp["beta"] = torch.full_like(inp["beta"], 1.5)
    _parity(w, inp, name=f"clamp v{variant}")


@pytest.mark.parametrize("variant,W,split", [(F2A, 1, 37), (F3A, 4, 2), (F3A, 3, 50)])
def test_inner_product_continuation(variant, W, split):
    """Two calls carrying S_final and the tail equal the oracle over the whole sequence."""
    w = I.WORKLOADS[HEAD].with_(variant=_IP[variant], window=W, chunk=32)
    T = 140
    inp = I.make_inputs(w, seed=33, seqlen=T, batch=1)
    a, b = slice_inputs(inp, 0, split), slice_inputs(inp, split, T)
    o1, S1, t1 = run_gpu(variant, a, window=W, chunk=32)
    o2, S2, t2 = run_gpu(variant, b, window=W, chunk=32, pos=split, S0=S1, tail=t1)
    ro, rS, rt = run_oracle(variant, inp, window=W)
    _check("out", torch.cat([o1, o2], dim=2), ro, torch.bfloat16)
    _check("S", S2, rS, torch.bfloat16)
    tk, tv = F.split_tail(t2, 1, 12, W, 64, 64)
    np.testing.assert_array_equal(tk.double().numpy(), rt[0])
    np.testing.assert_array_equal(tv.double().numpy(), rt[1])


@pytest.mark.parametrize("variant", [F2A, F3A])
@pytest.mark.parametrize("dk,dv", [(32, 32), (128, 64), (16, 128)])
def test_inner_product_head_sizes(variant, dk, dv):
    W = 2 if variant == F3A else 1
    w = I.WORKLOADS[HEAD].with_(variant=_IP[variant], window=W, chunk=32, dk=dk, dv=dv, heads=3)
    inp = I.make_inputs(w, seed=34, seqlen=90, batch=2)
    _parity(w, inp, name=f"dk{dk} dv{dv} v{variant}")
