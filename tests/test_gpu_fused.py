"""GPU parity of the fused tensor-core kernel (Falcon-1 / 1A, bf16, dk = dv = 64, chunk 64): one
persistent CTA per sequence, state on chip.

Every case runs through the C ABI and is compared with the fp64 oracle at the bf16 bound (both
checks of tests.gpu_util.check), covering the branches that kernel has: a nonzero and an aliased
initial state, the clamp (total log decay of a chunk below -30, so every factor is formed by its
own exp) and chunks where fast and exact exponential forms alternate, continuation from a tail at
every kind of split point, lengths around the chunk boundary, odd sequence counts, and the
headline shape.
"""

import numpy as np
import pytest
import torch

from tests.gpu_util import check, run_gpu, run_oracle, slice_inputs
from weight_linear_attention_gb300 import falcon as F
from weight_linear_attention_gb300 import inputs as I

pytestmark = pytest.mark.gpu

F1, F1A = 1, 2
HEAD = I.HEADLINE


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weight_linear_attention_gb300 import build

    build.build()
    F.load()


def _check(name, gpu, ref, bound=None):
    check(name, gpu, ref, torch.bfloat16, bound)


def _wl(variant, **kw):
    return I.WORKLOADS[HEAD].with_(variant="falcon1" if variant == F1 else "falcon1a", **kw)


def _fused(variant, inp, S0=None, pos=0, tail=None, eps_gamma=1e-6):
    dims = F.make_dims(*inp["q"].shape[:3], 64, 64, dtype=F.FALCON_BF16, pos=pos)
    T = inp["q"].shape[2]
    assert F.falcon_kernel_for(variant, dims, 64) == (4 if T == 1 else 6)
    assert F.falcon_workspace_bytes(variant, dims, 64) == 0
    return run_gpu(variant, inp, chunk=64, S0=S0, pos=pos, tail=tail, eps_gamma=eps_gamma)


@pytest.mark.parametrize("variant", [F1, F1A])
def test_nonzero_initial_state(variant):
    w = _wl(variant, nonzero_s0=True)
    inp = I.make_inputs(w, seed=21, seqlen=200, batch=2)
    out, S, _ = _fused(variant, inp, S0=inp["S0"])
    r_out, r_S, _ = run_oracle(variant, inp, S0=inp["S0"])
    _check(f"v{variant} S0 out", out, r_out)
    _check(f"v{variant} S0 S", S, r_S)


@pytest.mark.parametrize("variant", [F1, F1A])
def test_S_final_may_alias_S0(variant):
    w = _wl(variant, nonzero_s0=True)
    inp = I.make_inputs(w, seed=22, seqlen=130, batch=2)
    dev = {n: inp[n].cuda() for n in ("q", "k", "v", "beta", "lam")}
    S = inp["S0"].cuda().contiguous()
    out = torch.empty_like(dev["v"])
    d = F.make_dims(2, 12, 130, 64, 64, dtype=F.FALCON_BF16)
    st = F.falcon_fwd(variant, dev["q"], dev["k"], dev["v"], dev["beta"], dev["lam"], S, None, out, S, None, d, 64)
    assert st == 0
    torch.cuda.synchronize()
    assert F.falcon_device_status() == F.FALCON_OK
    r_out, r_S, _ = run_oracle(variant, inp, S0=inp["S0"])
    _check("alias out", out.cpu(), r_out)
    _check("alias S", S.cpu(), r_S)


@pytest.mark.parametrize("variant", [F1, F1A])
def test_clamp_stress(variant):
    """beta = 1.5, lambda = 1000: alpha = 1 - eps_gamma on every step, log decay ~ -13.8 per token."""
    w = _wl(variant, lam_const=1000.0, lam_shift=None)
    inp = I.make_inputs(w, seed=23, seqlen=150, batch=1)
    inp["beta"] = torch.full_like(inp["beta"], 1.5)
    out, S, _ = _fused(variant, inp)
    r_out, r_S, _ = run_oracle(variant, inp)
    _check(f"clamp v{variant} out", out, r_out)
    _check(f"clamp v{variant} S", S, r_S)


@pytest.mark.parametrize("variant", [F1, F1A])
def test_mixed_decay_chunks(variant):
    """Strong decay in some chunks only: the fast and the exact exp forms alternate across chunks."""
    w = _wl(variant)
    inp = I.make_inputs(w, seed=24, seqlen=256, batch=1)
    inp["lam"][:, :, 64:128] = 1000.0
    inp["lam"][:, :, 200:210] = 50.0
    out, S, _ = _fused(variant, inp)
    r_out, r_S, _ = run_oracle(variant, inp)
    _check(f"mixed v{variant} out", out, r_out)
    _check(f"mixed v{variant} S", S, r_S)


@pytest.mark.parametrize("variant,cut", [(F1, 1), (F1, 63), (F1, 64), (F1, 100), (F1A, 64), (F1A, 77)])
def test_segment_continuation(variant, cut):
    """Two calls carrying S_final and the tail (pos > 0: the first shifted key comes from the tail)."""
    w = _wl(variant)
    T = 200
    inp = I.make_inputs(w, seed=25, seqlen=T, batch=2)
    a, b = slice_inputs(inp, 0, cut), slice_inputs(inp, cut, T)
    o1, S1, t1 = run_gpu(variant, a, chunk=64)
    o2, S2, t2 = run_gpu(variant, b, chunk=64, pos=cut, S0=S1, tail=t1)
    ro, rS, rt = run_oracle(variant, inp)
    _check("cont out", torch.cat([o1, o2], dim=2), ro)
    _check("cont S", S2, rS)
    tk, tv = F.split_tail(t2, 2, 12, 1, 64, 64)
    np.testing.assert_array_equal(tk.double().numpy(), rt[0])


@pytest.mark.parametrize("T", [1, 2, 63, 64, 65, 127, 128, 129, 1000])
def test_lengths(T):
    w = I.WORKLOADS[HEAD]
    inp = I.make_inputs(w, seed=26, seqlen=T, batch=1)
    out, S, t = _fused(F1, inp)
    r_out, r_S, rt = run_oracle(F1, inp)
    _check(f"T={T} out", out, r_out)
    _check(f"T={T} S", S, r_S)
    np.testing.assert_array_equal(F.split_tail(t, 1, 12, 1, 64, 64)[0].double().numpy(), rt[0])


@pytest.mark.parametrize("variant", [F1, F1A])
def test_headline_shape_two_batch_rows(variant):
    """The headline shape's sequences (2 x 12 x 1024) against the oracle, every sequence compared."""
    w = _wl(variant)
    inp = I.make_inputs(w, seed=27, seqlen=1024, batch=2)
    r_out, r_S, _ = run_oracle(variant, inp)
    o, S, _ = _fused(variant, inp)
    _check("headline rows out", o, r_out)
    _check("headline rows S", S, r_S)


def test_rejected_call_leaves_outputs():
    w = I.WORKLOADS[HEAD]
    inp = I.make_inputs(w, seed=28, seqlen=64, batch=1)
    dev = {n: inp[n].cuda() for n in ("q", "k", "v", "beta", "lam")}
    out = torch.full_like(dev["v"], 7.0)
    d = F.make_dims(1, 12, 64, 64, 64, dtype=F.FALCON_BF16)
    # S_final over lambda: rejected before any launch
    st = F.falcon_fwd(F1, dev["q"], dev["k"], dev["v"], dev["beta"], dev["lam"], None, None, out,
                      dev["lam"].data_ptr(), None, d, 64)
    assert st == F.FALCON_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)


@pytest.mark.parametrize("variant", [F1, F1A])
def test_odd_sequence_count_with_state_and_tail(variant):
    """2 x 19 sequences (not a multiple of any launch width), from a nonzero state, continued
    from a tail after a cut inside the second chunk."""
    w = _wl(variant, heads=19, nonzero_s0=True)
    T = 200
    inp = I.make_inputs(w, seed=29, seqlen=T, batch=2)
    cut = 70
    a, b = slice_inputs(inp, 0, cut), slice_inputs(inp, cut, T)
    o1, S1, t1 = run_gpu(variant, a, chunk=64, S0=inp["S0"])
    o2, S2, t2 = run_gpu(variant, b, chunk=64, pos=cut, S0=S1, tail=t1)
    ro, rS, rt = run_oracle(variant, inp, S0=inp["S0"])
    _check("groups out", torch.cat([o1, o2], dim=2), ro)
    _check("groups S", S2, rS)
    np.testing.assert_array_equal(F.split_tail(t2, 2, 19, 1, 64, 64)[0].double().numpy(), rt[0])
