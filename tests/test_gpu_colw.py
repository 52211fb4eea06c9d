"""GPU parity of the per-column kernel (Falcon-2 / 2A, bf16, dk = dv = 64, chunk 64): one persistent
CTA per sequence, the shared Gram and scores one chunk ahead, one merged residual solve per value
column, the state on chip.

Every case runs through the C ABI and is compared with the fp64 oracle at the bf16 bound (both
checks of tests.gpu_util.check), covering the branches that kernel has: a nonzero and an aliased
initial state, columns whose chunk decay passes e^-30 (their steps run one by one) next to columns
that stay on the factored form in the same warp, continuation from a tail at every kind of split
point, lengths around the chunk boundary, odd sequence counts, a beta that is not 16-byte aligned
(the CUDA-core kernel runs instead), and the full Falcon-2 and 2A workload shape (8 x 12 x 2048),
every sequence compared.
"""

import numpy as np
import pytest
import torch

from tests.gpu_util import check, run_gpu, run_oracle, slice_inputs
from weight_linear_attention_gb300 import falcon as F
from weight_linear_attention_gb300 import inputs as I

pytestmark = pytest.mark.gpu

F2, F2A = 3, 4
NAME = {F2: "f2_b8h12t2048_bf16", F2A: "f2a_b8h12t2048_bf16"}


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
    return I.WORKLOADS[NAME[variant]].with_(**kw)


def _colw(variant, inp, S0=None, pos=0, tail=None, eps_gamma=1e-6):
    dims = F.make_dims(*inp["q"].shape[:3], 64, 64, dtype=F.FALCON_BF16, pos=pos)
    T = inp["q"].shape[2]
    assert F.falcon_kernel_for(variant, dims, 64) == (4 if T == 1 else 7)
    assert F.falcon_workspace_bytes(variant, dims, 64) == 0
    return run_gpu(variant, inp, chunk=64, S0=S0, pos=pos, tail=tail, eps_gamma=eps_gamma)


@pytest.mark.parametrize("variant", [F2, F2A])
def test_nonzero_initial_state(variant):
    inp = I.make_inputs(_wl(variant, nonzero_s0=True), seed=41, seqlen=200, batch=2)
    out, S, _ = _colw(variant, inp, S0=inp["S0"])
    r_out, r_S, _ = run_oracle(variant, inp, S0=inp["S0"])
    _check(f"v{variant} S0 out", out, r_out)
    _check(f"v{variant} S0 S", S, r_S)


@pytest.mark.parametrize("variant", [F2, F2A])
def test_S_final_may_alias_S0(variant):
    inp = I.make_inputs(_wl(variant, nonzero_s0=True), seed=42, seqlen=130, batch=2)
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


@pytest.mark.parametrize("variant", [F2, F2A])
def test_clamp_stress(variant):
    """beta = 1.5, lambda = 1000: alpha = 1 - eps_gamma on every step of every column (log decay
    ~ -13.8 per token), so every column of every chunk runs its steps one by one."""
    inp = I.make_inputs(_wl(variant, lam_const=1000.0), seed=43, seqlen=150, batch=1)
    inp["beta"] = torch.full_like(inp["beta"], 1.5)
    out, S, _ = _colw(variant, inp)
    r_out, r_S, _ = run_oracle(variant, inp)
    _check(f"clamp v{variant} out", out, r_out)
    _check(f"clamp v{variant} S", S, r_S)


@pytest.mark.parametrize("variant", [F2, F2A])
def test_mixed_decay_columns(variant):
    """Strong decay in some chunks, and within them only on some columns (beta 0 on the others, so
    their steps are 0 and their decay 1): factored and one-by-one columns share warps and chunks."""
    inp = I.make_inputs(_wl(variant), seed=44, seqlen=256, batch=1)
    inp["lam"][:, :, 64:128] = 1000.0
    inp["lam"][:, :, 200:210] = 50.0
    inp["beta"][:, :, 64:128, 1::3] = 0.0
    inp["beta"][:, :, 64:128, 0::5] = 1.5
    out, S, _ = _colw(variant, inp)
    r_out, r_S, _ = run_oracle(variant, inp)
    _check(f"mixed v{variant} out", out, r_out)
    _check(f"mixed v{variant} S", S, r_S)


@pytest.mark.parametrize("variant,cut", [(F2, 1), (F2, 63), (F2, 64), (F2, 100), (F2A, 64), (F2A, 77)])
def test_segment_continuation(variant, cut):
    """Two calls carrying S_final and the tail (pos > 0: the first shifted key comes from the tail)."""
    T = 200
    inp = I.make_inputs(_wl(variant), seed=45, seqlen=T, batch=2)
    a, b = slice_inputs(inp, 0, cut), slice_inputs(inp, cut, T)
    o1, S1, t1 = run_gpu(variant, a, chunk=64)
    o2, S2, t2 = run_gpu(variant, b, chunk=64, pos=cut, S0=S1, tail=t1)
    ro, rS, rt = run_oracle(variant, inp)
    _check("cont out", torch.cat([o1, o2], dim=2), ro)
    _check("cont S", S2, rS)
    tk, tv = F.split_tail(t2, 2, 12, 1, 64, 64)
    np.testing.assert_array_equal(tk.double().numpy(), rt[0])


@pytest.mark.parametrize("T", [0, 1, 2, 63, 64, 65, 127, 128, 129, 1000])
def test_lengths(T):
    inp = I.make_inputs(_wl(F2), seed=46, seqlen=max(T, 1), batch=1)
    if T == 0:
        inp = slice_inputs(inp, 0, 0)
    out, S, t = _colw(F2, inp)
    r_out, r_S, rt = run_oracle(F2, inp)
    if T > 0:
        _check(f"T={T} out", out, r_out)
    _check(f"T={T} S", S, r_S)
    np.testing.assert_array_equal(F.split_tail(t, 1, 12, 1, 64, 64)[0].double().numpy(), rt[0])


@pytest.mark.parametrize("variant", [F2, F2A])
def test_odd_sequence_count_with_state_and_tail(variant):
    """2 x 19 sequences from a nonzero state, continued from a tail after a cut inside the second chunk."""
    T = 200
    inp = I.make_inputs(_wl(variant, heads=19, nonzero_s0=True), seed=47, seqlen=T, batch=2)
    cut = 70
    a, b = slice_inputs(inp, 0, cut), slice_inputs(inp, cut, T)
    o1, S1, t1 = run_gpu(variant, a, chunk=64, S0=inp["S0"])
    o2, S2, t2 = run_gpu(variant, b, chunk=64, pos=cut, S0=S1, tail=t1)
    ro, rS, rt = run_oracle(variant, inp, S0=inp["S0"])
    _check("groups out", torch.cat([o1, o2], dim=2), ro)
    _check("groups S", S2, rS)
    np.testing.assert_array_equal(F.split_tail(t2, 2, 19, 1, 64, 64)[0].double().numpy(), rt[0])


def test_beta_not_16_byte_aligned_runs_cuda_core_kernel():
    """beta 4-byte aligned only: the TMA load cannot take it, the CUDA-core kernel runs; same results."""
    inp = I.make_inputs(_wl(F2), seed=48, seqlen=100, batch=1)
    dev = {n: inp[n].cuda() for n in ("q", "k", "v", "lam")}
    buf = torch.empty(inp["beta"].numel() + 1, dtype=torch.float32, device="cuda")
    beta = buf[1:].view_as(inp["beta"])
    beta.copy_(inp["beta"].cuda())
    assert beta.data_ptr() % 16 != 0
    out = torch.empty_like(dev["v"])
    S = torch.empty(1, 12, 64, 64, dtype=torch.float32, device="cuda")
    d = F.make_dims(1, 12, 100, 64, 64, dtype=F.FALCON_BF16)
    st = F.falcon_fwd(F2, dev["q"], dev["k"], dev["v"], beta, dev["lam"], None, None, out, S, None, d, 64)
    assert st == 0
    torch.cuda.synchronize()
    assert F.falcon_device_status() == F.FALCON_OK
    r_out, r_S, _ = run_oracle(F2, inp)
    _check("unaligned beta out", out.cpu(), r_out)
    _check("unaligned beta S", S.cpu(), r_S)


@pytest.mark.parametrize("variant", [F2, F2A])
def test_full_workload_shape_all_sequences(variant):
    """The bench's Falcon-2 / 2A workload (8 x 12 x 2048) in one call, every sequence against the oracle."""
    w = _wl(variant)
    inp = I.make_inputs(w, seed=49)
    r_out, r_S, _ = run_oracle(variant, inp)
    o, S, _ = _colw(variant, inp)
    _check(f"v{variant} full out", o, r_out)
    _check(f"v{variant} full S", S, r_S)
