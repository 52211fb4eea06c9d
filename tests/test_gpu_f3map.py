"""GPU parity of the tensor-core chunk maps of the scan path (Falcon-3 and 3A, bf16, dk = dv = 64,
window 4, chunk 32): the maps come from the tcgen05 kernel, chunks whose decay is too strong for its
factored form from the CUDA-core map kernel, and the scan over them as before.

Every case runs through the C ABI and is compared with the fp64 oracle at the bf16 bound (both
checks of tests.gpu_util.check); the tails are compared bit for bit. Cases: lengths around the chunk
boundary (the first chunk's windows are incomplete), a nonzero and an aliased initial state,
continuation from a tail at several cuts (a continuation's first chunk takes its earlier keys and
values from the tail), chunks with strong decay next to ordinary ones (both map kernels in one call),
the marks the tensor-core kernel leaves in the workspace, and the full Falcon-3 / 3A workload
(2 x 12 x 16384 as two 8192-token segments), every sequence compared.
"""

import numpy as np
import pytest
import torch

from tests.gpu_util import check, run_gpu, run_oracle, slice_inputs
from weight_linear_attention_gb300 import falcon as F
from weight_linear_attention_gb300 import inputs as I

pytestmark = pytest.mark.gpu

F3, F3A = 5, 6
NAME = {F3: "f3w4_b2h12t16384_bf16", F3A: "f3aw4_b2h12t16384_bf16"}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weight_linear_attention_gb300 import build

    build.build()
    F.load()


def _wl(variant, **kw):
    return I.WORKLOADS[NAME[variant]].with_(segments=1, **kw)


def _check(name, gpu, ref):
    check(name, gpu, ref, torch.bfloat16)


def _tails_equal(t, rt, B, H):
    tk, tv = F.split_tail(t, B, H, 4, 64, 64)
    np.testing.assert_array_equal(tk.double().numpy(), rt[0])
    np.testing.assert_array_equal(tv.double().numpy(), rt[1])


def _scan(variant, inp, S0=None, pos=0, tail=None):
    dims = F.make_dims(*inp["q"].shape[:3], 64, 64, window=4, dtype=F.FALCON_BF16, pos=pos)
    assert F.falcon_kernel_for(variant, dims, 32) == 5
    return run_gpu(variant, inp, window=4, chunk=32, S0=S0, pos=pos, tail=tail)


@pytest.mark.parametrize("variant", [F3, F3A])
@pytest.mark.parametrize("T", [128, 130, 161, 1500])
def test_lengths_and_initial_state(variant, T):
    inp = I.make_inputs(_wl(variant, nonzero_s0=True), seed=90 + T, seqlen=T, batch=2)
    out, S, t = _scan(variant, inp, S0=inp["S0"])
    ro, rS, rt = run_oracle(variant, inp, window=4, S0=inp["S0"])
    _check(f"v{variant} T={T} out", out, ro)
    _check(f"v{variant} T={T} S", S, rS)
    _tails_equal(t, rt, 2, 12)


@pytest.mark.parametrize("variant,cut", [(F3, 1), (F3, 2), (F3, 3), (F3, 37), (F3, 517), (F3A, 2), (F3A, 300)])
def test_continuation(variant, cut):
    """Two calls; the second starts at pos > 0 from the first's S_final and tail (its first chunk's
    windows reach back into the tail, partly past the sequence start for cuts below 4)."""
    T = 800
    inp = I.make_inputs(_wl(variant), seed=95, seqlen=T, batch=2)
    a, b = slice_inputs(inp, 0, cut), slice_inputs(inp, cut, T)
    o1, S1, t1 = run_gpu(variant, a, window=4, chunk=32)
    o2, S2, t2 = _scan(variant, b, S0=S1, pos=cut, tail=t1)
    ro, rS, rt = run_oracle(variant, inp, window=4)
    _check(f"v{variant} cut={cut} out", torch.cat([o1, o2], dim=2), ro)
    _check(f"v{variant} cut={cut} S", S2, rS)
    _tails_equal(t2, rt, 2, 12)


@pytest.mark.parametrize("variant", [F3, F3A])
def test_strong_decay_chunks_take_the_cuda_core_maps(variant):
    """beta 1.5 and lambda 1000 on two chunks (their decay passes e^-30), ordinary chunks around them:
    the tensor-core kernel leaves those two unmarked and the CUDA-core kernel forms their maps."""
    T = 600
    inp = I.make_inputs(_wl(variant, nonzero_s0=True), seed=96, seqlen=T, batch=1)
    inp["lam"][:, :, 64:128] = 1000.0
    inp["beta"][:, :, 64:128] = 1.5
    dev = {n: inp[n].cuda() for n in ("q", "k", "v", "beta", "lam")}
    d = F.make_dims(1, 12, T, 64, 64, window=4, dtype=F.FALCON_BF16)
    ws = F.workspace_for(variant, d, 32, "cuda")
    out = torch.empty_like(dev["v"])
    S = torch.empty(1, 12, 64, 64, dtype=torch.float32, device="cuda")
    st = F.falcon_fwd(variant, dev["q"], dev["k"], dev["v"], dev["beta"], dev["lam"], inp["S0"].cuda(), None, out, S,
                      None, d, 32, ws)
    assert st == 0
    torch.cuda.synchronize()
    assert F.falcon_device_status() == F.FALCON_OK
    ro, rS, _ = run_oracle(variant, inp, window=4, S0=inp["S0"])
    _check(f"v{variant} strong decay out", out.cpu(), ro)
    _check(f"v{variant} strong decay S", S.cpu(), rS)
    # the marks: chunk blocks of 5 x 64 x 64 floats, the state slot's first word
    N = -(-T // 32)
    marks = ws.view(torch.int32)[: 12 * N * 5 * 4096].view(12, N, 5 * 4096)[:, :, 2 * 4096].cpu().numpy()
    assert (marks[:, 2:4] == 0).all()  # chunks 2 and 3 (tokens 64-127) left to the CUDA-core kernel
    others = np.delete(marks, [2, 3], axis=1)
    assert (others == 1).all()


@pytest.mark.parametrize("variant", [F3, F3A])
def test_full_workload_all_sequences(variant):
    """The bench's Falcon-3 / 3A workload: 2 x 12 x 16384 as two 8192-token calls carrying S_final and
    the tail, every sequence against the oracle over the whole 16384 tokens."""
    w = I.WORKLOADS[NAME[variant]]
    inp = I.make_inputs(w, seed=97)
    T = inp["q"].shape[2]
    a, b = slice_inputs(inp, 0, T // 2), slice_inputs(inp, T // 2, T)
    o1, S1, t1 = _scan(variant, a)
    o2, S2, t2 = _scan(variant, b, S0=S1, pos=T // 2, tail=t1)
    ro, rS, rt = run_oracle(variant, inp, window=4)
    _check(f"v{variant} full out", torch.cat([o1, o2], dim=2), ro)
    _check(f"v{variant} full S", S2, rS)
    _tails_equal(t2, rt, 2, 12)
