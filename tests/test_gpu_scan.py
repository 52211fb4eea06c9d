"""GPU parity of the scan path (Falcon-1, 1A, 3, 3A with dk = dv = 64 and few sequences): every
chunk's affine state map, the associative scan over those maps (groups of 16 chunks, or of enough
chunks that the groups just fill the GPU when there are many), then every
chunk's outputs, against the fp64 oracle at the same bounds as the other paths (fp32 inputs:
max|err| / max|ref| <= 1e-4; bf16: max|err| / RMS(ref) <= 2e-2). Cases span one group and several,
both scan kernels (16-column slices for few groups; for many, one CTA per group with the state in
tensor memory and each step a tensor-core product),
ragged chunks, a nonzero initial state, continuation from a tail, the decay clamp, and the aliased
S_final = S0 call.
"""

import numpy as np
import pytest
import torch

from tests.gpu_util import check, rel_err, run_gpu, run_oracle, slice_inputs, tol
from weight_linear_attention_gb300 import falcon as F
from weight_linear_attention_gb300 import inputs as I

pytestmark = pytest.mark.gpu

F1, F1A, F3, F3A = 1, 2, 5, 6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weight_linear_attention_gb300 import build

    build.build()
    F.load()


def _wl(variant, dtype, **kw):
    base = {F1: "f1_b8h12t1024_bf16", F1A: "f1a_b8h12t1024_bf16", F3: "f3w4_b2h12t16384_bf16",
            F3A: "f3aw4_b2h12t16384_bf16"}[variant]
    return I.WORKLOADS[base].with_(dtype=dtype, segments=1, **kw)


def _check(name, gpu, ref, dtype):
    check(name, gpu, ref, dtype)


def _run(w, inp, chunk, S0=None, pos=0, tail=None, rtail=None, name=""):
    dims = F.make_dims(*inp["q"].shape[:3], 64, 64, window=w.window,
                       dtype=F.FALCON_F32 if w.dtype == "f32" else F.FALCON_BF16, pos=pos)
    assert F.falcon_kernel_for(w.variant_id, dims, chunk) == 5
    out, S, t = run_gpu(w.variant_id, inp, window=w.window, chunk=chunk, S0=S0, pos=pos, tail=tail)
    ro, rS, rt = run_oracle(w.variant_id, inp, window=w.window, S0=S0, pos=pos, tail=rtail)
    _check(f"{name} out", out, ro, w.torch_dtype)
    _check(f"{name} S", S, rS, torch.float32 if w.dtype == "f32" else w.torch_dtype)
    B, H = inp["q"].shape[:2]
    tk, tv = F.split_tail(t, B, H, w.window, 64, 64)
    np.testing.assert_array_equal(tk.double().numpy(), rt[0])
    np.testing.assert_array_equal(tv.double().numpy(), rt[1])
    return out, S, t, (ro, rS, rt)


@pytest.mark.parametrize("variant,dtype,chunk,T", [
    (F1, "f32", 64, 300),      # one group, ragged last chunk
    (F1, "f32", 16, 1000),     # 63 chunks: four groups, the last partial
    (F1A, "f32", 32, 1030),
    (F1, "bf16", 32, 700),     # bf16 at chunk 32 (no split path there)
    (F3, "bf16", 32, 1500),
    (F3A, "bf16", 32, 1500),
    (F3, "f32", 16, 600),
    (F1, "f32", 32, 4096),     # 2 x 12 sequences x 8 groups: the tensor-core steps (fp32 inputs: 1e-4 bound)
    (F3, "bf16", 32, 4096),
    (F3A, "bf16", 32, 4096),
    (F1, "f32", 64, 8300),     # the same kernel at chunk 64, 9 groups of 15 chunks, ragged last chunk
    (F1A, "f32", 16, 2100),    # and at chunk 16
    (F3, "bf16", 32, 4100),
])
def test_scan_path(variant, dtype, chunk, T):
    w = _wl(variant, dtype, nonzero_s0=True)
    inp = I.make_inputs(w, seed=60 + T, seqlen=T, batch=2)
    _run(w, inp, chunk, S0=inp["S0"], name=f"v{variant} {dtype} C={chunk} T={T}")


@pytest.mark.parametrize("variant,dtype,chunk,T", [(F1, "f32", 16, 3848), (F3, "bf16", 32, 7696)])
def test_tensor_core_scan_last_group_of_one_chunk(variant, dtype, chunk, T):
    """12 sequences of 241 chunks: 16 groups of 16, the last group a single ragged chunk (compose
    takes it as the group's map without a step; apply runs one step from its start state)."""
    w = _wl(variant, dtype, nonzero_s0=True)
    inp = I.make_inputs(w, seed=70 + T, seqlen=T, batch=1)
    _run(w, inp, chunk, S0=inp["S0"], name=f"v{variant} {dtype} C={chunk} T={T} one-chunk group")


@pytest.mark.parametrize("variant", [F1, F3])
def test_scan_continuation(variant):
    """Two calls: the second starts at pos > 0 from the first's S_final and tail."""
    w = _wl(variant, "bf16")
    T, cut = 1200, 517
    inp = I.make_inputs(w, seed=70, seqlen=T, batch=2)
    a, b = slice_inputs(inp, 0, cut), slice_inputs(inp, cut, T)
    o1, S1, t1, (_, _, rt1) = _run(w, a, 32, name=f"v{variant} first")
    W = w.window
    o2, S2, t2 = run_gpu(w.variant_id, b, window=W, chunk=32, S0=S1, pos=cut, tail=t1)
    ro, rS, _ = run_oracle(w.variant_id, inp, window=W)
    _check(f"v{variant} cont out", torch.cat([o1, o2], dim=2), ro, w.torch_dtype)
    _check(f"v{variant} cont S", S2, rS, w.torch_dtype)


def test_scan_clamp():
    w = _wl(F1, "f32", lam_const=1000.0, lam_shift=None)
    inp = I.make_inputs(w, seed=71, seqlen=500, batch=1)
    inp["beta"] = torch.full_like(inp["beta"], 1.5)
    _run(w, inp, 32, name="clamp")


def test_scan_state_alias():
    w = _wl(F3, "bf16", nonzero_s0=True)
    inp = I.make_inputs(w, seed=72, seqlen=900, batch=1)
    dev = {n: inp[n].cuda() for n in ("q", "k", "v", "beta", "lam")}
    S = inp["S0"].cuda().contiguous()
    out = torch.empty_like(dev["v"])
    d = F.make_dims(1, w.heads, 900, 64, 64, window=4, dtype=F.FALCON_BF16)
    ws = F.workspace_for(F3, d, 32, "cuda")
    assert ws is not None and F.falcon_kernel_for(F3, d, 32) == 5
    st = F.falcon_fwd(F3, dev["q"], dev["k"], dev["v"], dev["beta"], dev["lam"], S, None, out, S, None, d, 32, ws)
    assert st == 0
    torch.cuda.synchronize()
    ro, rS, _ = run_oracle(F3, inp, window=4, S0=inp["S0"])
    _check("alias out", out.cpu(), ro, torch.bfloat16)
    _check("alias S", S.cpu(), rS, torch.bfloat16)


def test_scan_path_on_static_scratch():
    """falcon_fwd_static: a small Falcon-3 call whose scan path fits the library's own scratch."""
    w = _wl(F3, "bf16", nonzero_s0=True, heads=2)
    inp = I.make_inputs(w, seed=73, seqlen=500, batch=1)
    dev = {n: inp[n].cuda() for n in ("q", "k", "v", "beta", "lam")}
    S0 = inp["S0"].cuda().contiguous()
    out = torch.empty_like(dev["v"])
    S = torch.empty_like(S0)
    d = F.make_dims(1, 2, 500, 64, 64, window=4, dtype=F.FALCON_BF16)
    assert F.falcon_kernel_for(F3, d, 32) == 5
    assert 0 < F.falcon_workspace_bytes(F3, d, 32) <= F.STATIC_WORKSPACE_BYTES
    st = F.falcon_fwd_static(F3, dev["q"], dev["k"], dev["v"], dev["beta"], dev["lam"], S0, None, out, S, None, d, 32)
    assert st == 0
    torch.cuda.synchronize()
    ro, rS, _ = run_oracle(F3, inp, window=4, S0=inp["S0"])
    _check("static out", out.cpu(), ro, torch.bfloat16)
    _check("static S", S.cpu(), rS, torch.bfloat16)


@pytest.mark.parametrize("variant", [F3, F3A])
@pytest.mark.parametrize("W,chunk", [(1, 64), (2, 32), (3, 32), (5, 16), (6, 16), (7, 16), (8, 16)])
def test_scan_path_window_sizes(variant, W, chunk):
    """Every window size on the scan path: the Falcon-3 block solve takes 16 // W tokens per block, so
    W = 3, 5, 6, 7 leave a partial last block and W = 1, 2, 8 do not."""
    w = _wl(variant, "bf16", window=W, chunk=chunk, nonzero_s0=True)
    inp = I.make_inputs(w, seed=80 + W, seqlen=300, batch=2)
    _run(w, inp, chunk, S0=inp["S0"], name=f"v{variant} W={W} C={chunk}")
