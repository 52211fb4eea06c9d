"""GPU parity of the backward pass (falcon_bwd: Falcon-1 and 1A, dk = dv = 64, chunk 64).

Every case runs the C ABI on the GPU and the fp64 autograd oracle on the same inputs and compares
every gradient element by element. The kernels read the inputs exactly (bf16 or fp32, widened)
and return fp32 gradients, so the only difference from the oracle is fp32 arithmetic: the bound is
max|gpu - ref| / max|ref| <= 2e-4 per gradient tensor, twice the forward pass's fp32 bound because
the backward chains two triangular systems (T and T^T) and the reverse state recurrence on top of
the forward one.
"""

import numpy as np
import pytest
import torch

from oracle import falcon_bwd as OB
from weight_linear_attention_gb300 import falcon as F
from weight_linear_attention_gb300 import inputs as I

pytestmark = pytest.mark.gpu

F1, F1A = 1, 2
TOL = 2e-4
NAMES = ("dq", "dk", "dv", "dbeta", "dlam", "dS0")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weight_linear_attention_gb300 import build

    build.build()
    F.load()


def _inputs(variant, seed, T, B=2, H=3, dtype="bf16", s0=True, pos=0, **kw):
    name = "f1_bwd_b8h12t1024_bf16" if variant == F1 else "f1a_bwd_b8h12t1024_bf16"
    w = I.WORKLOADS[name].with_(heads=H, dtype=dtype, nonzero_s0=s0, pos0=pos, **kw)
    inp = I.make_inputs(w, seed=seed, seqlen=T, batch=B)
    inp.update(I.make_adjoints(w, seed=seed, seqlen=T, batch=B))
    return inp


def _gpu(variant, inp, pos=0, want_dS=True, eps_gamma=1e-6):
    d = {n: (inp[n].cuda().contiguous() if inp.get(n) is not None else None)
         for n in ("q", "k", "v", "beta", "lam", "S0", "tail", "dout", "dS_final")}
    g = F.backward(variant, d["q"], d["k"], d["v"], d["beta"], d["lam"], d["dout"], d["S0"],
                   d["dS_final"] if want_dS else None, d["tail"], pos=pos, eps_gamma=eps_gamma)
    torch.cuda.synchronize()
    return {n: (t.cpu().double().numpy() if t is not None else None) for n, t in g.items()}


def _ref(variant, inp, pos=0, want_dS=True, eps_gamma=1e-6):
    tail = inp["tail"].reshape(inp["q"].shape[0], inp["q"].shape[1], -1) if inp.get("tail") is not None else None
    return OB.falcon_ref_bwd(variant, inp["q"], inp["k"], inp["v"], inp["beta"], inp["lam"], inp["dout"],
                             inp["S0"], inp["dS_final"] if want_dS else None, pos=pos, tail=tail,
                             eps_gamma=eps_gamma)


def _err(a, b):
    den = np.abs(b).max()
    return float(np.abs(a - b).max() / den) if den > 0 else float(np.abs(a).max())


def _check(tag, g, r, names=NAMES, bound=TOL):
    for n in names:
        if r.get(n) is None:
            continue
        e = _err(g[n], r[n])
        print(f"PARITY {tag} {n}: err {e:.3e} bound {bound:.1e}")
        assert np.isfinite(e) and e <= bound, f"{tag} {n}: {e:.3e} > {bound:.1e}"


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("variant", [F1, F1A])
@pytest.mark.parametrize("T", [1, 2, 63, 64, 65, 130, 200])
def test_lengths(variant, dtype, T):
    inp = _inputs(variant, 40 + T, T, dtype=dtype)
    _check(f"v{variant} {dtype} T={T}", _gpu(variant, inp), _ref(variant, inp))


@pytest.mark.parametrize("variant", [F1, F1A])
def test_zero_state_no_final_adjoint(variant):
    inp = _inputs(variant, 50, 150, s0=False)
    _check(f"v{variant} S0=0", _gpu(variant, inp, want_dS=False), _ref(variant, inp, want_dS=False))


@pytest.mark.parametrize("variant", [F1, F1A])
@pytest.mark.parametrize("pos", [1, 64, 77])
def test_continuation_from_tail(variant, pos):
    """pos > 0: x_1 is the tail key and the first step is a real one (its beta and lambda get gradients)."""
    inp = _inputs(variant, 51 + pos, 140, pos=pos)
    g, r = _gpu(variant, inp, pos=pos), _ref(variant, inp, pos=pos)
    _check(f"v{variant} pos={pos}", g, r, NAMES + ("dtail",))


@pytest.mark.parametrize("variant", [F1, F1A])
def test_clamp_stress(variant):
    """beta = 1.5, lambda = 1000: the clamp binds on every step (no gradient through alpha)."""
    inp = _inputs(variant, 52, 150, lam_const=1000.0, lam_shift=None)
    inp["beta"] = torch.full_like(inp["beta"], 1.5)
    _check(f"v{variant} clamp", _gpu(variant, inp), _ref(variant, inp))


@pytest.mark.parametrize("variant", [F1, F1A])
def test_mixed_decay_chunks(variant):
    """Strong decay in some chunks only, next to free ones, and a few clamped steps inside a free chunk."""
    inp = _inputs(variant, 53, 256)
    inp["lam"][:, :, 64:128] = 1000.0
    inp["lam"][:, :, 200:210] = 50.0
    _check(f"v{variant} mixed", _gpu(variant, inp), _ref(variant, inp))


def test_zero_beta_steps():
    """beta = 0 on some steps: eta = 0 there but beta's gradient is still defined (eta = beta / den)."""
    inp = _inputs(F1, 54, 100)
    inp["beta"][:, :, 10:20] = 0.0
    _check("beta=0", _gpu(F1, inp), _ref(F1, inp))


@pytest.mark.parametrize("variant", [F1, F1A])
def test_headline_shape_all_sequences(variant):
    """The bench's workload (8 x 12 x 1024, bf16) in one call; the oracle recomputes all 96 sequences,
    one batch row (12 heads) at a time to bound its autograd memory."""
    name = "f1_bwd_b8h12t1024_bf16" if variant == F1 else "f1a_bwd_b8h12t1024_bf16"
    w = I.WORKLOADS[name]
    inp = I.make_inputs(w, seed=55)
    inp.update(I.make_adjoints(w, seed=55))
    g = _gpu(variant, inp)
    for b in range(inp["q"].shape[0]):
        one = {n: (inp[n][b:b + 1] if inp.get(n) is not None else None)
               for n in ("q", "k", "v", "beta", "lam", "S0", "dout", "dS_final")}
        r = _ref(variant, one)
        gs = {n: (g[n][b:b + 1] if g.get(n) is not None else None) for n in NAMES}
        _check(f"v{variant} headline row {b}", gs, r)


@pytest.mark.parametrize("variant,dtype", [(F1, "bf16"), (F1A, "bf16"), (F1, "f32"), (F1A, "f32")])
@pytest.mark.parametrize("B,H", [(1, 1), (1, 3), (2, 2), (1, 15), (17, 1), (3, 11)])
def test_sequence_groups(B, H, variant, dtype):
    """A call runs its sequences unsplit (fewer than 4), in two groups (4 to 15) or in four groups
    (16 and more, here of unequal sizes: 17 and 33 sequences) on streams of their own; every
    sequence of every group is compared, with a ragged last chunk and a nonzero initial state."""
    inp = _inputs(variant, 57 + B * H, 150, B=B, H=H, dtype=dtype)
    _check(f"groups v{variant} {dtype} B={B} H={H}", _gpu(variant, inp), _ref(variant, inp))


def test_graph_capture():
    """One falcon_bwd call captured into a CUDA graph (two groups of sequences, so the library's own
    streams join the capture) and replayed on new inputs copied into the same buffers."""
    B, H, T = 2, 4, 150
    names = ("q", "k", "v", "beta", "lam", "S0", "dout", "dS_final")
    a, b = _inputs(F1, 61, T, B=B, H=H), _inputs(F1, 62, T, B=B, H=H)
    d = {n: a[n].cuda().contiguous() for n in names}
    f32 = dict(dtype=torch.float32, device="cuda")
    out = {"dq": torch.empty(B, H, T, 64, **f32), "dk": torch.empty(B, H, T, 64, **f32),
           "dv": torch.empty(B, H, T, 64, **f32), "dbeta": torch.empty(B, H, T, **f32),
           "dlam": torch.empty(B, H, T, **f32), "dS0": torch.empty(B, H, 64, 64, **f32)}
    dims = F.make_dims(B, H, T, 64, 64, dtype=F.FALCON_BF16)
    ws = torch.empty(F.falcon_bwd_workspace_bytes(F1, dims, 64), dtype=torch.uint8, device="cuda")

    def call():
        st = F.falcon_bwd(F1, d["q"], d["k"], d["v"], d["beta"], d["lam"], d["S0"], None, d["dout"], d["dS_final"],
                          out["dq"], out["dk"], out["dv"], out["dbeta"], out["dlam"], out["dS0"], None, dims, 64, ws,
                          stream=torch.cuda.current_stream().cuda_stream)
        assert st == 0

    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        call()  # the library's streams and kernel attributes exist before the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    for inp in (a, b):
        for n in names:
            d[n].copy_(inp[n])
        g.replay()
        torch.cuda.synchronize()
        got = {n: t.cpu().double().numpy() for n, t in out.items()}
        got["dtail"] = None
        _check("graph replay", got, _ref(F1, inp))


def test_argument_errors():
    inp = _inputs(F1, 56, 64)
    d = {n: inp[n].cuda() for n in ("q", "k", "v", "beta", "lam", "dout")}
    B, H, T, dk = d["q"].shape
    dims = F.make_dims(B, H, T, dk, 64, dtype=F.FALCON_BF16)
    n = F.falcon_bwd_workspace_bytes(F1, dims, 64)
    assert n == B * H * 1 * (6 * 64 * 64 * 4 + 3072)  # six 16 KiB slots and the scalars per chunk
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    outs = [torch.full((B, H, T, 64), 7.0, device="cuda") for _ in range(3)] + \
           [torch.full((B, H, T), 7.0, device="cuda") for _ in range(2)]
    args = lambda ws_, nbytes, ch=64, var=F1: F.falcon_bwd(var, d["q"], d["k"], d["v"], d["beta"], d["lam"], None,
                                                           None, d["dout"], None, *outs, None, None, dims, ch, ws_,
                                                           nbytes)
    assert args(None, 0) == F.FALCON_ERR_INVALID_ARG           # workspace required
    assert args(ws, n - 256) == F.FALCON_ERR_INVALID_ARG       # too small
    assert args(ws, n, ch=32) == F.FALCON_ERR_UNSUPPORTED      # chunk 64 only
    assert args(ws, n, var=3) == F.FALCON_ERR_UNSUPPORTED      # Falcon-2 has no backward kernel yet
    torch.cuda.synchronize()
    for o in outs:
        assert torch.all(o == 7.0)
    assert args(ws, n) == F.FALCON_OK
    torch.cuda.synchronize()
