"""falcon_fwd_static: the split path on the library's fixed scratch (no allocation anywhere).

Collected last on purpose: it must pass on its own and after every other GPU test (the scratch
is a module-level device array, so earlier calls through other entry points must not disturb it,
and two of its own calls in a row must agree with each other and with falcon_fwd)."""

import pytest
import torch

from weight_linear_attention_gb300 import falcon as F
from weight_linear_attention_gb300 import inputs as I

A = 1 << 40  # fake device addresses for the host-side checks: never dereferenced


def test_static_entry_rejects_oversize_without_launch():
    from weight_linear_attention_gb300 import build

    build.build()
    F.load()
    d = F.make_dims(8, 12, 1024, 64, 64)  # 1536 chunks x (66 KiB + 8 bytes) > 16 MiB
    assert F.falcon_workspace_bytes(F.FALCON_1, d, 64) > F.STATIC_WORKSPACE_BYTES
    st = F.falcon_fwd_static(F.FALCON_1, A, A + (1 << 30), A + (2 << 30), A + (3 << 30), A + (4 << 30), None, None,
                             A + (5 << 30), None, None, d, 64, stream=0)
    assert st == F.FALCON_ERR_UNSUPPORTED
    bad = F.make_dims(1, 12, 64, 48, 64)  # argument errors come first, as in falcon_fwd
    assert F.falcon_fwd_static(F.FALCON_1, A, A, A, A, A, None, None, A, None, None, bad, 64, stream=0) == \
        F.FALCON_ERR_UNSUPPORTED


def _run(entry, variant, dev, d, S0=None, ws=None):
    out = torch.empty_like(dev["v"])
    S = torch.empty(dev["q"].shape[0], dev["q"].shape[1], 64, 64, dtype=torch.float32, device="cuda")
    tail = torch.empty(F.falcon_tail_bytes(d) // 2, dtype=torch.bfloat16, device="cuda")
    args = (variant, dev["q"], dev["k"], dev["v"], dev["beta"], dev["lam"], S0, None, out, S, tail, d, 64)
    st = F.falcon_fwd(*args, ws) if entry == "fwd" else F.falcon_fwd_static(*args)
    assert st == F.FALCON_OK, F.status_string(st)
    torch.cuda.synchronize()
    assert F.falcon_device_status() == F.FALCON_OK
    return out, S, tail


@pytest.mark.gpu
@pytest.mark.parametrize("variant", [F.FALCON_1, F.FALCON_1A])
def test_static_matches_workspace_entry_on_consecutive_calls(variant):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weight_linear_attention_gb300 import build

    build.build()
    F.load()
    w = I.WORKLOADS[I.HEADLINE].with_(variant="falcon1" if variant == F.FALCON_1 else "falcon1a", nonzero_s0=True)
    d = F.make_dims(1, 12, 1024, 64, 64)  # 192 chunks: 12.4 MiB of scratch
    assert 0 < F.falcon_workspace_bytes(variant, d, 64) <= F.STATIC_WORKSPACE_BYTES
    dev = {}
    ref = None
    for seed in (31, 32):  # two consecutive calls with different inputs
        inp = I.make_inputs(w, seed=seed, seqlen=1024, batch=1)
        dev = {n: inp[n].cuda() for n in ("q", "k", "v", "beta", "lam")}
        S0 = inp["S0"].cuda()
        ws = F.workspace_for(variant, d, 64, "cuda")
        ref = _run("fwd", variant, dev, d, S0, ws)
        got = _run("static", variant, dev, d, S0)
        for a, b in zip(ref, got):
            assert torch.equal(a, b)  # the same kernels on the same inputs: bit-identical
    got2 = _run("static", variant, dev, d, inp["S0"].cuda())  # and again, after itself
    for a, b in zip(ref, got2):
        assert torch.equal(a, b)


@pytest.mark.gpu
def test_static_entry_without_split_path_runs_single_pass_kernels():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    w = I.WORKLOADS["f2_b8h12t2048_bf16"]
    inp = I.make_inputs(w, seed=33, seqlen=130, batch=1)
    dev = {n: inp[n].cuda() for n in ("q", "k", "v", "beta", "lam")}
    d = F.make_dims(1, 12, 130, 64, 64)
    assert F.falcon_workspace_bytes(F.FALCON_2, d, 64) == 0
    a = _run("fwd", F.FALCON_2, dev, d)
    b = _run("static", F.FALCON_2, dev, d)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
