"""falcon_fwd_static: the forward pass on the library's own fixed scratch, for callers that cannot
allocate device memory (a caller inside another runtime's memory pool, where an extra cudaMalloc
bypasses the pool's accounting and can fail under memory pressure, or a latency-critical loop that
must not pay cudaMalloc's implicit device synchronisation).

Of the forward paths only the scan path uses scratch, so these tests run shapes that take it and
compare with falcon_fwd given a workspace of its own. Collected last on purpose: the scratch is one
device array shared by every call, so the comparison must hold on a fresh process and after every
other test, and two calls in a row must agree with each other."""

import pytest
import torch

from weight_linear_attention_gb300 import falcon as F
from weight_linear_attention_gb300 import inputs as I

A = 1 << 40  # fake device addresses for the host-side checks: never dereferenced


def test_static_entry_checks_arguments_before_any_launch():
    from weight_linear_attention_gb300 import build

    build.build()
    F.load()
    bad = F.make_dims(1, 12, 64, 48, 64)  # argument errors come first, as in falcon_fwd
    assert F.falcon_fwd_static(F.FALCON_1, A, A, A, A, A, None, None, A, None, None, bad, 64, stream=0) == \
        F.FALCON_ERR_UNSUPPORTED
    d = F.make_dims(1, 4, 512, 64, 64)
    assert F.falcon_fwd_static(F.FALCON_1, A, A + (1 << 30), A + (2 << 30), A + (3 << 30), A + (4 << 30), None,
                               None, A + 4096, None, None, d, 32, stream=0) == F.FALCON_ERR_INVALID_ARG  # out on q


def _run(entry, variant, dev, d, chunk, S0=None, ws=None):
    out = torch.empty_like(dev["v"])
    S = torch.empty(dev["q"].shape[0], dev["q"].shape[1], 64, 64, dtype=torch.float32, device="cuda")
    tail = torch.empty(F.falcon_tail_bytes(d) // 2, dtype=torch.bfloat16, device="cuda")
    args = (variant, dev["q"], dev["k"], dev["v"], dev["beta"], dev["lam"], S0, None, out, S, tail, d, chunk)
    st = F.falcon_fwd(*args, ws) if entry == "fwd" else F.falcon_fwd_static(*args)
    assert st == F.FALCON_OK, F.status_string(st)
    torch.cuda.synchronize()
    assert F.falcon_device_status() == F.FALCON_OK
    return out, S, tail


def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weight_linear_attention_gb300 import build

    build.build()
    F.load()


@pytest.mark.gpu
@pytest.mark.parametrize("variant", [F.FALCON_1, F.FALCON_1A])
def test_static_matches_workspace_entry_on_consecutive_calls(variant):
    """Two calls in a row with different inputs, then the first inputs again: each equals falcon_fwd
    with a workspace of its own (the same kernels on the same inputs: bit-identical)."""
    _lib()
    w = I.WORKLOADS[I.HEADLINE].with_(variant="falcon1" if variant == F.FALCON_1 else "falcon1a", nonzero_s0=True,
                                      heads=4, chunk=32)
    d = F.make_dims(1, 4, 512, 64, 64)  # chunk 32: the scan path, 16 chunks per sequence
    assert F.falcon_kernel_for(variant, d, 32) == 5
    assert 0 < F.falcon_workspace_bytes(variant, d, 32) <= F.STATIC_WORKSPACE_BYTES
    runs = []
    for seed in (31, 32, 31):
        inp = I.make_inputs(w, seed=seed, seqlen=512, batch=1)
        dev = {n: inp[n].cuda() for n in ("q", "k", "v", "beta", "lam")}
        S0 = inp["S0"].cuda()
        ws = F.workspace_for(variant, d, 32, "cuda")
        ref = _run("fwd", variant, dev, d, 32, S0, ws)
        got = _run("static", variant, dev, d, 32, S0)
        for a, b in zip(ref, got):
            assert torch.equal(a, b)
        runs.append(got)
    for a, b in zip(runs[0], runs[2]):  # the scratch keeps nothing from one call to the next
        assert torch.equal(a, b)


@pytest.mark.gpu
def test_static_entry_runs_cuda_core_kernel_when_scan_scratch_does_not_fit():
    """A scan-path shape needing more than the fixed scratch runs the CUDA-core chunk kernel, as
    falcon_fwd does without a workspace."""
    _lib()
    w = I.WORKLOADS[I.HEADLINE].with_(chunk=32)
    d = F.make_dims(1, 12, 1024, 64, 64)
    assert F.falcon_workspace_bytes(F.FALCON_1, d, 32) > F.STATIC_WORKSPACE_BYTES
    inp = I.make_inputs(w, seed=34, seqlen=1024, batch=1)
    dev = {n: inp[n].cuda() for n in ("q", "k", "v", "beta", "lam")}
    a = _run("fwd", F.FALCON_1, dev, d, 32)  # no workspace: the CUDA-core kernel
    b = _run("static", F.FALCON_1, dev, d, 32)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


@pytest.mark.gpu
def test_static_entry_on_paths_without_scratch():
    """The fused and CUDA-core kernels need no scratch: the static entry point runs them unchanged."""
    _lib()
    for wname, variant in (("f1_b8h12t1024_bf16", F.FALCON_1), ("f2_b8h12t2048_bf16", F.FALCON_2)):
        w = I.WORKLOADS[wname]
        inp = I.make_inputs(w, seed=33, seqlen=130, batch=1)
        dev = {n: inp[n].cuda() for n in ("q", "k", "v", "beta", "lam")}
        d = F.make_dims(1, 12, 130, 64, 64)
        assert F.falcon_workspace_bytes(variant, d, 64) == 0
        a = _run("fwd", variant, dev, d, 64)
        b = _run("static", variant, dev, d, 64)
        for x, y in zip(a, b):
            assert torch.equal(x, y)
