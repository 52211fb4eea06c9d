"""Pins for the backward oracle (CPU only).

The autograd oracle differentiates a torch restatement of the recurrence. It is pinned here by
things other than itself:
  * its forward agrees with the C oracle's forward (an independent implementation);
  * every gradient agrees with central finite differences of the C oracle's forward (brute force
    on tiny inputs), so a wrong term in either restatement fails;
  * the pages' boundary rules: no gradient through the clamp where it binds, none to beta and
    lambda of the first step of a fresh sequence, none through a zero step size (no 0/0);
  * the chunk-parallel backward the CUDA kernels follow (tests/forms.py) agrees with it at
    several chunk sizes.
"""

import numpy as np
import pytest
import torch

import oracle
from oracle import falcon_bwd as OB
from tests import forms

F1, F1A, F2, F2A = 1, 2, 3, 4


def _case(seed, B=1, H=2, T=6, dk=3, dv=2, variant=F1, pos=0, lam_hi=0.5, beta_hi=1.0, s0=True):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, H, T, dk))
    k = rng.standard_normal((B, H, T, dk))
    v = rng.standard_normal((B, H, T, dv))
    beta = rng.uniform(0.05, beta_hi, (B, H, T, dv) if variant in (F2, F2A) else (B, H, T))
    lam = rng.uniform(0.0, lam_hi, (B, H, T))
    S0 = rng.standard_normal((B, H, dk, dv)) if s0 else None
    tail = rng.standard_normal((B, H, dk)) if pos > 0 else None
    dout = rng.standard_normal((B, H, T, dv))
    dS = rng.standard_normal((B, H, dk, dv))
    return dict(q=q, k=k, v=v, beta=beta, lam=lam, S0=S0, tail=tail, dout=dout, dS=dS, pos=pos)


def _c_loss(variant, c, **over):
    a = {**c, **over}
    tail = None if a["tail"] is None else (a["tail"][:, :, None, :], np.zeros(a["v"].shape[:2] + (0, a["v"].shape[3])))
    out, S, _ = oracle.falcon_ref_fwd(variant, a["q"], a["k"], a["v"], a["beta"], a["lam"], a["S0"], tail,
                                      pos=a["pos"], nthreads=1)
    return float(np.sum(out * a["dout"]) + np.sum(S * a["dS"]))


def _grads(variant, c):
    return OB.falcon_ref_bwd(variant, c["q"], c["k"], c["v"], c["beta"], c["lam"], c["dout"], c["S0"], c["dS"],
                             pos=c["pos"], tail=c["tail"])


@pytest.mark.parametrize("variant", [F1, F1A, F2, F2A])
@pytest.mark.parametrize("pos", [0, 5])
def test_forward_matches_c_oracle(variant, pos):
    c = _case(1, B=2, H=2, T=9, dk=4, dv=3, variant=variant, pos=pos)
    tail = None if pos == 0 else (c["tail"][:, :, None, :], np.zeros((2, 2, 0, 3)))
    ro, rS, _ = oracle.falcon_ref_fwd(variant, c["q"], c["k"], c["v"], c["beta"], c["lam"], c["S0"], tail, pos=pos)
    t = lambda a: torch.as_tensor(a)
    to, tS = OB.forward_torch(variant, t(c["q"]), t(c["k"]), t(c["v"]), t(c["beta"]), t(c["lam"]), t(c["S0"]),
                              pos=pos, tail=None if pos == 0 else t(c["tail"]))
    np.testing.assert_allclose(to.numpy(), ro, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(tS.numpy(), rS, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("variant,pos,lam_hi,beta_hi", [
    (F1, 0, 0.5, 1.0), (F1A, 0, 0.5, 1.0), (F1, 3, 0.5, 1.0), (F1A, 3, 0.5, 1.0),
    (F2, 0, 0.5, 1.0), (F2A, 2, 0.5, 1.0),
    (F1, 0, 50.0, 1.9),   # many steps clamped: alpha = 1 - eps_gamma
])
def test_gradients_match_finite_differences(variant, pos, lam_hi, beta_hi):
    c = _case(2 + pos, variant=variant, pos=pos, lam_hi=lam_hi, beta_hi=beta_hi)
    g = _grads(variant, c)
    names = [("q", "dq"), ("k", "dk"), ("v", "dv"), ("beta", "dbeta"), ("lam", "dlam"), ("S0", "dS0")]
    if pos > 0:
        names.append(("tail", "dtail"))
    h = 1e-6
    for name, gname in names:
        base = c[name]
        fd = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            up, dn = base.copy(), base.copy()
            up[idx] += h
            dn[idx] -= h
            fd[idx] = (_c_loss(variant, c, **{name: up}) - _c_loss(variant, c, **{name: dn})) / (2 * h)
        scale = max(1.0, np.max(np.abs(fd)))
        np.testing.assert_allclose(g[gname], fd, rtol=0, atol=2e-6 * scale, err_msg=name)


def test_clamp_blocks_the_decay_gradient():
    """Where eta lambda >= 1 - eps_gamma the decay is the constant eps_gamma: lambda's gradient is
    then only the one through the step-size denominator, -dbeta * eta (paperlayer §D.2, §G.3)."""
    c = _case(3, variant=F1, lam_hi=50.0, beta_hi=1.9)
    c["lam"][:] = 1000.0
    c["beta"][:] = 1.9
    g = _grads(F1, c)
    x = np.zeros_like(c["k"])
    x[:, :, 1:] = c["k"][:, :, :-1]
    den = np.sum(x * x, -1) + c["lam"] + 1e-6
    eta = c["beta"] / den
    assert np.all(eta * c["lam"] >= 1 - 1e-6)
    # d loss / d lam = d loss / d eta * d eta / d lam, and d eta / d lam = -eta / den
    dbeta = g["dbeta"]
    np.testing.assert_allclose(g["dlam"][:, :, 1:], -(dbeta * c["beta"] / den)[:, :, 1:], rtol=1e-10, atol=1e-14)


def test_first_step_and_zero_step_carry_no_gradient():
    c = _case(4, variant=F1)
    g = _grads(F1, c)
    assert np.all(g["dbeta"][:, :, 0] == 0) and np.all(g["dlam"][:, :, 0] == 0)
    # a zero key with lambda = eps = 0 gives a zero denominator: eta = 0, no 0/0 anywhere
    c["k"][:, :, 2] = 0.0
    c["lam"][:, :, 3] = 0.0
    d = OB.falcon_ref_bwd(F1, c["q"], c["k"], c["v"], c["beta"], c["lam"], c["dout"], c["S0"], c["dS"], eps=0.0)
    for a in d.values():
        if a is not None:
            assert np.all(np.isfinite(a))
    assert np.all(d["dbeta"][:, :, 3] == 0) and np.all(d["dlam"][:, :, 3] == 0)


def test_no_adjoint_no_gradient():
    c = _case(5, variant=F1)
    c["dout"][:] = 0
    c["dS"][:] = 0
    g = _grads(F1, c)
    for a in g.values():
        if a is not None:
            assert np.all(a == 0)


@pytest.mark.parametrize("variant", [F1, F1A])
@pytest.mark.parametrize("C,T,pos", [(1, 7, 0), (4, 11, 0), (4, 12, 3), (8, 8, 0), (64, 13, 2), (5, 23, 0)])
def test_chunk_backward_matches_oracle(variant, C, T, pos):
    c = _case(6 + C, B=1, H=1, T=T, dk=5, dv=4, variant=variant, pos=pos)
    g = _grads(variant, c)
    f = forms.chunk_backward(variant, c["q"][0, 0], c["k"][0, 0], c["v"][0, 0], c["beta"][0, 0], c["lam"][0, 0],
                             c["dout"][0, 0], c["S0"][0, 0], c["dS"][0, 0], C=C, pos=pos,
                             tail=None if pos == 0 else c["tail"][0, 0])
    for n in ("dq", "dk", "dv", "dbeta", "dlam", "dS0"):
        np.testing.assert_allclose(f[n], g[n][0, 0], rtol=1e-9, atol=1e-9, err_msg=n)
    if pos > 0:
        np.testing.assert_allclose(f["dtail"], g["dtail"][0, 0], rtol=1e-9, atol=1e-9)


@pytest.mark.parametrize("variant", [F1, F1A])
def test_chunk_backward_clamped_chunks(variant):
    """Chunks whose total log decay is far below -30 (every step clamped) next to free ones."""
    c = _case(30, B=1, H=1, T=20, dk=4, dv=3, variant=variant, beta_hi=1.5)
    c["lam"][:, :, 4:12] = 1000.0
    g = _grads(variant, c)
    f = forms.chunk_backward(variant, c["q"][0, 0], c["k"][0, 0], c["v"][0, 0], c["beta"][0, 0], c["lam"][0, 0],
                             c["dout"][0, 0], c["S0"][0, 0], c["dS"][0, 0], C=8)
    for n in ("dq", "dk", "dv", "dbeta", "dlam", "dS0"):
        np.testing.assert_allclose(f[n], g[n][0, 0], rtol=1e-9, atol=1e-9, err_msg=n)


@pytest.mark.parametrize("variant", [F2, F2A])
@pytest.mark.parametrize("C,pos", [(4, 0), (8, 3), (64, 0)])
def test_per_column_backward_matches_oracle(variant, C, pos):
    """Falcon-2 / 2A: the gradient split into one Falcon-1 / 1A backward per value column (the columns
    share only the keys) equals autograd of the per-column recurrence."""
    c = _case(90 + C, B=1, H=1, T=19, dk=5, dv=3, variant=variant, pos=pos)
    g = _grads(variant, c)
    f = forms.chunk_backward_per_column(variant, c["q"][0, 0], c["k"][0, 0], c["v"][0, 0], c["beta"][0, 0],
                                        c["lam"][0, 0], c["dout"][0, 0], c["S0"][0, 0], c["dS"][0, 0], C=C, pos=pos,
                                        tail=None if pos == 0 else c["tail"][0, 0])
    for n in ("dq", "dk", "dv", "dbeta", "dlam", "dS0"):
        np.testing.assert_allclose(f[n], g[n][0, 0], rtol=1e-9, atol=1e-9, err_msg=n)
    if pos > 0:
        np.testing.assert_allclose(f["dtail"], g["dtail"][0, 0], rtol=1e-9, atol=1e-9)
