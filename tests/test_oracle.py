"""Pins for the fp64 oracle (CPU only).

Each test checks the oracle against something other than itself: a hand-worked
example, a closed form, a library routine (autograd, eigvalsh, dense solve) or
an invariant the pages state. Together they are chosen so that a dropped term,
a wrong sign, a shifted index or a transposed operand in the recurrence fails
at least one of them.
"""

import json
import os

import numpy as np
import pytest
import torch

import oracle
from tests import forms

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
F1, F1A, F2, F3 = 1, 2, 3, 5


def _rand(seed, B, H, T, dk, dv, variant=F1, beta_hi=1.0, lam_hi=0.5, s0=True):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, H, T, dk))
    k = rng.standard_normal((B, H, T, dk))
    v = rng.standard_normal((B, H, T, dv))
    bshape = (B, H, T, dv) if variant == F2 else (B, H, T)
    beta = rng.uniform(0.05, beta_hi, bshape)
    lam = rng.uniform(0.0, lam_hi, (B, H, T))
    S0 = rng.standard_normal((B, H, dk, dv)) if s0 else None
    return q, k, v, beta, lam, S0


# ---------------------------------------------------------------- hand-worked goldens

@pytest.mark.parametrize("case", json.load(open(os.path.join(GOLDEN, "hand_worked.json")))["cases"],
                         ids=lambda c: c["name"])
def test_hand_worked(case):
    a = lambda x: np.asarray(x, dtype=np.float64)[None, None]
    out, S, (tk, tv) = oracle.falcon_ref_fwd(
        case["variant"], a(case["q"]), a(case["k"]), a(case["v"]), a(case["beta"]), a(case["lam"]),
        window=case["window"], eps=case["eps"], eps_gamma=case["eps_gamma"])
    np.testing.assert_allclose(out[0, 0], case["out"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(S[0, 0], case["S_final"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(tk[0, 0], case["tail_keys"], rtol=0, atol=0)
    if "tail_vals" in case:
        np.testing.assert_allclose(tv[0, 0], case["tail_vals"], rtol=0, atol=0)


# ---------------------------------------------------------------- closed forms / special cases

@pytest.mark.parametrize("variant", [F1, F1A, F2, F3])
def test_sentinel_step_is_noop(variant):
    """x_1 = 0 with eta_1 = alpha_1 = 0: the first step leaves S0 untouched (paperlayer §3, §4.6, §H.3)."""
    q, k, v, beta, lam, S0 = _rand(1, 2, 3, 1, 5, 4, variant, lam_hi=3.0)
    out, S, _ = oracle.falcon_ref_fwd(variant, q, k, v, beta, lam, S0, window=3 if variant == F3 else 1)
    assert np.array_equal(S, S0)
    np.testing.assert_allclose(out[:, :, 0], np.einsum("bhkv,bhk->bhv", S0, q[:, :, 0]), rtol=1e-14, atol=1e-14)


@pytest.mark.parametrize("variant", [F1, F2, F3])
def test_nlms_projection(variant):
    """lambda = eps = 0, beta = 1: after each step S_t^T x_t = y_t exactly, for any earlier state
    (classical NLMS, paperlayer §3.1, §2.3). With q_t = x_t = k_{t-1}, the read returns v_t."""
    B, H, T, d = 1, 2, 12, 6
    q, k, v, beta, lam, S0 = _rand(2, B, H, T, d, d, variant)
    beta = np.ones_like(beta)
    lam = np.zeros_like(lam)
    q = np.concatenate([np.zeros_like(k[:, :, :1]), k[:, :, :-1]], axis=2)  # q_t = k_{t-1}
    out, _, _ = oracle.falcon_ref_fwd(variant, q, k, v, beta, lam, S0, eps=0.0, window=1)
    np.testing.assert_allclose(out[:, :, 1:], v[:, :, 1:], rtol=0, atol=1e-11)


def test_nlms_single_step_from_zero():
    """From S = 0 one step writes x y^T / ||x||^2 (beta = 1, lambda = eps = 0)."""
    k = np.array([[[[3.0, 4.0, 0.0], [1.0, 1.0, 1.0]]]])
    v = np.array([[[[9.0, 9.0], [2.0, -1.0]]]])
    q = np.zeros((1, 1, 2, 3))
    out, S, _ = oracle.falcon_ref_fwd(F1, q, k, v, np.ones((1, 1, 2)), np.zeros((1, 1, 2)), eps=0.0)
    expect = np.outer([3.0, 4.0, 0.0], [2.0, -1.0]) / 25.0
    np.testing.assert_allclose(S[0, 0], expect, rtol=0, atol=1e-16)


def test_memorisation_orthonormal_keys():
    """Orthonormal write features, beta = 1, lambda = eps = 0: every stored pair is recalled
    exactly at the end (the delta rule edits only along the current key)."""
    d, dv = 8, 3
    rng = np.random.default_rng(3)
    Qm, _ = np.linalg.qr(rng.standard_normal((d, d)))
    T = d + 1
    k = np.zeros((1, 1, T, d))
    k[0, 0, :d] = Qm.T          # k_1..k_d orthonormal, k_T arbitrary (never written)
    k[0, 0, d] = rng.standard_normal(d)
    v = rng.standard_normal((1, 1, T, dv))
    _, S, _ = oracle.falcon_ref_fwd(F1, np.zeros((1, 1, T, d)), k, v, np.ones((1, 1, T)),
                                    np.zeros((1, 1, T)), eps=0.0)
    for j in range(2, T + 1):        # pair j = (k_{j-1}, v_j)
        np.testing.assert_allclose(S[0, 0].T @ k[0, 0, j - 2], v[0, 0, j - 1], atol=1e-12)


def test_falcon1a_no_ridge_is_shifted_linear_attention():
    """lambda = 0: Falcon-1A is additive (paperlayer §4.3): o_t = S0^T q_t +
    sum_{2<=j<=t} eta_j (q_t . k_{j-1}) v_j with eta_j = beta_j/(||k_{j-1}||^2 + eps)."""
    B, H, T, dk, dv = 2, 2, 16, 5, 4
    q, k, v, beta, lam, S0 = _rand(4, B, H, T, dk, dv, F1A)
    lam = np.zeros_like(lam)
    eps = 1e-3
    out, _, _ = oracle.falcon_ref_fwd(F1A, q, k, v, beta, lam, S0, eps=eps)
    x = np.concatenate([np.zeros_like(k[:, :, :1]), k[:, :, :-1]], axis=2)
    eta = beta / (np.sum(x * x, -1) + eps)
    eta[:, :, 0] = 0.0
    scores = np.einsum("bhtd,bhjd->bhtj", q, x) * np.tril(np.ones((T, T)))
    expect = np.einsum("bhtj,bhj,bhjv->bhtv", scores, eta, v) + np.einsum("bhkv,bhtk->bhtv", S0, q)
    np.testing.assert_allclose(out, expect, rtol=1e-12, atol=1e-12)


def test_clamp_binds_to_eps_gamma():
    """lambda huge, beta = 1.5: alpha = min(eta*lambda, 1-eps_gamma) clamps, so gamma = eps_gamma and
    (Falcon-1A) S_T = eps_gamma^(T-1) S0 + sum_j eps_gamma^(T-j) eta_j x_j y_j^T (paperlayer §C.1, §4.6)."""
    B, H, T, dk, dv = 1, 1, 5, 3, 2
    q, k, v, beta, lam, S0 = _rand(5, B, H, T, dk, dv, F1A)
    beta = np.full_like(beta, 1.5)
    lam = np.full_like(lam, 1e12)
    eg = 1e-2
    _, S, _ = oracle.falcon_ref_fwd(F1A, q, k, v, beta, lam, S0, eps=1e-6, eps_gamma=eg)
    expect = eg ** (T - 1) * S0[0, 0]
    for j in range(2, T + 1):
        x = k[0, 0, j - 2]
        eta = 1.5 / (x @ x + 1e12 + 1e-6)
        expect = expect + eg ** (T - j) * eta * np.outer(x, v[0, 0, j - 1])
    np.testing.assert_allclose(S[0, 0], expect, rtol=1e-12, atol=1e-300)


def test_zero_key_zero_denominator_gives_no_write():
    """||x||^2 + lambda + eps = 0 sets eta = 0 (paperlayer Appendix p.34): no NaN, no write."""
    B, H, T, d = 1, 1, 4, 3
    q, k, v, beta, lam, S0 = _rand(6, B, H, T, d, d, F1)
    k[0, 0, 1] = 0.0               # x_3 = k_2 = 0
    lam[:] = 0.0
    out_a, S_a, _ = oracle.falcon_ref_fwd(F1, q[:, :, :2], k[:, :, :2], v[:, :, :2], beta[:, :, :2],
                                          lam[:, :, :2], S0, eps=0.0)
    out_b, S_b, _ = oracle.falcon_ref_fwd(F1, q[:, :, :3], k[:, :, :3], v[:, :, :3], beta[:, :, :3],
                                          lam[:, :, :3], S0, eps=0.0)
    assert np.all(np.isfinite(out_b))
    assert np.array_equal(S_a, S_b)


# ---------------------------------------------------------------- library routines

@pytest.mark.parametrize("variant", [F1, F1A, F2, F3])
def test_matches_autograd_gradient_steps(variant):
    """Each step is one normalized gradient step of the stated objective (autograd + eigvalsh)."""
    B, H, T, dk, dv = 1, 2, 14, 4, 3
    W = 3 if variant == F3 else 1
    q, k, v, beta, lam, S0 = _rand(7, B, H, T, dk, dv, variant, beta_hi=1.0, lam_hi=0.8)
    out, S, _ = oracle.falcon_ref_fwd(variant, q, k, v, beta, lam, S0, window=W)
    for h in range(H):
        o_ref, S_ref = forms.ogd_steps(variant, q[0, h], k[0, h], v[0, h], beta[0, h], lam[0, h], S0[0, h], W=W)
        np.testing.assert_allclose(out[0, h], o_ref, rtol=1e-10, atol=1e-11)
        np.testing.assert_allclose(S[0, h], S_ref, rtol=1e-10, atol=1e-11)


@pytest.mark.parametrize("n", [1, 2, 3, 4, 6])
def test_lambda_max_vs_eigvalsh(n):
    rng = np.random.default_rng(n)
    for _ in range(20):
        X = rng.standard_normal((n, 7))
        g = X @ X.T / n
        assert abs(oracle.lambda_max(g) - np.linalg.eigvalsh(g).max()) <= 1e-12 * max(1.0, np.abs(g).max())


def test_falcon3_orthogonal_window_keys():
    """Orthogonal keys in the window: mu = max_j ||x_j||^2 / B, so eta = beta/(mu + lambda + eps)."""
    d = 6
    rng = np.random.default_rng(8)
    Qm, _ = np.linalg.qr(rng.standard_normal((d, d)))
    scales = np.array([1.0, 3.0, 2.0, 0.5])
    T = 5
    k = np.zeros((1, 1, T, d))
    k[0, 0, :4] = Qm[:, :4].T * scales[:, None]
    v = rng.standard_normal((1, 1, T, 2))
    lam = np.full((1, 1, T), 0.3)
    beta = np.full((1, 1, T), 0.7)
    # Falcon-1A-free check through a zero state: at t = 5 the window is pairs 2..5 (keys k1..k4),
    # and with S_4 known the step is gamma S_4 + (eta/4) sum x r^T.
    _, S4, _ = oracle.falcon_ref_fwd(F3, np.zeros((1, 1, 4, d)), k[:, :, :4], v[:, :, :4], beta[:, :, :4],
                                     lam[:, :, :4], window=4)
    _, S5, _ = oracle.falcon_ref_fwd(F3, np.zeros((1, 1, T, d)), k, v, beta, lam, window=4)
    mu = np.max(scales ** 2) / 4
    eta = 0.7 / (mu + 0.3 + 1e-6)
    X = k[0, 0, :4]
    Y = v[0, 0, 1:5]
    R = Y - X @ S4[0, 0]
    expect = (1 - eta * 0.3) * S4[0, 0] + (eta / 4) * X.T @ R
    np.testing.assert_allclose(S5[0, 0], expect, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- brute-force forms

@pytest.mark.parametrize("variant", [F1, F1A, F2, F3])
@pytest.mark.parametrize("C", [1, 4, 8, 64])
def test_chunk_and_masked_parallel_forms(variant, C):
    """Chunk-parallel form at C in {1,4,8} and the masked-parallel form (C >= T, one dense solve)
    agree with the recurrence, including a clamp-active stretch (lambda up to 500, beta up to 1.9)."""
    B, H, T, dk, dv = 1, 2, 24, 5, 4
    W = 3 if variant == F3 else 1
    q, k, v, beta, lam, S0 = _rand(9, B, H, T, dk, dv, variant, beta_hi=1.9, lam_hi=1.0)
    lam[0, 0, 6:14] = 500.0
    out, S, _ = oracle.falcon_ref_fwd(variant, q, k, v, beta, lam, S0, window=W)
    for h in range(H):
        o_c, S_c = forms.chunk_forward(variant, q[0, h], k[0, h], v[0, h], beta[0, h], lam[0, h], S0[0, h],
                                       C=C, W=W)
        scale = max(1.0, np.abs(out[0, h]).max())
        np.testing.assert_allclose(o_c, out[0, h], rtol=0, atol=1e-10 * scale)
        np.testing.assert_allclose(S_c, S[0, h], rtol=0, atol=1e-10 * max(1.0, np.abs(S[0, h]).max()))


# ---------------------------------------------------------------- invariants between variants

def test_falcon2_equal_columns_is_falcon1():
    q, k, v, beta, lam, S0 = _rand(10, 2, 2, 20, 5, 4, F1, beta_hi=1.9, lam_hi=2.0)
    o1, S1, _ = oracle.falcon_ref_fwd(F1, q, k, v, beta, lam, S0)
    beta2 = np.repeat(beta[..., None], 4, axis=-1)
    o2, S2, _ = oracle.falcon_ref_fwd(F2, q, k, v, beta2, lam, S0)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-13)
    np.testing.assert_allclose(S2, S1, rtol=0, atol=1e-13)


def test_falcon2_column_is_falcon1_on_that_column():
    """Column c of Falcon-2 evolves alone, as Falcon-1 with beta = beta[..., c] on v[..., c]."""
    q, k, v, beta, lam, S0 = _rand(11, 1, 2, 18, 5, 3, F2, beta_hi=1.5, lam_hi=2.0)
    o2, S2, _ = oracle.falcon_ref_fwd(F2, q, k, v, beta, lam, S0)
    for c in range(3):
        o1, S1, _ = oracle.falcon_ref_fwd(F1, q, k, v[..., c:c + 1], beta[..., c], lam, S0[..., c:c + 1])
        np.testing.assert_allclose(o2[..., c:c + 1], o1, rtol=0, atol=1e-13)
        np.testing.assert_allclose(S2[..., c:c + 1], S1, rtol=0, atol=1e-13)


def test_falcon3_window1_is_falcon1():
    q, k, v, beta, lam, S0 = _rand(12, 2, 2, 20, 5, 4, F1, beta_hi=1.9, lam_hi=2.0)
    o1, S1, _ = oracle.falcon_ref_fwd(F1, q, k, v, beta, lam, S0)
    o3, S3, _ = oracle.falcon_ref_fwd(F3, q, k, v, beta, lam, S0, window=1)
    np.testing.assert_allclose(o3, o1, rtol=0, atol=1e-13)
    np.testing.assert_allclose(S3, S1, rtol=0, atol=1e-13)


@pytest.mark.parametrize("variant,W", [(F1, 1), (F1A, 1), (F2, 1), (F3, 2), (F3, 4)])
@pytest.mark.parametrize("split", [1, 2, 3, 11])
def test_split_continuation_is_exact(variant, W, split):
    """S_final plus the tail of the last pairs continues a split sequence exactly (paperlayer §C.7, §4.4)."""
    q, k, v, beta, lam, S0 = _rand(13, 2, 2, 23, 5, 4, variant, beta_hi=1.9, lam_hi=2.0)
    full_o, full_S, full_tail = oracle.falcon_ref_fwd(variant, q, k, v, beta, lam, S0, window=W)
    s = split
    o1, S1, t1 = oracle.falcon_ref_fwd(variant, q[:, :, :s], k[:, :, :s], v[:, :, :s], beta[:, :, :s],
                                       lam[:, :, :s], S0, window=W)
    o2, S2, t2 = oracle.falcon_ref_fwd(variant, q[:, :, s:], k[:, :, s:], v[:, :, s:], beta[:, :, s:],
                                       lam[:, :, s:], S1, t1, pos=s, window=W)
    np.testing.assert_allclose(np.concatenate([o1, o2], axis=2), full_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(S2, full_S, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(t2[0], full_tail[0])
    np.testing.assert_array_equal(t2[1], full_tail[1])


def test_state_only_continuation_differs_for_falcon3():
    """Passing only the matrix state changes the boundary updates of Falcon-3 (paperlayer §C.7):
    the tail is needed, and dropping it is detectable."""
    q, k, v, beta, lam, S0 = _rand(14, 1, 1, 16, 4, 3, F3)
    full_o, _, _ = oracle.falcon_ref_fwd(F3, q, k, v, beta, lam, S0, window=4)
    o1, S1, t1 = oracle.falcon_ref_fwd(F3, q[:, :, :8], k[:, :, :8], v[:, :, :8], beta[:, :, :8],
                                       lam[:, :, :8], S0, window=4)
    zero_tail = (np.zeros_like(t1[0]), np.zeros_like(t1[1]))
    o2, _, _ = oracle.falcon_ref_fwd(F3, q[:, :, 8:], k[:, :, 8:], v[:, :, 8:], beta[:, :, 8:],
                                     lam[:, :, 8:], S1, zero_tail, pos=8, window=4)
    assert np.abs(o2 - full_o[:, :, 8:]).max() > 1e-3


def test_threads_do_not_change_results():
    q, k, v, beta, lam, S0 = _rand(15, 3, 4, 9, 4, 3, F3)
    a = oracle.falcon_ref_fwd(F3, q, k, v, beta, lam, S0, window=3, nthreads=1)
    b = oracle.falcon_ref_fwd(F3, q, k, v, beta, lam, S0, window=3, nthreads=5)
    for x, y in zip(a[:2], b[:2]):
        assert np.array_equal(x, y)


def test_rejects_bad_arguments():
    q, k, v, beta, lam, S0 = _rand(16, 1, 1, 4, 3, 3, F1)
    with pytest.raises(ValueError):
        oracle.falcon_ref_fwd(F1, q, k, v, beta, lam, S0, window=2)      # window only for Falcon-3
    with pytest.raises(ValueError):
        oracle.falcon_ref_fwd(7, q, k, v, beta, lam, S0)                  # no such variant
    with pytest.raises(ValueError):
        oracle.falcon_ref_fwd(F1, q, k, v, beta, lam, S0, pos=3)          # pos > 0 needs a tail


def test_torch_inputs_are_widened_exactly():
    t = torch.tensor([[[[1.0078125, -3.5]]]], dtype=torch.bfloat16)
    assert oracle._f64(t).tolist() == [[[[1.0078125, -3.5]]]]


# ---------------------------------------------------------------- the inner-product variants 2A and 3A

F2A, F3A = 4, 6


def test_falcon2a_equal_columns_is_falcon1a():
    """Falcon-2A with every column's gain equal to one beta is Falcon-1A, bitwise (same operations)."""
    q, k, v, beta, lam, S0 = _rand(41, 2, 3, 13, 5, 4, F1A, lam_hi=2.0)
    o1, S1, _ = oracle.falcon_ref_fwd(F1A, q, k, v, beta, lam, S0)
    b2 = np.repeat(beta[..., None], 4, axis=-1)
    o2, S2, _ = oracle.falcon_ref_fwd(F2A, q, k, v, b2, lam, S0)
    assert np.array_equal(o1, o2) and np.array_equal(S1, S2)


def test_falcon2a_column_is_falcon1a_on_that_column():
    """Each value column of Falcon-2A follows Falcon-1A on that column alone with that column's gains."""
    q, k, v, _, lam, S0 = _rand(42, 1, 2, 11, 5, 3, F1A, lam_hi=3.0)
    rng = np.random.default_rng(43)
    b2 = rng.uniform(0.05, 1.9, (1, 2, 11, 3))
    o2, S2, _ = oracle.falcon_ref_fwd(F2A, q, k, v, b2, lam, S0)
    for c in range(3):
        oc, Sc, _ = oracle.falcon_ref_fwd(F1A, q, k, v[..., c:c + 1], b2[..., c], lam, S0[..., c:c + 1])
        np.testing.assert_allclose(o2[..., c:c + 1], oc, rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(S2[..., c:c + 1], Sc, rtol=1e-13, atol=1e-13)


def test_falcon3a_window1_is_falcon1a():
    """A window of one pair reduces Falcon-3A to Falcon-1A (paperlayer §4.5)."""
    q, k, v, beta, lam, S0 = _rand(44, 2, 2, 17, 6, 5, F1A, beta_hi=1.9, lam_hi=4.0)
    o1, S1, _ = oracle.falcon_ref_fwd(F1A, q, k, v, beta, lam, S0)
    o3, S3, _ = oracle.falcon_ref_fwd(F3A, q, k, v, beta, lam, S0, window=1)
    np.testing.assert_allclose(o3, o1, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(S3, S1, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("W", [2, 3, 5])
def test_falcon3a_is_the_masked_attention_form(W):
    """Falcon-3A's parallel form (paperlayer §4.6): O = Diag(delta) Q S0 + (Q X^T (.) M) Y, with
    delta_t = prod_{s<=t} gamma_s and M_tj = sum over updates u <= t whose window holds pair j of
    (prod_{u<s<=t} gamma_s) eta_u / B_u. Built here by brute force over (t, u, j)."""
    T, dk, dv = 14, 4, 3
    q, k, v, beta, lam, S0 = _rand(45, 1, 1, T, dk, dv, F1A, beta_hi=1.9, lam_hi=3.0)
    eps, eps_g = 1e-6, 1e-6
    out, S, _ = oracle.falcon_ref_fwd(F3A, q, k, v, beta, lam, S0, window=W, eps=eps, eps_gamma=eps_g)
    X = np.vstack([np.zeros((1, dk)), k[0, 0, :-1]])  # x_tau = k_{tau-1}, x_1 = 0 (rows tau-1)
    Y = v[0, 0]
    gam, eta_b, win = np.ones(T), np.zeros(T), []
    for t in range(T):  # update at global step tau = t + 1
        tau = t + 1
        members = [j for j in range(max(2, tau - W + 1), tau + 1)] if tau >= 2 else []
        win.append(members)
        if not members:
            continue
        E = np.mean([X[j - 1] @ X[j - 1] for j in members])
        eta = beta[0, 0, t] / (E + lam[0, 0, t] + eps)
        alpha = min(eta * lam[0, 0, t], 1 - eps_g)
        gam[t] = 1 - alpha
        eta_b[t] = eta / len(members)
    ref = np.zeros((T, dv))
    for t in range(T):
        delta = np.prod(gam[: t + 1])
        ref[t] = delta * (S0[0, 0].T @ q[0, 0, t])
        for j in range(1, T + 1):
            m = sum(np.prod(gam[u + 1: t + 1]) * eta_b[u] for u in range(t + 1) if j in win[u])
            ref[t] += m * (q[0, 0, t] @ X[j - 1]) * Y[j - 1]
    np.testing.assert_allclose(out[0, 0], ref, rtol=1e-11, atol=1e-12)


def test_inner_product_variants_sentinel_and_arguments():
    """x_1 = 0: the first step is a no-op for 2A and 3A too; 2A takes per-column gains, 3A a window."""
    q, k, v, beta, lam, S0 = _rand(46, 2, 3, 1, 5, 4, F1A)
    b2 = np.repeat(beta[..., None], 4, axis=-1)
    _, S, _ = oracle.falcon_ref_fwd(F2A, q, k, v, b2, lam, S0)
    assert np.array_equal(S, S0)
    _, S, _ = oracle.falcon_ref_fwd(F3A, q, k, v, beta, lam, S0, window=3)
    assert np.array_equal(S, S0)
    with pytest.raises(AssertionError):
        oracle.falcon_ref_fwd(F2A, q, k, v, beta, lam, S0)  # gains must be per column


# ---------------------------------------------------------------- the scan path's algebra

@pytest.mark.parametrize("variant,W,pos", [(F1, 1, 0), (F1A, 1, 0), (F3, 3, 0), (F3, 4, 0), (F1, 1, 5), (F3, 3, 6)])
@pytest.mark.parametrize("C,G", [(4, 3), (5, 16), (3, 1)])
def test_scan_over_chunk_maps_is_exact(variant, W, pos, C, G):
    """Per-chunk affine maps of the state and of the outputs, composed in groups of G chunks, then the
    outputs from each chunk's start state (the scan path) give the oracle's outputs and final state
    (paperlayer §H.1: chunk maps compose associatively)."""
    q, k, v, beta, lam, S0 = _rand(40 + C + G, 1, 1, 29, 5, 4, variant)
    tail = None
    if pos > 0:
        rng = np.random.default_rng(7)
        tail = (rng.standard_normal((1, 1, W, 5)), rng.standard_normal((1, 1, W - 1, 4)))
    o, S = forms.scan_forward(variant, q[0, 0], k[0, 0], v[0, 0], beta[0, 0], lam[0, 0], S0[0, 0], C=C, G=G,
                              pos=pos, tail=None if tail is None else (tail[0][0, 0], tail[1][0, 0]), W=W)
    ro, rS, _ = oracle.falcon_ref_fwd(variant, q, k, v, beta, lam, S0, tail, pos=pos, window=W)
    np.testing.assert_allclose(o, ro[0, 0], rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(S, rS[0, 0], rtol=1e-10, atol=1e-10)
