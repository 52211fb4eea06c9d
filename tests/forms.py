"""Independent fp64 forms used to pin the oracle (test helpers, CPU only).

1. ``ogd_steps``: each step is literally "one normalized gradient step on the
   instantaneous objective" (agihunt explainer, Method; paperlayer §3.1, §4.4),
   with the gradient taken by torch autograd and the smoothness scale taken as
   the top eigenvalue (numpy ``eigvalsh``) of the data term's curvature
   (paperlayer §3.1: "L_t = ||x_t||^2 + lambda_t"; §C.6 / sungsoo post: Falcon-3
   uses lambda_max of the window covariance). It shares no arithmetic with the
   oracle's hand-written update. Valid only while the decay clamp is inactive.

2. ``chunk_forward``: the chunk-parallel form (paperlayer Figure 2, §D.1, §E.2,
   §F.2, §H.3): per chunk, one unit-lower-triangular solve whose right-hand side
   merges the value path and the projected-history path, log-prefix decay reset
   to zero at every chunk start, a read-after-write masked output and a carried
   state. With ``C >= T`` it is the masked-parallel form (one dense solve over
   the whole sequence, paperlayer Figure 2 "Masked-parallel form"). Its algebra
   comes from unrolling the recurrence inside a chunk; only exp(L_a - L_b) with
   a >= b is ever formed, so nothing overflows when the clamp binds.
"""

from __future__ import annotations

import numpy as np
import torch

F1, F1A, F2, F3 = 1, 2, 3, 5


def _np(a):
    if a is None:
        return None
    if hasattr(a, "detach"):
        a = a.detach().cpu().double().numpy()
    return np.asarray(a, dtype=np.float64)


def _global_pairs(k, v, pos, tail, W):
    """Key/value lookup by global 1-based index (0 for indices <= 0)."""
    T, dk = k.shape
    dv = v.shape[1]

    def key(i):
        if i <= 0:
            return np.zeros(dk)
        if i <= pos:
            return tail[0][i - (pos - W + 1)]
        return k[i - pos - 1]

    def val(i):
        if i <= 0:
            return np.zeros(dv)
        if i <= pos:
            return tail[1][i - (pos - W + 2)]
        return v[i - pos - 1]

    return key, val


# --------------------------------------------------------------------------------------
# 1. autograd gradient steps
# --------------------------------------------------------------------------------------

def ogd_steps(variant, q, k, v, beta, lam, S0=None, *, pos=0, tail=None, W=1, eps=1e-6, eps_gamma=1e-6):
    """One sequence: q,k [T,dk], v [T,dv], beta [T] or [T,dv], lam [T]."""
    q, k, v, beta, lam, S0 = (_np(a) for a in (q, k, v, beta, lam, S0))
    T, dk = q.shape
    dv = v.shape[1]
    key, val = _global_pairs(k, v, pos, tail, W)
    S = np.zeros((dk, dv)) if S0 is None else S0.copy()
    out = np.zeros((T, dv))
    for t in range(T):
        tau = pos + t + 1
        win = W if variant == F3 else 1
        js = [j for j in range(tau - win + 1, tau + 1) if j >= 2]
        if js:
            xs = [key(j - 1) for j in js]
            ys = [val(j) for j in js]
            nb = len(js)
            Sv = torch.tensor(S, requires_grad=True)
            lt = float(lam[t])
            if variant == F1A:
                x, y = torch.tensor(xs[0]), torch.tensor(ys[0])
                data = -(y @ (Sv.T @ x))
            else:
                data = sum(0.5 * torch.sum((torch.tensor(y) - Sv.T @ torch.tensor(x)) ** 2)
                           for x, y in zip(xs, ys)) / nb
            loss = data + 0.5 * lt * torch.sum(Sv ** 2)
            (grad,) = torch.autograd.grad(loss, Sv)
            grad = grad.numpy()
            if variant == F1A:
                smooth = float(np.dot(xs[0], xs[0]))  # write-energy normaliser (paperlayer "inner-product variants")
            else:
                cov = sum(np.outer(x, x) for x in xs) / nb  # curvature of the data term, per column
                smooth = float(np.linalg.eigvalsh(cov).max())
            den = smooth + lt + eps
            if variant == F2:
                eta = np.where(den == 0, 0.0, beta[t] / den)  # [dv]
                assert np.all(eta * lt < 1 - eps_gamma), "clamp active: autograd form does not apply"
                S = S - grad * eta[None, :]
            else:
                eta = 0.0 if den == 0 else float(beta[t]) / den
                assert eta * lt < 1 - eps_gamma, "clamp active: autograd form does not apply"
                S = S - eta * grad
        out[t] = S.T @ q[t]
    return out, S


# --------------------------------------------------------------------------------------
# 2. chunk-parallel (and, with C >= T, masked-parallel) form
# --------------------------------------------------------------------------------------

def _scalars(betas, lams, den, first_mask, eps_gamma):
    eta = np.where(den == 0, 0.0, betas / np.where(den == 0, 1.0, den))
    eta = np.where(first_mask, 0.0, eta)
    alpha = np.minimum(eta * lams, 1.0 - eps_gamma)
    alpha = np.where(first_mask, 0.0, alpha)
    return eta, alpha


def _lambda_max_small(g):
    return float(np.linalg.eigvalsh(g).max()) if g.size else 0.0


def chunk_forward(variant, q, k, v, beta, lam, S0=None, *, C, pos=0, tail=None, W=1, eps=1e-6,
                  eps_gamma=1e-6):
    """One sequence, fp64. Returns (out [T,dv], S_final [dk,dv])."""
    q, k, v, beta, lam, S0 = (_np(a) for a in (q, k, v, beta, lam, S0))
    T, dk = q.shape
    dv = v.shape[1]
    key, val = _global_pairs(k, v, pos, tail, W)
    S = np.zeros((dk, dv)) if S0 is None else S0.copy()
    out = np.zeros((T, dv))
    for t0 in range(0, T, C):
        t1 = min(T, t0 + C)
        n = t1 - t0
        taus = np.arange(pos + t0 + 1, pos + t1 + 1)
        Q = q[t0:t1]
        lm = lam[t0:t1]
        if variant in (F1, F1A, F2):
            X = np.stack([key(int(tau) - 1) for tau in taus])
            Y = v[t0:t1]
            first = taus == 1
            den = np.sum(X * X, axis=1) + lm + eps
            G = X @ X.T
            Sc = Q @ X.T
            if variant == F2:
                eta, alpha = _scalars(beta[t0:t1], lm[:, None], den[:, None], first[:, None], eps_gamma)
            else:
                eta, alpha = _scalars(beta[t0:t1], lm, den, first, eps_gamma)
            Lc = np.cumsum(np.log1p(-alpha), axis=0)            # inclusive prefix, reset per chunk
            Lx = np.concatenate([np.zeros_like(Lc[:1]), Lc[:-1]], axis=0)  # exclusive prefix
            LC = Lc[-1]
            lower = np.tril(np.ones((n, n)), -1)
            incl = np.tril(np.ones((n, n)), 0)
            if variant == F2:
                R = np.zeros((n, dv))
                O = np.zeros((n, dv))
                Snew = np.zeros_like(S)
                for c in range(dv):
                    Ec = np.exp(np.minimum(Lx[:, c][:, None] - Lc[:, c][None, :], 0.0)) * lower
                    A = eta[None, :, c] * Ec * G
                    rhs = Y[:, c] - np.exp(Lx[:, c]) * (X @ S[:, c])
                    r = np.linalg.solve(np.eye(n) + A, rhs)
                    Pc = eta[None, :, c] * np.exp(np.minimum(Lc[:, c][:, None] - Lc[:, c][None, :], 0.0)) * incl * Sc
                    O[:, c] = np.exp(Lc[:, c]) * (Q @ S[:, c]) + Pc @ r
                    w = eta[:, c] * np.exp(LC[c] - Lc[:, c])
                    Snew[:, c] = np.exp(LC[c]) * S[:, c] + X.T @ (w * r)
                out[t0:t1] = O
                S = Snew
                continue
            E = np.exp(np.minimum(Lx[:, None] - Lc[None, :], 0.0)) * lower
            A = eta[None, :] * E * G
            P = eta[None, :] * np.exp(np.minimum(Lc[:, None] - Lc[None, :], 0.0)) * incl * Sc
            if variant == F1:
                R = np.linalg.solve(np.eye(n) + A, Y - np.exp(Lx)[:, None] * (X @ S))
            else:
                R = Y
            out[t0:t1] = np.exp(Lc)[:, None] * (Q @ S) + P @ R
            w = eta * np.exp(LC - Lc)
            S = np.exp(LC) * S + X.T @ (w[:, None] * R)
        else:  # Falcon-3: rank-W system over (token, window slot) unknowns
            ne = n + W - 1
            js = np.arange(int(taus[0]) - W + 1, int(taus[-1]) + 1)     # global pair indices
            valid_e = js >= 2
            Xe = np.stack([key(int(j) - 1) if j >= 2 else np.zeros(dk) for j in js])
            Ye = np.stack([val(int(j)) if j >= 2 else np.zeros(dv) for j in js])
            Ge = Xe @ Xe.T
            Sce = Q @ Xe.T
            eta = np.zeros(n)
            alpha = np.zeros(n)
            kap = np.zeros(n)
            for i in range(n):
                ps = [i - a + W - 1 for a in range(W) if valid_e[i - a + W - 1]]
                if not ps:
                    continue
                nb = len(ps)
                mu = _lambda_max_small(Ge[np.ix_(ps, ps)] / nb)
                den = mu + lm[i] + eps
                eta[i] = 0.0 if den == 0 else beta[t0 + i] / den
                alpha[i] = min(eta[i] * lm[i], 1.0 - eps_gamma)
                kap[i] = eta[i] / nb
            Lc = np.cumsum(np.log1p(-alpha))
            Lx = np.concatenate([[0.0], Lc[:-1]])
            LC = Lc[-1]
            m = n * W
            A = np.zeros((m, m))
            rhs = np.zeros((m, dv))
            XeS = Xe @ S
            for i in range(n):
                for a in range(W):
                    pa = i - a + W - 1
                    if not valid_e[pa]:
                        continue
                    rhs[i * W + a] = Ye[pa] - np.exp(Lx[i]) * XeS[pa]
                    for l in range(i):
                        f = kap[l] * np.exp(Lx[i] - Lc[l])
                        for b in range(W):
                            pb = l - b + W - 1
                            if valid_e[pb]:
                                A[i * W + a, l * W + b] = f * Ge[pa, pb]
            R = np.linalg.solve(np.eye(m) + A, rhs)
            Ps = np.zeros((n, m))
            Xw = np.zeros((m, dk))
            for l in range(n):
                for b in range(W):
                    pb = l - b + W - 1
                    if not valid_e[pb]:
                        continue
                    Xw[l * W + b] = kap[l] * np.exp(LC - Lc[l]) * Xe[pb]
                    for i in range(l, n):
                        Ps[i, l * W + b] = kap[l] * np.exp(Lc[i] - Lc[l]) * Sce[i, pb]
            out[t0:t1] = np.exp(Lc)[:, None] * (Q @ S) + Ps @ R
            S = np.exp(LC) * S + Xw.T @ R
    return out, S


# --------------------------------------------------------------------------------------
# 3. chunk-parallel backward (Falcon-1, 1A)
# --------------------------------------------------------------------------------------

def chunk_backward(variant, q, k, v, beta, lam, dout, S0=None, dS_final=None, *, C, pos=0, tail=None,
                   eps=1e-6, eps_gamma=1e-6):
    """Gradients of sum(out * dout) + sum(S_final * dS_final) for one sequence by the chunk algebra
    the CUDA backward follows (paperlayer §D.2, §E.3, §G.3: reverse the output materialisation, the
    inter-chunk recurrence and the local structure). Three phases:
      1. per chunk, independent of the state: T = (I + A)^-1, the transition S -> M S + U and the
         state-free part V of the chunk's state adjoint, dS_n = M^T dS_{n+1} + V;
      2. the two scans: S_{n+1} = M S_n + U forward, dS_n = M^T dS_{n+1} + V backward;
      3. per chunk, from S_n and dS_{n+1}: every input gradient of the chunk.
    q, k [T,dk], v [T,dv], beta, lam [T], dout [T,dv]; tail = the pending key k_pos (pos > 0).
    Returns a dict like the oracle's (dq, dk, dv, dbeta, dlam, dS0, dtail)."""
    q, k, v, beta, lam, dout, S0, dS_final = (_np(a) for a in (q, k, v, beta, lam, dout, S0, dS_final))
    tail = None if tail is None else _np(tail).reshape(-1)
    T, dk = q.shape
    dv = v.shape[1]
    xs = np.zeros((T, dk))
    if T:
        xs[1:] = k[:-1]
        if pos > 0:
            xs[0] = tail
    taus = pos + np.arange(T) + 1
    first = taus == 1
    den = np.sum(xs * xs, axis=1) + lam + eps
    eta, alpha = _scalars(beta, lam, den, first, eps_gamma)
    lg = np.log1p(-alpha)
    chunks = [(t0, min(T, t0 + C)) for t0 in range(0, T, C)]
    inner = variant == F1A

    def local(t0, t1):
        X, Q, Y, dO = xs[t0:t1], q[t0:t1], v[t0:t1], dout[t0:t1]
        n = t1 - t0
        e = eta[t0:t1]
        L = np.cumsum(lg[t0:t1])
        Lx = np.concatenate([[0.0], L[:-1]])
        LC = L[-1]
        Ex = np.exp(np.minimum(Lx[:, None] - L[None, :], 0.0)) * np.tril(np.ones((n, n)), -1)
        Ep = np.exp(np.minimum(L[:, None] - L[None, :], 0.0)) * np.tril(np.ones((n, n)), 0)
        G, Sc = X @ X.T, Q @ X.T
        A = e[None, :] * Ex * G
        P = e[None, :] * Ep * Sc
        Tm = np.eye(n) if inner else np.linalg.inv(np.eye(n) + A)
        w = e * np.exp(LC - L)
        return dict(X=X, Q=Q, Y=Y, dO=dO, e=e, L=L, Lx=Lx, LC=LC, Ex=Ex, Ep=Ep, G=G, Sc=Sc, A=A, P=P,
                    T=Tm, w=w)

    # phase 1: state-free chunk operators
    ops = []
    for t0, t1 in chunks:
        c = local(t0, t1)
        D = np.exp(c["Lx"])[:, None] * c["X"]          # diag(e^Lx) X
        if inner:
            M = np.exp(c["LC"]) * np.eye(dk)
            V = c["Q"].T @ (np.exp(c["L"])[:, None] * c["dO"])
        else:
            M = np.exp(c["LC"]) * np.eye(dk) - c["X"].T @ (c["w"][:, None] * (c["T"] @ D))
            V = c["Q"].T @ (np.exp(c["L"])[:, None] * c["dO"]) - D.T @ (c["T"].T @ (c["P"].T @ c["dO"]))
        U = c["X"].T @ (c["w"][:, None] * (c["T"] @ c["Y"]))
        ops.append((M, U, V))
    # phase 2: scans
    S_in = [np.zeros((dk, dv)) if S0 is None else S0.copy()]
    for M, U, _ in ops:
        S_in.append(M @ S_in[-1] + U)
    dS_out = [None] * len(chunks)
    g = np.zeros((dk, dv)) if dS_final is None else dS_final.copy()
    for i in range(len(chunks) - 1, -1, -1):
        dS_out[i] = g
        M, _, V = ops[i]
        g = M.T @ g + V
    dS0 = g
    # phase 3: chunk gradients
    dq, dx, dvv = np.zeros_like(q), np.zeros_like(xs), np.zeros_like(v)
    deta, dL_all = np.zeros(T), np.zeros(T)
    for ci, (t0, t1) in enumerate(chunks):
        c = local(t0, t1)
        S, dSn = S_in[ci], dS_out[ci]
        X, Q, Y, dO, e, L, Lx, LC = (c[n] for n in ("X", "Q", "Y", "dO", "e", "L", "Lx", "LC"))
        n = t1 - t0
        H = np.exp(Lx)[:, None] * (X @ S)
        R = Y if inner else c["T"] @ (Y - H)
        XdS = X @ dSn
        dR = c["P"].T @ dO + c["w"][:, None] * XdS
        dOS = dO @ S.T
        dP = (dO @ R.T) * np.tril(np.ones((n, n)), 0)
        EP = dP * c["Ep"]                       # dP_ij e^{L_i - L_j}
        dSc = EP * e[None, :]
        dQ = np.exp(L)[:, None] * dOS + dSc @ X
        dX = dSc.T @ Q + c["w"][:, None] * (R @ dSn.T)
        de = np.sum(EP * c["Sc"], axis=0)
        dw = np.sum(XdS * R, axis=1)
        de += dw * np.exp(LC - L)
        PP = np.sum(dP * c["P"], axis=0)        # sum_i dP_ij P_ij  (by column j)
        dL = np.exp(L) * np.sum(Q * dOS, axis=1) + np.sum(dP * c["P"], axis=1) - PP
        dL[-1] += np.sum(dw * c["w"]) + np.exp(LC) * np.sum(dSn * S)
        dL -= dw * c["w"]
        dLx = np.zeros(n)
        if inner:
            dY = dR
        else:
            dZ = c["T"].T @ dR
            dY = dZ
            dA = -(dZ @ R.T) * np.tril(np.ones((n, n)), -1)
            EA = dA * c["Ex"]
            dG = EA * e[None, :]
            dX += (dG + dG.T) @ X
            de += np.sum(EA * c["G"], axis=0)
            AA = dA * c["A"]
            dLx += np.sum(AA, axis=1)
            dL -= np.sum(AA, axis=0)
            dZS = dZ @ S.T
            dX -= np.exp(Lx)[:, None] * dZS
            dLx -= np.exp(Lx) * np.sum(X * dZS, axis=1)
        dL[:-1] += dLx[1:]
        dq[t0:t1], dx[t0:t1], dvv[t0:t1] = dQ, dX, dY
        deta[t0:t1] = de
        dL_all[t0:t1] = dL
    # chunk-local prefixes: d log(gamma_u) = sum of dL_i over the chunk's i >= u
    dlg = np.zeros(T)
    for t0, t1 in chunks:
        dlg[t0:t1] = np.cumsum(dL_all[t0:t1][::-1])[::-1]
    unclamped = (eta * lam < 1.0 - eps_gamma) & ~first
    dalpha = np.where(unclamped, -dlg / (1.0 - alpha), 0.0)
    deta = deta + np.where(unclamped, dalpha * lam, 0.0)
    dlam = np.where(unclamped, dalpha * eta, 0.0)
    live = (den != 0) & ~first
    dbeta = np.where(live, deta / np.where(live, den, 1.0), 0.0)
    dden = np.where(live, -deta * eta / np.where(live, den, 1.0), 0.0)
    dlam = dlam + dden
    dx = dx + 2.0 * dden[:, None] * xs
    dk_ = np.zeros_like(k)
    if T:
        dk_[:-1] = dx[1:]
    return {"dq": dq, "dk": dk_, "dv": dvv, "dbeta": dbeta, "dlam": dlam,
            "dS0": dS0, "dtail": dx[0] if (T and pos > 0) else None}


# --------------------------------------------------------------------------------------
# 4. scan over chunk maps (Falcon-1, 1A, 3, 3A)
# --------------------------------------------------------------------------------------

def scan_forward(variant, q, k, v, beta, lam, S0=None, *, C, G=16, pos=0, tail=None, W=1, eps=1e-6, eps_gamma=1e-6):
    """Falcon-1, 1A and 3 (the variants chunk_forward covers). The scan path's algebra for one sequence, fp64 (paperlayer §H.1: chunk maps compose
    associatively). Every chunk n acts affinely on its start state, S_{n+1} = M_n S_n + U_n and
    O_n = Ao_n S_n + Bo_n; the four maps are read off the chunk form run over that chunk alone (its
    window and shifted-key history passed as a tail): from the unit states e_c without targets (the
    columns of M_n and Ao_n) and from the zero state with the targets (U_n, Bo_n). The start states
    are then formed in groups of G chunks: each group's composed map, the group start states, and
    each chunk's start state from its group's; the outputs come from the output maps.
    Returns (out [T,dv], S_final [dk,dv])."""
    q, k, v, beta, lam, S0 = (_np(a) for a in (q, k, v, beta, lam, S0))
    T, dk = q.shape
    dv = v.shape[1]
    key, val = _global_pairs(k, v, pos, tail, W)
    S = np.zeros((dk, dv)) if S0 is None else S0
    maps = []
    for t0 in range(0, T, C):
        t1 = min(T, t0 + C)
        P = pos + t0  # tokens before the chunk
        tl = None
        if P > 0:
            tl = (np.stack([key(g) for g in range(P - W + 1, P + 1)]),
                  np.stack([val(g) for g in range(P - W + 2, P + 1)]) if W > 1 else np.zeros((0, dv)))

        def run(Sst, targets):  # without targets, the window's earlier values are zero too
            vv = v[t0:t1] if targets else np.zeros((t1 - t0, dv))
            tt = tl if (targets or tl is None) else (tl[0], np.zeros_like(tl[1]))
            return chunk_forward(variant, q[t0:t1], k[t0:t1], vv, beta[t0:t1], lam[t0:t1], Sst, C=t1 - t0, pos=P,
                                 tail=tt, W=W, eps=eps, eps_gamma=eps_gamma)

        M = np.zeros((dk, dk))
        Ao = np.zeros((t1 - t0, dk))
        for c in range(dk):  # every value column starts at e_c: the columns of M and Ao
            Sst = np.zeros((dk, dv))
            Sst[c, :] = 1.0
            o, Se = run(Sst, False)
            M[:, c] = Se[:, 0]
            Ao[:, c] = o[:, 0]
        Bo, U = run(np.zeros((dk, dv)), True)
        maps.append((M, U, Ao, Bo))
    N = len(maps)
    starts = []
    for g0 in range(0, N, G):  # group maps, then the group start states
        Mg, Ug = np.eye(dk), np.zeros((dk, dv))
        for n in range(g0, min(N, g0 + G)):
            Mg, Ug = maps[n][0] @ Mg, maps[n][0] @ Ug + maps[n][1]
        starts.append(S)
        S = Mg @ S + Ug
    out = np.zeros((T, dv))
    for gi, g0 in enumerate(range(0, N, G)):  # each group's chunks from its start state
        Sn = starts[gi]
        for n in range(g0, min(N, g0 + G)):
            M, U, Ao, Bo = maps[n]
            out[n * C:n * C + Ao.shape[0]] = Ao @ Sn + Bo
            Sn = M @ Sn + U
    return out, S


def chunk_backward_per_column(variant, q, k, v, beta, lam, dout, S0=None, dS_final=None, *, C, pos=0, tail=None,
                              eps=1e-6, eps_gamma=1e-6):
    """Falcon-2 / 2A gradients by columns: every value column evolves on its own given the shared keys
    (its own beta, so its own step sizes, decay and triangular system), so the loss splits into one
    term per column and each column's term is the Falcon-1 / 1A backward of that column with its beta.
    The per-column gradients of v, beta, S0 are that column's; those of q, k, lambda and the tail key
    are summed over the columns. beta [T,dv]."""
    q, k, v, beta, lam, dout, S0, dS_final = (_np(a) for a in (q, k, v, beta, lam, dout, S0, dS_final))
    T, dk = q.shape
    dv = v.shape[1]
    base = F1 if variant == F2 else F1A
    acc = {"dq": np.zeros_like(q), "dk": np.zeros_like(k), "dv": np.zeros_like(v), "dbeta": np.zeros_like(beta),
           "dlam": np.zeros_like(lam), "dS0": np.zeros((dk, dv)), "dtail": None if pos == 0 else np.zeros(dk)}
    for c in range(dv):
        g = chunk_backward(base, q, k, v[:, c:c + 1], beta[:, c], lam, dout[:, c:c + 1],
                           None if S0 is None else S0[:, c:c + 1], None if dS_final is None else dS_final[:, c:c + 1],
                           C=C, pos=pos, tail=tail, eps=eps, eps_gamma=eps_gamma)
        acc["dq"] += g["dq"]
        acc["dk"] += g["dk"]
        acc["dlam"] += g["dlam"]
        acc["dv"][:, c] = g["dv"][:, 0]
        acc["dbeta"][:, c] = g["dbeta"]
        acc["dS0"][:, c] = g["dS0"][:, 0]
        if pos > 0:
            acc["dtail"] += g["dtail"]
    return acc
