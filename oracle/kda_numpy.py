"""Numpy restatements of the KDA core in fp64, for cross-checking the C++ oracle.

TEST INFRASTRUCTURE ONLY: used by tests/, __graft_entry__.smoke() and bench.py's
CPU-baseline leg, never by the product path.  Shares no code with the CUDA library.

Every function works on ONE problem (one sequence of one head): q, k, g [T, dk],
v [T, dv], beta [T], S0 [dk, dv] (or None), all cast to float64.  The forward ones
return (o [T, dv], S_T [dk, dv]); backward_chunked returns a dict of gradients.

Sources (page title, section / equation):
  * recurrence_three_step  - "Kimi K3 核心算子拆解" (devpress.csdn.net) §2.2 state update
    and §2.3 three-step decomposition (decay, rank-1 correction, write).
  * recurrence_full_matrix - same page §2.3 complexity table ("naive DPLR": form the
    whole d_k x d_k transition); "尝试对Kimi KDA的数学推导&算子实现分析"
    (hjcheng0602.cn/blog/kdd) eq. (3).
  * chunkwise              - hjcheng0602.cn/blog/kdd eqs. (9), (15)-(16), (45)-(52)
    for U, (36)/(63) for the output (inclusive lower triangle, eq. (34) sums j <= t),
    (64)-(66) for the state passed to the next chunk.
  * backward_chunked       - the exact reverse-mode derivative of `chunkwise`, chunk by
    chunk (the pages give only the forward); pinned to torch autograd of the token loop.
  * segment_transition     - "Kimi K3 技术报告解读" (marsggbo.github.io) §7.3: a segment's
    effect is an input-independent transition M plus a zero-start local state S~,
    S_out = M S_in + S~ ; hjcheng0602.cn/blog/kdd eq. (6) for the product form.
"""
from __future__ import annotations

import numpy as np


def _f64(x):
    """Exact fp64 copy of a numpy array or a torch tensor of any float dtype (bf16
    and fp32 widen exactly; fp64 stays as it is)."""
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().cpu().double().numpy()
    return np.asarray(x, dtype=np.float64)


def _prep(q, k, v, g, beta, S0):
    q, k, v, g, beta = (_f64(a) for a in (q, k, v, g, beta))
    dk, dv = k.shape[1], v.shape[1]
    S = np.zeros((dk, dv)) if S0 is None else _f64(S0).copy()
    return q, k, v, g, beta, S


def recurrence_three_step(q, k, v, g, beta, S0, scale):
    """Token loop: S <- Diag(a)S ; S <- S - b k (k^T S) ; S <- S + b k v^T ; o = scale S^T q."""
    q, k, v, g, beta, S = _prep(q, k, v, g, beta, S0)
    T = q.shape[0]
    o = np.zeros((T, v.shape[1]))
    for t in range(T):
        S = S * np.exp(g[t])[:, None]
        kS = k[t] @ S
        S = S - beta[t] * np.outer(k[t], kS)
        S = S + beta[t] * np.outer(k[t], v[t])
        o[t] = scale * (S.T @ q[t])
    return o, S


def recurrence_full_matrix(q, k, v, g, beta, S0, scale):
    """Token loop with the explicit transition M_t = (I - b k k^T) Diag(exp(g_t))."""
    q, k, v, g, beta, S = _prep(q, k, v, g, beta, S0)
    T, dk = k.shape
    o = np.zeros((T, v.shape[1]))
    eye = np.eye(dk)
    for t in range(T):
        M = (eye - beta[t] * np.outer(k[t], k[t])) @ np.diag(np.exp(g[t]))
        S = M @ S + beta[t] * np.outer(k[t], v[t])
        o[t] = scale * (S.T @ q[t])
    return o, S


def chunkwise(q, k, v, g, beta, S0, scale, C):
    """Chunked form with chunk length C (the last chunk may be partial).

    Inside a chunk, G_t is the inclusive cumulative log-decay from the chunk start
    (eq. 9), K+ = K e^G, K- = K e^-G, Q+ = Q e^G (eqs. 15, 16, 54),
    L = StrictTril(B_beta K+ K-^T) (eq. 51), U = (I + L)^-1 B_beta (V - K+ S) (eq. 52),
    O = scale (Q+ S + Tril_incl(Q+ K-^T) U) (eqs. 36, 63),
    S_next = Diag(e^{G_C}) S + (K e^{G_C - G})^T U (eqs. 64-66).
    Exponents up to 5*C stay finite in fp64 for C <= 128.
    """
    q, k, v, g, beta, S = _prep(q, k, v, g, beta, S0)
    T = q.shape[0]
    o = np.zeros((T, v.shape[1]))
    for c0 in range(0, T, C):
        c1 = min(T, c0 + C)
        Qc, Kc, Vc, gc, bc = q[c0:c1], k[c0:c1], v[c0:c1], g[c0:c1], beta[c0:c1]
        n = c1 - c0
        G = np.cumsum(gc, axis=0)
        Kp, Km, Qp = Kc * np.exp(G), Kc * np.exp(-G), Qc * np.exp(G)
        L = np.tril(bc[:, None] * (Kp @ Km.T), k=-1)
        U = np.linalg.solve(np.eye(n) + L, bc[:, None] * (Vc - Kp @ S))
        o[c0:c1] = scale * (Qp @ S + np.tril(Qp @ Km.T) @ U)
        Kend = Kc * np.exp(G[-1] - G)
        S = np.exp(G[-1])[:, None] * S + Kend.T @ U
    return o, S


def segment_transition(k, g, beta, v):
    """(M, S~) of a segment: S_out = M S_in + S~ for any S_in.

    M = D_T ... D_1 with D_t = (I - b_t k_t k_t^T) Diag(exp(g_t)) and S~ the state
    reached from zero (product form of eq. 6)."""
    k, g, beta, v = (_f64(a) for a in (k, g, beta, v))
    T, dk = k.shape
    M = np.eye(dk)
    St = np.zeros((dk, v.shape[1]))
    for t in range(T):
        D = (np.eye(dk) - beta[t] * np.outer(k[t], k[t])) @ np.diag(np.exp(g[t]))
        M = D @ M
        St = D @ St + beta[t] * np.outer(k[t], v[t])
    return M, St


def backward_chunked(q, k, v, g, beta, S0, scale, d_out, d_final, C):
    """Gradients of the chunked form (`chunkwise`) by hand, chunk by chunk in reverse.

    The forward of each chunk is the one in `chunkwise` (hjcheng0602.cn/blog/kdd eqs.
    (9), (15)-(16), (36), (51)-(52), (63)-(66)); the pages derive no backward, so this
    is the exact reverse-mode derivative of those equations, taken factor by factor:
    the read-out O = scale (Q+ S + A_Q U), the write S' = Diag(e^{G_C}) S + K_end^T U,
    the solve U = T Y with T = (I + L)^-1 (dL = -T^T dT T^T on the strict lower
    triangle), Y = B_beta (V - K+ S), and the exponential factors of K+, K-, Q+ and
    K_end into the cumulative log-decay G, whose gradient is summed back to g by a
    reverse cumulative sum.  The state gradient is carried to the previous chunk.

    d_out [T, dv], d_final [dk, dv] or None.  Returns dq, dk, dv, dg [T, dk|dv],
    dbeta [T] and dS0 [dk, dv].
    """
    q, k, v, g, beta, S = _prep(q, k, v, g, beta, S0)
    do = _f64(d_out)
    T, dk = k.shape
    dvd = v.shape[1]
    spans = [(c0, min(T, c0 + C)) for c0 in range(0, T, C)]
    starts = []
    for c0, c1 in spans:
        starts.append(S.copy())
        Kc, Vc, bc = k[c0:c1], v[c0:c1], beta[c0:c1]
        G = np.cumsum(g[c0:c1], axis=0)
        Kp, Km = Kc * np.exp(G), Kc * np.exp(-G)
        L = np.tril(bc[:, None] * (Kp @ Km.T), k=-1)
        U = np.linalg.solve(np.eye(c1 - c0) + L, bc[:, None] * (Vc - Kp @ S))
        S = np.exp(G[-1])[:, None] * S + (Kc * np.exp(G[-1] - G)).T @ U
    dq, dkk, dg = np.zeros((T, dk)), np.zeros((T, dk)), np.zeros((T, dk))
    dvv, dbeta = np.zeros((T, dvd)), np.zeros(T)
    dS1 = np.zeros((dk, dvd)) if d_final is None else _f64(d_final).copy()
    for (c0, c1), S in zip(reversed(spans), reversed(starts)):
        n = c1 - c0
        Qc, Kc, Vc, bc, dO = q[c0:c1], k[c0:c1], v[c0:c1], beta[c0:c1], do[c0:c1]
        G = np.cumsum(g[c0:c1], axis=0)
        gC = G[-1]
        E, Ei, Ee = np.exp(G), np.exp(-G), np.exp(gC - G)
        Kp, Km, Qp, Ke = Kc * E, Kc * Ei, Qc * E, Kc * Ee
        A = Kp @ Km.T
        L = np.tril(bc[:, None] * A, k=-1)
        Tm = np.linalg.inv(np.eye(n) + L)
        R = Vc - Kp @ S
        Y = bc[:, None] * R
        U = Tm @ Y
        AQ = np.tril(Qp @ Km.T)
        # O = scale (Q+ S + A_Q U)
        dAQ = scale * np.tril(dO @ U.T)
        dU = scale * AQ.T @ dO
        dQp = scale * dO @ S.T + dAQ @ Km
        dKm = dAQ.T @ Qp
        dS = scale * Qp.T @ dO
        # S' = Diag(e^{G_C}) S + K_end^T U
        dS += np.exp(gC)[:, None] * dS1
        dgC = np.exp(gC) * np.sum(S * dS1, axis=1)
        dKe = U @ dS1.T
        dU += Ke @ dS1
        # U = T Y, T = (I + L)^-1, L = StrictTril(B_beta A)
        dY = Tm.T @ dU
        dL = np.tril(-Tm.T @ (dU @ Y.T) @ Tm.T, k=-1)
        dA = bc[:, None] * dL
        db = np.sum(A * dL, axis=1)
        dKp = dA @ Km
        dKm += dA.T @ Kp
        # Y = B_beta (V - K+ S)
        db += np.sum(R * dY, axis=1)
        dR = bc[:, None] * dY
        dvv[c0:c1] = dR
        dKp -= dR @ S.T
        dS -= Kp.T @ dR
        # exponential factors into G, then G = cumsum(g)
        dkk[c0:c1] = dKp * E + dKm * Ei + dKe * Ee
        dq[c0:c1] = dQp * E
        dG = dKp * Kp - dKm * Km + dQp * Qp - dKe * Ke
        dG[-1] += dgC + np.sum(dKe * Ke, axis=0)
        dg[c0:c1] = np.cumsum(dG[::-1], axis=0)[::-1]
        dbeta[c0:c1] = db
        dS1 = dS
    return dict(dq=dq, dk=dkk, dv=dvv, dg=dg, dbeta=dbeta, d_initial_state=dS1)
