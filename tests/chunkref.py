"""fp64 numpy statement of the chunked (WY) algebra that the CUDA kernels implement.

This is a test helper, not the oracle: it restates, chunk by chunk, the four
steps of the chunked form (onedev.kr FlashQLA talk summary, paragraph on the
WY representation: intra-chunk K K^T and its inverse, W and U, the
chunk-to-chunk state pass, the output), the diagonal gamma factoring (same
page, paragraph on SFU load), the segment transition used for intra-card
sequence parallelism (paragraph on parallelism) and the chunk backward with
the dA + dA^T batching (paragraph on SFU load, last sentence).  The tests
check it against the token-by-token oracle; the CUDA kernels follow the same
algebra in fp32/bf16.

Per chunk of C tokens, with G = inclusive cumsum of g inside the chunk,
gamma = exp(G), c_i = gamma_C / gamma_i, state S in R^{dv x dk}:

  N   = strict_tril(K K^T)
  Ahat = (I + diag(beta) N)^{-1}                  (no exp inside the inverse)
  W   = diag(gamma) Ahat diag(beta) K
  U   = diag(gamma) Ahat diag(beta/gamma) V
  Ut  = U - W S0^T                                (corrected values)
  O   = diag(gamma) Q S0^T + (tril_incl(Gamma) * Q K^T) Ut,  Gamma_ri = gamma_r/gamma_i
  S_C = gamma_C S0 + Ut^T diag(c) K
"""
from __future__ import annotations

import numpy as np

C = 64


def _prep(x, l2, mul=1.0):
    if l2:
        x = x / np.sqrt((x * x).sum(-1, keepdims=True) + 1e-6)
    return x * mul


def chunk_wy(K, V, g, beta):
    G = np.cumsum(g)
    gam = np.exp(G)
    N = np.tril(K @ K.T, -1)
    Ahat = np.linalg.inv(np.eye(len(g)) + beta[:, None] * N)
    W = gam[:, None] * (Ahat @ (beta[:, None] * K))
    U = gam[:, None] * (Ahat @ ((beta / gam)[:, None] * V))
    return G, gam, Ahat, W, U


def chunk_fwd(Q, K, V, g, beta, S0):
    G, gam, Ahat, W, U = chunk_wy(K, V, g, beta)
    Ut = U - W @ S0.T
    Gam = np.tril(np.exp(G[:, None] - G[None, :]))
    O = gam[:, None] * (Q @ S0.T) + (Gam * (Q @ K.T)) @ Ut
    c = np.exp(G[-1] - G)
    S1 = gam[-1] * S0 + Ut.T @ (c[:, None] * K)
    return O, S1


def chunk_transition(K, g, beta):
    """M with S_C = S0 M + (S_C from S0 = 0):  M = gamma_C I - W^T diag(c) K."""
    G, gam, Ahat, W, _ = chunk_wy(K, np.zeros_like(K), g, beta)
    c = np.exp(G[-1] - G)
    return gam[-1] * np.eye(K.shape[1]) - W.T @ (c[:, None] * K)


def fwd(q, k, v, g, beta, S0=None, *, scale=1.0, l2norm=False):
    """Single sequence, single head: q,k [T,dk], v [T,dv], g,beta [T]."""
    T, dk = k.shape
    dv = v.shape[1]
    Q, K = _prep(q, l2norm, scale), _prep(k, l2norm)
    S = np.zeros((dv, dk)) if S0 is None else S0.copy()
    O = np.zeros((T, dv))
    for a in range(0, T, C):
        b = min(a + C, T)
        O[a:b], S = chunk_fwd(Q[a:b], K[a:b], v[a:b], g[a:b], beta[a:b], S)
    return O, S


def chunk_bwd(Q, K, V, g, beta, S0, dO, dS1):
    """Gradients of one chunk given dO and dS_C (gradient w.r.t. its end state).

    Returns dQ, dK, dV, dg, dbeta (w.r.t. the normalised/scaled Q, K) and dS0.
    """
    Cn = len(g)
    G, gam, Ahat, W, U = chunk_wy(K, V, g, beta)
    Ut = U - W @ S0.T
    Gam = np.tril(np.exp(G[:, None] - G[None, :]))
    P = Gam * (Q @ K.T)
    c = np.exp(G[-1] - G)
    # state chain
    Y = K @ dS1.T                                  # C x dv
    dUt = P.T @ dO + c[:, None] * Y
    dS0 = gam[-1] * dS1 + dO.T @ (gam[:, None] * Q) - dUt.T @ W
    # Gate gradient.  dG_r collects the terms whose decay factor starts or ends at token r: the
    # derivative of gamma_r (decay from the chunk start) and of each ratio gamma_r / gamma_i
    # (i < r: + at r, - at i; the diagonal ratio is 1 and contributes nothing, so it is left out
    # of every row and column sum).  dg_t = sum_{r >= t} dG_r, plus the state terms, which depend
    # on g_t through gamma_C (every t) and through c_r = gamma_C / gamma_r for r < t only.
    lo = np.tril(np.ones((Cn, Cn)), -1)
    dQ = gam[:, None] * (dO @ S0)
    dG = (dQ * Q).sum(1)                          # gamma_r <dO_r, S0 q_r>
    dP = dO @ Ut.T
    Z = dP * P * lo
    dG += Z.sum(1) - Z.sum(0)
    dPm = Gam * dP
    dQ += dPm @ K
    dK = dPm.T @ Q + c[:, None] * (Ut @ dS1)
    y = c * (Ut * Y).sum(1)                       # c_r <dS_C, ut_r k_r^T>
    # through Ut = U - W S0^T, with W = diag(gamma) Ahat diag(beta) K and U = X2 V,
    # X2 = Gamma * Ahat diag(beta)
    dW = -dUt @ S0
    dU = dUt
    dWp = gam[:, None] * dW
    M1 = dWp @ K.T                                # gamma_r <dW_r, k_i>
    M2 = dU @ V.T                                 # <dU_r, v_i>
    X2 = Gam * Ahat * beta[None, :]
    dG += (Ahat * M1 * beta[None, :]).sum(1)      # <dW_r, W_r>
    XM = X2 * M2 * lo
    dG += XM.sum(1) - XM.sum(0)
    dUp = gam[:, None] * dU
    AdW = Ahat.T @ dWp
    AdU = Ahat.T @ dUp
    dK += beta[:, None] * AdW
    dV = (beta / gam)[:, None] * AdU
    dbeta = (K * AdW).sum(1) + (V * AdU).sum(1) / gam
    dAhat = dWp @ (beta[:, None] * K).T + dUp @ ((beta / gam)[:, None] * V).T
    dT = -Ahat.T @ dAhat @ Ahat.T
    N = np.tril(K @ K.T, -1)
    dTl = np.tril(dT, -1)
    dbeta += (dTl * N).sum(1)
    dN = beta[:, None] * dTl
    dK += (dN + dN.T) @ K                          # dA and dA^T batched into one product with K
    dg = np.cumsum(dG[::-1])[::-1] + gam[-1] * (dS1 * S0).sum() + (np.cumsum(y) - y)
    return dQ, dK, dV, dg, dbeta, dS0


def bwd(q, k, v, g, beta, dO, S0=None, dST=None, *, scale=1.0, l2norm=False):
    T, dk = k.shape
    dv = v.shape[1]
    Q, K = _prep(q, l2norm, scale), _prep(k, l2norm)
    S = np.zeros((dv, dk)) if S0 is None else S0.copy()
    starts = list(range(0, T, C))
    states = []
    for a in starts:
        b = min(a + C, T)
        states.append(S)
        _, S = chunk_fwd(Q[a:b], K[a:b], v[a:b], g[a:b], beta[a:b], S)
    dS = np.zeros((dv, dk)) if dST is None else dST.copy()
    dQ = np.zeros_like(Q); dK = np.zeros_like(K); dV = np.zeros_like(v)
    dg = np.zeros(T); db = np.zeros(T)
    for i in reversed(range(len(starts))):
        a = starts[i]
        b = min(a + C, T)
        dQ[a:b], dK[a:b], dV[a:b], dg[a:b], db[a:b], dS = chunk_bwd(
            Q[a:b], K[a:b], v[a:b], g[a:b], beta[a:b], states[i], dO[a:b], dS)
    # normalisation Jacobians
    if l2norm:
        nq = np.sqrt((q * q).sum(-1, keepdims=True) + 1e-6)
        nk = np.sqrt((k * k).sum(-1, keepdims=True) + 1e-6)
        qt, kt = q / nq, k / nk
        dQs = scale * dQ
        dq = (dQs - qt * (qt * dQs).sum(-1, keepdims=True)) / nq
        dkk = (dK - kt * (kt * dK).sum(-1, keepdims=True)) / nk
    else:
        dq, dkk = scale * dQ, dK
    return dq, dkk, dV, dg, db, dS
