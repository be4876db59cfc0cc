"""Pins for the CPU oracle, independent of the oracle's own code.

Each test checks the oracle against something fixed by the mathematics of the
gated delta rule (S_t = alpha_t S_{t-1}(I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
o_t = S_t q_t): a dense brute-force product of the per-token factors, closed
forms, invariants, a hand-worked example and central finite differences.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(rng, T, H, Dk, Dv, *, B=1, l2=False, gate=(-0.5, 0.0)):
    q = rng.standard_normal((B, T, H, Dk))
    k = rng.standard_normal((B, T, H, Dk))
    if l2:
        k = k / np.linalg.norm(k, axis=-1, keepdims=True)
        q = q / np.linalg.norm(q, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, Dv))
    g = rng.uniform(gate[0], gate[1], (B, T, H))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, H))))
    return q, k, v, g, beta


def _brute(q, k, v, g, beta, S0):
    """S_T and o_t from explicit products of dense per-token factors.

    Phi_t = alpha_t (I - beta_t k_t k_t^T);  S_t = S0 Phi_1..Phi_t +
    sum_{s<=t} beta_s v_s k_s^T Phi_{s+1}..Phi_t.  Single sequence, single head.
    """
    T, Dk = k.shape
    Dv = v.shape[1]
    Phi = [math.exp(g[t]) * (np.eye(Dk) - beta[t] * np.outer(k[t], k[t])) for t in range(T)]
    o = np.zeros((T, Dv))
    S_t = None
    for t in range(T):
        prod = np.eye(Dk)
        for s in range(t + 1):
            prod = prod @ Phi[s]
        S_t = S0 @ prod
        for s in range(t + 1):
            tail = np.eye(Dk)
            for r in range(s + 1, t + 1):
                tail = tail @ Phi[r]
            S_t = S_t + beta[s] * np.outer(v[s], k[s]) @ tail
        o[t] = S_t @ q[t]
    return o, S_t


@pytest.mark.parametrize("seed,T,Dk,Dv", [(0, 1, 3, 2), (1, 7, 4, 4), (2, 16, 8, 5), (3, 12, 6, 8)])
def test_bruteforce_products(seed, T, Dk, Dv):
    rng = np.random.default_rng(seed)
    q, k, v, g, beta = _rand(rng, T, 1, Dk, Dv)
    S0 = rng.standard_normal((1, 1, Dv, Dk))
    o, ST = oracle.fwd(q, k, v, g, beta, S0)
    ob, Sb = _brute(q[0, :, 0], k[0, :, 0], v[0, :, 0], g[0, :, 0], beta[0, :, 0], S0[0, 0])
    np.testing.assert_allclose(o[0, :, 0], ob, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(ST[0, 0], Sb, rtol=1e-11, atol=1e-11)


def test_hand_worked_golden():
    with open(os.path.join(GOLDEN, "hand_worked_d2_t2.json")) as f:
        gd = json.load(f)
    q = np.array(gd["q"])[None, :, None, :]
    k = np.array(gd["k"])[None, :, None, :]
    v = np.array(gd["v"])[None, :, None, :]
    g = np.array(gd["g"])[None, :, None]
    beta = np.array(gd["beta"])[None, :, None]
    S0 = np.array(gd["S0"])[None, None]
    o, ST = oracle.fwd(q, k, v, g, beta, S0)
    np.testing.assert_allclose(o[0, :, 0], np.array(gd["o"]), rtol=0, atol=1e-14)
    np.testing.assert_allclose(ST[0, 0], np.array(gd["S_T"]), rtol=0, atol=1e-14)


def test_identity_state_alpha1_beta0():
    """alpha = 1 and beta = 0: the state never changes, o_t = S0 q_t."""
    rng = np.random.default_rng(5)
    q, k, v, g, beta = _rand(rng, 20, 2, 6, 5)
    g[:] = 0.0
    beta[:] = 0.0
    S0 = rng.standard_normal((1, 2, 5, 6))
    o, ST = oracle.fwd(q, k, v, g, beta, S0)
    np.testing.assert_allclose(ST, S0, rtol=0, atol=0)
    np.testing.assert_allclose(o[0], np.einsum("hab,thb->tha", S0[0], q[0]), rtol=1e-13, atol=1e-13)


def test_single_token_from_zero():
    """One token from S = 0:  S = beta v k^T and o = beta v (k . q)."""
    rng = np.random.default_rng(6)
    q, k, v, g, beta = _rand(rng, 1, 3, 5, 4)
    o, ST = oracle.fwd(q, k, v, g, beta, None, scale=0.7)
    for h in range(3):
        S = beta[0, 0, h] * np.outer(v[0, 0, h], k[0, 0, h])
        np.testing.assert_allclose(ST[0, h], S, rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(o[0, 0, h], beta[0, 0, h] * v[0, 0, h] * (k[0, 0, h] @ (0.7 * q[0, 0, h])),
                                   rtol=1e-13, atol=1e-14)


def test_exact_recall_orthonormal_keys():
    """alpha = 1, beta = 1, orthonormal keys, S0 = 0: S_T = sum v k^T, S_T k_j = v_j."""
    rng = np.random.default_rng(7)
    d = 8
    Qm, _ = np.linalg.qr(rng.standard_normal((d, d)))
    k = Qm.T[None, :, None, :]                   # rows are orthonormal keys
    v = rng.standard_normal((1, d, 1, 5))
    q = rng.standard_normal((1, d, 1, d))
    g = np.zeros((1, d, 1))
    beta = np.ones((1, d, 1))
    _, ST = oracle.fwd(q, k, v, g, beta)
    np.testing.assert_allclose(ST[0, 0], sum(np.outer(v[0, t, 0], k[0, t, 0]) for t in range(d)), atol=1e-12)
    for j in range(d):
        np.testing.assert_allclose(ST[0, 0] @ k[0, j, 0], v[0, j, 0], atol=1e-12)


def test_repeated_key_overwrites():
    """The same unit key written twice with beta = 1: recall returns the last value."""
    rng = np.random.default_rng(8)
    kk = rng.standard_normal(6)
    kk /= np.linalg.norm(kk)
    k = np.stack([kk, kk])[None, :, None, :]
    v = rng.standard_normal((1, 2, 1, 4))
    q = rng.standard_normal((1, 2, 1, 6))
    S0 = rng.standard_normal((1, 1, 4, 6))
    _, ST = oracle.fwd(q, k, v, np.zeros((1, 2, 1)), np.ones((1, 2, 1)), S0)
    np.testing.assert_allclose(ST[0, 0] @ kk, v[0, 1, 0], atol=1e-12)


def test_memoryless_alpha0():
    """g = -inf (alpha = 0): S_t = beta_t v_t k_t^T regardless of the past."""
    rng = np.random.default_rng(9)
    q, k, v, g, beta = _rand(rng, 9, 2, 5, 3)
    g[:] = -np.inf
    S0 = rng.standard_normal((1, 2, 3, 5))
    o, ST = oracle.fwd(q, k, v, g, beta, S0)
    for h in range(2):
        for t in range(9):
            S = beta[0, t, h] * np.outer(v[0, t, h], k[0, t, h])
            np.testing.assert_allclose(o[0, t, h], S @ q[0, t, h], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(ST[0, h], beta[0, 8, h] * np.outer(v[0, 8, h], k[0, 8, h]), atol=1e-13)


def test_affine_in_start_state():
    """S_end(S_start) = S_end(0) + S_start M, M = the recurrence run with v = 0 from I."""
    rng = np.random.default_rng(10)
    T, Dk, Dv = 40, 6, 4
    q, k, v, g, beta = _rand(rng, T, 2, Dk, Dv, l2=True)
    S0 = rng.standard_normal((1, 2, Dv, Dk))
    _, S_full = oracle.fwd(q, k, v, g, beta, S0)
    _, S_zero = oracle.fwd(q, k, v, g, beta, None)
    I = np.broadcast_to(np.eye(Dk), (1, 2, Dk, Dk)).copy()
    _, M = oracle.fwd(q, k, np.zeros((1, T, 2, Dk)), g, beta, I)
    np.testing.assert_allclose(S_full[0], S_zero[0] + np.einsum("hab,hbc->hac", S0[0], M[0]), atol=1e-12)


def test_continuation():
    """Splitting a sequence and carrying S_T -> S0 gives the same outputs and state."""
    rng = np.random.default_rng(11)
    q, k, v, g, beta = _rand(rng, 50, 3, 5, 5, l2=True)
    S0 = rng.standard_normal((1, 3, 5, 5))
    o, ST = oracle.fwd(q, k, v, g, beta, S0, scale=0.5, l2norm=True)
    o1, S1 = oracle.fwd(q[:, :23], k[:, :23], v[:, :23], g[:, :23], beta[:, :23], S0, scale=0.5, l2norm=True)
    o2, S2 = oracle.fwd(q[:, 23:], k[:, 23:], v[:, 23:], g[:, 23:], beta[:, 23:], S1, scale=0.5, l2norm=True)
    np.testing.assert_allclose(np.concatenate([o1, o2], axis=1), o, atol=1e-12)
    np.testing.assert_allclose(S2, ST, atol=1e-12)


def test_varlen_equals_separate_calls():
    rng = np.random.default_rng(12)
    lens = [5, 17, 1, 9]
    q, k, v, g, beta = _rand(rng, sum(lens), 2, 4, 3)
    S0 = rng.standard_normal((4, 2, 3, 4))
    cu = np.concatenate([[0], np.cumsum(lens)])
    o, ST = oracle.fwd(q, k, v, g, beta, S0, cu_seqlens=cu)
    for n in range(4):
        a, b = cu[n], cu[n + 1]
        on, Sn = oracle.fwd(q[:, a:b], k[:, a:b], v[:, a:b], g[:, a:b], beta[:, a:b], S0[n:n + 1])
        np.testing.assert_allclose(o[:, a:b], on, atol=1e-13)
        np.testing.assert_allclose(ST[n], Sn[0], atol=1e-13)


def test_l2norm_option_matches_prenormalised():
    """The normalisation option equals feeding x/sqrt(|x|^2+1e-6) (and scale*q) directly."""
    rng = np.random.default_rng(13)
    q, k, v, g, beta = _rand(rng, 30, 2, 8, 8)
    nq = q / np.sqrt((q * q).sum(-1, keepdims=True) + 1e-6)
    nk = k / np.sqrt((k * k).sum(-1, keepdims=True) + 1e-6)
    o1, S1 = oracle.fwd(q, k, v, g, beta, scale=0.3, l2norm=True)
    o2, S2 = oracle.fwd(0.3 * nq, nk, v, g, beta)
    np.testing.assert_allclose(o1, o2, atol=1e-13)
    np.testing.assert_allclose(S1, S2, atol=1e-13)


def test_window_bound():
    """Starting w tokens early from zero: error <= exp(sum g over the warm-up) * |S_{b-w}|.

    |I - beta k k^T|_2 <= 1 for unit k and beta in [0, 1], so the start-state
    error contracts at least by prod alpha over the warm-up.
    """
    rng = np.random.default_rng(14)
    T, b, w = 120, 90, 30
    q, k, v, g, beta = _rand(rng, T, 2, 6, 6, l2=True, gate=(-0.3, -0.05))
    _, S_bw = oracle.fwd(q[:, :b - w], k[:, :b - w], v[:, :b - w], g[:, :b - w], beta[:, :b - w])
    _, S_b = oracle.fwd(q[:, :b], k[:, :b], v[:, :b], g[:, :b], beta[:, :b])
    _, S_star = oracle.fwd(q[:, b - w:b], k[:, b - w:b], v[:, b - w:b], g[:, b - w:b], beta[:, b - w:b])
    for h in range(2):
        bound = math.exp(g[0, b - w:b, h].sum()) * np.linalg.norm(S_bw[0, h], 2)
        err = np.linalg.norm(S_b[0, h] - S_star[0, h], 2)
        assert err <= bound * (1 + 1e-9) + 1e-15
        assert err > 0.01 * bound          # the bound is not vacuous here


# ----------------------------------------------------------------------------- backward

def _loss(q, k, v, g, beta, S0, dO, dST, **kw):
    o, ST = oracle.fwd(q, k, v, g, beta, S0, **kw)
    val = (o * dO).sum()
    if dST is not None:
        val += (ST * dST).sum()
    return val


@pytest.mark.parametrize("l2norm", [False, True])
@pytest.mark.parametrize("seed,T,Dk,Dv", [(20, 6, 3, 2), (21, 11, 4, 3)])
def test_backward_finite_differences_all_coords(seed, T, Dk, Dv, l2norm):
    rng = np.random.default_rng(seed)
    H = 2
    q, k, v, g, beta = _rand(rng, T, H, Dk, Dv)
    S0 = rng.standard_normal((1, H, Dv, Dk))
    dO = rng.standard_normal((1, T, H, Dv))
    dST = rng.standard_normal((1, H, Dv, Dk))
    kw = dict(scale=0.8, l2norm=l2norm)
    gr = oracle.bwd(q, k, v, g, beta, dO, S0, dST, **kw)
    args = dict(q=q, k=k, v=v, g=g, beta=beta, S0=S0)
    names = dict(q="dq", k="dk", v="dv", g="dg", beta="dbeta", S0="dS0")
    h = 1e-6
    for name, arr in args.items():
        flat = arr.reshape(-1)
        num = np.zeros_like(flat)
        for i in range(flat.size):
            old = flat[i]
            flat[i] = old + h
            fp = _loss(dO=dO, dST=dST, **args, **kw)
            flat[i] = old - h
            fm = _loss(dO=dO, dST=dST, **args, **kw)
            flat[i] = old
            num[i] = (fp - fm) / (2 * h)
        ana = gr[names[name]].reshape(-1)
        np.testing.assert_allclose(ana, num, rtol=1e-6, atol=1e-7, err_msg=name)


def test_backward_fd_sampled_tiny_workload():
    """200 random coordinates on the tiny fp32 workload's shape (T=256, d=64), l2norm on."""
    rng = np.random.default_rng(22)
    T, H, D = 256, 1, 64
    q = rng.standard_normal((1, T, H, D)); k = rng.standard_normal((1, T, H, D))
    v = rng.standard_normal((1, T, H, D))
    g = rng.uniform(-0.1, -0.001, (1, T, H)); beta = 1 / (1 + np.exp(-rng.standard_normal((1, T, H))))
    S0 = 0.02 * rng.standard_normal((1, H, D, D)); dO = rng.standard_normal((1, T, H, D))
    kw = dict(scale=1 / 8, l2norm=True)
    gr = oracle.bwd(q, k, v, g, beta, dO, S0, None, **kw)
    args = dict(q=q, k=k, v=v, g=g, beta=beta, S0=S0)
    names = dict(q="dq", k="dk", v="dv", g="dg", beta="dbeta", S0="dS0")
    h = 1e-6
    picks = [(n, int(rng.integers(args[n].size))) for n in rng.choice(list(args), 200)]
    for name, i in picks:
        flat = args[name].reshape(-1)
        old = flat[i]
        flat[i] = old + h
        fp = _loss(dO=dO, dST=None, **args, **kw)
        flat[i] = old - h
        fm = _loss(dO=dO, dST=None, **args, **kw)
        flat[i] = old
        num = (fp - fm) / (2 * h)
        ana = gr[names[name]].reshape(-1)[i]
        assert abs(ana - num) <= 1e-5 * max(1.0, abs(num)), (name, i, ana, num)


def test_backward_homogeneity():
    """O is linear in q, and (O, S_T) is jointly linear in (v, S0):
    <q, dq> = <dO, O> and <v, dv> + <S0, dS0> = <dO, O> + <dS_T, S_T> (l2norm off)."""
    rng = np.random.default_rng(23)
    q, k, v, g, beta = _rand(rng, 70, 3, 7, 5, l2=True)
    S0 = rng.standard_normal((1, 3, 5, 7))
    dO = rng.standard_normal((1, 70, 3, 5)); dST = rng.standard_normal((1, 3, 5, 7))
    o, ST = oracle.fwd(q, k, v, g, beta, S0, scale=0.6)
    gr = oracle.bwd(q, k, v, g, beta, dO, S0, dST, scale=0.6)
    rhs = (dO * o).sum()
    np.testing.assert_allclose((q * gr["dq"]).sum(), rhs, rtol=1e-11)
    np.testing.assert_allclose((v * gr["dv"]).sum() + (S0 * gr["dS0"]).sum(), rhs + (dST * ST).sum(), rtol=1e-11)


def test_backward_varlen_equals_separate():
    rng = np.random.default_rng(24)
    lens = [3, 11, 6]
    q, k, v, g, beta = _rand(rng, sum(lens), 2, 4, 4)
    S0 = rng.standard_normal((3, 2, 4, 4)); dO = rng.standard_normal((1, sum(lens), 2, 4))
    cu = np.concatenate([[0], np.cumsum(lens)])
    gr = oracle.bwd(q, k, v, g, beta, dO, S0, None, cu_seqlens=cu, l2norm=True)
    for n in range(3):
        a, b = cu[n], cu[n + 1]
        gn = oracle.bwd(q[:, a:b], k[:, a:b], v[:, a:b], g[:, a:b], beta[:, a:b], dO[:, a:b], S0[n:n + 1],
                        None, l2norm=True)
        for key in ("dq", "dk", "dv", "dg", "dbeta"):
            np.testing.assert_allclose(gr[key][:, a:b], gn[key], atol=1e-13)
        np.testing.assert_allclose(gr["dS0"][n], gn["dS0"][0], atol=1e-13)
