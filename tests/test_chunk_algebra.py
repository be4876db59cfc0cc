"""The chunked WY algebra (tests/chunkref.py) reproduces the token-by-token oracle
in fp64, forward and backward, including partial chunks and the segment
transition used for intra-card sequence parallelism."""
import numpy as np
import pytest

import oracle
from tests import chunkref


def _case(seed, T, dk, dv, gate=(-0.2, -0.001)):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((T, dk)); k = rng.standard_normal((T, dk)); v = rng.standard_normal((T, dv))
    g = rng.uniform(*gate, T); beta = 1 / (1 + np.exp(-rng.standard_normal(T)))
    S0 = 0.3 * rng.standard_normal((dv, dk)); dO = rng.standard_normal((T, dv))
    dST = rng.standard_normal((dv, dk))
    return q, k, v, g, beta, S0, dO, dST


def _o(x):
    return x[None, :, None]


@pytest.mark.parametrize("T", [1, 63, 64, 65, 200])
def test_chunk_forward_matches_oracle(T):
    q, k, v, g, beta, S0, _, _ = _case(T, T, 16, 12)
    O, S = chunkref.fwd(q, k, v, g, beta, S0, scale=0.25, l2norm=True)
    o_ref, S_ref = oracle.fwd(_o(q), _o(k), _o(v), g[None, :, None], beta[None, :, None], S0[None, None],
                              scale=0.25, l2norm=True)
    np.testing.assert_allclose(O, o_ref[0, :, 0], atol=1e-11)
    np.testing.assert_allclose(S, S_ref[0, 0], atol=1e-11)


def test_inverse_is_textbook_solve():
    """Ahat equals a triangular solve of (I + diag(beta) N) X = I."""
    import scipy.linalg
    q, k, v, g, beta, *_ = _case(3, 64, 32, 32)
    k = k / np.linalg.norm(k, axis=1, keepdims=True)
    _, _, Ahat, _, _ = chunkref.chunk_wy(k, v, g, beta)
    T = np.eye(64) + beta[:, None] * np.tril(k @ k.T, -1)
    X = scipy.linalg.solve_triangular(T, np.eye(64), lower=True, unit_diagonal=True)
    np.testing.assert_allclose(Ahat, X, atol=1e-12)


def test_segment_transition_composes():
    """S_end(S_start) = S_end(0) + S_start * prod_chunks M_c."""
    q, k, v, g, beta, S0, _, _ = _case(4, 64 * 5, 16, 16)
    k = k / np.linalg.norm(k, axis=1, keepdims=True)
    _, S_full = chunkref.fwd(q, k, v, g, beta, S0)
    _, S_zero = chunkref.fwd(q, k, v, g, beta, None)
    M = np.eye(16)
    for a in range(0, 320, 64):
        M = M @ chunkref.chunk_transition(k[a:a + 64], g[a:a + 64], beta[a:a + 64])
    np.testing.assert_allclose(S_full, S_zero + S0 @ M, atol=1e-11)


@pytest.mark.parametrize("T,l2", [(1, False), (64, True), (100, True), (130, False)])
def test_chunk_backward_matches_oracle(T, l2):
    q, k, v, g, beta, S0, dO, dST = _case(100 + T, T, 16, 12)
    if not l2:
        k = k / 4.0          # keep beta |k|^2 < 2 so the recurrence is contractive
    got = chunkref.bwd(q, k, v, g, beta, dO, S0, dST, scale=0.5, l2norm=l2)
    ref = oracle.bwd(_o(q), _o(k), _o(v), g[None, :, None], beta[None, :, None], _o(dO), S0[None, None],
                     dST[None, None], scale=0.5, l2norm=l2)
    for name, a, b in zip(["dq", "dk", "dv", "dg", "dbeta", "dS0"], got,
                          [ref["dq"][0, :, 0], ref["dk"][0, :, 0], ref["dv"][0, :, 0], ref["dg"][0, :, 0],
                           ref["dbeta"][0, :, 0], ref["dS0"][0, 0]]):
        np.testing.assert_allclose(a, b, atol=1e-10, rtol=1e-9, err_msg=name)
