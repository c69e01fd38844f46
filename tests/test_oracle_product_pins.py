"""Pins of the oracle's token-ordered ("product") reading of the frame transition.

The summary page "SANA-WM: Efficient Minute-Scale World Modeling with Hybrid
Linear Diffusion Transformer" prints the frame transition as
gamma_t I - K^_t beta_t K^_t^T (section 方法步骤详情, module 2) and calls the
layer a frame-wise generalisation of token-wise GDN (section 技术新颖性).  The
product reading applies the frame's tokens in order, prod_n (I - beta_n k^_n k^_n^T),
which the oracle evaluates through the UT transform over sub-chunks.  These
CPU tests pin that evaluation to things that do not reuse it: dense token-by-
token matrix products, the plain token-wise delta rule, and closed forms.
"""
import numpy as np
import pytest

import oracle
from tests.test_oracle_pins import rand_inputs, unit


def brute_force_frame(k, v, beta, gamma, key_scale):
    """Dense sequential products for one chain: (P_f, W_f) per frame, token order."""
    _, FN, _, D = k.shape
    F = gamma.shape[1]
    N = FN // F
    out = []
    for f in range(F):
        P = np.eye(D)
        W = np.zeros((D, D))
        for n in range(f * N, (f + 1) * N):
            kh = unit(k[0, n, 0]) * key_scale
            b = float(beta[0, n, 0])
            E = np.eye(D) - b * np.outer(kh, kh)
            P = P @ E
            W = W @ E + b * np.outer(v[0, n, 0].astype(np.float64), kh)
        out.append((P, W))
    return out


def ut_transform_frame(kh, vv, bb, sub):
    """(Abar, W) of one frame through the UT transform over sub-chunks of `sub` tokens.

    kh [N, D] are the scaled unit keys, vv [N, D] the values, bb [N] the write
    strengths.  For each sub-chunk c, T_c = (I + StrictLower(diag(b_c) K_c K_c^T))^-1 diag(b_c)
    gives prod_{n in c} (I - b_n k_n k_n^T) = I - K_c^T T_c K_c, and the pair
    (Abar = I - P, W) of the tokens so far is advanced by the delta rule with the
    keys as Abar's values: X = T_c ([K_c | V_c] - K_c [Abar; W]^T), pair += X^T K_c.
    This is the blocked (WY) evaluation that the GPU kernel uses; the oracle does
    not use it.
    """
    N, D = kh.shape
    Ab = np.zeros((D, D))
    W = np.zeros((D, D))
    for n0 in range(0, N, sub):
        Kc, Vc, bc = kh[n0:n0 + sub], vv[n0:n0 + sub], bb[n0:n0 + sub]
        m = len(bc)
        L = np.eye(m) + np.tril(bc[:, None] * (Kc @ Kc.T), -1)
        T = np.linalg.solve(L, np.diag(bc))
        Xa = T @ (Kc - Kc @ Ab.T)
        Xw = T @ (Vc - Kc @ W.T)
        Ab = Ab + Xa.T @ Kc
        W = W + Xw.T @ Kc
    return Ab, W


@pytest.mark.parametrize("sub", [1, 3, 8, 64])
def test_ut_transform_matches_oracle_and_dense_products(sub):
    """The oracle's token-by-token transition equals the dense product of the frame's token
    factors, and the UT transform over sub-chunks of any size; U_f is the state the frame's
    tokens reach from zero."""
    rng = np.random.default_rng(40 + sub)
    N = 70 if sub == 64 else 8   # several sub-chunks and a ragged tail
    q, k, v, beta, gamma, _ = rand_inputs(rng, 1, 1, 2, N, 16, s0=False)
    ks = 0.9 if N == 8 else 0.35  # large keys: the product differs from the sum at first order in beta
    M, U = oracle.frame_transitions(k, v, beta, gamma, key_scale=ks, mode="product")
    Ms, _ = oracle.frame_transitions(k, v, beta, gamma, key_scale=ks, mode="sum")
    for f, (P, W) in enumerate(brute_force_frame(k, v, beta, gamma, ks)):
        g = float(gamma[0, f, 0])
        np.testing.assert_allclose(M[0, 0, f] + (1 - g) * np.eye(16), P, rtol=0, atol=1e-12)
        np.testing.assert_allclose(U[0, 0, f], W, rtol=0, atol=1e-12)
        sl = slice(f * N, (f + 1) * N)
        kh = np.stack([unit(x) * ks for x in k[0, sl, 0]])
        Ab, Wut = ut_transform_frame(kh, v[0, sl, 0].astype(np.float64), beta[0, sl, 0].astype(np.float64), sub)
        np.testing.assert_allclose(M[0, 0, f], g * np.eye(16) - Ab, rtol=0, atol=1e-12)
        np.testing.assert_allclose(U[0, 0, f], Wut, rtol=0, atol=1e-12)
        assert np.abs(M[0, 0, f] - Ms[0, 0, f]).max() > 1e-3   # the two readings really differ here


def test_product_forward_is_the_token_wise_delta_rule():
    """S_f = R_f - (1 - gamma_f) S_{f-1}, R_f the token-wise delta rule run from S_{f-1}; o = S_f q^."""
    rng = np.random.default_rng(7)
    B, H, F, N, D = 1, 1, 3, 8, 16
    q, k, v, beta, gamma, S0 = rand_inputs(rng, B, H, F, N, D)
    ks = 0.8
    o, S_out = oracle.frame_fwd(q, k, v, beta, gamma, S0, key_scale=ks, mode="product")
    S = S0[0, 0].astype(np.float64)
    for f in range(F):
        R = S.copy()
        for n in range(f * N, (f + 1) * N):
            kh = unit(k[0, n, 0]) * ks
            b = float(beta[0, n, 0])
            R = R + b * np.outer(v[0, n, 0] - R @ kh, kh)
        S = R - (1 - float(gamma[0, f, 0])) * S
        for n in range(f * N, (f + 1) * N):
            np.testing.assert_allclose(o[0, n, 0], S @ unit(q[0, n, 0]), rtol=0, atol=1e-10)
    np.testing.assert_allclose(S_out[0, 0], S, rtol=0, atol=1e-10)


def test_product_equals_sum_for_orthogonal_keys():
    """Mutually orthogonal keys commute and annihilate cross terms: product == sum exactly."""
    rng = np.random.default_rng(3)
    B, H, F, N, D = 1, 2, 2, 6, 16
    q, k, v, beta, gamma, S0 = rand_inputs(rng, B, H, F, N, D)
    for h in range(H):
        for f in range(F):
            Qm, _ = np.linalg.qr(rng.standard_normal((D, N)))
            scale = rng.uniform(0.5, 2.0, N)
            k[0, f * N:(f + 1) * N, h] = (Qm * scale).T.astype(np.float32)
    o_p, S_p = oracle.frame_fwd(q, k, v, beta, gamma, S0, key_scale=1.0, mode="product")
    o_s, S_s = oracle.frame_fwd(q, k, v, beta, gamma, S0, key_scale=1.0, mode="sum")
    # fp32 keys are orthogonal only to ~1e-7: the cross terms are that small
    np.testing.assert_allclose(S_p, S_s, rtol=0, atol=1e-5)
    np.testing.assert_allclose(o_p, o_s, rtol=0, atol=1e-5)


def test_repeated_unit_key_projector_and_last_write():
    """N copies of one unit key with beta = 1: (I - k k^T)^N = I - k k^T (a projector), and the
    state from zero keeps only the last value, U = v_N k^T.  The sum reading gives N k k^T and
    sum_n v_n k^T instead."""
    D, N = 5, 3
    kvec = np.array([1.0, 2.0, -2.0, 0.0, 4.0], np.float32)
    kh = unit(kvec)
    k = np.tile(kvec, (N, 1)).reshape(1, N, 1, D)
    v = np.arange(N * D, dtype=np.float32).reshape(1, N, 1, D) - 4.0
    beta = np.ones((1, N, 1), np.float32)
    gamma = np.array([[[0.75]]], np.float32)
    M, U = oracle.frame_transitions(k, v, beta, gamma, key_scale=1.0, mode="product")
    np.testing.assert_allclose(M[0, 0, 0], 0.75 * np.eye(D) - np.outer(kh, kh), rtol=0, atol=1e-12)
    np.testing.assert_allclose(U[0, 0, 0], np.outer(v[0, -1, 0], kh), rtol=0, atol=1e-12)
    Ms, Us = oracle.frame_transitions(k, v, beta, gamma, key_scale=1.0, mode="sum")
    np.testing.assert_allclose(Ms[0, 0, 0], 0.75 * np.eye(D) - N * np.outer(kh, kh), rtol=0, atol=1e-12)
    np.testing.assert_allclose(Us[0, 0, 0], np.outer(v[0, :, 0].sum(0), kh), rtol=0, atol=1e-12)


def test_product_ut_invariance_and_default_scale_gap():
    """The UT evaluation at every sub-chunk size reproduces the oracle's transition; at the
    default key scale 1/sqrt(D N) the product differs from the sum only at second order in the
    keys (cross terms ~ c^4)."""
    rng = np.random.default_rng(11)
    q, k, v, beta, gamma, S0 = rand_inputs(rng, 1, 1, 2, 40, 24)
    ref = oracle.frame_transitions(k, v, beta, gamma, mode="product")
    c = 1 / np.sqrt(24 * 40)
    for f in range(2):
        sl = slice(f * 40, (f + 1) * 40)
        kh = np.stack([unit(x) * c for x in k[0, sl, 0]])
        for sub in (1, 2, 7, 16, 64):
            Ab, W = ut_transform_frame(kh, v[0, sl, 0].astype(np.float64), beta[0, sl, 0].astype(np.float64), sub)
            np.testing.assert_allclose(float(gamma[0, f, 0]) * np.eye(24) - Ab, ref[0][0, 0, f], rtol=0, atol=1e-14)
            np.testing.assert_allclose(W, ref[1][0, 0, f], rtol=0, atol=1e-12)
    Ms, Us = oracle.frame_transitions(k, v, beta, gamma, mode="sum")
    gap = np.abs(ref[0] - Ms).max()
    assert 0 < gap < 5 * 40 * c ** 4      # N^2/2 cross terms of size c^4 |cos|, cos ~ 1/sqrt(D)
    # halving the key scale divides the gap by 2^4
    Mh, _ = oracle.frame_transitions(k, v, beta, gamma, key_scale=c / 2, mode="product")
    Msh, _ = oracle.frame_transitions(k, v, beta, gamma, key_scale=c / 2, mode="sum")
    ratio = gap / np.abs(Mh - Msh).max()
    assert 14.0 < ratio < 18.5, ratio
