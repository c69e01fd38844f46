"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Every test here runs on the CPU.  The oracle is checked against closed forms,
invariants and a hand-worked example; each is chosen so that a plausible slip
(dropped decay, wrong sign of the delta term, transposed write, pre-update
output, wrong key scale or normalisation, mixed-up token/head/frame axes)
fails at least one of them.

Method: summary page "SANA-WM: Efficient Minute-Scale World Modeling with Hybrid
Linear Diffusion Transformer", section 方法步骤详情 module 2 (recurrence, output,
key scale), section 前置知识 "Gated DeltaNet" (S_t = S_{t-1} M_t + U_t, state
size independent of length), section 技术新颖性 (norm bound, exact composite
prefix scan).
"""
import os

import numpy as np
import pytest

import oracle
from tests.conftest import rel_fro

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_inputs(rng, B, H, F, N, D, s0=True):
    q = rng.standard_normal((B, F * N, H, D)).astype(np.float32)
    k = rng.standard_normal((B, F * N, H, D)).astype(np.float32)
    v = rng.standard_normal((B, F * N, H, D)).astype(np.float32)
    beta = (1 / (1 + np.exp(-rng.standard_normal((B, F * N, H))))).astype(np.float32)
    gamma = (1 / (1 + np.exp(rng.standard_normal((B, F, H))))).astype(np.float32)
    S0 = rng.standard_normal((B, H, D, D)).astype(np.float32) if s0 else None
    return q, k, v, beta, gamma, S0


def unit(x):
    x = np.asarray(x, np.float64)
    return x / np.sqrt((x * x).sum(-1, keepdims=True) + 1e-12)


def test_worked_example_d2():
    """Hand-derived two-frame example (tests/golden/worked_d2.txt)."""
    rows = {}
    with open(os.path.join(GOLDEN, "worked_d2.txt")) as fh:
        for line in fh:
            if line.startswith("#") or not line.strip():
                continue
            name, *vals = line.split()
            rows[name] = np.array([float(x) for x in vals])
    B, H, F, N, D = 1, 1, 2, 1, 2
    q = rows["q"].reshape(B, F * N, H, D)
    k = rows["k"].reshape(B, F * N, H, D)
    v = rows["v"].reshape(B, F * N, H, D)
    beta = rows["beta"].reshape(B, F * N, H)
    gamma = rows["gamma"].reshape(B, F, H)
    o, S = oracle.frame_fwd(q, k, v, beta, gamma)
    np.testing.assert_allclose(o.ravel(), rows["o"], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(S.ravel(), rows["S_out"], rtol=1e-12, atol=1e-12)


def test_beta_zero_is_pure_decay():
    """beta = 0: S_f = (prod_{f'<=f} gamma_f') S_0, and o reads the post-update state."""
    rng = np.random.default_rng(1)
    B, H, F, N, D = 2, 3, 5, 4, 8
    q, k, v, beta, gamma, S0 = rand_inputs(rng, B, H, F, N, D)
    beta[:] = 0
    o, S = oracle.frame_fwd(q, k, v, beta, gamma, S0)
    g = gamma.astype(np.float64)
    cum = np.cumprod(g, axis=1)                          # [B, F, H]
    np.testing.assert_allclose(S, cum[:, -1][:, :, None, None] * S0, rtol=1e-13, atol=1e-13)
    qh = unit(q).reshape(B, F, N, H, D)
    expect = np.einsum("bfh,bhij,bfnhj->bfnhi", cum, S0.astype(np.float64), qh)
    np.testing.assert_allclose(o, expect.reshape(B, F * N, H, D), rtol=1e-12, atol=1e-12)


def test_unit_key_projection_and_retrieval():
    """gamma=1, beta=1, N=1, key_scale=1: M = I - k^k^T projects onto k^-perp and S_f k^ = v_f."""
    rng = np.random.default_rng(2)
    B, H, F, N, D = 1, 2, 4, 1, 6
    q, k, v, beta, gamma, S0 = rand_inputs(rng, B, H, F, N, D)
    k *= 3.0                       # non-unit raw keys: the oracle must normalise
    beta[:] = 1
    gamma[:] = 1
    M, U = oracle.frame_transitions(k, v, beta, gamma, key_scale=1.0)
    kh = unit(k)                   # [B, F, H, D] with N = 1
    for h in range(H):
        S = S0[0, h].astype(np.float64)
        for f in range(F):
            kf = kh[0, f, h]
            P = np.eye(D) - np.outer(kf, kf)
            np.testing.assert_allclose(M[0, h, f], P, atol=1e-14)
            np.testing.assert_allclose(M[0, h, f] @ M[0, h, f], M[0, h, f], atol=1e-13)
            S = S @ M[0, h, f] + U[0, h, f]
            np.testing.assert_allclose(S @ kf, v[0, f, h], rtol=1e-12, atol=1e-12)
            x = rng.standard_normal(D)
            x -= kf * (kf @ x)
            Sprev = S0[0, h].astype(np.float64) if f == 0 else Sp
            np.testing.assert_allclose(S @ x, Sprev @ x, rtol=1e-11, atol=1e-11)
            Sp = S
    o, S_out = oracle.frame_fwd(q, k, v, beta, gamma, S0, key_scale=1.0)
    # retrieval through the public forward: the last frame's state maps k^ to v
    for h in range(H):
        np.testing.assert_allclose(S_out[0, h] @ kh[0, F - 1, h], v[0, F - 1, h], rtol=1e-12, atol=1e-12)


def test_rank_one_frame_closed_form():
    """All keys of a frame share one direction e (raw magnitudes/signs differ).

    With the default scale c = 1/sqrt(D N): A = c^2 (sum beta_n) e e^T and
    U = c (sum_n beta_n sign(a_n) v_n) e^T, so after one frame
    S_1 = gamma S_0 - c^2 (sum beta) (S_0 e) e^T + c w e^T.  This pins the key scale,
    the key normalisation, the sign of the delta term and the write orientation.
    """
    rng = np.random.default_rng(3)
    B, H, F, N, D = 1, 1, 1, 7, 5
    e = unit(rng.standard_normal(D))
    a = rng.standard_normal(N) * 4
    k = (a[:, None] * e[None, :]).reshape(B, N, H, D).astype(np.float64)
    k = k.astype(np.float32)
    e = unit(k[0, 0, 0]) * np.sign(a[0])     # the fp32-rounded direction
    v = rng.standard_normal((B, N, H, D)).astype(np.float32)
    q = rng.standard_normal((B, N, H, D)).astype(np.float32) * 2.5
    beta = rng.uniform(0.1, 0.9, (B, N, H)).astype(np.float32)
    gamma = np.array([[[0.7]]], np.float32)
    S0 = rng.standard_normal((B, H, D, D)).astype(np.float32)
    o, S = oracle.frame_fwd(q, k, v, beta, gamma, S0)
    c = 1 / np.sqrt(D * N)
    sb = beta[0, :, 0].astype(np.float64).sum()
    w = (beta[0, :, 0, None] * np.sign(a)[:, None] * v[0, :, 0].astype(np.float64)).sum(0)
    S0d = S0[0, 0].astype(np.float64)
    S1 = 0.7 * S0d - c * c * sb * np.outer(S0d @ e, e) + c * np.outer(w, e)
    np.testing.assert_allclose(S[0, 0], S1, rtol=1e-6, atol=1e-6)   # e is fp32-rounded
    np.testing.assert_allclose(o[0, :, 0], (S1 @ unit(q[0, :, 0]).T).T, rtol=1e-6, atol=1e-6)


def test_norm_bound_and_symmetry():
    """||M_f||_2 <= gamma_f <= 1 and M_f = M_f^T at the default key scale (novelty section)."""
    rng = np.random.default_rng(4)
    for (N, D) in [(8, 16), (64, 32), (200, 24)]:
        B, H, F = 1, 2, 6
        q, k, v, beta, gamma, _ = rand_inputs(rng, B, H, F, N, D, s0=False)
        gamma[0, 0, 0] = 0.02          # small gate: the bound still needs gamma >= lambda_max(A)/2
        M, _ = oracle.frame_transitions(k, v, beta, gamma)
        for h in range(H):
            for f in range(F):
                Mf = M[0, h, f]
                np.testing.assert_allclose(Mf, Mf.T, atol=1e-15)
                lam = np.linalg.eigvalsh(Mf)
                assert np.max(np.abs(lam)) <= float(gamma[0, f, h]) + 1e-12
                # trace(A) = sum_n beta_n / (D N) exactly at the default scale
                trA = D * float(gamma[0, f, h]) - np.trace(Mf)
                assert abs(trA - beta[0, f * N:(f + 1) * N, h].astype(np.float64).sum() / (D * N)) < 1e-12


def test_two_formulations_agree():
    rng = np.random.default_rng(5)
    for (B, H, F, N, D) in [(1, 1, 4, 8, 16), (2, 3, 3, 5, 7), (1, 2, 6, 33, 12)]:
        q, k, v, beta, gamma, S0 = rand_inputs(rng, B, H, F, N, D)
        o1, S1 = oracle.frame_fwd(q, k, v, beta, gamma, S0, formulation="recurrence")
        o2, S2 = oracle.frame_fwd(q, k, v, beta, gamma, S0, formulation="tokacc")
        assert rel_fro(o2, o1) < 1e-13
        assert rel_fro(S2, S1) < 1e-13


@pytest.mark.parametrize("F", [1, 2, 5, 9])
def test_composite_prefix_scan_is_exact(F):
    """Every split of the frame axis into two runs composes back to the sequential state."""
    rng = np.random.default_rng(10 + F)
    B, H, N, D = 1, 1, 6, 8
    q, k, v, beta, gamma, S0 = rand_inputs(rng, B, H, F, N, D)
    _, S_ref = oracle.frame_fwd(q, k, v, beta, gamma, S0)
    M, U = oracle.frame_transitions(k, v, beta, gamma)
    M, U = M[0, 0], U[0, 0]
    C_all, H_all = oracle.composite(M, U)
    s0 = S0[0, 0].astype(np.float64)
    np.testing.assert_allclose(s0 @ C_all + H_all, S_ref[0, 0], rtol=1e-12, atol=1e-12)
    for p in range(0, F + 1):
        C1, H1 = oracle.composite(M[:p], U[:p])
        C2, H2 = oracle.composite(M[p:], U[p:])
        C, Hc = oracle.compose(C1, H1, C2, H2)
        np.testing.assert_allclose(C, C_all, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(Hc, H_all, rtol=1e-12, atol=1e-12)


def test_linear_in_values_and_initial_state():
    rng = np.random.default_rng(6)
    B, H, F, N, D = 1, 2, 3, 5, 6
    q, k, v1, beta, gamma, S1 = rand_inputs(rng, B, H, F, N, D)
    _, _, v2, _, _, S2 = rand_inputs(rng, B, H, F, N, D)
    a = 1.75
    oA, SA = oracle.frame_fwd(q, k, v1, beta, gamma, S1)
    oB, SB = oracle.frame_fwd(q, k, v2, beta, gamma, S2)
    oC, SC = oracle.frame_fwd(q, k, (a * v1.astype(np.float64) + v2).astype(np.float32), beta, gamma,
                              (a * S1.astype(np.float64) + S2).astype(np.float32))
    # the combined inputs were rounded to fp32 once; compare at that precision
    assert rel_fro(oC, a * oA + oB) < 1e-6
    assert rel_fro(SC, a * SA + SB) < 1e-6


def test_axes_heads_batches_and_frames():
    """Heads/batches are independent chains; frames are causal across frames but not within one."""
    rng = np.random.default_rng(7)
    B, H, F, N, D = 2, 3, 4, 5, 6
    q, k, v, beta, gamma, S0 = rand_inputs(rng, B, H, F, N, D)
    o, S = oracle.frame_fwd(q, k, v, beta, gamma, S0)
    # perturb head 1 of batch 0 everywhere
    k2 = k.copy(); k2[0, :, 1] += 1.0
    o2, S2 = oracle.frame_fwd(q, k2, v, beta, gamma, S0)
    mask = np.zeros_like(o, bool); mask[0, :, 1] = True
    np.testing.assert_array_equal(o2[~mask], o[~mask])
    assert np.abs(o2[mask] - o[mask]).max() > 1e-3
    # perturb the last token of frame 2 of chain (1, 2): earlier frames unchanged,
    # every token of frame 2 (including earlier ones) changes.
    f, n = 2, N - 1
    v3 = v.copy(); v3[1, f * N + n, 2] += 1.0
    o3, _ = oracle.frame_fwd(q, k, v3, beta, gamma, S0)
    np.testing.assert_array_equal(o3[1, :f * N, 2], o[1, :f * N, 2])
    assert np.all(np.abs(o3[1, f * N:(f + 1) * N, 2] - o[1, f * N:(f + 1) * N, 2]).max(-1) > 1e-6)
    # gamma of frame f acts from frame f on
    g4 = gamma.copy(); g4[1, f, 2] *= 0.5
    o4, _ = oracle.frame_fwd(q, k, v, beta, g4, S0)
    np.testing.assert_array_equal(o4[1, :f * N, 2], o[1, :f * N, 2])
    assert np.abs(o4[1, f * N:, 2] - o[1, f * N:, 2]).max() > 1e-6


def test_state_size_independent_of_length():
    rng = np.random.default_rng(8)
    for F in (1, 3, 17):
        q, k, v, beta, gamma, S0 = rand_inputs(rng, 1, 2, F, 3, 4)
        _, S = oracle.frame_fwd(q, k, v, beta, gamma, S0)
        assert S.shape == (1, 2, 4, 4)


def test_split_call_equals_one_call():
    """The state is the checkpoint: two calls carrying S equal one call."""
    rng = np.random.default_rng(9)
    B, H, F, N, D = 1, 2, 6, 4, 5
    q, k, v, beta, gamma, S0 = rand_inputs(rng, B, H, F, N, D)
    o, S = oracle.frame_fwd(q, k, v, beta, gamma, S0)
    p = 4
    oa, Sa = oracle.frame_fwd(q[:, :p * N], k[:, :p * N], v[:, :p * N], beta[:, :p * N], gamma[:, :p], S0)
    ob, Sb = oracle.frame_fwd(q[:, p * N:], k[:, p * N:], v[:, p * N:], beta[:, p * N:], gamma[:, p:],
                              Sa.astype(np.float32))
    np.testing.assert_allclose(np.concatenate([oa, ob], 1), o, rtol=1e-6, atol=1e-6)
    np.testing.assert_allclose(Sb, S, rtol=1e-6, atol=1e-6)


def test_zero_keys_are_inert():
    """An all-zero key (and a padded token) contributes nothing: k^ = 0 under the eps-guarded norm."""
    rng = np.random.default_rng(11)
    B, H, F, N, D = 1, 1, 2, 4, 6
    q, k, v, beta, gamma, S0 = rand_inputs(rng, B, H, F, N, D)
    k0 = k.copy(); k0[0, 1, 0] = 0.0
    o_ref, S_ref = oracle.frame_fwd(q, k, v, beta, gamma, S0)
    o0, S0_ = oracle.frame_fwd(q, k0, v, beta, gamma, S0)
    # same as removing token 1 from frame 0 by zeroing its beta
    b0 = beta.copy(); b0[0, 1, 0] = 0.0
    o1, S1 = oracle.frame_fwd(q, k, v, b0, gamma, S0)
    np.testing.assert_allclose(o0, o1, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(S0_, S1, rtol=1e-13, atol=1e-13)
    assert rel_fro(o0, o_ref) > 1e-6
