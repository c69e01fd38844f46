"""Pins of the oracle's reverse-direction scan (bidirectional stage-1 model,
summary page section 局限与改进) to something other than its own code path:
the oracle computes it by running the forward scan on the frame-reversed
sequence; here it is rebuilt from the per-frame transitions (M_f, U_f),
composed explicitly from the last frame to the first."""
import numpy as np
import pytest

import oracle

B, H, D = 1, 2, 8


def _inputs(F, N, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, F * N, H, D)).astype(np.float32)
    k = rng.standard_normal((B, F * N, H, D)).astype(np.float32)
    v = rng.standard_normal((B, F * N, H, D)).astype(np.float32)
    beta = (1 / (1 + np.exp(-rng.standard_normal((B, F * N, H))))).astype(np.float32)
    gamma = (1 / (1 + np.exp(rng.standard_normal((B, F, H))))).astype(np.float32)
    S0 = rng.standard_normal((B, H, D, D)).astype(np.float32)
    return q, k, v, beta, gamma, S0


@pytest.mark.parametrize("mode", ["sum", "product"])
def test_reverse_is_the_transitions_composed_from_the_last_frame(mode):
    F, N, ks = 4, 5, 0.7
    q, k, v, beta, gamma, S0 = _inputs(F, N, 3)
    o, S = oracle.frame_fwd(q, k, v, beta, gamma, S0, key_scale=ks, mode=mode, reverse=True)
    M, U = oracle.frame_transitions(k, v, beta, gamma, key_scale=ks, mode=mode)
    for h in range(H):
        St = S0[0, h].astype(np.float64)
        for f in reversed(range(F)):
            St = St @ M[0, h, f] + U[0, h, f]
            for n in range(N):
                qn = q[0, f * N + n, h].astype(np.float64)
                np.testing.assert_allclose(o[0, f * N + n, h], St @ qn / np.linalg.norm(qn), rtol=1e-9, atol=1e-9)
        np.testing.assert_allclose(S[0, h], St, rtol=1e-9, atol=1e-9)


def test_single_frame_reverse_equals_forward():
    q, k, v, beta, gamma, S0 = _inputs(1, 6, 4)
    of, Sf = oracle.frame_fwd(q, k, v, beta, gamma, S0, key_scale=0.5)
    orv, Sr = oracle.frame_fwd(q, k, v, beta, gamma, S0, key_scale=0.5, reverse=True)
    np.testing.assert_array_equal(of, orv)
    np.testing.assert_array_equal(Sf, Sr)


def test_reverse_differs_from_forward_when_frames_differ():
    q, k, v, beta, gamma, S0 = _inputs(3, 4, 5)
    of, Sf = oracle.frame_fwd(q, k, v, beta, gamma, S0, key_scale=0.5)
    orv, Sr = oracle.frame_fwd(q, k, v, beta, gamma, S0, key_scale=0.5, reverse=True)
    assert np.abs(Sf - Sr).max() > 1e-3 * np.abs(Sf).max()
