"""Pins of the oracle's backward pass (sum reading) to the pinned forward:
every gradient is compared with a fourth-order central finite difference of
L = sum(dO * o) + sum(dS_out * S_out), the forward run by the oracle itself
(formulation and code independent of the backward).  Inputs are dyadic
rationals and the steps powers of two, so every perturbed input is exact in
fp32 and the difference quotient carries only its O(h^4) truncation."""
import numpy as np
import pytest

import oracle

B, H, F, N, D = 1, 2, 3, 4, 6
KS = 0.7


def _dyadic(rng, shape, scale=1.0):
    return (np.round(rng.standard_normal(shape) * scale * 256) / 256).astype(np.float32)


def _inputs(seed):
    rng = np.random.default_rng(seed)
    x = dict(q=_dyadic(rng, (B, F * N, H, D)), k=_dyadic(rng, (B, F * N, H, D)), v=_dyadic(rng, (B, F * N, H, D)),
             beta=(np.round(rng.uniform(0.1, 0.9, (B, F * N, H)) * 256) / 256).astype(np.float32),
             gamma=(np.round(rng.uniform(0.5, 0.95, (B, F, H)) * 256) / 256).astype(np.float32),
             S_in=_dyadic(rng, (B, H, D, D), 0.5))
    dO = _dyadic(rng, (B, F * N, H, D))
    dS = _dyadic(rng, (B, H, D, D))
    return x, dO, dS


def _loss(x, dO, dS):
    o, S = oracle.frame_fwd(x["q"], x["k"], x["v"], x["beta"], x["gamma"], x["S_in"], key_scale=KS)
    return float((o * dO).sum() + ((S * dS).sum() if dS is not None else 0.0))


def _fd(x, name, idx, dO, dS, h=2.0 ** -6):
    vals = []
    for m in (2, 1, -1, -2):
        y = {kk: vv.copy() for kk, vv in x.items()}
        y[name][idx] += np.float32(m * h)
        vals.append(_loss(y, dO, dS))
    return (8 * (vals[1] - vals[2]) - (vals[0] - vals[3])) / (12 * h)


@pytest.mark.parametrize("with_dS", [True, False])
def test_gradients_match_finite_differences(with_dS):
    x, dO, dS = _inputs(5)
    dS = dS if with_dS else None
    g = dict(zip(["q", "k", "v", "beta", "gamma", "S_in"],
                 oracle.frame_bwd(x["q"], x["k"], x["v"], x["beta"], x["gamma"], x["S_in"], dO, dS, key_scale=KS)))
    rng = np.random.default_rng(1)
    for name, grad in g.items():
        flat = list(np.ndindex(grad.shape))
        picks = [flat[i] for i in rng.choice(len(flat), size=min(24, len(flat)), replace=False)]
        scale = np.abs(grad).max()
        for idx in picks:
            fd = _fd(x, name, idx, dO, dS)
            assert abs(fd - grad[idx]) <= 2e-6 * scale + 1e-9, (name, idx, fd, grad[idx])


def test_only_state_gradient_flows_through_the_decay():
    """dO = 0, beta = 0: S_out = (prod gamma) S_in, so dS_in = (prod gamma) dS_out and
    dgamma_f = (prod_{g != f} gamma_g) <S_in, dS_out>; no token gradient."""
    x, _, dS = _inputs(6)
    x["beta"][:] = 0
    dO = np.zeros_like(x["q"])
    dq, dk, dv, db, dg, dSin = oracle.frame_bwd(x["q"], x["k"], x["v"], x["beta"], x["gamma"], x["S_in"], dO, dS,
                                                key_scale=KS)
    gp = x["gamma"].astype(np.float64).prod(1)                       # [B, H]
    np.testing.assert_allclose(dSin, gp[:, :, None, None] * dS, rtol=1e-12)
    inner = (x["S_in"].astype(np.float64) * dS).sum((2, 3))          # [B, H]
    np.testing.assert_allclose(dg, gp[:, None, :] / x["gamma"] * inner[:, None, :], rtol=1e-12)
    assert np.abs(dq).max() == 0 and np.abs(dk).max() == 0 and np.abs(dv).max() == 0
