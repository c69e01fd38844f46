"""Pins of the oracle's GDN block (input projection, frame-wise forward, output projection).

Summary page "SANA-WM: Efficient Minute-Scale World Modeling with Hybrid Linear
Diffusion Transformer", section 方法步骤详情 module 1: the GDN blocks have
d_model = 20 heads x 112.  The projection shapes and gate activations are a
reading (the pages print none): [q | k | v | a | g] = x W_in^T,
beta = sigmoid(a), gamma = exp(-softplus(frame mean of g)), y = o W_out^T.
These CPU tests tie the oracle's block to closed forms and to brute-force loops,
and its layer part to the already-pinned frame_fwd.
"""
import numpy as np

import oracle

D = 112


def _weights(rng, H, scale=None):
    HD = H * D
    s = scale if scale is not None else 1 / np.sqrt(HD)
    W_in = (rng.standard_normal((3 * HD + 2 * H, HD)) * s).astype(np.float32)
    W_out = (rng.standard_normal((HD, HD)) * s).astype(np.float32)
    return oracle._round_bf16(W_in), oracle._round_bf16(W_out)


def test_identity_projections_reduce_to_the_layer():
    """W_q = W_k = W_v = I, zero gate rows, W_out = I: q = k = v = x, beta = gamma = 1/2 exactly,
    and the block is frame_fwd(x, x, x, 1/2, 1/2) with y = o."""
    rng = np.random.default_rng(1)
    B, H, F, N = 1, 2, 3, 5
    HD = H * D
    x = oracle._round_bf16(rng.standard_normal((B, F * N, HD)))
    W_in = np.zeros((3 * HD + 2 * H, HD), np.float32)
    for i in range(3):
        W_in[i * HD:(i + 1) * HD] = np.eye(HD)
    W_out = np.eye(HD, dtype=np.float32)
    q, k, v, beta, gamma = oracle.block_in_proj(x, W_in, F)
    xs = x.reshape(B, F * N, H, D)
    for t in (q, k, v):
        np.testing.assert_array_equal(t, xs)
    np.testing.assert_array_equal(beta, 0.5)
    np.testing.assert_array_equal(gamma, 0.5)
    y, S = oracle.block_fwd(x, W_in, W_out, None, F=F)
    o_ref, S_ref = oracle.frame_fwd(xs, xs, xs, np.full((B, F * N, H), 0.5, np.float32),
                                    np.full((B, F, H), 0.5, np.float32), None)
    np.testing.assert_allclose(y, o_ref.reshape(B, F * N, HD), rtol=0, atol=1e-13)
    np.testing.assert_allclose(S, S_ref, rtol=0, atol=1e-13)


def test_gates_pick_a_channel_closed_form():
    """Gate rows that pick channel j of x: beta = sigmoid(x_j) per token; gamma_f =
    1 / (1 + exp(mean_n x_{n,j})) per frame (exp(-softplus(t)) = 1 / (1 + e^t))."""
    rng = np.random.default_rng(2)
    B, H, F, N = 2, 2, 4, 6
    HD = H * D
    x = oracle._round_bf16(rng.standard_normal((B, F * N, HD)))
    W_in = np.zeros((3 * HD + 2 * H, HD), np.float32)
    picks_a, picks_g = [5, 130], [17, 200]
    for h in range(H):
        W_in[3 * HD + h, picks_a[h]] = 1.0
        W_in[3 * HD + H + h, picks_g[h]] = 1.0
    _, _, _, beta, gamma = oracle.block_in_proj(x, W_in, F)
    for b in range(B):
        for h in range(H):
            for n in range(F * N):
                xa = float(x[b, n, picks_a[h]])
                assert abs(beta[b, n, h] - 1 / (1 + np.exp(-xa))) < 1e-15
            for f in range(F):
                m = float(np.mean(x[b, f * N:(f + 1) * N, picks_g[h]].astype(np.float64)))
                assert abs(gamma[b, f, h] - 1 / (1 + np.exp(m))) < 1e-15


def test_projection_equals_brute_force_loops():
    """The library matmul step against explicit loops, on a tiny shape (one head of D = 112
    would be slow: a 2-head slice of the rows is checked), and the bf16 rounding of q, k, v."""
    rng = np.random.default_rng(3)
    B, H, F, N = 1, 1, 2, 3
    HD = H * D
    x = oracle._round_bf16(rng.standard_normal((B, F * N, HD)))
    W_in, _ = _weights(rng, H)
    q, k, v, beta, gamma = oracle.block_in_proj(x, W_in, F)
    for n in range(F * N):
        for c in list(range(0, 3 * HD, 37)) + [3 * HD, 3 * HD + 1]:
            s = 0.0
            for j in range(HD):
                s += float(x[0, n, j]) * float(W_in[c, j])
            if c < 3 * HD:
                t = (q, k, v)[c // HD][0, n, 0, c % HD]
                assert t == oracle._round_bf16(np.array([s]))[0]
            elif c == 3 * HD:
                assert abs(beta[0, n, 0] - 1 / (1 + np.exp(-s))) < 1e-14
    # gamma: mean over each frame of the g logit
    for f in range(F):
        g = [sum(float(x[0, n, j]) * float(W_in[3 * HD + 1, j]) for j in range(HD)) for n in range(f * N, (f + 1) * N)]
        assert abs(gamma[0, f, 0] - 1 / (1 + np.exp(np.mean(g)))) < 1e-14


def test_output_projection_is_linear_in_w_out():
    """y = o W_out^T: doubling W_out doubles y exactly; the state does not depend on W_out."""
    rng = np.random.default_rng(4)
    B, H, F, N = 1, 2, 2, 4
    x = oracle._round_bf16(rng.standard_normal((B, F * N, H * D)))
    W_in, W_out = _weights(rng, H)
    y1, S1 = oracle.block_fwd(x, W_in, W_out, None, F=F)
    y2, S2 = oracle.block_fwd(x, W_in, 2 * W_out, None, F=F)
    np.testing.assert_array_equal(y2, 2 * y1)
    np.testing.assert_array_equal(S1, S2)
