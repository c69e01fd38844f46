"""Token-ordered ("product") reading on the GPU (gdn_frame_fwd_product) against
the fp64 oracle's product mode, through the C ABI.

The UT-transform kernel works in 64-token sub-chunks, so the token counts
cover one token, exactly one sub-chunk, a one-token tail, several sub-chunks
with a ragged tail and the layer's 880.  Unit keys (key_scale = 1) are the
regime where the product and the sum readings differ at first order; the
tests check that the GPU follows the product there and not the sum.
Tolerance: relative Frobenius error <= 5e-3 on o and S_out (bf16 I/O, fp32 state).
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_wise_b300 import gdn
from gated_deltanet_wise_b300.inputs import make_inputs
from tests.conftest import check_every_chain, rel_fro

pytestmark = pytest.mark.gpu

TOL = 5e-3
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    gdn.lib()
    yield
    assert gdn.gdn_device_status() == gdn.GDN_OK


def _check(x, key_scale, S_in=None):
    o, S = gdn.frame_fwd_product(x.q, x.k, x.v, x.beta, x.gamma, S_in, key_scale=key_scale)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    o_ref, S_ref = oracle.frame_fwd(x.q, x.k, x.v, x.beta, x.gamma, S_in, key_scale=key_scale, mode="product")
    e_o = rel_fro(o.float().cpu().numpy(), o_ref)
    e_s = rel_fro(S.cpu().numpy(), S_ref)
    assert e_o <= TOL and e_s <= TOL, (e_o, e_s)
    return o, S, o_ref, S_ref


@pytest.mark.parametrize("B,H,F,N", [(1, 1, 2, 1), (1, 1, 3, 64), (1, 2, 2, 65), (2, 1, 3, 200),
                                     (1, 3, 4, 300), (1, 2, 3, 880)])
@pytest.mark.parametrize("key_scale", [0.0, 0.3, 1.0])
def test_product_matches_oracle(B, H, F, N, key_scale):
    x = make_inputs(B, H, F, N, 112, dtype="bf16", seed=100 + N + F, device=DEV)
    _check(x, key_scale)


def test_unit_keys_follow_the_product_not_the_sum():
    x = make_inputs(1, 2, 3, 200, 112, dtype="bf16", seed=7, device=DEV)
    o, S, o_ref, S_ref = _check(x, 1.0)
    o_sum, S_sum = oracle.frame_fwd(x.q, x.k, x.v, x.beta, x.gamma, None, key_scale=1.0, mode="sum")
    assert rel_fro(o_sum, o_ref) > 20 * TOL  # the readings really differ here
    assert rel_fro(o.float().cpu().numpy(), o_sum) > 10 * TOL


def test_start_state_and_aliasing():
    x = make_inputs(1, 2, 3, 150, 112, dtype="bf16", seed=11, device=DEV, s0_std=0.1)
    o, S, _, _ = _check(x, 0.5, S_in=x.S0)
    S_alias = x.S0.clone()
    o2, _ = gdn.frame_fwd_product(x.q, x.k, x.v, x.beta, x.gamma, S_alias, key_scale=0.5, S_out=S_alias)
    torch.cuda.synchronize()
    torch.testing.assert_close(S_alias, S, rtol=0, atol=0)
    torch.testing.assert_close(o2, o, rtol=0, atol=0)


def test_zero_beta_is_pure_decay():
    x = make_inputs(1, 2, 3, 130, 112, dtype="bf16", seed=12, device=DEV, s0_std=0.1)
    beta = torch.zeros_like(x.beta)
    _, S = gdn.frame_fwd_product(x.q, x.k, x.v, beta, x.gamma, x.S0, key_scale=1.0)
    torch.cuda.synchronize()
    ref = x.S0 * x.gamma.prod(1)[:, :, None, None]
    torch.testing.assert_close(S, ref, rtol=1e-5, atol=1e-6)


def test_default_scale_agrees_with_sum_path():
    """At the default key scale the two readings agree to ~1e-8, so the product
    path must match the sum path within the bf16 output rounding."""
    x = make_inputs(1, 4, 5, 300, 112, dtype="bf16", seed=13, device=DEV, s0_std=0.1)
    o_p, S_p = gdn.frame_fwd_product(x.q, x.k, x.v, x.beta, x.gamma, x.S0)
    o_s, S_s = gdn.frame_fwd(x.q, x.k, x.v, x.beta, x.gamma, x.S0)
    torch.cuda.synchronize()
    assert rel_fro(o_p.float().cpu().numpy(), o_s.float().cpu().numpy()) <= TOL
    assert rel_fro(S_p.cpu().numpy(), S_s.cpu().numpy()) <= TOL


@pytest.mark.parametrize("key_scale", [0.0, 1.0])
def test_layer_size_every_head(key_scale):
    """The 60 s 720p layer (B=1, H=20, F=121, N=880) in one call; the oracle
    checks all 20 chains."""
    x = make_inputs(1, 20, 121, 880, 112, dtype="bf16", seed=21, device=DEV)
    o, S = gdn.frame_fwd_product(x.q, x.k, x.v, x.beta, x.gamma, None, key_scale=key_scale)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    check_every_chain(x, o, S, lambda q, k, v, b, g, s0: oracle.frame_fwd(q, k, v, b, g, s0, key_scale=key_scale,
                                                                             mode="product"), TOL)


def test_workspace_and_degenerate_sizes():
    x = make_inputs(1, 2, 2, 70, 112, dtype="bf16", seed=14, device=DEV, s0_std=0.1)
    nbytes = gdn.gdn_frame_fwd_product_workspace_size(1, 2, 2, 70, 112)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    o = torch.empty_like(x.q)
    S = torch.empty(1, 2, 112, 112, device=DEV)
    st = gdn.gdn_frame_fwd_product(x.q, x.k, x.v, x.beta, x.gamma, x.S0, S, o, 1, 2, 2, 70, 112, 0.0, ws,
                                   nbytes - 1)
    assert st == gdn.GDN_ERR_WORKSPACE
    assert gdn.gdn_frame_fwd_product(x.q, x.k, x.v, x.beta, x.gamma, x.S0, S, o, 1, 2, 2, 70, 96, 0.0, ws,
                                     nbytes) == gdn.GDN_ERR_UNSUPPORTED
    # no tokens: S_out = (prod gamma) S_in
    e = torch.empty(1, 0, 2, 112, dtype=torch.bfloat16, device=DEV)
    st = gdn.gdn_frame_fwd_product(e, e, e, torch.empty(1, 0, 2, device=DEV), x.gamma, x.S0, S, e, 1, 2, 2, 0,
                                   112, 0.0, None, 0)
    assert st == gdn.GDN_OK
    torch.cuda.synchronize()
    torch.testing.assert_close(S, x.S0 * x.gamma.prod(1)[:, :, None, None], rtol=1e-6, atol=1e-7)


@pytest.mark.parametrize("key_scale", [0.0, 1.0])
def test_long_frames_cfg_batch(key_scale):
    """Frames of 3520 tokens (55 sub-chunks each) with B=2, the longest frame of the CFG sweep."""
    x = make_inputs(2, 3, 6, 3520, 112, dtype="bf16", seed=23, device=DEV, s0_std=0.1)
    _check(x, key_scale, S_in=x.S0)
