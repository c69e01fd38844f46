"""The fused single-frame streaming step (gdn_frame_step) against the fp64 oracle.

One cluster of CTAs per (batch, head) chain splits the frame's tokens, so the
cases below cover token counts around the 64-token stats stages and 128-token
output tiles, several chains per launch, a zero and a random initial state,
state aliasing, and the layer's streaming shape (B=1, H=20, N=880).
Tolerance: relative Frobenius error <= 5e-3 on o and S_out (bf16 I/O, fp32 state).
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_wise_b300 import gdn
from gated_deltanet_wise_b300.inputs import make_inputs
from tests.conftest import rel_fro

pytestmark = pytest.mark.gpu

TOL_BF16 = 5e-3
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    gdn.lib()
    yield
    assert gdn.gdn_device_status() == gdn.GDN_OK


def step_inputs(B, H, N, seed, s0_std=0.1):
    x = make_inputs(B, H, 1, N, 112, dtype="bf16", seed=seed, device=DEV, s0_std=s0_std)
    return x, x.gamma[:, 0].contiguous()


@pytest.mark.parametrize("B,H,N", [(1, 1, 1), (1, 1, 63), (1, 1, 64), (1, 2, 65), (2, 1, 127), (1, 1, 128),
                                   (1, 3, 129), (2, 3, 200), (1, 20, 880), (1, 2, 1000), (1, 2, 3520)])
def test_step_matches_oracle(B, H, N):
    x, g = step_inputs(B, H, N, seed=N + 17 * H)
    o, S = gdn.frame_step(x.q, x.k, x.v, x.beta, g, x.S0)
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.frame_fwd(x.q, x.k, x.v, x.beta, x.gamma, x.S0)
    eo = rel_fro(o.float().cpu().numpy(), o_ref)
    es = rel_fro(S.cpu().numpy(), S_ref)
    assert eo <= TOL_BF16 and es <= TOL_BF16, (eo, es)
    assert es < 1e-4   # the state path keeps fp32 accuracy through hi/lo splits


def test_step_zero_initial_state_and_no_state_out():
    x, g = step_inputs(1, 4, 300, seed=3, s0_std=0.0)
    o = torch.empty_like(x.q)
    st = gdn.gdn_frame_step(x.q, x.k, x.v, x.beta, g, None, None, o, 1, 4, 300, 112, 0.0, None, 0)
    assert st == gdn.GDN_OK
    torch.cuda.synchronize()
    o_ref, _ = oracle.frame_fwd(x.q, x.k, x.v, x.beta, x.gamma, None)
    assert rel_fro(o.float().cpu().numpy(), o_ref) <= TOL_BF16


def test_step_state_aliasing_and_determinism():
    x, g = step_inputs(2, 5, 880, seed=9, s0_std=0.3)
    o1, S1 = gdn.frame_step(x.q, x.k, x.v, x.beta, g, x.S0)
    o2, S2 = gdn.frame_step(x.q, x.k, x.v, x.beta, g, x.S0)
    assert torch.equal(o1, o2) and torch.equal(S1, S2)
    S_alias = x.S0.clone()
    o3, S3 = gdn.frame_step(x.q, x.k, x.v, x.beta, g, S_alias, S_out=S_alias)
    assert S3.data_ptr() == S_alias.data_ptr()
    assert torch.equal(o3, o1) and torch.equal(S3, S1)


def test_step_equals_full_forward_with_one_frame():
    x, g = step_inputs(1, 6, 500, seed=5, s0_std=0.2)
    o_s, S_s = gdn.frame_step(x.q, x.k, x.v, x.beta, g, x.S0)
    o_f, S_f = gdn.frame_fwd(x.q, x.k, x.v, x.beta, x.gamma, x.S0)
    assert rel_fro(o_s.float().cpu().numpy(), o_f.float().cpu().numpy()) <= TOL_BF16
    assert rel_fro(S_s.cpu().numpy(), S_f.cpu().numpy()) <= 1e-4


def test_step_output_canaries_untouched():
    B, H, N, D = 1, 3, 150, 112
    x, g = step_inputs(B, H, N, seed=8)
    n = B * N * H * D
    pad = 4096
    buf = torch.full((n + 2 * pad,), 7.0, dtype=torch.bfloat16, device=DEV)
    o = buf[pad:pad + n].view(B, N, H, D)
    S_buf = torch.full((B * H * D * D + 2 * pad,), 3.0, dtype=torch.float32, device=DEV)
    S_out = S_buf[pad:pad + B * H * D * D].view(B, H, D, D)
    gdn.frame_step(x.q, x.k, x.v, x.beta, g, x.S0, o=o, S_out=S_out)
    torch.cuda.synchronize()
    assert torch.all(buf[:pad] == 7.0) and torch.all(buf[pad + n:] == 7.0)
    assert torch.all(S_buf[:pad] == 3.0) and torch.all(S_buf[pad + B * H * D * D:] == 3.0)
    o_ref, S_ref = oracle.frame_fwd(x.q, x.k, x.v, x.beta, x.gamma, x.S0)
    assert rel_fro(o.float().cpu().numpy(), o_ref) <= TOL_BF16
    assert rel_fro(S_out.cpu().numpy(), S_ref) <= TOL_BF16


def test_step_beta_zero_is_pure_decay():
    x, g = step_inputs(1, 2, 256, seed=12, s0_std=0.5)
    x.beta.zero_()
    o, S = gdn.frame_step(x.q, x.k, x.v, x.beta, g, x.S0)
    expect = g[:, :, None, None] * x.S0
    assert rel_fro(S.cpu().numpy(), expect.cpu().numpy()) < 1e-6
