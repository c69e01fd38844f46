"""Backward pass (gdn_frame_bwd) on the GPU against the fp64 oracle backward
(which tests/test_oracle_backward_pins.py checks against finite differences of
the forward).  Every gradient tensor must match within a relative Frobenius
error of 5e-3; the cases cover a ragged token tail, several frame chunks, a
zero and a random dS_out, a non-default key scale, and four heads of the
20-head layer."""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_wise_b300 import gdn
from gated_deltanet_wise_b300.inputs import make_inputs
from tests.conftest import rel_fro

pytestmark = pytest.mark.gpu
TOL = 5e-3
DEV = "cuda"
NAMES = ("dq", "dk", "dv", "dbeta", "dgamma", "dS_in")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    gdn.lib()
    yield
    assert gdn.gdn_device_status() == gdn.GDN_OK


def _upstream(x, seed, with_dS=True):
    g = torch.Generator(device=DEV).manual_seed(seed)
    dO = torch.randn(x.q.shape, generator=g, device=DEV).to(torch.bfloat16)
    dS = torch.randn(x.B, x.H, x.D, x.D, generator=g, device=DEV) * 0.1 if with_dS else None
    return dO, dS


def _compare(got, ref, tol=TOL):
    errs = {}
    for n, a, b in zip(NAMES, got, ref):
        errs[n] = rel_fro(a.cpu().numpy().astype(np.float64), b)
    assert all(e <= tol for e in errs.values()), errs
    return errs


@pytest.mark.parametrize("B,H,F,N,ks,with_dS", [(1, 2, 3, 200, 0.0, True), (2, 1, 4, 130, 0.5, True),
                                                (1, 3, 9, 64, 0.0, False), (1, 2, 2, 1, 0.3, True)])
def test_backward_matches_oracle(B, H, F, N, ks, with_dS):
    x = make_inputs(B, H, F, N, 112, dtype="bf16", seed=80 + F + N, device=DEV, s0_std=0.1)
    dO, dS = _upstream(x, 5 + F, with_dS)
    got = gdn.frame_bwd(x.q, x.k, x.v, x.beta, x.gamma, x.S0, dO, dS, key_scale=ks)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    ref = oracle.frame_bwd(x.q, x.k, x.v, x.beta, x.gamma, x.S0, dO, dS, key_scale=ks)
    _compare(got, ref)


def test_backward_without_initial_state():
    x = make_inputs(1, 2, 4, 150, 112, dtype="bf16", seed=91, device=DEV)
    dO, dS = _upstream(x, 9)
    got = gdn.frame_bwd(x.q, x.k, x.v, x.beta, x.gamma, None, dO, dS)
    torch.cuda.synchronize()
    ref = oracle.frame_bwd(x.q, x.k, x.v, x.beta, x.gamma, None, dO, dS)
    _compare(got, ref)


def test_backward_layer_size_four_heads():
    """The 20-head layer (F=121, N=880); the oracle checks four heads spread over the
    layer (chains are independent; first, last and two inner head offsets)."""
    x = make_inputs(1, 20, 121, 880, 112, dtype="bf16", seed=92, device=DEV)
    dO, dS = _upstream(x, 10)
    got = gdn.frame_bwd(x.q, x.k, x.v, x.beta, x.gamma, None, dO, dS)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    heads = torch.tensor([0, 6, 13, 19], device=DEV)
    sl = lambda t: t.index_select(2, heads).contiguous()
    ref = oracle.frame_bwd(sl(x.q), sl(x.k), sl(x.v), sl(x.beta), sl(x.gamma), None, sl(dO),
                           dS.index_select(1, heads).contiguous())
    got_h = [sl(got[0]), sl(got[1]), sl(got[2]), sl(got[3]), sl(got[4]), got[5].index_select(1, heads)]
    head = lambda t, i, j: t[:, j:j + 1] if i == 5 else t[:, :, j:j + 1]   # dS_in has heads on axis 1
    for j in range(len(heads)):   # every head on its own
        _compare([head(g, i, j) for i, g in enumerate(got_h)], [head(r, i, j) for i, r in enumerate(ref)])


def test_backward_degenerate_sizes():
    x = make_inputs(1, 2, 2, 16, 112, dtype="bf16", seed=93, device=DEV, s0_std=0.1)
    dO, dS = _upstream(x, 11)
    z = torch.empty(0, device=DEV)
    dS_in = torch.empty(1, 2, 112, 112, device=DEV)
    e = torch.empty(1, 0, 2, 112, dtype=torch.bfloat16, device=DEV)
    g0 = torch.empty(1, 0, 2, device=DEV)
    # no frames: dS_in = dS_out
    st = gdn.gdn_frame_bwd(e, e, e, g0, g0, x.S0, e, dS, z, z, z, z, z, dS_in, 1, 2, 0, 0, 112, 0.0, None, 0)
    assert st == gdn.GDN_OK
    torch.cuda.synchronize()
    torch.testing.assert_close(dS_in, dS, rtol=0, atol=0)
    assert gdn.gdn_frame_bwd_workspace_size(1, 2, 2, 0, 112) == 2 ** 64 - 1
    assert gdn.gdn_frame_bwd_workspace_size(1, 2, 2, 16, 96) == 2 ** 64 - 1
    nb = gdn.gdn_frame_bwd_workspace_size(1, 2, 2, 16, 112)
    ws = torch.empty(nb, dtype=torch.uint8, device=DEV)
    dq = torch.empty(x.q.shape, device=DEV)
    dbeta = torch.empty(x.beta.shape, device=DEV)
    dgamma = torch.empty(x.gamma.shape, device=DEV)
    assert gdn.gdn_frame_bwd(x.q, x.k, x.v, x.beta, x.gamma, x.S0, dO, dS, dq, dq, dq, dbeta, dgamma, dS_in,
                             1, 2, 2, 16, 112, 0.0, ws, nb - 256) == gdn.GDN_ERR_WORKSPACE
