"""The GDN block with its projections on the GPU (gdn_block_in_proj, gdn_block_out_proj,
gdn_block_fwd) against the fp64 oracle block (tests/test_oracle_block_pins.py pins it).

The input projection's epilogue writes q, k, v (bf16), beta and the per-frame decay
logits; q, k, v must equal the oracle's bf16-rounded fp64 products up to the few
elements (about 0.1 % at K = 2240) whose fp32 and fp64 sums round to neighbouring
bf16 values.  Shapes span
several 128-row and 256-column tiles with ragged tails in rows, columns and K.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_wise_b300 import gdn
from gated_deltanet_wise_b300.inputs import make_block_inputs
from tests.conftest import rel_fro

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL = 5e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    gdn.lib()
    yield
    assert gdn.gdn_device_status() == gdn.GDN_OK


def _in_proj(xb):
    B, H, F, N, D = xb.B, xb.H, xb.F, xb.N, xb.D
    q = torch.empty(B, F * N, H, D, dtype=torch.bfloat16, device=DEV)
    k, v = torch.empty_like(q), torch.empty_like(q)
    beta = torch.empty(B, F * N, H, device=DEV)
    gamma = torch.empty(B, F, H, device=DEV)
    st = gdn.gdn_block_in_proj(xb.x, xb.W_in, q, k, v, beta, gamma, B, H, F, N, D)
    assert st == gdn.GDN_OK, gdn.status_string(st)
    torch.cuda.synchronize()
    return q, k, v, beta, gamma


@pytest.mark.parametrize("B,H,F,N", [(1, 2, 3, 100), (2, 20, 2, 150), (1, 1, 1, 1)])
def test_in_proj_matches_oracle(B, H, F, N):
    xb = make_block_inputs(B, H, F, N, seed=70 + H + N, device=DEV)
    got = _in_proj(xb)
    ref = oracle.block_in_proj(xb.x, xb.W_in, F)
    for name, a, r in zip(("q", "k", "v"), got[:3], ref[:3]):
        a = a.float().cpu().numpy()
        assert rel_fro(a, r) <= 1e-3, name
        assert np.mean(a != r) < 1e-2, name   # nearly every element is the same bf16 value (K = 2240 sums)
    assert rel_fro(got[3].cpu().numpy(), ref[3]) <= 1e-5
    assert rel_fro(got[4].cpu().numpy(), ref[4]) <= 1e-5


@pytest.mark.parametrize("B,H,F,N", [(1, 2, 3, 100), (2, 20, 2, 150)])
def test_out_proj_matches_fp64(B, H, F, N):
    xb = make_block_inputs(B, H, F, N, seed=80 + N, device=DEV)
    HD = H * 112
    o = torch.randn(B, F * N, HD, device=DEV).to(torch.bfloat16)
    y = torch.empty_like(o)
    st = gdn.gdn_block_out_proj(o, xb.W_out, y, B, H, F, N, 112)
    assert st == gdn.GDN_OK
    torch.cuda.synchronize()
    ref = o.double().cpu().numpy() @ xb.W_out.double().cpu().numpy().T
    assert rel_fro(y.float().cpu().numpy(), ref) <= TOL


@pytest.mark.parametrize("B,H,F,N,s0", [(1, 20, 4, 220, 0.0), (2, 3, 5, 130, 0.1), (1, 20, 8, 880, 0.0)])
def test_block_fwd_matches_oracle(B, H, F, N, s0):
    xb = make_block_inputs(B, H, F, N, seed=90 + F + N, device=DEV, s0_std=s0)
    y, S = gdn.block_fwd(xb.x, xb.W_in, xb.W_out, xb.S0, F=F)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    y_ref, S_ref = oracle.block_fwd(xb.x, xb.W_in, xb.W_out, xb.S0, F=F)
    ey = rel_fro(y.float().cpu().numpy(), y_ref)
    es = rel_fro(S.cpu().numpy(), S_ref)
    print(f"block B={B} H={H} F={F} N={N}: rel_fro y={ey:.2e} S={es:.2e}")
    assert ey <= TOL and es <= TOL


def test_block_degenerate_and_rejected_sizes():
    xb = make_block_inputs(1, 2, 2, 8, seed=3, device=DEV, s0_std=0.2)
    S = torch.empty(1, 2, 112, 112, device=DEV)
    e = torch.empty(0, dtype=torch.bfloat16, device=DEV)
    # no frames: the state passes through
    assert gdn.gdn_block_fwd(e, xb.W_in, xb.W_out, xb.S0, S, e, 1, 2, 0, 8, 112, 0.0, None, 0) == gdn.GDN_OK
    torch.cuda.synchronize()
    assert torch.equal(S, xb.S0)
    assert gdn.gdn_block_fwd(xb.x, xb.W_in, xb.W_out, None, S, xb.x, 1, 2, 2, 0, 112, 0.0, None, 0) == \
        gdn.GDN_ERR_UNSUPPORTED
    assert gdn.gdn_block_fwd(xb.x, xb.W_in, xb.W_out, None, S, xb.x, 1, 2, 2, 8, 64, 0.0, None, 0) == \
        gdn.GDN_ERR_UNSUPPORTED
    nb = gdn.gdn_block_fwd_workspace_size(1, 2, 2, 8, 112)
    ws = torch.empty(nb, dtype=torch.uint8, device=DEV)
    y = torch.empty_like(xb.x)
    assert gdn.gdn_block_fwd(xb.x, xb.W_in, xb.W_out, None, S, y, 1, 2, 2, 8, 112, 0.0, ws, nb - 256) == \
        gdn.GDN_ERR_WORKSPACE
