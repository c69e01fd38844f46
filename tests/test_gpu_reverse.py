"""Reverse-direction scan (gdn_frame_fwd_ex with GDN_FWD_REVERSE) on the GPU:
the frames are visited from the last to the first, for the sum and the
product readings, against the fp64 oracle's reverse mode, and bit for bit
against the forward scan of the frame-reversed sequence (same plan, same
arithmetic, only the frame addressing differs).
Tolerance: relative Frobenius error <= 5e-3 on o and S_out."""
import pytest
import torch

import oracle
from gated_deltanet_wise_b300 import gdn
from gated_deltanet_wise_b300.inputs import make_inputs
from tests.conftest import rel_fro

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


def _flip(x, F):
    B, FN = x.shape[:2]
    return x.reshape(B, F, FN // F, *x.shape[2:]).flip(1).reshape(x.shape).contiguous()


@pytest.mark.parametrize("product", [False, True])
@pytest.mark.parametrize("B,H,F,N,ks", [(1, 2, 9, 150, 0.0), (2, 1, 5, 200, 0.5), (1, 3, 12, 64, 1.0)])
def test_reverse_matches_oracle(product, B, H, F, N, ks):
    x = make_inputs(B, H, F, N, 112, dtype="bf16", seed=60 + F, device=DEV, s0_std=0.1)
    o, S = gdn.frame_fwd_ex(x.q, x.k, x.v, x.beta, x.gamma, x.S0, product=product, reverse=True, key_scale=ks)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    o_ref, S_ref = oracle.frame_fwd(x.q, x.k, x.v, x.beta, x.gamma, x.S0, key_scale=ks,
                                    mode="product" if product else "sum", reverse=True)
    assert rel_fro(o.float().cpu().numpy(), o_ref) <= TOL
    assert rel_fro(S.cpu().numpy(), S_ref) <= TOL


@pytest.mark.parametrize("product", [False, True])
def test_reverse_is_forward_of_the_reversed_frames_bit_for_bit(product):
    B, H, F, N = 1, 3, 11, 300
    x = make_inputs(B, H, F, N, 112, dtype="bf16", seed=71, device=DEV, s0_std=0.1)
    o_r, S_r = gdn.frame_fwd_ex(x.q, x.k, x.v, x.beta, x.gamma, x.S0, product=product, reverse=True)
    o_f, S_f = gdn.frame_fwd_ex(_flip(x.q, F), _flip(x.k, F), _flip(x.v, F), _flip(x.beta, F),
                                x.gamma.flip(1).contiguous(), x.S0, product=product)
    torch.cuda.synchronize()
    assert torch.equal(o_r, _flip(o_f, F))
    assert torch.equal(S_r, S_f)


def test_reverse_layer_size_sampled_heads():
    """The 20-head layer (F=121, N=880) reversed in one call; two heads checked."""
    x = make_inputs(1, 20, 121, 880, 112, dtype="bf16", seed=72, device=DEV)
    o, S = gdn.frame_fwd_ex(x.q, x.k, x.v, x.beta, x.gamma, None, reverse=True)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    for h in (3, 17):
        sl = lambda t: t[:, :, h:h + 1].contiguous()
        o_ref, S_ref = oracle.frame_fwd(sl(x.q), sl(x.k), sl(x.v), sl(x.beta), sl(x.gamma), None, reverse=True)
        assert rel_fro(o[:, :, h:h + 1].float().cpu().numpy(), o_ref) <= TOL
        assert rel_fro(S[:, h:h + 1].cpu().numpy(), S_ref) <= TOL
