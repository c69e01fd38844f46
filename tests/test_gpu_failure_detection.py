"""Failure detection on the GPU without a fault: a bounded device-side wait runs out.

The test entry gdn_test_frame_fwd_expired_wait runs the forward with the
frame-statistics kernel's loads withheld, so the first pipeline stage never
fills.  The consumers' waits on it are bounded (about 2 s of GPU time); when
they expire the kernel raises its abort flag, every role leaves its loop, the
tensor memory is freed and the kernel returns.  Nothing traps, faults or waits
without a limit.  The host then reads GDN_ERR_TIMEOUT from the status word, and
the same process goes on to run a normal forward that matches the oracle.
"""
import pytest
import torch

import oracle
from gated_deltanet_wise_b300 import gdn
from gated_deltanet_wise_b300.inputs import make_inputs
from tests.conftest import rel_fro

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    gdn.lib()
    assert gdn.gdn_device_status() == gdn.GDN_OK   # nothing left over from earlier tests


def test_expired_wait_reports_timeout_and_context_survives():
    x = make_inputs(1, 2, 3, 96, 112, dtype="bf16", seed=31, device=DEV, s0_std=0.1)
    B, H, F, N, D = x.B, x.H, x.F, x.N, x.D
    nb = gdn.gdn_frame_fwd_workspace_size(B, H, F, N, D)
    ws = torch.empty(nb, dtype=torch.uint8, device=DEV)
    o = torch.empty_like(x.q)
    S = torch.empty(B, H, D, D, device=DEV)
    st = gdn.gdn_test_frame_fwd_expired_wait(x.q, x.k, x.v, x.beta, x.gamma, x.S0, S, o, B, H, F, N, D, 0.0,
                                             ws, nb)
    assert st == gdn.GDN_OK   # the call itself enqueues normally
    assert gdn.gdn_device_status() == gdn.GDN_ERR_TIMEOUT
    assert gdn.gdn_device_status() == gdn.GDN_OK   # reading the word clears it
    # the context is intact: a normal forward right after is correct
    o2, S2 = gdn.frame_fwd(x.q, x.k, x.v, x.beta, x.gamma, x.S0)
    assert gdn.gdn_device_status() == gdn.GDN_OK
    o_ref, S_ref = oracle.frame_fwd(x.q, x.k, x.v, x.beta, x.gamma, x.S0)
    assert rel_fro(o2.float().cpu().numpy(), o_ref) <= 5e-3
    assert rel_fro(S2.cpu().numpy(), S_ref) <= 5e-3
