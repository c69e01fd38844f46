"""The streaming step that allocates nothing (gdn_frame_step_noalloc).

Some callers cannot allocate device memory where they run a frame (a host that
owns the device memory budget, a real-time per-frame loop, code inside a stream
capture), so this entry point takes its scratch from a fixed array inside the
library instead of a caller workspace.  The test calls it through the C ABI and
checks it against gdn_frame_step, which takes a caller workspace, on two calls
in a row with different inputs: the shared array keeps the previous call's
contents, so the second call also shows that nothing stale leaks through.

Kept in a file of its own, collected last.
"""
import pytest
import torch

from gated_deltanet_wise_b300 import gdn
from gated_deltanet_wise_b300.inputs import make_inputs
from tests.conftest import rel_fro

pytestmark = pytest.mark.gpu

TOL_BF16 = 5e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    gdn.lib()


def _step_inputs(seed, B, H, N):
    x = make_inputs(B, H, 1, N, 112, dtype="bf16", seed=seed, device="cuda", s0_std=0.1)
    return x.q, x.k, x.v, x.beta, x.gamma[:, 0].contiguous(), x.S0


def test_noalloc_step_matches_workspace_step_on_two_calls():
    B, H, N, D = 1, 20, 880, 112
    assert gdn.gdn_frame_fwd_workspace_size(B, H, 1, N, D) <= gdn.gdn_frame_step_noalloc_limit_bytes()
    for call, seed in enumerate((21, 22)):
        q, k, v, beta, gamma, S0 = _step_inputs(seed, B, H, N)
        o_ref, S_ref = gdn.frame_step(q, k, v, beta, gamma, S0)
        o = torch.empty_like(q)
        S = torch.empty_like(S_ref)
        st = gdn.gdn_frame_step_noalloc(q, k, v, beta, gamma, S0, S, o, B, H, N, D, 0.0)
        assert st == gdn.GDN_OK, (call, gdn.status_string(st))
        torch.cuda.synchronize()
        assert rel_fro(o.float().cpu().numpy(), o_ref.float().cpu().numpy()) <= TOL_BF16, call
        assert rel_fro(S.cpu().numpy(), S_ref.cpu().numpy()) <= TOL_BF16, call
    assert gdn.gdn_device_status() == gdn.GDN_OK


def test_noalloc_step_rejects_requests_beyond_its_scratch():
    limit = gdn.gdn_frame_step_noalloc_limit_bytes()
    B, H = 4, 40   # 160 chains: beyond the fixed scratch
    assert gdn.gdn_frame_fwd_workspace_size(B, H, 1, 880, 112) > limit
    fake = torch.empty(16, dtype=torch.uint8, device="cuda")   # never touched: rejected on the host
    st = gdn.gdn_frame_step_noalloc(fake, fake, fake, fake, fake, None, fake, fake, B, H, 880, 112, 0.0)
    assert st == gdn.GDN_ERR_WORKSPACE
