"""GPU entry points of the context-parallel path: per-run composites
(gdn_frame_composite), composition onto a state (gdn_state_compose), and a
frame split emulated on one GPU (no collective: the runs execute one after
another) against one gdn_frame_fwd call and the fp64 oracle.
Tolerance: relative Frobenius error <= 5e-3 (bf16 inputs, fp32 state)."""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_wise_b300 import gdn
from gated_deltanet_wise_b300.context_parallel import frame_split, library_ops, start_state
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


def test_frame_composite_matches_oracle():
    x = make_inputs(1, 3, 5, 200, 112, dtype="bf16", seed=31, device=DEV)
    C, Hc = gdn.frame_composite(x.k, x.v, x.beta, x.gamma)
    torch.cuda.synchronize()
    M, U = oracle.frame_transitions(x.k, x.v, x.beta, x.gamma)
    for h in range(3):
        C_ref, H_ref = oracle.composite(M[0, h], U[0, h])
        assert rel_fro(C[0, h].cpu().numpy(), C_ref) <= 1e-3
        assert rel_fro(Hc[0, h].cpu().numpy(), H_ref) <= TOL


def test_frame_composite_without_tokens_is_pure_decay():
    gamma = torch.rand(2, 4, 3, device=DEV) * 0.9 + 0.05
    e = torch.empty(2, 0, 3, 112, dtype=torch.bfloat16, device=DEV)
    C, Hc = gdn.frame_composite(e, e, torch.empty(2, 0, 3, device=DEV), gamma)
    torch.cuda.synchronize()
    eye = torch.eye(112, device=DEV)
    torch.testing.assert_close(C, gamma.prod(1)[:, :, None, None] * eye, rtol=1e-6, atol=1e-7)
    assert torch.count_nonzero(Hc) == 0


def test_state_compose_matches_fp64():
    g = torch.Generator(device=DEV).manual_seed(3)
    S, C, Hc = (torch.randn(5, 112, 112, generator=g, device=DEV) for _ in range(3))
    out = gdn.state_compose(S, C, Hc)
    ref = S.double() @ C.double() + Hc.double()
    assert rel_fro(out.cpu().numpy(), ref.cpu().numpy()) < 1e-5
    out0 = gdn.state_compose(None, C, Hc)
    torch.testing.assert_close(out0, Hc)
    S_alias = S.clone()
    gdn.state_compose(S_alias, C, Hc, out=S_alias)
    torch.testing.assert_close(S_alias, out)


@pytest.mark.parametrize("world", [2, 3])
def test_split_runs_equal_one_forward(world):
    """Frames split into runs: composites, exclusive prefix, per-run forward == one forward."""
    B, H, F, N = 1, 4, 9, 300
    x = make_inputs(B, H, F, N, 112, dtype="bf16", seed=40 + world, device=DEV, s0_std=0.1)
    o_ref, S_ref = gdn.frame_fwd(x.q, x.k, x.v, x.beta, x.gamma, x.S0)
    runs = frame_split(F, world)
    ops = [library_ops() for _ in runs]   # one per emulated rank: each keeps its statistics
    sl = lambda t, f0, f1: t[:, f0 * N:f1 * N].contiguous()
    comps = []
    for i, r in enumerate(runs):
        args = (sl(x.k, *r), sl(x.v, *r), sl(x.beta, *r), x.gamma[:, r[0]:r[1]].contiguous())
        if i == len(runs) - 1:
            # the last run, as cp_forward runs it: the statistics pass alone; its placeholders
            # are filled with NaN, so a rank that composed them would show it
            C, Hc = ops[i].statistics(*args)
            C.fill_(float("nan"))
            Hc.fill_(float("nan"))
            comps.append((C, Hc))
        else:
            comps.append(ops[i].composite(*args))
    outs, S_end = [], None
    for rank, r in enumerate(runs):
        S_start = start_state(x.S0, comps, rank, ops[rank].compose)
        o, S_end = ops[rank].forward(sl(x.q, *r), sl(x.k, *r), sl(x.v, *r), sl(x.beta, *r),
                                     x.gamma[:, r[0]:r[1]].contiguous(), S_start)
        outs.append(o)
    torch.cuda.synchronize()
    o = torch.cat(outs, 1)
    assert rel_fro(o.float().cpu().numpy(), o_ref.float().cpu().numpy()) <= TOL
    assert rel_fro(S_end.cpu().numpy(), S_ref.cpu().numpy()) <= TOL
    o_orc, S_orc = oracle.frame_fwd(x.q, x.k, x.v, x.beta, x.gamma, x.S0)
    assert rel_fro(o.float().cpu().numpy(), o_orc) <= TOL
    assert rel_fro(S_end.cpu().numpy(), S_orc) <= TOL


@pytest.mark.parametrize("outputs", [True, False])
def test_resume_equals_forward_and_reads_no_keys(outputs):
    """gdn_frame_fwd_resume after gdn_frame_composite on the same frames equals the three-launch forward
    (several chunks, a random start state), also when the composite call forms no composites
    (C_out = H_out = NULL, the last rank's form); k, v and beta are not read again (they are
    overwritten with NaN before the resume)."""
    B, H, F, N = 2, 3, 23, 150
    x = make_inputs(B, H, F, N, 112, dtype="bf16", seed=77, device=DEV, s0_std=0.1)
    o_ref, S_ref = gdn.frame_fwd_ex(x.q, x.k, x.v, x.beta, x.gamma, x.S0)  # three launches
    ws = gdn.Workspace()
    C, Hc = gdn.frame_composite(x.k, x.v, x.beta, x.gamma, workspace=ws, outputs=outputs)
    assert (C is None) == (not outputs)
    for t in (x.k, x.v, x.beta):
        t.fill_(float("nan"))
    o, S = gdn.frame_fwd_resume(x.q, x.gamma, x.S0, workspace=ws)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status() == gdn.GDN_OK
    assert rel_fro(o.float().cpu().numpy(), o_ref.float().cpu().numpy()) <= 1e-6
    assert rel_fro(S.cpu().numpy(), S_ref.cpu().numpy()) <= 1e-6
    if outputs:  # the composites describe the same run: S_out = S_in C + H
        S_comp = gdn.state_compose(x.S0, C, Hc)
        assert rel_fro(S_comp.cpu().numpy(), S_ref.cpu().numpy()) <= TOL
