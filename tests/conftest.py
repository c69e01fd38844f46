import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU oracle case")


def rel_fro(a, b):
    """Relative Frobenius error ||a - b||_F / ||b||_F in fp64."""
    import numpy as np
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b.ravel())
    return float(np.linalg.norm((a - b).ravel()) / (nb if nb > 0 else 1.0))


def chain_groups(B, H, bytes_per_chain, budget=32e9):
    """(b, h0, h1) head groups covering every (batch, head) chain, each group small
    enough that the oracle's fp32 inputs and fp64 outputs for it stay within
    `budget` bytes of host memory.  The oracle runs the chains of one call in
    parallel, so larger groups use more host cores."""
    per = max(1, min(H, int(budget // max(1, bytes_per_chain))))
    for b in range(B):
        for h0 in range(0, H, per):
            yield b, h0, min(H, h0 + per)


def check_every_chain(x, o, S, ref_fn, tol):
    """Compare the GPU outputs o [B, F*N, H, D] and S [B, H, D, D] with ref_fn on
    every (batch, head) chain; ref_fn(q, k, v, beta, gamma, S0) returns the fp64
    (o, S_out) of the head group it is given.  Returns the worst chain error."""
    B, FN, H, D = x.q.shape
    per_chain = FN * D * (3 * 4 + 8 + 8) + 4 * D * D * 8
    worst = 0.0
    for b, h0, h1 in chain_groups(B, H, per_chain):
        def sl(t):
            return None if t is None else t[b:b + 1, :, h0:h1].contiguous()
        S0 = None if x.S0 is None else x.S0[b:b + 1, h0:h1].contiguous()
        o_ref, S_ref = ref_fn(sl(x.q), sl(x.k), sl(x.v), sl(x.beta), sl(x.gamma), S0)
        for j, h in enumerate(range(h0, h1)):
            eo = rel_fro(o[b:b + 1, :, h:h + 1].float().cpu().numpy(), o_ref[:, :, j:j + 1])
            es = rel_fro(S[b:b + 1, h:h + 1].float().cpu().numpy(), S_ref[:, j:j + 1])
            assert eo <= tol and es <= tol, ((b, h), eo, es)
            worst = max(worst, eo, es)
        del o_ref, S_ref
    return worst
