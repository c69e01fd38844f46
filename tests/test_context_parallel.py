"""Context-parallel exchange (frames split across ranks) on CPU gloo ranks.

Two (and three) processes each own a contiguous run of frames, compute their
composites, all-gather them, compose the exclusive prefix onto S_in and run
their frames.  The per-rank arithmetic is the fp64 oracle here, passed in as
the operations, so these tests exercise the split and the exchange of
gated_deltanet_wise_b300.context_parallel without a GPU; together the ranks
must reproduce one sequential pass over all frames (the exactness the summary
page's section 技术新颖性 states for the C_p / H_p prefix exchange).
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from gated_deltanet_wise_b300.context_parallel import CpOps, cp_forward, frame_split, start_state

B, H, N, D = 1, 2, 6, 8


def _inputs(F, seed=0):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, F * N, H, D)).astype(np.float32)
    k = rng.standard_normal((B, F * N, H, D)).astype(np.float32)
    v = rng.standard_normal((B, F * N, H, D)).astype(np.float32)
    beta = (1 / (1 + np.exp(-rng.standard_normal((B, F * N, H))))).astype(np.float32)
    gamma = (1 / (1 + np.exp(rng.standard_normal((B, F, H))))).astype(np.float32)
    S0 = rng.standard_normal((B, H, D, D)).astype(np.float32)
    return q, k, v, beta, gamma, S0


def _oracle_ops(with_statistics=False):
    import oracle

    def composite(k, v, beta, gamma):
        M, U = oracle.frame_transitions(k.numpy(), v.numpy(), beta.numpy(), gamma.numpy(), key_scale=0.5)
        C = np.zeros((B, H, D, D)); Hc = np.zeros((B, H, D, D))
        for b in range(B):
            for h in range(H):
                C[b, h], Hc[b, h] = oracle.composite(M[b, h], U[b, h])
        return torch.from_numpy(C), torch.from_numpy(Hc)

    def compose(S, C, Hc):
        return Hc.clone() if S is None else torch.matmul(S, C) + Hc

    def forward(q, k, v, beta, gamma, S):
        o, S_out = oracle.frame_fwd(q.numpy(), k.numpy(), v.numpy(), beta.numpy(), gamma.numpy(),
                                    None if S is None else S.numpy().astype(np.float32), key_scale=0.5)
        return torch.from_numpy(o), torch.from_numpy(S_out)

    def statistics(k, v, beta, gamma):
        # the last rank's placeholders: NaN, so that a rank composing them would show it
        nan = torch.full((B, H, D, D), float("nan"), dtype=torch.float64)
        return nan, nan.clone()

    return CpOps(composite, compose, forward, statistics if with_statistics else None)


def _rank_main(rank, world, port, F, out_dir, with_statistics=False):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q, k, v, beta, gamma, S0 = _inputs(F)
        f0, f1 = frame_split(F, world)[rank]
        sl = slice(f0 * N, f1 * N)
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
        o, S_end = cp_forward(t(q[:, sl]), t(k[:, sl]), t(v[:, sl]), t(beta[:, sl]), t(gamma[:, f0:f1]),
                              torch.from_numpy(S0.astype(np.float64)), ops=_oracle_ops(with_statistics))
        np.save(os.path.join(out_dir, f"o_{rank}.npy"), o.numpy())
        np.save(os.path.join(out_dir, f"S_{rank}.npy"), S_end.numpy())
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("world,F,with_statistics", [(2, 6, False), (2, 5, False), (3, 7, False), (3, 7, True)])
def test_ranks_reproduce_one_sequential_pass(tmp_path, world, F, with_statistics):
    """with_statistics: the last rank forms no composites (NaN placeholders go into the
    all-gather); the result is unchanged because no rank composes them."""
    import oracle
    mp.spawn(_rank_main, args=(world, _free_port(), F, str(tmp_path), with_statistics), nprocs=world, join=True)
    q, k, v, beta, gamma, S0 = _inputs(F)
    o_ref, S_ref = oracle.frame_fwd(q, k, v, beta, gamma, S0, key_scale=0.5)
    o = np.concatenate([np.load(tmp_path / f"o_{r}.npy") for r in range(world)], axis=1)
    # the composites and the prefix are fp64; the only rounding is the oracle's
    # fp32 interface for a run's initial state (relative 2^-24 on S_start)
    tol = 1e-6
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=tol * np.abs(o_ref).max())
    np.testing.assert_allclose(np.load(tmp_path / f"S_{world - 1}.npy"), S_ref, rtol=0, atol=tol * np.abs(S_ref).max())


def test_frame_split_is_contiguous_and_balanced():
    for F in range(0, 13):
        for world in range(1, 6):
            runs = frame_split(F, world)
            assert runs[0][0] == 0 and runs[-1][1] == F
            assert all(a[1] == b[0] for a, b in zip(runs, runs[1:]))
            sizes = [r[1] - r[0] for r in runs]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        frame_split(4, 0)


def test_start_state_is_the_exclusive_prefix():
    rng = np.random.default_rng(2)
    comps = [(rng.standard_normal((3, 3)), rng.standard_normal((3, 3))) for _ in range(4)]
    S0 = rng.standard_normal((3, 3))
    compose = lambda S, C, Hc: Hc if S is None else S @ C + Hc
    assert start_state(S0, comps, 0, compose) is S0
    S2 = start_state(S0, comps, 2, compose)
    np.testing.assert_allclose(S2, (S0 @ comps[0][0] + comps[0][1]) @ comps[1][0] + comps[1][1])
    np.testing.assert_allclose(start_state(None, comps, 1, compose), comps[0][1])
