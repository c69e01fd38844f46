"""Context-parallel frame-wise GDN forward: the frame axis split across ranks.

Summary page "SANA-WM: Efficient Minute-Scale World Modeling with Hybrid Linear
Diffusion Transformer", section 技术新颖性: for context-parallel training the
frames are split across devices, and a prefix-sum exchange of each device's
transition composite C_p and input composite H_p recovers the single-device
result exactly.

A run of frames acts on the state as the affine map S -> S C_p + H_p
(C_p = M_{f0} ... M_{f1-1}, H_p = the state the run reaches from zero).  Rank p
owns a contiguous run of frames.  It computes (C_p, H_p) from its own k, v,
beta, gamma; one all-gather gives every rank every (C_r, H_r); rank p composes
the maps of ranks 0..p-1 onto the initial state,

    S_start(p) = (...((S_in C_0 + H_0) C_1 + H_1) ...) C_{p-1} + H_{p-1},

and runs its frames from S_start(p).  The last rank's final state is the
layer's S_out, and its own composites are never composed, so it runs only the
statistics pass its forward resumes from.  The arithmetic runs in the CUDA
library (gdn_frame_composite, gdn_state_compose, gdn_frame_fwd_resume); this
module holds only the split and the exchange, and takes its operations as
arguments so that the exchange logic can be exercised without a GPU.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Callable, List, Optional, Sequence, Tuple


def frame_split(F: int, world: int) -> List[Tuple[int, int]]:
    """Contiguous frame runs [f0, f1) per rank, sizes differing by at most one."""
    if world <= 0 or F < 0:
        raise ValueError("world must be positive and F non-negative")
    base, extra = divmod(F, world)
    out, f0 = [], 0
    for r in range(world):
        n = base + (1 if r < extra else 0)
        out.append((f0, f0 + n))
        f0 += n
    return out


@dataclass
class CpOps:
    """The per-rank operations: composite(k, v, beta, gamma) -> (C, H);
    compose(S or None, C, H) -> S C + H; forward(q, k, v, beta, gamma, S) -> (o, S_out);
    and optionally statistics(k, v, beta, gamma) -> placeholders shaped and typed like
    (C, H), called instead of composite on the last rank, whose composites no rank reads
    (the library form still runs the statistics pass its forward resumes from)."""
    composite: Callable
    compose: Callable
    forward: Callable
    statistics: Optional[Callable] = None


def library_ops(key_scale: float = 0.0) -> CpOps:
    """The CUDA library's operations (device tensors) for one rank.

    The composite pass is the forward's frame-statistics pass over the rank's
    frames; its per-frame statistics stay in this rank's workspace, and the
    forward resumes from them (gdn_frame_fwd_resume), so each rank reads its k,
    v and beta once.  Use one instance per rank and call composite before
    forward on the same frames."""
    from gated_deltanet_wise_b300 import gdn
    ws = gdn.Workspace()

    def composite(k, v, beta, gamma):
        return gdn.frame_composite(k, v, beta, gamma, key_scale=key_scale, workspace=ws)

    def statistics(k, v, beta, gamma):
        import torch
        gdn.frame_composite(k, v, beta, gamma, key_scale=key_scale, workspace=ws, outputs=False)
        z = torch.zeros(k.shape[0], k.shape[2], k.shape[3], k.shape[3], dtype=torch.float32, device=k.device)
        return z, z

    def compose(S, C, H):
        return gdn.state_compose(S, C, H)

    def forward(q, k, v, beta, gamma, S):
        return gdn.frame_fwd_resume(q, gamma, S, workspace=ws)

    return CpOps(composite, compose, forward, statistics)


def start_state(S_in, composites: Sequence[Tuple[object, object]], rank: int, compose: Callable):
    """Exclusive prefix: the state at the start of `rank`'s run of frames."""
    S = S_in
    for r in range(rank):
        C, H = composites[r]
        S = compose(S, C, H)
    return S


def cp_forward(q, k, v, beta, gamma, S_in=None, *, ops: Optional[CpOps] = None, group=None):
    """Forward pass of this rank's run of frames (its slices of q, k, v, beta, gamma).

    S_in is the layer's initial state (the same on every rank, or None for zero).
    Returns (o for this rank's frames, this rank's final state); on the last
    rank the final state is the layer's S_out.  The only communication is one
    all-gather of the per-rank composites.
    """
    import torch
    import torch.distributed as dist

    ops = ops or library_ops()
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    # the last rank's composites are gathered but no rank composes them
    last = rank == world - 1 and ops.statistics is not None
    C, H = (ops.statistics if last else ops.composite)(k, v, beta, gamma)
    CH = torch.stack([C, H]).contiguous()   # one message per rank: (C_p, H_p) back to back
    parts = [torch.empty_like(CH) for _ in range(world)]
    dist.all_gather(parts, CH, group=group)
    S_start = start_state(S_in, [(x[0], x[1]) for x in parts], rank, ops.compose)
    return ops.forward(q, k, v, beta, gamma, S_start)
