"""Sequence parallelism for causal linear attention (LASP-2).

A sequence too long for one device is split into consecutive parts, one per
rank.  Every rank summarises its own part as a fixed-size state U_r (its final
state from a zero start), the ranks all-gather those states -- B*H*(d*dv + d)
floats each, independent of the sequence length -- and each rank forms the
state before its part as the exclusive prefix

    P_0 = 0,   P_{r+1} = gamma^(len_r) P_r + U_r

then runs its part's forward from P_r ("Linear Attention and SSM", LASP-2
section: one gather of fixed-size states instead of passing the state from
rank to rank; "Efficient Attention Variants", sections 5 and 7.1).

Every step runs in the library's kernels (la_state, la_state_prefix,
la_forward_with_state); the only exchange is the all-gather, done by
torch.distributed.  `ops` lets a caller substitute the three steps (the
multi-rank CPU tests drive the exchange with other implementations of them).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Callable

import torch


@dataclass
class LaspOps:
    """The three local steps of a rank."""
    local_state: Callable  # (k, v, feature_map, gamma) -> (S [B,H,d,dv], z [B,H,d])
    prefix: Callable       # (S_parts, z_parts, lens, upto, gamma) -> (S, z)
    forward: Callable      # (q, k, v, S0, z0, feature_map, gamma) -> out [B,H,N,dv]


def library_ops() -> LaspOps:
    from . import _binding as b

    return LaspOps(
        local_state=lambda k, v, fm, g: b.la_state(k, v, feature_map=fm, gamma=g),
        prefix=lambda S, z, lens, upto, g: b.la_state_prefix(S, z, lens, upto, gamma=g),
        forward=lambda q, k, v, S0, z0, fm, g: b.la_forward_with_state(
            q, k, v, S0=S0, z0=z0, feature_map=fm, gamma=g, return_state=False)[0],
    )


def lasp2_forward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, group=None,
                  feature_map="elu1", gamma=None, ops: LaspOps | None = None) -> torch.Tensor:
    """Causal forward of this rank's part (q, k [B,H,n_r,d], v [B,H,n_r,dv]) of
    a sequence split over the ranks of `group` in rank order."""
    import torch.distributed as dist

    ops = ops or library_ops()
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    S, z = ops.local_state(k, v, feature_map, gamma)
    S_all = [torch.empty_like(S) for _ in range(world)]
    z_all = [torch.empty_like(z) for _ in range(world)]
    n = torch.tensor([k.shape[2]], dtype=torch.int64, device=S.device)
    n_all = [torch.empty_like(n) for _ in range(world)]
    dist.all_gather(S_all, S.contiguous(), group=group)
    dist.all_gather(z_all, z.contiguous(), group=group)
    dist.all_gather(n_all, n, group=group)
    lens = [int(x.item()) for x in n_all]
    S0, z0 = ops.prefix(torch.stack(S_all), torch.stack(z_all), lens, rank, gamma)
    return ops.forward(q, k, v, S0, z0, feature_map, gamma)


def lasp2_forward_emulated(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, parts, *,
                           feature_map="elu1", gamma=None,
                           ops: LaspOps | None = None) -> torch.Tensor:
    """The same split on one device: the sequence [B,H,N,*] is cut at the
    token counts `parts` (summing to N), every part's state is computed on its
    own, the "all-gather" is a stack, and each part runs from its prefix.
    Returns the concatenated outputs [B,H,N,dv]."""
    ops = ops or library_ops()
    assert sum(parts) == q.shape[2]
    cuts, lo = [], 0
    for n in parts:
        cuts.append((lo, lo + n))
        lo += n
    sl = [(q[:, :, a:b].contiguous(), k[:, :, a:b].contiguous(), v[:, :, a:b].contiguous())
          for a, b in cuts]
    states = [ops.local_state(kk, vv, feature_map, gamma) for _, kk, vv in sl]
    S_all = torch.stack([s for s, _ in states])
    z_all = torch.stack([z for _, z in states])
    outs = []
    for r, (qq, kk, vv) in enumerate(sl):
        S0, z0 = ops.prefix(S_all, z_all, list(parts), r, gamma)
        outs.append(ops.forward(qq, kk, vv, S0, z0, feature_map, gamma))
    return torch.cat(outs, dim=2)
