"""Context parallelism: one batch of sequences split along time into contiguous
shards, one per rank (cross-GPU sequence parallelism).

The recurrence is affine in the state (onedev.kr FlashQLA talk summary,
paragraph on parallelism across cards): over a shard,

    S_end = S_start @ M + E,       M = S_end(v = 0, S_start = I),  E = S_end(S_start = 0)

(S is d_v x d_k, M is d_k x d_k), and the reverse recurrence of the gradient is

    dS_start = dS_end @ R + F,     R = M^T,  F = dS_start(dS_end = 0)

because every per-token factor alpha (I - beta k k^T) is symmetric.  So each rank
summarises its shard (E, M), the summaries are all-gathered (the one exchange
step), every rank composes the summaries of the ranks before it into its exact
start state and reruns its shard; the backward does the same in reverse order
with (F, M^T).  No tensor other than the per-(sequence, head) summaries crosses
ranks.

The per-shard work goes through the library's own entry points
(``chunk_gated_delta_rule_fwd`` / ``_bwd``); ``ShardFns`` lets a caller supply
other implementations with the same signatures.  ``compose_forward`` /
``compose_backward`` are the pure composition steps, usable without a process
group (all shards in one process).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Callable, List, Optional, Sequence

import torch


@dataclass
class ShardFns:
    """fwd(q, k, v, g, beta, S0) -> (o, S_T);  bwd(q, k, v, g, beta, dO, S0, dS_T) -> (dq, dk, dv, dg, dbeta, dS0)."""
    fwd: Callable
    bwd: Callable


def library_fns(scale: Optional[float] = None, l2norm: bool = False) -> ShardFns:
    from . import chunk_gated_delta_rule_bwd, chunk_gated_delta_rule_fwd

    def fwd(q, k, v, g, beta, S0):
        return chunk_gated_delta_rule_fwd(q, k, v, g, beta, S0, True, None, scale, l2norm)

    def bwd(q, k, v, g, beta, dO, S0, dS_T):
        return chunk_gated_delta_rule_bwd(q, k, v, g, beta, dO, S0, dS_T, None, scale, l2norm)

    return ShardFns(fwd, bwd)


def _identity_state(B: int, H: int, D: int, like: torch.Tensor) -> torch.Tensor:
    return torch.eye(D, dtype=torch.float32, device=like.device).expand(B, H, D, D).contiguous()


def shard_summary(fns: ShardFns, q, k, v, g, beta):
    """(E, M) of one shard: end state from a zero start, and the transition (v = 0 from I)."""
    B, _, H, D = q.shape
    _, E = fns.fwd(q, k, v, g, beta, torch.zeros(B, H, v.shape[-1], D, dtype=torch.float32, device=q.device))
    _, M = fns.fwd(q, k, torch.zeros_like(v), g, beta, _identity_state(B, H, D, q))
    return E, M


def compose_forward(S0: Optional[torch.Tensor], summaries: Sequence, rank: int) -> torch.Tensor:
    """Exact start state of shard `rank`: fold S <- S @ M_j + E_j over the shards j < rank."""
    E0, M0 = summaries[0]
    S = torch.zeros_like(E0) if S0 is None else S0.to(E0.dtype)
    for j in range(rank):
        E, M = summaries[j]
        S = torch.matmul(S, M) + E
    return S


def compose_backward(dS_T: Optional[torch.Tensor], F_list: Sequence, M_list: Sequence, rank: int) -> torch.Tensor:
    """Exact end gradient of shard `rank`: fold X <- X @ M_j^T + F_j over the shards j > rank, from the last."""
    n = len(F_list)
    X = torch.zeros_like(F_list[0]) if dS_T is None else dS_T.to(F_list[0].dtype)
    for j in range(n - 1, rank, -1):
        X = torch.matmul(X, M_list[j].transpose(-1, -2)) + F_list[j]
    return X


def _all_gather(t: torch.Tensor, group) -> List[torch.Tensor]:
    import torch.distributed as dist
    out = [torch.empty_like(t) for _ in range(dist.get_world_size(group))]
    dist.all_gather(out, t.contiguous(), group=group)
    return out


def cp_forward(q, k, v, g, beta, initial_state=None, *, fns: ShardFns, group=None):
    """Forward of this rank's shard [B, T_rank, H, d] of a sequence split across the ranks of
    `group` in rank order.  `initial_state` is the whole sequence's S0 (used by every rank; only
    rank 0's shard starts from it).  Returns (o_shard, S_end_shard, S_start_shard, M_shard)."""
    import torch.distributed as dist
    rank = dist.get_rank(group)
    E, M = shard_summary(fns, q, k, v, g, beta)
    Es, Ms = _all_gather(E, group), _all_gather(M, group)
    S_start = compose_forward(initial_state, list(zip(Es, Ms)), rank)
    o, S_end = fns.fwd(q, k, v, g, beta, S_start)
    return o, S_end, S_start, M


def cp_backward(q, k, v, g, beta, dO, S_start, M, dS_T=None, *, fns: ShardFns, group=None):
    """Backward of this rank's shard, given its exact start state and transition from cp_forward.
    `dS_T` is the gradient of the whole sequence's final state (used by the last rank's shard).
    Returns (dq, dk, dv, dg, dbeta, dS_start): dS_start of rank 0 is the gradient of S0."""
    import torch.distributed as dist
    rank = dist.get_rank(group)
    B, _, H, D = q.shape
    zero = torch.zeros(B, H, v.shape[-1], D, dtype=torch.float32, device=q.device)
    F = fns.bwd(q, k, v, g, beta, dO, S_start, zero)[5]
    Fs, Ms = _all_gather(F, group), _all_gather(M, group)
    dS_end = compose_backward(dS_T, Fs, Ms, rank)
    return fns.bwd(q, k, v, g, beta, dO, S_start, dS_end)
