"""Expert-parallel sharding of the routed layer: the dispatch and combine plans.

This is the host-side index logic of expert parallelism for a box with
several GPUs -- each rank holds E/N routed experts (contiguous blocks of
expert ids) and a replica of the shared expert and the router, and serves
its own tokens.  Every box this library runs on has one GPU, so no GPU step
uses it; it is the plan that a multi-GPU layer call would execute, tested on
CPU ranks.

One step on N ranks (token-parallel over ranks, expert-parallel inside):
  1. route the rank's own tokens (the router is replicated);
  2. dispatch: every route (token t, slot j) goes to the rank that owns
     expert ids[t, j]; the send buffer is ordered by (destination rank,
     expert, token, slot), so each peer receives its routes already grouped
     by expert (the CSR route table of PocketLLM's "Xing4.0-29B-A4B: the
     design record", section 4) and runs them with the batched kernels,
     weight 1, no shared expert;
  3. combine: the expert outputs travel back in the same order, and the
     source rank adds a token's routes in slot order, then its own shared
     expert -- the same order as the single-GPU deterministic combine, so the
     sum does not depend on which rank computed which expert.
The pages rejected tensor parallelism for this model (PocketLLM design
record, section 8 "What was rejected"); experts are whole on one rank here.
"""
from __future__ import annotations

import dataclasses

import numpy as np


def expert_owner(E: int, n_ranks: int) -> np.ndarray:
    """Rank of each routed expert: contiguous blocks, rank r owns experts
    [r*E/N, (r+1)*E/N) (integer split; E need not be a multiple of N)."""
    if not (1 <= n_ranks <= E):
        raise ValueError(f"need 1 <= n_ranks <= E (got {n_ranks}, {E})")
    e = np.arange(E, dtype=np.int64)
    return (e * n_ranks // E).astype(np.int32)


def local_experts(E: int, n_ranks: int, rank: int) -> np.ndarray:
    """Global ids of the experts rank `rank` holds, ascending."""
    return np.nonzero(expert_owner(E, n_ranks) == rank)[0].astype(np.int32)


@dataclasses.dataclass
class DispatchPlan:
    """Routes of one rank's tokens, in send order.

    order[i]       route index t*k + j of the i-th row sent
    dest[i]        rank it goes to
    expert[i]      global expert id of that row
    send_counts[r] rows sent to rank r (rows for rank r are contiguous)
    pos[t, j]      row of route (t, j) in the send (and returned) order
    """
    order: np.ndarray
    dest: np.ndarray
    expert: np.ndarray
    send_counts: np.ndarray
    pos: np.ndarray


def dispatch_plan(ids: np.ndarray, E: int, n_ranks: int) -> DispatchPlan:
    """Order the routes of [T, k] ids by (owner rank, expert, token, slot)."""
    ids = np.asarray(ids, np.int64)
    if ids.ndim != 2:
        raise ValueError("ids must be [T, k]")
    if ids.size and (ids.min() < 0 or ids.max() >= E):
        raise ValueError("expert id outside [0, E)")
    T, k = ids.shape
    owner = expert_owner(E, n_ranks)
    flat = ids.reshape(-1)
    route = np.arange(T * k, dtype=np.int64)
    dest = owner[flat].astype(np.int64)
    # stable lexicographic sort: rank, then expert, then route index (= token, slot)
    order = np.lexsort((route, flat, dest))
    pos = np.empty(T * k, dtype=np.int64)
    pos[order] = np.arange(T * k)
    return DispatchPlan(order=order, dest=dest[order].astype(np.int32), expert=flat[order].astype(np.int32),
                        send_counts=np.bincount(dest, minlength=n_ranks).astype(np.int64),
                        pos=pos.reshape(T, k))


def receive_groups(recv_experts: np.ndarray):
    """The rows a rank received (concatenated over source ranks, each source's
    block already in expert order) as (expert, row indices) groups, experts
    ascending -- the input of the rank's local expert kernels."""
    recv_experts = np.asarray(recv_experts, np.int64)
    rows = np.argsort(recv_experts, kind="stable")
    groups = []
    for e in np.unique(recv_experts):
        groups.append((int(e), rows[recv_experts[rows] == e]))
    return groups


def combine(y_back: np.ndarray, plan: DispatchPlan, weights: np.ndarray,
            shared: np.ndarray | None) -> np.ndarray:
    """out[t] = sum over slots j, in slot order, of weights[t, j] *
    y_back[pos[t, j]], then + shared[t].  y_back: the expert outputs of this
    rank's routes, returned in send order."""
    w = np.asarray(weights, np.float64)
    T, k = w.shape
    out = np.zeros((T, y_back.shape[1]), dtype=np.float64)
    for j in range(k):
        out += w[:, j:j + 1] * y_back[plan.pos[:, j]]
    if shared is not None:
        out += shared
    return out
