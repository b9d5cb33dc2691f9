"""Expert-parallel dispatch and combine on two CPU ranks (gloo), against the
oracle's single-process layer.

Each rank routes its own tokens with the replicated router, sends every route
to the rank that owns its expert (contiguous blocks of expert ids), runs only
its own experts on what it received, sends the outputs back, and adds a
token's routes in slot order plus its own replica of the shared expert.  The
result must equal the oracle's layer on the same tokens to fp64 rounding,
whichever rank held which expert.  The expert FFNs here are the oracle's
(CPU); the plan and the exchange are the library's host index logic.
"""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from quantized_moe_expert_sigmoid_gb300 import ep, synth

E, H, F, K, T = 8, 64, 32, 2, 5


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class _One:
    """One expert's matrices as a one-expert layer without a shared expert."""

    def __init__(self, up, gate, down):
        self.up, self.gate, self.down = up[None], gate[None], down[None]
        self.sh_up = self.sh_gate = self.sh_down = None


def _layer():
    ew = synth.expert_weights(21, 0, E, H, F)
    wr = synth.router_weights(21, 0, E, H, 0.2)
    return ew, wr


def _tokens(rank):
    return oracle.to_f64(synth.activations(21, "ep", T, H, np.full(T, rank), "fp32"), "fp32")


def _exchange(rows: np.ndarray, send_counts, recv_counts):
    """all_to_all of float64 rows (and a matching int64 vector when rows is 1-D)."""
    t = torch.from_numpy(np.ascontiguousarray(rows))
    out = torch.empty((int(sum(recv_counts)),) + tuple(t.shape[1:]), dtype=t.dtype)
    dist.all_to_all_single(out, t, [int(c) for c in recv_counts], [int(c) for c in send_counts])
    return out.numpy()


def _rank_step(rank, world, force_ids, result):
    oracle.build()
    ew, wr = _layer()
    x = _tokens(rank)
    ids, w, _ = oracle.route(x, wr, K, 2.0)
    if force_ids is not None:
        ids = np.asarray(force_ids[rank], np.int32)
    plan = ep.dispatch_plan(ids, E, world)
    send_counts = plan.send_counts
    recv_counts = _exchange(send_counts.astype(np.int64), np.ones(world), np.ones(world))
    x_send = x[plan.order // K]
    x_recv = _exchange(x_send, send_counts, recv_counts)
    e_recv = _exchange(plan.expert.astype(np.int64), send_counts, recv_counts)
    mine = set(ep.local_experts(E, world, rank).tolist())
    assert set(e_recv.tolist()) <= mine, "a route reached a rank that does not hold its expert"
    y = np.zeros_like(x_recv)
    for e, rows in ep.receive_groups(e_recv):
        y[rows] = oracle.dense_ffn(x_recv[rows], _One(ew.up[e], ew.gate[e], ew.down[e]))
    y_back = _exchange(y, recv_counts, send_counts)
    shared = oracle.dense_ffn(x, _One(ew.sh_up, ew.sh_gate, ew.sh_down))
    out = ep.combine(y_back, plan, w, shared)
    ref = oracle.moe_forward(x, ids, w, ew)
    err = np.abs(out - ref).max() / np.abs(ref).max()
    result[rank] = (err, int(recv_counts.sum()))


def _worker(rank, world, port, force_ids, result):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        _rank_step(rank, world, force_ids, result)
    finally:
        dist.destroy_process_group()


def _run(force_ids=None, world=2):
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        result = m.dict()
        mp.start_processes(_worker, args=(world, _free_port(), force_ids, result), nprocs=world,
                           start_method="spawn")
        return dict(result)


def test_two_rank_dispatch_and_combine_equal_the_oracle():
    res = _run()
    assert sorted(res) == [0, 1]
    for rank, (err, n_recv) in res.items():
        assert err <= 1e-12, f"rank {rank}: relative error {err:.3e}"


def test_rank_that_receives_nothing():
    # every route of both ranks on experts 0..3, which rank 0 holds
    force = [[[0, 1], [2, 3], [1, 0], [3, 2], [0, 3]], [[1, 2], [0, 1], [3, 0], [2, 1], [0, 2]]]
    res = _run(force)
    assert res[1][1] == 0 and res[0][1] == 2 * T * K
    for rank, (err, _) in res.items():
        assert err <= 1e-12, f"rank {rank}: relative error {err:.3e}"


def test_dispatch_plan_orders_routes_by_rank_then_expert():
    ids = np.array([[7, 0], [3, 4], [0, 7], [5, 2]], np.int32)
    plan = ep.dispatch_plan(ids, 8, 2)
    assert plan.send_counts.tolist() == [4, 4]
    assert plan.expert.tolist() == [0, 0, 2, 3, 4, 5, 7, 7]
    assert plan.dest.tolist() == [0, 0, 0, 0, 1, 1, 1, 1]
    # equal experts keep token order; pos inverts order
    assert plan.order[:2].tolist() == [1, 4]
    for t in range(4):
        for j in range(2):
            assert plan.order[plan.pos[t, j]] == t * 2 + j
    assert ep.expert_owner(100, 8).tolist().count(0) == 13  # 100 experts over 8 ranks: 12 or 13 each
    with pytest.raises(ValueError):
        ep.dispatch_plan(np.array([[8, 0]]), 8, 2)
