"""GPU parity of the single-launch batch kernel (2..16 tokens in one launch
per layer call): the Xing4 layer on both sides of the point where x no
longer fits shared memory whole (up to 9 tokens one pass over the hidden
dimension, above that two), the K2-Horizon shape, caller-given routes with
an invalid id, a repeated id and every token on the same expert, a
per-token logit bias, and bit-reproducibility -- each against the fp64
oracle (routing ids bit for bit, outputs within tests/parity.py).
"""
import functools

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from oracle import cases
from quantized_moe_expert_sigmoid_gb300 import MoeError, MoeLayer, moe_launch_count, synth
from tests import parity

pytestmark = pytest.mark.gpu


@functools.lru_cache(maxsize=None)
def _layer(name):
    wl = synth.WORKLOADS[name]
    ew = parity.weights(0, 0, wl.E, wl.H, wl.F, 1)
    return wl, ew, MoeLayer.from_weights(ew, k=wl.k, scale=wl.scale, max_tokens=16)


def _inputs(c):
    x = torch.from_numpy(c.x.view(np.int16)).cuda().view(torch.bfloat16)
    return x, torch.from_numpy(c.wr).cuda()


@pytest.mark.parametrize("name,T", [("decode1", 2), ("decode1", 5), ("decode1", 9), ("decode1", 10),
                                    ("decode1", 16), ("k2h_decode1", 3), ("k2h_decode1", 16)])
def test_routed_batch_matches_oracle(name, T):
    """Route + layer in one launch: ids bit for bit, weights within 2e-6,
    fp32 output within tolerance on every token; the bf16 output is the
    fp32 one rounded once."""
    wl, ew, L = _layer(name)
    c = cases.make_case(wl, T=T, ew=ew, seed=5)
    x, wr = _inputs(c)
    before = moe_launch_count()
    out, ids, w = L.forward_routed(x, wr, out_dtype=torch.float32)
    assert moe_launch_count() - before == 1
    L.check()
    np.testing.assert_array_equal(ids.cpu().numpy(), c.ids)
    np.testing.assert_allclose(w.cpu().numpy(), c.w, rtol=0, atol=2e-6)
    ref = parity.oracle_forward(c.x64, c.ids, c.w, ew)
    parity.assert_close_fp32(out.cpu().numpy(), ref, f"{name} T={T}")
    out_b, _, _ = L.forward_routed(x, wr)
    L.check()
    parity.assert_close_bf16(out_b.float().cpu().numpy(), ref, f"{name} T={T} bf16")
    np.testing.assert_array_equal(out_b.float().cpu().numpy(),
                                  out.to(torch.bfloat16).float().cpu().numpy())


@pytest.mark.parametrize("T", [6, 12])
def test_given_routes_bad_repeated_and_shared_ids(T):
    """Token 0 names an expert outside [0, E) (dropped and reported) and one
    expert twice; tokens 1.. all put slot 0 on the same expert, so one
    expert carries every token of the batch."""
    wl, ew, L = _layer("decode1")
    c = cases.make_case(wl, T=T, ew=ew, seed=6)
    x, _ = _inputs(c)
    ids = c.ids.copy()
    ids[0, 1] = wl.E + 3
    ids[0, 2] = ids[0, 0]
    hot = int(ids[1, 0])
    for t in range(1, T):
        if hot not in ids[t, 1:]:
            ids[t, 0] = hot
    w = (np.linspace(0.2, 0.9, T * wl.k, dtype=np.float32).reshape(T, wl.k))
    out = L.forward(x, torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(), out_dtype=torch.float32)
    with pytest.raises(MoeError) as e:
        L.check()
    assert e.value.name == "MOE_ERR_BAD_EXPERT_ID"
    L.check()
    keep_ids, keep_w = ids.copy(), w.astype(np.float64)
    keep_ids[0, 1], keep_w[0, 1] = 0, 0.0
    ref = parity.oracle_forward(c.x64, keep_ids, keep_w, ew)
    parity.assert_close_fp32(out.cpu().numpy(), ref, f"given routes T={T}")


def test_every_slot_on_two_experts():
    """16 tokens whose four slots name only experts 5 and 9 (twice each):
    two plan entries of 32 routes each."""
    wl, ew, L = _layer("decode1")
    c = cases.make_case(wl, T=16, ew=ew, seed=7)
    x, _ = _inputs(c)
    ids = np.tile(np.array([5, 9, 5, 9], np.int32), (16, 1))
    w = np.tile(np.array([0.5, 0.25, 0.125, 1.0], np.float32), (16, 1))
    out = L.forward(x, torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(), out_dtype=torch.float32)
    L.check()
    ref = parity.oracle_forward(c.x64, ids, w.astype(np.float64), ew)
    parity.assert_close_fp32(out.cpu().numpy(), ref, "two experts")


def test_per_token_logit_bias():
    """A [T, E] logit bias (added before the sigmoid) that lifts each
    token's best unselected expert by 4 (into its top-k)."""
    wl, ew, L = _layer("decode1")
    T = 7
    c = cases.make_case(wl, T=T, ew=ew, seed=8)
    x, wr = _inputs(c)
    bias = np.zeros((T, wl.E), np.float32)
    for t in range(T):
        bias[t, np.argsort(-c.logits[t], kind="stable")[wl.k]] = 4.0
    out, ids, w = L.forward_routed(x, wr, torch.from_numpy(bias).cuda(), out_dtype=torch.float32)
    L.check()
    ref_ids, ref_w, logits = oracle.route(c.x64, c.wr, wl.k, wl.scale, bias)
    clear = oracle.min_topk_gap(logits, wl.k) >= 1e-4  # (the bias may bring two scores close)
    assert clear.sum() >= T - 1
    ids_g, w_g = ids.cpu().numpy(), w.cpu().numpy()
    np.testing.assert_array_equal(ids_g[clear], ref_ids[clear])
    np.testing.assert_allclose(w_g[clear], ref_w[clear], rtol=0, atol=2e-6)
    assert sum(int(bias[t, ids_g[t]].max() > 0) for t in range(T)) >= T - 1  # the lifted expert is taken
    ref = parity.oracle_forward(c.x64, ids_g, w_g.astype(np.float64), ew)
    parity.assert_close_fp32(out.cpu().numpy(), ref, "per-token bias")


def test_batch_is_bit_reproducible():
    """Repeated calls (alternating counter sets) give the same bits."""
    wl, ew, L = _layer("decode1")
    c = cases.make_case(wl, T=11, ew=ew, seed=9)
    x, wr = _inputs(c)
    outs = []
    for _ in range(3):
        o, _, _ = L.forward_routed(x, wr, out_dtype=torch.float32)
        outs.append(o.clone())
    L.check()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])


@pytest.mark.parametrize("T", [4, 13])
def test_fp32_activations_and_a_shared_bias_row(T):
    """fp32 x (bf16 values exactly, so routing is unchanged) takes the
    kernel's path that reads x from global memory; a single [E] logit bias
    row applies to every token; the bf16 output is the fp32 one rounded once."""
    wl, ew, L = _layer("decode1")
    c = cases.make_case(wl, T=T, ew=ew, seed=10)
    x32 = torch.from_numpy(synth.bf16_bits_to_f32(c.x).reshape(T, wl.H)).cuda()
    wr = torch.from_numpy(c.wr).cuda()
    row = np.zeros(wl.E, np.float32)
    row[int(np.argsort(-c.logits[0], kind="stable")[wl.k])] = 3.0  # token 0's best unselected expert
    out, ids, w = L.forward_routed(x32, wr, torch.from_numpy(row).cuda(), out_dtype=torch.float32)
    L.check()
    ref_ids, ref_w, logits = oracle.route(c.x64, c.wr, wl.k, wl.scale, row)
    clear = oracle.min_topk_gap(logits, wl.k) >= 1e-4
    assert clear.sum() >= T - 1
    ids_g, w_g = ids.cpu().numpy(), w.cpu().numpy()
    np.testing.assert_array_equal(ids_g[clear], ref_ids[clear])
    np.testing.assert_allclose(w_g[clear], ref_w[clear], rtol=0, atol=2e-6)
    ref = parity.oracle_forward(c.x64, ids_g, w_g.astype(np.float64), ew)
    parity.assert_close_fp32(out.cpu().numpy(), ref, f"fp32 x T={T}")
    out_b, _, _ = L.forward_routed(x32, wr, torch.from_numpy(row).cuda(), out_dtype=torch.bfloat16)
    L.check()
    np.testing.assert_array_equal(out_b.float().cpu().numpy(), out.to(torch.bfloat16).float().cpu().numpy())


@pytest.mark.parametrize("H,E,k,F,T,S", [(3488, 40, 3, 992, 6, 1), (2528, 100, 8, 736, 11, 0)])
def test_ragged_shapes_on_the_batch_kernel(H, E, k, F, T, S):
    """H and F that are not multiples of 256 (x copied row by row, the pad
    columns read as zero; padded outputs with zero weights), an odd expert
    count, k = 3 and k = 8, with and without the shared expert: one launch,
    ids bit for bit, output within tolerance."""
    wl = synth.Workload("ragged batch", H, E, k, F, T, "bf16", 1.2 / H ** 0.5, n_shared=S)
    ew = synth.expert_weights(13, 0, E, H, F, S)
    if not S:
        ew.sh_up = ew.sh_gate = ew.sh_down = None
    c = cases.make_case(wl, seed=13, ew=ew)
    L = MoeLayer.from_weights(ew, k=k, scale=2.0, max_tokens=16)
    x, wr = _inputs(c)
    before = moe_launch_count()
    out, ids, w = L.forward_routed(x, wr, out_dtype=torch.float32)
    assert moe_launch_count() - before == 1
    L.check()
    np.testing.assert_array_equal(ids.cpu().numpy(), c.ids)
    ref = parity.oracle_forward(c.x64, c.ids, c.w, ew)
    parity.assert_close_fp32(out.cpu().numpy(), ref, f"H{H} E{E} k{k} F{F} T{T}")
    L.close()
