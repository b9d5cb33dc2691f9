"""GPU parity of the one-token decode kernel (one launch per layer call at
T = 1 on the Xing4 and K2-Horizon hidden sizes) on the paths the workload
tests do not reach: caller-given routes with an invalid id and with one
expert named in two slots, a plain logit bias (added before the sigmoid),
and fp32 activations with a bf16 output -- each against the fp64 oracle.
"""
import functools

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from oracle import cases
from quantized_moe_expert_sigmoid_gb300 import MOE_FLAG_COOPERATIVE, MoeError, MoeLayer, moe_launch_count, synth
from tests import parity

pytestmark = pytest.mark.gpu


@functools.lru_cache(maxsize=None)
def _setup(name):
    wl = synth.WORKLOADS[name]
    ew = parity.weights(0, 0, wl.E, wl.H, wl.F, 1)
    L = MoeLayer.from_weights(ew, k=wl.k, scale=wl.scale, max_tokens=8)
    c = cases.make_case(wl, T=1, ew=ew, seed=3)
    x = torch.from_numpy(c.x.view(np.int16)).cuda().view(torch.bfloat16)
    wr = torch.from_numpy(c.wr).cuda()
    return wl, ew, L, c, x, wr


@pytest.mark.parametrize("name", ["decode1", "k2h_decode1"])
def test_given_routes_with_a_bad_and_a_repeated_id(name):
    """Slot 1 names an expert outside [0, E): that route is dropped and
    reported; slot 2 repeats slot 0's expert with another weight, so the
    expert's output counts twice (w0 + w2)."""
    wl, ew, L, c, x, wr = _setup(name)
    ids = c.ids.copy()
    ids[0, 1] = wl.E
    ids[0, 2] = ids[0, 0]
    w = np.linspace(0.3, 0.9, wl.k, dtype=np.float32)[None, :]
    before = moe_launch_count()
    out = L.forward(x, torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(), out_dtype=torch.float32)
    assert moe_launch_count() - before == 1  # the whole layer in one launch
    with pytest.raises(MoeError) as e:
        L.check()
    assert e.value.name == "MOE_ERR_BAD_EXPERT_ID"
    L.check()
    keep_ids, keep_w = ids.copy(), w.astype(np.float64)
    keep_ids[0, 1], keep_w[0, 1] = 0, 0.0
    ref = oracle.moe_forward(c.x64, keep_ids, keep_w, ew)
    parity.assert_close_fp32(out.cpu().numpy(), ref, f"{name} bad and repeated ids")


@pytest.mark.parametrize("name", ["decode1", "k2h_decode1"])
def test_logit_bias_moves_the_selection(name):
    """A [E] logit bias (added before the sigmoid, so it moves both the
    selection and the weights) on one expert that the plain router did not
    pick: ids must follow the oracle's biased routing."""
    wl, ew, L, c, x, wr = _setup(name)
    row = np.zeros(wl.E, np.float32)
    outside = [e for e in range(wl.E) if e not in set(c.ids[0].tolist())]
    row[outside[0]] = 4.0
    out, ids, w = L.forward_routed(x, wr, torch.from_numpy(row).cuda(), out_dtype=torch.float32)
    L.check()
    ref_ids, ref_w, logits = oracle.route(c.x64, c.wr, wl.k, wl.scale, row)
    assert oracle.min_topk_gap(logits, wl.k)[0] >= 1e-4
    assert outside[0] in ref_ids[0]
    np.testing.assert_array_equal(ids.cpu().numpy(), ref_ids)
    np.testing.assert_allclose(w.cpu().numpy(), ref_w, rtol=0, atol=2e-6)
    ref = oracle.moe_forward(c.x64, ref_ids, ref_w, ew)
    parity.assert_close_fp32(out.cpu().numpy(), ref, f"{name} logit bias")


def test_fp32_activations_and_bf16_output():
    """The same token as fp32 (bf16 values exactly) routes identically; the
    bf16 output is the fp32 result rounded once."""
    wl, ew, L, c, x, wr = _setup("decode1")
    x32 = torch.from_numpy(synth.bf16_bits_to_f32(c.x).reshape(1, wl.H)).cuda()
    out, ids, w = L.forward_routed(x32, wr, out_dtype=torch.bfloat16)
    L.check()
    np.testing.assert_array_equal(ids.cpu().numpy(), c.ids)
    np.testing.assert_allclose(w.cpu().numpy(), c.w, rtol=0, atol=2e-6)
    ref = oracle.moe_forward(c.x64, c.ids, c.w, ew)
    parity.assert_close_bf16(out.float().cpu().numpy(), ref, "fp32 x, bf16 out")


@pytest.mark.parametrize("name", ["decode1", "k2h_decode1"])
@pytest.mark.parametrize("delta_kind", ["none", "bf16", "fp32"])
def test_residual_step_in_the_one_token_launch(name, delta_kind):
    """moe_layer_forward_routed_resid at one token forms the residual update
    and the RMSNorm inside the one-token kernel's single launch.  Its r_out,
    u, ids, weights and output must equal, bit for bit, the same step taken
    as a residual-RMSNorm launch followed by moe_layer_forward_routed; and u
    must be the bf16 RMSNorm of r_in + delta within one bf16 ulp of the
    fp64 oracle."""
    from quantized_moe_expert_sigmoid_gb300 import (moe_layer_forward_routed, moe_layer_forward_routed_resid,
                                                    moe_residual_rmsnorm)
    wl, ew, L, c, x, wr = _setup(name)
    g = torch.Generator().manual_seed(11)
    r_in = (torch.randn(1, wl.H, generator=g) * 0.7).cuda()
    delta = None
    if delta_kind != "none":
        d = torch.randn(1, wl.H, generator=g) * 0.3
        delta = (d.to(torch.bfloat16) if delta_kind == "bf16" else d).cuda()
    eps = 1e-6

    def bufs():
        return (torch.full((1, wl.H), float("nan"), device="cuda"),
                torch.zeros(1, wl.H, dtype=torch.bfloat16, device="cuda"),
                torch.full((1, wl.k), -7, dtype=torch.int32, device="cuda"),
                torch.zeros(1, wl.k, device="cuda"), torch.zeros(1, wl.H, device="cuda"))

    r1, u1, i1, w1, o1 = bufs()
    before = moe_launch_count()
    moe_layer_forward_routed_resid(L.handle, r_in, delta, r1, u1, eps, wr, i1, w1, o1)
    assert moe_launch_count() - before == 1  # residual, RMSNorm and the layer in one launch
    L.check()
    r2, u2, i2, w2, o2 = bufs()
    r2.copy_(r_in)
    moe_residual_rmsnorm(r2, delta, u2, eps)
    moe_layer_forward_routed(L.handle, u2, wr, i2, w2, o2)
    L.check()
    for a, b, what in ((r1, r2, "r_out"), (u1.view(torch.int16), u2.view(torch.int16), "u"), (i1, i2, "ids"),
                       (w1, w2, "weights"), (o1, o2, "out")):
        assert torch.equal(a, b), f"{name} delta {delta_kind}: {what} differs from the two-launch step"
    r_ref = r_in.cpu().numpy().astype(np.float32)
    if delta is not None:
        r_ref = (r_ref + delta.float().cpu().numpy()).astype(np.float32)
    np.testing.assert_array_equal(r1.cpu().numpy(), r_ref)
    u_ref = synth.to_bf16_bits(np.asarray(oracle.rmsnorm(r_ref.astype(np.float64), eps), np.float32))
    u_bits = u1.cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.abs(u_bits.astype(np.int32) - u_ref.astype(np.int32)).max() <= 1
    # the input buffer is read only
    assert torch.isfinite(r_in).all()


def test_residual_step_rejects_overlap():
    from quantized_moe_expert_sigmoid_gb300 import moe_layer_forward_routed_resid
    wl, ew, L, c, x, wr = _setup("decode1")
    r = torch.zeros(2, wl.H, device="cuda")
    u = torch.zeros(1, wl.H, dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros(1, wl.k, dtype=torch.int32, device="cuda")
    w = torch.zeros(1, wl.k, device="cuda")
    out = torch.zeros(1, wl.H, device="cuda")
    before = moe_launch_count()
    with pytest.raises(MoeError) as e:  # resid_out is resid_in
        moe_layer_forward_routed_resid(L.handle, r[:1], None, r[:1], u, 1e-6, wr, ids, w, out)
    assert e.value.name == "MOE_ERR_INVALID_ARG"
    with pytest.raises(MoeError) as e:  # delta is resid_out
        moe_layer_forward_routed_resid(L.handle, r[:1], r[1:], r[1:], u, 1e-6, wr, ids, w, out)
    assert e.value.name == "MOE_ERR_INVALID_ARG"
    assert moe_launch_count() == before


@pytest.mark.parametrize("name,T", [("decode1", 1), ("decode1", 4), ("tiny", 3)])
def test_cooperative_flag_gives_the_same_bits(name, T):
    """MOE_FLAG_COOPERATIVE changes only how the single-launch kernels are
    launched (the one-token kernel at T = 1, the batch kernel at 4 tokens,
    the multi-token kernel on a small hidden size): one launch each, and the
    same ids, weights and output bits as the layer without it."""
    wl = synth.WORKLOADS[name]
    ew = parity.weights(0, 0, wl.E, wl.H, wl.F, 1)
    c = cases.make_case(wl, T=T, ew=ew, seed=21)
    if wl.x_dtype == "fp32":
        x = torch.from_numpy(c.x).cuda()
    else:
        x = torch.from_numpy(c.x.view(np.int16)).cuda().view(torch.bfloat16)
    wr = torch.from_numpy(c.wr).cuda()
    res = []
    for flags in (0, MOE_FLAG_COOPERATIVE):
        L = MoeLayer.from_weights(ew, k=wl.k, scale=wl.scale, max_tokens=8, flags=flags)
        before = moe_launch_count()
        out, ids, w = L.forward_routed(x, wr, out_dtype=torch.float32)
        assert moe_launch_count() - before == 1
        L.check()
        res.append((out.cpu(), ids.cpu(), w.cpu()))
        L.close()
    for a, b in zip(*res):
        assert torch.equal(a, b)
    np.testing.assert_array_equal(res[0][1].numpy(), c.ids)
    parity.assert_close_fp32(res[0][0].numpy(), parity.oracle_forward(c.x64, c.ids, c.w, ew), f"{name} T={T}")
