"""GPU parity of the selection-only score bias (noaux_tc): with
MOE_FLAG_SELECTION_BIAS the layer ranks expert e by sigmoid(l_e) + b_e and
weights the chosen experts by their unbiased scores.  Each router path of
the library is covered against the fp64 oracle router (oracle.route_selbias):
the single-launch decode kernel (T <= 8), the SIMT router (small batches), and
the tensor-core router (>= 256 bf16 tokens), with one [E] bias row for every
token and with a [T, E] bias matrix.  The inputs keep every token's k+1
largest selection keys >= 1e-4 apart, so ids must match bit for bit.
"""
import functools

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from oracle import cases
from quantized_moe_expert_sigmoid_gb300 import MOE_FLAG_SELECTION_BIAS, MoeLayer, synth
from tests import parity

pytestmark = pytest.mark.gpu


@functools.lru_cache(maxsize=None)
def _xing4_layer(flags):
    wl = synth.WORKLOADS["decode1"]
    ew = parity.weights(0, 0, wl.E, wl.H, wl.F, 1)
    return MoeLayer.from_weights(ew, k=wl.k, scale=wl.scale, max_tokens=512, flags=flags)


def _x(c):
    x = torch.from_numpy(c.x.view(np.int16) if c.wl.x_dtype == "bf16" else c.x).cuda()
    return x.view(torch.bfloat16) if c.wl.x_dtype == "bf16" else x


def _check_routes(c, ids, w):
    np.testing.assert_array_equal(ids.cpu().numpy(), c.ids)
    np.testing.assert_allclose(w.cpu().numpy(), c.w, rtol=0, atol=2e-6)


@pytest.mark.parametrize("T,per_token", [(1, False), (1, True), (5, False), (8, True)])
def test_single_launch_decode(T, per_token):
    wl = synth.WORKLOADS["decode1"]
    b = synth.selection_bias(3, wl.E, T if per_token else None)
    c = cases.make_case(wl, T=T, ew=parity.weights(0, 0, wl.E, wl.H, wl.F, 1), selection_bias=b)
    L = _xing4_layer(MOE_FLAG_SELECTION_BIAS)
    x, wr = _x(c), torch.from_numpy(c.wr).cuda()
    out, ids, w = L.forward_routed(x, wr, torch.from_numpy(b).cuda(), out_dtype=torch.float32)
    L.check()
    _check_routes(c, ids, w)
    ref = oracle.moe_forward(c.x64, c.ids, c.w, c.ew)
    parity.assert_close_fp32(out.cpu().numpy(), ref, f"decode T={T}")


@pytest.mark.parametrize("T,per_token", [(16, False), (64, True), (512, True)])
def test_batched_router_and_layer(T, per_token):
    """T = 16 and 64 take the SIMT router, T = 512 the tensor-core router;
    the layer output of every token against the oracle."""
    wl = synth.WORKLOADS["decode1"]
    b = synth.selection_bias(5, wl.E, T if per_token else None)
    c = cases.make_case(wl, T=T, ew=parity.weights(0, 0, wl.E, wl.H, wl.F, 1), selection_bias=b)
    L = _xing4_layer(MOE_FLAG_SELECTION_BIAS)
    x, wr = _x(c), torch.from_numpy(c.wr).cuda()
    bias = torch.from_numpy(b).cuda()
    ids, w = L.route(x, wr, bias)
    L.check()
    _check_routes(c, ids, w)
    out, ids2, w2 = L.forward_routed(x, wr, bias, out_dtype=torch.float32)
    L.check()
    _check_routes(c, ids2, w2)
    ref = parity.oracle_forward(c.x64, c.ids, c.w, c.ew)
    parity.assert_close_fp32(out.cpu().numpy(), ref, f"batched T={T}")


@pytest.mark.parametrize("T", [1, 300])
def test_without_bias_equals_plain_router(T):
    """With the flag and no bias the routes are the plain sigmoid router's."""
    wl = synth.WORKLOADS["decode1"]
    c = cases.make_case(wl, T=T, ew=parity.weights(0, 0, wl.E, wl.H, wl.F, 1))
    x, wr = _x(c), torch.from_numpy(c.wr).cuda()
    ids_s, w_s = _xing4_layer(MOE_FLAG_SELECTION_BIAS).route(x, wr)
    ids_p, w_p = _xing4_layer(0).route(x, wr)
    torch.cuda.synchronize()
    assert torch.equal(ids_s, ids_p) and torch.equal(w_s, w_p)
    _check_routes(c, ids_s, w_s)


def test_small_shape_many_experts():
    """E = 100, top-8 (two logits per lane in the top-k warp, an 8-wide
    selection), fp32 x, per-token bias, through the SIMT and tensor-core
    routers' shapes at H = 288."""
    for T, dt in ((40, "fp32"), (300, "bf16")):
        wl = synth.Workload(f"selection bias: H 288, E 100, top-8, {T} tokens", 288, 100, 8, 64, T, dt, 0.05)
        ew = synth.expert_weights(0, 0, wl.E, wl.H, wl.F)
        b = synth.selection_bias(7, wl.E, T)
        c = cases.make_case(wl, ew=ew, selection_bias=b)
        L = MoeLayer.from_weights(ew, k=wl.k, scale=wl.scale, max_tokens=T, flags=MOE_FLAG_SELECTION_BIAS)
        x, wr = _x(c), torch.from_numpy(c.wr).cuda()
        out, ids, w = L.forward_routed(x, wr, torch.from_numpy(b).cuda(), out_dtype=torch.float32)
        L.check()
        _check_routes(c, ids, w)
        ref = oracle.moe_forward(c.x64, c.ids, c.w, c.ew)
        parity.assert_close_fp32(out.cpu().numpy(), ref, f"E 100 T={T}")
        L.close()
