"""GPU parity of the other parameterisations of the same sigmoid router and
expert layer (K2-Horizon, as integrated into zLLM: the FFN router picks 8 of
100 routed experts next to one shared expert, normalises the chosen weights
and scales them by 2.5; the value-path router picks 4 of 64 with plain
normalised weights; hidden size 2,560).  The expert width of K2-Horizon is
not given; the workloads take 768.  Ids bit for bit against the fp64
oracle router, outputs within the parity tolerance: decode batch 1 (single
launch), batched decode 64 and a 1,024-token prefill (tensor-core path).
"""
import functools

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from oracle import cases
from quantized_moe_expert_sigmoid_gb300 import MOE_FLAG_DETERMINISTIC, MoeLayer, synth
from tests import parity

pytestmark = pytest.mark.gpu


@functools.lru_cache(maxsize=None)
def _weights():
    wl = synth.WORKLOADS["k2h_decode1"]
    return synth.expert_weights(0, 0, wl.E, wl.H, wl.F, 1)


@functools.lru_cache(maxsize=None)
def _layer(flags=0):
    wl = synth.WORKLOADS["k2h_decode1"]
    return MoeLayer.from_weights(_weights(), k=wl.k, scale=wl.scale, max_tokens=1024, flags=flags)


@functools.lru_cache(maxsize=None)
def _case(name):
    return cases.make_case(synth.WORKLOADS[name], ew=_weights())


def _dev(c):
    x = torch.from_numpy(c.x.view(np.int16)).cuda().view(torch.bfloat16)
    return x, torch.from_numpy(c.wr).cuda()


@pytest.mark.parametrize("name", ["k2h_decode1", "k2h_decode64", "k2h_prefill1024"])
def test_k2_horizon_layer(name):
    c = _case(name)
    T = c.wl.T
    L = _layer()
    x, wr = _dev(c)
    ids, w = L.route(x, wr)
    L.check()
    np.testing.assert_array_equal(ids.cpu().numpy(), c.ids)
    np.testing.assert_allclose(w.cpu().numpy(), c.w, rtol=0, atol=2e-6)
    np.testing.assert_allclose(w.cpu().numpy().sum(1), 2.5, atol=3e-6)
    out, ids2, _ = L.forward_routed(x, wr, out_dtype=torch.float32)
    L.check()
    np.testing.assert_array_equal(ids2.cpu().numpy(), c.ids)
    ref = parity.oracle_forward(c.x64, c.ids, c.w, c.ew, key=(name, "w64"))
    parity.assert_close_fp32(out.cpu().numpy(), ref, name)
    out_b, _, _ = L.forward_routed(x, wr)
    L.check()
    parity.assert_close_bf16(out_b.float().cpu().numpy(), ref, name + " bf16")


def test_k2_horizon_deterministic_prefill():
    c = _case("k2h_prefill1024")
    L = _layer(MOE_FLAG_DETERMINISTIC)
    x, wr = _dev(c)
    a = L.forward_routed(x, wr, out_dtype=torch.float32)[0].cpu().numpy()
    b = L.forward_routed(x, wr, out_dtype=torch.float32)[0].cpu().numpy()
    L.check()
    np.testing.assert_array_equal(a.view(np.int32), b.view(np.int32))
    ref = parity.oracle_forward(c.x64, c.ids, c.w, c.ew, key=("k2h_prefill1024", "w64"))
    parity.assert_close_fp32(a, ref, "k2h prefill deterministic")


@pytest.mark.parametrize("T", [1, 300])
def test_value_path_router_4_of_64(T):
    """The value-path router's parameters (4 of 64, scale 1, H 2,560) through
    moe_route: the single-token GEMV router and the tensor-core router."""
    wl = synth.Workload(f"K2-Horizon value router, {T} tokens", 2560, 64, 4, 256, T, "bf16", 0.024,
                        scale=1.0)
    ew = synth.expert_weights(0, 0, wl.E, wl.H, wl.F, 1)
    c = cases.make_case(wl, ew=ew)
    L = MoeLayer.from_weights(ew, k=wl.k, scale=wl.scale, max_tokens=T)
    x, wr = _dev(c)
    ids, w = L.route(x, wr)
    L.check()
    np.testing.assert_array_equal(ids.cpu().numpy(), c.ids)
    np.testing.assert_allclose(w.cpu().numpy(), c.w, rtol=0, atol=2e-6)
    np.testing.assert_allclose(w.cpu().numpy().sum(1), 1.0, atol=2e-6)
    L.close()
