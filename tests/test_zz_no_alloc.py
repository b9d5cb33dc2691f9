"""moe_route_noalloc: the router for callers that cannot allocate device memory.

Some callers may not call cudaMalloc (their host framework owns every device
allocation, or the serving step must not allocate once it runs).  This entry
point takes no layer and allocates nothing: its logits scratch is a fixed
array inside the library.  It must give what moe_route gives, call after
call, since every call reuses that one array.

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import quantized_moe_expert_sigmoid_gb300 as moe
from oracle import cases
from quantized_moe_expert_sigmoid_gb300 import MoeError, MoeLayer, synth

pytestmark = pytest.mark.gpu


def _inputs(c):
    x = torch.from_numpy(c.x.view(np.int16)).cuda().view(torch.bfloat16) \
        if c.wl.x_dtype == "bf16" else torch.from_numpy(c.x).cuda()
    wr = torch.from_numpy(c.wr).cuda()
    bias = None if c.bias is None else torch.from_numpy(c.bias).cuda()
    return x, wr, bias


def _both(layer, c):
    x, wr, bias = _inputs(c)
    T, k = x.shape[0], c.wl.k
    ids_a = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w_a = torch.empty((T, k), dtype=torch.float32, device="cuda")
    moe.moe_route(layer.handle, x, wr, ids_a, w_a, bias)
    ids_b = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    w_b = torch.full((T, k), -7.0, dtype=torch.float32, device="cuda")
    moe.moe_route_noalloc(x, wr, ids_b, w_b, k, c.wl.scale, bias)
    torch.cuda.synchronize()
    return ids_a.cpu().numpy(), w_a.cpu().numpy(), ids_b.cpu().numpy(), w_b.cpu().numpy()


def test_noalloc_router_matches_moe_route_on_consecutive_calls():
    tiny = synth.WORKLOADS["tiny"]
    ew = synth.expert_weights(0, 0, tiny.E, tiny.H, tiny.F)
    layer = MoeLayer.from_weights(ew, k=tiny.k, scale=tiny.scale, max_tokens=64)
    wl = synth.Workload("router-only: H 3584, 64 experts top-4, 64 tokens", 3584, 64, 4, 32, 64,
                        "bf16", 0.02)
    big = MoeLayer.from_weights(synth.expert_weights(0, 0, 64, 3584, 32), k=4, scale=2.0,
                                max_tokens=64)
    # two calls in a row with different inputs (and the second one larger)
    for lay, c in ((layer, cases.make_case(tiny, ew=ew)),
                   (big, cases.make_case(wl, ew=synth.expert_weights(0, 0, 64, 3584, 32)))):
        ids_a, w_a, ids_b, w_b = _both(lay, c)
        np.testing.assert_array_equal(ids_b, ids_a)
        np.testing.assert_allclose(w_b, w_a, rtol=0, atol=2e-6)
        np.testing.assert_array_equal(ids_b, c.ids)
    layer.close()
    big.close()


def test_noalloc_router_rejects_more_than_its_scratch():
    x = torch.zeros((4097, 64), dtype=torch.float32, device="cuda")
    wr = torch.zeros((64, 64), dtype=torch.float32, device="cuda")
    ids = torch.empty((4097, 2), dtype=torch.int32, device="cuda")
    w = torch.empty((4097, 2), dtype=torch.float32, device="cuda")
    with pytest.raises(MoeError) as e:
        moe.moe_route_noalloc(x, wr, ids, w, 2)
    assert e.value.name == "MOE_ERR_UNSUPPORTED_SHAPE"
    assert "scratch" in str(e.value)


@pytest.mark.parametrize("T", [256, 4096])
def test_noalloc_router_large_bf16_batches(T):
    """At 256 and more bf16 tokens moe_route runs the tensor-core router and
    moe_route_noalloc the CUDA-core one: both must give the oracle's ids on
    gap-resampled inputs, and weights within the router tolerance of each
    other.  T = 4,096 with 64 experts fills the scratch exactly."""
    wl = synth.Workload(f"router-only: H 3584, 64 experts top-4, {T} tokens", 3584, 64, 4, 32, T,
                        "bf16", 0.02)
    ew = synth.expert_weights(0, 0, 64, 3584, 32)
    layer = MoeLayer.from_weights(ew, k=4, scale=2.0, max_tokens=T)
    c = cases.make_case(wl, ew=ew)
    for _ in range(2):  # two calls in a row through the shared scratch
        ids_a, w_a, ids_b, w_b = _both(layer, c)
        np.testing.assert_array_equal(ids_a, c.ids)
        np.testing.assert_array_equal(ids_b, c.ids)
        np.testing.assert_allclose(w_b, w_a, rtol=0, atol=2e-6)
        np.testing.assert_allclose(w_b, c.w, rtol=0, atol=2e-6)
    layer.close()
