"""moe_layer_forward_routed_host: x and out in pinned host memory, the copies
enqueued with the layer call.  Its output must equal the device-memory call's
bit for bit (the same kernels run on the same values), for the one-token
and batch kernels (x imported inside the kernel, out through the host
mapping) and the multi-launch path (both copied), bf16 and fp32 out."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import cases
from quantized_moe_expert_sigmoid_gb300 import (MOE_FLAG_DETERMINISTIC, MOE_FLAG_HOST_IO, MoeError, MoeLayer,
                                                moe_layer_forward_routed, moe_layer_forward_routed_host, synth)
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T", [1, 5, 16, 64])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_host_call_equals_device_call(T, out_dtype):
    wl = synth.WORKLOADS["decode1"]
    ew = parity.weights(0, 0, wl.E, wl.H, wl.F, 1)
    c = cases.make_case(wl, T=T, ew=ew)
    L = MoeLayer.from_weights(ew, k=wl.k, scale=wl.scale, max_tokens=64,
                              flags=MOE_FLAG_HOST_IO | MOE_FLAG_DETERMINISTIC)
    xh = torch.from_numpy(c.x.view(np.int16)).view(torch.bfloat16).pin_memory()
    xd = xh.cuda()
    wr = torch.from_numpy(c.wr).cuda()
    ids = torch.empty((T, wl.k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, wl.k), dtype=torch.float32, device="cuda")
    out_d = torch.empty((T, wl.H), dtype=out_dtype, device="cuda")
    moe_layer_forward_routed(L.handle, xd, wr, ids, w, out_d)
    ref = out_d.cpu()
    out_h = torch.empty((T, wl.H), dtype=out_dtype).pin_memory()
    for _ in range(2):
        out_h.zero_()
        moe_layer_forward_routed_host(L.handle, xh, wr, ids, w, out_h)
        torch.cuda.current_stream().synchronize()
        assert torch.equal(out_h, ref)
    np.testing.assert_array_equal(ids.cpu().numpy(), c.ids)
    L.check()
    L.close()


def test_host_call_needs_the_flag():
    wl = synth.WORKLOADS["decode1"]
    ew = parity.weights(0, 0, wl.E, wl.H, wl.F, 1)
    L = MoeLayer.from_weights(ew, k=wl.k, scale=wl.scale, max_tokens=1)
    xh = torch.zeros((1, wl.H), dtype=torch.bfloat16).pin_memory()
    out_h = torch.empty((1, wl.H), dtype=torch.bfloat16).pin_memory()
    wr = torch.zeros((wl.E, wl.H), dtype=torch.float32, device="cuda")
    ids = torch.empty((1, wl.k), dtype=torch.int32, device="cuda")
    w = torch.empty((1, wl.k), dtype=torch.float32, device="cuda")
    with pytest.raises(MoeError) as e:
        moe_layer_forward_routed_host(L.handle, xh, wr, ids, w, out_h)
    assert e.value.name == "MOE_ERR_INVALID_ARG"
    L.close()


def test_one_token_host_and_device_calls_interleaved():
    """At one token the host-buffer call brings x to the device inside the
    kernel, each CTA its share, behind an arrival counter whose target
    follows the layer's call count; calls without that step (device x, a
    4-token batch on another kernel) in any order between them must keep
    the count right: every host call gives the device call's bits."""
    wl = synth.WORKLOADS["decode1"]
    ew = parity.weights(0, 0, wl.E, wl.H, wl.F, 1)
    c = cases.make_case(wl, T=4, ew=ew, seed=31)
    L = MoeLayer.from_weights(ew, k=wl.k, scale=wl.scale, max_tokens=16, flags=MOE_FLAG_HOST_IO)
    x4 = torch.from_numpy(c.x.view(np.int16)).view(torch.bfloat16)
    wr = torch.from_numpy(c.wr).cuda()
    ids = torch.empty((4, wl.k), dtype=torch.int32, device="cuda")
    w = torch.empty((4, wl.k), dtype=torch.float32, device="cuda")
    refs = []
    for t in range(4):
        o = torch.empty((1, wl.H), dtype=torch.float32, device="cuda")
        moe_layer_forward_routed(L.handle, x4[t:t + 1].cuda(), wr, ids[:1], w[:1], o)
        refs.append(o.cpu())
    out4 = torch.empty((4, wl.H), dtype=torch.float32, device="cuda")
    xh = [x4[t:t + 1].clone().pin_memory() for t in range(4)]
    oh = torch.empty((1, wl.H), dtype=torch.float32).pin_memory()
    for step, t in enumerate([0, 1, 1, 2, 3, 0, 2]):
        if step % 3 == 1:
            moe_layer_forward_routed(L.handle, x4.cuda(), wr, ids, w, out4)
        if step % 2 == 0:
            o = torch.empty((1, wl.H), dtype=torch.float32, device="cuda")
            moe_layer_forward_routed(L.handle, xh[t].cuda(), wr, ids[:1], w[:1], o)
            assert torch.equal(o.cpu(), refs[t])
        oh.zero_()
        moe_layer_forward_routed_host(L.handle, xh[t], wr, ids[:1], w[:1], oh)
        torch.cuda.current_stream().synchronize()
        assert torch.equal(oh, refs[t]), f"step {step}, token {t}"
    L.check()
    parity.assert_close_fp32(refs[0].numpy(), parity.oracle_forward(c.x64[:1], c.ids[:1], c.w[:1], ew), "token 0")
    L.close()


def test_batch_host_calls_with_changing_x():
    """The batch kernel takes bf16 x from host memory the same way (each CTA
    copies its share into the layer's device buffer, one arrival counter,
    then one bulk copy of x into shared memory).  x changes on every call,
    with one-token host calls and device calls between, so a stale or
    partly written import would show: every host call gives the device
    call's bits for its own x."""
    wl = synth.WORKLOADS["decode1"]
    ew = parity.weights(0, 0, wl.E, wl.H, wl.F, 1)
    c = cases.make_case(wl, T=12, ew=ew, seed=33)
    L = MoeLayer.from_weights(ew, k=wl.k, scale=wl.scale, max_tokens=16, flags=MOE_FLAG_HOST_IO)
    x = torch.from_numpy(c.x.view(np.int16)).view(torch.bfloat16)
    wr = torch.from_numpy(c.wr).cuda()
    batches = [(0, 4), (4, 8), (0, 12), (3, 5), (5, 6)]  # the last one is a single token
    ids = torch.empty((12, wl.k), dtype=torch.int32, device="cuda")
    w = torch.empty((12, wl.k), dtype=torch.float32, device="cuda")
    refs = []
    for a, b in batches:
        o = torch.empty((b - a, wl.H), dtype=torch.bfloat16, device="cuda")
        moe_layer_forward_routed(L.handle, x[a:b].cuda(), wr, ids[:b - a], w[:b - a], o)
        refs.append(o.cpu())
    xh = [x[a:b].clone().pin_memory() for a, b in batches]
    for step, i in enumerate([0, 1, 2, 0, 4, 1, 3, 2, 4, 3, 0]):
        a, b = batches[i]
        if step % 4 == 3:
            o = torch.empty((b - a, wl.H), dtype=torch.bfloat16, device="cuda")
            moe_layer_forward_routed(L.handle, xh[i].cuda(), wr, ids[:b - a], w[:b - a], o)
        oh = torch.zeros((b - a, wl.H), dtype=torch.bfloat16).pin_memory()
        moe_layer_forward_routed_host(L.handle, xh[i], wr, ids[:b - a], w[:b - a], oh)
        torch.cuda.current_stream().synchronize()
        assert torch.equal(oh, refs[i]), f"step {step}, tokens {a}..{b}"
    L.check()
    ref = parity.oracle_forward(c.x64, c.ids, c.w, ew)
    parity.assert_close_bf16(refs[2].float().numpy(), ref, "12 tokens")
    L.close()
