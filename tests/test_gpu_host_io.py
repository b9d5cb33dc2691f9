"""moe_layer_forward_routed_host: x and out in pinned host memory, the copies
enqueued with the layer call.  Its output must equal the device-memory call's
bit for bit (the same kernels run on the same values), for the one-token
kernel (x and out through the host mapping), the batch kernel (x copied in,
out through the host mapping) and the multi-launch path (both copied), bf16
and fp32 out."""
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
