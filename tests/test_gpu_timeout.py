"""The bounded grid-wide waits of the single-launch decode kernel.  The
barrier-slack test hook makes the kernel expect one arrival more than its
grid has at the wait for every CTA's h, so the wait can never be met: each
CTA must give up after its poll limit and finish the call, the call must
report MOE_ERR_TIMEOUT through moe_layer_check, and the layer's next calls
must be exact again -- no hang, and the CUDA context stays usable.
"""
import time

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import cases
from quantized_moe_expert_sigmoid_gb300 import MoeError, MoeLayer, moe_test_barrier_slack, synth
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T", [1, 5])
def test_h_wait_gives_up_and_the_layer_recovers(T):
    wl = synth.WORKLOADS["decode1"]
    ew = parity.weights(0, 0, wl.E, wl.H, wl.F, 1)
    c = cases.make_case(wl, T=T, ew=ew)
    L = MoeLayer.from_weights(ew, k=wl.k, scale=wl.scale, max_tokens=8)
    x = torch.from_numpy(c.x.view(np.int16)).cuda().view(torch.bfloat16)
    wr = torch.from_numpy(c.wr).cuda()
    good = L.forward_routed(x, wr, out_dtype=torch.float32)[0].clone()
    L.check()

    moe_test_barrier_slack(L.handle, 1)
    t0 = time.monotonic()
    _, ids, _ = L.forward_routed(x, wr, out_dtype=torch.float32)
    with pytest.raises(MoeError) as e:
        L.check()
    assert e.value.name == "MOE_ERR_TIMEOUT"
    assert time.monotonic() - t0 < 60.0
    # the routing ran before the wait that gave up
    np.testing.assert_array_equal(ids.cpu().numpy(), c.ids)

    moe_test_barrier_slack(L.handle, 0)
    for _ in range(2):
        out = L.forward_routed(x, wr, out_dtype=torch.float32)[0]
        L.check()
        assert torch.equal(out, good)
    L.close()
