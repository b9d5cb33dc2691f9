"""GPU parity of the dense FFN blocks (the first two of the Xing4 model's
forty blocks, FFN width 9,216): a one-expert, top-1 layer without a shared
expert, run by moe_dense_forward on the routed layer's kernels, against the
fp64 oracle's dense FFN.  Decode sizes (1 and 3 tokens), a batch of 64 and a
ragged small shape (H and F not multiples of 256)."""
import functools

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from quantized_moe_expert_sigmoid_gb300 import MoeError, MoeLayer, synth
from tests import parity

pytestmark = pytest.mark.gpu


@functools.lru_cache(maxsize=None)
def _dense(H, F, max_tokens):
    ew = synth.dense_ffn_weights(0, 0, H, F)
    return ew, MoeLayer.from_weights(ew, k=1, scale=1.0, max_tokens=max_tokens)


def _x(T, H, seed=0):
    bits = synth.activations(seed, "dense", T, H)
    return bits, torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)


@pytest.mark.parametrize("T", [1, 3, 64])
def test_xing4_dense_block(T):
    H, F = 3584, 9216
    ew, L = _dense(H, F, 64)
    bits, x = _x(T, H)
    out = L.dense_forward(x, out_dtype=torch.float32)
    L.check()
    ref = parity.oracle_dense(oracle.to_f64(bits, "bf16"), ew)
    parity.assert_close_fp32(out.cpu().numpy(), ref, f"dense T={T}")
    out_b = L.dense_forward(x)
    L.check()
    parity.assert_close_bf16(out_b.float().cpu().numpy(), ref, f"dense bf16 T={T}")


@pytest.mark.parametrize("T", [5, 40])
def test_ragged_dense_block(T):
    H, F = 288, 320
    ew, L = _dense(H, F, 64)
    bits, x = _x(T, H, seed=3)
    out = L.dense_forward(x, out_dtype=torch.float32)
    L.check()
    ref = oracle.dense_ffn(oracle.to_f64(bits, "bf16"), ew)
    parity.assert_close_fp32(out.cpu().numpy(), ref, f"ragged dense T={T}")


def test_dense_forward_needs_a_one_expert_layer():
    ew = synth.expert_weights(0, 0, 4, 256, 128)
    L = MoeLayer.from_weights(ew, k=2, scale=2.0, max_tokens=4)
    x = torch.zeros((2, 256), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(MoeError) as e:
        L.dense_forward(x)
    assert e.value.name == "MOE_ERR_INVALID_ARG"
    L.close()
