"""Bit-reproducible output.  A layer created with MOE_FLAG_DETERMINISTIC adds
each token's routed outputs in slot order (the shared expert last) from a
per-route buffer with one writer per element, instead of float atomics; the
single-launch decode kernel (T <= 8) reduces in a fixed order with or
without the flag.  Repeated calls, eager and graph-replayed, must give
identical bits, and the result must still meet the oracle tolerance.
"""
import functools

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from oracle import cases
from quantized_moe_expert_sigmoid_gb300 import (MOE_FLAG_DETERMINISTIC, MoeError, MoeLayer,
                                                moe_layer_forward_routed, synth)
from tests import parity

pytestmark = pytest.mark.gpu


@functools.lru_cache(maxsize=None)
def _xing4(flags, max_tokens):
    wl = synth.WORKLOADS["decode1"]
    ew = parity.weights(0, 0, wl.E, wl.H, wl.F, 1)
    return MoeLayer.from_weights(ew, k=wl.k, scale=wl.scale, max_tokens=max_tokens, flags=flags)


@functools.lru_cache(maxsize=None)
def _case(name, T=None):
    wl = synth.WORKLOADS[name]
    return cases.make_case(wl, T=T, ew=parity.weights(0, 0, wl.E, wl.H, wl.F, 1))


def _dev(c):
    x = torch.from_numpy(c.x.view(np.int16)).cuda().view(torch.bfloat16)
    bias = None if c.bias is None else torch.from_numpy(c.bias).cuda()
    return x, torch.from_numpy(c.wr).cuda(), bias


def _bits(t):
    return t.contiguous().view(torch.int32 if t.dtype == torch.float32 else torch.int16).cpu().numpy()


@pytest.mark.parametrize("name,T", [("decode64", 16), ("decode64", None), ("prefill4096", None)])
def test_deterministic_combine_repeats_bit_for_bit(name, T):
    c = _case(name, T)
    T = c.wl.T if T is None else T
    L = _xing4(MOE_FLAG_DETERMINISTIC, 4096)
    x, wr, bias = _dev(c)
    outs = []
    for _ in range(3):
        out, ids, w = L.forward_routed(x, wr, bias, out_dtype=torch.float32)
        outs.append(_bits(out))
    L.check()
    for o in outs[1:]:
        np.testing.assert_array_equal(o, outs[0])
    np.testing.assert_array_equal(ids.cpu().numpy(), c.ids)
    ref = parity.oracle_forward(c.x64, c.ids, c.w, c.ew, key=(name, T, "w64"))
    got = outs[0].view(np.float32)
    parity.assert_close_fp32(got, ref, f"{name} deterministic")
    # bf16 output: the same fp32 sum rounded once
    out_b, _, _ = L.forward_routed(x, wr, bias)
    L.check()
    f32 = torch.from_numpy(outs[0].view(np.float32)).cuda()
    assert torch.equal(out_b, f32.bfloat16())


def test_deterministic_and_atomic_combines_agree():
    """The slot-ordered sum and the atomic sum add the same fp32 terms in
    different orders: they differ by a few fp32 roundings at most."""
    c = _case("decode64")
    x, wr, bias = _dev(c)
    a, _, _ = _xing4(MOE_FLAG_DETERMINISTIC, 4096).forward_routed(x, wr, bias, out_dtype=torch.float32)
    b, _, _ = _xing4(0, 4096).forward_routed(x, wr, bias, out_dtype=torch.float32)
    torch.cuda.synchronize()
    d = (a - b).abs().max().item()
    assert d <= 1e-5 * b.abs().max().item(), d


def test_deterministic_graph_replay_equals_eager():
    c = _case("decode64")
    L = _xing4(MOE_FLAG_DETERMINISTIC, 4096)
    x, wr, bias = _dev(c)
    eager, _, _ = L.forward_routed(x, wr, bias, out_dtype=torch.float32)
    eager = _bits(eager)
    T = x.shape[0]
    ids = torch.empty((T, 4), dtype=torch.int32, device="cuda")
    w = torch.empty((T, 4), dtype=torch.float32, device="cuda")
    out = torch.empty((T, 3584), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        moe_layer_forward_routed(L.handle, x, wr, ids, w, out, bias)
    for _ in range(3):
        g.replay()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(_bits(out), eager)
    L.check()


def test_deterministic_drops_bad_ids():
    """A dropped route (id outside [0, E)) adds nothing to the ordered sum."""
    c = _case("decode64", 16)
    L = _xing4(MOE_FLAG_DETERMINISTIC, 4096)
    x, _, _ = _dev(c)
    ids = c.ids.copy()
    ids[3, 1] = 64
    ids[9, 0] = -5
    w32 = c.w.astype(np.float32)
    out = L.forward(x, torch.from_numpy(ids).cuda(), torch.from_numpy(w32).cuda(), out_dtype=torch.float32)
    with pytest.raises(MoeError) as e:
        L.check()
    assert e.value.name == "MOE_ERR_BAD_EXPERT_ID"
    keep_ids, keep_w = ids.copy(), w32.astype(np.float64)
    for t, j in ((3, 1), (9, 0)):
        keep_ids[t, j], keep_w[t, j] = 0, 0.0
    ref = oracle.moe_forward(c.x64, keep_ids, keep_w, c.ew)
    parity.assert_close_fp32(out.cpu().numpy(), ref, "deterministic, dropped routes")


@pytest.mark.parametrize("flags", [0, MOE_FLAG_DETERMINISTIC])
@pytest.mark.parametrize("T", [1, 3, 8])
def test_single_launch_decode_repeats_bit_for_bit(T, flags):
    c = _case("decode1", T)
    L = _xing4(flags, 4096)
    x, wr, _ = _dev(c)
    outs = [_bits(L.forward_routed(x, wr, out_dtype=torch.float32)[0]) for _ in range(4)]
    L.check()
    for o in outs[1:]:
        np.testing.assert_array_equal(o, outs[0])


@pytest.mark.parametrize("F", [768, 1536])
def test_ragged_shape_deterministic(F):
    """The decode kernel's row reduction with three parts per row: F = 768
    (48 units per row, 16-lane groups) and F = 1,536 (96 units, 32-lane
    groups); H = 288, no shared expert, decode and batched."""
    H, E, k = 288, 16, 4
    ew = synth.expert_weights(13, 0, E, H, F, 0)
    ew.sh_up = ew.sh_gate = ew.sh_down = None
    L = MoeLayer.from_weights(ew, k=k, scale=2.0, max_tokens=40, flags=MOE_FLAG_DETERMINISTIC)
    for T in (2, 40):
        wl = synth.Workload("ragged deterministic", H, E, k, F, T, "bf16", 1.2 / H ** 0.5, n_shared=0)
        c = cases.make_case(wl, seed=13, ew=ew)
        x = torch.from_numpy(c.x.view(np.int16)).cuda().view(torch.bfloat16)
        wr = torch.from_numpy(c.wr).cuda()
        outs = [_bits(L.forward_routed(x, wr, out_dtype=torch.float32)[0]) for _ in range(3)]
        L.check()
        for o in outs[1:]:
            np.testing.assert_array_equal(o, outs[0])
        ref = oracle.moe_forward(c.x64, c.ids, c.w, ew)
        parity.assert_close_fp32(outs[0].view(np.float32), ref, f"ragged deterministic T={T}")
    L.close()
