"""GPU parity: the CUDA path through the C ABI against the fp64 CPU oracle.

Workloads (seeded, synthetic): the tiny layer (H 256, E 8, top-2, F 128,
4 tokens, fp32 x), and the Xing4-shaped layer (H 3584, E 64, top-4, F 1024,
one shared expert) at decode batch 1, batched decode 64 and a 4,096-token
prefill with Zipf-skewed routing.  Routing ids must match bit for bit (the
inputs keep every token's top-k+1 scores >= 1e-4 apart); outputs must meet
the tolerance in tests/parity.py, element by element over every token (at
4,096 tokens the oracle runs on all host cores, tokens split into chunks).
"""
import functools

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from oracle import cases
from quantized_moe_expert_sigmoid_gb300 import MoeError, MoeLayer, synth
from tests import parity

pytestmark = pytest.mark.gpu

WORKLOADS = ["tiny", "decode1", "decode64", "prefill4096"]


@functools.lru_cache(maxsize=None)
def _case(name):
    wl = synth.WORKLOADS[name]
    ew = parity.weights(0, 0, wl.E, wl.H, wl.F, wl.n_shared)
    return cases.make_case(wl, ew=ew)


@functools.lru_cache(maxsize=None)
def _layer(E, H, F, k, max_tokens):
    ew = parity.weights(0, 0, E, H, F, 1)
    return MoeLayer.from_weights(ew, k=k, scale=2.0, max_tokens=max_tokens)


def _layer_for(name):
    wl = synth.WORKLOADS[name]
    return _layer(wl.E, wl.H, wl.F, wl.k, 4096 if wl.H == 3584 else 64)


def _dev_inputs(c):
    x = torch.from_numpy(c.x.view(np.int16) if c.wl.x_dtype == "bf16" else c.x).cuda()
    if c.wl.x_dtype == "bf16":
        x = x.view(torch.bfloat16)
    wr = torch.from_numpy(c.wr).cuda()
    bias = None if c.bias is None else torch.from_numpy(c.bias).cuda()
    return x, wr, bias


@pytest.mark.parametrize("name", WORKLOADS)
def test_route_ids_bit_exact(name):
    c = _case(name)
    L = _layer_for(name)
    x, wr, bias = _dev_inputs(c)
    ids, w = L.route(x, wr, bias)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(ids.cpu().numpy(), c.ids)
    np.testing.assert_allclose(w.cpu().numpy(), c.w, rtol=0, atol=2e-6)
    assert np.allclose(w.cpu().numpy().sum(1), 2.0, atol=2e-6)


@pytest.mark.parametrize("name", WORKLOADS)
def test_forward_fp32_matches_oracle(name):
    c = _case(name)
    L = _layer_for(name)
    x, _, _ = _dev_inputs(c)
    ids = torch.from_numpy(c.ids).cuda()
    w32 = c.w.astype(np.float32)
    out = L.forward(x, ids, torch.from_numpy(w32).cuda(), out_dtype=torch.float32)
    L.check()
    ref = parity.oracle_forward(c.x64, c.ids, w32.astype(np.float64), c.ew, key=(name, "w32"))
    parity.assert_close_fp32(out.cpu().numpy(), ref, name)


@pytest.mark.parametrize("name", WORKLOADS)
def test_forward_routed_matches_oracle_layer(name):
    c = _case(name)
    L = _layer_for(name)
    x, wr, bias = _dev_inputs(c)
    out, ids, w = L.forward_routed(x, wr, bias)
    L.check()
    np.testing.assert_array_equal(ids.cpu().numpy(), c.ids)
    ref = parity.oracle_forward(c.x64, c.ids, c.w, c.ew, key=(name, "w64"))
    got = out.float().cpu().numpy()
    if c.wl.x_dtype == "bf16":
        parity.assert_close_bf16(got, ref, name)
    else:
        parity.assert_close_fp32(got, ref, name)


RAGGED = [  # (H, E, k, F, T, n_shared): padding of H and F to 256, odd E, k = 1, no shared
    (96, 7, 3, 64, 5, 1),
    (160, 5, 1, 96, 33, 1),
    (288, 16, 4, 320, 100, 0),
    (512, 3, 3, 32, 17, 1),
]


@pytest.mark.parametrize("H,E,k,F,T,S", RAGGED)
def test_ragged_shapes(H, E, k, F, T, S):
    wl = synth.Workload("ragged", H, E, k, F, T, "bf16", 1.2 / H ** 0.5, n_shared=S)
    ew = synth.expert_weights(11, 0, E, H, F, S)
    if not S:
        ew.sh_up = ew.sh_gate = ew.sh_down = None
    c = cases.make_case(wl, seed=11, ew=ew)
    L = MoeLayer.from_weights(ew, k=k, scale=2.0, max_tokens=T + 3)
    x, wr, _ = _dev_inputs(c)
    out, ids, w = L.forward_routed(x, wr, out_dtype=torch.float32)
    L.check()
    np.testing.assert_array_equal(ids.cpu().numpy(), c.ids)
    ref = oracle.moe_forward(c.x64, c.ids, c.w, ew)
    parity.assert_close_fp32(out.cpu().numpy(), ref, f"H{H} E{E} k{k} F{F} T{T}")
    L.close()


def test_empty_batch_launches_nothing():
    L = _layer_for("tiny")
    x = torch.zeros((0, 256), device="cuda")
    wr = torch.zeros((8, 256), device="cuda")
    out, ids, w = L.forward_routed(x, wr)
    L.check()
    assert out.shape == (0, 256) and ids.shape == (0, 2)


def test_too_many_tokens_rejected():
    L = _layer_for("tiny")
    x = torch.zeros((65, 256), device="cuda")
    wr = torch.zeros((8, 256), device="cuda")
    with pytest.raises(MoeError) as e:
        L.route(x, wr)
    assert e.value.name == "MOE_ERR_TOO_MANY_TOKENS"


def test_misaligned_base_pointer_rejected():
    L = _layer_for("tiny")
    buf = torch.zeros(4 * 256 + 1, device="cuda")
    x = buf[1:].view(4, 256)  # 4-byte offset view: contiguous but not 16-byte aligned
    wr = torch.zeros((8, 256), device="cuda")
    with pytest.raises(MoeError) as e:
        L.route(x, wr)
    assert e.value.name == "MOE_ERR_MISALIGNED"


def test_bad_expert_id_is_reported_and_dropped():
    c = _case("tiny")
    L = _layer_for("tiny")
    x, _, _ = _dev_inputs(c)
    ids = c.ids.copy()
    ids[1, 0] = 8          # outside [0, 8)
    ids[2, 1] = -1
    w32 = c.w.astype(np.float32)
    out = L.forward(x, torch.from_numpy(ids).cuda(), torch.from_numpy(w32).cuda(),
                    out_dtype=torch.float32)
    with pytest.raises(MoeError) as e:
        L.check()
    assert e.value.name == "MOE_ERR_BAD_EXPERT_ID"
    L.check()  # the error word is cleared after being reported
    keep_w = w32.astype(np.float64).copy()
    keep_ids = ids.copy()
    for t, j in ((1, 0), (2, 1)):
        keep_w[t, j] = 0.0
        keep_ids[t, j] = 0
    ref = oracle.moe_forward(c.x64, keep_ids, keep_w, c.ew)
    parity.assert_close_fp32(out.cpu().numpy(), ref, "dropped routes")


def test_shared_bias_row_and_permuted_routes():
    """A [E] bias row (stride 0) is added to every token; and listing the
    same routes in another slot order gives the same output."""
    c = _case("decode64")
    L = _layer_for("decode64")
    x, wr, _ = _dev_inputs(c)
    row = np.zeros(64, np.float32)
    row[5] = 3.0
    ids, w = L.route(x, wr, torch.from_numpy(row).cuda())
    ref_ids, ref_w, _ = oracle.route(c.x64, c.wr, 4, 2.0, row)
    gap = oracle.min_topk_gap(c.logits + row[None, :].astype(np.float64), 4)
    ok = gap >= 1e-4
    np.testing.assert_array_equal(ids.cpu().numpy()[ok], ref_ids[ok])
    perm = np.array([2, 0, 3, 1])
    ids2 = torch.from_numpy(c.ids[:, perm].copy()).cuda()
    w2 = torch.from_numpy(np.ascontiguousarray(c.w[:, perm], dtype=np.float32)).cuda()
    out1 = L.forward(x, torch.from_numpy(c.ids).cuda(), torch.from_numpy(c.w.astype(np.float32)).cuda(),
                     out_dtype=torch.float32)
    out2 = L.forward(x, ids2, w2, out_dtype=torch.float32)
    torch.cuda.synchronize()
    a, b = out1.cpu().numpy(), out2.cpu().numpy()
    assert np.abs(a - b).max() <= 1e-5 * np.abs(a).max()


def test_binding_refuses_strided_and_mistyped_tensors():
    c = _case("tiny")
    L = _layer_for("tiny")
    x, wr, _ = _dev_inputs(c)
    ids = torch.from_numpy(c.ids).cuda()
    w_t = torch.from_numpy(np.asfortranarray(c.w.astype(np.float32))).cuda()  # column-major
    with pytest.raises(ValueError):
        L.forward(x, ids, w_t)
    with pytest.raises(TypeError):
        L.forward(x, ids.long(), torch.from_numpy(c.w.astype(np.float32)).cuda())
    with pytest.raises(ValueError):
        L.route(x.t().contiguous().t(), wr)


@pytest.mark.parametrize("T", [1, 2, 3, 5, 8])
def test_single_launch_decode_matches_oracle(T):
    """Batches of up to 8 tokens run the whole layer in one launch."""
    import quantized_moe_expert_sigmoid_gb300 as moe
    wl = synth.WORKLOADS["decode1"]
    ew = parity.weights(0, 0, wl.E, wl.H, wl.F, 1)
    c = cases.make_case(wl, T=T, ew=ew, seed=0)
    L = _layer_for("decode1")
    x, wr, _ = _dev_inputs(c)
    before = moe.moe_launch_count()
    out, ids, w = L.forward_routed(x, wr, out_dtype=torch.float32)
    assert moe.moe_launch_count() - before == 1
    L.check()
    np.testing.assert_array_equal(ids.cpu().numpy(), c.ids)
    np.testing.assert_allclose(w.cpu().numpy(), c.w, rtol=0, atol=2e-6)
    ref = oracle.moe_forward(c.x64, c.ids, c.w, c.ew)
    parity.assert_close_fp32(out.cpu().numpy(), ref, f"T={T}")
    out2 = L.forward(x, ids, w, out_dtype=torch.float32)
    L.check()
    parity.assert_close_fp32(out2.cpu().numpy(), ref, f"T={T} given routes")


def test_graph_replay_matches_eager():
    """Layer calls captured in a CUDA graph (with programmatic dependent
    launch between them) give the eager results."""
    import quantized_moe_expert_sigmoid_gb300 as moe
    c = _case("decode1")
    L = _layer_for("decode1")
    x, wr, _ = _dev_inputs(c)
    xs = [x.clone() for _ in range(4)]
    for i, xi in enumerate(xs):
        xi.mul_(1.0 + 0.25 * i)
    ids = [torch.empty((1, 4), dtype=torch.int32, device="cuda") for _ in xs]
    ws = [torch.empty((1, 4), dtype=torch.float32, device="cuda") for _ in xs]
    outs = [torch.empty((1, 3584), dtype=torch.bfloat16, device="cuda") for _ in xs]
    eager = []
    for i, xi in enumerate(xs):
        o, _, _ = L.forward_routed(xi, wr)
        eager.append(o.float().cpu())
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for i, xi in enumerate(xs):
            moe.moe_layer_forward_routed(L.handle, xi, wr, ids[i], ws[i], outs[i])
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    L.check()
    for i in range(len(xs)):
        assert torch.allclose(outs[i].float().cpu(), eager[i], rtol=0, atol=2e-2 * eager[i].abs().max().item())


@pytest.mark.parametrize("H,E,k,T,zipf", [(256, 8, 2, 256, False), (288, 100, 8, 300, True),
                                          (3584, 64, 4, 512, False)])
def test_large_batch_router_bit_exact(H, E, k, T, zipf):
    """Batches of >= 256 bf16 tokens take the tensor-core router (the fp32
    router rows split into three exact bf16 parts): ids must still equal
    the fp64 oracle's bit for bit; E > 64 exercises two rows per splitting
    thread, H = 288 a K tail that is half a 64-wide step."""
    wl = synth.Workload(f"router: H {H}, E {E}, top-{k}, {T} tokens", H, E, k, 32, T, "bf16", 0.05,
                        zipf=zipf)
    ew = synth.expert_weights(0, 0, E, H, 32)
    c = cases.make_case(wl, ew=ew)
    L = MoeLayer.from_weights(ew, k=k, scale=wl.scale, max_tokens=T)
    x, wr, bias = _dev_inputs(c)
    ids, w = L.route(x, wr, bias)
    torch.cuda.synchronize()
    L.check()
    np.testing.assert_array_equal(ids.cpu().numpy(), c.ids)
    np.testing.assert_allclose(w.cpu().numpy(), c.w, rtol=0, atol=2e-6)
    L.close()


@pytest.mark.parametrize("T,boost", [(1, 2.0 ** 8), (3, 2.0 ** 15), (8, 2.0 ** 11)])
def test_decode_activation_blocks_with_wide_range(T, boost):
    """The single-launch decode kernel (T <= 8) holds x and the SwiGLU output
    h as 16-bit integers with one power-of-two scale per 32-element block:
    an element is exact while its exponent is within 6 of the block's
    largest, and smaller ones are rounded to the block's step (at most 2^-14
    of the block's largest).  Worst case for that reading of the
    fp32-accumulating GEMV: one element of every 32-block scaled up by
    2^8 .. 2^15 (so most of the block sits 8 to 15 binades below its
    maximum), given routes, against the oracle within the parity tolerance."""
    wl = synth.WORKLOADS["decode1"]
    ew = parity.weights(0, 0, wl.E, wl.H, wl.F, 1)
    c = cases.make_case(wl, T=T, ew=ew)
    x32 = synth.bf16_bits_to_f32(c.x).reshape(T, wl.H // 32, 32).copy()
    for t in range(T):
        for b in range(wl.H // 32):
            x32[t, b, (7 * t + 3 * b) % 32] *= boost * (1.0 if b % 2 else -1.0)
    bits = synth.to_bf16_bits(x32.reshape(T, wl.H))
    x64 = oracle.to_f64(bits, "bf16")
    x = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
    L = _layer_for("decode1")
    w32 = c.w.astype(np.float32)
    out = L.forward(x, torch.from_numpy(c.ids).cuda(), torch.from_numpy(w32).cuda(), out_dtype=torch.float32)
    L.check()
    ref = oracle.moe_forward(x64, c.ids, w32.astype(np.float64), ew)
    parity.assert_close_fp32(out.cpu().numpy(), ref, f"wide-range blocks T={T} boost 2^{int(np.log2(boost))}")


def test_max_tokens_boundary():
    """T == max_tokens runs; T == max_tokens + 1 is refused before any launch."""
    import quantized_moe_expert_sigmoid_gb300 as moe
    wl = synth.WORKLOADS["decode1"]
    ew = parity.weights(0, 0, wl.E, wl.H, wl.F, 1)
    c = cases.make_case(wl, T=9, ew=ew)
    L = MoeLayer.from_weights(ew, k=wl.k, scale=wl.scale, max_tokens=8)
    x, wr, _ = _dev_inputs(c)
    out, ids, w = L.forward_routed(x[:8], wr, out_dtype=torch.float32)
    L.check()
    np.testing.assert_array_equal(ids.cpu().numpy(), c.ids[:8])
    ref = oracle.moe_forward(c.x64[:8], c.ids[:8], c.w[:8], ew)
    parity.assert_close_fp32(out.cpu().numpy(), ref, "T = max_tokens")
    before = moe.moe_launch_count()
    with pytest.raises(MoeError) as e:
        L.forward_routed(x, wr)
    assert e.value.name == "MOE_ERR_TOO_MANY_TOKENS"
    assert moe.moe_launch_count() == before
    L.close()


@pytest.mark.parametrize("T", [9, 16, 40, 64])
def test_batched_decode_path_matches_oracle(T):
    """9..64 tokens run the batched decode path (register dequantisation,
    mma.sync, route-ordered activations): ids bit-exact, fp32 and bf16
    outputs within tolerance of the oracle on every token."""
    wl = synth.WORKLOADS["decode64"]
    ew = parity.weights(0, 0, wl.E, wl.H, wl.F, 1)
    c = cases.make_case(wl, T=T, ew=ew, seed=3)
    L = _layer_for("decode64")
    x, wr, _ = _dev_inputs(c)
    out, ids, w = L.forward_routed(x, wr, out_dtype=torch.float32)
    L.check()
    np.testing.assert_array_equal(ids.cpu().numpy(), c.ids)
    ref = parity.oracle_forward(c.x64, c.ids, c.w, ew)
    parity.assert_close_fp32(out.cpu().numpy(), ref, f"batched decode T={T}")
    out_b, _, _ = L.forward_routed(x, wr)
    L.check()
    parity.assert_close_bf16(out_b.float().cpu().numpy(), ref, f"batched decode bf16 T={T}")


def test_batched_decode_expert_with_more_than_64_routes():
    """Given routes may name an expert more than once per token: 64 tokens
    with every slot on experts 5 and 9 put 128 routes on each, more than one
    pass of the batched kernels' 64-route activation tile."""
    wl = synth.WORKLOADS["decode64"]
    ew = parity.weights(0, 0, wl.E, wl.H, wl.F, 1)
    c = cases.make_case(wl, T=64, ew=ew, seed=4)
    L = _layer_for("decode64")
    x, _, _ = _dev_inputs(c)
    ids = np.tile(np.array([5, 9, 5, 9], np.int32), (64, 1))
    w = np.tile(np.array([0.7, 0.5, 0.3, 0.5], np.float32), (64, 1))
    out = L.forward(x, torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(), out_dtype=torch.float32)
    L.check()
    ref = parity.oracle_forward(c.x64, ids, w.astype(np.float64), ew)
    parity.assert_close_fp32(out.cpu().numpy(), ref, "128 routes per expert")
