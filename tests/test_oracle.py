"""Pins for the CPU oracle: each checks it against something other than itself.

Sources: HelloSun/xing4_0-29b-IQ4_NL_EPQ model card ("模型與路由": sigmoid
router, expert_weights_norm, scale 2.0, top-4 of 64, one shared expert;
"對純 NumPy": IQ4_NL = 16-entry table x one fp16 scale; "權重組成": byte sizes),
PocketLLM "Xing4.0-29B-A4B: the design record" (section 2: shared expert added
to the routed sum), zhuai.tech "FFN: feature processing inside each layer"
(gated MLP with SiLU).

``test_planted_mistakes_are_caught`` plants plausible mistakes in a copy of
oracle.c and checks that at least one pin fails for each.
"""
import itertools
import math
import os
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
from quantized_moe_expert_sigmoid_gb300 import synth

# The IQ4_NL table, as given with the synthetic workload definition.
CODEBOOK = np.array([-127, -104, -83, -65, -49, -35, -22, -10,
                     1, 13, 25, 38, 53, 69, 89, 113], dtype=np.float64)
HERE = os.path.dirname(os.path.abspath(__file__))


def _read_golden(name):
    path = os.path.join(HERE, "golden", name)
    with open(path) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def _fp16_bits(v):
    return int(np.array([v], dtype=np.float16).view(np.uint16)[0])


def _pack_rows(d_rows, q):
    """Rows of blocks with one fp16 scale per row and index matrix q [N, K],
    packed with weight j in the low nibble and weight j+16 in the high nibble
    of index byte j (the reading the golden blocks fix)."""
    N, K = q.shape
    nb = K // 32
    out = np.zeros((N, nb, 18), dtype=np.uint8)
    for n in range(N):
        bits = _fp16_bits(d_rows[n])
        for b in range(nb):
            out[n, b, 0] = bits & 0xFF
            out[n, b, 1] = bits >> 8
            qq = q[n, 32 * b:32 * b + 32]
            out[n, b, 2:] = (qq[:16] | (qq[16:] << 4)).astype(np.uint8)
    return out


def _silu(v):
    return v / (1.0 + np.exp(-v))


# --------------------------------------------------------------------------
# pins (plain functions so the mutation test can run them on a planted copy)
# --------------------------------------------------------------------------

def pin_fp16_values():
    for bits, val in _read_golden("fp16_values.txt"):
        got = oracle.fp16_to_double(int(bits, 16))
        want = float(val)
        assert got == want and math.copysign(1, got) == math.copysign(1, want), (bits, got, want)
    assert math.isinf(oracle.fp16_to_double(0x7C00))


def pin_golden_blocks():
    rows = _read_golden("iq4nl_blocks.txt")
    assert len(rows) % 2 == 0 and len(rows) >= 6
    for blk, w in zip(rows[0::2], rows[1::2]):
        assert blk[0] == "block" and w[0] == "w"
        b = np.array([int(h, 16) for h in blk[1:]], dtype=np.uint8).reshape(1, 18)
        want = np.array([float(v) for v in w[1:]])
        got = oracle.iq4nl_dequant(b).ravel()
        assert np.array_equal(got, want), (got, want)


def pin_matrix_bytes():
    # "權重組成": gate/up/down are 2,064,384 B each, 6,193,152 B per expert
    m = synth.iq4nl_blocks(0, "size", 1024, 3584)
    assert m.nbytes == 2_064_384
    assert 3 * m.nbytes == 6_193_152
    assert oracle.iq4nl_dequant(m[:2]).shape == (2, 3584)


def pin_roundtrip():
    blocks = synth.iq4nl_blocks(7, "rt", 16, 256).reshape(-1, 18)
    w = oracle.iq4nl_dequant(blocks.reshape(1, -1, 18)).ravel()
    d_bits = blocks[:, 0].astype(np.uint16) | (blocks[:, 1].astype(np.uint16) << 8)
    again = oracle.iq4nl_quantize(w, d_bits)
    assert np.array_equal(again, blocks)


def pin_router_hand_case():
    # x = e_0, logits = first column of Wr: [0.5, 2, -1, 1] (+ bias on expert 2)
    x = np.array([[1.0, 0.0]])
    wr = np.array([[0.5, 0.3], [2.0, -1.0], [-1.0, 4.0], [1.0, 0.0]])
    ids, w, logits = oracle.route(x, wr, k=2, scale=2.0)
    assert np.array_equal(logits, [[0.5, 2.0, -1.0, 1.0]])
    assert ids.tolist() == [[1, 3]]
    s1, s3 = 1 / (1 + math.exp(-2.0)), 1 / (1 + math.exp(-1.0))
    assert np.allclose(w, [[2 * s1 / (s1 + s3), 2 * s3 / (s1 + s3)]], rtol=0, atol=1e-15)
    # a bias of +2.5 on expert 2 makes its logit 1.5: selected second, and the
    # biased score enters the weights
    bias = np.array([[0.0, 0.0, 2.5, 0.0]])
    ids, w, _ = oracle.route(x, wr, k=2, scale=2.0, bias=bias)
    assert ids.tolist() == [[1, 2]]
    s2 = 1 / (1 + math.exp(-1.5))
    assert np.allclose(w, [[2 * s1 / (s1 + s2), 2 * s2 / (s1 + s2)]], rtol=0, atol=1e-15)
    # equal scores go to the lower expert id
    wr_tie = np.array([[1.0, 0.0], [3.0, 0.0], [1.0, 0.0], [3.0, 0.0]])
    ids, _, _ = oracle.route(x, wr_tie, k=3, scale=2.0)
    assert ids.tolist() == [[1, 3, 0]]


def pin_router_brute_force():
    wl = synth.WORKLOADS["tiny"]
    wr = synth.router_weights(3, 0, wl.E, wl.H, wl.router_sigma)
    x = oracle.to_f64(synth.activations(3, "x", 16, wl.H, dtype="fp32"), "fp32")
    ids, w, _ = oracle.route(x, wr, wl.k, wl.scale)
    s = 1 / (1 + np.exp(-(x @ wr.astype(np.float64).T)))
    for t in range(x.shape[0]):
        best = max(itertools.combinations(range(wl.E), wl.k), key=lambda c: sum(s[t, list(c)]))
        assert set(best) == set(ids[t].tolist())
        assert all(s[t, ids[t, j]] > s[t, ids[t, j + 1]] for j in range(wl.k - 1))
        assert abs(w[t].sum() - wl.scale) < 1e-12
        assert np.allclose(w[t], wl.scale * s[t, ids[t]] / s[t, ids[t]].sum(), rtol=1e-12)


def pin_weights_sum_to_scale():
    wl = synth.WORKLOADS["decode1"]
    wr = synth.router_weights(0, 0, wl.E, wl.H, wl.router_sigma)
    x = oracle.to_f64(synth.activations(0, "x", 8, wl.H), "bf16")
    for scale in (2.0, 2.5, 1.0):
        _, w, _ = oracle.route(x, wr, 4, scale)
        assert np.all(np.abs(w.sum(axis=1) - scale) <= 1e-12)


class _EW:
    def __init__(self, up, gate, down, sh_up=None, sh_gate=None, sh_down=None):
        self.up, self.gate, self.down = up, gate, down
        self.sh_up, self.sh_gate, self.sh_down = sh_up, sh_gate, sh_down


def pin_rank_one_closed_form():
    """Every matrix is diag(d) x C with C's column c = table[q_c]: then
    W x = d * (table[q] . x) and the FFN has a closed form per row.  F != H,
    so a transposed operand or a permuted nibble order changes the answer."""
    rng = np.random.default_rng(11)
    H, F, E, k, T = 96, 64, 3, 2, 2
    params = []
    up, gate, down = [], [], []
    for e in range(E + 1):
        dg = 2.0 ** rng.integers(-9, -6, F) * rng.integers(1, 4, F)
        du = 2.0 ** rng.integers(-9, -6, F) * rng.integers(1, 4, F)
        dd = 2.0 ** rng.integers(-9, -6, H) * rng.integers(1, 4, H)
        qg, qu = rng.integers(0, 16, H), rng.integers(0, 16, H)
        qd = rng.integers(0, 16, F)
        params.append((dg, du, dd, qg, qu, qd))
        up.append(_pack_rows(du, np.tile(qu, (F, 1))))
        gate.append(_pack_rows(dg, np.tile(qg, (F, 1))))
        down.append(_pack_rows(dd, np.tile(qd, (H, 1))))
    ew = _EW(np.stack(up[:E]), np.stack(gate[:E]), np.stack(down[:E]), up[E], gate[E], down[E])
    x = rng.standard_normal((T, H))
    ids = np.array([[2, 0], [1, 2]], dtype=np.int32)
    wts = np.array([[1.25, 0.75], [0.5, 1.5]])

    def ffn(e, xt):
        dg, du, dd, qg, qu, qd = params[e]
        g = dg * float(CODEBOOK[qg] @ xt)
        u = du * float(CODEBOOK[qu] @ xt)
        h = _silu(g) * u
        return dd * float(CODEBOOK[qd] @ h)

    want = np.stack([sum(wts[t, j] * ffn(ids[t, j], x[t]) for j in range(k)) + ffn(E, x[t])
                     for t in range(T)])
    got = oracle.moe_forward(x, ids, wts, ew)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12 * np.abs(want).max())


def _tiny_layer(seed=5, E=8, H=64, F=32):
    ew = synth.expert_weights(seed, 0, E, H, F)
    wr = synth.router_weights(seed, 0, E, H, 0.2)
    x = oracle.to_f64(synth.activations(seed, "x", 3, H, dtype="fp32"), "fp32")
    return ew, wr, x


def _dense_ffn(blocks_up, blocks_gate, blocks_down, xt):
    wu = oracle.iq4nl_dequant(blocks_up)
    wg = oracle.iq4nl_dequant(blocks_gate)
    wd = oracle.iq4nl_dequant(blocks_down)
    return wd @ (_silu(wg @ xt) * (wu @ xt))


def pin_all_experts_equals_dense():
    ew, wr, x = _tiny_layer()
    E = ew.up.shape[0]
    out, ids, w = oracle.moe_layer(x, wr, ew, k=E, scale=2.0)
    for t in range(x.shape[0]):
        s = 1 / (1 + np.exp(-(wr.astype(np.float64) @ x[t])))
        dense = sum(2.0 * s[e] / s.sum() * _dense_ffn(ew.up[e], ew.gate[e], ew.down[e], x[t])
                    for e in range(E))
        dense = dense + _dense_ffn(ew.sh_up, ew.sh_gate, ew.sh_down, x[t])
        assert np.allclose(out[t], dense, rtol=1e-10, atol=1e-12 * np.abs(dense).max())


def pin_top1_special_case():
    ew, wr, x = _tiny_layer(seed=6)
    out, ids, w = oracle.moe_layer(x, wr, ew, k=1, scale=2.0)
    assert np.all(w == 2.0)
    for t in range(x.shape[0]):
        s = 1 / (1 + np.exp(-(wr.astype(np.float64) @ x[t])))
        e = int(np.argmax(s))
        assert ids[t, 0] == e
        want = 2.0 * _dense_ffn(ew.up[e], ew.gate[e], ew.down[e], x[t]) + \
            _dense_ffn(ew.sh_up, ew.sh_gate, ew.sh_down, x[t])
        assert np.allclose(out[t], want, rtol=1e-10, atol=1e-12 * np.abs(want).max())


def pin_permutation_and_token_independence():
    ew, wr, x = _tiny_layer(seed=8)
    E = ew.up.shape[0]
    out, ids, w = oracle.moe_layer(x, wr, ew, k=3)
    perm = np.random.default_rng(1).permutation(E)
    ew_p = _EW(ew.up[perm], ew.gate[perm], ew.down[perm], ew.sh_up, ew.sh_gate, ew.sh_down)
    out_p, ids_p, w_p = oracle.moe_layer(x, wr[perm], ew_p, k=3)
    assert np.allclose(out_p, out, rtol=1e-12, atol=1e-12 * np.abs(out).max())
    assert np.array_equal(perm[ids_p], ids)
    for t in range(x.shape[0]):
        o1, _, _ = oracle.moe_layer(x[t:t + 1], wr, ew, k=3)
        assert np.array_equal(o1[0], out[t])


def pin_zero_weight_route_contributes_nothing():
    ew, wr, x = _tiny_layer(seed=9)
    ids = np.array([[0, 5], [3, 3], [7, 1]], dtype=np.int32)
    w = np.array([[1.0, 0.0], [0.5, 0.5], [0.0, 2.0]])
    out = oracle.moe_forward(x, ids, w, ew)
    sh = [_dense_ffn(ew.sh_up, ew.sh_gate, ew.sh_down, x[t]) for t in range(3)]
    f = lambda e, t: _dense_ffn(ew.up[e], ew.gate[e], ew.down[e], x[t])
    want = np.stack([f(0, 0) + sh[0], f(3, 1) + sh[1], 2.0 * f(1, 2) + sh[2]])
    assert np.allclose(out, want, rtol=1e-10, atol=1e-12 * np.abs(want).max())


def pin_repeated_expert_in_one_token():
    # out[t] sums w * FFN over the slots, so an expert named in every slot of
    # a token contributes (sum of its weights) * FFN_e once per token; four
    # tokens with three slots each put twelve routes on one expert
    ew, wr, x = _tiny_layer(seed=11)
    x = np.concatenate([x, x[:1] * 0.5])
    ids = np.array([[2, 2, 2], [6, 6, 6], [2, 2, 2], [6, 2, 6]], dtype=np.int32)
    w = np.array([[0.5, 0.25, 1.0], [1.0, 0.5, 0.5], [0.125, 0.125, 0.25], [0.75, 1.5, 0.25]])
    out = oracle.moe_forward(x, ids, w, ew)
    f = lambda e, t: _dense_ffn(ew.up[e], ew.gate[e], ew.down[e], x[t])
    sh = lambda t: _dense_ffn(ew.sh_up, ew.sh_gate, ew.sh_down, x[t])
    want = np.stack([1.75 * f(2, 0) + sh(0), 2.0 * f(6, 1) + sh(1), 0.5 * f(2, 2) + sh(2),
                     1.0 * f(6, 3) + 1.5 * f(2, 3) + sh(3)])
    assert np.allclose(out, want, rtol=1e-10, atol=1e-12 * np.abs(want).max())


def pin_rmsnorm_closed_form():
    r = np.array([[3.0] * 8, [-0.5] * 8, [0.0] * 8])
    u = oracle.rmsnorm(r, 1e-6)
    for i, c in enumerate([3.0, -0.5, 0.0]):
        assert np.allclose(u[i], c / math.sqrt(c * c + 1e-6), rtol=1e-15, atol=0)
    r2 = np.array([[1.0, -1.0, 2.0, -2.0]])
    assert np.allclose(oracle.rmsnorm(r2, 0.0), r2 / math.sqrt(2.5), rtol=1e-15)


def pin_invalid_ids_rejected():
    ew, wr, x = _tiny_layer(seed=10)
    with pytest.raises(ValueError):
        oracle.moe_forward(x, np.array([[0, 8]] * 3, dtype=np.int32), np.ones((3, 2)), ew)


def pin_selection_bias_hand_case():
    """noaux_tc [EPQ "模型與路由": sigmoid + ffn_exp_probs_b]: the bias moves
    expert 1 ahead of expert 0, the weights stay the unbiased scores."""
    x = np.array([[1.0]])
    wr = np.array([[2.0], [1.0], [0.0]])                 # l = 2, 1, 0
    s = 1.0 / (1.0 + np.exp(-np.array([2.0, 1.0, 0.0])))  # 0.8808, 0.7311, 0.5
    b = np.array([0.0, 0.2, 0.0])                        # keys 0.8808, 0.9311, 0.5
    ids, w, _ = oracle.route_selbias(x, wr, 2, 2.0, b)
    assert ids.tolist() == [[1, 0]]
    np.testing.assert_allclose(w[0], 2.0 * np.array([s[1], s[0]]) / (s[1] + s[0]), rtol=1e-15)
    ids1, w1, _ = oracle.route_selbias(x, wr, 1, 2.0, b)
    assert ids1.tolist() == [[1]] and w1[0, 0] == 2.0
    # equal keys go to the lower id: b makes expert 2's key equal expert 1's
    b2 = np.array([-1.0, 0.0, s[1] - s[2]])
    ids2, _, _ = oracle.route_selbias(x, wr, 1, 2.0, b2)
    assert ids2.tolist() == [[1]]


def pin_selection_bias_zero_and_forcing():
    """b = 0 is the plain router; a large bias on one expert puts it first
    for every token without changing the other weights' ratios."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal((6, 32))
    wr = rng.standard_normal((8, 32)) * 0.3
    ids0, w0, _ = oracle.route(x, wr, 3, 2.0)
    ids1, w1, l1 = oracle.route_selbias(x, wr, 3, 2.0, np.zeros(8))
    np.testing.assert_array_equal(ids1, ids0)
    np.testing.assert_array_equal(w1, w0)
    b = np.zeros(8)
    b[5] = 10.0
    ids2, w2, _ = oracle.route_selbias(x, wr, 3, 2.0, b)
    assert (ids2[:, 0] == 5).all()
    s = 1.0 / (1.0 + np.exp(-l1))
    for t in range(6):
        sel = s[t, ids2[t]]
        np.testing.assert_allclose(w2[t], 2.0 * sel / sel.sum(), rtol=1e-14)


def pin_dense_block():
    # a one-expert layer with weight 1 and no shared expert is the plain FFN,
    # checked against the dense loop above
    ew = synth.dense_ffn_weights(9, 0, 64, 96)
    x = oracle.to_f64(synth.activations(9, "x", 4, 64, dtype="fp32"), "fp32")
    out = oracle.dense_ffn(x, ew)
    for t in range(x.shape[0]):
        want = _dense_ffn(ew.up[0], ew.gate[0], ew.down[0], x[t])
        assert np.allclose(out[t], want, rtol=1e-10, atol=1e-12 * np.abs(want).max())


PINS = [pin_fp16_values, pin_golden_blocks, pin_matrix_bytes, pin_roundtrip,
        pin_router_hand_case, pin_router_brute_force, pin_weights_sum_to_scale,
        pin_rank_one_closed_form, pin_all_experts_equals_dense, pin_top1_special_case,
        pin_permutation_and_token_independence, pin_zero_weight_route_contributes_nothing,
        pin_repeated_expert_in_one_token, pin_rmsnorm_closed_form, pin_invalid_ids_rejected, pin_selection_bias_hand_case,
        pin_selection_bias_zero_and_forcing, pin_dense_block]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin()


def test_empty_batch():
    ew, wr, x = _tiny_layer()
    out = oracle.moe_forward(x[:0], np.zeros((0, 2), np.int32), np.zeros((0, 2)), ew)
    assert out.shape == (0, x.shape[1])


# Plausible mistakes, each planted in a copy of oracle.c; the pins must catch all.
MUTANTS = {
    "nibble order swapped": ("kCodebook[qs[j] & 15]", "kCodebook[qs[j] >> 4]"),
    "fp16 exponent bias": ("ex - 25", "ex - 24"),
    "sigmoid sign": ("1.0 / (1.0 + exp(-v))", "1.0 / (1.0 + exp(v))"),
    "bias dropped": ("if (bias) acc +=", "if (0) acc +="),
    "selects smallest": ("s[e] > s[best]", "s[e] < s[best]"),
    "ties to higher id": ("s[e] > s[best]", "s[e] >= s[best]"),
    "scale dropped": ("weights[t * k + j] = scale *", "weights[t * k + j] = 1.0 *"),
    "shared expert dropped": ("e < E + n_shared", "e < E"),
    "silu replaced by sigmoid": ("h[f] = g * sigmoid(g) * u", "h[f] = sigmoid(g) * u"),
    "gate/up swapped": ("h[f] = g * sigmoid(g) * u", "h[f] = u * sigmoid(u) * g"),
    "down transposed": ("wd[r * F + f]", "wd[f * H + r]"),
    "route weight dropped": ("ot[r] += wt[i] * y", "ot[r] += y"),
    "rmsnorm mean": ("ss / (double)H", "ss / (double)(H - 1)"),
    "selection bias subtracted": ("choice[e] = prob[e] + bias", "choice[e] = prob[e] - bias"),
    "selection by smallest key": ("choice[e] > choice[best]", "choice[e] < choice[best]"),
    "selection bias in the weights": ("sum += prob[best]", "sum += choice[best]"),
    "selection bias ignored": ("choice[e] = prob[e] + bias[t * bias_stride + e]", "choice[e] = prob[e]"),
}


def test_planted_mistakes_are_caught():
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    escaped = []
    with tempfile.TemporaryDirectory() as tmp:
        for name, (a, b) in MUTANTS.items():
            assert src.count(a) >= 1, name
            mut = os.path.join(tmp, "m.c")
            lib = os.path.join(tmp, f"m{len(escaped)}_{abs(hash(name))}.so")
            with open(mut, "w") as f:
                f.write(src.replace(a, b, 1))
            subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", mut, "-o", lib, "-lm"])
            with oracle.using_library(lib):
                caught = False
                for pin in PINS:
                    try:
                        pin()
                    except Exception:
                        caught = True
                        break
            if not caught:
                escaped.append(name)
    assert not escaped, f"mistakes no pin catches: {escaped}"


def test_selection_bias_cases_change_routes_and_keep_gaps():
    """The parity cases with a drawn selection bias: it changes the chosen
    set of most tokens (so the GPU tests exercise it), every token's k+1
    largest keys stay >= 1e-4 apart, and the weights, free of the bias,
    still sum to routed_scaling."""
    from oracle import cases
    wl = synth.Workload("selection bias: H 256, E 64, top-4, 64 tokens", 256, 64, 4, 32, 64, "bf16", 0.05)
    ew = synth.expert_weights(0, 0, wl.E, wl.H, wl.F)
    for b in (synth.selection_bias(0, wl.E), synth.selection_bias(1, wl.E, wl.T)):
        c = cases.make_case(wl, ew=ew, selection_bias=b)
        assert c.selection_bias
        plain_ids, _, _ = oracle.route(c.x64, c.wr, wl.k, wl.scale)
        assert (np.sort(plain_ids, 1) != np.sort(c.ids, 1)).any(axis=1).sum() >= wl.T // 4
        assert oracle.min_selection_gap(c.logits, b, wl.k).min() >= cases.GAP
        np.testing.assert_allclose(c.w.sum(1), wl.scale, rtol=1e-12)
