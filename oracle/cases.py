"""Seeded parity cases -- TEST INFRASTRUCTURE ONLY.

Draws a workload's inputs with the product-independent generator
(``quantized_moe_expert_sigmoid_gb300.synth``) and redraws any token whose
routing would be ambiguous: a token is kept only when, among its k+1 largest
selection keys (fp64, from this oracle's router: the sigmoid scores, or with
a selection-only bias the scores plus that bias), adjacent keys differ by at
least ``GAP``.  That keeps the selected set and its order unique, so a
kernel computing the logits in fp32 must return the same ids bit for bit.
"""
from __future__ import annotations

import dataclasses
import numpy as np

from quantized_moe_expert_sigmoid_gb300 import synth
from . import route, route_selbias, to_f64, min_topk_gap, min_selection_gap

GAP = 1e-4


@dataclasses.dataclass
class Case:
    wl: synth.Workload
    x: np.ndarray          # bf16 bits (uint16) or fp32, [T, H]
    x64: np.ndarray        # the same values in fp64
    wr: np.ndarray         # fp32 [E, H]
    bias: np.ndarray | None  # fp32 [T, E] or [E], or None
    ew: synth.ExpertWeights
    ids: np.ndarray        # oracle routes, int32 [T, k]
    w: np.ndarray          # oracle weights, fp64 [T, k]
    logits: np.ndarray     # fp64 [T, E]
    attempts: np.ndarray
    selection_bias: bool = False  # bias ranks experts only (noaux_tc)


def draw_routed_inputs(wl: synth.Workload, wr: np.ndarray, seed: int = 0,
                       layer: int = 0, T: int | None = None,
                       bias: np.ndarray | None = None, tag: str = "x",
                       max_rounds: int = 64, selection_bias: bool = False):
    """x for T tokens with every token's top-k+1 selection keys >= GAP apart.
    selection_bias: bias ([T, E] or [E]) is the noaux_tc selection bias."""
    T = wl.T if T is None else T
    attempts = np.zeros(T, dtype=np.int64)
    x = synth.activations(seed, tag, T, wl.H, attempts, wl.x_dtype, layer)
    x64 = to_f64(x, wl.x_dtype)

    def rows_bias(rows):
        if bias is None or bias.ndim == 1 or rows is None:
            return bias
        return bias[rows]

    def do_route(xr, rows=None):
        b = rows_bias(rows)
        if selection_bias:
            return route_selbias(xr, wr, wl.k, wl.scale, np.zeros(wr.shape[0]) if b is None else b)
        return route(xr, wr, wl.k, wl.scale, b)

    def gaps(logits, rows=None):
        if selection_bias:
            b = rows_bias(rows)
            return min_selection_gap(logits, 0.0 if b is None else b, wl.k)
        return min_topk_gap(logits, wl.k)

    ids, w, logits = do_route(x64)
    for _ in range(max_rounds):
        bad = np.nonzero(gaps(logits, np.arange(T)) < GAP)[0]
        if bad.size == 0:
            return x, x64, ids, w, logits, attempts
        attempts[bad] += 1
        # regenerate only the ambiguous rows
        xb = np.stack([_row(seed, tag, wl, layer, int(t), int(attempts[t])) for t in bad])
        x[bad] = xb
        x64[bad] = to_f64(xb, wl.x_dtype)
        i2, w2, l2 = do_route(x64[bad], bad)
        ids[bad], w[bad], logits[bad] = i2, w2, l2
    raise RuntimeError("could not draw tie-free routing inputs")


def _row(seed, tag, wl, layer, t, attempt):
    """Row t of the activation stream at the given attempt."""
    key = synth.stream_key(seed, tag, layer, t, attempt)
    v = synth.normal(key, wl.H)
    return synth.to_bf16_bits(v) if wl.x_dtype == "bf16" else v.astype(np.float32)


def make_case(wl: synth.Workload | str, seed: int = 0, layer: int = 0,
              T: int | None = None, ew: synth.ExpertWeights | None = None,
              selection_bias: np.ndarray | None = None) -> Case:
    """selection_bias ([T, E] or [E]): route with that noaux_tc selection
    bias instead of the workload's logit bias."""
    if isinstance(wl, str):
        wl = synth.WORKLOADS[wl]
    T = wl.T if T is None else T
    wr = synth.router_weights(seed, layer, wl.E, wl.H, wl.router_sigma)
    sel = selection_bias is not None
    if sel:
        bias = np.asarray(selection_bias, np.float32)
    else:
        bias = synth.zipf_logit_bias(seed, T, wl.E) if wl.zipf else None
    if ew is None:
        ew = synth.expert_weights(seed, layer, wl.E, wl.H, wl.F, wl.n_shared)
    x, x64, ids, w, logits, att = draw_routed_inputs(wl, wr, seed, layer, T, bias,
                                                     selection_bias=sel)
    return Case(wl, x, x64, wr, bias, ew, ids, w, logits, att, sel)
