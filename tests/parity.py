"""Helpers shared by the GPU parity tests: cached inputs and the tolerance.

Tolerance (stated with the workloads): routing ids bit-exact; layer outputs
within max|err| <= 2e-3 * max|ref| and sum|err| / sum|ref| <= 1e-3 against
the fp64 oracle, for fp32 outputs.  A bf16 output adds one rounding of at
most half a bf16 ulp per element on top (and run-to-run fp32 atomics may
push an element across a rounding boundary), so bf16 outputs are checked
elementwise to max(2e-3 * max|ref|, one bf16 ulp of ref) and in the mean
against the oracle rounded to bf16.
"""
from __future__ import annotations

import functools

import numpy as np

from quantized_moe_expert_sigmoid_gb300 import synth

MAX_REL = 2e-3
MEAN_REL = 1e-3


@functools.lru_cache(maxsize=4)
def weights(seed: int, layer: int, E: int, H: int, F: int, n_shared: int = 1):
    return synth.expert_weights(seed, layer, E, H, F, n_shared)


def errors(out: np.ndarray, ref: np.ndarray):
    out = np.asarray(out, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(out - ref)
    return err.max() / max(np.abs(ref).max(), 1e-300), err.sum() / max(np.abs(ref).sum(), 1e-300)


def assert_close_fp32(out, ref, what=""):
    mx, mean = errors(out, ref)
    assert mx <= MAX_REL and mean <= MEAN_REL, f"{what}: max {mx:.3e} mean {mean:.3e}"
    return mx, mean


def bf16_round(a: np.ndarray) -> np.ndarray:
    return synth.bf16_bits_to_f32(synth.to_bf16_bits(np.asarray(a, np.float32))).astype(np.float64)


def bf16_ulp(a: np.ndarray) -> np.ndarray:
    a = np.abs(np.asarray(a, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return 2.0 ** (e - 7)


def assert_close_bf16(out, ref, what=""):
    out = np.asarray(out, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(out - ref)
    bound = np.maximum(MAX_REL * np.abs(ref).max(), bf16_ulp(ref))
    assert np.all(err <= bound), f"{what}: worst excess {(err - bound).max():.3e}"
    mean = np.abs(out - bf16_round(ref)).sum() / np.abs(ref).sum()
    assert mean <= MEAN_REL, f"{what}: mean vs rounded oracle {mean:.3e}"
