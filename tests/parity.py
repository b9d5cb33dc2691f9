"""Helpers shared by the GPU parity tests: cached inputs, the tolerance and
the full-size oracle reference.

Tolerance (stated with the workloads): routing ids bit-exact; layer outputs
within max|err| <= 2e-3 * max|ref| and sum|err| / sum|ref| <= 1e-3 against
the fp64 oracle, for fp32 outputs.  A bf16 output is that fp32 sum rounded
once to nearest, which moves an element by at most half a bf16 ulp of the
rounded value, so bf16 outputs are checked elementwise to
2e-3 * max|ref| + 0.5 ulp(out) and in the mean against the oracle rounded
to bf16.

Every parity test compares every output element with the oracle.  The
oracle is single-threaded C; for the large batches its tokens are split
into contiguous chunks run on all host cores at once (ctypes releases the
interpreter lock during the call).  A token's output does not depend on the
other tokens of its batch -- tests/test_oracle.py pins that -- so the
chunked result is the oracle's own.
"""
from __future__ import annotations

import concurrent.futures as cf
import functools
import os

import numpy as np

import oracle
from quantized_moe_expert_sigmoid_gb300 import synth

MAX_REL = 2e-3
MEAN_REL = 1e-3


@functools.lru_cache(maxsize=4)
def weights(seed: int, layer: int, E: int, H: int, F: int, n_shared: int = 1):
    return synth.expert_weights(seed, layer, E, H, F, n_shared)


def host_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


_REF = {}


def oracle_ready():
    """Build and load the oracle library before threads call into it."""
    oracle.build()
    oracle.fp16_to_double(0)


def oracle_forward(x64, ids, w, ew, key=None):
    """oracle.moe_forward over every token of the batch, the tokens split
    into one contiguous chunk per host thread.  `key` (hashable) memoises
    the result for tests that share inputs."""
    if key is not None and key in _REF:
        return _REF[key]
    x64 = np.asarray(x64, np.float64)
    ids = np.asarray(ids, np.int32)
    w = np.asarray(w, np.float64)
    T = x64.shape[0]
    n = max(1, min(host_threads(), T // 4))
    oracle_ready()
    if n == 1:
        out = oracle.moe_forward(x64, ids, w, ew)
    else:
        chunks = [c for c in np.array_split(np.arange(T), n) if c.size]
        with cf.ThreadPoolExecutor(len(chunks)) as ex:
            parts = list(ex.map(lambda c: oracle.moe_forward(x64[c], ids[c], w[c], ew), chunks))
        out = np.concatenate(parts, axis=0)
    if key is not None:
        if len(_REF) >= 8:
            _REF.pop(next(iter(_REF)))
        _REF[key] = out
    return out


def errors(out: np.ndarray, ref: np.ndarray):
    out = np.asarray(out, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(out - ref)
    return err.max() / max(np.abs(ref).max(), 1e-300), err.sum() / max(np.abs(ref).sum(), 1e-300)


def assert_close_fp32(out, ref, what=""):
    assert np.shape(out) == np.shape(ref), f"{what}: shape {np.shape(out)} vs {np.shape(ref)}"
    mx, mean = errors(out, ref)
    assert mx <= MAX_REL and mean <= MEAN_REL, f"{what}: max {mx:.3e} mean {mean:.3e}"
    return mx, mean


def bf16_round(a: np.ndarray) -> np.ndarray:
    return synth.bf16_bits_to_f32(synth.to_bf16_bits(np.asarray(a, np.float32))).astype(np.float64)


def bf16_ulp(a: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at |a| (8 significant bits)."""
    a = np.abs(np.asarray(a, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return 2.0 ** (e - 7)


def assert_close_bf16(out, ref, what=""):
    out = np.asarray(out, np.float64)
    ref = np.asarray(ref, np.float64)
    assert out.shape == ref.shape, f"{what}: shape {out.shape} vs {ref.shape}"
    err = np.abs(out - ref)
    bound = MAX_REL * np.abs(ref).max() + 0.5 * bf16_ulp(out)
    assert np.all(err <= bound), f"{what}: worst excess {(err - bound).max():.3e}"
    mean = np.abs(out - bf16_round(ref)).sum() / np.abs(ref).sum()
    assert mean <= MEAN_REL, f"{what}: mean vs rounded oracle {mean:.3e}"


def oracle_dense(x64, ew):
    """oracle.dense_ffn over every token, chunked over the host cores like
    oracle_forward."""
    x64 = np.asarray(x64, np.float64)
    T = x64.shape[0]
    n = max(1, min(host_threads(), T // 4))
    oracle_ready()
    chunks = [c for c in np.array_split(np.arange(T), n) if c.size]
    with cf.ThreadPoolExecutor(len(chunks)) as ex:
        parts = list(ex.map(lambda c: oracle.dense_ffn(x64[c], ew), chunks))
    return np.concatenate(parts, axis=0)
