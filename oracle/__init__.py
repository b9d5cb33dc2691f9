"""CPU oracle for the routed IQ4_NL MoE layer -- TEST INFRASTRUCTURE ONLY.

A ctypes front end to ``oracle.c`` (plain C, fp64, single thread).  Only the
test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package; the product library never does, and the two share
no code.  Sources and readings are listed at the top of ``oracle.c``.

Parity status of each function (what pins it lives in tests/test_oracle.py):
  fp16_to_double, iq4nl_dequant   pinned: hand-decoded golden blocks, fp16
                                  special values, 2,064,384-byte matrix size
  iq4nl_quantize                  pinned: decode/encode round trip
  route                           pinned: hand-computed two-expert case,
                                  brute force over all subsets, sum = scale
  moe_forward                     pinned: rank-one closed form, k = 1 special
                                  case, all-experts = dense sum, permutation
                                  and token independence
  rmsnorm                         pinned: closed form on constant rows
Layer outputs at the full Xing4 shapes have no printed values on the pages:
beyond the pins above, their parity is "parity unpinned".
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (-O2, IEEE fp64, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                               "-fno-fast-math", "-ffp-contract=off",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        _lib = _configure(ctypes.CDLL(build()))
    return _lib


def _configure(lib):
    P = ctypes.c_void_p
    I = ctypes.c_int64
    D = ctypes.c_double
    lib.oracle_fp16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_fp16_to_double.restype = D
    lib.oracle_iq4nl_dequant.argtypes = [P, I, P]
    lib.oracle_iq4nl_dequant.restype = None
    lib.oracle_iq4nl_quantize.argtypes = [P, P, I, P]
    lib.oracle_iq4nl_quantize.restype = None
    lib.oracle_route.argtypes = [I, I, I, I, D, P, P, P, I, P, P, P]
    lib.oracle_route.restype = ctypes.c_int
    lib.oracle_route_selbias.argtypes = [I, I, I, I, D, P, P, P, I, P, P, P]
    lib.oracle_route_selbias.restype = ctypes.c_int
    lib.oracle_moe_forward.argtypes = [I, I, I, I, I, I, P, P, P, P, P, P, P, P, P, P]
    lib.oracle_moe_forward.restype = ctypes.c_int
    lib.oracle_rmsnorm.argtypes = [I, I, P, D, P]
    lib.oracle_rmsnorm.restype = None
    return lib


@contextlib.contextmanager
def using_library(path: str):
    """Run the oracle from another build of oracle.c (the planted-mistake
    tests compile modified copies) for the duration of a with-block."""
    global _lib
    saved = _lib
    _lib = None
    lib = ctypes.CDLL(path)
    try:
        _lib = _configure(lib)
        yield
    finally:
        _lib = saved


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def to_f64(x: np.ndarray, dtype: str) -> np.ndarray:
    """Exact widening of the layer input: 'bf16' (uint16 bits) or 'fp32'."""
    if dtype == "bf16":
        return (np.asarray(x, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    if dtype == "fp32":
        return np.asarray(x, np.float32).astype(np.float64)
    if dtype == "fp64":
        return np.asarray(x, np.float64)
    raise ValueError(dtype)


def fp16_to_double(bits: int) -> float:
    return _load().oracle_fp16_to_double(int(bits))


def iq4nl_dequant(blocks: np.ndarray) -> np.ndarray:
    """uint8 [..., n, 18] blocks -> float64 [..., 32*n] weights."""
    b = np.ascontiguousarray(blocks, dtype=np.uint8)
    assert b.shape[-1] == 18
    nb = b.size // 18
    out = np.empty(nb * 32, dtype=np.float64)
    _load().oracle_iq4nl_dequant(_p(b), nb, _p(out))
    return out.reshape(b.shape[:-2] + (b.shape[-2] * 32,))


def iq4nl_quantize(w: np.ndarray, d_bits: np.ndarray) -> np.ndarray:
    """float64 [n*32] weights + uint16 [n] fp16 scales -> uint8 [n, 18]."""
    w = np.ascontiguousarray(w, dtype=np.float64).ravel()
    d = np.ascontiguousarray(d_bits, dtype=np.uint16).ravel()
    nb = d.size
    assert w.size == nb * 32
    out = np.empty((nb, 18), dtype=np.uint8)
    _load().oracle_iq4nl_quantize(_p(w), _p(d), nb, _p(out))
    return out


def route(x: np.ndarray, wr: np.ndarray, k: int, scale: float = 2.0,
          bias: np.ndarray | None = None):
    """Sigmoid top-k router.  x float64 [T,H], wr [E,H] (any float dtype),
    bias [T,E] or [E] or None.  Returns (ids int32 [T,k], weights [T,k],
    logits [T,E])."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    wr = np.ascontiguousarray(wr, dtype=np.float64)
    T, H = x.shape
    E = wr.shape[0]
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    logits = np.empty((T, E), dtype=np.float64)
    bp, bstride = None, 0
    if bias is not None:
        bias = np.ascontiguousarray(bias, dtype=np.float64)
        bstride = E if bias.ndim == 2 else 0
        bp = _p(bias)
    rc = _load().oracle_route(T, H, E, k, float(scale), _p(x), _p(wr), bp, bstride,
                              _p(logits), _p(ids), _p(w))
    if rc != 0:
        raise ValueError(f"oracle_route: invalid sizes (rc={rc})")
    return ids, w, logits


def route_selbias(x: np.ndarray, wr: np.ndarray, k: int, scale: float, sel_bias: np.ndarray):
    """Sigmoid top-k router whose bias only steers the selection (noaux_tc):
    experts chosen by sigmoid(l) + b, weights from sigmoid(l).  sel_bias
    [T,E] or [E].  Returns (ids, weights, logits)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    wr = np.ascontiguousarray(wr, dtype=np.float64)
    T, H = x.shape
    E = wr.shape[0]
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    logits = np.empty((T, E), dtype=np.float64)
    b = np.ascontiguousarray(sel_bias, dtype=np.float64)
    rc = _load().oracle_route_selbias(T, H, E, k, float(scale), _p(x), _p(wr), _p(b),
                                      E if b.ndim == 2 else 0, _p(logits), _p(ids), _p(w))
    if rc != 0:
        raise ValueError(f"oracle_route_selbias: invalid sizes (rc={rc})")
    return ids, w, logits


def min_selection_gap(logits: np.ndarray, sel_bias: np.ndarray, k: int) -> np.ndarray:
    """Per token, the smallest gap between adjacent selection keys
    sigmoid(l) + b among the k+1 largest (fp64)."""
    s = 1.0 / (1.0 + np.exp(-np.asarray(logits, np.float64)))
    key = s + np.asarray(sel_bias, np.float64)
    kk = min(k + 1, key.shape[1])
    if kk < 2:
        return np.full(key.shape[0], np.inf)
    top = -np.sort(-key, axis=1)[:, :kk]
    return np.min(top[:, :-1] - top[:, 1:], axis=1)


def moe_forward(x: np.ndarray, ids: np.ndarray, weights: np.ndarray, ew) -> np.ndarray:
    """Layer output for given routes.  ew: an object with up/gate/down
    ([E,F,H/32,18] / [E,H,F/32,18]) and sh_up/sh_gate/sh_down arrays, or
    sh_up None for no shared expert."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    T, H = x.shape
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    w = np.ascontiguousarray(weights, dtype=np.float64)
    k = ids.shape[1] if ids.ndim == 2 else 1
    up = np.ascontiguousarray(ew.up, dtype=np.uint8)
    gate = np.ascontiguousarray(ew.gate, dtype=np.uint8)
    down = np.ascontiguousarray(ew.down, dtype=np.uint8)
    E, F = up.shape[0], up.shape[1]
    assert up.shape[2] * 32 == H and down.shape[1] == H and down.shape[2] * 32 == F
    n_shared = 0 if getattr(ew, "sh_up", None) is None else 1
    if n_shared:
        su = np.ascontiguousarray(ew.sh_up, dtype=np.uint8)
        sg = np.ascontiguousarray(ew.sh_gate, dtype=np.uint8)
        sd = np.ascontiguousarray(ew.sh_down, dtype=np.uint8)
        sp = (_p(su), _p(sg), _p(sd))
    else:
        sp = (None, None, None)
    out = np.empty((T, H), dtype=np.float64)
    rc = _load().oracle_moe_forward(T, H, E, k, F, n_shared, _p(x), _p(ids), _p(w),
                                    _p(up), _p(gate), _p(down), *sp, _p(out))
    if rc == -2:
        raise ValueError("oracle_moe_forward: expert id out of range")
    if rc != 0:
        raise ValueError(f"oracle_moe_forward: invalid sizes (rc={rc})")
    return out


def moe_layer(x: np.ndarray, wr: np.ndarray, ew, k: int, scale: float = 2.0,
              bias: np.ndarray | None = None):
    """Route then forward: returns (out [T,H] float64, ids, weights)."""
    ids, w, _ = route(x, wr, k, scale, bias)
    return moe_forward(x, ids, w, ew), ids, w


def rmsnorm(r: np.ndarray, eps: float) -> np.ndarray:
    r = np.ascontiguousarray(r, dtype=np.float64)
    T, H = r.shape
    u = np.empty_like(r)
    _load().oracle_rmsnorm(T, H, _p(r), float(eps), _p(u))
    return u


def dense_ffn(x: np.ndarray, ew) -> np.ndarray:
    """Dense FFN block [PocketLLM "Xing4.0-29B-A4B: the design record",
    section 1: the first two blocks are dense]: out[t] = W_down (silu(W_gate
    x[t]) * (W_up x[t])) with ew holding one expert (up/gate/down [1, ...])
    and no shared expert -- the layer forward with every token routed to
    expert 0 at weight 1."""
    assert ew.up.shape[0] == 1 and getattr(ew, "sh_up", None) is None
    T = np.asarray(x).shape[0]
    return moe_forward(x, np.zeros((T, 1), np.int32), np.ones((T, 1)), ew)


def min_topk_gap(logits: np.ndarray, k: int) -> np.ndarray:
    """Per token, the smallest gap between adjacent sigmoid scores among the
    k+1 largest (fp64).  The routing of a token is unambiguous when it is
    positive; inputs are drawn so that it is at least 1e-4."""
    s = 1.0 / (1.0 + np.exp(-np.asarray(logits, np.float64)))
    kk = min(k + 1, s.shape[1])
    top = -np.sort(-s, axis=1)[:, :kk]
    if kk < 2:
        return np.full(s.shape[0], np.inf)
    return np.min(top[:, :-1] - top[:, 1:], axis=1)
