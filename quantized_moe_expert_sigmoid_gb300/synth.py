"""Seeded synthetic inputs for the routed IQ4_NL MoE layer.

This module only draws random numbers and lays them out in the storage
formats the layer consumes.  It holds none of the layer's arithmetic (no
dequantisation, no router, no FFN): the CUDA path and the CPU oracle both
take its arrays as inputs, and neither is used here.

Every value comes from SplitMix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014), evaluated on a counter, so any
row of any tensor can be regenerated on its own and the streams are identical
on every machine (the arithmetic is plain uint64 wrap-around).

Workload recipes follow the synthetic layer shapes of the Xing4.0-29B-A4B
design record (PocketLLM, section 1 "The shape of the thing": 64 routed
experts top-4, one shared expert, expert_ffn 1,024, hidden 3,584, sigmoid
router, routed_scaling_factor 2.0) and the IQ4_NL storage described on the
HelloSun/xing4_0-29b-IQ4_NL_EPQ model card ("模型與路由" and "權重組成":
4.5 bpw, 18-byte blocks of 32 weights, 2,064,384 B per expert matrix).
"""
from __future__ import annotations

import dataclasses
import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

QK = 32            # weights per IQ4_NL block
BLOCK_BYTES = 18   # fp16 scale + 16 bytes of 4-bit indices


def _mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function on a uint64 array (wrap-around arithmetic)."""
    with np.errstate(over="ignore"):
        z = z.astype(np.uint64, copy=True)
        z ^= z >> np.uint64(30)
        z *= _M1
        z ^= z >> np.uint64(27)
        z *= _M2
        z ^= z >> np.uint64(31)
    return z


def _tag_hash(tag: str) -> int:
    """FNV-1a over the tag's bytes: names a stream."""
    h = 0xCBF29CE484222325
    for b in tag.encode():
        h ^= b
        h = (h * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    return h


def stream_key(seed: int, tag: str, *ints: int) -> np.uint64:
    """64-bit key of the stream named by (seed, tag, ints...)."""
    k = np.array([(seed * 0xD1B54A32D192ED03 + _tag_hash(tag)) & 0xFFFFFFFFFFFFFFFF],
                 dtype=np.uint64)
    for i in ints:
        with np.errstate(over="ignore"):
            k = _mix(k ^ np.uint64(i & 0xFFFFFFFFFFFFFFFF)) + _GOLDEN
    return k[0]


def u64(key, n: int, start: int = 0) -> np.ndarray:
    """n consecutive SplitMix64 outputs of stream `key` from counter `start`."""
    with np.errstate(over="ignore"):
        c = np.arange(start, start + n, dtype=np.uint64)
        return _mix(np.uint64(key) + c * _GOLDEN)


def uniform(key, n: int, start: int = 0) -> np.ndarray:
    """U[0,1) doubles from the top 53 bits."""
    return (u64(key, n, start) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal(key, n: int, start: int = 0) -> np.ndarray:
    """N(0,1) doubles by the Box-Muller transform on pairs of uniforms."""
    m = (n + 1) // 2
    u = uniform(key, 2 * m, 2 * start)
    u1 = 1.0 - u[0::2]          # (0, 1]
    u2 = u[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    z = np.empty(2 * m)
    z[0::2] = r * np.cos(2.0 * np.pi * u2)
    z[1::2] = r * np.sin(2.0 * np.pi * u2)
    return z[:n]


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float values to bfloat16 (round-to-nearest-even); returns uint16 bits."""
    f = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    with np.errstate(over="ignore"):
        r = f + np.uint32(0x7FFF) + ((f >> np.uint32(16)) & np.uint32(1))
    return (r >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bits to float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# --------------------------------------------------------------------------
# IQ4_NL weight blocks
# --------------------------------------------------------------------------

def iq4nl_blocks(seed: int, tag: str, rows: int, cols: int, *ids: int,
                 d_lo: float = 5e-4, d_hi: float = 2e-3) -> np.ndarray:
    """Random IQ4_NL matrix [rows x cols] stored as uint8 [rows, cols/32, 18].

    Each block is a little-endian fp16 scale d ~ U[d_lo, d_hi] (rounded to
    fp32 then to fp16, nearest-even each time) followed by 16 bytes whose 32
    nibbles are uniform on 0..15.  Uniform random bytes give uniform nibbles in both halves, so this
    generator does not depend on the order of the nibbles inside a block.
    """
    assert cols % QK == 0
    nb = rows * (cols // QK)
    kd = stream_key(seed, tag + "/d", *ids)
    kq = stream_key(seed, tag + "/q", *ids)
    d = (d_lo + (d_hi - d_lo) * uniform(kd, nb)).astype(np.float32).astype(np.float16)
    q = u64(kq, 2 * nb).view(np.uint8).reshape(nb, 16)
    out = np.empty((nb, BLOCK_BYTES), dtype=np.uint8)
    out[:, 0:2] = d.view(np.uint8).reshape(nb, 2)
    out[:, 2:] = q
    return out.reshape(rows, cols // QK, BLOCK_BYTES)


@dataclasses.dataclass
class ExpertWeights:
    """IQ4_NL weights of one layer: E routed experts plus the shared one."""
    up: np.ndarray       # [E, F, H/32, 18]
    gate: np.ndarray     # [E, F, H/32, 18]
    down: np.ndarray     # [E, H, F/32, 18]
    sh_up: np.ndarray    # [F, H/32, 18]
    sh_gate: np.ndarray
    sh_down: np.ndarray  # [H, F/32, 18]


def expert_weights(seed: int, layer: int, E: int, H: int, F: int,
                   n_shared: int = 1) -> ExpertWeights:
    """Weights of layer `layer`: expert e's matrices are streams (layer, e)."""
    up = np.stack([iq4nl_blocks(seed, "up", F, H, layer, e) for e in range(E)])
    gate = np.stack([iq4nl_blocks(seed, "gate", F, H, layer, e) for e in range(E)])
    down = np.stack([iq4nl_blocks(seed, "down", H, F, layer, e) for e in range(E)])
    if n_shared:
        s_up = iq4nl_blocks(seed, "sh_up", F, H, layer)
        s_gate = iq4nl_blocks(seed, "sh_gate", F, H, layer)
        s_down = iq4nl_blocks(seed, "sh_down", H, F, layer)
    else:
        s_up = np.zeros((F, H // QK, BLOCK_BYTES), np.uint8)
        s_gate = np.zeros_like(s_up)
        s_down = np.zeros((H, F // QK, BLOCK_BYTES), np.uint8)
    return ExpertWeights(up, gate, down, s_up, s_gate, s_down)


def dense_ffn_weights(seed: int, layer: int, H: int, F: int) -> ExpertWeights:
    """A dense FFN block's IQ4_NL matrices as a one-expert layer with no
    shared expert (streams of their own, distinct from any expert's)."""
    up = iq4nl_blocks(seed, "dense/up", F, H, layer)[None]
    gate = iq4nl_blocks(seed, "dense/gate", F, H, layer)[None]
    down = iq4nl_blocks(seed, "dense/down", H, F, layer)[None]
    return ExpertWeights(up, gate, down, None, None, None)


def expert_subset_weights(seed: int, layer: int, experts, H: int, F: int,
                          n_shared: int = 1) -> ExpertWeights:
    """The matrices of the routed experts `experts` (in that order) of layer
    `layer`, plus the shared expert: the same bytes as expert_weights(...)
    for those experts, without drawing the others."""
    ids = [int(e) for e in experts]
    up = np.stack([iq4nl_blocks(seed, "up", F, H, layer, e) for e in ids])
    gate = np.stack([iq4nl_blocks(seed, "gate", F, H, layer, e) for e in ids])
    down = np.stack([iq4nl_blocks(seed, "down", H, F, layer, e) for e in ids])
    if n_shared:
        s_up = iq4nl_blocks(seed, "sh_up", F, H, layer)
        s_gate = iq4nl_blocks(seed, "sh_gate", F, H, layer)
        s_down = iq4nl_blocks(seed, "sh_down", H, F, layer)
    else:
        s_up = np.zeros((F, H // QK, BLOCK_BYTES), np.uint8)
        s_gate = np.zeros_like(s_up)
        s_down = np.zeros((H, F // QK, BLOCK_BYTES), np.uint8)
    return ExpertWeights(up, gate, down, s_up, s_gate, s_down)


# --------------------------------------------------------------------------
# Activations, router weights, logit bias
# --------------------------------------------------------------------------

def activations(seed: int, tag: str, T: int, H: int, attempts=None,
                dtype: str = "bf16", layer: int = 0) -> np.ndarray:
    """x ~ N(0,1) [T x H]; row t is stream (layer, t, attempts[t]).

    `attempts` lets a caller redraw single rows (for example to keep routing
    free of near-ties) without changing the others.  Returns uint16 bf16 bits
    for dtype 'bf16' and float32 for 'fp32'.
    """
    if attempts is None:
        attempts = np.zeros(T, dtype=np.int64)
    rows = np.empty((T, H), dtype=np.float64)
    for t in range(T):
        rows[t] = normal(stream_key(seed, tag, layer, t, int(attempts[t])), H)
    if dtype == "bf16":
        return to_bf16_bits(rows)
    if dtype == "fp32":
        return rows.astype(np.float32)
    raise ValueError(dtype)


def router_weights(seed: int, layer: int, E: int, H: int, sigma: float) -> np.ndarray:
    """Router matrix Wr [E x H] fp32 ~ N(0, sigma^2)."""
    return (sigma * normal(stream_key(seed, "router", layer), E * H)).astype(np.float32).reshape(E, H)


ZIPF_S = 1.1
ZIPF_BETA = 0.3


def zipf_logit_bias(seed: int, T: int, E: int, s: float = ZIPF_S,
                    beta: float = ZIPF_BETA) -> np.ndarray:
    """Per-token Zipf(s) bias over expert ids, [T x E] fp32.

    Expert e gets rank pi(e) from a seeded permutation and prior
    p_e = (pi(e)+1)^-s / sum_r (r+1)^-s.  Token t's bias is
    b[t,e] = beta * ln(E * p_e) + beta * g[t,e] with g ~ N(0,1)/4, a fixed
    Zipf-shaped preference plus per-token jitter.  beta is a constant of the
    recipe, chosen once so that the per-expert loads of the 4,096-token
    workload spread over roughly 64..1,000 routes.
    """
    rank = np.argsort(u64(stream_key(seed, "zipf/perm"), E), kind="stable")
    pi = np.empty(E, dtype=np.int64)
    pi[rank] = np.arange(E)
    p = (pi + 1.0) ** (-s)
    p /= p.sum()
    base = beta * np.log(E * p)
    jit = normal(stream_key(seed, "zipf/jitter"), T * E).reshape(T, E) * 0.25
    return (base[None, :] + beta * jit).astype(np.float32)


def selection_bias(seed: int, E: int, T: int | None = None, sigma: float = 0.1) -> np.ndarray:
    """Per-expert selection bias (the noaux_tc probability bias): N(0, sigma)
    values, [E] fp32, or [T x E] when T is given (one row per token).  Scores
    are sigmoid outputs in (0, 1), so sigma 0.1 reorders a good share of the
    close candidates without overriding the router."""
    shape = (E,) if T is None else (T, E)
    tag = "selbias" if T is None else "selbias/rows"
    return (normal(stream_key(seed, tag, E), int(np.prod(shape))).reshape(shape) * sigma).astype(np.float32)


# --------------------------------------------------------------------------
# Workloads
# --------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    H: int
    E: int
    k: int
    F: int
    T: int
    x_dtype: str        # 'bf16' or 'fp32'
    router_sigma: float
    zipf: bool = False
    n_layers: int = 1
    n_shared: int = 1
    scale: float = 2.0


WORKLOADS = {
    "tiny": Workload("tiny: H256 E8 top-2 F128, 4 tokens, fp32 x", 256, 8, 2, 128, 4, "fp32", 0.05),
    "decode1": Workload("Xing4 MoE layer, decode batch 1 (H3584 E64 top-4 F1024)", 3584, 64, 4, 1024, 1, "bf16", 0.02),
    "decode8": Workload("Xing4 MoE layer, batched decode 8 tokens", 3584, 64, 4, 1024, 8, "bf16", 0.02),
    "decode64": Workload("Xing4 MoE layer, batched decode 64 tokens", 3584, 64, 4, 1024, 64, "bf16", 0.02),
    "prefill4096": Workload("Xing4 MoE layer, prefill 4,096 tokens, Zipf-skewed routing", 3584, 64, 4, 1024, 4096, "bf16", 0.02, zipf=True),
    "trunk38_t1": Workload("38-layer Xing4 MoE trunk, batch 1", 3584, 64, 4, 1024, 1, "bf16", 0.02, n_layers=38),
    "trunk38_t16": Workload("38-layer Xing4 MoE trunk, batch 16", 3584, 64, 4, 1024, 16, "bf16", 0.02, n_layers=38),
    # the K2-Horizon FFN router: 8 of 100 routed experts + 1 shared, weights
    # normalised and scaled by 2.5, hidden 2,560.  The expert width is not
    # given: 10.00 GiB for 4,500 expert groups at IQ3_XS's ~3.3 bits per
    # weight is ~5.8 M weights = 3 x 2,560 x ~750 per expert; 768 is taken.
    "k2h_decode1": Workload("K2-Horizon-shaped MoE layer, decode batch 1 (H2560 E100 top-8 F768, x2.5)",
                            2560, 100, 8, 768, 1, "bf16", 0.024, scale=2.5),
    "k2h_decode64": Workload("K2-Horizon-shaped MoE layer, batched decode 64 tokens",
                             2560, 100, 8, 768, 64, "bf16", 0.024, scale=2.5),
    "k2h_prefill1024": Workload("K2-Horizon-shaped MoE layer, prefill 1,024 tokens",
                                2560, 100, 8, 768, 1024, "bf16", 0.024, scale=2.5),
}


# --------------------------------------------------------------------------
# The same weight streams drawn on a torch device (bit-identical to the
# numpy functions above; used to fill many layers quickly)
# --------------------------------------------------------------------------

def _s64(v: int) -> int:
    v &= 0xFFFFFFFFFFFFFFFF
    return v - (1 << 64) if v >= (1 << 63) else v


def _mix_t(z):
    """SplitMix64 output function on an int64 tensor (wrap-around, logical shifts)."""
    z = z ^ ((z >> 30) & ((1 << 34) - 1))
    z = z * _s64(int(_M1))
    z = z ^ ((z >> 27) & ((1 << 37) - 1))
    z = z * _s64(int(_M2))
    z = z ^ ((z >> 31) & ((1 << 33) - 1))
    return z


def u64_torch(key, n: int, device, start: int = 0):
    import torch
    c = torch.arange(start, start + n, dtype=torch.int64, device=device)
    return _mix_t(c * _s64(int(_GOLDEN)) + _s64(int(key)))


def uniform_torch(key, n: int, device, start: int = 0):
    import torch
    u = (u64_torch(key, n, device, start) >> 11) & ((1 << 53) - 1)
    return u.to(torch.float64) * (2.0 ** -53)


def iq4nl_blocks_torch(seed: int, tag: str, rows: int, cols: int, *ids: int, device="cuda",
                       d_lo: float = 5e-4, d_hi: float = 2e-3):
    """Same bytes as iq4nl_blocks, as a uint8 tensor on `device`."""
    import torch
    assert cols % QK == 0
    nb = rows * (cols // QK)
    kd = stream_key(seed, tag + "/d", *ids)
    kq = stream_key(seed, tag + "/q", *ids)
    d = (d_lo + (d_hi - d_lo) * uniform_torch(kd, nb, device)).to(torch.float32).to(torch.float16)
    q = u64_torch(kq, 2 * nb, device).view(torch.uint8).reshape(nb, 16)
    out = torch.empty((nb, BLOCK_BYTES), dtype=torch.uint8, device=device)
    out[:, 0:2] = d.view(torch.uint8).reshape(nb, 2)
    out[:, 2:] = q
    return out.reshape(rows, cols // QK, BLOCK_BYTES)


def expert_weights_torch(seed: int, layer: int, E: int, H: int, F: int, n_shared: int = 1,
                         device="cuda") -> ExpertWeights:
    """expert_weights(...) drawn directly on `device` (torch uint8 tensors)."""
    import torch
    up = torch.stack([iq4nl_blocks_torch(seed, "up", F, H, layer, e, device=device) for e in range(E)])
    gate = torch.stack([iq4nl_blocks_torch(seed, "gate", F, H, layer, e, device=device) for e in range(E)])
    down = torch.stack([iq4nl_blocks_torch(seed, "down", H, F, layer, e, device=device) for e in range(E)])
    if n_shared:
        su = iq4nl_blocks_torch(seed, "sh_up", F, H, layer, device=device)
        sg = iq4nl_blocks_torch(seed, "sh_gate", F, H, layer, device=device)
        sd = iq4nl_blocks_torch(seed, "sh_down", H, F, layer, device=device)
    else:
        su = sg = sd = None
    return ExpertWeights(up, gate, down, su, sg, sd)
