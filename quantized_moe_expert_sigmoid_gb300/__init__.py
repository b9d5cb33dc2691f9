"""GB300-native routed IQ4_NL Mixture-of-Experts layer with a sigmoid router.

A thin ctypes binding over libmoe_gb300.so (include/moe_gb300.h).  The
functions below have the C entry points' names and only marshal arguments:
torch tensors on the GPU become device pointers, the current torch CUDA
stream becomes the stream argument, and a non-OK status raises MoeError.
Every step of the layer runs in the library's CUDA kernels; there is no
other implementation to fall back to, and importing the library fails
loudly when it has not been built.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB as _LIB_PATH

MOE_OK = 0
MOE_DT_BF16 = 0
MOE_DT_FP32 = 1
MOE_FLAG_SELECTION_BIAS = 1  # the bias ranks experts only (noaux_tc); weights stay unbiased
MOE_FLAG_DETERMINISTIC = 2   # slot-ordered combine: equal inputs give equal output bits
MOE_FLAG_HOST_IO = 4         # device copy buffers for moe_layer_forward_routed_host
MOE_FLAG_COOPERATIVE = 8     # cooperative launches for the single-launch decode kernels

STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED_SHAPE",
          3: "MOE_ERR_MISALIGNED", 4: "MOE_ERR_OUT_OF_MEMORY", 5: "MOE_ERR_CUDA",
          6: "MOE_ERR_TIMEOUT", 7: "MOE_ERR_BAD_EXPERT_ID", 8: "MOE_ERR_TOO_MANY_TOKENS",
          9: "MOE_ERR_OVERFLOW"}

EXPORTS = ["moe_layer_create", "moe_layer_destroy", "moe_route", "moe_forward",
           "moe_layer_forward_routed", "moe_residual_rmsnorm", "moe_layer_check",
           "moe_layer_weight_bytes", "moe_launch_count", "moe_status_string", "moe_last_error",
           "moe_route_noalloc", "moe_dense_forward", "moe_layer_forward_routed_resid"]


class MoeError(RuntimeError):
    def __init__(self, status: int, detail: str):
        self.status = status
        self.name = STATUS.get(status, f"status {status}")
        super().__init__(f"{self.name}: {detail}")


class _Shapes(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("expert_ffn", ctypes.c_int32),
                ("n_shared", ctypes.c_int32), ("routed_scaling", ctypes.c_float),
                ("max_tokens", ctypes.c_int32), ("flags", ctypes.c_uint32)]


class _Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("up", "gate", "down", "sh_up", "sh_gate", "sh_down")]


_lib = None


def library_path() -> str:
    return _LIB_PATH


def load_library(path: str | None = None):
    """Load libmoe_gb300.so (built by build.build()); raises if it is absent."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or _LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"libmoe_gb300.so is not built ({path}); run "
                           "quantized_moe_expert_sigmoid_gb300.build.build() first")
    lib = ctypes.CDLL(path)
    P, I32, I64, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    lib.moe_layer_create.argtypes = [ctypes.POINTER(_Shapes), ctypes.POINTER(_Weights), P,
                                     ctypes.POINTER(P)]
    lib.moe_layer_destroy.argtypes = [P]
    lib.moe_route.argtypes = [P, P, I32, I32, P, P, I64, P, P, P]
    lib.moe_forward.argtypes = [P, P, I32, I32, P, P, P, I32, P]
    lib.moe_dense_forward.argtypes = [P, P, I32, I32, P, I32, P]
    lib.moe_layer_forward_routed.argtypes = [P, P, I32, I32, P, P, I64, P, P, P, I32, P]
    lib.moe_layer_forward_routed_host.argtypes = [P, P, I32, I32, P, P, I64, P, P, P, I32, P]
    lib.moe_residual_rmsnorm.argtypes = [P, P, I32, P, I32, I32, F, P]
    lib.moe_layer_forward_routed_resid.argtypes = [P, P, P, I32, P, P, F, I32, P, P, I64, P, P, P, I32, P]
    lib.moe_layer_check.argtypes = [P]
    lib.moe_layer_weight_bytes.argtypes = [P]
    lib.moe_layer_weight_bytes.restype = I64
    lib.moe_route_noalloc.argtypes = [P, I32, I32, I32, I32, I32, F, P, P, I64, P, P, P]
    lib.moe_route_noalloc.restype = I32
    lib.moe_launch_count.argtypes = []
    lib.moe_launch_count.restype = I64
    lib.moe_status_string.argtypes = [I32]
    lib.moe_status_string.restype = ctypes.c_char_p
    lib.moe_last_error.argtypes = []
    lib.moe_last_error.restype = ctypes.c_char_p
    lib.moe_layer_enable_timing.argtypes = [P, I32]
    lib.moe_test_barrier_slack.argtypes = [P, I32]
    lib.moe_layer_stage_times.argtypes = [P, P, I32, ctypes.POINTER(I32)]
    for n in ("moe_layer_create", "moe_layer_destroy", "moe_route", "moe_forward",
              "moe_layer_forward_routed", "moe_residual_rmsnorm", "moe_layer_check",
              "moe_layer_enable_timing", "moe_layer_stage_times", "moe_dense_forward",
              "moe_test_barrier_slack", "moe_layer_forward_routed_host", "moe_layer_forward_routed_resid"):
        getattr(lib, n).restype = I32
    _lib = lib
    return lib


def _check(status: int):
    if status != MOE_OK:
        raise MoeError(status, load_library().moe_last_error().decode(errors="replace"))


def _ptr(t, name="tensor", dtypes=None):
    """Device pointer of a dense tensor; the C ABI takes dense row-major
    arrays, so a strided view or a wrong dtype is refused here."""
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous (row-major); got strides {tuple(t.stride())}")
    if dtypes is not None and t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}; expected one of {dtypes}")
    if t.numel() and not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    return ctypes.c_void_p(t.data_ptr())


_DT = None


def _dt():
    global _DT
    if _DT is None:  # (built once: the marshalling runs on every call)
        import torch
        _DT = {"x": (torch.bfloat16, torch.float32), "f32": (torch.float32,),
               "i32": (torch.int32,), "u8": (torch.uint8,)}
    return _DT


def _dtype(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return MOE_DT_BF16
    if t.dtype == torch.float32:
        return MOE_DT_FP32
    raise TypeError(f"unsupported dtype {t.dtype}: bf16 or fp32")


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


# ---------------------------------------------------------------------------
# Entry points (same names as the C ABI)
# ---------------------------------------------------------------------------

def moe_layer_create(hidden, n_experts, top_k, expert_ffn, n_shared, routed_scaling,
                     max_tokens, up, gate, down, sh_up=None, sh_gate=None, sh_down=None,
                     stream=None, flags=0):
    """Returns an opaque handle (int).  Weight tensors: uint8 on the GPU in
    the IQ4_NL block layout of include/moe_gb300.h; flags: MOE_FLAG_* bits."""
    lib = load_library()
    sh = _Shapes(hidden, n_experts, top_k, expert_ffn, n_shared, routed_scaling, max_tokens, flags)
    w = _Weights(*(_ptr(t, n, _dt()["u8"]) for t, n in ((up, "up"), (gate, "gate"), (down, "down"),
                                                         (sh_up, "sh_up"), (sh_gate, "sh_gate"),
                                                         (sh_down, "sh_down"))))
    out = ctypes.c_void_p()
    _check(lib.moe_layer_create(ctypes.byref(sh), ctypes.byref(w), _stream(stream), ctypes.byref(out)))
    return out.value


def moe_layer_destroy(layer):
    _check(load_library().moe_layer_destroy(ctypes.c_void_p(layer)))


def moe_route(layer, x, router_w, ids, weights, logit_bias=None, bias_row_stride=None,
              stream=None):
    if bias_row_stride is None:
        bias_row_stride = 0 if logit_bias is None or logit_bias.dim() == 1 else logit_bias.stride(0)
    d = _dt()
    if logit_bias is not None and logit_bias.dim() == 2 and logit_bias.stride(1) == 1 \
            and bias_row_stride == logit_bias.stride(0):
        bias_p = ctypes.c_void_p(logit_bias.data_ptr())  # row-strided [T][E] view is allowed
    else:
        bias_p = _ptr(logit_bias, "logit_bias", d["f32"])
    _check(load_library().moe_route(ctypes.c_void_p(layer), _ptr(x, "x", d["x"]), _dtype(x),
                                    x.shape[0], _ptr(router_w, "router_w", d["f32"]), bias_p,
                                    bias_row_stride, _ptr(ids, "ids", d["i32"]),
                                    _ptr(weights, "weights", d["f32"]), _stream(stream)))


def moe_forward(layer, x, ids, weights, out, stream=None):
    d = _dt()
    _check(load_library().moe_forward(ctypes.c_void_p(layer), _ptr(x, "x", d["x"]), _dtype(x),
                                      x.shape[0], _ptr(ids, "ids", d["i32"]),
                                      _ptr(weights, "weights", d["f32"]), _ptr(out, "out", d["x"]),
                                      _dtype(out), _stream(stream)))


def moe_dense_forward(layer, x, out, stream=None):
    d = _dt()
    _check(load_library().moe_dense_forward(ctypes.c_void_p(layer), _ptr(x, "x", d["x"]), _dtype(x),
                                            x.shape[0], _ptr(out, "out", d["x"]), _dtype(out),
                                            _stream(stream)))


def moe_layer_forward_routed(layer, x, router_w, ids, weights, out, logit_bias=None,
                             bias_row_stride=None, stream=None):
    if bias_row_stride is None:
        bias_row_stride = 0 if logit_bias is None or logit_bias.dim() == 1 else logit_bias.stride(0)
    d = _dt()
    if logit_bias is not None and logit_bias.dim() == 2 and logit_bias.stride(1) == 1 \
            and bias_row_stride == logit_bias.stride(0):
        bias_p = ctypes.c_void_p(logit_bias.data_ptr())
    else:
        bias_p = _ptr(logit_bias, "logit_bias", d["f32"])
    _check(load_library().moe_layer_forward_routed(
        ctypes.c_void_p(layer), _ptr(x, "x", d["x"]), _dtype(x), x.shape[0],
        _ptr(router_w, "router_w", d["f32"]), bias_p, bias_row_stride,
        _ptr(ids, "ids", d["i32"]), _ptr(weights, "weights", d["f32"]), _ptr(out, "out", d["x"]),
        _dtype(out), _stream(stream)))


def moe_layer_forward_routed_resid(layer, resid_in, delta, resid_out, u_out, eps, router_w, ids, weights, out,
                                   logit_bias=None, stream=None):
    T = resid_in.shape[0]
    d = _dt()
    ddt = MOE_DT_FP32 if delta is None else _dtype(delta)
    bias_stride = 0 if logit_bias is None or logit_bias.dim() == 1 else logit_bias.stride(0)
    _check(load_library().moe_layer_forward_routed_resid(
        ctypes.c_void_p(layer), _ptr(resid_in, "resid_in", d["f32"]), _ptr(delta, "delta", d["x"]), ddt,
        _ptr(resid_out, "resid_out", d["f32"]), _ptr(u_out, "u_out", (d["x"][0],)), float(eps), T,
        _ptr(router_w, "router_w", d["f32"]), _ptr(logit_bias, "logit_bias", d["f32"]), bias_stride,
        _ptr(ids, "ids", d["i32"]), _ptr(weights, "weights", d["f32"]), _ptr(out, "out", d["x"]),
        _dtype(out), _stream(stream)))


def _host_ptr(t, name, dtypes):
    """Host pointer of a dense CPU tensor (page-locked for asynchronous copies)."""
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous (row-major); got strides {tuple(t.stride())}")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}; expected one of {dtypes}")
    if t.is_cuda:
        raise ValueError(f"{name} must be in host memory")
    return ctypes.c_void_p(t.data_ptr())


def moe_layer_forward_routed_host(layer, x_host, router_w, ids, weights, out_host, logit_bias=None,
                                  bias_row_stride=None, stream=None):
    """moe_layer_forward_routed with x and out in host memory (pinned CPU
    tensors), for a layer created with MOE_FLAG_HOST_IO: the copies in and
    out are enqueued on the stream with the layer call; out_host is written
    once the stream has passed the call."""
    if bias_row_stride is None:
        bias_row_stride = 0 if logit_bias is None or logit_bias.dim() == 1 else logit_bias.stride(0)
    d = _dt()
    if logit_bias is not None and logit_bias.dim() == 2 and logit_bias.stride(1) == 1 \
            and bias_row_stride == logit_bias.stride(0):
        bias_p = ctypes.c_void_p(logit_bias.data_ptr())
    else:
        bias_p = _ptr(logit_bias, "logit_bias", d["f32"])
    _check(load_library().moe_layer_forward_routed_host(
        ctypes.c_void_p(layer), _host_ptr(x_host, "x_host", d["x"]), _dtype(x_host), x_host.shape[0],
        _ptr(router_w, "router_w", d["f32"]), bias_p, bias_row_stride,
        _ptr(ids, "ids", d["i32"]), _ptr(weights, "weights", d["f32"]),
        _host_ptr(out_host, "out_host", d["x"]), _dtype(out_host), _stream(stream)))


def moe_route_noalloc(x, router_w, ids, weights, top_k, routed_scaling=2.0, logit_bias=None,
                      bias_row_stride=None, stream=None):
    """moe_route without a layer and without any device allocation: the
    logits scratch is a fixed array inside the library (T * n_experts <=
    262,144).  For callers that may not allocate device memory; the first
    call on a device should come before any stream capture, and calls that
    overlap on the GPU share (and race on) the one scratch array."""
    if bias_row_stride is None:
        bias_row_stride = 0 if logit_bias is None or logit_bias.dim() == 1 else logit_bias.stride(0)
    d = _dt()
    if logit_bias is not None and logit_bias.dim() == 2 and logit_bias.stride(1) == 1 \
            and bias_row_stride == logit_bias.stride(0):
        bias_p = ctypes.c_void_p(logit_bias.data_ptr())
    else:
        bias_p = _ptr(logit_bias, "logit_bias", d["f32"])
    T, H = x.shape
    E = router_w.shape[0]
    _check(load_library().moe_route_noalloc(
        _ptr(x, "x", d["x"]), _dtype(x), T, H, E, top_k, float(routed_scaling),
        _ptr(router_w, "router_w", d["f32"]), bias_p, bias_row_stride,
        _ptr(ids, "ids", d["i32"]), _ptr(weights, "weights", d["f32"]), _stream(stream)))


def moe_residual_rmsnorm(resid, delta, u, eps, stream=None):
    T, H = resid.shape
    ddt = MOE_DT_FP32 if delta is None else _dtype(delta)
    d = _dt()
    _check(load_library().moe_residual_rmsnorm(_ptr(resid, "resid", d["f32"]),
                                               _ptr(delta, "delta", d["x"]), ddt,
                                               _ptr(u, "u", (d["x"][0],)), T, H,
                                               float(eps), _stream(stream)))


def moe_layer_check(layer):
    _check(load_library().moe_layer_check(ctypes.c_void_p(layer)))


def moe_layer_enable_timing(layer, calls: int):
    """Record per-stage CUDA events for the next calls on the layer (a ring of
    `calls` slots; 0 disables)."""
    _check(load_library().moe_layer_enable_timing(ctypes.c_void_p(layer), int(calls)))


def moe_test_barrier_slack(layer, slack: int):
    """Test hook: slack 1 makes the single-launch decode kernel's h wait run
    out (the call then reports MOE_ERR_TIMEOUT through moe_layer_check);
    0 restores normal calls."""
    _check(load_library().moe_test_barrier_slack(ctypes.c_void_p(layer), int(slack)))


STAGES = ("route+plan+gather", "up/gate", "down", "combine")


def moe_layer_stage_times(layer, max_calls: int):
    """Per-stage milliseconds of the recorded calls, oldest first: a list of
    4-tuples in the order of STAGES."""
    import numpy as np
    ms = np.zeros((max(1, max_calls), 4), np.float32)
    n = ctypes.c_int32(0)
    _check(load_library().moe_layer_stage_times(ctypes.c_void_p(layer),
                                                ms.ctypes.data_as(ctypes.c_void_p),
                                                int(max_calls), ctypes.byref(n)))
    return [tuple(float(v) for v in row) for row in ms[:n.value]]


def moe_layer_weight_bytes(layer) -> int:
    return int(load_library().moe_layer_weight_bytes(ctypes.c_void_p(layer)))


def moe_launch_count() -> int:
    return int(load_library().moe_launch_count())


def moe_status_string(status: int) -> str:
    return load_library().moe_status_string(status).decode()


def moe_last_error() -> str:
    return load_library().moe_last_error().decode(errors="replace")


class MoeLayer:
    """Owns one layer handle; keeps nothing else alive (the library copied
    the weights).  Methods are the entry points with the handle bound."""

    def __init__(self, hidden, n_experts, top_k, expert_ffn, n_shared=1, routed_scaling=2.0,
                 max_tokens=1, *, up, gate, down, sh_up=None, sh_gate=None, sh_down=None,
                 stream=None, flags=0):
        self.H, self.E, self.k, self.F, self.S = hidden, n_experts, top_k, expert_ffn, n_shared
        self.scale, self.max_tokens, self.flags = routed_scaling, max_tokens, flags
        self.handle = moe_layer_create(hidden, n_experts, top_k, expert_ffn, n_shared,
                                       routed_scaling, max_tokens, up, gate, down, sh_up,
                                       sh_gate, sh_down, stream, flags)

    @classmethod
    def from_weights(cls, ew, k, scale=2.0, max_tokens=1, device="cuda", stream=None, flags=0):
        """Upload synth.ExpertWeights-like numpy arrays and create the layer."""
        import torch
        t = lambda a: None if a is None else torch.from_numpy(a).to(device)
        E, F, nbh = ew.up.shape[0], ew.up.shape[1], ew.up.shape[2]
        H = nbh * 32
        S = 0 if getattr(ew, "sh_up", None) is None else 1
        return cls(H, E, k, F, S, scale, max_tokens, up=t(ew.up), gate=t(ew.gate), down=t(ew.down),
                   sh_up=t(ew.sh_up) if S else None, sh_gate=t(ew.sh_gate) if S else None,
                   sh_down=t(ew.sh_down) if S else None, stream=stream, flags=flags)

    def route(self, x, router_w, logit_bias=None, stream=None):
        import torch
        T = x.shape[0]
        ids = torch.empty((T, self.k), dtype=torch.int32, device=x.device)
        w = torch.empty((T, self.k), dtype=torch.float32, device=x.device)
        moe_route(self.handle, x, router_w, ids, w, logit_bias, stream=stream)
        return ids, w

    def forward(self, x, ids, weights, out_dtype=None, stream=None):
        import torch
        out = torch.empty((x.shape[0], self.H), dtype=out_dtype or x.dtype, device=x.device)
        moe_forward(self.handle, x, ids, weights, out, stream=stream)
        return out

    def dense_forward(self, x, out_dtype=None, stream=None):
        """The FFN of a dense block (a layer of one expert, top-1) on every token."""
        import torch
        out = torch.empty((x.shape[0], self.H), dtype=out_dtype or x.dtype, device=x.device)
        moe_dense_forward(self.handle, x, out, stream=stream)
        return out

    def forward_routed(self, x, router_w, logit_bias=None, out_dtype=None, stream=None):
        import torch
        T = x.shape[0]
        ids = torch.empty((T, self.k), dtype=torch.int32, device=x.device)
        w = torch.empty((T, self.k), dtype=torch.float32, device=x.device)
        out = torch.empty((T, self.H), dtype=out_dtype or x.dtype, device=x.device)
        moe_layer_forward_routed(self.handle, x, router_w, ids, w, out, logit_bias, stream=stream)
        return out, ids, w

    def check(self):
        moe_layer_check(self.handle)

    def weight_bytes(self):
        return moe_layer_weight_bytes(self.handle)

    def close(self):
        if self.handle:
            moe_layer_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class MoeTrunk:
    """A stack of MoE layers on an fp32 residual stream (the 38-layer trunk
    of the Xing4.0-29B-A4B model card, MoE blocks only):
        r_0 = x,  u_l = bf16(r_l / sqrt(mean(r_l^2) + eps)),  r_{l+1} = r_l + MoE_l(u_l).
    Per layer one moe_layer_forward_routed_resid call: the residual update,
    the RMSNorm and the layer (at one token a single launch of the one-token
    kernel; otherwise a residual-RMSNorm launch and the layer's launches).
    The residual alternates between two buffers (a step reads one and writes
    the other); layer outputs are fp32.  Every tensor it uses is preallocated
    at construction, so forward() can be captured in a CUDA graph."""

    def __init__(self, layers, routers, max_tokens, eps=1e-6, device="cuda"):
        import torch
        assert len(layers) == len(routers) and layers
        self.layers, self.routers, self.eps = list(layers), list(routers), float(eps)
        H, k = layers[0].H, layers[0].k
        n = len(layers)
        self.rbuf = [torch.empty((max_tokens, H), dtype=torch.float32, device=device) for _ in range(2)]
        self.u = [torch.empty((max_tokens, H), dtype=torch.bfloat16, device=device) for _ in range(n)]
        self.out = [torch.empty((max_tokens, H), dtype=torch.float32, device=device) for _ in range(n)]
        self.ids = [torch.empty((max_tokens, k), dtype=torch.int32, device=device) for _ in range(n)]
        self.w = [torch.empty((max_tokens, k), dtype=torch.float32, device=device) for _ in range(n)]
        self.u_final = torch.empty((max_tokens, H), dtype=torch.bfloat16, device=device)

    def forward(self, x, stream=None):
        """x: fp32 or bf16 [T, H] on the device.  Returns the final residual
        r_L [T, H] fp32 (a view of one of the trunk's buffers); the per-layer
        u, out, ids and w stay readable in self.u / self.out / self.ids /
        self.w."""
        T = x.shape[0]
        cur = 0
        self.rbuf[0][:T].copy_(x)
        prev = None
        for l, (L, wr) in enumerate(zip(self.layers, self.routers)):
            r_in, r_out = self.rbuf[cur][:T], self.rbuf[1 - cur][:T]
            moe_layer_forward_routed_resid(L.handle, r_in, prev, r_out, self.u[l][:T], self.eps, wr,
                                           self.ids[l][:T], self.w[l][:T], self.out[l][:T], stream=stream)
            prev = self.out[l][:T]
            cur = 1 - cur
        r = self.rbuf[cur][:T]
        moe_residual_rmsnorm(r, prev, self.u_final[:T], self.eps, stream=stream)  # r_L = r_{L-1} + out
        return r

    def check(self):
        for L in self.layers:
            L.check()
