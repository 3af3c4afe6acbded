"""CPU oracle of the sparse MoE FFN sublayer (ctypes wrapper of moe_oracle.c).

TEST INFRASTRUCTURE ONLY.  Only the test-suite, ``__graft_entry__.smoke()``
and the benchmark's CPU-baseline leg may import this package.  The product
library (``sparse_mixture_experts_gb300``) never does, and the two share no
code: the only common dependency is the seeded input generator ``synth``.

Every function follows the equations in ``moe_oracle.h``; all arithmetic is
double precision.  Inputs are numpy arrays of the exact stored values
(float32, or uint16 bf16 bit patterns when the layer's dtype is bf16).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_HDR = os.path.join(_HERE, "moe_oracle.h")
_LIB = os.path.join(_HERE, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None

ROUTER_MODES = {"softmax_topk": 0, "topk_softmax": 1}
ACTS = {"swiglu": 0, "clamp_glu": 1}
DTYPES = {"f32": 0, "bf16": 1}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP when available)."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= newest:
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-fPIC", "-shared", "-std=c99", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB)
    return _LIB


class _Config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("n_expert", ctypes.c_int), ("top_k", ctypes.c_int),
                ("expert_ff", ctypes.c_int), ("shared_ff", ctypes.c_int), ("router_mode", ctypes.c_int),
                ("norm_topk_prob", ctypes.c_int), ("weights_scale", ctypes.c_double), ("act", ctypes.c_int),
                ("act_alpha", ctypes.c_double), ("act_limit", ctypes.c_double), ("has_bias", ctypes.c_int),
                ("gate_up_interleaved", ctypes.c_int), ("w_dtype", ctypes.c_int), ("x_dtype", ctypes.c_int)]


_WNAMES = ("router_w", "router_b", "gate_w", "up_w", "gate_up_w", "gate_up_b", "down_w", "down_b",
           "sh_gate_w", "sh_up_w", "sh_down_w", "sh_gate_inp")


class _Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in _WNAMES]


def _get():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P, I, VP = ctypes.POINTER, ctypes.c_int, ctypes.c_void_p
            C, W = P(_Config), P(_Weights)
            lib.orc_check_config.argtypes = [C]
            lib.orc_router_logits.argtypes = [C, W, VP, I, VP, VP]
            lib.orc_select.argtypes = [C, VP, VP, VP]
            lib.orc_weights_for_selection.argtypes = [C, VP, VP, VP]
            lib.orc_expert.argtypes = [C, W, I, VP, VP, VP]
            lib.orc_shared.argtypes = [C, W, VP, VP, VP, VP]
            lib.orc_token_output.argtypes = [C, W, VP, VP, VP, VP]
            lib.orc_forward.argtypes = [C, W, VP, I, VP, I, VP, VP, VP, I]
            lib.orc_max_threads.argtypes = []
            for fn in ("orc_check_config", "orc_router_logits", "orc_select", "orc_weights_for_selection",
                       "orc_expert", "orc_shared", "orc_token_output", "orc_forward", "orc_max_threads"):
                getattr(lib, fn).restype = ctypes.c_int
            lib.orc_e2m1_value.argtypes = [ctypes.c_uint]
            lib.orc_e2m1_value.restype = ctypes.c_double
            lib.orc_e8m0_scale.argtypes = [ctypes.c_uint]
            lib.orc_e8m0_scale.restype = ctypes.c_double
            lib.orc_mxfp4_dequant.argtypes = [VP, VP, ctypes.c_int64, I, VP]
            lib.orc_mxfp4_dequant.restype = ctypes.c_int
            lib.orc_fp16_value.argtypes = [ctypes.c_uint]
            lib.orc_fp16_value.restype = ctypes.c_double
            lib.orc_q4_dequant.argtypes = [VP, ctypes.c_int64, I, VP]
            lib.orc_q4_dequant.restype = ctypes.c_int
            _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data


def e2m1_value(code: int) -> float:
    """Value of one E2M1 code (see moe_oracle.h)."""
    return _get().orc_e2m1_value(int(code))


def e8m0_scale(e: int) -> float:
    """Scale of one E8M0 byte: 2^(e - 127)."""
    return _get().orc_e8m0_scale(int(e))


def mxfp4_dequant(blocks: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """[..., cols/32, 16] uint8 blocks and [..., cols/32] uint8 scales ->
    [..., cols] float32 (exact)."""
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    if blocks.shape[-1] != 16 or blocks.shape[:-1] != scales.shape:
        raise ValueError("blocks must be [..., nb, 16] and scales [..., nb]")
    nb = scales.shape[-1]
    rows = int(np.prod(scales.shape[:-1]))
    out = np.empty(scales.shape[:-1] + (nb * 32,), dtype=np.float32)
    if _get().orc_mxfp4_dequant(_p(blocks), _p(scales), rows, nb * 32, _p(out)) != 0:
        raise ValueError("bad MXFP4 tensor")
    return out


def fp16_value(h: int) -> float:
    """Value of one binary16 bit pattern."""
    return _get().orc_fp16_value(int(h))


def q4_dequant(blocks: np.ndarray) -> np.ndarray:
    """[..., cols/32, 18] uint8 Q4 blocks -> [..., cols] float32 (exact)."""
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
    if blocks.shape[-1] != 18:
        raise ValueError("blocks must be [..., nb, 18]")
    nb = blocks.shape[-2]
    rows = int(np.prod(blocks.shape[:-2]))
    out = np.empty(blocks.shape[:-2] + (nb * 32,), dtype=np.float32)
    if _get().orc_q4_dequant(_p(blocks), rows, nb * 32, _p(out)) != 0:
        raise ValueError("bad Q4 tensor")
    return out


def _bf16_to_f32(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return (a.astype(np.uint32) << 16).view(np.float32)


def dense_weights_of_q4(weights: dict) -> dict:
    """The float32 weights a layer with Q4 expert records stands for: the
    routed experts dequantised, every bf16 tensor widened (both exact)."""
    w = {}
    for n, a in weights.items():
        if n.endswith("_q4"):
            continue
        w[n] = _bf16_to_f32(a)
    for n in ("gate_up_w", "gate_w", "up_w", "down_w"):
        if n + "_q4" in weights:
            w[n] = q4_dequant(weights[n + "_q4"])
    return w


def dense_weights_of_mxfp4(weights: dict) -> dict:
    """The float32 weights an MXFP4 layer stands for: the routed experts
    dequantised, every bf16 tensor widened (both exact)."""
    w = {}
    for n, a in weights.items():
        if n in ("gate_up_blocks", "gate_up_scales", "down_blocks", "down_scales"):
            continue
        w[n] = _bf16_to_f32(a)
    w["gate_up_w"] = mxfp4_dequant(weights["gate_up_blocks"], weights["gate_up_scales"])
    w["down_w"] = mxfp4_dequant(weights["down_blocks"], weights["down_scales"])
    return w


class Oracle:
    """One layer: a spec (synth.LayerSpec or anything with the same fields)
    and its weight arrays (dict name -> numpy array)."""

    def __init__(self, spec, weights: dict):
        self.spec = spec
        c = _Config()
        c.hidden, c.n_expert, c.top_k = spec.hidden, spec.n_expert, spec.top_k
        c.expert_ff, c.shared_ff = spec.expert_ff, spec.shared_ff
        c.router_mode = ROUTER_MODES[spec.router_mode]
        c.norm_topk_prob = int(spec.norm_topk_prob)
        c.weights_scale = float(spec.weights_scale)
        c.act = ACTS[spec.act]
        c.act_alpha, c.act_limit = float(spec.act_alpha), float(spec.act_limit)
        c.has_bias = int(spec.has_bias)
        c.gate_up_interleaved = int(spec.gate_up_interleaved)
        fmt = getattr(spec, "expert_format", "dense")
        mx = fmt in ("mxfp4", "q4")
        if fmt == "mxfp4":
            # MXFP4 experts: the layer is evaluated on its exact float32 expansion
            weights = dense_weights_of_mxfp4(weights)
        elif fmt == "q4":
            weights = dense_weights_of_q4(weights)
        c.w_dtype = DTYPES["f32" if mx else spec.dtype]
        c.x_dtype = DTYPES[spec.dtype]
        self._c = c
        self._keep = {}
        w = _Weights()
        wdt = np.float32 if mx else (np.uint16 if spec.dtype == "bf16" else np.float32)
        for n in _WNAMES:
            a = weights.get(n)
            if a is not None:
                a = np.ascontiguousarray(a)
                if a.dtype != wdt:
                    raise TypeError(f"{n}: expected {wdt} storage, got {a.dtype}")
                self._keep[n] = a
                setattr(w, n, a.ctypes.data)
        self._w = w
        self.lib = _get()
        if self.lib.orc_check_config(ctypes.byref(c)) != 0:
            raise ValueError("invalid layer configuration")

    # -- helpers ---------------------------------------------------------
    def _x(self, x):
        wdt = np.uint16 if self.spec.dtype == "bf16" else np.float32
        x = np.ascontiguousarray(x)
        if x.dtype != wdt or x.ndim != 2 or x.shape[1] != self.spec.hidden:
            raise TypeError("x must be [T, H] in the layer's storage dtype")
        return x

    def _check(self, rc, what):
        if rc != 0:
            raise RuntimeError(f"oracle {what} failed ({rc})")

    # -- API -------------------------------------------------------------
    def router_logits(self, x):
        """logits [T, E] (bias included when the layer has one) and the
        shared-gate logit [T] (zeros without a shared expert)."""
        x = self._x(x)
        T = x.shape[0]
        l = np.zeros((T, self.spec.n_expert))
        s = np.zeros(T)
        self._check(self.lib.orc_router_logits(ctypes.byref(self._c), ctypes.byref(self._w), _p(x), T, _p(l), _p(s)),
                    "router")
        return l, s

    def select(self, logits_row):
        l = np.ascontiguousarray(logits_row, dtype=np.float64)
        idx = np.zeros(self.spec.top_k, dtype=np.int32)
        wt = np.zeros(self.spec.top_k)
        self._check(self.lib.orc_select(ctypes.byref(self._c), _p(l), _p(idx), _p(wt)), "select")
        return idx, wt

    def weights_for_selection(self, logits_row, idx):
        l = np.ascontiguousarray(logits_row, dtype=np.float64)
        idx = np.ascontiguousarray(idx, dtype=np.int32)
        wt = np.zeros(self.spec.top_k)
        self._check(self.lib.orc_weights_for_selection(ctypes.byref(self._c), _p(l), _p(idx), _p(wt)), "weights")
        return wt

    def expert(self, e, x_row):
        """(h[F], y[H]) of routed expert e on one token (x_row as float64)."""
        xr = np.ascontiguousarray(x_row, dtype=np.float64)
        h = np.zeros(self.spec.expert_ff)
        y = np.zeros(self.spec.hidden)
        self._check(self.lib.orc_expert(ctypes.byref(self._c), ctypes.byref(self._w), int(e), _p(xr), _p(h), _p(y)),
                    "expert")
        return h, y

    def shared(self, x_row):
        """(h[Fs], y[H] ungated, gate sigmoid) of the shared expert."""
        xr = np.ascontiguousarray(x_row, dtype=np.float64)
        h = np.zeros(self.spec.shared_ff)
        y = np.zeros(self.spec.hidden)
        g = np.zeros(1)
        self._check(self.lib.orc_shared(ctypes.byref(self._c), ctypes.byref(self._w), _p(xr), _p(h), _p(y), _p(g)),
                    "shared")
        return h, y, float(g[0])

    def token_output(self, x_row, idx, wt):
        xr = np.ascontiguousarray(x_row, dtype=np.float64)
        idx = np.ascontiguousarray(idx, dtype=np.int32)
        wt = np.ascontiguousarray(wt, dtype=np.float64)
        out = np.zeros(self.spec.hidden)
        self._check(self.lib.orc_token_output(ctypes.byref(self._c), ctypes.byref(self._w), _p(xr), _p(idx), _p(wt),
                                              _p(out)), "token_output")
        return out

    def forward(self, x, rows=None, n_threads: int = 0):
        """out [R, H] (float64), idx [R, k], wt [R, k] for the listed token
        rows of x (all rows when rows is None)."""
        x = self._x(x)
        T = x.shape[0]
        r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
        R = T if r is None else len(r)
        out = np.zeros((R, self.spec.hidden))
        idx = np.zeros((R, self.spec.top_k), dtype=np.int32)
        wt = np.zeros((R, self.spec.top_k))
        rc = self.lib.orc_forward(ctypes.byref(self._c), ctypes.byref(self._w), _p(x), T, _p(r), R, _p(out), _p(idx),
                                  _p(wt), int(n_threads))
        self._check(rc, "forward")
        return out, idx, wt


def max_threads() -> int:
    return int(_get().orc_max_threads())
