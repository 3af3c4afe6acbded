"""Seeded synthetic inputs for the sparse MoE FFN layer.

This module is shared by the oracle's tests and by the CUDA path's tests and
benchmark.  It only *draws* numbers (weights, biases, activations) and
describes layer shapes; it contains none of the layer's arithmetic.

Recipe (the pages publish no weights; all inputs are synthetic):

* every weight matrix ~ N(0, 1/fan_in) (the second parameter read as the
  variance), fan_in = H for router / gate / up / shared-gate vector, F (or Fs)
  for the down projections;
* biases ~ N(0, 0.02) (variance), i.e. std sqrt(0.02);
* activations x ~ N(0, 1);
* ``router_init="uniform"``: router rows ~ U(-a, a) with a = sqrt(3/H) (same
  variance as the normal case);
* ``router_init="zipf"``: expert load skewed as Zipf(s) over a seeded
  permutation of the experts: with p_r proportional to r^-s, a seeded unit
  vector u and alpha = 8, router row e = G_e + (ln p_e / alpha) u and token
  x_t = z_t + alpha u, so logit_e ~ ln p_e + N(0, ~1): top-k then behaves like
  drawing k experts without replacement from the Zipf law.
* bf16 tensors are rounded to nearest-even once; both sides read those values.

The generator is counter-based (SplitMix64 hash + Box-Muller, ``synth.c``), so
value i of a tensor does not depend on chunking or threads, and token row t of
x is the same for every token count.
"""
from __future__ import annotations

import ctypes
import dataclasses
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile synth.c into libsynth.so next to it (gcc, OpenMP if present)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-fPIC", "-shared", "-std=c99", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB)
    return _LIB


def _get():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u64, i64, dbl, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
            for name in ("synth_normal_f32", "synth_normal_bf16", "synth_uniform_f32", "synth_uniform_bf16"):
                fn = getattr(lib, name)
                fn.argtypes = [u64, u64, u64, i64, dbl, dbl, vp]
                fn.restype = None
            lib.synth_u64.argtypes = [u64, u64, u64, i64, vp]
            lib.synth_u64.restype = None
            lib.synth_f32_to_bf16.argtypes = [vp, i64, vp]
            lib.synth_f32_to_bf16.restype = None
            lib.synth_bf16_to_f32.argtypes = [vp, i64, vp]
            lib.synth_bf16_to_f32.restype = None
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def normal(shape, std: float, seed: int, stream: int, dtype: str, offset: int = 0, mean: float = 0.0) -> np.ndarray:
    n = int(np.prod(shape))
    if dtype == "bf16":
        out = np.empty(shape, dtype=np.uint16)
        _get().synth_normal_bf16(seed, stream, offset, n, mean, std, _ptr(out))
    else:
        out = np.empty(shape, dtype=np.float32)
        _get().synth_normal_f32(seed, stream, offset, n, mean, std, _ptr(out))
    return out


def uniform(shape, lo: float, hi: float, seed: int, stream: int, dtype: str, offset: int = 0) -> np.ndarray:
    n = int(np.prod(shape))
    if dtype == "bf16":
        out = np.empty(shape, dtype=np.uint16)
        _get().synth_uniform_bf16(seed, stream, offset, n, lo, hi, _ptr(out))
    else:
        out = np.empty(shape, dtype=np.float32)
        _get().synth_uniform_f32(seed, stream, offset, n, lo, hi, _ptr(out))
    return out


def u64(n: int, seed: int, stream: int, offset: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    _get().synth_u64(seed, stream, offset, n, _ptr(out))
    return out


def to_bf16(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    out = np.empty(a.shape, dtype=np.uint16)
    _get().synth_f32_to_bf16(_ptr(a), a.size, _ptr(out))
    return out


def bf16_to_f32(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.uint16)
    out = np.empty(a.shape, dtype=np.float32)
    _get().synth_bf16_to_f32(_ptr(a), a.size, _ptr(out))
    return out


def as_f32(a: np.ndarray, dtype: str) -> np.ndarray:
    """The exact stored values of an f32 or bf16 tensor as float32."""
    return bf16_to_f32(a) if dtype == "bf16" else a


# ----------------------------------------------------------------------------
# layer shapes
# ----------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class LayerSpec:
    name: str
    hidden: int
    n_expert: int
    top_k: int
    expert_ff: int
    shared_ff: int = 0
    router_mode: str = "softmax_topk"      # or "topk_softmax" (gpt-oss)
    norm_topk_prob: bool = True
    weights_scale: float = 1.0
    act: str = "swiglu"                    # or "clamp_glu" (gpt-oss)
    act_alpha: float = 1.702
    act_limit: float = 7.0
    has_bias: bool = False
    gate_up_interleaved: bool = False
    dtype: str = "bf16"                    # weights and activations: "f32" / "bf16"
    router_init: str = "normal"            # "normal" / "uniform" / "zipf"
    zipf_s: float = 1.1
    expert_format: str = "dense"           # "dense" (dtype), "mxfp4" or "q4" (routed experts; rest bf16)
    resident_experts: int = 0              # layer option (not an input): device slots for routed experts

    def replace(self, **kw) -> "LayerSpec":
        return dataclasses.replace(self, **kw)


TINY = LayerSpec("tiny-f32 (H=64, E=8, top-2, F=32)", 64, 8, 2, 32, dtype="f32")
QWEN = LayerSpec("qwen35moe-shaped (H=2048, E=256, top-8, F=512, shared 512)", 2048, 256, 8, 512, shared_ff=512)
QWEN_ZIPF = QWEN.replace(name="qwen35moe-shaped, Zipf s=1.1 expert load (H=2048, E=256, top-8, F=512, shared 512)",
                         router_init="zipf")
GPTOSS = LayerSpec("gpt-oss-20b-shaped (H=2880, E=32, top-4, F=2880, biases, clamped GLU)", 2880, 32, 4, 2880,
                   router_mode="topk_softmax", act="clamp_glu", has_bias=True, gate_up_interleaved=True)
MIXTRAL = LayerSpec("mixtral-shaped (H=4096, E=8, top-2, F=14336)", 4096, 8, 2, 14336, router_init="uniform")
GPTOSS_MXFP4 = GPTOSS.replace(name="gpt-oss-20b-shaped, MXFP4 experts (H=2880, E=32, top-4, F=2880, biases)",
                              expert_format="mxfp4")

QWEN_Q4 = QWEN.replace(name="qwen35moe-shaped routed experts, Q4 records (H=2048, E=256, top-8, F=512)",
                       shared_ff=0, expert_format="q4")
GPTOSS_Q4 = GPTOSS.replace(name="gpt-oss-20b-shaped, Q4 expert records (H=2880, E=32, top-4, F=2880, biases)",
                           expert_format="q4")

QWEN_STREAMED = QWEN.replace(name="qwen35moe-shaped, 128 of 256 experts resident, the rest streamed from host memory",
                             resident_experts=128)

# workload -> token counts exercised
WORKLOADS = {
    "tiny": (TINY, (16,)),
    "qwen_decode": (QWEN, (1, 4, 8)),
    "qwen_prefill_zipf": (QWEN_ZIPF, (4096,)),
    "gptoss": (GPTOSS, (1, 64, 2048)),
    "mixtral": (MIXTRAL, (1, 16, 256, 4096, 16384)),
    "gptoss_mxfp4": (GPTOSS_MXFP4, (1, 4, 16, 64)),
    "qwen_q4": (QWEN_Q4, (1, 8, 300)),
    "gptoss_q4": (GPTOSS_Q4, (1, 16, 2048)),
}

# stream ids, one per tensor
_S = dict(router_w=1, router_b=2, gate_w=3, up_w=4, gate_up_w=5, gate_up_b=6, down_w=7, down_b=8,
          sh_gate_w=9, sh_up_w=10, sh_down_w=11, sh_gate_inp=12, zipf_perm=20, zipf_dir=21,
          gate_up_blocks=30, gate_up_scales=31, down_blocks=32, down_scales=33,
          gate_up_q4=40, gate_q4=41, up_q4=42, down_q4=43, q4_scales=44, x=100)
_ZIPF_ALPHA = 8.0
_BIAS_STD = math.sqrt(0.02)


def _zipf_parts(spec: LayerSpec, seed: int):
    """Seeded expert permutation -> log p_e, and the unit direction u."""
    E, H = spec.n_expert, spec.hidden
    keys = u64(E, seed, _S["zipf_perm"])
    order = np.argsort(keys, kind="stable")          # rank r of expert order[r]
    p = np.arange(1, E + 1, dtype=np.float64) ** (-spec.zipf_s)
    p /= p.sum()
    logp = np.empty(E, dtype=np.float64)
    logp[order] = np.log(p)
    u = normal((H,), 1.0, seed, _S["zipf_dir"], "f32").astype(np.float64)
    u /= np.linalg.norm(u)
    return logp, u


def _mxfp4(rows_shape, cols: int, seed: int, blocks_stream: int, scales_stream: int):
    """MXFP4 tensor [*rows_shape][cols]: blocks [..][cols/32][16] of uniformly
    drawn bytes (every E2M1 code equally likely) and one E8M0 scale per block
    drawn from {119, 120, 121}: |code value| has RMS 2.93, so the values have
    RMS near 1/sqrt(cols) for cols around 2880, like the dense layers."""
    nb = cols // 32
    n_rows = int(np.prod(rows_shape))
    raw = u64((n_rows * nb * 16 + 7) // 8, seed, blocks_stream)
    blocks = raw.view(np.uint8)[: n_rows * nb * 16].reshape(tuple(rows_shape) + (nb, 16)).copy()
    sc = u64(n_rows * nb, seed, scales_stream)
    scales = (119 + (sc % np.uint64(3))).astype(np.uint8).reshape(tuple(rows_shape) + (nb,))
    return blocks, scales


def _q4(rows_shape, cols: int, seed: int, stream: int):
    """Q4 records [*rows_shape][cols/32][18]: per block a binary16 scale d
    (little-endian) and 16 bytes of uniformly drawn 4-bit codes.  The codes
    minus 8 have RMS 4.64, so d = 2^u / (4.64 sqrt(cols)) with u uniform in
    [-0.5, 0.5) per block gives values of RMS near 1/sqrt(cols), like the
    dense layers."""
    nb = cols // 32
    n = int(np.prod(rows_shape)) * nb
    raw = u64((n * 16 + 7) // 8, seed, stream)
    codes = raw.view(np.uint8)[: n * 16].reshape(n, 16)
    u = (u64(n, seed, _S["q4_scales"] * 1000 + stream) >> np.uint64(11)).astype(np.float64) / float(1 << 53)
    d = (np.exp2(u - 0.5) / (4.64 * math.sqrt(cols))).astype(np.float16).view(np.uint16)
    out = np.empty((n, 18), dtype=np.uint8)
    out[:, 0] = (d & 0xFF).astype(np.uint8)
    out[:, 1] = (d >> 8).astype(np.uint8)
    out[:, 2:] = codes
    return out.reshape(tuple(rows_shape) + (nb, 18))


def make_weights(spec: LayerSpec, seed: int = 0) -> dict:
    """All weight/bias tensors of one layer as numpy arrays (float32, or
    uint16 bf16 bit patterns when spec.dtype == "bf16").  With
    expert_format == "mxfp4" the routed experts come as MXFP4 blocks and
    scales (uint8): gate_up_blocks [E][2F][H/32][16] (rows interleaved gate,
    up), gate_up_scales [E][2F][H/32], down_blocks [E][H][F/32][16],
    down_scales [E][H][F/32]; router, biases and activations stay bf16."""
    H, E, F, Fs, dt = spec.hidden, spec.n_expert, spec.expert_ff, spec.shared_ff, spec.dtype
    w = {}
    if spec.expert_format == "mxfp4":
        if dt != "bf16" or not spec.gate_up_interleaved or Fs or H % 32 or F % 32:
            raise ValueError("mxfp4 layers: bf16, interleaved gate_up, no shared expert, H and F multiples of 32")
    if spec.expert_format == "q4":
        if dt != "bf16" or Fs or H % 32 or F % 32:
            raise ValueError("q4 layers: bf16, no shared expert, H and F multiples of 32")
    if spec.router_init == "uniform":
        a = math.sqrt(3.0 / H)
        w["router_w"] = uniform((E, H), -a, a, seed, _S["router_w"], dt)
    elif spec.router_init == "zipf":
        g = normal((E, H), 1.0 / math.sqrt(H), seed, _S["router_w"], "f32").astype(np.float64)
        logp, u = _zipf_parts(spec, seed)
        r = (g + (logp / _ZIPF_ALPHA)[:, None] * u[None, :]).astype(np.float32)
        w["router_w"] = to_bf16(r) if dt == "bf16" else r
    else:
        w["router_w"] = normal((E, H), 1.0 / math.sqrt(H), seed, _S["router_w"], dt)
    if spec.has_bias:
        w["router_b"] = normal((E,), _BIAS_STD, seed, _S["router_b"], dt)
        w["gate_up_b"] = normal((E, 2 * F), _BIAS_STD, seed, _S["gate_up_b"], dt)
        w["down_b"] = normal((E, H), _BIAS_STD, seed, _S["down_b"], dt)
    if spec.expert_format == "mxfp4":
        w["gate_up_blocks"], w["gate_up_scales"] = _mxfp4((E, 2 * F), H, seed, _S["gate_up_blocks"],
                                                          _S["gate_up_scales"])
        w["down_blocks"], w["down_scales"] = _mxfp4((E, H), F, seed, _S["down_blocks"], _S["down_scales"])
        return w
    if spec.expert_format == "q4":
        if spec.gate_up_interleaved:
            w["gate_up_w_q4"] = _q4((E, 2 * F), H, seed, _S["gate_up_q4"])
        else:
            w["gate_w_q4"] = _q4((E, F), H, seed, _S["gate_q4"])
            w["up_w_q4"] = _q4((E, F), H, seed, _S["up_q4"])
        w["down_w_q4"] = _q4((E, H), F, seed, _S["down_q4"])
        return w
    if spec.gate_up_interleaved:
        w["gate_up_w"] = normal((E, 2 * F, H), 1.0 / math.sqrt(H), seed, _S["gate_up_w"], dt)
    else:
        w["gate_w"] = normal((E, F, H), 1.0 / math.sqrt(H), seed, _S["gate_w"], dt)
        w["up_w"] = normal((E, F, H), 1.0 / math.sqrt(H), seed, _S["up_w"], dt)
    w["down_w"] = normal((E, H, F), 1.0 / math.sqrt(F), seed, _S["down_w"], dt)
    if Fs > 0:
        w["sh_gate_w"] = normal((Fs, H), 1.0 / math.sqrt(H), seed, _S["sh_gate_w"], dt)
        w["sh_up_w"] = normal((Fs, H), 1.0 / math.sqrt(H), seed, _S["sh_up_w"], dt)
        w["sh_down_w"] = normal((H, Fs), 1.0 / math.sqrt(Fs), seed, _S["sh_down_w"], dt)
        w["sh_gate_inp"] = normal((H,), 1.0 / math.sqrt(H), seed, _S["sh_gate_inp"], dt)
    return w


def make_x(spec: LayerSpec, n_tokens: int, seed: int = 0, first_token: int = 0) -> np.ndarray:
    """Token activations [n_tokens, H]; row t is token first_token + t of the
    seeded stream (the same values whatever n_tokens is)."""
    H = spec.hidden
    off = first_token * H
    if spec.router_init == "zipf":
        z = normal((n_tokens, H), 1.0, seed, _S["x"], "f32", offset=off).astype(np.float64)
        _, u = _zipf_parts(spec, seed)
        x = (z + _ZIPF_ALPHA * u[None, :]).astype(np.float32)
        return to_bf16(x) if spec.dtype == "bf16" else x
    return normal((n_tokens, H), 1.0, seed, _S["x"], spec.dtype, offset=off)


def weight_bytes_per_expert(spec: LayerSpec) -> int:
    """Bytes of one routed expert's weights (and biases) as stored."""
    if spec.expert_format == "mxfp4":
        n = 3 * spec.hidden * spec.expert_ff  # codes: half a byte each; a scale byte per 32
        return n // 2 + n // 32 + (2 * spec.expert_ff + spec.hidden) * 2
    if spec.expert_format == "q4":
        n = 3 * spec.hidden * spec.expert_ff  # 18 bytes per 32 elements
        return n // 32 * 18 + ((2 * spec.expert_ff + spec.hidden) * 2 if spec.has_bias else 0)
    el = 2 if spec.dtype == "bf16" else 4
    n = 3 * spec.hidden * spec.expert_ff
    if spec.has_bias:
        n += 2 * spec.expert_ff + spec.hidden
    return n * el
