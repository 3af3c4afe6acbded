"""Python binding of libmoe, the GB300 (sm_103a) sparse-MoE FFN layer.

Argument marshalling only: every step of the layer runs in the CUDA kernels of
``libmoe.so`` behind the C ABI in ``include/moe.h``.  PyTorch supplies device
memory and streams.  There is no CPU or PyTorch fallback: if the library is
not built, importing the binding works but creating a layer raises.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import sys
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

# moe_status
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_OOM, ERR_CUDA, ERR_TOO_MANY_TOKENS, ERR_DEVICE_TIMEOUT = 0, -1, -2, -3, -4, -5, -6
_STATUS_NAMES = {0: "OK", -1: "INVALID_ARG", -2: "UNSUPPORTED", -3: "OOM", -4: "CUDA", -5: "TOO_MANY_TOKENS",
                 -6: "DEVICE_TIMEOUT"}
DT_F32, DT_BF16, DT_MXFP4, DT_Q4 = 0, 1, 2, 3
ROUTER_SOFTMAX_TOPK, ROUTER_TOPK_SOFTMAX = 0, 1
ACT_SWIGLU, ACT_CLAMP_GLU = 0, 1
PATH_AUTO, PATH_STREAM, PATH_TC, PATH_FUSED, PATH_DECODE_TC = 0, 1, 2, 3, 4
INTER_OFFSETS, INTER_PERM, INTER_H, INTER_YS = 0, 1, 2, 3
KERNEL_KINDS = ("router", "select", "group", "up", "down", "combine", "gather", "fused", "experts",
                "experts_mxfp4", "experts_q4", "residency")

_DT = {"f32": DT_F32, "bf16": DT_BF16}
_TORCH_DT = {DT_F32: torch.float32, DT_BF16: torch.bfloat16}


class MoEError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class _Config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("n_expert", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("expert_ff", ctypes.c_int32), ("shared_ff", ctypes.c_int32), ("router_mode", ctypes.c_int32),
                ("norm_topk_prob", ctypes.c_int32), ("weights_scale", ctypes.c_float), ("act", ctypes.c_int32),
                ("act_alpha", ctypes.c_float), ("act_limit", ctypes.c_float), ("has_bias", ctypes.c_int32),
                ("gate_up_interleaved", ctypes.c_int32), ("w_dtype", ctypes.c_int32), ("act_dtype", ctypes.c_int32),
                ("out_dtype", ctypes.c_int32), ("max_tokens", ctypes.c_int32), ("resident_experts", ctypes.c_int32)]


WEIGHT_NAMES = ("router_w", "router_b", "gate_w", "up_w", "gate_up_w", "gate_up_b", "down_w", "down_b",
                "sh_gate_w", "sh_up_w", "sh_down_w", "sh_gate_inp", "gate_up_scales", "down_scales")


class _Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in WEIGHT_NAMES]


_lib = None


def load_library(path: str = LIB_PATH):
    """Load libmoe.so and declare its signatures (raises if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libmoe.so is not built ({path}); run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    P, VP, I32 = ctypes.POINTER, ctypes.c_void_p, ctypes.c_int32
    sigs = {
        "moe_layer_create": ([P(_Config), P(_Weights), P(VP)], ctypes.c_int),
        "moe_forward": ([VP, VP, I32, VP, VP], ctypes.c_int),
        "moe_forward_host": ([VP, VP, I32, VP, VP], ctypes.c_int),
        "moe_get_routing": ([VP, VP, VP, VP], ctypes.c_int),
        "moe_get_logits": ([VP, VP, VP, VP], ctypes.c_int),
        "moe_get_expert_counts": ([VP, VP, VP], ctypes.c_int),
        "moe_set_path": ([VP, I32], ctypes.c_int),
        "moe_get_status": ([VP], ctypes.c_int),
        "moe_timing_enable": ([VP, I32], ctypes.c_int),
        "moe_timing_read": ([VP, VP, VP], ctypes.c_int),
        "moe_last_launch_count": ([VP], I32),
        "moe_last_token_count": ([VP], I32),
        "moe_device_bytes": ([VP], ctypes.c_size_t),
        "moe_destroy": ([VP], None),
        "moe_last_error": ([], ctypes.c_char_p),
        "moe_abi_version": ([], I32),
        "moe_route_noalloc": ([VP, VP, VP, I32, I32, I32, I32, I32, I32, ctypes.c_float, I32, VP, VP, VP, VP],
                              ctypes.c_int),
        "moe_get_intermediate": ([VP, I32, VP, ctypes.c_size_t, P(ctypes.c_size_t), VP], ctypes.c_int),
        "moe_set_wait_limit": ([VP, ctypes.c_int64], ctypes.c_int),
        "moe_set_fault_injection": ([VP, I32], ctypes.c_int),
        "moe_get_residency": ([VP, VP, VP], ctypes.c_int),
        "moe_ep_send_plan": ([I32, I32, VP, VP, VP, VP], ctypes.c_int),
        "moe_ep_recv_plan": ([I32, I32, VP, VP, VP, VP, VP], ctypes.c_int),
    }
    for name, (args, res) in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def _check(rc: int):
    if rc != OK:
        raise MoEError(rc, _lib.moe_last_error().decode(errors="replace"))


@dataclasses.dataclass
class MoEConfig:
    hidden: int
    n_expert: int
    top_k: int
    expert_ff: int
    shared_ff: int = 0
    router_mode: int = ROUTER_SOFTMAX_TOPK
    norm_topk_prob: bool = True
    weights_scale: float = 1.0
    act: int = ACT_SWIGLU
    act_alpha: float = 1.702
    act_limit: float = 7.0
    has_bias: bool = False
    gate_up_interleaved: bool = False
    w_dtype: int = DT_BF16
    act_dtype: int = DT_BF16
    out_dtype: int = DT_F32
    max_tokens: int = 1
    resident_experts: int = 0  # 0: every routed expert in device memory; else slots (see include/moe.h)

    def _c(self) -> _Config:
        c = _Config()
        for f in _Config._fields_:
            setattr(c, f[0], type(getattr(c, f[0]))(getattr(self, f[0])))
        return c


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


class MoELayer:
    """A created layer.  ``weights`` maps the names in ``WEIGHT_NAMES`` to
    tensors (device or host) in the config's weight dtype; they are copied at
    creation.  With ``w_dtype == DT_MXFP4`` the expert weights are uint8
    tensors: gate_up_w / down_w the MXFP4 blocks, gate_up_scales /
    down_scales the E8M0 scales; with ``w_dtype == DT_Q4`` gate_up_w (or
    gate_w and up_w) and down_w are uint8 tensors of 18-byte Q4 records (the
    rest bf16; see include/moe.h)."""

    def __init__(self, config: MoEConfig, weights: dict, device: Optional[torch.device] = None):
        lib = load_library()
        self.config = config
        self.device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        w = _Weights()
        keep = []
        for n in WEIGHT_NAMES:
            t = weights.get(n)
            if t is not None:
                if not t.is_contiguous():
                    t = t.contiguous()
                keep.append(t)
                setattr(w, n, t.data_ptr())
        handle = ctypes.c_void_p()
        with torch.cuda.device(self.device):
            _check(lib.moe_layer_create(ctypes.byref(config._c()), ctypes.byref(w), ctypes.byref(handle)))
        self._h = handle
        self.out_dtype = _TORCH_DT[config.out_dtype]
        self.mxfp4 = config.w_dtype == DT_MXFP4
        self.q4 = config.w_dtype == DT_Q4
        self.x_dtype = _TORCH_DT[config.act_dtype]

    # ------------------------------------------------------------------
    def _rows(self, t: torch.Tensor, name: str, dtype: torch.dtype, T: Optional[int], host: bool) -> int:
        """The C ABI takes bare pointers, so the shape, dtype, layout and
        device of a token-row tensor are checked here: a tensor that is
        smaller than the layer assumes would be read or written past its
        end.  Returns the number of rows."""
        H = self.config.hidden
        if t.dim() != 2 or t.shape[1] != H or (T is not None and t.shape[0] != T):
            want = f"({T if T is not None else 'n_tokens'}, {H})"
            raise ValueError(f"{name}: expected shape {want}, got {tuple(t.shape)}")
        if t.dtype != dtype:
            raise ValueError(f"{name}: expected dtype {dtype}, got {t.dtype}")
        if not t.is_contiguous():
            raise ValueError(f"{name}: expected a contiguous tensor")
        if host and t.device.type != "cpu":
            raise ValueError(f"{name}: expected a host (CPU) tensor, got {t.device}")
        if not host and t.device != self.device:
            raise ValueError(f"{name}: expected a tensor on {self.device}, got {t.device}")
        return int(t.shape[0])

    def forward(self, x: torch.Tensor, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        """out = the layer applied to the token rows x [n_tokens, hidden] (the
        activation dtype, on the layer's device); out [n_tokens, hidden] in
        the output dtype is allocated when not given.  Asynchronous on
        `stream` (default: the current stream)."""
        T = self._rows(x, "x", self.x_dtype, None, host=False)
        if out is None:
            out = torch.empty((T, self.config.hidden), dtype=self.out_dtype, device=x.device)
        else:
            self._rows(out, "out", self.out_dtype, T, host=False)
        _check(_lib.moe_forward(self._h, x.data_ptr() if T else None, T, out.data_ptr() if T else None,
                                _stream_handle(stream)))
        return out

    __call__ = forward

    def forward_host(self, x_host: torch.Tensor, out_host: torch.Tensor, stream=None) -> None:
        """x_host / out_host: CPU tensors (pinned for asynchronous copies).
        The caller synchronises the stream before reading out_host."""
        T = self._rows(x_host, "x_host", self.x_dtype, None, host=True)
        self._rows(out_host, "out_host", self.out_dtype, T, host=True)
        _check(_lib.moe_forward_host(self._h, x_host.data_ptr() if T else None, T,
                                     out_host.data_ptr() if T else None, _stream_handle(stream)))

    def _last_tokens(self, n_tokens: Optional[int]) -> int:
        """Rows of the last successful forward, which the getters write; a
        caller's n_tokens must agree (a smaller buffer would overflow)."""
        n = int(_lib.moe_last_token_count(self._h))
        if n_tokens is not None and int(n_tokens) != n:
            raise ValueError(f"the last forward had {n} tokens, not {n_tokens}")
        return n

    def routing(self, n_tokens: Optional[int] = None, stream=None):
        """(idx [n, k] int32, w [n, k] fp32) of the last forward."""
        n_tokens = self._last_tokens(n_tokens)
        k = self.config.top_k
        idx = torch.empty((n_tokens, k), dtype=torch.int32, device=self.device)
        w = torch.empty((n_tokens, k), dtype=torch.float32, device=self.device)
        _check(_lib.moe_get_routing(self._h, idx.data_ptr(), w.data_ptr(), _stream_handle(stream)))
        return idx, w

    def logits(self, n_tokens: Optional[int] = None, stream=None):
        """(router logits [n, E] fp32, shared-expert gate logits [n]) of the
        last forward."""
        n_tokens = self._last_tokens(n_tokens)
        l = torch.empty((n_tokens, self.config.n_expert), dtype=torch.float32, device=self.device)
        s = torch.zeros((n_tokens,), dtype=torch.float32, device=self.device)
        _check(_lib.moe_get_logits(self._h, l.data_ptr(), s.data_ptr(), _stream_handle(stream)))
        return l, s

    def expert_counts(self, stream=None):
        c = torch.empty((self.config.n_expert,), dtype=torch.int32, device=self.device)
        _check(_lib.moe_get_expert_counts(self._h, c.data_ptr(), _stream_handle(stream)))
        return c

    def intermediate(self, which: int, stream=None) -> torch.Tensor:
        """A grouped-path intermediate of the last forward as a flat uint8
        device tensor (see moe_get_intermediate in include/moe.h)."""
        n = ctypes.c_size_t()
        _check(_lib.moe_get_intermediate(self._h, int(which), None, 0, ctypes.byref(n), _stream_handle(stream)))
        buf = torch.empty((n.value,), dtype=torch.uint8, device=self.device)
        if n.value:
            _check(_lib.moe_get_intermediate(self._h, int(which), buf.data_ptr(), n.value, None,
                                             _stream_handle(stream)))
        return buf

    def set_wait_limit(self, ns: int) -> None:
        """Bound of the kernels' waits on other thread blocks (0 = default 1 s)."""
        _check(_lib.moe_set_wait_limit(self._h, int(ns)))

    def set_fault_injection(self, on: bool) -> None:
        """Test only: the next forwards wait for what never happens and report
        MOE_ERR_DEVICE_TIMEOUT through status()."""
        _check(_lib.moe_set_fault_injection(self._h, int(bool(on))))

    def set_path(self, path: int) -> None:
        _check(_lib.moe_set_path(self._h, int(path)))

    def residency(self):
        """Expert residency: (expert held by each slot, {"hits", "misses",
        "bytes"} counted over every chunk since creation)."""
        S = self.config.resident_experts
        slots = (ctypes.c_int32 * max(S, 1))()
        stats = (ctypes.c_int64 * 3)()
        _check(_lib.moe_get_residency(self._h, slots, stats))
        return list(slots[:S]), {"hits": int(stats[0]), "misses": int(stats[1]), "bytes": int(stats[2])}

    def status(self) -> None:
        _check(_lib.moe_get_status(self._h))

    def timing_enable(self, max_forwards: int) -> None:
        """Record per-kernel CUDA events for up to max_forwards forwards."""
        _check(_lib.moe_timing_enable(self._h, int(max_forwards)))

    def timing_read(self) -> dict:
        """{kernel kind: (total ms, launches)} since the last read (syncs)."""
        n = len(KERNEL_KINDS)
        ms = (ctypes.c_float * n)()
        cnt = (ctypes.c_int32 * n)()
        _check(_lib.moe_timing_read(self._h, ctypes.cast(ms, ctypes.c_void_p), ctypes.cast(cnt, ctypes.c_void_p)))
        return {k: (float(ms[i]), int(cnt[i])) for i, k in enumerate(KERNEL_KINDS)}

    @property
    def last_launch_count(self) -> int:
        return int(_lib.moe_last_launch_count(self._h))

    @property
    def device_bytes(self) -> int:
        return int(_lib.moe_device_bytes(self._h))

    def close(self) -> None:
        if getattr(self, "_h", None) is not None and self._h.value:
            _lib.moe_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        # At interpreter shutdown the CUDA runtime may already be tearing down;
        # destroying the layer then (it synchronises the device and frees
        # memory) can crash the process, and process exit frees the memory
        # anyway.  Layers closed explicitly are unaffected.
        if sys.is_finalizing():
            return
        try:
            self.close()
        except Exception:
            pass
