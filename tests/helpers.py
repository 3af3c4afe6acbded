"""Test helpers: build layers from synth specs, run the oracle beside the CUDA
path and compare them the way the parity bar states.

Parity bar (per layer):
  * expert indices bit-exact, ties to the lower index; a token whose k-th and
    (k+1)-th logits (or two adjacent selected logits) differ by < 1e-5 is a
    near tie: it is reported, its selection must still be a valid top-k, and
    its output is compared with the oracle's output for that selection;
  * relative L2 error of the output <= 1e-5 for fp32 layers, <= 1e-2 for
    bf16 layers (fp32 accumulation);
  * max |gpu - ref| <= 2e-2 * max |ref|.
"""
from __future__ import annotations

import dataclasses

import numpy as np

import synth

NEAR_TIE = 1e-5
REL_L2 = {"f32": 1e-5, "bf16": 1e-2}
MAX_ABS_FRAC = 2e-2


def moe_config(spec: synth.LayerSpec, max_tokens: int, out_dtype: str = "f32"):
    import sparse_mixture_experts_gb300 as moe
    dt = {"f32": moe.DT_F32, "bf16": moe.DT_BF16}
    return moe.MoEConfig(
        hidden=spec.hidden, n_expert=spec.n_expert, top_k=spec.top_k, expert_ff=spec.expert_ff,
        shared_ff=spec.shared_ff,
        router_mode=moe.ROUTER_SOFTMAX_TOPK if spec.router_mode == "softmax_topk" else moe.ROUTER_TOPK_SOFTMAX,
        norm_topk_prob=spec.norm_topk_prob, weights_scale=spec.weights_scale,
        act=moe.ACT_SWIGLU if spec.act == "swiglu" else moe.ACT_CLAMP_GLU,
        act_alpha=spec.act_alpha, act_limit=spec.act_limit, has_bias=spec.has_bias,
        gate_up_interleaved=spec.gate_up_interleaved,
        w_dtype={"mxfp4": moe.DT_MXFP4, "q4": moe.DT_Q4}.get(getattr(spec, "expert_format", "dense"),
                                                              dt[spec.dtype]),
        act_dtype=dt[spec.dtype],
        out_dtype=dt[out_dtype], max_tokens=max_tokens,
        resident_experts=getattr(spec, "resident_experts", 0))


def to_torch(a: np.ndarray, device="cuda"):
    """numpy float32 or uint16 (bf16 bits) -> torch tensor on `device`."""
    import torch
    if a.dtype == np.uint16:
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    elif a.dtype == np.uint8:
        t = torch.from_numpy(np.ascontiguousarray(a))
    else:
        t = torch.from_numpy(a)
    return t.to(device) if device != "cpu" else t


def make_layer(spec, weights: dict, max_tokens: int, out_dtype: str = "f32", path: int = 0):
    import sparse_mixture_experts_gb300 as moe
    w = {k: to_torch(v) for k, v in weights.items()}
    if getattr(spec, "expert_format", "dense") == "mxfp4":
        # the ABI takes the MXFP4 blocks in the gate_up_w / down_w slots
        w["gate_up_w"] = w.pop("gate_up_blocks")
        w["down_w"] = w.pop("down_blocks")
    elif getattr(spec, "expert_format", "dense") == "q4":
        # and the Q4 records in the slots of the tensors they stand for
        for n in [n for n in w if n.endswith("_q4")]:
            w[n[:-3]] = w.pop(n)
    layer = moe.MoELayer(moe_config(spec, max_tokens, out_dtype), w)
    if path:
        layer.set_path(path)
    return layer


@dataclasses.dataclass
class ParityReport:
    rel_l2: float
    max_abs: float
    max_ref: float
    n_tokens: int
    index_mismatch: list          # tokens whose selection differs without a near tie
    near_ties: list               # tokens with a near tie (reported)
    invalid_near_tie: list        # near-tie tokens whose selection is not a valid top-k

    def ok(self, dtype: str) -> bool:
        return (not self.index_mismatch and not self.invalid_near_tie and self.rel_l2 <= REL_L2[dtype]
                and self.max_abs <= MAX_ABS_FRAC * self.max_ref)

    def __str__(self):
        return (f"rel_l2={self.rel_l2:.3e} max_abs={self.max_abs:.3e} (bound {MAX_ABS_FRAC * self.max_ref:.3e}) "
                f"tokens={self.n_tokens} index_mismatch={self.index_mismatch[:8]} near_ties={self.near_ties[:8]} "
                f"invalid_near_tie={self.invalid_near_tie[:8]}")


def _near_tie(l_row: np.ndarray, k: int) -> bool:
    order = np.argsort(-l_row, kind="stable")
    v = l_row[order[:k + 1]]
    return bool(np.any(np.abs(np.diff(v)) < NEAR_TIE))


def _valid_topk(l_row: np.ndarray, sel: np.ndarray) -> bool:
    E = l_row.shape[0]
    if len(set(sel.tolist())) != len(sel) or np.any(sel < 0) or np.any(sel >= E):
        return False
    mask = np.zeros(E, bool)
    mask[sel] = True
    if (~mask).any() and l_row[mask].min() < l_row[~mask].max() - NEAR_TIE:
        return False
    return bool(np.all(np.diff(l_row[sel]) <= NEAR_TIE))


def compare(orc, x: np.ndarray, rows, gpu_out: np.ndarray, gpu_idx: np.ndarray, n_threads: int = 0) -> ParityReport:
    """Compare GPU outputs on token rows `rows` of x (gpu_out / gpu_idx hold
    those rows) with the oracle."""
    spec = orc.spec
    rows = np.asarray(rows, dtype=np.int32)
    ref, ref_idx, _ = orc.forward(x, rows=rows, n_threads=n_threads)
    logits, _ = orc.router_logits(np.ascontiguousarray(x[rows]))
    mism, ties, invalid = [], [], []
    xf = synth.as_f32(np.ascontiguousarray(x[rows]), spec.dtype).astype(np.float64)
    for i, t in enumerate(rows.tolist()):
        if np.array_equal(ref_idx[i], gpu_idx[i]):
            continue
        if _near_tie(logits[i], spec.top_k):
            ties.append(t)
            if not _valid_topk(logits[i], gpu_idx[i]):
                invalid.append(t)
                continue
            wt = orc.weights_for_selection(logits[i], gpu_idx[i])
            ref[i] = orc.token_output(xf[i], gpu_idx[i], wt)
        else:
            mism.append(t)
    g = gpu_out.astype(np.float64)
    diff = g - ref
    rel = float(np.linalg.norm(diff) / max(np.linalg.norm(ref), 1e-300))
    return ParityReport(rel, float(np.abs(diff).max()), float(np.abs(ref).max()), len(rows), mism, ties, invalid)


def index_parity_all(orc, x: np.ndarray, gpu_idx: np.ndarray):
    """Selection parity on every token (cheap: router logits + select only).
    Returns (mismatches without near tie, near-tie tokens, invalid near ties)."""
    spec = orc.spec
    logits, _ = orc.router_logits(x)
    mism, ties, invalid = [], [], []
    for t in range(x.shape[0]):
        idx, _ = orc.select(logits[t])
        if np.array_equal(idx, gpu_idx[t]):
            continue
        if _near_tie(logits[t], spec.top_k):
            ties.append(t)
            if not _valid_topk(logits[t], gpu_idx[t]):
                invalid.append(t)
        else:
            mism.append(t)
    return mism, ties, invalid, logits


def sample_rows(T: int, n: int, seed: int = 0) -> np.ndarray:
    """Up to n token rows: the first and last 8 (ragged tails) and a seeded
    spread in between."""
    if T <= n:
        return np.arange(T, dtype=np.int32)
    head = np.arange(8)
    tail = np.arange(T - 8, T)
    keys = synth.u64(T, seed, 999)
    mid = np.argsort(keys[8:T - 8], kind="stable")[: n - 16] + 8
    return np.unique(np.concatenate([head, mid, tail])).astype(np.int32)
