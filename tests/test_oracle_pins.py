"""Pins of the CPU oracle against facts fixed by the pages and by mathematics.

Each test would fail on a plausible mistake in the oracle: a dropped bias, a
swapped gate/up interleave, a transposed operand, a wrong tie-break, a missing
clamp or renormalisation, a wrong shared-expert gate.  None of them compares
the oracle with itself: they use hand-worked closed forms (tests/golden), a
dense brute-force restatement in numpy with a full sort, closed-form
equivalences between the two router forms and special cases that reduce to a
dense SwiGLU FFN.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def sig(z):
    return 1.0 / (1.0 + math.exp(-z))


def _ev(expr):
    return eval(expr, {"sig": sig, "exp": math.exp})


def _spec_from(d):
    kw = dict(d)
    return synth.LayerSpec(name="hand", **kw)


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        g = json.load(f)
    spec = _spec_from(g["layer"])
    w = {k: np.ascontiguousarray(np.array(v, dtype=np.float32)) for k, v in g["weights"].items()}
    x = np.array(g["x"], dtype=np.float32)
    return g, spec, w, x


# ----------------------------------------------------------------------------
# hand-worked examples
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["hand_example_softmax_shared.json", "hand_example_gptoss.json"])
def test_hand_example(golden_dir, name):
    g, spec, w, x = _load(golden_dir, name)
    o = oracle.Oracle(spec, w)
    exp = g["expected"]
    logits, _ = o.router_logits(x)
    np.testing.assert_allclose(logits[0], [_ev(v) for v in exp["logits"]], rtol=0, atol=1e-15)
    out, idx, wt = o.forward(x)
    assert idx[0].tolist() == exp["idx"]
    np.testing.assert_allclose(wt[0], [_ev(v) for v in exp["weights"]], rtol=1e-14, atol=0)
    np.testing.assert_allclose(out[0], [_ev(v) for v in exp["out"]], rtol=1e-13, atol=1e-15)


def test_hand_example_probabilities(golden_dir):
    g, spec, w, x = _load(golden_dir, "hand_example_softmax_shared.json")
    o = oracle.Oracle(spec.replace(norm_topk_prob=False), w)
    logits, _ = o.router_logits(x)
    idx, wt = o.select(logits[0])
    probs = [_ev(v) for v in g["expected"]["probs"]]
    np.testing.assert_allclose(wt, [probs[i] for i in idx], rtol=1e-14)


def test_weights_scale_applies_after_renormalisation(golden_dir):
    g, spec, w, x = _load(golden_dir, "hand_example_softmax_shared.json")
    o = oracle.Oracle(spec.replace(weights_scale=2.5), w)
    _, _, wt = o.forward(x)
    np.testing.assert_allclose(wt[0], [2.5 * sig(1), 2.5 * (1 - sig(1))], rtol=1e-14)


# ----------------------------------------------------------------------------
# activations at chosen points (E = 1, k = 1, H = 1, F = 1 layer: out = act)
# ----------------------------------------------------------------------------

def _act_layer(act, gate, up):
    spec = synth.LayerSpec("act", 1, 1, 1, 1, act=act, gate_up_interleaved=(act == "clamp_glu"), dtype="f32",
                           router_mode="topk_softmax" if act == "clamp_glu" else "softmax_topk",
                           has_bias=(act == "clamp_glu"))
    w = {"router_w": np.array([[1.0]], np.float32), "down_w": np.array([[[1.0]]], np.float32)}
    if act == "clamp_glu":
        # gate row 0, up row 1; the values enter through the biases (x = 0)
        w["gate_up_w"] = np.zeros((1, 2, 1), np.float32)
        w["gate_up_b"] = np.array([[gate, up]], np.float32)
        w["router_b"] = np.zeros(1, np.float32)
        w["down_b"] = np.zeros((1, 1), np.float32)
        x = np.zeros((1, 1), np.float32)
    else:
        w["gate_w"] = np.array([[[gate]]], np.float32)
        w["up_w"] = np.array([[[up]]], np.float32)
        x = np.ones((1, 1), np.float32)
    out, _, wt = oracle.Oracle(spec, w).forward(x)
    assert wt[0, 0] == 1.0
    return out[0, 0]


@pytest.mark.parametrize("gate,up,expected", [
    (10.0, 10.0, "8*7*sig(1.702*7)"),        # both clamped to the limit
    (1.0, 0.0, "sig(1.702)"),
    (-2.0, -9.0, "(-7+1)*(-2)*sig(-1.702*2)"),  # up clamped from below
    (0.0, 3.0, "0"),
    (-8.0, 0.5, "1.5*(-8)*sig(-1.702*8)"),    # gate has no lower clamp
    (7.5, -7.5, "(-7+1)*7*sig(1.702*7)"),
    (3.0, 6.5, "7.5*3*sig(1.702*3)"),         # inside the limits
])
def test_clamp_glu_points(gate, up, expected):
    assert _act_layer("clamp_glu", gate, up) == pytest.approx(_ev(expected), rel=1e-14, abs=1e-300)


@pytest.mark.parametrize("gate,up", [(1.0, 1.0), (-3.0, 2.0), (0.5, -4.0), (12.0, 0.25)])
def test_swiglu_points(gate, up):
    assert _act_layer("swiglu", gate, up) == pytest.approx(gate * sig(gate) * up, rel=1e-14)


def test_clamp_glu_bound_on_large_inputs():
    """|h| <= 8 * 7 * sig(1.702 * 7) whatever the expert's pre-activations."""
    spec = synth.GPTOSS.replace(name="small gpt-oss", hidden=48, n_expert=4, top_k=2, expert_ff=24, dtype="f32")
    w = synth.make_weights(spec, seed=3)
    w["gate_up_w"] = (w["gate_up_w"] * 40.0).astype(np.float32)
    x = synth.make_x(spec, 4, seed=3)
    o = oracle.Oracle(spec, w)
    bound = 8 * 7 * sig(1.702 * 7)
    hit_limit = False
    for t in range(4):
        for e in range(spec.n_expert):
            h, _ = o.expert(e, x[t].astype(np.float64))
            assert np.all(np.abs(h) <= bound * (1 + 1e-15))
            hit_limit |= bool(np.any(np.abs(h) > 0.999 * bound))
    assert hit_limit  # the scaled weights do drive pairs into both clamps


# ----------------------------------------------------------------------------
# ties and top-k
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("mode", ["softmax_topk", "topk_softmax"])
def test_tie_breaks_to_lower_index(mode):
    spec = synth.LayerSpec("tie", 2, 3, 1, 1, router_mode=mode, dtype="f32")
    o = oracle.Oracle(spec, {"router_w": np.zeros((3, 2), np.float32)})
    idx, wt = o.select(np.array([1.0, 1.0, 0.0]))
    assert idx.tolist() == [0] and wt[0] == 1.0
    idx, _ = o.select(np.array([0.0, 2.0, 2.0]))
    assert idx.tolist() == [1]


@pytest.mark.parametrize("mode", ["softmax_topk", "topk_softmax"])
def test_topk_matches_full_stable_sort(mode):
    E, k = 16, 5
    spec = synth.LayerSpec("sort", 2, E, k, 1, router_mode=mode, dtype="f32")
    o = oracle.Oracle(spec, {"router_w": np.zeros((E, 2), np.float32)})
    rng = np.random.default_rng(7)
    for trial in range(200):
        l = rng.normal(size=E)
        if trial % 2:
            l = np.round(l * 2) / 2          # many exact ties
        idx, wt = o.select(l)
        want = np.argsort(-l, kind="stable")[:k]   # stable: equal keys keep index order
        assert idx.tolist() == want.tolist()
        assert np.all(np.diff(wt) <= 0)             # descending weights


def test_renormalised_weights_sum_to_one():
    E, k = 64, 8
    spec = synth.LayerSpec("sum", 2, E, k, 1, dtype="f32")
    o = oracle.Oracle(spec, {"router_w": np.zeros((E, 2), np.float32)})
    rng = np.random.default_rng(1)
    for _ in range(100):
        _, wt = o.select(rng.normal(scale=3.0, size=E))
        assert abs(wt.sum() - 1.0) <= 4 * np.finfo(np.float64).eps


def test_without_renormalisation_weights_are_probabilities():
    E, k = 10, 3
    spec = synth.LayerSpec("p", 2, E, k, 1, norm_topk_prob=False, dtype="f32")
    o = oracle.Oracle(spec, {"router_w": np.zeros((E, 2), np.float32)})
    l = np.linspace(-1, 2, E)
    idx, wt = o.select(l)
    p = np.exp(l - l.max()) / np.exp(l - l.max()).sum()
    np.testing.assert_allclose(wt, p[idx], rtol=1e-14)


# ----------------------------------------------------------------------------
# brute force: dense evaluation of every expert + scatter of the scores
# ----------------------------------------------------------------------------

def _silu(z):
    return z / (1.0 + np.exp(-z))


def _dense_reference(spec, w, x):
    """Scatter-dense form: evaluate every expert on every token, scatter the
    routing scores into an [T, E] matrix that is zero outside the top-k (full
    stable sort), and contract.  Independent restatement in numpy."""
    f64 = lambda a: synth.as_f32(a, spec.dtype).astype(np.float64)
    X = f64(x)
    T, E, F, H = X.shape[0], spec.n_expert, spec.expert_ff, spec.hidden
    L = X @ f64(w["router_w"]).T
    if spec.has_bias:
        L = L + f64(w["router_b"])[None, :]
    scores = np.zeros((T, E))
    for t in range(T):
        order = np.argsort(-L[t], kind="stable")[:spec.top_k]
        if spec.router_mode == "softmax_topk":
            p = np.exp(L[t] - L[t].max())
            p /= p.sum()
            s = p[order]
            if spec.norm_topk_prob:
                s = s / s.sum()
            s = s * spec.weights_scale
        else:
            v = L[t, order]
            s = np.exp(v - v.max()) / np.exp(v - v.max()).sum()
        scores[t, order] = s
    Y = np.zeros((T, E, H))
    for e in range(E):
        if spec.gate_up_interleaved:
            Z = X @ f64(w["gate_up_w"][e]).T
            if spec.has_bias:
                Z = Z + f64(w["gate_up_b"][e])[None, :]
            G, U = Z[:, 0::2], Z[:, 1::2]
        else:
            G = X @ f64(w["gate_w"][e]).T
            U = X @ f64(w["up_w"][e]).T
            if spec.has_bias:
                b = f64(w["gate_up_b"][e])
                G, U = G + b[None, :F], U + b[None, F:]
        if spec.act == "swiglu":
            Hh = _silu(G) * U
        else:
            G = np.minimum(G, spec.act_limit)
            U = np.clip(U, -spec.act_limit, spec.act_limit)
            Hh = (U + 1.0) * G / (1.0 + np.exp(-spec.act_alpha * G))
        Ye = Hh @ f64(w["down_w"][e]).T
        if spec.has_bias:
            Ye = Ye + f64(w["down_b"][e])[None, :]
        Y[:, e, :] = Ye
    out = np.einsum("te,teh->th", scores, Y)
    if spec.shared_ff > 0:
        Hs = _silu(X @ f64(w["sh_gate_w"]).T) * (X @ f64(w["sh_up_w"]).T)
        gate = 1.0 / (1.0 + np.exp(-(X @ f64(w["sh_gate_inp"]))))
        out = out + gate[:, None] * (Hs @ f64(w["sh_down_w"]).T)
    return out, scores


SMALL_SPECS = [
    synth.TINY,
    synth.TINY.replace(name="tiny bf16 + shared", dtype="bf16", shared_ff=24),
    synth.LayerSpec("small gpt-oss f32", 40, 6, 3, 20, router_mode="topk_softmax", act="clamp_glu", has_bias=True,
                    gate_up_interleaved=True, dtype="f32"),
    synth.LayerSpec("small gpt-oss bf16", 40, 8, 4, 24, router_mode="topk_softmax", act="clamp_glu", has_bias=True,
                    gate_up_interleaved=True, dtype="bf16"),
    synth.LayerSpec("small, biased swiglu, unnormalised", 32, 5, 2, 12, has_bias=True, norm_topk_prob=False,
                    weights_scale=1.7, dtype="f32"),
    synth.QWEN_ZIPF.replace(name="small zipf", hidden=48, n_expert=8, top_k=3, expert_ff=16, shared_ff=8),
    synth.MIXTRAL.replace(name="small uniform router", hidden=40, n_expert=4, top_k=2, expert_ff=28),
]


@pytest.mark.parametrize("spec", SMALL_SPECS, ids=lambda s: s.name)
def test_brute_force_dense_scatter(spec):
    w = synth.make_weights(spec, seed=11)
    x = synth.make_x(spec, 9, seed=11)
    out, idx, wt = oracle.Oracle(spec, w).forward(x)
    ref, scores = _dense_reference(spec, w, x)
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-12 * np.abs(ref).max())
    for t in range(x.shape[0]):
        nz = np.flatnonzero(scores[t])
        assert sorted(idx[t].tolist()) == sorted(nz.tolist())
        np.testing.assert_allclose(wt[t], scores[t, idx[t]], rtol=1e-13)


def test_brute_force_with_exact_ties():
    """Router rows repeated exactly, so logits tie; the lower index must win."""
    spec = synth.LayerSpec("ties", 16, 6, 2, 8, dtype="f32")
    w = synth.make_weights(spec, seed=5)
    w["router_w"][3] = w["router_w"][1]
    w["router_w"][5] = w["router_w"][0]
    x = synth.make_x(spec, 12, seed=5)
    out, idx, _ = oracle.Oracle(spec, w).forward(x)
    ref, scores = _dense_reference(spec, w, x)
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-13)
    for t in range(12):
        assert sorted(idx[t].tolist()) == sorted(np.flatnonzero(scores[t]).tolist())


# ----------------------------------------------------------------------------
# closed-form equivalences and invariants
# ----------------------------------------------------------------------------

def test_top_k_equal_to_n_expert_is_dense_softmax_mixture():
    spec = synth.LayerSpec("k=E", 24, 5, 5, 10, shared_ff=6, dtype="f32")
    w = synth.make_weights(spec, seed=2)
    x = synth.make_x(spec, 6, seed=2)
    out, _, wt = oracle.Oracle(spec, w).forward(x)
    X = x.astype(np.float64)
    L = X @ w["router_w"].astype(np.float64).T
    P = np.exp(L - L.max(1, keepdims=True))
    P /= P.sum(1, keepdims=True)
    dense = np.zeros_like(out)
    for e in range(5):
        He = _silu(X @ w["gate_w"][e].astype(np.float64).T) * (X @ w["up_w"][e].astype(np.float64).T)
        dense += P[:, e:e + 1] * (He @ w["down_w"][e].astype(np.float64).T)
    Hs = _silu(X @ w["sh_gate_w"].astype(np.float64).T) * (X @ w["sh_up_w"].astype(np.float64).T)
    g = 1 / (1 + np.exp(-(X @ w["sh_gate_inp"].astype(np.float64))))
    dense += g[:, None] * (Hs @ w["sh_down_w"].astype(np.float64).T)
    np.testing.assert_allclose(out, dense, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(np.sort(wt, 1)[:, ::-1], np.sort(P, 1)[:, ::-1], rtol=1e-13)


def test_single_expert_is_dense_swiglu_ffn():
    """E = 1, k = 1: weight 1, so the layer is the dense SwiGLU FFN
    out = W_down (silu(W_gate x) * (W_up x))."""
    spec = synth.LayerSpec("dense", 32, 1, 1, 48, dtype="f32")
    w = synth.make_weights(spec, seed=4)
    x = synth.make_x(spec, 5, seed=4)
    out, idx, wt = oracle.Oracle(spec, w).forward(x)
    assert np.all(idx == 0) and np.all(wt == 1.0)
    X = x.astype(np.float64)
    Wg, Wu, Wd = (w[n][0].astype(np.float64) for n in ("gate_w", "up_w", "down_w"))
    G = X @ Wg.T
    ffn = ((G / (1 + np.exp(-G))) * (X @ Wu.T)) @ Wd.T
    np.testing.assert_allclose(out, ffn, rtol=1e-12, atol=1e-14)


def test_router_forms_agree_without_bias():
    """Without a bias, softmax over all E then renormalising over the k kept
    equals softmax over the k kept logits: the full denominator cancels."""
    base = synth.LayerSpec("forms", 32, 8, 3, 16, dtype="f32")
    w = synth.make_weights(base, seed=6)
    x = synth.make_x(base, 10, seed=6)
    a = oracle.Oracle(base, w).forward(x)
    b = oracle.Oracle(base.replace(router_mode="topk_softmax"), w).forward(x)
    assert np.array_equal(a[1], b[1])
    np.testing.assert_allclose(a[2], b[2], rtol=1e-13)
    np.testing.assert_allclose(a[0], b[0], rtol=1e-12, atol=1e-14)


def test_router_bias_changes_selection():
    spec = synth.LayerSpec("bias", 16, 4, 1, 4, router_mode="topk_softmax", act="clamp_glu", has_bias=True,
                           gate_up_interleaved=True, dtype="f32")
    w = synth.make_weights(spec, seed=8)
    x = synth.make_x(spec, 1, seed=8)
    o = oracle.Oracle(spec, w)
    l, _ = o.router_logits(x)
    loser = int(np.argmin(l[0]))
    w2 = dict(w)
    w2["router_b"] = w["router_b"].copy()
    w2["router_b"][loser] = 100.0
    _, idx, _ = oracle.Oracle(spec, w2).forward(x)
    assert idx[0, 0] == loser


def test_token_permutation_equivariance():
    spec = SMALL_SPECS[2]
    w = synth.make_weights(spec, seed=9)
    x = synth.make_x(spec, 7, seed=9)
    o = oracle.Oracle(spec, w)
    out, idx, _ = o.forward(x)
    perm = np.array([3, 0, 6, 1, 5, 2, 4])
    out2, idx2, _ = o.forward(np.ascontiguousarray(x[perm]))
    np.testing.assert_array_equal(out2, out[perm])
    np.testing.assert_array_equal(idx2, idx[perm])


@pytest.mark.parametrize("spec", [SMALL_SPECS[1], SMALL_SPECS[3]], ids=lambda s: s.name)
def test_expert_permutation_invariance(spec):
    """Relabelling the experts (router rows together with their weights) maps
    the indices and leaves the outputs unchanged."""
    w = synth.make_weights(spec, seed=10)
    x = synth.make_x(spec, 6, seed=10)
    out, idx, _ = oracle.Oracle(spec, w).forward(x)
    E = spec.n_expert
    pi = np.roll(np.arange(E), 3)            # new expert j is old expert pi[j]
    w2 = {}
    for n, a in w.items():
        if n in ("router_w", "router_b", "gate_w", "up_w", "gate_up_w", "gate_up_b", "down_w", "down_b"):
            w2[n] = np.ascontiguousarray(a[pi])
        else:
            w2[n] = a
    out2, idx2, _ = oracle.Oracle(spec, w2).forward(x)
    np.testing.assert_allclose(out2, out, rtol=1e-12, atol=1e-14)
    inv = np.argsort(pi)
    assert np.array_equal(np.sort(inv[idx], 1), np.sort(idx2, 1))


def test_batch_independence_and_row_selection():
    spec = SMALL_SPECS[1]
    w = synth.make_weights(spec, seed=12)
    x = synth.make_x(spec, 8, seed=12)
    o = oracle.Oracle(spec, w)
    out, _, _ = o.forward(x)
    for t in (0, 5, 7):
        single, _, _ = o.forward(np.ascontiguousarray(x[t:t + 1]))
        np.testing.assert_array_equal(single[0], out[t])
    rows = np.array([7, 2, 2])
    sub, _, _ = o.forward(x, rows=rows)
    np.testing.assert_array_equal(sub, out[rows])
    # the generator gives the same token rows whatever the token count
    np.testing.assert_array_equal(synth.make_x(spec, 3, seed=12), x[:3])


def test_bf16_storage_reads_exact_values():
    spec = SMALL_SPECS[1]
    w = synth.make_weights(spec, seed=13)
    x = synth.make_x(spec, 4, seed=13)
    o = oracle.Oracle(spec, w)
    f32spec = spec.replace(dtype="f32")
    o32 = oracle.Oracle(f32spec, {k: synth.bf16_to_f32(v) for k, v in w.items()})
    a = o.forward(x)
    b = o32.forward(synth.bf16_to_f32(x))
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_threads_do_not_change_results():
    spec = SMALL_SPECS[3]
    w = synth.make_weights(spec, seed=14)
    x = synth.make_x(spec, 32, seed=14)
    o = oracle.Oracle(spec, w)
    a = o.forward(x, n_threads=1)
    b = o.forward(x, n_threads=4)
    for u, v in zip(a, b):
        np.testing.assert_array_equal(u, v)


def test_invalid_configs_are_rejected():
    with pytest.raises(ValueError):
        oracle.Oracle(synth.LayerSpec("bad", 8, 4, 5, 4, dtype="f32"), {})
    with pytest.raises(ValueError):
        oracle.Oracle(synth.LayerSpec("bad", 8, 4, 0, 4, dtype="f32"), {})


# ----------------------------------------------------------------------------
# MXFP4 expert weights ("Phase 19: MoE -- gpt-oss-20b": MXFP4 packing note and
# section 3, dequantisation; E2M1 values from the OCP Microscaling formats)
# ----------------------------------------------------------------------------

# the sixteen E2M1 values as the OCP definition lists them
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def test_e2m1_code_table():
    vals = [oracle.e2m1_value(c) for c in range(16)]
    assert vals == E2M1_TABLE
    # sign bit 3, magnitudes of 0..7 strictly increasing from 0, largest 6
    for c in range(8):
        assert vals[c + 8] == -vals[c] and math.copysign(1.0, vals[c + 8]) == -1.0
    assert all(vals[c] < vals[c + 1] for c in range(7)) and max(vals) == 6.0


def test_e8m0_scale():
    assert oracle.e8m0_scale(127) == 1.0
    assert oracle.e8m0_scale(128) == 2.0 and oracle.e8m0_scale(126) == 0.5
    assert oracle.e8m0_scale(0) == 2.0 ** -127 and oracle.e8m0_scale(254) == 2.0 ** 127
    assert math.isnan(oracle.e8m0_scale(255))


def test_mxfp4_nibble_order_and_block_direction():
    # one row of 64 elements = two blocks along the input dimension
    blocks = np.zeros((1, 2, 16), dtype=np.uint8)
    scales = np.array([[127, 129]], dtype=np.uint8)
    blocks[0, 0, 0] = 0x21   # element 0 = code 1 (low nibble), element 1 = code 2 (high nibble)
    blocks[0, 1, 15] = 0xF7  # element 32 + 30 = code 7, element 32 + 31 = code 15
    v = oracle.mxfp4_dequant(blocks, scales)[0]
    assert v[0] == 0.5 and v[1] == 1.0
    assert v[62] == 6.0 * 4 and v[63] == -6.0 * 4
    assert np.count_nonzero(v) == 4


def _numpy_dequant(blocks, scales):
    """The same definition restated with numpy bit operations (table lookup)."""
    lo, hi = blocks & 0x0F, blocks >> 4
    codes = np.stack([lo, hi], axis=-1).reshape(blocks.shape[:-1] + (32,))
    vals = np.array(E2M1_TABLE)[codes] * np.ldexp(1.0, scales.astype(np.int64) - 127)[..., None]
    return vals.reshape(scales.shape[:-1] + (scales.shape[-1] * 32,))


def test_mxfp4_dequant_matches_table_restatement():
    spec = synth.GPTOSS_MXFP4.replace(hidden=96, n_expert=3, expert_ff=64, top_k=2)
    w = synth.make_weights(spec, seed=3)
    for b, s in (("gate_up_blocks", "gate_up_scales"), ("down_blocks", "down_scales")):
        np.testing.assert_array_equal(oracle.mxfp4_dequant(w[b], w[s]), _numpy_dequant(w[b], w[s]))


def test_hand_example_mxfp4(golden_dir):
    with open(os.path.join(golden_dir, "hand_example_mxfp4.json")) as f:
        g = json.load(f)
    spec = _spec_from(g["layer"])
    H, E, F = spec.hidden, spec.n_expert, spec.expert_ff
    w = {
        "router_w": synth.to_bf16(np.zeros((E, H), np.float32)),
        "router_b": synth.to_bf16(np.array(g["router_b"], np.float32)),
        "gate_up_b": synth.to_bf16(np.zeros((E, 2 * F), np.float32)),
        "down_b": synth.to_bf16(np.zeros((E, H), np.float32)),
        "gate_up_blocks": np.zeros((E, 2 * F, H // 32, 16), np.uint8),
        "gate_up_scales": np.full((E, 2 * F, H // 32), g["scales_default"], np.uint8),
        "down_blocks": np.zeros((E, H, F // 32, 16), np.uint8),
        "down_scales": np.full((E, H, F // 32), g["scales_default"], np.uint8),
    }
    for nz in g["nonzero_bytes"]:
        w[nz["tensor"]][nz["expert"], nz["row"], 0, nz["byte"]] = int(nz["value"], 16)
    for so in g["scale_overrides"]:
        w[so["tensor"]][so["expert"], so["row"], so["block"]] = so["value"]
    x = np.zeros((1, H), np.float32)
    x[0, :len(g["x"])] = g["x"]
    out, idx, wt = oracle.Oracle(spec, w).forward(synth.to_bf16(x))
    assert idx[0].tolist() == [0] and wt[0].tolist() == [1.0]
    exp = [_ev(v) for v in g["expected_out_first2"]]
    np.testing.assert_allclose(out[0, :2], exp, rtol=1e-13, atol=0)
    assert np.count_nonzero(out[0, 2:]) == 0


def test_mxfp4_layer_equals_dense_layer_of_its_values():
    # the MXFP4 layer is the dense layer whose weights are the dequantised values
    spec = synth.GPTOSS_MXFP4.replace(hidden=64, n_expert=4, expert_ff=64, top_k=2)
    w = synth.make_weights(spec, seed=5)
    dense = {k: synth.bf16_to_f32(v) for k, v in w.items() if v.dtype == np.uint16}
    dense["gate_up_w"] = _numpy_dequant(w["gate_up_blocks"], w["gate_up_scales"]).astype(np.float32)
    dense["down_w"] = _numpy_dequant(w["down_blocks"], w["down_scales"]).astype(np.float32)
    x = synth.make_x(spec, 5, seed=2)
    out_mx, idx_mx, _ = oracle.Oracle(spec, w).forward(x)
    dspec = spec.replace(dtype="f32", expert_format="dense")
    out_d, idx_d, _ = oracle.Oracle(dspec, dense).forward(synth.bf16_to_f32(x))
    np.testing.assert_array_equal(idx_mx, idx_d)
    np.testing.assert_array_equal(out_mx, out_d)


# ----------------------------------------------------------------------------
# Q4 records: binary16 scale, 32 four-bit codes offset by 8, element j in the
# low nibble of byte j and element j + 16 in its high nibble
# ----------------------------------------------------------------------------

def test_fp16_values():
    assert oracle.fp16_value(0x3C00) == 1.0 and oracle.fp16_value(0xC000) == -2.0
    assert oracle.fp16_value(0x3800) == 0.5 and oracle.fp16_value(0x3E00) == 1.5
    assert oracle.fp16_value(0x7BFF) == 65504.0           # largest finite
    assert oracle.fp16_value(0x0400) == 2.0 ** -14         # smallest normal
    assert oracle.fp16_value(0x0001) == 2.0 ** -24         # smallest subnormal
    assert oracle.fp16_value(0x0000) == 0.0 and math.copysign(1.0, oracle.fp16_value(0x8000)) == -1.0
    assert math.isinf(oracle.fp16_value(0x7C00)) and math.isnan(oracle.fp16_value(0x7E00))
    # every pattern agrees with numpy's binary16
    pats = np.arange(1 << 16, dtype=np.uint16)
    ref = pats.view(np.float16).astype(np.float64)
    got = np.array([oracle.fp16_value(int(h)) for h in pats[::97]])
    np.testing.assert_array_equal(got, ref[::97])


def test_q4_block_hand_worked():
    # d = 0.5; byte j holds code j (element j) and code 15 - j (element j + 16)
    blk = np.zeros((1, 1, 18), np.uint8)
    blk[0, 0, 0], blk[0, 0, 1] = 0x00, 0x38               # 0x3800 little-endian
    for j in range(16):
        blk[0, 0, 2 + j] = j | ((15 - j) << 4)
    v = oracle.q4_dequant(blk)[0]
    assert v[:16].tolist() == [(j - 8) * 0.5 for j in range(16)]      # -4.0 .. 3.5
    assert v[16:].tolist() == [(15 - j - 8) * 0.5 for j in range(16)]  # 3.5 .. -4.0
    assert v[8] == 0.0 and v[0] == -4.0                                # code 8 is zero


def test_q4_block_direction_and_scale_per_block():
    # two blocks along the input dimension, each with its own scale
    blk = np.zeros((1, 2, 18), np.uint8)
    blk[0, 0, :2] = [0x00, 0x3C]    # d = 1
    blk[0, 1, :2] = [0x00, 0xC0]    # d = -2
    blk[0, :, 2:] = 0x88            # every code 8 -> 0
    blk[0, 0, 2] = 0x09             # element 0 = code 9 (+1), element 16 = code 0 (-8)
    blk[0, 1, 17] = 0xF8            # element 32 + 15 = code 8 (0), element 32 + 31 = code 15 (+7)
    v = oracle.q4_dequant(blk)[0]
    assert v[0] == 1.0 and v[16] == -8.0 and v[63] == -14.0
    assert np.count_nonzero(v) == 3


def _numpy_q4(blocks):
    """The same definition restated with numpy bit operations."""
    d = (blocks[..., 0].astype(np.uint16) | (blocks[..., 1].astype(np.uint16) << 8)).view(np.float16)
    q = blocks[..., 2:]
    codes = np.concatenate([q & 0x0F, q >> 4], axis=-1).astype(np.float64) - 8.0
    vals = codes * d.astype(np.float64)[..., None]
    return vals.reshape(blocks.shape[:-2] + (blocks.shape[-2] * 32,))


def test_q4_dequant_matches_numpy_restatement():
    spec = synth.QWEN_Q4.replace(hidden=96, n_expert=3, expert_ff=64, top_k=2)
    w = synth.make_weights(spec, seed=3)
    for n in ("gate_w_q4", "up_w_q4", "down_w_q4"):
        np.testing.assert_array_equal(oracle.q4_dequant(w[n]), _numpy_q4(w[n]))


@pytest.mark.parametrize("interleaved", [False, True])
def test_q4_layer_equals_dense_layer_of_its_values(interleaved):
    spec = synth.QWEN_Q4.replace(hidden=64, n_expert=4, expert_ff=64, top_k=2, gate_up_interleaved=interleaved)
    w = synth.make_weights(spec, seed=5)
    dense = {k: synth.bf16_to_f32(v) for k, v in w.items() if v.dtype == np.uint16}
    for n in ("gate_up_w", "gate_w", "up_w", "down_w"):
        if n + "_q4" in w:
            dense[n] = _numpy_q4(w[n + "_q4"]).astype(np.float32)
    x = synth.make_x(spec, 5, seed=2)
    out_q, idx_q, _ = oracle.Oracle(spec, w).forward(x)
    dspec = spec.replace(dtype="f32", expert_format="dense")
    out_d, idx_d, _ = oracle.Oracle(dspec, dense).forward(synth.bf16_to_f32(x))
    np.testing.assert_array_equal(idx_q, idx_d)
    np.testing.assert_array_equal(out_q, out_d)
