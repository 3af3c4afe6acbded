"""The synthetic inputs follow their stated recipe: normal weights of variance
1/fan_in, biases of variance 0.02, bf16 rounded once to nearest even, a
counter-based stream (value i independent of chunking and token count), the
Zipf-skewed router's expert load, and the MXFP4 / Q4 code and scale
distributions.  Host only."""
import math

import numpy as np
import pytest

import synth


def _f32(a, dtype="bf16"):
    return synth.as_f32(a, dtype).astype(np.float64)


def test_normal_moments_and_bias_variance():
    spec = synth.QWEN.replace(name="moments", hidden=1024, n_expert=8, top_k=2, expert_ff=256, shared_ff=256)
    w = synth.make_weights(spec, seed=3)
    for name, fan_in in (("router_w", 1024), ("gate_w", 1024), ("up_w", 1024), ("down_w", 256),
                         ("sh_gate_w", 1024), ("sh_down_w", 256)):
        v = _f32(w[name])
        assert abs(v.mean()) < 5 * v.std() / math.sqrt(v.size), name
        assert v.std() == pytest.approx(1 / math.sqrt(fan_in), rel=0.01), name
    g = synth.GPTOSS.replace(name="biases", hidden=256, n_expert=32, top_k=4, expert_ff=256)
    wb = synth.make_weights(g, seed=4)
    b = np.concatenate([_f32(wb["gate_up_b"]).ravel(), _f32(wb["down_b"]).ravel()])
    assert b.std() == pytest.approx(math.sqrt(0.02), rel=0.02)


def test_bf16_is_round_to_nearest_even_once():
    f = synth.normal((1 << 16,), 1.0, 9, 77, "f32")
    bits = f.view(np.uint32).astype(np.uint64)
    # round to nearest, ties to even, on the upper 16 bits (all values finite)
    rne = ((bits + 0x7FFF + ((bits >> 16) & 1)) >> 16).astype(np.uint16)
    assert np.array_equal(synth.to_bf16(f), rne)
    b = synth.normal((1 << 16,), 1.0, 9, 77, "bf16")
    assert np.array_equal(b, rne)
    ties = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8)], dtype=np.float32)
    assert np.array_equal(synth.bf16_to_f32(synth.to_bf16(ties)),
                          np.array([1.0, 1.0 + 4 * 2.0 ** -8, -1.0], dtype=np.float32))


def test_stream_is_counter_based():
    a = synth.normal((1000,), 1.0, 5, 6, "f32")
    b = synth.normal((4000,), 1.0, 5, 6, "f32")
    c = synth.normal((500,), 1.0, 5, 6, "f32", offset=700)
    assert np.array_equal(a, b[:1000]) and np.array_equal(c, b[700:1200])
    assert not np.array_equal(a, synth.normal((1000,), 1.0, 5, 7, "f32"))   # another stream
    assert not np.array_equal(a, synth.normal((1000,), 1.0, 6, 6, "f32"))   # another seed
    spec = synth.GPTOSS.replace(name="rows", hidden=192)
    x5, x9 = synth.make_x(spec, 5, seed=2), synth.make_x(spec, 9, seed=2)
    assert np.array_equal(x5, x9[:5])
    assert np.array_equal(synth.make_x(spec, 4, seed=2, first_token=5), x9[5:])


def test_uniform_router_rows():
    spec = synth.MIXTRAL.replace(name="uniform router", hidden=1024, expert_ff=64)
    r = _f32(synth.make_weights(spec, seed=1)["router_w"])
    a = math.sqrt(3 / 1024)
    assert r.min() >= -a * (1 + 2 ** -8) and r.max() <= a * (1 + 2 ** -8)
    assert r.var() == pytest.approx(1 / 1024, rel=0.03)


def test_zipf_router_skews_the_expert_load():
    """logit_e is about ln p_e + N(0, ~1): the experts' selection counts fall
    with their Zipf rank, and the most loaded experts are the head of the law."""
    spec = synth.QWEN_ZIPF
    E, k, T = spec.n_expert, spec.top_k, 2048
    w = synth.make_weights(spec, seed=0)
    x = _f32(synth.make_x(spec, T, seed=0))
    logits = x @ _f32(w["router_w"]).T
    top = np.argsort(-logits, axis=1, kind="stable")[:, :k]
    counts = np.bincount(top.ravel(), minlength=E)
    logp, _ = synth._zipf_parts(spec, 0)
    # the noise of the logits against ln p_e has unit-order spread
    resid = (logits - logits.mean(axis=1, keepdims=True)) - (logp - logp.mean())[None, :]
    assert 0.5 < resid.std() < 2.0
    # counts decrease with the Zipf rank (rank correlation), and are skewed
    rank_p = np.argsort(np.argsort(-logp))
    rank_c = np.argsort(np.argsort(-counts, kind="stable"), kind="stable")
    rho = 1 - 6 * np.sum((rank_p - rank_c) ** 2.0) / (E * (E * E - 1))
    assert rho > 0.8, rho
    assert counts.max() > 8 * counts.mean()
    head = set(np.argsort(-logp)[:8])
    assert len(head & set(np.argsort(-counts)[:8])) >= 5


def test_mxfp4_codes_and_scales():
    spec = synth.GPTOSS_MXFP4.replace(name="mxfp4 draw", hidden=512, n_expert=4, expert_ff=256)
    w = synth.make_weights(spec, seed=8)
    blocks = np.concatenate([w["gate_up_blocks"].ravel(), w["down_blocks"].ravel()])
    codes = np.concatenate([blocks & 0xF, blocks >> 4])
    freq = np.bincount(codes, minlength=16) / codes.size
    assert np.all(np.abs(freq - 1 / 16) < 0.004), freq
    scales = np.concatenate([w["gate_up_scales"].ravel(), w["down_scales"].ravel()])
    assert set(np.unique(scales)) == {119, 120, 121}
    assert np.all(np.abs(np.bincount(scales)[119:] / scales.size - 1 / 3) < 0.02)
    assert w["gate_up_blocks"].shape == (4, 512, 512 // 32, 16) and w["down_scales"].shape == (4, 512, 256 // 32)


def test_q4_codes_and_scales():
    spec = synth.QWEN_Q4.replace(name="q4 draw", hidden=512, n_expert=4, top_k=2, expert_ff=256)
    w = synth.make_weights(spec, seed=8)
    for name, cols in (("gate_w_q4", 512), ("up_w_q4", 512), ("down_w_q4", 256)):
        rec = w[name].reshape(-1, 18)
        d = rec[:, :2].copy().view(np.float16).astype(np.float64).ravel()
        u = np.log2(d * 4.64 * math.sqrt(cols))
        assert u.min() >= -0.5 - 1e-3 and u.max() < 0.5 + 1e-3, name
        assert abs(u.mean()) < 0.02, name
        codes = np.concatenate([rec[:, 2:] & 0xF, rec[:, 2:] >> 4]).ravel()
        freq = np.bincount(codes, minlength=16) / codes.size
        assert np.all(np.abs(freq - 1 / 16) < 0.006), (name, freq)
