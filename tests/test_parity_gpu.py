"""GPU parity: the CUDA path through the C ABI against the CPU oracle, on the
seeded synthetic layers (tiny fp32; qwen35moe-shaped decode and Zipf-skewed
prefill; gpt-oss-20b-shaped; mixtral-shaped token sweep), on both kernel paths
(weight-streaming CUDA-core kernels and tcgen05 grouped GEMMs).

At the full sizes the oracle computes a sample of token rows (the first and
last 8, for the ragged tail, plus a seeded spread); the selection is checked
on every token."""
import gc

import numpy as np
import pytest

import oracle
import synth
from tests import helpers

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import sparse_mixture_experts_gb300 as moe  # noqa: E402

# workload -> (token counts, oracle rows sampled per case)
CASES = [
    ("tiny", 16, 16),
    ("qwen_decode", 1, 1), ("qwen_decode", 4, 4), ("qwen_decode", 8, 8),
    ("qwen_prefill_zipf", 4096, 160),
    ("gptoss", 1, 1), ("gptoss", 64, 64), ("gptoss", 2048, 64),
    ("mixtral", 1, 1), ("mixtral", 16, 16), ("mixtral", 256, 40), ("mixtral", 4096, 24), ("mixtral", 16384, 24),
    # MXFP4 experts: both tensor-core paths widen the packed codes and scales on chip
    ("gptoss_mxfp4", 1, 1), ("gptoss_mxfp4", 4, 4), ("gptoss_mxfp4", 16, 16), ("gptoss_mxfp4", 64, 32),
    # Q4 expert records: both tensor-core paths widen them on chip
    ("qwen_q4", 1, 1), ("qwen_q4", 8, 8), ("qwen_q4", 300, 40),
    ("gptoss_q4", 1, 1), ("gptoss_q4", 16, 16), ("gptoss_q4", 2048, 48),
]

# CUDA-core flops budget for the streaming path in a test (it is the decode path)
STREAM_MAX_FLOP = 6e11


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_mixture_experts_gb300 import build
    build.build()


class _Workload:
    def __init__(self, name):
        self.spec, counts = synth.WORKLOADS[name]
        self.Tmax = max(counts)
        self.w = synth.make_weights(self.spec, seed=0)
        self.x = synth.make_x(self.spec, self.Tmax, seed=0)
        self.orc = oracle.Oracle(self.spec, self.w)
        self.layer = helpers.make_layer(self.spec, self.w, self.Tmax)
        self.x_dev = helpers.to_torch(self.x)

    def close(self):
        self.layer.close()


_cache = {}


def workload(name):
    if name not in _cache:
        for k in list(_cache):
            _cache.pop(k).close()
        gc.collect()
        torch.cuda.empty_cache()
        _cache[name] = _Workload(name)
    return _cache[name]


def _flops(spec, T):
    return 2.0 * T * spec.top_k * 3 * spec.hidden * spec.expert_ff


PATHS = [moe.PATH_STREAM, moe.PATH_TC, moe.PATH_FUSED, moe.PATH_DECODE_TC]
PATH_IDS = ["stream", "tc", "fused", "dectc"]
FUSED_MAX_TOKENS = 8
DECODE_TC_MAX_TOKENS = 16


def _applies(spec, path, T=None):
    """Which kernel path a case can take, decided from the layer's shape alone:
    the CUDA-core paths read bf16 or fp32 weights, the fused decode kernel
    covers up to 8 tokens and F a multiple of 16 (its rows per work item), the tensor-core paths need bf16 weights with H, F
    and the shared F multiples of 64, the weight-streaming tensor-core kernels
    cover up to 16 tokens, and the streaming CUDA-core path is kept to
    decode-sized work.  T=None asks about the layer only.  Every case generated
    from this must run: a path the library refuses for it fails the test."""
    lowbit = spec.expert_format != "dense"
    tc = spec.dtype == "bf16" and spec.hidden % 64 == 0 and spec.expert_ff % 64 == 0 and spec.shared_ff % 64 == 0
    if path == moe.PATH_FUSED:
        return not lowbit and spec.expert_ff % 16 == 0 and (T is None or T <= FUSED_MAX_TOKENS)
    if path == moe.PATH_STREAM:
        return not lowbit and (T is None or _flops(spec, T) <= STREAM_MAX_FLOP)
    if path == moe.PATH_DECODE_TC:
        return tc and (T is None or T <= DECODE_TC_MAX_TOKENS)
    return path == moe.PATH_AUTO or tc


PARITY = [pytest.param(name, T, n_rows, path, id=f"{pid}-{name}-T{T}")
          for name, T, n_rows in CASES for path, pid in zip(PATHS, PATH_IDS)
          if _applies(synth.WORKLOADS[name][0], path, T)]


@pytest.mark.parametrize("name,T,n_rows,path", PARITY)
def test_layer_parity(name, T, n_rows, path):
    wl = workload(name)
    spec = wl.spec
    wl.layer.set_path(path)
    x = wl.x[:T]
    out = wl.layer.forward(wl.x_dev[:T])
    idx, wt = wl.layer.routing(T)
    torch.cuda.synchronize()
    wl.layer.status()
    out = out.cpu().numpy()
    idx = idx.cpu().numpy()
    wt = wt.cpu().numpy()

    # selection on every token
    mism, ties, invalid, logits = helpers.index_parity_all(wl.orc, x, idx)
    assert not mism, f"expert indices differ without a near tie at tokens {mism[:10]}"
    assert not invalid, f"near-tie tokens with an invalid selection: {invalid[:10]}"
    if ties:
        print(f"[{name} T={T}] near ties reported (not failed): {ties[:10]}")
    # routing weights and logits as intermediates
    ok = np.array([t not in set(ties) for t in range(T)])
    for t in np.flatnonzero(ok)[:256]:
        _, w_ref = wl.orc.select(logits[t])
        np.testing.assert_allclose(wt[t], w_ref, rtol=2e-5, atol=2e-6)
    gl, _ = wl.layer.logits(T)
    gl = gl.cpu().numpy()
    scale = np.abs(logits).max()
    assert np.abs(gl - logits).max() <= 1e-5 * max(scale, 1.0)
    # expert histogram (bit-exact when no near tie changed a selection)
    if not ties:
        counts = wl.layer.expert_counts().cpu().numpy()
        ref_counts = np.bincount(idx.reshape(-1), minlength=spec.n_expert)
        np.testing.assert_array_equal(counts, ref_counts)

    rows = helpers.sample_rows(T, n_rows)
    rep = helpers.compare(wl.orc, x, rows, out[rows], idx[rows])
    print(f"[{name} T={T} path={path}] {rep}")
    assert rep.ok(spec.dtype), str(rep)


DETERMINISM = [
    ("qwen_prefill_zipf", 1024, moe.PATH_STREAM), ("qwen_prefill_zipf", 1024, moe.PATH_TC),
    ("qwen_prefill_zipf", 8, moe.PATH_FUSED), ("qwen_prefill_zipf", 8, moe.PATH_DECODE_TC),
    # low-bit experts: the widening warps' rings and the split-K sums of both
    # tensor-core paths, at sizes with many stages per CTA
    ("gptoss_q4", 2048, moe.PATH_TC), ("gptoss_q4", 16, moe.PATH_DECODE_TC),
    ("gptoss_mxfp4", 64, moe.PATH_TC), ("gptoss_mxfp4", 16, moe.PATH_DECODE_TC),
    ("qwen_q4", 8, moe.PATH_DECODE_TC), ("qwen_q4", 300, moe.PATH_TC),
]


@pytest.mark.parametrize("name,T,path", DETERMINISM,
                         ids=[f"{n}-T{T}-{PATH_IDS[PATHS.index(p)]}" for n, T, p in DETERMINISM])
def test_deterministic_bitwise(name, T, path):
    """The same input gives the same bits on every forward (no race, and no
    reduction whose order depends on scheduling)."""
    wl = workload(name)
    wl.layer.set_path(path)
    a = wl.layer.forward(wl.x_dev[:T]).clone()
    for _ in range(4):
        b = wl.layer.forward(wl.x_dev[:T])
        torch.cuda.synchronize()
        assert torch.equal(a, b)


def test_forward_host_matches_forward():
    wl = workload("qwen_decode")
    wl.layer.set_path(moe.PATH_AUTO)
    T = 8
    dev = wl.layer.forward(wl.x_dev[:T]).cpu()
    x_host = helpers.to_torch(wl.x[:T], device="cpu").pin_memory()
    out_host = torch.empty((T, wl.spec.hidden), dtype=torch.float32).pin_memory()
    s = torch.cuda.current_stream()
    wl.layer.forward_host(x_host, out_host, s)
    s.synchronize()
    assert torch.equal(dev, out_host)


def test_forward_host_back_to_back():
    """Several host-buffer forwards queued without a synchronisation between
    them (the input copies overlap the work queued before them) give each
    batch's own result."""
    wl = workload("qwen_decode")
    wl.layer.set_path(moe.PATH_AUTO)
    T, n = 8, 4
    x_host = helpers.to_torch(synth.make_x(wl.spec, T * n, seed=7), device="cpu").pin_memory()
    outs = [torch.empty((T, wl.spec.hidden), dtype=torch.float32).pin_memory() for _ in range(n)]
    s = torch.cuda.current_stream()
    for i in range(n):
        wl.layer.forward_host(x_host[i * T:(i + 1) * T], outs[i], s)
    s.synchronize()
    for i in range(n):
        ref = wl.layer.forward(x_host[i * T:(i + 1) * T].cuda()).cpu()
        assert torch.equal(ref, outs[i]), i


def test_zero_tokens_and_too_many():
    wl = workload("qwen_decode")
    empty = torch.empty((0, wl.spec.hidden), dtype=torch.bfloat16, device="cuda")
    out = wl.layer.forward(empty)
    assert out.shape == (0, wl.spec.hidden)
    too_many = torch.zeros((wl.Tmax + 1, wl.spec.hidden), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe.MoEError) as ei:
        wl.layer.forward(too_many)
    assert ei.value.status == moe.ERR_TOO_MANY_TOKENS


def test_misaligned_and_overlapping_pointers_rejected():
    wl = workload("qwen_decode")
    H = wl.spec.hidden
    buf = torch.zeros((4 * H + 8,), dtype=torch.bfloat16, device="cuda")
    lib = moe.load_library()
    out = torch.empty((2, H), dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    rc = lib.moe_forward(wl.layer._h, buf.data_ptr() + 2, 2, out.data_ptr(), s)
    assert rc == moe.ERR_INVALID_ARG
    both = torch.zeros((4 * H,), dtype=torch.float32, device="cuda")
    rc = lib.moe_forward(wl.layer._h, both.data_ptr(), 2, both.data_ptr() + 16, s)
    assert rc == moe.ERR_INVALID_ARG


def _small_case(spec, T, path, seed=21, out_dtype="f32", mutate=None, repeats=0):
    if path == moe.PATH_FUSED and T > FUSED_MAX_TOKENS:
        T = 7  # a ragged decode batch
    if path == moe.PATH_DECODE_TC and T > DECODE_TC_MAX_TOKENS:
        T = 13
    w = synth.make_weights(spec, seed=seed)
    if mutate:
        mutate(w)
    x = synth.make_x(spec, T, seed=seed)
    layer = helpers.make_layer(spec, w, T, out_dtype=out_dtype)
    try:
        layer.set_path(path)
        xt = helpers.to_torch(x)
        out = layer.forward(xt).float().cpu().numpy()
        for _ in range(repeats):  # the same bits on every forward
            again = layer.forward(xt).float().cpu().numpy()
            assert np.array_equal(out, again, equal_nan=True)
    except moe.MoEError:
        layer.close()
        raise
    idx, _ = layer.routing(T)
    idx = idx.cpu().numpy()
    layer.status()
    layer.close()
    orc = oracle.Oracle(spec, w)
    mism, ties, invalid, _ = helpers.index_parity_all(orc, x, idx)
    assert not mism and not invalid
    return helpers.compare(orc, x, np.arange(T), out, idx)


EDGE_SPECS = [
    # every expert selected (k = E)
    ("k_equals_E", synth.LayerSpec("k=E", 128, 4, 4, 64, shared_ff=64), 37),
    # one expert: the layer is a dense SwiGLU FFN
    ("single_expert", synth.LayerSpec("E=1", 128, 1, 1, 128), 45),
    # ragged token count spanning several 128-row tiles with a tail
    ("ragged_tail", synth.QWEN.replace(name="qwen-like small", hidden=256, n_expert=16, top_k=4, expert_ff=128,
                                       shared_ff=192), 300),
    # gpt-oss form on a small layer with a ragged tail
    ("gptoss_small", synth.GPTOSS.replace(name="gpt-oss-like small", hidden=192, n_expert=8, top_k=4, expert_ff=128),
     133),
    # fp32 layer larger than the tiny one, unnormalised weights with a scale
    ("f32_unnormalised", synth.LayerSpec("f32 mid", 96, 12, 3, 40, shared_ff=24, norm_topk_prob=False,
                                         weights_scale=2.5, dtype="f32"), 70),
    # MXFP4 experts: every expert selected, a single expert, a ragged tail
    ("mxfp4_k_equals_E", synth.GPTOSS_MXFP4.replace(name="mxfp4 k=E", hidden=128, n_expert=4, top_k=4,
                                                    expert_ff=64), 37),
    ("mxfp4_single_expert", synth.GPTOSS_MXFP4.replace(name="mxfp4 E=1", hidden=192, n_expert=1, top_k=1,
                                                       expert_ff=128), 45),
    ("mxfp4_ragged", synth.GPTOSS_MXFP4.replace(name="mxfp4 small", hidden=192, n_expert=8, top_k=4,
                                                expert_ff=128), 133),
    # Q4 records: every expert selected, a single expert, ragged tails in both forms
    ("q4_k_equals_E", synth.QWEN_Q4.replace(name="q4 k=E", hidden=128, n_expert=4, top_k=4, expert_ff=64), 37),
    ("q4_single_expert", synth.QWEN_Q4.replace(name="q4 E=1", hidden=192, n_expert=1, top_k=1, expert_ff=128), 45),
    ("q4_ragged", synth.QWEN_Q4.replace(name="q4 small", hidden=256, n_expert=16, top_k=4, expert_ff=192), 300),
    ("q4_gptoss_ragged", synth.GPTOSS_Q4.replace(name="q4 gpt-oss-like small", hidden=192, n_expert=8, top_k=4,
                                                 expert_ff=128), 133),
    # more than 128 rows per expert: the low-bit GEMMs' 256-row tiles (two M
    # halves), with ragged second tiles and halves
    ("q4_many_rows", synth.QWEN_Q4.replace(name="q4 many rows", hidden=256, n_expert=4, top_k=2, expert_ff=192), 700),
    ("mxfp4_many_rows", synth.GPTOSS_MXFP4.replace(name="mxfp4 many rows", hidden=192, n_expert=4, top_k=2,
                                                   expert_ff=128), 600),
]

# Deep K (16 K blocks for gate/up, 8 for down) over few tiles, fewer than
# half the SMs, in bf16 and both low-bit forms, with 128- and 256-row tiles
DEEP_K_SPECS = [
    ("deep_k_bf16", synth.QWEN.replace(name="deep K bf16", hidden=1024, n_expert=8, top_k=2, expert_ff=512,
                                      shared_ff=512), 150),
    ("deep_k_q4", synth.QWEN_Q4.replace(name="deep K q4", hidden=1024, n_expert=8, top_k=2, expert_ff=512), 150),
    ("deep_k_q4_two_halves", synth.QWEN_Q4.replace(name="deep K q4 256 rows", hidden=1024, n_expert=4, top_k=2,
                                                  expert_ff=512), 700),
    ("deep_k_mxfp4", synth.GPTOSS_MXFP4.replace(name="deep K mxfp4", hidden=1024, n_expert=8, top_k=4,
                                               expert_ff=512), 64),
]
EDGE_SPECS += DEEP_K_SPECS


EDGE = [pytest.param(name, spec, T, path, id=f"{pid}-{name}")
        for name, spec, T in EDGE_SPECS for path, pid in zip(PATHS, PATH_IDS) if _applies(spec, path)]


@pytest.mark.parametrize("name,spec,T,path", EDGE)
def test_edge_cases(name, spec, T, path):
    rep = _small_case(spec, T, path)
    print(f"[{name} path={path}] {rep}")
    assert rep.ok(spec.dtype), str(rep)


@pytest.mark.parametrize("name,spec,T", DEEP_K_SPECS, ids=[n for n, _, _ in DEEP_K_SPECS])
def test_deep_k_deterministic(name, spec, T):
    rep = _small_case(spec, T, moe.PATH_TC, repeats=3)
    assert rep.ok(spec.dtype), str(rep)


@pytest.mark.parametrize("path", PATHS, ids=PATH_IDS)
def test_all_tokens_to_one_expert(path):
    """Degenerate routing: one router row dominates, so every token picks
    expert 5 first through its router bias (the hot-expert case of a skewed
    load)."""
    spec = synth.LayerSpec("hot expert", 128, 8, 2, 64, shared_ff=64, has_bias=True)

    def mutate(w):
        b = synth.bf16_to_f32(w["router_b"])
        b[5] = 100.0
        w["router_b"] = synth.to_bf16(b)

    rep = _small_case(spec, 260, path, mutate=mutate)
    assert rep.ok(spec.dtype), str(rep)


@pytest.mark.parametrize("T", [5, 24])
def test_bf16_output(T):
    spec = synth.QWEN.replace(name="qwen-like bf16 out", hidden=256, n_expert=32, top_k=8, expert_ff=128,
                              shared_ff=128)
    rep = _small_case(spec, T, moe.PATH_AUTO, out_dtype="bf16")
    assert rep.ok("bf16"), str(rep)


def test_fused_path_rejects_large_batches():
    spec = synth.TINY
    w = synth.make_weights(spec, seed=3)
    layer = helpers.make_layer(spec, w, 16)
    layer.set_path(moe.PATH_FUSED)
    x = helpers.to_torch(synth.make_x(spec, 16, seed=3))
    with pytest.raises(moe.MoEError) as ei:
        layer.forward(x)
    assert ei.value.status == moe.ERR_UNSUPPORTED
    layer.forward(x[:8])
    torch.cuda.synchronize()
    layer.close()


def test_paths_agree_on_decode_batch():
    """The three kernel paths give the same selection and outputs within the
    bf16 bar on one decode batch."""
    wl = workload("qwen_decode")
    outs = {}
    for path in PATHS:
        wl.layer.set_path(path)
        outs[path] = wl.layer.forward(wl.x_dev[:8]).cpu().numpy().astype(np.float64)
        idx, _ = wl.layer.routing(8)
        outs[(path, "idx")] = idx.cpu().numpy()
    wl.layer.set_path(moe.PATH_AUTO)
    for path in PATHS[1:]:
        np.testing.assert_array_equal(outs[(path, "idx")], outs[(PATHS[0], "idx")])
        ref = outs[PATHS[0]]
        assert np.linalg.norm(outs[path] - ref) <= 1e-2 * np.linalg.norm(ref)


MXFP4_SMALL = synth.GPTOSS_MXFP4.replace(name="gpt-oss-like, MXFP4 experts, small", hidden=256, n_expert=8, top_k=2,
                                         expert_ff=192)


@pytest.mark.parametrize("scales", ["synthetic", "spread_100_150", "edges"])
@pytest.mark.parametrize("T", [5, 200])
def test_mxfp4_scales_take_the_packed_path(scales, T):
    """MXFP4 experts stay packed for every scale byte: a decode batch runs the
    kernel that streams the codes and scales (timed as its own kind) and a
    prefill batch the grouped GEMMs that widen them, and both agree with the
    oracle on the same weights -- with the synthetic scales, with scales
    spread over 100..150, and with the edge bytes 1 (subnormal products), 113
    and 140, and 254 on blocks whose codes are all zero (so that no product
    leaves the fp32 range)."""
    spec = MXFP4_SMALL
    w = synth.make_weights(spec, seed=5)
    if scales == "spread_100_150":
        for name in ("gate_up_scales", "down_scales"):
            r = synth.u64(w[name].size, 5, 77 if name == "down_scales" else 76)
            w[name] = (100 + (r % np.uint64(51))).astype(np.uint8).reshape(w[name].shape)
    if scales == "edges":
        for name, blocks in (("gate_up_scales", "gate_up_blocks"), ("down_scales", "down_blocks")):
            sc = w[name].copy()
            sc.flat[3::97] = 113
            sc.flat[11::89] = 140
            sc.flat[5::53] = 1
            b = w[blocks].copy().reshape(-1, 16)
            zero = np.arange(sc.size)[7::61]
            sc.flat[zero] = 254
            b[zero] = 0
            w[name], w[blocks] = sc, b.reshape(w[blocks].shape)
    x = synth.make_x(spec, T, seed=5)
    layer = helpers.make_layer(spec, w, T)
    layer.timing_enable(4)
    out = layer.forward(helpers.to_torch(x)).float().cpu().numpy()
    kinds = layer.timing_read()
    idx, _ = layer.routing(T)
    idx = idx.cpu().numpy()
    layer.status()
    layer.close()
    if T <= DECODE_TC_MAX_TOKENS:
        assert kinds["experts_mxfp4"][1] == 1 and kinds["experts"][1] == 0, kinds
    else:
        assert kinds["up"][1] == 1 and kinds["down"][1] == 1, kinds
    orc = oracle.Oracle(spec, w)
    mism, ties, invalid, _ = helpers.index_parity_all(orc, x, idx)
    assert not mism and not invalid
    rep = helpers.compare(orc, x, np.arange(T), out, idx)
    assert rep.ok(spec.dtype), str(rep)


def test_mxfp4_layer_keeps_only_the_packed_experts():
    """An MXFP4 gpt-oss-shaped layer holds its experts as codes and scales:
    its device bytes are the packed experts plus the rest of the layer and the
    workspace, far below the bf16 experts' 1.6 GB."""
    spec = synth.GPTOSS_MXFP4
    w = synth.make_weights(spec, seed=0)
    layer = helpers.make_layer(spec, w, 16)
    nbytes = layer.device_bytes
    layer.close()
    E, H, F = spec.n_expert, spec.hidden, spec.expert_ff
    packed = E * 3 * H * F * (0.5 + 1 / 32)          # 423 MB
    bf16_experts = E * 3 * H * F * 2                 # 1.59 GB
    assert packed <= nbytes <= packed + 0.1e9, (nbytes, packed)
    assert nbytes < 0.3 * bf16_experts


@pytest.mark.parametrize("T", [1, 7, 16])
def test_mxfp4_small_layer_paths_agree(T):
    """Ragged batches on a small MXFP4 layer: both tensor-core paths (the
    weight-streaming decode kernel and the grouped GEMMs) give the oracle's
    result; the CUDA-core paths, which read bf16 or fp32 weights only, are
    refused."""
    for path in (moe.PATH_DECODE_TC, moe.PATH_TC):
        rep = _small_case(MXFP4_SMALL, T, path, seed=9)
        assert rep.ok(MXFP4_SMALL.dtype), (path, str(rep))
    layer = helpers.make_layer(MXFP4_SMALL, synth.make_weights(MXFP4_SMALL, seed=9), T)
    for path in (moe.PATH_STREAM, moe.PATH_FUSED):
        with pytest.raises(moe.MoEError) as ei:
            layer.set_path(path)
        assert ei.value.status == moe.ERR_UNSUPPORTED
    layer.close()


Q4_SMALL = synth.QWEN_Q4.replace(name="qwen-like, Q4 expert records, small", hidden=256, n_expert=8, top_k=2,
                                 expert_ff=192)


def _q4_records(w):
    return [n for n in w if n.endswith("_q4")]


@pytest.mark.parametrize("scales", ["synthetic", "edges"])
@pytest.mark.parametrize("T", [5, 200])
def test_q4_scales_take_the_packed_path(scales, T):
    """Q4 records stay packed: a decode batch runs the kernel that streams them
    (timed as its own kind) and a prefill batch the grouped GEMMs that widen
    them; both agree with the oracle on the same records -- with the synthetic
    scales, and with edge scales: 0, negative, the smallest binary16
    subnormal, the largest finite binary16 (65504) on blocks of codes 8 (value
    0), and blocks whose codes are all 0 or all 15 (values -8 d and 7 d)."""
    spec = Q4_SMALL
    w = synth.make_weights(spec, seed=6)
    if scales == "edges":
        for name in _q4_records(w):
            r = w[name].copy().reshape(-1, 18)
            d = r[:, 0].astype(np.uint16) | (r[:, 1].astype(np.uint16) << 8)
            d[3::97] = 0x0000                       # 0
            d[11::89] = d[11::89] | 0x8000          # negative
            d[5::53] = 0x0001                       # 2^-24
            r[19::71, 2:] = 0x00                    # codes 0: -8 d
            r[23::67, 2:] = 0xFF                    # codes 15: 7 d
            big = np.arange(d.size)[7::61]
            d[big] = 0x7BFF                         # 65504
            r[big, 2:] = 0x88                       # codes 8: value 0
            r[:, 0] = (d & 0xFF).astype(np.uint8)
            r[:, 1] = (d >> 8).astype(np.uint8)
            w[name] = r.reshape(w[name].shape)
    x = synth.make_x(spec, T, seed=6)
    layer = helpers.make_layer(spec, w, T)
    layer.timing_enable(4)
    out = layer.forward(helpers.to_torch(x)).float().cpu().numpy()
    kinds = layer.timing_read()
    idx, _ = layer.routing(T)
    idx = idx.cpu().numpy()
    layer.status()
    layer.close()
    if T <= DECODE_TC_MAX_TOKENS:
        assert kinds["experts_q4"][1] == 1 and kinds["experts"][1] == 0 and kinds["experts_mxfp4"][1] == 0, kinds
    else:
        assert kinds["up"][1] == 1 and kinds["down"][1] == 1, kinds
    orc = oracle.Oracle(spec, w)
    mism, ties, invalid, _ = helpers.index_parity_all(orc, x, idx)
    assert not mism and not invalid
    rep = helpers.compare(orc, x, np.arange(T), out, idx)
    print(f"[q4 {scales} T={T}] {rep}")
    assert rep.ok(spec.dtype), str(rep)


def test_q4_layer_keeps_only_the_packed_experts():
    """A Q4 gpt-oss-shaped layer holds its experts as 4.5-bit records: its
    device bytes are the packed experts plus the rest of the layer and the
    workspace."""
    spec = synth.GPTOSS_Q4
    w = synth.make_weights(spec, seed=0)
    layer = helpers.make_layer(spec, w, 16)
    nbytes = layer.device_bytes
    layer.close()
    E, H, F = spec.n_expert, spec.hidden, spec.expert_ff
    packed = E * 3 * H * F * (0.5 + 2 / 32)          # 448 MB: 0.28 of the bf16 experts
    bf16_experts = E * 3 * H * F * 2                 # 1.59 GB
    assert packed <= nbytes <= packed + 0.1e9, (nbytes, packed)
    assert nbytes < 0.35 * bf16_experts


@pytest.mark.parametrize("T", [1, 7, 16])
def test_q4_small_layer_paths_agree(T):
    """Ragged batches on a small Q4 layer: both tensor-core paths give the
    oracle's result; the CUDA-core paths are refused."""
    for path in (moe.PATH_DECODE_TC, moe.PATH_TC):
        rep = _small_case(Q4_SMALL, T, path, seed=10)
        assert rep.ok(Q4_SMALL.dtype), (path, str(rep))
    layer = helpers.make_layer(Q4_SMALL, synth.make_weights(Q4_SMALL, seed=10), T)
    for path in (moe.PATH_STREAM, moe.PATH_FUSED):
        with pytest.raises(moe.MoEError) as ei:
            layer.set_path(path)
        assert ei.value.status == moe.ERR_UNSUPPORTED
    layer.close()


def _bf16_bits_to_f32(a):
    return (a.astype(np.uint32) << 16).view(np.float32)


INTER_CASES = [
    # name, tokens, path, routed rows sampled, shared rows sampled
    ("tiny", 16, moe.PATH_STREAM, 32, 0),
    ("qwen_prefill_zipf", 4096, moe.PATH_TC, 48, 8),
    ("qwen_prefill_zipf", 300, moe.PATH_STREAM, 32, 8),
    ("gptoss", 64, moe.PATH_TC, 24, 0),
    ("mixtral", 256, moe.PATH_TC, 12, 0),
    ("gptoss_mxfp4", 64, moe.PATH_TC, 16, 0),
    ("qwen_q4", 300, moe.PATH_TC, 24, 0),
]


@pytest.mark.parametrize("name,T,path,n_routed,n_shared", INTER_CASES,
                         ids=[f"{c[0]}-T{c[1]}-{'tc' if c[2] == moe.PATH_TC else 'stream'}" for c in INTER_CASES])
def test_intermediates_match_oracle(name, T, path, n_routed, n_shared):
    """Each grouped-path intermediate against the oracle: the expert offsets
    and the pair permutation bit-exact with a stable sort of the selection by
    expert; the activations h of sampled routed rows (and shared-expert rows)
    against the oracle's expert evaluation at the parity tolerance; and, where
    the path keeps them, the weighted per-slot outputs."""
    wl = workload(name)
    spec = wl.spec
    wl.layer.set_path(path)
    x = wl.x[:T]
    wl.layer.forward(wl.x_dev[:T])
    idx, wt = wl.layer.routing(T)
    torch.cuda.synchronize()
    wl.layer.status()
    idx, wt = idx.cpu().numpy(), wt.cpu().numpy()
    E, K, H, F, Fs = spec.n_expert, spec.top_k, spec.hidden, spec.expert_ff, spec.shared_ff
    Fmax = max(F, Fs)
    mism, ties, invalid, logits = helpers.index_parity_all(wl.orc, x, idx)
    assert not mism and not invalid
    # the grouping of the selection (the oracle's, which equals the GPU's off near ties)
    sel = idx if ties else np.stack([wl.orc.select(logits[t])[0] for t in range(T)])
    offsets = wl.layer.intermediate(moe.INTER_OFFSETS).cpu().numpy().view(np.int32)
    perm = wl.layer.intermediate(moe.INTER_PERM).cpu().numpy().view(np.int32)
    counts = np.bincount(sel.reshape(-1), minlength=E)
    np.testing.assert_array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
    np.testing.assert_array_equal(perm, np.argsort(sel.reshape(-1), kind="stable"))

    raw = wl.layer.intermediate(moe.INTER_H).cpu().numpy()
    rows = T * K + (T if Fs else 0)
    h = (_bf16_bits_to_f32(raw.view(np.uint16)) if spec.dtype == "bf16" else raw.view(np.float32)).reshape(rows, Fmax)
    xf = synth.as_f32(np.ascontiguousarray(x), spec.dtype).astype(np.float64)
    pick = helpers.sample_rows(T * K, n_routed, seed=7)
    got, ref, yref, ykey = [], [], [], []
    for j in pick:
        p = int(perm[j])
        t, slot = divmod(p, K)
        hr, yr = wl.orc.expert(int(idx[t, slot]), xf[t])
        got.append(h[j, :F])
        ref.append(hr)
        w_ref = wl.orc.weights_for_selection(logits[t], idx[t])
        yref.append(w_ref[slot] * yr)
        ykey.append((t, slot))
    for t in (helpers.sample_rows(T, n_shared, seed=8) if Fs else []):
        hr, yr, g = wl.orc.shared(xf[t])
        got.append(h[T * K + t, :Fs])
        ref.append(hr)
        yref.append(g * yr)
        ykey.append((int(t), K))
    got, ref = np.concatenate(got).astype(np.float64), np.concatenate(ref)
    tol = helpers.REL_L2[spec.dtype]
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel <= tol, f"h rel-L2 {rel:.3e}"
    assert np.abs(got - ref).max() <= helpers.MAX_ABS_FRAC * np.abs(ref).max()

    if path == moe.PATH_STREAM:
        ys = wl.layer.intermediate(moe.INTER_YS).cpu().numpy().view(np.float32).reshape(T, K + 1, H)
        gy = np.concatenate([ys[t, s] for t, s in ykey]).astype(np.float64)
        ry = np.concatenate(yref)
        rel = np.linalg.norm(gy - ry) / np.linalg.norm(ry)
        assert rel <= tol, f"Ys rel-L2 {rel:.3e}"
        assert np.abs(gy - ry).max() <= helpers.MAX_ABS_FRAC * np.abs(ry).max()
    wl.layer.set_path(moe.PATH_AUTO)
