"""moe_route_noalloc: the routing step for callers that cannot allocate device
memory (an application that hands all device memory out of its own pool, an
allocator frozen after start-up, a real-time loop).  It keeps its logits in a
static device array instead of a layer's workspace.  Its routing is checked
against the oracle and against what moe_forward reports through
moe_get_routing.

This file is collected last so that, in a run stopping at the first failure,
every other test has already run.  It creates its own layers, so it passes
alone in a fresh process as well as after the other tests."""
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

# the tolerance the parity tests use for routing weights
W_RTOL, W_ATOL = 2e-5, 2e-6

SPECS = [
    # softmax -> top-8 -> renormalise, 256 experts (the router is full size)
    synth.QWEN.replace(name="qwen-like router", expert_ff=64, shared_ff=64),
    # top-4 -> softmax over the 4, router bias
    synth.GPTOSS.replace(name="gpt-oss-like router", expert_ff=64),
    # fp32, unnormalised weights with a scale
    synth.TINY.replace(name="tiny unnormalised", norm_topk_prob=False, weights_scale=2.5),
]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_mixture_experts_gb300 import build
    build.build()


def _noalloc(lib, spec, x_dev, router_w, router_b, stream):
    T, k, E = x_dev.shape[0], spec.top_k, spec.n_expert
    idx = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
    w = torch.full((T, k), -1.0, dtype=torch.float32, device="cuda")
    counts = torch.full((E,), -7, dtype=torch.int32, device="cuda")
    rc = lib.moe_route_noalloc(
        x_dev.data_ptr(), router_w.data_ptr(), router_b.data_ptr() if router_b is not None else None, T,
        spec.hidden, E, k, moe.ROUTER_SOFTMAX_TOPK if spec.router_mode == "softmax_topk" else moe.ROUTER_TOPK_SOFTMAX,
        int(spec.norm_topk_prob), float(spec.weights_scale), moe.DT_BF16 if spec.dtype == "bf16" else moe.DT_F32,
        idx.data_ptr(), w.data_ptr(), counts.data_ptr(), stream.cuda_stream)
    assert rc == moe.OK, lib.moe_last_error()
    return idx, w, counts


@pytest.mark.parametrize("spec", SPECS, ids=lambda s: s.name)
def test_route_noalloc_matches_forward_routing(spec):
    """Two calls in a row (different tokens; the shared scratch keeps the last
    call's logits and must not leak into the next call).  Each call's routing
    is checked against the oracle (indices bit-exact, near ties reported, and
    weights within the parity tests' tolerance) and against what moe_forward
    reports for the same tokens.  The two entry points sum the router's dot
    products in different orders, so they may disagree only on near-tie
    tokens, and there each selection must be a valid top-k."""
    lib = moe.load_library()
    weights = synth.make_weights(spec, seed=4)
    orc = oracle.Oracle(spec, weights)
    T = 24
    layer = helpers.make_layer(spec, weights, T)
    router_w = helpers.to_torch(weights["router_w"])
    router_b = helpers.to_torch(weights["router_b"]) if "router_b" in weights else None
    stream = torch.cuda.current_stream()
    for call, n_tok in enumerate((T, 17)):
        x_np = synth.make_x(spec, n_tok, seed=100 + call)
        x = helpers.to_torch(x_np)
        layer.forward(x)
        ref_idx, ref_w = layer.routing(n_tok)
        idx, w, counts = _noalloc(lib, spec, x, router_w, router_b, stream)
        torch.cuda.synchronize()
        idx, w, counts = idx.cpu().numpy(), w.cpu().numpy(), counts.cpu().numpy()
        ref_idx, ref_w = ref_idx.cpu().numpy(), ref_w.cpu().numpy()

        # against the oracle
        mism, ties, invalid, logits = helpers.index_parity_all(orc, x_np, idx)
        assert not mism, f"call {call}: indices differ from the oracle without a near tie at {mism}"
        assert not invalid, f"call {call}: near-tie tokens with an invalid selection: {invalid}"
        if ties:
            print(f"[{spec.name} call {call}] near ties reported (not failed): {ties}")
        for t in range(n_tok):
            if t in ties:
                continue
            _, w_ref = orc.select(logits[t])
            np.testing.assert_allclose(w[t], w_ref, rtol=W_RTOL, atol=W_ATOL)
        np.testing.assert_array_equal(counts, np.bincount(idx.reshape(-1), minlength=spec.n_expert))

        # against moe_forward's routing
        differ = [t for t in range(n_tok) if not np.array_equal(idx[t], ref_idx[t])]
        mism_f, ties_f, invalid_f, _ = helpers.index_parity_all(orc, x_np, ref_idx)
        assert not mism_f and not invalid_f
        assert set(differ) <= set(ties) | set(ties_f), f"call {call}: entry points disagree off near ties: {differ}"
        same = [t for t in range(n_tok) if t not in differ]
        np.testing.assert_allclose(w[same], ref_w[same], rtol=W_RTOL, atol=W_ATOL)
    layer.close()


def test_route_noalloc_rejects_sizes_beyond_its_scratch():
    lib = moe.load_library()
    E, H = 256, 64
    T = 262144 // E + 1
    x = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
    rw = torch.zeros((E, H), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((T, 8), dtype=torch.int32, device="cuda")
    w = torch.empty((T, 8), dtype=torch.float32, device="cuda")
    counts = torch.empty((E,), dtype=torch.int32, device="cuda")
    rc = lib.moe_route_noalloc(x.data_ptr(), rw.data_ptr(), None, T, H, E, 8, moe.ROUTER_SOFTMAX_TOPK, 1, 1.0,
                               moe.DT_BF16, idx.data_ptr(), w.data_ptr(), counts.data_ptr(),
                               torch.cuda.current_stream().cuda_stream)
    assert rc == moe.ERR_TOO_MANY_TOKENS
    assert b"scratch" in lib.moe_last_error()
