"""Failure detection without a GPU fault ("Qwen3.5-MoE Model Implementation",
Gotchas and Fragile Spots: failure modes must not be silent).

Every wait of the layer's kernels on another thread block is bounded.  Test-only
fault injection makes one forward wait for a condition nothing satisfies -- a
grid barrier one arrival short (fused cooperative decode kernel), a group's
activations one tile short (weight-streaming tensor-core decode kernel), a
device word that stays zero (tensor-core GEMMs) -- with a 1 ms limit.  The wait
runs out, the kernels stop issuing work and drain what they have in flight,
moe_get_status reports MOE_ERR_DEVICE_TIMEOUT, and the next forward, without
injection, gives the same bits as before and the oracle's result."""
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

SPEC = synth.QWEN.replace(name="qwen-like small", hidden=256, n_expert=16, top_k=4, expert_ff=128, shared_ff=128)
CASES = [("fused", moe.PATH_FUSED, 5), ("dectc", moe.PATH_DECODE_TC, 8), ("tc", moe.PATH_TC, 200)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_mixture_experts_gb300 import build
    build.build()


@pytest.mark.parametrize("name,path,T", CASES, ids=[c[0] for c in CASES])
def test_injected_wait_runs_out_and_the_layer_recovers(name, path, T):
    w = synth.make_weights(SPEC, seed=11)
    x = synth.make_x(SPEC, T, seed=11)
    layer = helpers.make_layer(SPEC, w, T)
    try:
        layer.set_path(path)
    except moe.MoEError:
        layer.close()
        raise
    xd = helpers.to_torch(x)
    ref = layer.forward(xd).clone()
    torch.cuda.synchronize()
    layer.status()
    layer.set_wait_limit(1_000_000)  # 1 ms
    for _ in range(2):
        layer.set_fault_injection(True)
        layer.forward(xd)
        with pytest.raises(moe.MoEError) as ei:
            layer.status()
        assert ei.value.status == moe.ERR_DEVICE_TIMEOUT, str(ei.value)
        layer.set_fault_injection(False)
        out = layer.forward(xd).clone()
        torch.cuda.synchronize()
        layer.status()
        assert torch.equal(out, ref), "the forward after a timeout differs from the one before"
    layer.set_wait_limit(0)
    idx, _ = layer.routing(T)
    idx = idx.cpu().numpy()
    layer.close()
    rep = helpers.compare(oracle.Oracle(SPEC, w), x, np.arange(T), ref.cpu().numpy(), idx)
    assert rep.ok(SPEC.dtype), str(rep)
