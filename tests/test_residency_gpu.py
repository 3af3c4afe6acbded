"""GPU tests of expert residency (config.resident_experts = S > 0): the
routed experts live in pinned host memory, S device slots hold the resident
ones, and every chunk of up to 16 tokens copies its missing experts into the
least recently used free slots before the weight-streaming kernel runs.

* outputs are bitwise those of the same layer with every expert resident
  (the same kernel, the same arithmetic order, only the weight addresses
  differ), and agree with the oracle;
* the slot table and the hit / miss / byte counters follow the policy's
  definition, simulated here from the layer's own selections;
* bf16, MXFP4 and Q4 experts; batches of 1, 5, 16 and several chunks."""
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

# E above 16 * top_k, so that S can sit below E
BF16 = synth.QWEN.replace(name="qwen-like, 128 experts", hidden=256, n_expert=128, top_k=2, expert_ff=128,
                          shared_ff=128)
MXFP4 = synth.GPTOSS_MXFP4.replace(name="gpt-oss-like, MXFP4, 64 experts", hidden=256, n_expert=64, top_k=2,
                                   expert_ff=192)
Q4 = synth.QWEN_Q4.replace(name="qwen-like, Q4, 64 experts", hidden=256, n_expert=64, top_k=2, expert_ff=128)
BATCHES = (1, 5, 16, 37, 3, 16)


def _layers(spec, S, seed, Tmax=48):
    import dataclasses
    w = synth.make_weights(spec, seed=seed)
    full = helpers.make_layer(spec, w, Tmax)
    cfg = dataclasses.replace(helpers.moe_config(spec, Tmax), resident_experts=S)
    wt = {k: helpers.to_torch(v) for k, v in w.items()}
    if spec.expert_format == "mxfp4":
        wt["gate_up_w"] = wt.pop("gate_up_blocks")
        wt["down_w"] = wt.pop("down_blocks")
    elif spec.expert_format == "q4":
        for n in [n for n in wt if n.endswith("_q4")]:
            wt[n[:-3]] = wt.pop(n)
    res = moe.MoELayer(cfg, wt)
    return w, full, res


def _simulate(S, chunks):
    """The policy's definition: per chunk, hits stamp their slots; the misses,
    in ascending expert order, take the slots with the lowest (stamp, slot)."""
    expert_of = list(range(S))
    slot_of = {e: e for e in range(S)}
    last = [0] * S
    hits = misses = 0
    for stamp, sel in enumerate(chunks, 1):
        miss = []
        for e in sorted(sel):
            if e in slot_of:
                last[slot_of[e]] = stamp
                hits += 1
            else:
                miss.append(e)
        order = sorted(range(S), key=lambda v: (last[v], v))
        for r, e in enumerate(miss):
            v = order[r]
            assert last[v] < stamp
            slot_of.pop(expert_of[v], None)
            expert_of[v] = e
            slot_of[e] = v
            last[v] = stamp
        misses += len(miss)
    return expert_of, hits, misses


@pytest.mark.parametrize("spec,S", [(BF16, 40), (BF16, 100), (MXFP4, 40), (Q4, 33)],
                         ids=["bf16-S40", "bf16-S100", "mxfp4-S40", "q4-S33"])
def test_streamed_experts_match_the_resident_layer(spec, S):
    w, full, res = _layers(spec, S, seed=4)
    orc = oracle.Oracle(spec, w)
    x_all = synth.make_x(spec, sum(BATCHES), seed=4)
    chunks = []
    t = 0
    E, H = spec.n_expert, spec.hidden
    per_expert = 3 * H * spec.expert_ff * {"mxfp4": 0.5 + 1 / 32, "q4": 0.5 + 2 / 32}.get(spec.expert_format, 2)
    for T in BATCHES:
        x = x_all[t:t + T]
        t += T
        xd = helpers.to_torch(x)
        # the resident layer on the same chunks of 16 (a longer batch would take its prefill path)
        a = torch.cat([full.forward(xd[c0:c0 + 16]).clone() for c0 in range(0, T, 16)])
        b = res.forward(xd).clone()
        idx, _ = res.routing(T)
        torch.cuda.synchronize()
        res.status()
        assert torch.equal(a, b), f"T={T}: streamed layer differs from the resident one"
        idx = idx.cpu().numpy()
        for c0 in range(0, T, 16):
            chunks.append(set(idx[c0:c0 + 16].reshape(-1).tolist()))
        rep = helpers.compare(orc, x, np.arange(T), b.cpu().numpy(), idx)
        assert rep.ok(spec.dtype), str(rep)
    slots, stats = res.residency()
    want_slots, want_hits, want_misses = _simulate(S, chunks)
    assert slots == want_slots
    assert stats["hits"] == want_hits and stats["misses"] == want_misses
    assert stats["bytes"] == want_misses * int(per_expert)
    assert want_misses > 0  # the sequence did stream experts in
    full.close()
    res.close()


def test_streamed_layer_keeps_only_its_slots():
    _, full, res = _layers(BF16, 40, seed=1)
    E, H, F = BF16.n_expert, BF16.hidden, BF16.expert_ff
    per_expert = 3 * H * F * 2
    saved = full.device_bytes - res.device_bytes
    # the experts left out, less the slot tables (a few KB)
    assert (E - 40) * per_expert - 65536 <= saved <= (E - 40) * per_expert
    full.close()
    res.close()


def test_streamed_layer_refuses_the_other_paths():
    _, full, res = _layers(BF16, 40, seed=2)
    for path in (moe.PATH_STREAM, moe.PATH_TC, moe.PATH_FUSED):
        with pytest.raises(moe.MoEError) as ei:
            res.set_path(path)
        assert ei.value.status == moe.ERR_UNSUPPORTED
    res.set_path(moe.PATH_DECODE_TC)
    res.set_path(moe.PATH_AUTO)
    with pytest.raises(moe.MoEError) as ei:
        full.residency()
    assert ei.value.status == moe.ERR_UNSUPPORTED
    full.close()
    res.close()


def test_streamed_layer_timing_kinds():
    """A forward of 20 tokens runs two chunks, each a router, a residency step
    (slot assignment + copies) and an experts kernel."""
    w, full, res = _layers(BF16, 40, seed=3)
    x = helpers.to_torch(synth.make_x(BF16, 20, seed=3))
    res.timing_enable(2)
    res.forward(x)
    kinds = res.timing_read()
    assert kinds["router"][1] == 2 and kinds["residency"][1] == 2 and kinds["experts"][1] == 2, kinds
    assert res.last_launch_count == 2 * 4
    full.close()
    res.close()
