"""Expert parallelism on the host: the index arithmetic of libmoe's
dispatch/combine plan against a brute-force restatement, and two gloo ranks
that exchange token rows and expert outputs through it and reproduce the
oracle's layer output (the oracle stands in for the experts' arithmetic; the
exchange, the permutations and the slot-order combine are what is tested).
No GPU is needed."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_mixture_experts_gb300 import build
    build.build()


def test_contiguous_partition():
    from sparse_mixture_experts_gb300 import expert_parallel as ep
    assert ep.contiguous_partition(8, 2) == [0, 4, 8]
    assert ep.contiguous_partition(10, 4) == [0, 3, 6, 8, 10]
    with pytest.raises(ValueError):
        ep.contiguous_partition(2, 3)


@pytest.mark.parametrize("G,E,seed", [(2, 8, 0), (3, 10, 1), (4, 32, 2), (1, 5, 3)])
def test_plans_against_brute_force(G, E, seed):
    """Simulate the exchange in one process: every rank's pairs, tagged
    (source, position), go out by the send plan; the receiver's order must be
    expert-major, then source, then the source's order, and sending the
    outputs back in arrival order must return every source its own pairs."""
    from sparse_mixture_experts_gb300 import expert_parallel as ep
    rng = np.random.default_rng(seed)
    first = ep.contiguous_partition(E, G)
    counts = [rng.integers(0, 6, size=E).astype(np.int32) for _ in range(G)]
    # each source's pairs in expert order, tagged (source, position, expert)
    sent = []
    for g in range(G):
        experts = np.repeat(np.arange(E), counts[g])
        sent.append([(g, i, int(e)) for i, e in enumerate(experts)])
        sc, sd = ep.send_plan(counts[g], first)
        for r in range(G):
            want = counts[g][first[r]:first[r + 1]].sum()
            assert sc[r] == want and sd[r] == counts[g][:first[r]].sum()
    for r in range(G):
        n_local = first[r + 1] - first[r]
        cf = np.stack([counts[g][first[r]:first[r + 1]] for g in range(G)])
        rc, rd, order, go = ep.recv_plan(cf)
        arrived = []
        for g in range(G):
            sc, sd = ep.send_plan(counts[g], first)
            arrived += sent[g][int(sd[r]):int(sd[r]) + int(sc[r])]
        assert [len(arrived)] == [int(rc.sum())]
        local = [arrived[i] for i in order.tolist()]
        want = sorted(arrived, key=lambda t: (t[2], t[0], t[1]))
        assert local == want
        for e in range(n_local):
            seg = local[int(go[e]):int(go[e + 1])]
            assert all(t[2] == first[r] + e for t in seg)
        # outputs back in arrival order
        back = [None] * len(local)
        for i, o in enumerate(order.tolist()):
            back[o] = local[i]
        assert back == arrived


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


SPEC_ARGS = dict(name="ep small", hidden=64, n_expert=8, top_k=2, expert_ff=32, shared_ff=32)
TOKENS = (37, 20)
FIRST = (0, 3, 8)  # uneven: rank 0 owns experts 0-2, rank 1 owns 3-7


def _ep_rank(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    import synth
    from sparse_mixture_experts_gb300 import expert_parallel as ep
    spec = synth.QWEN.replace(**SPEC_ARGS)
    w = synth.make_weights(spec, seed=3)
    orc = oracle.Oracle(spec, w)
    T = TOKENS[rank]
    x = synth.make_x(spec, T, seed=3, first_token=sum(TOKENS[:rank]))
    xf = synth.as_f32(x, spec.dtype).astype(np.float64)
    ref, idx, wt = orc.forward(x)
    K, E = spec.top_k, spec.n_expert
    # the grouping step: pairs p = t K + slot in a stable order by expert
    perm = np.argsort(idx.reshape(-1), kind="stable")
    counts = np.bincount(idx.reshape(-1), minlength=E).astype(np.int32)
    rows = torch.from_numpy(xf[perm // K])
    par = ep.ExpertParallel(E, first=list(FIRST))
    d = par.dispatch(rows, counts)
    # this rank's experts on the rows it received (the oracle computes them)
    y = torch.zeros((d.rows.shape[0], spec.hidden), dtype=torch.float64)
    go = d.group_offsets.tolist()
    for e in range(par.n_local):
        for i in range(go[e], go[e + 1]):
            y[i] = torch.from_numpy(orc.expert(FIRST[rank] + e, d.rows[i].numpy())[1])
    back = par.combine(y, d).numpy()
    # scatter to (token, slot), weight, combine in slot order, add the shared expert
    ys = np.zeros((T, K, spec.hidden))
    for j, p in enumerate(perm.tolist()):
        t, s = divmod(p, K)
        ys[t, s] = wt[t, s] * back[j]
    out = np.zeros((T, spec.hidden))
    for t in range(T):
        acc = np.zeros(spec.hidden)
        for s in range(K):
            acc = acc + ys[t, s]
        _, ysh, g = orc.shared(xf[t])
        out[t] = acc + g * ysh
    results[rank] = float(np.abs(out - ref).max() / np.abs(ref).max())
    dist.destroy_process_group()


def test_two_gloo_ranks_reproduce_the_oracle():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    results = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_ep_rank, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    assert set(results.keys()) == {0, 1}
    assert max(results.values()) <= 1e-12, dict(results)


def test_plans_reject_bad_partitions_and_counts():
    """Bounds that run past n_expert, descend, or leave experts out are
    refused before any count is read; a count list of the wrong length is
    refused by the binding."""
    import ctypes
    import sparse_mixture_experts_gb300 as moe
    from sparse_mixture_experts_gb300 import expert_parallel as ep
    lib = moe.load_library()
    counts = (ctypes.c_int32 * 8)(*range(8))
    sc, sd = (ctypes.c_int32 * 2)(), (ctypes.c_int32 * 2)()
    for first in ([0, 10, 8], [0, 5, 3, 8][:3], [1, 4, 8], [0, 4, 7]):
        f = (ctypes.c_int32 * len(first))(*first)
        assert lib.moe_ep_send_plan(8, 2, f, counts, sc, sd) == moe.ERR_INVALID_ARG, first
    f = (ctypes.c_int32 * 3)(0, 4, 8)
    assert lib.moe_ep_send_plan(8, 2, f, counts, sc, sd) == moe.OK
    assert list(sc) == [0 + 1 + 2 + 3, 4 + 5 + 6 + 7] and list(sd) == [0, 6]
    with pytest.raises(ValueError):
        ep.send_plan(list(range(7)), [0, 4, 8])
    with pytest.raises(ValueError):
        ep.recv_plan([1, 2, 3])
