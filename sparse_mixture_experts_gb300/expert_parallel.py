"""Expert parallelism across ranks: the exchange of token rows after the
grouping step and of the experts' outputs before the combine.

Rank g owns a contiguous range of the experts.  Every rank routes its own
tokens and groups its (token, slot) pairs by expert (the layer's grouping
step, MOE_INTER_PERM): in that order the pairs are already grouped by owning
rank, so one all-to-all of the rows dispatches them, and one all-to-all in the
other direction brings the outputs back in the same order.  The index
arithmetic (who sends which rows, and the receiver's expert-major order) is in
libmoe (moe_ep_send_plan / moe_ep_recv_plan); torch.distributed carries the
rows (NCCL between GPUs, gloo on the host).  The pages list expert parallelism
as not done ("Phase 19: MoE -- gpt-oss-20b", section 6).
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import torch
import torch.distributed as dist

from . import _check, load_library


def contiguous_partition(n_expert: int, n_ranks: int) -> list:
    """first_expert[n_ranks + 1]: rank g owns [first[g], first[g+1]); the
    remainder of n_expert / n_ranks goes to the lowest ranks."""
    if n_ranks < 1 or n_expert < n_ranks:
        raise ValueError("need 1 <= n_ranks <= n_expert")
    base, extra = divmod(n_expert, n_ranks)
    first = [0]
    for g in range(n_ranks):
        first.append(first[-1] + base + (1 if g < extra else 0))
    return first


def _i32(t: torch.Tensor) -> int:
    return ctypes.c_void_p(t.data_ptr()).value


def send_plan(counts, first):
    """(send_counts[G], send_displs[G]) from the local per-expert counts."""
    lib = load_library()
    G = len(first) - 1
    c = torch.as_tensor(counts, dtype=torch.int32).contiguous().cpu()
    f = torch.tensor(first, dtype=torch.int32)
    if G < 1 or c.dim() != 1 or c.numel() != int(f[-1]):
        raise ValueError("counts must hold one entry per expert of the partition")
    sc = torch.empty(G, dtype=torch.int32)
    sd = torch.empty(G, dtype=torch.int32)
    _check(lib.moe_ep_send_plan(int(f[-1]), G, _i32(f), _i32(c), _i32(sc), _i32(sd)))
    return sc, sd


def recv_plan(counts_from):
    """(recv_counts, recv_displs, order, group_offsets) from the [G][n_local]
    counts the ranks send this one."""
    lib = load_library()
    cf = torch.as_tensor(counts_from, dtype=torch.int32).contiguous().cpu()
    if cf.dim() != 2:
        raise ValueError("counts_from must be [n_ranks][n_local]")
    G, n_local = cf.shape
    rc = torch.empty(G, dtype=torch.int32)
    rd = torch.empty(G, dtype=torch.int32)
    n = int(cf.sum())
    order = torch.empty(max(n, 1), dtype=torch.int32)
    go = torch.empty(n_local + 1, dtype=torch.int32)
    _check(lib.moe_ep_recv_plan(G, n_local, _i32(cf), _i32(rc), _i32(rd), _i32(order), _i32(go)))
    return rc, rd, order[:n], go


@dataclass
class Dispatched:
    """The rows this rank computes: rows[i] belongs to local expert e for
    group_offsets[e] <= i < group_offsets[e + 1] (experts of this rank,
    ascending); the rest is what combine() needs."""
    rows: torch.Tensor
    group_offsets: torch.Tensor
    order: torch.Tensor
    send_counts: list
    recv_counts: list


class ExpertParallel:
    """Dispatch and combine for one process group; the group's rank g owns
    the experts [first[g], first[g+1])."""

    def __init__(self, n_expert: int, group=None, first=None):
        self.group = group
        self.G = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        self.first = list(first) if first is not None else contiguous_partition(n_expert, self.G)
        if len(self.first) != self.G + 1 or self.first[-1] != n_expert:
            raise ValueError("first must hold n_ranks + 1 ascending bounds ending at n_expert")
        self.n_local = self.first[self.rank + 1] - self.first[self.rank]

    def dispatch(self, rows_by_expert: torch.Tensor, counts) -> Dispatched:
        """rows_by_expert: the token rows of this rank's (token, slot) pairs in
        expert order (the grouping step's gather); counts: pairs per expert."""
        sc, _ = send_plan(counts, self.first)
        c = torch.as_tensor(counts, dtype=torch.int32).cpu()
        # each rank tells each other rank how many rows of each of its experts follow
        send_rows = [c[self.first[g]:self.first[g + 1]] for g in range(self.G)]
        n_local_of = [self.first[g + 1] - self.first[g] for g in range(self.G)]
        flat = torch.cat(send_rows).to(rows_by_expert.device)
        got = torch.empty(self.G * self.n_local, dtype=torch.int32, device=rows_by_expert.device)
        dist.all_to_all_single(got, flat, [self.n_local] * self.G, n_local_of, group=self.group)
        rc, _, order, go = recv_plan(got.cpu().view(self.G, self.n_local))
        arrived = rows_by_expert.new_empty((int(rc.sum()),) + tuple(rows_by_expert.shape[1:]))
        dist.all_to_all_single(arrived, rows_by_expert.contiguous(), rc.tolist(), sc.tolist(), group=self.group)
        rows = arrived.index_select(0, order.to(arrived.device).long())
        return Dispatched(rows, go, order, sc.tolist(), rc.tolist())

    def combine(self, outputs: torch.Tensor, d: Dispatched) -> torch.Tensor:
        """outputs[i]: the expert output of d.rows[i].  Returns this rank's
        outputs back in its own expert order (one row per dispatched row)."""
        back = torch.empty_like(outputs)
        back.index_copy_(0, d.order.to(outputs.device).long(), outputs)  # to arrival order
        mine = outputs.new_empty((sum(d.send_counts),) + tuple(outputs.shape[1:]))
        dist.all_to_all_single(mine, back.contiguous(), d.send_counts, d.recv_counts, group=self.group)
        return mine
