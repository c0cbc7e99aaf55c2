"""Expert parallelism for the routed MoE layer over a torch.distributed group.

The pages place expert stacks across devices (llama.cpp PR #26185 "model: add
Kimi-K3 text model": the runs that split the model with --tensor-split and
interleaved -ot layer placement).  Here the experts of one layer are split
over G ranks: rank r holds experts [r E_l, (r + 1) E_l), E_l = E / G, and its
own tokens.  One forward on every rank:

1. route its tokens (every rank holds the router): idx [T, k], w [T, k];
2. dispatch: each (token, slot) pair goes to the rank that owns its expert,
   in the order (owner, token, slot); an all-to-all of the pair counts, then of
   the token rows, the experts' local indices and the combine weights;
3. compute: the owner runs its experts on the rows it received, one expert
   and one weight per row (k3moe_forward_routed with k = 1 on the GPU), and
   returns w * expert(row);
4. combine: a second all-to-all brings the rows back in the order they were
   sent, and each rank adds its tokens' k rows in slot order (fp32), so the
   sum's order is fixed whatever the split.

Only the index arithmetic and the data movement live here; the routing and
the expert computation are passed in (the library's kernels on a GPU; the
tests give the CPU oracle, over gloo ranks).  The collectives are
torch.distributed.all_to_all_single, so NCCL on GPUs and gloo on CPUs both
serve.  No TMA multicast or peer access is involved: received rows land in
the receiving rank's own memory before any kernel reads them.
"""
from __future__ import annotations

import torch
import torch.distributed as dist


class ExpertParallel:
    """The split of E experts over the ranks of ``group`` and the dispatch /
    combine of one layer call."""

    def __init__(self, E: int, k: int, group=None):
        self.group = group
        self.world = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        if E % self.world:
            raise ValueError("the experts must split evenly over the ranks")
        self.E, self.k, self.E_local = E, k, E // self.world

    def owned(self) -> range:
        """The global indices of this rank's experts."""
        return range(self.rank * self.E_local, (self.rank + 1) * self.E_local)

    def plan(self, idx: torch.Tensor) -> dict:
        """Send order of the (token, slot) pairs of idx [T, k]: grouped by owner
        rank, then token, then slot (a stable sort of the owners), with the
        pairs' counts per destination and the experts' local indices."""
        T, k = idx.shape
        flat = idx.reshape(-1).to(torch.int64)
        owner = torch.div(flat, self.E_local, rounding_mode="floor")
        order = torch.sort(owner, stable=True).indices
        counts = torch.bincount(owner, minlength=self.world)
        return {"T": T, "k": k, "order": order, "send_counts": counts,
                "local": (flat - owner * self.E_local)[order].to(torch.int32)}

    def _exchange(self, t: torch.Tensor, send: list, recv: list) -> torch.Tensor:
        out = t.new_empty((sum(recv),) + tuple(t.shape[1:]))
        dist.all_to_all_single(out, t.contiguous(), recv, send, group=self.group)
        return out

    def dispatch(self, x: torch.Tensor, idx: torch.Tensor, w: torch.Tensor) -> dict:
        """Send every pair's token row, local expert and weight to the owner.
        Returns the received rows [R, d], local experts [R] int32, weights [R]
        (fp32, or float64 for float64 weights) and the plan (with both sides'
        counts) for the combine."""
        p = self.plan(idx)
        counts = p["send_counts"].to(torch.int64)
        recv_counts = torch.empty_like(counts)
        dist.all_to_all_single(recv_counts, counts, group=self.group)
        send, recv = counts.tolist(), recv_counts.tolist()
        token = torch.div(p["order"], p["k"], rounding_mode="floor")
        rows = self._exchange(x[token], send, recv)
        local = self._exchange(p["local"], send, recv)
        wdt = torch.float64 if w.dtype == torch.float64 else torch.float32
        wts = self._exchange(w.reshape(-1)[p["order"]].to(wdt), send, recv)
        p.update(send=send, recv=recv)
        return {"rows": rows, "local": local, "w": wts, "plan": p}

    def combine(self, y: torch.Tensor, plan: dict) -> torch.Tensor:
        """Return the weighted expert rows y [R, d] to their senders and add
        each token's k rows in slot order (fp32, or float64 for float64 rows).
        Returns [T, d]."""
        back = self._exchange(y, plan["recv"], plan["send"])  # in this rank's send order
        T, k = plan["T"], plan["k"]
        acc = torch.float64 if y.dtype == torch.float64 else torch.float32
        pair_rows = torch.empty_like(back)
        pair_rows[plan["order"]] = back  # row p = t * k + j
        pair_rows = pair_rows.reshape(T, k, back.shape[-1]).to(acc)
        out = torch.zeros((T, pair_rows.shape[-1]), dtype=acc, device=y.device)
        for j in range(k):
            out += pair_rows[:, j]
        return out

    def forward(self, x: torch.Tensor, route_fn, experts_fn) -> torch.Tensor:
        """One layer call on this rank's tokens x [T, d]: route_fn(x) -> (idx
        [T, k], w [T, k]) with global expert indices; experts_fn(rows, local
        [R, 1] int32, w [R, 1] fp32) -> the rows' weighted outputs [R, d] from
        this rank's experts.  Returns [T, d] (fp32, or float64 for float64 rows)."""
        idx, w = route_fn(x)
        d = self.dispatch(x, idx, w)
        y = experts_fn(d["rows"], d["local"].reshape(-1, 1), d["w"].reshape(-1, 1))
        return self.combine(y, d["plan"])


def routed_experts_fn(local_layer, ws=None):
    """experts_fn for ExpertParallel.forward on a GPU: k3moe_forward_routed on
    this rank's experts (``local_layer``: a MoELayer of the E_l local experts
    with k = 1)."""
    from . import k3moe_forward_routed

    def fn(rows, local, w):
        if rows.shape[0] == 0:
            return rows.new_zeros(rows.shape)
        return k3moe_forward_routed(local_layer, rows, local.contiguous(), w.contiguous(), ws=ws)

    return fn
