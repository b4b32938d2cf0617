"""Expert parallelism across the ranks of a process group: the exchange of one MoE layer call.

Unmeasured on hardware: every run of this build has one GPU. The exchange and the combine are
tested on CPU in two gloo processes (tests/test_ep_gloo.py); on GPUs the same calls run over
NCCL.

Rank r of N owns experts [floor(r*E/N), floor((r+1)*E/N)) (equal blocks when N divides E) and
is the home rank of its own tokens. The experts are independent and each token fires K of them ("Qwen3.6-35B-A3B --
Architecture Overview", MoE FFN: 256 Experts), so the experts are sharded and the token rows
travel. One call:
  1. routing on the home rank (the router weights are replicated): ids [T, K], w [T, K] and
     the shared-expert gate sg [T];
  2. counts all-to-all: n[r -> d], the pairs (t, k) of rank r routed to experts of rank d;
  3. dispatch all-to-all: each pair's token row with its (expert, token, slot), in the order
     (owner, expert, token, slot) -- the stable counting sort of the one-GPU dispatch, so an
     owner receives each expert's rows from each source rank contiguously;
  4. on the owner, each local expert's received rows go through that expert (`expert_fn`; on a
     GPU the grouped GEMMs over the received rows);
  5. return all-to-all: the unscaled expert outputs, in the order the owner received the rows;
  6. on the home rank, the fixed-order combine
         out[t] = residual[t] + sg[t] * shared(x[t]) + sum_{k=0..K-1} w[t, k] * y[t, k],
     the order of the one-GPU combine, so the result depends neither on N nor on the order in
     which rows arrive.
Each received row lands in local memory before anything reads it; nothing is multicast.
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def owners(ids: torch.Tensor, E: int, world: int) -> torch.Tensor:
    """Rank that owns each expert id: rank r owns [floor(r*E/world), floor((r+1)*E/world)), so
    expert e belongs to the largest r with floor(r*E/world) <= e, i.e. floor(((e+1)*world - 1) / E)."""
    if not 1 <= world <= E:
        raise ValueError(f"{world} ranks cannot share {E} experts")
    return torch.div((ids.to(torch.int64) + 1) * world - 1, E, rounding_mode="floor")


def dispatch_order(ids: torch.Tensor, E: int, world: int):
    """The send order of the pairs p = t * K + k: sorted by expert (hence by owner), ties by p
    (token, then slot); and the number of pairs for each owner."""
    flat = ids.reshape(-1).to(torch.int64)
    if flat.numel() and (int(flat.min()) < 0 or int(flat.max()) >= E):
        raise ValueError("expert id out of range")
    order = torch.sort(flat, stable=True).indices
    counts = torch.bincount(owners(flat, E, world), minlength=world)
    return order, counts


def ep_layer(x: torch.Tensor, ids: torch.Tensor, w: torch.Tensor, sg: torch.Tensor, ys: torch.Tensor, expert_fn,
             E: int, residual: torch.Tensor | None = None, group=None) -> dict:
    """One layer call of this rank's T tokens under expert parallelism.

    x [T, H] token rows (any dtype; sent as they are), ids [T, K] expert ids, w [T, K] routing
    weights, sg [T] shared gate, ys [T, H] the shared expert's output (computed on the home
    rank), residual [T, H] or None. expert_fn(e, rows) -> [n, H] is expert e applied to rows
    [n, H]; it is called on the rank that owns e. Every rank of `group` must call this.

    Returns out [T, H] (dtype of ys) and, for checking, what this rank received: meta [R, 3]
    (expert, source-local token, slot), src [R] (source rank) and the rows [R, H]."""
    world = dist.get_world_size(group)
    T, K = ids.shape
    H = x.shape[1]
    order, send_counts = dispatch_order(ids, E, world)
    recv_counts = torch.empty_like(send_counts)
    dist.all_to_all_single(recv_counts, send_counts, group=group)
    sc, rc = send_counts.tolist(), recv_counts.tolist()
    R = sum(rc)

    tok = torch.div(order, K, rounding_mode="floor")
    meta = torch.stack([ids.reshape(-1).to(torch.int64)[order], tok, order - tok * K], dim=1).contiguous()
    rows = x[tok].contiguous()
    r_meta = torch.empty(R, 3, dtype=torch.int64)
    r_rows = torch.empty(R, H, dtype=x.dtype)
    dist.all_to_all_single(r_meta, meta, rc, sc, group=group)
    dist.all_to_all_single(r_rows, rows, rc, sc, group=group)
    src = torch.repeat_interleave(torch.arange(world), torch.tensor(rc, dtype=torch.int64))

    # each local expert over every row it received (in received order within the expert)
    y_recv = torch.empty(R, H, dtype=ys.dtype)
    if R:
        by_expert = torch.sort(r_meta[:, 0], stable=True).indices
        experts, n_per = torch.unique_consecutive(r_meta[by_expert, 0], return_counts=True)
        start = 0
        for e, n in zip(experts.tolist(), n_per.tolist()):
            sel = by_expert[start:start + n]
            y_recv[sel] = expert_fn(e, r_rows[sel]).to(ys.dtype)
            start += n

    y_back = torch.empty(T * K, H, dtype=ys.dtype)
    dist.all_to_all_single(y_back, y_recv, sc, rc, group=group)
    y = torch.empty(T * K, H, dtype=ys.dtype)
    y[order] = y_back
    y = y.reshape(T, K, H)

    out = residual.to(ys.dtype).clone() if residual is not None else torch.zeros(T, H, dtype=ys.dtype)
    out += sg.to(ys.dtype)[:, None] * ys
    for k in range(K):
        out += w[:, k].to(ys.dtype)[:, None] * y[:, k]
    return dict(out=out, meta=r_meta, src=src, rows=r_rows, recv_counts=recv_counts, send_counts=send_counts)
