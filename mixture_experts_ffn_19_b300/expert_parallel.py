"""Expert-parallel dispatch and combine across ranks: the exchange plan.

Expert parallelism as the pages describe it: the routed experts are divided
among the ranks, every rank routes its own tokens, the rows of each kept
assignment travel to the rank that owns its expert, that rank runs the expert,
and the results travel back to the token's rank for the gate-weighted combine
(«DeepSeek-V2 ...» summary, §3.1 and the ``expert_parallel_forward`` example of
§4.2; «为什么MoE有效？稀疏激活的数学直觉与工程实践» §4.1: both moves are
all-to-all exchanges).  Shared experts are replicated: each rank runs them on
its own tokens.

Capacity stays exactly that of one device running the concatenation of every
rank's batch in rank order (global token order): C is computed on the global
token count, and an expert keeps an assignment when its place in global order
is below C.  That place is the assignment's rank inside its own rank's batch
plus the number of assignments of the same expert on lower ranks, so one
all-gather of the [E] per-rank histogram and an exclusive scan over ranks make
the drop decisions identical to one device's.  Reroute ("next-best unfilled
expert", rounds) takes one all-gather of the per-rank proposal histogram per
round for the same reason.

Everything here is integer bookkeeping and the two exchanges; the arithmetic
(routing, expert FFNs) is supplied by the caller.  The planning functions are
pure (they take the gathered histograms), so a single process can check them
for any number of ranks; ``ep_forward`` runs them with ``torch.distributed``
collectives (gloo on CPU; the row exchange is one ``all_to_all_single`` each
way).

Inside an expert's segment the owner lays rows out by source rank, then as
that rank placed them (primary assignments in token order, then reroutes in
(round, token, slot) order); one device orders a segment by global primary,
then global reroute order.  Output rows do not depend on that order.
"""
from __future__ import annotations

import numpy as np

__all__ = ["expert_owner", "local_experts", "capacity_for", "primary_plan", "propose",
           "reroute_round", "exchange_plan", "ep_forward"]


def expert_owner(n_experts: int, world: int) -> np.ndarray:
    """Owner rank of each routed expert: contiguous, balanced blocks."""
    return (np.arange(n_experts, dtype=np.int64) * world // n_experts).astype(np.int64)


def local_experts(n_experts: int, world: int, rank: int) -> np.ndarray:
    return np.nonzero(expert_owner(n_experts, world) == rank)[0]


def capacity_for(n_tokens_global: int, n_experts: int, top_k: int, cap_mode: int,
                 alpha: float) -> int | None:
    """C = floor(floor(k N / E) alpha) on the global token count («大模型MoE架构揭秘»
    §3.1); None without a capacity limit.  Same formula as the library's
    moe_capacity, restated for the global batch."""
    if cap_mode == 0:
        return None
    return int(np.floor(((top_k * n_tokens_global) // n_experts) * float(alpha)))


def _local_order(topk_idx: np.ndarray, n_experts: int):
    """Per expert, this rank's assignments (t, j) in ascending token order."""
    N, k = topk_idx.shape
    lists = [[] for _ in range(n_experts)]
    for t in range(N):
        for j in range(k):
            e = int(topk_idx[t, j])
            if 0 <= e < n_experts:
                lists[e].append((t, j))
    return lists


def primary_plan(topk_idx: np.ndarray, hist_all: np.ndarray, rank: int, cap: int | None):
    """Drop decisions of one rank given every rank's histogram hist_all[R, E].

    An assignment of expert e with local rank rho is kept when
    base[e] + rho < C, base = the exclusive scan of hist_all over ranks.
    Returns (final_idx with -1 for overflow, blocks: per expert the kept (t, j)
    in block order, pending: overflowed (t, j) in (t, j) order)."""
    E = hist_all.shape[1]
    base = hist_all[:rank].sum(axis=0)
    final = topk_idx.astype(np.int32).copy()
    blocks = [[] for _ in range(E)]
    pending = []
    for e, lst in enumerate(_local_order(topk_idx, E)):
        for rho, (t, j) in enumerate(lst):
            if cap is None or base[e] + rho < cap:
                blocks[e].append((t, j))
            else:
                final[t, j] = -1
                pending.append((t, j))
    pending.sort()
    return final, blocks, pending


def propose(final: np.ndarray, key: np.ndarray, pending, full: np.ndarray):
    """One round's proposals of one rank (reading R4): each pending slot, in (t, j)
    order, proposes the best-keyed expert (ties to the lower index) that was not
    full when the round began and that its token neither holds nor proposed
    earlier this round.  Returns (proposals [(t, j, e)], dropped [(t, j)])."""
    proposals, dropped = [], []
    cur, proposed = -1, []
    for (t, j) in pending:
        if t != cur:
            cur, proposed = t, []
        held = set(int(e) for e in final[t] if e >= 0) | set(proposed)
        best = -1
        for e in range(key.shape[1]):
            if full[e] or e in held:
                continue
            if best < 0 or key[t, e] > key[t, best]:
                best = e
        if best < 0:
            dropped.append((t, j))
        else:
            proposed.append(best)
            proposals.append((t, j, best))
    return proposals, dropped


def reroute_round(proposals, prop_hist_all: np.ndarray, rank: int, fill: np.ndarray, cap: int):
    """Acceptance of one rank's proposals given every rank's proposal histogram:
    proposal number rho of this rank to expert e is accepted when
    fill[e] + (proposals to e on lower ranks) + rho < C.  Returns (accepted
    [(t, j, e)], rejected [(t, j)] in (t, j) order, next fill levels)."""
    base = prop_hist_all[:rank].sum(axis=0)
    seen = np.zeros(prop_hist_all.shape[1], dtype=np.int64)
    accepted, rejected = [], []
    for (t, j, e) in proposals:
        if fill[e] + base[e] + seen[e] < cap:
            accepted.append((t, j, e))
        else:
            rejected.append((t, j))
        seen[e] += 1
    new_fill = np.minimum(cap, fill + prop_hist_all.sum(axis=0))
    return accepted, rejected, new_fill


def exchange_plan(blocks, kept_all: np.ndarray, rank: int):
    """Row movements of one rank.

    blocks: per expert the kept (t, j) of this rank in block order.
    kept_all[R, E]: every rank's kept count per expert.
    Returns a dict:
      send_slots  [(t, j)] in send order (by owner, expert, block order)
      send_counts [R] rows to each owner
      recv_counts [R] rows from each source
      segments    per local expert e: indices into the receive buffer, in
                  segment order (source rank ascending, then block order)
    The return exchange sends the owner's rows back in receive order, so the
    source gets them in its own send order."""
    R, E = kept_all.shape
    owner = expert_owner(E, R)
    send_slots, send_counts = [], np.zeros(R, dtype=np.int64)
    for o in range(R):
        for e in np.nonzero(owner == o)[0]:
            send_slots += blocks[e]
            send_counts[o] += len(blocks[e])
    mine = np.nonzero(owner == rank)[0]
    recv_counts = kept_all[:, mine].sum(axis=1)
    # receive buffer: source-major, then this rank's experts ascending
    starts = np.concatenate([[0], np.cumsum(recv_counts)])
    segments = {}
    for e in mine:
        idx = []
        for r in range(R):
            off = starts[r] + kept_all[r, mine[mine < e]].sum()
            idx += list(range(int(off), int(off + kept_all[r, e])))
        segments[int(e)] = np.asarray(idx, dtype=np.int64)
    return {"send_slots": send_slots, "send_counts": send_counts, "recv_counts": recv_counts,
            "segments": segments}


def _all_gather_np(a: np.ndarray, group=None) -> np.ndarray:
    import torch
    import torch.distributed as dist
    t = torch.as_tensor(np.ascontiguousarray(a))
    out = [torch.empty_like(t) for _ in range(dist.get_world_size(group))]
    dist.all_gather(out, t, group=group)
    return np.stack([o.numpy() for o in out])


def ep_forward(x, topk_idx, gates, key, n_experts, cap_mode, alpha, expert_fn, shared_fn=None,
               group=None):
    """Expert-parallel MoE layer on this rank's tokens.

    x         [N_r, d] torch tensor (CPU): this rank's token rows, as stored
              (bf16 bit patterns as int16, or float32); these bytes travel
    topk_idx  [N_r, k] int, gates [N_r, k] float32, key [N_r, E] float32: this
              rank's routing (key ranks reroute candidates)
    expert_fn(e, rows) -> float64 [n, d]: routed expert e (owned here) on rows
    shared_fn(x) -> float64 [N_r, d] or None: sum of the shared experts
    Returns (y float64 [N_r, d], info) with this rank's final_idx and the global
    per-expert kept counts, n_dropped and n_rerouted.
    """
    import torch
    import torch.distributed as dist
    R, rank = dist.get_world_size(group), dist.get_rank(group)
    topk_idx = np.asarray(topk_idx)
    N, k = topk_idx.shape
    E = n_experts
    n_global = int(_all_gather_np(np.array([N], dtype=np.int64), group).sum())
    cap = capacity_for(n_global, E, k, cap_mode, alpha)

    hist = np.bincount(topk_idx[(topk_idx >= 0) & (topk_idx < E)].ravel(), minlength=E)
    hist_all = _all_gather_np(hist.astype(np.int64), group)
    final, blocks, pending = primary_plan(topk_idx, hist_all, rank, cap)
    n_dropped_local, n_rerouted_local = 0, 0
    if cap_mode == 2:
        fill = np.minimum(cap, hist_all.sum(axis=0))
        while True:
            if int(_all_gather_np(np.array([len(pending)], dtype=np.int64), group).sum()) == 0:
                break
            full = fill >= cap
            proposals, dropped = propose(final, np.asarray(key), pending, full)
            n_dropped_local += len(dropped)
            ph = np.zeros(E, dtype=np.int64)
            for (_, _, e) in proposals:
                ph[e] += 1
            ph_all = _all_gather_np(ph, group)
            accepted, pending, fill = reroute_round(proposals, ph_all, rank, fill, cap)
            for (t, j, e) in accepted:
                final[t, j] = e
                blocks[e].append((t, j))
            n_rerouted_local += len(accepted)
    elif cap_mode == 1:
        n_dropped_local = len(pending)
    kept = np.array([len(b) for b in blocks], dtype=np.int64)
    kept_all = _all_gather_np(kept, group)

    plan = exchange_plan(blocks, kept_all, rank)
    d = x.shape[1]
    rows = [t for (t, _) in plan["send_slots"]]
    # rows travel as their raw bytes, whatever their element type
    xb = x.contiguous().view(torch.uint8).reshape(x.shape[0], -1)
    send = xb[torch.as_tensor(rows, dtype=torch.long)] if rows else xb.new_empty((0, xb.shape[1]))
    recv_b = xb.new_empty((int(plan["recv_counts"].sum()), xb.shape[1]))
    dist.all_to_all_single(recv_b, send.contiguous(), [int(c) for c in plan["recv_counts"]],
                           [int(c) for c in plan["send_counts"]], group=group)
    recv = recv_b.view(x.dtype).reshape(-1, d)

    out = torch.zeros((recv.shape[0], d), dtype=torch.float64)
    for e, seg in plan["segments"].items():
        if len(seg):
            out[torch.as_tensor(seg)] = torch.as_tensor(
                np.asarray(expert_fn(e, recv[torch.as_tensor(seg)]), dtype=np.float64))
    back = torch.empty((len(rows), d), dtype=torch.float64)
    dist.all_to_all_single(back, out, [int(c) for c in plan["send_counts"]],
                           [int(c) for c in plan["recv_counts"]], group=group)

    # combine: shared experts first, then the kept slots in slot order
    where = {tj: i for i, tj in enumerate(plan["send_slots"])}
    y = np.zeros((N, d)) if shared_fn is None else np.array(shared_fn(x), dtype=np.float64)
    g = np.asarray(gates, dtype=np.float32)
    bk = back.numpy()
    for t in range(N):
        for j in range(k):
            if final[t, j] >= 0:
                y[t] = y[t] + float(g[t, j]) * bk[where[(t, j)]]
    totals = _all_gather_np(np.array([n_dropped_local, n_rerouted_local], dtype=np.int64), group)
    return y, {"final": final, "counts": kept_all.sum(axis=0), "n_dropped": int(totals[:, 0].sum()),
               "n_rerouted": int(totals[:, 1].sum()), "capacity": cap,
               "send_counts": plan["send_counts"], "recv_counts": plan["recv_counts"]}
