"""Expert-parallel dispatch and combine of the routed MoE layer across ranks.

"Why can super-large MoE be distributed for inference", the swarm section: the backbone keeps
the router authoritative and sends the expert computation to the machines that hold the
experts.  Here expert e lives on rank e mod G (as local expert e // G) and tokens are
data-parallel: every rank routes its own tokens, ships each (token, expert) pair's input row
to the expert's rank, the ranks evaluate the experts they hold on what they received, the
outputs travel back, and every rank combines its tokens' k outputs in slot order j, as the
single-GPU layer does.

The exchange is two all-to-alls over torch.distributed (NCCL between GPUs, gloo on CPU ranks):
  1. counts: pairs per destination rank, so that every rank knows how many rows it receives;
  2. dispatch: the pairs' input rows and local expert indices, in send order -- sorted by
     (destination rank, expert, pair id t*k + j), so each destination receives its rows grouped
     by expert and, within an expert, in pair order (the stable sort of the single-GPU layer);
  3. the expert ranks evaluate (`run_local(rows, local_expert) -> outputs`);
  4. return: the outputs travel back with the split sizes swapped, and land at their pairs;
  5. combine: out[t] = sum_j w[t, j] * y[t, j], in slot order.
Only the routing metadata and the rows move: no rank needs another rank's expert weights.
"""
from __future__ import annotations

import numpy as np


def expert_rank(e, world: int):
    """Rank that holds expert e (array-wise)."""
    return np.asarray(e) % world


def local_expert(e, world: int):
    """Index of expert e among the experts its rank holds."""
    return np.asarray(e) // world


def dispatch_plan(idx: np.ndarray, world: int):
    """Send order and per-destination counts of this rank's T*k pairs.

    idx: int [T, k] global expert ids.  Returns (order [P] pair ids in send order, counts [world]):
    pairs sorted by destination rank, then expert, then pair id (a stable order)."""
    flat = np.asarray(idx, dtype=np.int64).ravel()
    pair = np.arange(flat.size, dtype=np.int64)
    order = np.lexsort((pair, flat, expert_rank(flat, world)))
    counts = np.bincount(expert_rank(flat, world), minlength=world).astype(np.int64)
    return order, counts


def combine(w: np.ndarray, y_pair, k: int):
    """out[t] = sum_j w[t, j] * y[t*k + j], summed in slot order j (y_pair [P, d], torch or numpy)."""
    T = w.shape[0]
    out = None
    for j in range(k):
        yj = y_pair[j::k][:T]
        wj = w[:, j:j + 1]
        term = wj * yj
        out = term if out is None else out + term
    return out


def ep_forward(x, idx: np.ndarray, w, run_local, group=None):
    """One expert-parallel layer step on this rank.

    x: torch [T, d] this rank's expert inputs; idx: int [T, k] the routing this rank computed;
    w: torch [T, k] its combine weights (same dtype as x); run_local(rows [n, d], local_ids
    int64 [n]) -> torch [n, d]: the experts this rank holds, on the rows it received.
    Returns out [T, d] (x's dtype and device)."""
    import torch
    import torch.distributed as dist

    world = dist.get_world_size(group)
    T, k = np.asarray(idx).shape
    d = x.shape[1]
    order, send_counts = dispatch_plan(idx, world)
    dev = x.device
    # 1. counts
    sc = torch.from_numpy(send_counts).to(dev)     # (NCCL exchanges device tensors only)
    rc = torch.empty_like(sc)
    dist.all_to_all_single(rc, sc, group=group)
    recv_counts = rc.cpu().tolist()
    send_list = send_counts.tolist()
    n_recv = int(sum(recv_counts))
    # 2. dispatch rows and their local expert indices
    order_t = torch.from_numpy(order).to(dev)
    send_x = x[order_t // k].contiguous()
    send_e = torch.from_numpy(local_expert(np.asarray(idx).ravel()[order], world).astype(np.int64)).to(dev)
    recv_x = torch.empty((n_recv, d), dtype=x.dtype, device=dev)
    recv_e = torch.empty(n_recv, dtype=torch.int64, device=dev)
    dist.all_to_all_single(recv_x, send_x, recv_counts, send_list, group=group)
    dist.all_to_all_single(recv_e, send_e, recv_counts, send_list, group=group)
    # 3. the experts this rank holds
    y_recv = run_local(recv_x, recv_e) if n_recv > 0 else torch.empty((0, d), dtype=x.dtype, device=dev)
    # 4. back to the pairs' ranks, in send order
    y_sent = torch.empty((T * k, d), dtype=y_recv.dtype, device=dev)
    dist.all_to_all_single(y_sent, y_recv.contiguous(), send_list, recv_counts, group=group)
    y_pair = torch.empty_like(y_sent)
    y_pair[order_t] = y_sent
    # 5. combine in slot order
    return combine(w, y_pair, k)


class LocalExperts:
    """The experts one rank holds, evaluated by libmoe: a layer over the E_local local experts
    with k = 1 and supplied routing (each received row is one pair with weight 1), so every
    row's output is its expert's y exactly as the single-GPU layer computes it."""

    def __init__(self, d, f, E_local, act, wfmt, gate_up, down, gate_up_tscale=None, down_tscale=None,
                 path: str = "auto"):
        import torch

        from . import native
        dummy_router = torch.zeros((d, E_local), dtype=torch.float32, device=gate_up.device)
        self.layer = native.MoELayer(d, f, E_local, 1, act, wfmt, dummy_router, gate_up, down, gate_up_tscale,
                                     down_tscale, path=path)

    def __call__(self, rows, local_ids):
        import torch
        n = rows.shape[0]
        ids = local_ids.to(torch.int32).reshape(n, 1).contiguous()
        ones = torch.ones((n, 1), dtype=torch.float32, device=rows.device)
        return self.layer.forward(rows.contiguous(), idx_in=ids, w_in=ones)
