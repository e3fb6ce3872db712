"""Expert-parallel partition of the routed MoE layer: the host-side plan.

The pages run the layer with expert parallelism across the GPUs of a node
("Inkling-2-Small" cookbook, section 2, Parallelism paragraph: TP4 with EP4,
the expert-parallel size equal to the tensor-parallel size; MegaMoE
paragraph: dispatch, both expert GEMMs, the capped SwiGLU and the combine
fused with the all-to-all, at most 4,096 tokens per rank).  NVFP4 experts are
not split by tensor parallelism, because an activation row's scales span the
expert's full input width (the same paragraph); so experts are partitioned
whole, each rank owning a contiguous range.

This module computes, from each rank's routing, everything an exchange needs
and nothing that moves data: the owner of every expert, the send order and
counts of the pairs (t, j) a rank routes, the order in which a receiver
regroups the rows it gets, and the inverse orders that bring the experts'
outputs back for the combine.  The exchange itself (an all-to-all of the
encoded activation rows, and one of the outputs) is the caller's.

Orders (G ranks, rank s holds T_s tokens; a global token id is the rank's
offset plus its local id):
  * send order of rank s = its own dispatch order: pairs sorted by (expert,
    token).  Each owner's experts are a contiguous range, so the pairs for
    owner d form one contiguous block (send_counts[d] rows), already sorted
    by (expert, token) inside it.
  * received order at rank d: source rank s ascending, then (expert, token)
    inside each source's block.
  * grouped order at rank d: (expert, source rank, token) = (expert, global
    token), i.e. exactly the dispatch order that a single GPU would give the
    whole batch, restricted to d's experts.  The expert GEMMs read this
    order; its per-expert counts come from one small exchange of the
    [G, experts of d] count matrix before the rows move.
  * the outputs go back in received order (the inverse regrouping), and
    arrive at rank s in its send order, which is its dispatch order, so the
    combine reads them through its own pair_pos unchanged.

Remote rows land in the receiver's local memory (a staging buffer in HBM)
before any of its kernels read them; the expert GEMMs' TMA loads then read
only local memory, and no kernel loads a peer's memory.
"""
from __future__ import annotations

import numpy as np


def expert_ranges(E: int, G: int):
    """[(lo, hi)] of the G ranks: contiguous, sizes differing by at most one
    (the first E % G ranks hold one expert more)."""
    if not (1 <= G <= E):
        raise ValueError(f"need 1 <= G <= E, got G={G}, E={E}")
    base, extra = divmod(E, G)
    out, lo = [], 0
    for r in range(G):
        hi = lo + base + (1 if r < extra else 0)
        out.append((lo, hi))
        lo = hi
    return out


def expert_owner(E: int, G: int) -> np.ndarray:
    """int32 [E]: the rank that owns each expert."""
    own = np.empty(E, np.int32)
    for r, (lo, hi) in enumerate(expert_ranges(E, G)):
        own[lo:hi] = r
    return own


def local_dispatch(topk_idx: np.ndarray, E: int):
    """The dispatch order of one rank's pairs (as moe_dispatch computes it):
    counts [E], offsets [E+1], perm [T*k] (pair id t*k + j, sorted by
    (expert, token)), pair_pos [T, k] (its inverse)."""
    idx = np.ascontiguousarray(topk_idx, np.int64)
    T, k = idx.shape
    if idx.size and (idx.min() < 0 or idx.max() >= E):
        raise ValueError("expert id out of range")
    flat = idx.ravel()
    counts = np.bincount(flat, minlength=E).astype(np.int32)
    offsets = np.zeros(E + 1, np.int32)
    np.cumsum(counts, out=offsets[1:])
    pair = np.arange(T * k, dtype=np.int64)
    # stable sort by expert keeps pair ids (hence tokens) ascending per expert
    perm = pair[np.argsort(flat, kind="stable")].astype(np.int32)
    pair_pos = np.empty(T * k, np.int32)
    pair_pos[perm] = np.arange(T * k, dtype=np.int32)
    return dict(counts=counts, offsets=offsets, perm=perm, pair_pos=pair_pos.reshape(T, k))


def plan_send(topk_idx: np.ndarray, E: int, G: int):
    """What rank s sends: its dispatch order (`perm`: row i of the send
    buffer is the token perm[i] // k), rows per destination (`send_counts`
    [G]), and the per-expert counts of each destination's block
    (`expert_counts` [G][n_d], the row of the count matrix destination d
    receives from this rank)."""
    d = local_dispatch(topk_idx, E)
    ranges = expert_ranges(E, G)
    send_counts = np.array([d["counts"][lo:hi].sum() for lo, hi in ranges], np.int64)
    expert_counts = [d["counts"][lo:hi].astype(np.int64) for lo, hi in ranges]
    return dict(d, send_counts=send_counts, expert_counts=expert_counts, send_tokens=d["perm"] // topk_idx.shape[1])


def plan_receive(count_matrix: np.ndarray):
    """At a receiver: count_matrix [G, n_d] = rows of each of its n_d experts
    from each source rank (sources ascending).  Returns
      recv_counts [G]          rows from each source (its all-to-all split),
      grouped_from_recv [R]    row i of the grouped (expert, source, token)
                               order is row grouped_from_recv[i] of the
                               received (source, expert, token) order,
      recv_from_grouped [R]    the inverse (outputs go back in received
                               order: recv_out[j] = grouped_out[recv_from_grouped[j]]),
      expert_offsets [n_d+1]   the grouped order's per-expert segments."""
    cm = np.asarray(count_matrix, np.int64)
    G, n = cm.shape
    recv_counts = cm.sum(1)
    # start of (source s, local expert e) inside the received buffer
    src_start = np.zeros(G, np.int64)
    np.cumsum(recv_counts[:-1], out=src_start[1:])
    within = np.zeros((G, n), np.int64)
    np.cumsum(cm[:, :-1], axis=1, out=within[:, 1:])
    recv_block = src_start[:, None] + within
    expert_offsets = np.zeros(n + 1, np.int64)
    np.cumsum(cm.sum(0), out=expert_offsets[1:])
    R = int(recv_counts.sum())
    grouped_from_recv = np.empty(R, np.int64)
    pos = 0
    for e in range(n):
        for s in range(G):
            c = int(cm[s, e])
            grouped_from_recv[pos:pos + c] = recv_block[s, e] + np.arange(c)
            pos += c
    recv_from_grouped = np.empty(R, np.int64)
    recv_from_grouped[grouped_from_recv] = np.arange(R)
    return dict(recv_counts=recv_counts, grouped_from_recv=grouped_from_recv, recv_from_grouped=recv_from_grouped,
                expert_offsets=expert_offsets)
