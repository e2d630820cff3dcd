"""Expert parallelism across ranks: the exchange around the local slice.

Each rank of an expert-parallel group holds T_r tokens and the weights of
E / ep experts (H20 article, para. 2: the fused-MoE call takes the EP size and
rank; para. 3: 400 expert slots over 8 GPUs).  ``ep_forward`` computes the
full layer output for the rank's own tokens:

1. route: the rank's tokens are routed over all E experts (ids, weights);
2. dispatch: every token is sent once to each rank that owns at least one of
   its picks, with all k ids and weights (``all_to_all_single``: first the
   counts, then the rows, ids and weights);
3. local slice: the owner runs its experts on the received rows with the
   received picks; picks owned by other ranks are skipped
   (``MoELayer.forward_with_ids`` on an expert-parallel plan);
4. combine: each partial row goes back to the token's rank, which adds the
   partials of all owners in rank order, so the result does not depend on
   arrival order.

The module holds no arithmetic of the layer: routing and the expert MLPs are
the callables it is given; it only indexes and moves rows.  Every rank must
call it collectively, with the same k and E.  On GPUs (one rank per GPU,
NCCL)::

    layer = MoELayer(w13_local, w2_local, k=k, dtype=BF16, ep_size=ep, ep_rank=rank)
    out = ep_forward(x, logits, k=k, E=E,
                     route=lambda lg: route_topk(lg, k),
                     local_forward=layer.forward_with_ids)
"""
from __future__ import annotations

from typing import Callable

import torch
import torch.distributed as dist


def _exchange(send: torch.Tensor, send_counts: list, recv_counts: list, row: int, group):
    """all_to_all_single of a [sum(send_counts), *] tensor by row counts."""
    out = torch.empty((sum(recv_counts),) + tuple(send.shape[1:]), dtype=send.dtype,
                      device=send.device)
    dist.all_to_all_single(out.view(-1), send.contiguous().view(-1),
                           output_split_sizes=[c * row for c in recv_counts],
                           input_split_sizes=[c * row for c in send_counts], group=group)
    return out


def ep_forward(x: torch.Tensor, logits: torch.Tensor, *, k: int, E: int,
               route: Callable, local_forward: Callable, group=None) -> torch.Tensor:
    """Full MoE layer output for this rank's tokens under expert parallelism.

    x [T, H], logits [T, E] of this rank's tokens.  ``route(logits)`` returns
    (ids int32 [T, k], w float32 [T, k]) over all E experts;
    ``local_forward(x_recv, ids_recv, w_recv)`` returns this rank's partial
    output [T_recv, H] for received rows (its own experts' picks only).
    Returns [T, H] in float32 (the sum of the owners' partials).
    """
    ws = dist.get_world_size(group)
    if E % ws != 0:
        raise ValueError(f"E={E} experts do not split over {ws} ranks")
    e_local = E // ws
    T, H = x.shape
    ids, w = route(logits)
    if tuple(ids.shape) != (T, k) or tuple(w.shape) != (T, k):
        raise ValueError("route() must return ids and weights of shape [T, k]")
    owner = ids.long() // e_local  # [T, k]; rank that holds each pick's expert

    # tokens for each destination rank, in token order
    dest_tokens = [torch.nonzero((owner == d).any(dim=1)).flatten() for d in range(ws)]
    send_counts = [int(t.numel()) for t in dest_tokens]
    counts = torch.tensor(send_counts, dtype=torch.int64, device=x.device)
    recv = torch.empty_like(counts)
    dist.all_to_all_single(recv, counts, group=group)
    recv_counts = [int(c) for c in recv.tolist()]

    order = torch.cat(dest_tokens) if T else torch.empty(0, dtype=torch.long, device=x.device)
    x_recv = _exchange(x[order], send_counts, recv_counts, H, group)
    ids_recv = _exchange(ids[order], send_counts, recv_counts, k, group)
    w_recv = _exchange(w[order], send_counts, recv_counts, k, group)

    partial = local_forward(x_recv, ids_recv, w_recv)
    if tuple(partial.shape) != (sum(recv_counts), H):
        raise ValueError("local_forward() must return [rows received, H]")
    back = _exchange(partial.float(), recv_counts, send_counts, H, group)

    out = torch.zeros(T, H, dtype=torch.float32, device=x.device)
    start = 0
    for d in range(ws):  # owners in rank order: a fixed order of additions
        n = send_counts[d]
        if n:
            out.index_add_(0, dest_tokens[d], back[start:start + n])
        start += n
    return out
