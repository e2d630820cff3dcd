"""Expert parallelism across ranks: the exchange around the local slice.

Each rank of an expert-parallel group holds T_r tokens and the weights of
E / ep experts (H20 article, para. 2: the fused-MoE call takes the EP size and
rank; para. 3: 400 expert slots over 8 GPUs).  ``ep_forward`` computes the
full layer output for the rank's own tokens:

1. route: the rank's tokens are routed over all E experts (ids, weights);
2. plan and pack (library: ``moe_ep_dispatch``, ``moe_ep_pack``): every token
   goes once to each rank that owns at least one of its picks, with all k ids
   and weights, grouped by destination rank in rank order;
3. exchange (``all_to_all_single``): counts first, then rows, ids, weights;
4. local slice: the owner runs its experts on the received rows with the
   received picks; picks owned by other ranks are skipped
   (``MoELayer.forward_with_ids`` on an expert-parallel plan);
5. return and combine (library: ``moe_ep_combine``): each partial row goes
   back to the token's rank, which adds the partials of all owners in rank
   order, so the result does not depend on arrival order.

This module moves rows and holds no arithmetic of the layer: routing and the
expert MLPs are the callables it is given, the send plan and the combine are
the library's.  The host waits once per call, for the split sizes that
``all_to_all_single`` takes.  Every rank must call it collectively, with the
same k and E.  On GPUs (one rank per GPU, NCCL)::

    layer = MoELayer(w13_local, w2_local, k=k, dtype=BF16, ep_size=ep, ep_rank=rank)
    out = ep_forward(x, logits, k=k, E=E,
                     route=lambda lg: route_topk(lg, k),
                     local_forward=layer.forward_with_ids)
"""
from __future__ import annotations

from typing import Callable

import torch
import torch.distributed as dist

from . import _binding as B


class LibraryEpOps:
    """The exchange's send plan, packing and combine, run by the CUDA library
    on the tensors' device and the current stream."""

    @staticmethod
    def _stream(t):
        return torch.cuda.current_stream(t.device).cuda_stream

    def dispatch(self, ids: torch.Tensor, e_local: int, ep_size: int):
        T, k = ids.shape
        dev = ids.device
        send_counts = torch.zeros(ep_size, dtype=torch.int32, device=dev)
        send_tokens = torch.empty(max(1, T * ep_size), dtype=torch.int32, device=dev)
        row_of = torch.empty(max(1, T * ep_size), dtype=torch.int32, device=dev)
        B._check(B.moe_ep_dispatch(ids.data_ptr(), T, k, e_local, ep_size,
                                   send_counts.data_ptr(), send_tokens.data_ptr(),
                                   row_of.data_ptr(), self._stream(ids)), "moe_ep_dispatch")
        return send_counts, send_tokens, row_of[:T * ep_size].view(T, ep_size)

    def pack(self, x, ids, w, send_counts, send_tokens, ep_size: int):
        T, H = x.shape
        k = ids.shape[1]
        dt = {torch.float32: B.MOE_DTYPE_F32, torch.bfloat16: B.MOE_DTYPE_BF16}[x.dtype]
        rows = max(1, T * ep_size)
        x_send = torch.empty(rows, H, dtype=x.dtype, device=x.device)
        ids_send = torch.empty(rows, k, dtype=torch.int32, device=x.device)
        w_send = torch.empty(rows, k, dtype=torch.float32, device=x.device)
        B._check(B.moe_ep_pack(x.data_ptr(), dt, ids.data_ptr(), w.data_ptr(), T, H, k, ep_size,
                               send_counts.data_ptr(), send_tokens.data_ptr(),
                               x_send.data_ptr(), ids_send.data_ptr(), w_send.data_ptr(),
                               self._stream(x)), "moe_ep_pack")
        return x_send, ids_send, w_send

    def combine(self, back, row_of, T: int, H: int, ep_size: int):
        out = torch.empty(T, H, dtype=torch.float32, device=row_of.device)
        if T:
            B._check(B.moe_ep_combine(back.data_ptr(), row_of.data_ptr(), T, H, ep_size,
                                      out.data_ptr(), self._stream(row_of)), "moe_ep_combine")
        return out


def _exchange(send: torch.Tensor, send_counts: list, recv_counts: list, row: int, group):
    """all_to_all_single of a [sum(send_counts), *] tensor by row counts."""
    out = torch.empty((sum(recv_counts),) + tuple(send.shape[1:]), dtype=send.dtype,
                      device=send.device)
    dist.all_to_all_single(out.view(-1), send.contiguous().view(-1),
                           output_split_sizes=[c * row for c in recv_counts],
                           input_split_sizes=[c * row for c in send_counts], group=group)
    return out


def ep_forward(x: torch.Tensor, logits: torch.Tensor, *, k: int, E: int,
               route: Callable, local_forward: Callable, group=None, ops=None) -> torch.Tensor:
    """Full MoE layer output for this rank's tokens under expert parallelism.

    x [T, H], logits [T, E] of this rank's tokens.  ``route(logits)`` returns
    (ids int32 [T, k], w float32 [T, k]) over all E experts;
    ``local_forward(x_recv, ids_recv, w_recv)`` returns this rank's partial
    output [T_recv, H] for received rows (its own experts' picks only).
    ``ops`` supplies dispatch / pack / combine (default: the CUDA library).
    Returns [T, H] in float32 (the sum of the owners' partials).
    """
    ops = ops or LibraryEpOps()
    ws = dist.get_world_size(group)
    if E % ws != 0:
        raise ValueError(f"E={E} experts do not split over {ws} ranks")
    e_local = E // ws
    T, H = x.shape
    ids, w = route(logits)
    if tuple(ids.shape) != (T, k) or tuple(w.shape) != (T, k):
        raise ValueError("route() must return ids and weights of shape [T, k]")

    send_counts, send_tokens, row_of = ops.dispatch(ids, e_local, ws)
    recv_counts_t = torch.empty_like(send_counts)
    dist.all_to_all_single(recv_counts_t, send_counts, group=group)
    counts = torch.cat([send_counts, recv_counts_t]).tolist()  # the one host wait
    send_counts_l, recv_counts_l = counts[:ws], counts[ws:]
    n_send = sum(send_counts_l)

    x_send, ids_send, w_send = ops.pack(x, ids, w, send_counts, send_tokens, ws)
    x_recv = _exchange(x_send[:n_send], send_counts_l, recv_counts_l, H, group)
    ids_recv = _exchange(ids_send[:n_send], send_counts_l, recv_counts_l, k, group)
    w_recv = _exchange(w_send[:n_send], send_counts_l, recv_counts_l, k, group)

    partial = local_forward(x_recv, ids_recv, w_recv)
    if tuple(partial.shape) != (sum(recv_counts_l), H):
        raise ValueError("local_forward() must return [rows received, H]")
    back = _exchange(partial.float(), recv_counts_l, send_counts_l, H, group)
    return ops.combine(back, row_of, T, H, ws)
