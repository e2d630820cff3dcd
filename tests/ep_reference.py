"""Plain-torch statement of the expert-parallel exchange's send plan, packing
and combine (test infrastructure): the CPU gloo test runs ep_forward with it,
and the GPU test compares the library's moe_ep_* calls against it."""
from __future__ import annotations

import torch


class TorchEpOps:
    def dispatch(self, ids: torch.Tensor, e_local: int, ep_size: int):
        T, k = ids.shape
        owner = ids.long() // e_local
        valid = (ids >= 0) & (owner < ep_size)
        send_counts = torch.zeros(ep_size, dtype=torch.int32)
        send_tokens = torch.full((max(1, T * ep_size),), -1, dtype=torch.int32)
        row_of = torch.full((T, ep_size), -1, dtype=torch.int32)
        row = 0
        for d in range(ep_size):  # destination ranks in rank order
            for t in range(T):    # tokens in token order
                if bool(((owner[t] == d) & valid[t]).any()):
                    row_of[t, d] = row
                    send_tokens[row] = t
                    send_counts[d] += 1
                    row += 1
        return send_counts, send_tokens, row_of

    def pack(self, x, ids, w, send_counts, send_tokens, ep_size: int):
        n = int(send_counts.sum())
        rows = max(1, x.shape[0] * ep_size)
        x_send = torch.zeros(rows, x.shape[1], dtype=x.dtype)
        ids_send = torch.zeros(rows, ids.shape[1], dtype=torch.int32)
        w_send = torch.zeros(rows, w.shape[1], dtype=torch.float32)
        for r in range(n):
            t = int(send_tokens[r])
            x_send[r], ids_send[r], w_send[r] = x[t], ids[t], w[t]
        return x_send, ids_send, w_send

    def combine(self, back, row_of, T: int, H: int, ep_size: int):
        out = torch.zeros(T, H, dtype=torch.float32)
        for t in range(T):
            for d in range(ep_size):  # owners in rank order
                r = int(row_of[t, d])
                if r >= 0:
                    out[t] += back[r].float()
        return out
