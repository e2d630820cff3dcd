"""Expert parallelism across ranks on CPU: two gloo ranks run ep_forward
(route, send plan, all-to-all dispatch, local slice, all-to-all return,
combine); the output for each rank's tokens must equal the oracle's full
layer.  The local slice here is a float64 dense reference of the rank's own
experts, and the send plan, packing and combine are the plain-torch reference
of tests/ep_reference.py; on GPUs they are an expert-parallel MoELayer and
the library's moe_ep_* calls."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _silu(z):
    return z / (1.0 + np.exp(-z))


def _rank_main(rank, world, port, split, q):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from serving_moe_route_gb300 import workloads as W
        from ep_reference import TorchEpOps
        from serving_moe_route_gb300.ep import ep_forward

        T, H, I, E, k = sum(split), 128, 64, 8, 2
        wl = W.custom("ep_x", T=T, H=H, I=I, E=E, k=k, dtype=W.F32, seed=61, logits="nan_rows")
        inp = W.make_inputs(wl)
        x_all = inp["x"].float()
        lg_all = inp["logits"].float()
        w13 = inp["w13"].double().numpy()
        w2 = inp["w2"].double().numpy()
        t0 = sum(split[:rank])
        tok = slice(t0, t0 + split[rank])
        e_local = E // world

        def route(logits):
            ids, w = oracle.route(logits.numpy(), k)
            return torch.from_numpy(ids), torch.from_numpy(w.astype(np.float32))

        def local_forward(xr, idr, wr):
            out = np.zeros((xr.shape[0], H))
            xs = xr.double().numpy()
            for t in range(xs.shape[0]):
                for j in range(k):
                    e = int(idr[t, j])
                    if rank * e_local <= e < (rank + 1) * e_local:
                        h = w13[e] @ xs[t]
                        out[t] += float(wr[t, j]) * (w2[e] @ (_silu(h[:I]) * h[I:]))
            return torch.from_numpy(out.astype(np.float32))

        got = ep_forward(x_all[tok].contiguous(), lg_all[tok].contiguous(), k=k, E=E,
                         route=route, local_forward=local_forward, ops=TorchEpOps())
        ref, _, _ = oracle.moe_forward(
            T=T, H=H, I=I, E=E, k=k, dtype=wl.dtype, scoring=wl.scoring, renorm=wl.renorm,
            x=W.storage_numpy(inp["x"]), logits=W.storage_numpy(inp["logits"]),
            w13=W.storage_numpy(inp["w13"]), w2=W.storage_numpy(inp["w2"]))
        ref = ref[tok]
        err = float(np.abs(got.numpy() - ref).max()) if ref.size else 0.0
        scale = float(np.abs(ref).max()) if ref.size else 1.0
        q.put((rank, got.shape[0], err, scale))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("split", [(6, 6), (5, 9), (0, 7)])
def test_ep_forward_two_gloo_ranks_equals_full_layer(split):
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, split, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(180)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, n, err, scale in got:
        assert n == split[rank]
        assert err <= 1e-5 * max(scale, 1e-30), (rank, err, scale)
