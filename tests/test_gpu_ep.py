"""GPU checks of the expert-parallel exchange's library calls (moe_ep_dispatch,
moe_ep_pack, moe_ep_combine) against the plain-torch statement of the same
steps, bit for bit, on several ranks' worth of picks held by one GPU (no
communication: the calls are per-rank arithmetic)."""
import pytest
import torch

import oracle
from ep_reference import TorchEpOps
from serving_moe_route_gb300 import workloads as W
from serving_moe_route_gb300.ep import LibraryEpOps

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,E,k,ep,H", [(50, 32, 4, 4, 256), (37, 30, 3, 3, 96), (1, 16, 8, 8, 64),
                                        (1500, 64, 6, 8, 128), (0, 16, 2, 2, 64)])
def test_ep_calls_match_reference(T, E, k, ep, H):
    dev = torch.device("cuda", 0)
    wl = W.custom("ep_calls", T=max(T, 1), H=H, I=64, E=E, k=k, dtype=W.BF16, seed=70 + T,
                  logits="nan_rows")
    act = W.make_activations(wl)
    ids, w = oracle.route(act["logits"].float().numpy(), k)
    ids = torch.from_numpy(ids)[:T].contiguous()
    w = torch.from_numpy(w).float()[:T].contiguous()
    x = act["x"][:T].contiguous()
    ref, lib = TorchEpOps(), LibraryEpOps()
    e_local = E // ep

    rc, rt, rr = ref.dispatch(ids, e_local, ep)
    gc, gt, gr = lib.dispatch(ids.to(dev), e_local, ep)
    n = int(rc.sum())
    assert torch.equal(gc.cpu(), rc)
    assert torch.equal(gt.cpu()[:n], rt[:n])
    assert torch.equal(gr.cpu(), rr)

    xs, is_, ws_ = lib.pack(x.to(dev), ids.to(dev), w.to(dev), gc, gt, ep)
    rxs, ris, rws = ref.pack(x, ids, w, rc, rt, ep)
    assert torch.equal(xs.cpu()[:n], rxs[:n])
    assert torch.equal(is_.cpu()[:n], ris[:n])
    assert torch.equal(ws_.cpu()[:n], rws[:n])

    g = torch.Generator().manual_seed(5)
    back = torch.randn(max(n, 1), H, generator=g)
    got = lib.combine(back.to(dev), gr, T, H, ep).cpu()
    want = ref.combine(back, rr, T, H, ep)
    assert torch.equal(got, want)  # same additions in the same (rank) order
