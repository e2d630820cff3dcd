"""GPU parity of step a-1 (moe_route_topk through the C ABI) against the
oracle: ids bit-exact (ties to the lower expert index, NaN -> -FLT_MAX,
k distinct ids), weights within 2e-6."""
import numpy as np
import pytest
import torch

import oracle
from serving_moe_route_gb300 import route_topk
from serving_moe_route_gb300 import workloads as W

pytestmark = pytest.mark.gpu

WL = W.workloads()


def _compare(logits_cpu, k, scoring, renorm):
    dev = torch.device("cuda", 0)
    ids, w = route_topk(logits_cpu.to(dev), k, scoring=scoring, renorm=renorm)
    torch.cuda.synchronize()
    ids_ref, w_ref = oracle.route(logits_cpu.float().numpy(), k, scoring=scoring, renorm=renorm)
    np.testing.assert_array_equal(ids.cpu().numpy(), ids_ref)
    np.testing.assert_allclose(w.cpu().numpy(), w_ref, rtol=0, atol=2e-6)
    ids_np = ids.cpu().numpy()
    for row in ids_np:
        assert len(set(row.tolist())) == k
    return ids_np


@pytest.mark.parametrize("name", ["tiny_f32", "decode_bf16", "sparse_uniform_bf16",
                                  "sparse_concentrated_bf16", "skewed_prefill_bf16",
                                  "skewed_prefill_sigmoid_bf16", "fp8_T4096"])
@pytest.mark.parametrize("renorm", [True, False])
def test_route_workloads(name, renorm):
    wl = WL[name]
    x = None
    if wl.logits == "router":
        x = W.make_inputs(W.custom(T=wl.T, H=wl.H, I=wl.I, E=wl.E, k=wl.k, dtype=wl.dtype,
                                   seed=wl.seed))["x"]
    lg = W.make_logits(wl, x)
    _compare(lg, wl.k, wl.scoring, renorm)


@pytest.mark.parametrize("scoring", [0, 1])
@pytest.mark.parametrize("E,k", [(8, 2), (40, 3), (128, 8), (400, 6), (1024, 32), (33, 32),
                                 (1, 1), (64, 1), (250, 6), (260, 6)])
def test_route_edge_rows(E, k, scoring):
    g = torch.Generator().manual_seed(E * 100 + k)
    T = 70
    lg = torch.randn(T, E, generator=g)
    lg[0] = float("nan")                      # all-NaN row
    lg[1] = 0.5                               # all-equal row
    lg[2, : E // 2] = float("nan")            # half NaN
    lg[3] = torch.randint(-2, 3, (E,), generator=g).float()  # heavy ties
    lg[4, 0] = float("inf")
    lg[4, E - 1] = float("-inf")
    lg[5] = -1e30
    # signed zeros tie (they compare equal), so the lower expert wins either way
    lg[6] = -1.0
    lg[6, 1::2] = 0.0
    lg[6, 0::2] = -0.0
    lg[7] = float("-inf")
    lg[7, E - 1] = -0.0
    lg[7, 0] = 0.0
    for dt in (torch.float32, torch.bfloat16):
        ids = _compare(lg.to(dt), k, scoring, True)
        assert list(ids[0]) == list(range(k))
        assert list(ids[1]) == list(range(k))


def test_route_unaligned_logits_pointer():
    # logits read several to a load need an aligned pointer; a view that
    # starts one element into its buffer takes the one-per-load path and
    # must pick the same experts
    g = torch.Generator().manual_seed(11)
    T, E, k = 40, 128, 8
    lg = torch.randn(T, E, generator=g)
    dev = torch.device("cuda", 0)
    for dt in (torch.float32, torch.bfloat16):
        buf = torch.empty(T * E + 1, dtype=dt, device=dev)
        view = buf[1:].view(T, E)
        view.copy_(lg.to(dt).to(dev))
        assert view.data_ptr() % 16 != 0
        ids_u, w_u = route_topk(view, k)
        ids_ref, w_ref = oracle.route(lg.to(dt).float().numpy(), k)
        np.testing.assert_array_equal(ids_u.cpu().numpy(), ids_ref)
        np.testing.assert_allclose(w_u.cpu().numpy(), w_ref, rtol=0, atol=2e-6)


def test_route_rejects_k_above_32():
    from serving_moe_route_gb300 import MoeError
    lg = torch.randn(4, 40, device="cuda")
    with pytest.raises(MoeError):
        route_topk(lg, 33)


def test_route_empty_and_single_token():
    dev = torch.device("cuda", 0)
    ids, w = route_topk(torch.empty(0, 128, dtype=torch.bfloat16, device=dev), 8)
    assert ids.shape == (0, 8)
    lg = torch.full((1, 128), float("nan"), dtype=torch.bfloat16)
    ids = _compare(lg, 8, 0, True)
    assert list(ids[0]) == list(range(8))


@pytest.mark.parametrize("scoring", [0, 1])
@pytest.mark.parametrize("E,k,n_group,topk_group", [(128, 8, 8, 4), (64, 6, 4, 2), (40, 3, 8, 2),
                                                    (256, 8, 32, 4), (16, 4, 16, 4)])
def test_grouped_route_matches_oracle(E, k, n_group, topk_group, scoring):
    g = torch.Generator().manual_seed(E + k + n_group)
    T = 70
    lg = torch.randn(T, E, generator=g)
    lg[0] = float("nan")                      # all-NaN row: distinct, lowest groups
    lg[1] = 0.5
    lg[2, : E // 2] = float("nan")
    lg[3] = torch.randint(-2, 3, (E,), generator=g).float()
    dev = torch.device("cuda", 0)
    for dt in (torch.float32, torch.bfloat16):
        x = lg.to(dt)
        ids, w = route_topk(x.to(dev), k, scoring=scoring, renorm=True, n_group=n_group,
                            topk_group=topk_group)
        torch.cuda.synchronize()
        ids_ref, w_ref = oracle.route_grouped(x.float().numpy(), k, n_group, topk_group,
                                              scoring=scoring, renorm=True)
        np.testing.assert_array_equal(ids.cpu().numpy(), ids_ref)
        np.testing.assert_allclose(w.cpu().numpy(), w_ref, rtol=0, atol=2e-6)
        assert list(ids_ref[0]) == list(range(k))
