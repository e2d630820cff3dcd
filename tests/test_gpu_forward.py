"""GPU parity of the whole layer (moe_forward through the C ABI) against the
oracle on every named workload (all that the benchmark times) and on edge
cases: routing and permutation bit-exact on every token, outputs within
tolerance on every token."""
import numpy as np
import pytest
import torch

import oracle
import parity_util as PU
from serving_moe_route_gb300 import MoELayer
from serving_moe_route_gb300 import workloads as W
from serving_moe_route_gb300 import _binding as B

pytestmark = pytest.mark.gpu

WL = W.workloads()


@pytest.mark.parametrize("name", list(WL))
def test_forward_workload(name):
    wl = WL[name]
    inp = PU.inputs(wl)
    out, inter, _ = PU.run_gpu(wl, inp)
    PU.check_routing_and_permutation(wl, inp, inter)
    tokens = PU.all_tokens(wl)
    ref, ids_o, _ = PU.run_oracle(wl, inp, tokens)
    np.testing.assert_array_equal(inter["ids"], ids_o)
    PU.check_outputs(wl, out, ref, tokens)


EDGE = [
    # ragged: E not a multiple of 32, T not a multiple of the routing chunk
    W.custom("ragged_bf16", T=37, H=256, I=128, E=40, k=3, dtype=W.BF16, seed=21),
    W.custom("ragged_fp8", T=37, H=256, I=128, E=40, k=3, dtype=W.FP8, seed=22),
    W.custom("ragged_f32", T=29, H=96, I=64, E=12, k=4, dtype=W.F32, seed=23),
    W.custom("single_token", T=1, H=2048, I=768, E=128, k=8, dtype=W.BF16, seed=24),
    W.custom("k1", T=50, H=128, I=128, E=16, k=1, dtype=W.BF16, seed=25),
    W.custom("one_expert", T=33, H=128, I=64, E=1, k=1, dtype=W.BF16, seed=26),
    W.custom("all_nan", T=40, H=256, I=128, E=64, k=8, dtype=W.BF16, seed=27, logits="nan_rows"),
    W.custom("sigmoid_no_renorm", T=45, H=256, I=128, E=64, k=4, dtype=W.BF16, seed=28,
             scoring=W.SIGMOID, renorm=False),
    W.custom("softmax_no_renorm", T=45, H=256, I=128, E=64, k=4, dtype=W.FP8, seed=29,
             renorm=False),
    W.custom("many_tiles", T=600, H=256, I=256, E=8, k=2, dtype=W.BF16, seed=30),
    W.custom("big_tiles_fp8", T=300, H=256, I=256, E=4, k=2, dtype=W.FP8, seed=31),
    W.custom("forced_est", T=100, H=256, I=128, E=64, k=4, dtype=W.BF16, seed=32, force_est=100),
    W.custom("prefill_chunks", T=2500, H=128, I=128, E=32, k=4, dtype=W.BF16, seed=33),
    W.custom("grouped_fp8", T=70, H=256, I=128, E=32, k=4, dtype=W.FP8, seed=42,
             logits="nan_rows", n_group=8, topk_group=2),
    W.custom("grouped_sigmoid", T=70, H=256, I=128, E=48, k=6, dtype=W.BF16, seed=43,
             scoring=W.SIGMOID, n_group=6, topk_group=3),
    # CTA-pair GEMMs: TF32; I and H not multiples of 256 (the second CTA's
    # rows are masked in the last block); the single-CTA path forced on a
    # prefill-sized plan and the pair path forced on a decode-sized one
    W.custom("pair_f32", T=300, H=160, I=96, E=8, k=2, dtype=W.F32, seed=44),
    W.custom("pair_odd_blocks", T=600, H=384, I=384, E=8, k=2, dtype=W.BF16, seed=45),
    W.custom("single_cta_prefill", T=600, H=256, I=256, E=8, k=2, dtype=W.BF16, seed=46,
             gemm_pair=0),
    W.custom("pair_decode", T=64, H=256, I=256, E=32, k=4, dtype=W.BF16, seed=47,
             logits="nan_rows", gemm_pair=1),
    # FP8 with experts averaging more than half a tile: the kernel one width
    # up and per-expert widths (est 12 -> 32-wide kernel; est 24 -> 64)
    W.custom("fp8_wider_32", T=96, H=256, I=256, E=32, k=4, dtype=W.FP8, seed=48),
    W.custom("fp8_wider_64", T=192, H=256, I=256, E=32, k=4, dtype=W.FP8, seed=49,
             logits="nan_rows"),
    # token-major FP8 GEMMs (tokens on the MMA's M side, 128-row tiles):
    # forced on small and ragged shapes (partial tiles, every token box
    # height, H not a multiple of 256 so GEMM2's last item has one valid
    # 128-row block), a hot expert with many tiles, and the other FP8 path
    # forced on a plan that would pick token-major
    W.custom("tm_ragged", T=37, H=384, I=256, E=40, k=3, dtype=W.FP8, seed=63, gemm_tm=1),
    W.custom("tm_small", T=1, H=256, I=128, E=8, k=2, dtype=W.FP8, seed=64, gemm_tm=1),
    W.custom("tm_many_tiles", T=700, H=256, I=384, E=8, k=2, dtype=W.FP8, seed=65,
             logits="nan_rows"),
    W.custom("tm_concentrated", T=400, H=256, I=256, E=64, k=4, dtype=W.FP8, seed=66,
             logits="concentrated", gemm_tm=1),
    W.custom("tm_sigmoid", T=300, H=256, I=256, E=16, k=4, dtype=W.FP8, seed=67,
             scoring=W.SIGMOID),
    W.custom("swap_ab_large_fp8", T=700, H=256, I=384, E=8, k=2, dtype=W.FP8, seed=65,
             gemm_tm=0),
    # the kernel family chosen on the device (BF16, est <= 32, T >= 256): hot
    # experts (>= 256 rows) select CTA pairs, uniform routing one CTA per tile
    # (concentrated: ~90% of the picks on 6 experts, so each holds ~T*k*0.15 rows)
    W.custom("family_pair", T=520, H=256, I=256, E=128, k=4, dtype=W.BF16, seed=68,
             logits="concentrated"),
    W.custom("family_single", T=300, H=256, I=256, E=64, k=4, dtype=W.BF16, seed=69),
    W.custom("family_pair_f32", T=1000, H=128, I=96, E=128, k=2, dtype=W.F32, seed=71,
             logits="concentrated"),
]


@pytest.mark.parametrize("wl", EDGE, ids=[w.name for w in EDGE])
def test_forward_edge(wl):
    inp = W.make_inputs(wl)
    if wl.name == "all_nan":
        inp["logits"][:] = float("nan")
    out, inter, _ = PU.run_gpu(wl, inp)
    PU.check_routing_and_permutation(wl, inp, inter)
    tokens = PU.all_tokens(wl)
    ref, _, _ = PU.run_oracle(wl, inp, tokens)
    PU.check_outputs(wl, out, ref, tokens)


def test_all_tokens_on_the_same_experts():
    # every token routed to the same k experts: the crash repro shape of
    # PR #39593 (one expert gets T rows, the rest none)
    wl = W.custom("same_experts", T=300, H=256, I=128, E=64, k=4, dtype=W.BF16, seed=34)
    inp = W.make_inputs(wl)
    lg = torch.zeros(wl.T, wl.E)
    lg[:, [5, 17, 2, 60]] = torch.tensor([4.0, 3.0, 2.0, 1.0])
    inp["logits"] = lg.to(torch.bfloat16)
    out, inter, _ = PU.run_gpu(wl, inp)
    PU.check_routing_and_permutation(wl, inp, inter)
    assert sorted(np.nonzero(inter["counts"])[0].tolist()) == [2, 5, 17, 60]
    tokens = PU.all_tokens(wl)
    ref, _, _ = PU.run_oracle(wl, inp, tokens)
    PU.check_outputs(wl, out, ref, tokens)


def test_fp8_activation_quantisation_bit_exact():
    wl = WL["fp8_T16"]
    inp = PU.inputs(wl)
    _, inter, _ = PU.run_gpu(wl, inp)
    x = inp["x"].float().numpy()
    src = inter["src"]
    for slot in range(wl.T * wl.k):
        t = src[slot] // wl.k
        codes, scales = oracle.quant_group128(x[t])
        np.testing.assert_array_equal(inter["xq"][slot], codes)
        np.testing.assert_array_equal(inter["xs"][slot], scales)


def test_empty_batch_enqueues_nothing():
    wl = W.custom("empty", T=0, H=256, I=128, E=8, k=2, dtype=W.BF16, seed=35)
    dev = torch.device("cuda", 0)
    inp = W.make_inputs(W.custom(T=1, H=256, I=128, E=8, k=2, dtype=W.BF16, seed=35))
    layer = PU.make_layer(wl, inp)
    out = layer.forward(torch.empty(0, 256, dtype=torch.bfloat16, device=dev),
                        torch.empty(0, 8, dtype=torch.bfloat16, device=dev))
    assert out.shape == (0, 256)


def test_repeated_calls_are_deterministic():
    wl = W.custom("repeat", T=64, H=256, I=128, E=16, k=4, dtype=W.BF16, seed=36)
    inp = W.make_inputs(wl)
    layer = PU.make_layer(wl, inp)
    a, _, _ = PU.run_gpu(wl, inp, layer)
    b, _, _ = PU.run_gpu(wl, inp, layer)
    # the combine sums each token's k rows in pick order: bit-identical calls
    np.testing.assert_array_equal(a, b)


def test_with_ids_matches_routed_forward():
    wl = W.custom("with_ids", T=64, H=256, I=128, E=32, k=4, dtype=W.BF16, seed=37)
    inp = W.make_inputs(wl)
    out, inter, layer = PU.run_gpu(wl, inp)
    dev = layer.device
    ids = torch.from_numpy(inter["ids"]).to(dev)
    w = torch.from_numpy(inter["w"]).to(dev)
    out2 = layer.forward_with_ids(inp["x"].to(dev), ids, w)
    rc, bits = layer.check(wl.T)
    assert rc == 0 and bits == 0
    o2 = out2.float().cpu().double().numpy()
    np.testing.assert_array_equal(o2, out)


def test_with_ids_reports_bad_and_duplicate_ids():
    # duplicate / out-of-range ids are reported in the error word and skipped,
    # never used as an index (the PR #39593 failure mode)
    wl = W.custom("bad_ids", T=32, H=256, I=128, E=16, k=4, dtype=W.BF16, seed=38)
    inp = W.make_inputs(wl)
    layer = PU.make_layer(wl, inp)
    dev = layer.device
    ids = torch.tensor([[0, 1, 2, 3]] * wl.T, dtype=torch.int32)
    ids[3] = torch.tensor([7, 7, 7, 7])          # duplicates
    ids[9] = torch.tensor([1, 99, -4, 2])        # out of range
    w = torch.full((wl.T, wl.k), 0.25)
    out = layer.forward_with_ids(inp["x"].to(dev), ids.to(dev), w.to(dev))
    rc, bits = layer.check(wl.T)
    assert rc == B.MOE_ERR_DEVICE
    assert bits & B.MOE_DEVERR_DUP_ID and bits & B.MOE_DEVERR_BAD_ID
    inter = layer.intermediates(wl.T)
    got_ids = inter["ids"].cpu().numpy()
    assert list(got_ids[3]) == [7, -1, -1, -1]
    assert list(got_ids[9]) == [1, -1, -1, 2]
    assert int(inter["counts"].sum()) == wl.T * wl.k - 5
    assert torch.isfinite(out.float()).all()
    # the context is still healthy: a normal call succeeds afterwards
    PU.run_gpu(wl, inp, layer)


def test_forward_in_a_cuda_graph():
    # the whole forward (its launches and the error-word memset) captures
    # into one CUDA graph and replays with new inputs in the same buffers
    wl = W.custom("graph", T=80, H=256, I=128, E=24, k=4, dtype=W.FP8, seed=39)
    inp = W.make_inputs(wl)
    inp2 = W.make_activations(W.custom(T=80, H=256, I=128, E=24, k=4, dtype=W.FP8, seed=40))
    layer = PU.make_layer(wl, inp)
    dev = layer.device
    x = inp["x"].to(dev)
    lg = inp["logits"].to(dev)
    out = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device=dev)
    eager1 = layer.forward(x, lg).clone()
    eager2 = layer.forward(inp2["x"].to(dev), inp2["logits"].to(dev)).clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        layer.forward(x, lg, out)
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layer.forward(x, lg, out)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager1)
    x.copy_(inp2["x"])
    lg.copy_(inp2["logits"])
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager2)
    rc, bits = layer.check(wl.T)
    assert rc == 0, bits


def test_per_call_family_in_a_cuda_graph():
    # a plan that picks the GEMM kernel family per call, captured once and
    # replayed on inputs that alternate between concentrated routing (CTA
    # pairs) and uniform routing (one CTA per tile), the launches of the
    # family not picked returning at once.  Each input's eager output matches
    # the oracle; every replay equals it bit for bit, so no replay reads
    # permuted rows, tile lists or a family word left by the one before.
    shape = dict(T=520, H=256, I=256, E=128, k=4, dtype=W.BF16)
    kinds = [(72, "concentrated", 2), (73, "concentrated", 2), (74, "normal", 1)]
    wl = W.custom("family_graph", seed=72, logits="concentrated", **shape)
    inp = W.make_inputs(wl)
    layer = PU.make_layer(wl, inp)
    assert layer.plan(wl.T).gemm_dyn == 1
    dev = layer.device
    tokens = PU.all_tokens(wl)
    acts = [W.make_activations(W.custom(seed=s, logits=lk, **shape)) for s, lk, _ in kinds]
    eager = []
    for a, (_, _, fam) in zip(acts, kinds):
        o = layer.forward(a["x"].to(dev), a["logits"].to(dev)).clone()
        rc, bits = layer.check(wl.T)
        assert rc == 0, bits
        assert int(layer.intermediates(wl.T)["family"][0]) == fam
        full = dict(inp)
        full.update(a)
        ref, _, _ = PU.run_oracle(wl, full, tokens)
        PU.check_outputs(wl, o.float().cpu().double().numpy(), ref, tokens)
        eager.append(o)
    x = acts[0]["x"].to(dev)
    lg = acts[0]["logits"].to(dev)
    out = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device=dev)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        layer.forward(x, lg, out)
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layer.forward(x, lg, out)
    for i in range(24):
        j = i % len(kinds)
        x.copy_(acts[j]["x"])
        lg.copy_(acts[j]["logits"])
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager[j]), (i, j)
        assert int(layer.intermediates(wl.T)["family"][0]) == kinds[j][2]
    rc, bits = layer.check(wl.T)
    assert rc == 0, bits


@pytest.mark.parametrize("dtype", [W.BF16, W.FP8])
def test_expert_parallel_slices(dtype):
    # each expert-parallel rank computes its experts' share (ids global and
    # bit-exact, local counts and permutation bit-exact, outputs against the
    # oracle's rank slice); the ranks' outputs add up to the whole layer
    ep, E = 4, 16
    full_wl = W.custom("ep_full", T=60, H=256, I=128, E=E, k=3, dtype=dtype, seed=41,
                       logits="nan_rows")
    inp = W.make_inputs(full_wl)
    full_out, _, _ = PU.run_gpu(full_wl, inp)
    ids_ref, _ = oracle.route(PU.logits_f32(inp), full_wl.k)
    flat = ids_ref.reshape(-1)
    el = E // ep
    total = np.zeros_like(full_out)
    for r in range(ep):
        wl = W.custom("ep_rank", T=60, H=256, I=128, E=E, k=3, dtype=dtype, seed=41,
                      logits="nan_rows", ep_size=ep, ep_rank=r)
        inp_r = dict(inp)
        for key in ("w13", "w2", "s13", "s2"):
            if inp[key] is not None:
                inp_r[key] = inp[key][r * el:(r + 1) * el].contiguous()
        out, inter, _ = PU.run_gpu(wl, inp_r)
        np.testing.assert_array_equal(inter["ids"], ids_ref)
        local = flat - r * el
        valid = (local >= 0) & (local < el)
        np.testing.assert_array_equal(inter["counts"], np.bincount(local[valid], minlength=el))
        order = np.nonzero(valid)[0][np.argsort(local[valid], kind="stable")]
        n_valid = int(valid.sum())
        np.testing.assert_array_equal(inter["src"][:n_valid], order)
        pos = np.full(flat.size, -1, np.int32)
        pos[order] = np.arange(n_valid, dtype=np.int32)
        np.testing.assert_array_equal(inter["pos"], pos)
        ref, _, _ = PU.run_oracle(wl, inp_r, np.arange(wl.T, dtype=np.int32))
        PU.check_outputs(wl, out, ref, np.arange(wl.T))
        total += out
    tol = PU.TOL[dtype] * np.abs(full_out).max()
    assert np.abs(total - full_out).max() <= tol



@pytest.mark.gpu
def test_ep_forward_single_rank_nccl():
    # the expert-parallel exchange driving the GPU layer through NCCL; with
    # one rank every pick is local, so it must reproduce the plain layer
    import socket

    import torch.distributed as dist

    from serving_moe_route_gb300 import route_topk
    from serving_moe_route_gb300.ep import ep_forward

    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1)
    try:
        wl = W.custom("ep_nccl", T=40, H=256, I=128, E=16, k=4, dtype=W.BF16, seed=62,
                      logits="nan_rows")
        inp = W.make_inputs(wl)
        layer = PU.make_layer(wl, inp)
        dev = layer.device
        x, lg = inp["x"].to(dev), inp["logits"].to(dev)
        got = ep_forward(x, lg, k=wl.k, E=wl.E, route=lambda t: route_topk(t, wl.k),
                         local_forward=layer.forward_with_ids)
        torch.cuda.synchronize()
        tokens = np.arange(wl.T, dtype=np.int32)
        ref, _, _ = PU.run_oracle(wl, inp, tokens)
        PU.check_outputs(wl, got.double().cpu().numpy(), ref, tokens)
    finally:
        dist.destroy_process_group()
