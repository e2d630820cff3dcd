"""Shared helpers of the GPU parity tests: run a workload through the CUDA
path (via the C ABI) and through the oracle, compare.  Tolerances:
bit-exact for ids, counts, offsets, src, pos and tile lists; for outputs
max|gpu - oracle| <= tol * max|oracle| over every token, with
tol = 2e-2 for bf16 and for the TF32 path of the f32 layer, 5e-2 for FP8;
routing weights within 2e-6 absolute (fp32 exp against the oracle's
double exp)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from serving_moe_route_gb300 import MoELayer
from serving_moe_route_gb300 import workloads as W

TOL = {W.F32: 2e-2, W.BF16: 2e-2, W.FP8: 5e-2}
W_ATOL = 2e-6

_WEIGHT_CACHE: dict = {}


def inputs(wl: W.Workload) -> dict:
    """make_inputs(wl), with the weights (which depend on H, I, E, dtype,
    seed and the expert-parallel slice only) kept for the next workload
    that shares them."""
    key = (wl.H, wl.I, wl.E, wl.dtype, wl.seed, wl.ep_size, wl.ep_rank)
    if key not in _WEIGHT_CACHE:
        _WEIGHT_CACHE.clear()
        _WEIGHT_CACHE[key] = W.make_weights(wl)
    out = dict(_WEIGHT_CACHE[key])
    out.update(W.make_activations(wl))
    return out


def all_tokens(wl) -> np.ndarray:
    return np.arange(wl.T, dtype=np.int32)


def logits_f32(inp) -> np.ndarray:
    return inp["logits"].float().numpy()


def make_layer(wl, inp) -> MoELayer:
    dev = torch.device("cuda", 0)
    s13 = inp["s13"].to(dev) if inp["s13"] is not None else None
    s2 = inp["s2"].to(dev) if inp["s2"] is not None else None
    return MoELayer(inp["w13"].to(dev), inp["w2"].to(dev), k=wl.k, dtype=wl.dtype,
                    scoring=wl.scoring, renorm=wl.renorm, s13=s13, s2=s2, force_est=wl.force_est,
                    ep_size=wl.ep_size, ep_rank=wl.ep_rank, n_group=wl.n_group,
                    topk_group=wl.topk_group, gemm_pair=wl.gemm_pair,
                    gemm_tm=wl.gemm_tm)


def run_gpu(wl, inp, layer=None):
    layer = layer or make_layer(wl, inp)
    dev = layer.device
    x = inp["x"].to(dev)
    lg = inp["logits"].to(dev)
    out = layer.forward(x, lg)
    rc, bits = layer.check(wl.T)
    assert rc == 0, f"device error word {bits:#x}"
    inter = {k: v.cpu().numpy().copy() for k, v in layer.intermediates(wl.T).items()}
    inter["tile_n"] = layer.plan(wl.T).tile_n
    inter["gemm_pair"] = layer.plan(wl.T).gemm_pair
    inter["gemm_tm"] = layer.plan(wl.T).gemm_tm
    # plans that pick the GEMM kernel family on the device: an expert with 256
    # or more rows selects CTA pairs
    inter["dyn_family"] = bool(layer.plan(wl.T).gemm_dyn)
    inter["est"] = layer.plan(wl.T).est
    return out.float().cpu().double().numpy(), inter, layer


def run_oracle(wl, inp, tokens):
    return oracle.moe_forward(
        T=wl.T, H=wl.H, I=wl.I, E=wl.E, k=wl.k, dtype=wl.dtype, scoring=wl.scoring,
        renorm=wl.renorm, x=W.storage_numpy(inp["x"]), logits=W.storage_numpy(inp["logits"]),
        w13=W.storage_numpy(inp["w13"]), w2=W.storage_numpy(inp["w2"]),
        s13=W.storage_numpy(inp["s13"]), s2=W.storage_numpy(inp["s2"]), tokens=tokens,
        ep_size=wl.ep_size, ep_rank=wl.ep_rank, n_group=wl.n_group, topk_group=wl.topk_group)


def check_routing_and_permutation(wl, inp, inter):
    """ids / w / counts / offsets / src / pos against the oracle, all tokens."""
    if wl.n_group > 1:
        ids_ref, w_ref = oracle.route_grouped(logits_f32(inp), wl.k, wl.n_group, wl.topk_group,
                                              scoring=wl.scoring, renorm=wl.renorm)
    else:
        ids_ref, w_ref = oracle.route(logits_f32(inp), wl.k, scoring=wl.scoring,
                                      renorm=wl.renorm)
    np.testing.assert_array_equal(inter["ids"], ids_ref)
    np.testing.assert_allclose(inter["w"], w_ref, rtol=0, atol=W_ATOL)
    flat = ids_ref.reshape(-1)
    E_loc = wl.E // wl.ep_size
    if wl.ep_size == 1:
        counts, offsets, src, pos = oracle.permute(flat, wl.E)
        np.testing.assert_array_equal(inter["src"], src)
    else:
        # an expert-parallel slice permutes only the picks of its own experts,
        # in (local expert, flat index) order; the other picks get pos -1
        local = flat - wl.ep_rank * E_loc
        valid = (local >= 0) & (local < E_loc)
        counts = np.bincount(local[valid], minlength=E_loc).astype(np.int32)
        offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
        order = np.nonzero(valid)[0][np.argsort(local[valid], kind="stable")]
        pos = np.full(flat.size, -1, np.int32)
        pos[order] = np.arange(order.size, dtype=np.int32)
        np.testing.assert_array_equal(inter["src"][:order.size], order)
    np.testing.assert_array_equal(inter["counts"], counts)
    np.testing.assert_array_equal(inter["offsets"], offsets)
    np.testing.assert_array_equal(inter["pos"], pos)
    # the tile list covers every expert's rows exactly once, in expert order,
    # each tile at most its width; the width is the plan's tile (from the
    # estimate) widened per expert to 32/64/128 by its row count (BF16/F32);
    # GEMM2's list of a prefill-sized plan goes up to 256, and CTA-pair
    # plans share one list with widths up to 256
    tile_n = int(inter["tile_n"])
    # FP8: the kernel width is the plan's tile, or twice it (at most 64) when
    # experts average more than half a tile; then widths grow per expert too
    est = int(inter["est"])
    fp8_nt = 2 * tile_n if (2 * est > tile_n and tile_n < 64) else tile_n
    tm = wl.dtype == W.FP8 and int(inter["gemm_tm"])
    if inter.get("dyn_family"):
        hot = int(counts.max()) >= 256 if counts.size else False
        assert int(inter["family"][0]) == (2 if hot else 1), (inter["family"], counts.max())
    if (int(inter["gemm_pair"]) or (inter.get("dyn_family") and int(inter["family"][0]) == 2)) \
            and wl.dtype != W.FP8:
        lists = [("tiles", "ntiles", 256)]
    elif tm:  # token-major FP8: every expert's rows in tiles of 128
        lists = [("tiles", "ntiles", 128)]
    elif wl.dtype == W.FP8:
        lists = [("tiles", "ntiles", fp8_nt)]
    else:
        lists = [("tiles", "ntiles", 128)]
        if wl.dtype != W.FP8 and tile_n >= 128:
            lists.append(("tiles2", "ntiles2", 256))  # GEMM2's own list, widths up to 256
    for key, nkey, n_max in lists:
        nt = int(inter[nkey][0])
        rows = np.zeros(E_loc, np.int64)
        for e, r0, n, width in inter[key][:nt]:
            assert 0 <= e < E_loc and 1 <= n <= width
            assert offsets[e] <= r0 and r0 + n <= offsets[e + 1]
            c = counts[e]
            bucket = 16 if c <= 16 else 32 if c <= 32 else 64 if c <= 64 else 128 if c <= 128 \
                else 256
            if tm:
                want = 128
            elif wl.dtype == W.FP8 and fp8_nt == tile_n:
                want = tile_n
            else:
                want = min(n_max, max(tile_n, bucket))
            assert width == want, (key, e, c, width, want)
            # an expert's rows are split evenly over ceil(c / width) tiles:
            # every tile but the last holds `step` rows (the even share
            # rounded up to 16, at most the width), in row order
            ntl = -(-c // width)
            step = width if ntl == 1 else min(width, -(-(-(-c // ntl)) // 16) * 16)
            i = (r0 - offsets[e]) // step
            assert r0 == offsets[e] + i * step and i < ntl, (key, e, c, r0, step)
            assert n == min(step, c - i * step), (key, e, c, i, n, step)
            rows[e] += n
        np.testing.assert_array_equal(rows, counts)
    return ids_ref, w_ref


def check_outputs(wl, out_gpu, out_ref, tokens):
    got = out_gpu[tokens]
    assert np.isfinite(got).all(), "non-finite output"
    err = np.abs(got - out_ref).max()
    scale = np.abs(out_ref).max()
    assert scale > 0
    assert err <= TOL[wl.dtype] * scale, f"max|err| {err:.3e} > {TOL[wl.dtype]} * {scale:.3e}"
    return err / scale
