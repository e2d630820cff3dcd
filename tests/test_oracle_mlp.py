"""Pins for the oracle's expert MLP and weighted combine (a-4 .. a-7).

References here are written with numpy float64 matrix products and torch's
own bf16 / e4m3 conversions -- a different route to the same definition:
  E=1, k=1 reduces the layer to one dense SwiGLU MLP; identical experts make
  the output independent of routing (weights sum to one); and in general the
  layer equals the dense-gating sum over experts with zero gates off the
  top-k (picks from brute force in test_oracle_route)."""
import numpy as np
import pytest
import torch
from scipy.special import expit, softmax

from serving_moe_route_gb300 import workloads as W


def _silu(z):
    return z * expit(z)


def _mlp(x, w13, w2, I):
    """x [n,H] f64, w13 [2I,H], w2 [H,I] -> [n,H]; gate rows first, up second."""
    g = x @ w13[:I].T
    u = x @ w13[I:].T
    return (_silu(g) * u) @ w2.T


def _f64(t):
    return t.float().double().numpy()


def _run(oracle, wl, inp, tokens=None):
    return oracle.moe_forward(
        T=wl.T, H=wl.H, I=wl.I, E=wl.E, k=wl.k, dtype=wl.dtype, scoring=wl.scoring,
        renorm=wl.renorm, x=W.storage_numpy(inp["x"]), logits=W.storage_numpy(inp["logits"]),
        w13=W.storage_numpy(inp["w13"]), w2=W.storage_numpy(inp["w2"]),
        s13=W.storage_numpy(inp["s13"]), s2=W.storage_numpy(inp["s2"]), tokens=tokens)


@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
def test_single_expert_is_dense_mlp(oracle, dtype):
    wl = W.custom(T=9, H=64, I=32, E=1, k=1, dtype=dtype, seed=4)
    inp = W.make_inputs(wl)
    out, ids, w = _run(oracle, wl, inp)
    assert np.all(ids == 0) and np.allclose(w, 1.0)
    ref = _mlp(_f64(inp["x"]), _f64(inp["w13"][0]), _f64(inp["w2"][0]), wl.I)
    np.testing.assert_allclose(out, ref, rtol=1e-9, atol=1e-12)


def test_identical_experts_ignore_routing(oracle):
    wl = W.custom(T=12, H=64, I=32, E=6, k=3, dtype=W.BF16, seed=5, logits="nan_rows")
    inp = W.make_inputs(wl)
    inp["w13"][:] = inp["w13"][0]
    inp["w2"][:] = inp["w2"][0]
    out, _, w = _run(oracle, wl, inp)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=1e-12)
    ref = _mlp(_f64(inp["x"]), _f64(inp["w13"][0]), _f64(inp["w2"][0]), wl.I)
    np.testing.assert_allclose(out, ref, rtol=1e-9, atol=1e-12)


@pytest.mark.parametrize("scoring", [W.SOFTMAX, W.SIGMOID])
def test_dense_gating_sum(oracle, scoring):
    wl = W.custom(T=10, H=64, I=32, E=8, k=3, dtype=W.BF16, seed=6, scoring=scoring)
    inp = W.make_inputs(wl)
    out, ids, w = _run(oracle, wl, inp)
    x = _f64(inp["x"])
    l = inp["logits"].float().double().numpy()
    ref = np.zeros_like(out)
    for t in range(wl.T):
        top = np.argsort(-l[t], kind="stable")[:wl.k]
        assert list(top) == list(ids[t])
        if scoring == W.SOFTMAX:
            gates = softmax(l[t][top])
        else:
            s = expit(l[t][top])
            gates = s / s.sum()
        for gj, e in zip(gates, top):
            ref[t] += gj * _mlp(x[t:t + 1], _f64(inp["w13"][e]), _f64(inp["w2"][e]), wl.I)[0]
    np.testing.assert_allclose(out, ref, rtol=1e-9, atol=1e-12)


def _torch_fake_quant64(v):
    """per-128-group e4m3 round trip through torch's own conversion; the
    code x scale product is formed in float64, where it is exact"""
    v = torch.from_numpy(np.ascontiguousarray(v, np.float32))
    out = torch.empty(v.numel(), dtype=torch.float64)
    for g0 in range(0, v.numel(), 128):
        grp = v[g0:g0 + 128]
        scale = torch.clamp(grp.abs().max(), min=1e-10) / 448.0
        q = (grp / scale).clamp(-448, 448).to(torch.float8_e4m3fn)
        out[g0:g0 + 128] = q.double() * scale.double()
    return out.numpy()


def test_fp8_block_scaled_against_torch_codec(oracle):
    wl = W.custom(T=5, H=256, I=128, E=4, k=2, dtype=W.FP8, seed=9)
    inp = W.make_inputs(wl)
    out, ids, w = _run(oracle, wl, inp)
    # dequantise with torch's e4m3 conversion and explicit block broadcast
    s13 = inp["s13"].repeat_interleave(128, 1).repeat_interleave(128, 2)
    s2 = inp["s2"].repeat_interleave(128, 1).repeat_interleave(128, 2)
    # products formed in float64, where code x scale is exact
    w13 = (inp["w13"].float().double() * s13.double()).numpy()
    w2 = (inp["w2"].float().double() * s2.double()).numpy()
    x = inp["x"].float().numpy()
    for t in range(wl.T):
        xq = _torch_fake_quant64(x[t])
        acc = np.zeros(wl.H)
        for j in range(wl.k):
            e = ids[t, j]
            g = w13[e, :wl.I] @ xq
            u = w13[e, wl.I:] @ xq
            a = _torch_fake_quant64((_silu(g) * u).astype(np.float32))
            acc += w[t, j] * (w2[e] @ a)
        # a 1-ulp difference in an fp32 activation can move its code; allow that
        np.testing.assert_allclose(out[t], acc, rtol=1e-6, atol=1e-6 * np.abs(acc).max())


def test_token_subset_matches_full(oracle):
    wl = W.custom(T=20, H=64, I=32, E=8, k=2, dtype=W.BF16, seed=10)
    inp = W.make_inputs(wl)
    full, ids_full, _ = _run(oracle, wl, inp)
    sub, ids_sub, _ = _run(oracle, wl, inp, tokens=np.array([19, 0, 7], np.int32))
    np.testing.assert_array_equal(sub, full[[19, 0, 7]])
    np.testing.assert_array_equal(ids_sub, ids_full[[19, 0, 7]])


def test_expert_parallel_slices(oracle):
    # one expert per rank: rank r's partial output is exactly the dense-gating
    # term of expert r (numpy); and the ranks' partial outputs add up to the
    # whole layer
    wl = W.custom(T=7, H=64, I=32, E=4, k=2, dtype=W.BF16, seed=12)
    inp = W.make_inputs(wl)
    full, ids, w = _run(oracle, wl, inp)
    x = _f64(inp["x"])
    total = np.zeros_like(full)
    for r in range(wl.E):
        part, ids_r, w_r = oracle.moe_forward(
            T=wl.T, H=wl.H, I=wl.I, E=wl.E, k=wl.k, dtype=wl.dtype, scoring=wl.scoring,
            renorm=wl.renorm, x=W.storage_numpy(inp["x"]), logits=W.storage_numpy(inp["logits"]),
            w13=W.storage_numpy(inp["w13"][r:r + 1]), w2=W.storage_numpy(inp["w2"][r:r + 1]),
            ep_size=wl.E, ep_rank=r)
        np.testing.assert_array_equal(ids_r, ids)
        gate = np.where(ids == r, w, 0.0).sum(1)  # routing weight of expert r per token
        ref = gate[:, None] * _mlp(x, _f64(inp["w13"][r]), _f64(inp["w2"][r]), wl.I)
        np.testing.assert_allclose(part, ref, rtol=1e-9, atol=1e-12)
        total += part
    np.testing.assert_allclose(total, full, rtol=1e-9, atol=1e-12)
