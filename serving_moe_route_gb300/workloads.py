"""Seeded synthetic inputs for the fused MoE layer forward.

This module draws inputs and nothing else: it holds none of the layer's
arithmetic (no routing, no permutation, no expert math, no activation
quantisation).  Both the CUDA path and the CPU oracle consume exactly the
tensors made here, byte for byte.

Workloads follow the shapes the pages measure on:
  * H20 article (288 tokens, top-6, 400 expert slots, uniform routing; the
    concentrated case is reported separately),
  * PR #39593 micro-benchmark (128 tokens x 128 experts, top-8, bf16,
    10% all-NaN rows),
  * Lab notes #6 (E=128, N=768, FP8 [128,128] blocks, batch 1 ... 4096).
Hidden size 2048 and intermediate 768 are the Qwen3-30B-A3B MoE shapes
those pages run.

All tensors are CPU torch tensors: fp32, bf16 or float8_e4m3fn.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

F32, BF16, FP8 = 0, 1, 2
SOFTMAX, SIGMOID = 0, 1
DTYPE_NAMES = {F32: "f32", BF16: "bf16", FP8: "fp8_block128"}

FP8_SWEEP = (1, 2, 4, 16, 64, 128, 256, 1024, 4096)


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    I: int
    E: int
    k: int
    dtype: int
    scoring: int = SOFTMAX
    renorm: bool = True
    logits: str = "normal"  # normal | router | nan_rows | concentrated | zipf
    seed: int = 0
    force_est: int = 0
    ep_size: int = 1  # expert-parallel ranks; this workload is rank ep_rank's slice
    ep_rank: int = 0
    n_group: int = 1  # group-limited routing (1 = off)
    topk_group: int = 1
    gemm_pair: object = None  # None: the plan's choice; 0 / 1: forced
    gemm_tm: object = None  # FP8 token-major GEMMs: None the plan's choice; 0 / 1 forced
    extra: dict = field(default_factory=dict, compare=False, hash=False)


def _wl(name, T, H, I, E, k, dtype, seed, **kw):
    return Workload(name=name, T=T, H=H, I=I, E=E, k=k, dtype=dtype, seed=seed, **kw)


def workloads() -> dict:
    """Every named workload, keyed by name.  Seeds are 1000 + group index."""
    w = {}
    w["tiny_f32"] = _wl("tiny_f32", 16, 128, 64, 8, 2, F32, 1000, logits="router")
    w["decode_bf16"] = _wl("decode_bf16", 128, 2048, 768, 128, 8, BF16, 1001, logits="nan_rows")
    w["sparse_uniform_bf16"] = _wl("sparse_uniform_bf16", 288, 2048, 768, 400, 6, BF16, 1002)
    w["sparse_concentrated_bf16"] = _wl("sparse_concentrated_bf16", 288, 2048, 768, 400, 6, BF16,
                                        1002, logits="concentrated")
    w["sparse_uniform_bf16_old_est"] = _wl("sparse_uniform_bf16_old_est", 288, 2048, 768, 400, 6,
                                           BF16, 1002, force_est=288)
    w["sparse_concentrated_bf16_old_est"] = _wl("sparse_concentrated_bf16_old_est", 288, 2048, 768,
                                                400, 6, BF16, 1002, logits="concentrated",
                                                force_est=288)
    for T in FP8_SWEEP:
        w[f"fp8_T{T}"] = _wl(f"fp8_T{T}", T, 2048, 768, 128, 8, FP8, 1003)
    # the FP8 batch sweep's decode sizes with the token-major GEMMs forced
    # (the plan picks them from 32 rows per expert on)
    for T in (1, 2, 4, 16, 64, 128, 256):
        w[f"fp8_T{T}_tm"] = _wl(f"fp8_T{T}_tm", T, 2048, 768, 128, 8, FP8, 1003, gemm_tm=1)
    # the H20 article's setting: 400 expert slots over 8 GPUs, local MoE of one rank
    w["sparse_uniform_bf16_ep8"] = _wl("sparse_uniform_bf16_ep8", 288, 2048, 768, 400, 6, BF16,
                                       1002, ep_size=8)
    w["sparse_uniform_bf16_ep8_old_est"] = _wl("sparse_uniform_bf16_ep8_old_est", 288, 2048, 768,
                                               400, 6, BF16, 1002, ep_size=8, force_est=288)
    # group-limited routing on the decode shape: 8 groups of 16, 4 kept
    w["decode_grouped_bf16"] = _wl("decode_grouped_bf16", 128, 2048, 768, 128, 8, BF16, 1001,
                                   logits="nan_rows", n_group=8, topk_group=4)
    w["skewed_prefill_bf16"] = _wl("skewed_prefill_bf16", 4096, 2048, 768, 128, 8, BF16, 1004,
                                   logits="zipf")
    w["skewed_prefill_sigmoid_bf16"] = _wl("skewed_prefill_sigmoid_bf16", 4096, 2048, 768, 128, 8,
                                           BF16, 1004, logits="zipf", scoring=SIGMOID)
    return w


def _gen(seed: int, salt: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed * 1_000_003 + salt)
    return g


def _normal(shape, std, g, dtype=torch.float32):
    return (torch.randn(*shape, generator=g, dtype=torch.float32) * std).to(dtype)


def make_logits(wl: Workload, x: torch.Tensor | None = None) -> torch.Tensor:
    """Router logits [T, E]: fp32 for the fp32 workload, bf16 otherwise."""
    T, E = wl.T, wl.E
    g = _gen(wl.seed, 1)
    out_dtype = torch.float32 if wl.dtype == F32 else torch.bfloat16
    if wl.logits == "router":
        # gating logits from a random router matrix: the router GEMM sits
        # outside the layer boundary, so it is part of input synthesis
        wr = _normal((E, wl.H), 0.02, g)
        return (x.float() @ wr.t()).to(out_dtype)
    z = torch.randn(T, E, generator=g, dtype=torch.float32)
    if wl.logits == "nan_rows":
        # 10% of rows entirely NaN (padding rows under DP + CUDA graphs)
        n_nan = max(1, round(0.1 * T))
        rows = torch.randperm(T, generator=g)[:n_nan]
        z[rows] = float("nan")
    elif wl.logits == "concentrated":
        # bias b on a seeded set S of 6 experts so that the expected softmax
        # mass on S is 90%: 6 e^b / (6 e^b + (E - 6)) = 0.9
        s = torch.randperm(E, generator=g)[:6]
        b = math.log(0.9 * (E - 6) / (6 * 0.1))
        z[:, s] += b
    elif wl.logits == "zipf":
        # Zipf(1.2) expert popularity: logit offset ln p over ranks 1..E,
        # ranks assigned to experts by a seeded permutation
        ranks = torch.arange(1, E + 1, dtype=torch.float64)
        p = ranks.pow(-1.2)
        p = p / p.sum()
        perm = torch.randperm(E, generator=g)
        off = torch.empty(E, dtype=torch.float64)
        off[perm] = p.log()
        z = z + off.to(torch.float32)
    elif wl.logits != "normal":
        raise ValueError(f"unknown logits kind {wl.logits!r}")
    return z.to(out_dtype)


def make_activations(wl: Workload) -> dict:
    """x [T,H] (fp32 for the fp32 workload, else bf16) and logits [T,E]."""
    gx = _gen(wl.seed, 0)
    if wl.dtype == F32:
        x = _normal((wl.T, wl.H), 0.02, gx)
    else:
        x = _normal((wl.T, wl.H), 1.0, gx, torch.bfloat16)
    return {"x": x, "logits": make_logits(wl, x)}


def make_weights(wl: Workload) -> dict:
    """w13 [E,2I,H] and w2 [E,H,I]; for the FP8 workloads float8_e4m3fn
    codes with fp32 block scales s13 [E,2I/128,H/128] and s2 [E,H/128,I/128].
    Depends only on (H, I, E, dtype, seed), not on T.  With ep_size > 1 only
    rank ep_rank's E/ep_size experts (the same tensors as in the full set)."""
    if wl.ep_size > 1:
        full = make_weights(Workload(name=wl.name, T=wl.T, H=wl.H, I=wl.I, E=wl.E, k=wl.k,
                                     dtype=wl.dtype, seed=wl.seed)) if wl.ep_rank else None
        el = wl.E // wl.ep_size
        if full is None:  # rank 0: the first experts of the stream, no need for the rest
            part = make_weights(Workload(name=wl.name, T=wl.T, H=wl.H, I=wl.I, E=el, k=wl.k,
                                         dtype=wl.dtype, seed=wl.seed))
            if wl.dtype == FP8:  # block scales are drawn after all codes: take them from E
                full = make_weights(Workload(name=wl.name, T=wl.T, H=wl.H, I=wl.I, E=wl.E,
                                             k=wl.k, dtype=wl.dtype, seed=wl.seed))
            else:
                return part
        sl = slice(wl.ep_rank * el, (wl.ep_rank + 1) * el)
        return {k2: (None if v is None else v[sl].contiguous()) for k2, v in full.items()}
    H, I, E = wl.H, wl.I, wl.E
    gw = _gen(wl.seed, 2)
    if wl.dtype in (F32, BF16):
        dt = torch.float32 if wl.dtype == F32 else torch.bfloat16
        w13 = torch.empty(E, 2 * I, H, dtype=dt)
        w2 = torch.empty(E, H, I, dtype=dt)
        for e in range(E):  # per expert, to bound the fp32 temporaries
            w13[e] = _normal((2 * I, H), 0.02, gw, dt)
            w2[e] = _normal((H, I), 0.02, gw, dt)
        return {"w13": w13, "w2": w2, "s13": None, "s2": None}
    if H % 128 or I % 128:
        raise ValueError("FP8 block-scaled weights need H and I multiples of 128")
    # codes from a clipped normal in code space and one positive fp32 scale
    # per [128,128] block, so that code * scale ~ N(0, 0.02)
    sigma_code = 112.0
    w13 = torch.empty(E, 2 * I, H, dtype=torch.float8_e4m3fn)
    w2 = torch.empty(E, H, I, dtype=torch.float8_e4m3fn)
    for e in range(E):
        w13[e] = (torch.randn(2 * I, H, generator=gw) * sigma_code).clamp_(-448, 448).to(
            torch.float8_e4m3fn)
        w2[e] = (torch.randn(H, I, generator=gw) * sigma_code).clamp_(-448, 448).to(
            torch.float8_e4m3fn)
    base = 0.02 / sigma_code
    s13 = base * (0.75 + 0.5 * torch.rand(E, 2 * I // 128, H // 128, generator=gw))
    s2 = base * (0.75 + 0.5 * torch.rand(E, H // 128, I // 128, generator=gw))
    return {"w13": w13, "w2": w2, "s13": s13.float().contiguous(), "s2": s2.float().contiguous()}


def make_inputs(wl: Workload) -> dict:
    """All inputs of one workload as CPU tensors: make_activations and
    make_weights together."""
    out = make_activations(wl)
    out.update(make_weights(wl))
    return out


def custom(name="custom", *, T, H, I, E, k, dtype, scoring=SOFTMAX, renorm=True, logits="normal",
           seed=7, force_est=0, ep_size=1, ep_rank=0, n_group=1, topk_group=1,
           gemm_pair=None, gemm_tm=None) -> Workload:
    """An ad-hoc workload (edge cases in tests)."""
    return Workload(name=name, T=T, H=H, I=I, E=E, k=k, dtype=dtype, scoring=scoring,
                    renorm=renorm, logits=logits, seed=seed, force_est=force_est,
                    ep_size=ep_size, ep_rank=ep_rank, n_group=n_group, topk_group=topk_group,
                    gemm_pair=gemm_pair, gemm_tm=gemm_tm)


# ------------------------------------------------------------ numpy views
def storage_numpy(t: torch.Tensor | None):
    """A tensor's bytes as numpy in storage form: fp32 values, bf16 bit
    patterns (uint16) or e4m3 codes (uint8).  No conversion of values."""
    import numpy as np

    if t is None:
        return None
    t = t.contiguous()
    if t.dtype == torch.float32:
        return t.numpy()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    if t.dtype == torch.int32:
        return t.numpy()
    raise TypeError(f"unsupported dtype {t.dtype}")
