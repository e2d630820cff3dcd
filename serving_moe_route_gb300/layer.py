"""Torch-facing wrapper over the C ABI.  PyTorch provides device memory and
the stream; all of the layer's arithmetic runs in ``libmoe_route.so``."""
from __future__ import annotations

import torch

from . import _binding as B

F32, BF16, FP8 = B.MOE_DTYPE_F32, B.MOE_DTYPE_BF16, B.MOE_DTYPE_FP8_BLOCK128
SOFTMAX, SIGMOID = B.MOE_SCORING_SOFTMAX, B.MOE_SCORING_SIGMOID

_ACT_DTYPE = {F32: torch.float32, BF16: torch.bfloat16, FP8: torch.bfloat16}
_W_DTYPE = {F32: torch.float32, BF16: torch.bfloat16, FP8: torch.float8_e4m3fn}


def _stream(stream):
    return (stream if stream is not None else torch.cuda.current_stream()).cuda_stream


def _p(t):
    return 0 if t is None else t.data_ptr()


def _need(t, dtype, shape, name):
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


class MoELayer:
    """One fused MoE layer: weights resident on the GPU, a plan and a
    workspace per batch size, ``forward(x, logits) -> out``."""

    def __init__(self, w13, w2, *, k, dtype, scoring=SOFTMAX, renorm=True, s13=None, s2=None,
                 force_est=0, ep_size=1, ep_rank=0, n_group=1, topk_group=1, gemm_pair=None,
                 gemm_tm=None):
        """w13/w2 (and s13/s2) hold this expert-parallel rank's experts: all
        of them when ep_size == 1, else E/ep_size of E = w13.shape[0] * ep_size;
        forward() then returns this rank's partial sum.  gemm_pair=None keeps
        the plan's choice of CTA-pair GEMMs (BF16/F32), gemm_tm=None its
        choice of token-major GEMMs (FP8); 0 or 1 overrides either."""
        E, I2, H = w13.shape  # experts held by this rank
        I = I2 // 2
        _need(w13, _W_DTYPE[dtype], (E, 2 * I, H), "w13")
        _need(w2, _W_DTYPE[dtype], (E, H, I), "w2")
        if dtype == FP8:
            _need(s13, torch.float32, (E, 2 * I // 128, H // 128), "s13")
            _need(s2, torch.float32, (E, H // 128, I // 128), "s2")
        elif s13 is not None or s2 is not None:
            raise ValueError("block scales are only used by the FP8 layer")
        self.e_local, self.E, self.H, self.I, self.k = E, E * ep_size, H, I, k
        self.ep_size, self.ep_rank = ep_size, ep_rank
        self.n_group, self.topk_group = n_group, topk_group
        self.gemm_pair = gemm_pair
        self.gemm_tm = gemm_tm
        self.dtype, self.scoring, self.renorm, self.force_est = dtype, scoring, renorm, force_est
        self.w13, self.w2, self.s13, self.s2 = w13, w2, s13, s2
        self.device = w13.device
        self._plans = {}
        self._ws = None

    # ------------------------------------------------------------ planning
    def plan(self, T: int) -> B.MoePlan:
        p = self._plans.get(T)
        if p is None:
            p = B.moe_plan_ep(T, self.H, self.I, self.E, self.k, self.dtype, self.scoring,
                              self.renorm, self.force_est, self.ep_size, self.ep_rank)
            if self.n_group > 1:
                B.moe_plan_set_groups(p, self.n_group, self.topk_group)
            if self.gemm_pair is not None:
                p.gemm_pair = int(bool(self.gemm_pair))
            if self.gemm_tm is not None:
                p.gemm_tm = int(bool(self.gemm_tm))
            self._plans[T] = p
        return p

    def workspace(self, T: int) -> torch.Tensor:
        need = int(self.plan(T).workspace_bytes)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.empty(max(need, 256), dtype=torch.uint8, device=self.device)
        return self._ws

    # ------------------------------------------------------------ forward
    def forward(self, x, logits, out=None, stream=None):
        T = x.shape[0]
        _need(x, _ACT_DTYPE[self.dtype], (T, self.H), "x")
        _need(logits, _ACT_DTYPE[self.dtype], (T, self.E), "logits")
        if out is None:
            out = torch.empty(T, self.H, dtype=_ACT_DTYPE[self.dtype], device=self.device)
        _need(out, _ACT_DTYPE[self.dtype], (T, self.H), "out")
        p = self.plan(T)
        ws = self.workspace(T)
        rc = B.moe_forward(p, _p(x), _p(logits), _p(self.w13), _p(self.s13), _p(self.w2),
                           _p(self.s2), _p(out), _p(ws), ws.numel(), _stream(stream))
        B._check(rc, "moe_forward")
        return out

    __call__ = forward

    def forward_with_ids(self, x, ids, topk_w, out=None, stream=None):
        T = x.shape[0]
        _need(x, _ACT_DTYPE[self.dtype], (T, self.H), "x")
        _need(ids, torch.int32, (T, self.k), "ids")
        _need(topk_w, torch.float32, (T, self.k), "topk_w")
        if out is None:
            out = torch.empty(T, self.H, dtype=_ACT_DTYPE[self.dtype], device=self.device)
        p = self.plan(T)
        ws = self.workspace(T)
        rc = B.moe_forward_with_ids(p, _p(x), _p(ids), _p(topk_w), _p(self.w13), _p(self.s13),
                                    _p(self.w2), _p(self.s2), _p(out), _p(ws), ws.numel(),
                                    _stream(stream))
        B._check(rc, "moe_forward_with_ids")
        return out

    def check(self, T: int, stream=None):
        """Synchronise and return (rc, device error bits)."""
        return B.moe_check(self.plan(T), _p(self.workspace(T)), _stream(stream))

    # ------------------------------------------------------------ inspection
    def intermediates(self, T: int) -> dict:
        """Views into the workspace of the last forward with batch T."""
        p = self.plan(T)
        ws = self.workspace(T)
        R = T * self.k

        def view(off, n, dt):
            esz = torch.tensor([], dtype=dt).element_size()
            return ws[off:off + n * esz].view(dt)

        out = {
            "ids": view(p.off_ids, R, torch.int32).view(T, self.k),
            "w": view(p.off_w, R, torch.float32).view(T, self.k),
            "counts": view(p.off_counts, self.e_local, torch.int32),
            "offsets": view(p.off_offsets, self.e_local + 1, torch.int32),
            "src": view(p.off_src, R, torch.int32),
            "pos": view(p.off_pos, R, torch.int32),
            "tiles": view(p.off_tiles, p.max_tiles * 4, torch.int32).view(p.max_tiles, 4),
            "ntiles": view(p.off_ntiles, 1, torch.int32),
            "tiles2": view(p.off_tiles2, p.max_tiles * 4, torch.int32).view(p.max_tiles, 4),
            "ntiles2": view(p.off_ntiles2, 1, torch.int32),
            # the GEMM kernel family a plan that chooses it on the device ran
            # (1 one CTA per tile, 2 CTA pairs; left as it was otherwise)
            "family": view(p.off_err + 8, 1, torch.int32),
        }
        if self.dtype == FP8:
            out["xq"] = view(p.off_xq, R * self.H, torch.uint8).view(R, self.H)
            out["xs"] = view(p.off_xs, R * (self.H // 128), torch.float32).view(R, self.H // 128)
        return out


def route_topk(logits, k, scoring=SOFTMAX, renorm=True, stream=None, n_group=1, topk_group=1):
    """Step a-1 alone: logits [T, E] (f32 or bf16) -> (ids int32 [T,k], w f32 [T,k]);
    n_group > 1 selects group-limited routing."""
    if logits.device.type != "cuda" or not logits.is_contiguous() or logits.dim() != 2:
        raise ValueError("logits must be a contiguous 2-D CUDA tensor")
    if logits.dtype == torch.float32:
        ldt = B.MOE_LOGITS_F32
    elif logits.dtype == torch.bfloat16:
        ldt = B.MOE_LOGITS_BF16
    else:
        raise ValueError("logits must be float32 or bfloat16")
    T, E = logits.shape
    ids = torch.empty(T, k, dtype=torch.int32, device=logits.device)
    w = torch.empty(T, k, dtype=torch.float32, device=logits.device)
    rc = B.moe_route_grouped_topk(_p(logits), ldt, T, E, k, n_group, topk_group, scoring,
                                  renorm, _p(ids), _p(w), _stream(stream))
    B._check(rc, "moe_route_grouped_topk")
    return ids, w
