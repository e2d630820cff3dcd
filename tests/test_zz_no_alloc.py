"""The allocation-free entry point, moe_forward_noalloc, against moe_forward.

Some callers cannot allocate device memory: code that runs inside an
allocator hook or a memory pool, and hosts that forbid device allocation
after start-up.  moe_forward_noalloc runs the same layer on a workspace that
lives in the library's own device image, and moe_check_noalloc reads that
workspace's error word.  The two entry points launch the same deterministic
kernels, so their outputs must agree bit for bit.  This file is collected
last on purpose: a run that stops at its first failure has run every other
test by then."""
import numpy as np
import pytest
import torch

import parity_util as PU
from serving_moe_route_gb300 import _binding as B
from serving_moe_route_gb300 import workloads as W

CASES = [
    W.custom("noalloc_bf16", T=96, H=512, I=256, E=32, k=4, dtype=W.BF16, seed=51,
             logits="nan_rows"),
    W.custom("noalloc_fp8", T=40, H=256, I=256, E=16, k=4, dtype=W.FP8, seed=52),
]


def _lib_or_skip():
    try:
        return B.lib()
    except (OSError, RuntimeError) as exc:  # no built library or no CUDA runtime here
        pytest.skip(f"library not loadable: {exc}")


def test_noalloc_rejects_oversized_plan_before_launch():
    # 4096 tokens x top-8 at H=2048 needs far more than the 16 MiB built in;
    # rejected on the host before anything touches a device
    _lib_or_skip()
    p = B.moe_plan(4096, 2048, 768, 128, 8, B.MOE_DTYPE_BF16)
    assert p.workspace_bytes > 16 << 20
    fake = 1 << 20
    rc = B.moe_forward_noalloc(p, fake, fake, fake, 0, fake, 0, fake, 0)
    assert rc == B.MOE_ERR_WORKSPACE
    rc, _ = B.moe_check_noalloc(p, 0)
    assert rc == B.MOE_ERR_WORKSPACE


@pytest.mark.gpu
@pytest.mark.parametrize("wl", CASES, ids=[w.name for w in CASES])
def test_noalloc_matches_moe_forward_twice(wl):
    inp = W.make_inputs(wl)
    layer = PU.make_layer(wl, inp)
    dev = layer.device
    x = inp["x"].to(dev)
    lg = inp["logits"].to(dev)
    ref = layer.forward(x, lg)
    rc, bits = layer.check(wl.T)
    assert rc == 0, bits
    ref = ref.cpu()
    p = layer.plan(wl.T)
    assert p.workspace_bytes <= 16 << 20
    stream = torch.cuda.current_stream(dev).cuda_stream
    for _ in range(2):  # two calls in a row share the built-in workspace
        out = torch.full((wl.T, wl.H), float("nan"), dtype=x.dtype, device=dev)
        rc = B.moe_forward_noalloc(
            p, x.data_ptr(), lg.data_ptr(), layer.w13.data_ptr(),
            0 if layer.s13 is None else layer.s13.data_ptr(), layer.w2.data_ptr(),
            0 if layer.s2 is None else layer.s2.data_ptr(), out.data_ptr(), stream)
        assert rc == B.MOE_OK, B.strerror(rc)
        rc, bits = B.moe_check_noalloc(p, stream)
        assert rc == B.MOE_OK and bits == 0, (rc, bits)
        got = out.cpu()
        # same kernels on the same inputs: identical bits, no tolerance
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
        assert np.isfinite(got.float().numpy()).all()
