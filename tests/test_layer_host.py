"""Host-side behaviour of the Python layer (no GPU): the product path has no
CPU fallback -- it refuses CPU tensors and a missing CUDA library loudly."""
import pytest
import torch

from serving_moe_route_gb300 import _binding as B
from serving_moe_route_gb300 import MoELayer, route_topk


def test_layer_refuses_cpu_tensors():
    w13 = torch.zeros(4, 256, 128, dtype=torch.bfloat16)
    w2 = torch.zeros(4, 128, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        MoELayer(w13, w2, k=2, dtype=B.MOE_DTYPE_BF16)


def test_route_topk_refuses_cpu_tensors():
    with pytest.raises(ValueError, match="CUDA"):
        route_topk(torch.zeros(4, 8), 2)


def test_missing_library_raises(monkeypatch, tmp_path):
    monkeypatch.setattr(B, "_lib", None)
    monkeypatch.setattr(B, "lib_path", lambda: str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError, match="missing"):
        B.lib()

