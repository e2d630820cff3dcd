"""CPU checks of the C ABI: the library builds, loads and exports every
symbol the header declares; the header compiles as C and its struct layout
matches the binding; moe_plan's host arithmetic (estimate, tile table,
worst-case workspace before the estimate, argument errors).  No compute
call is made -- there is no GPU here."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_route.h")


@pytest.fixture(scope="module")
def B():
    from serving_moe_route_gb300 import _binding, _build

    _build.build()
    _binding.lib()
    return _binding


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(moe_\w+)\s*\(", text, re.M)))


def test_exports_every_declared_symbol(B):
    names = _declared()
    assert set(B.EXPORTED) <= set(names)
    out = subprocess.run(["nm", "-D", "--defined-only", B.lib_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (moe_\w+)$", out, re.M))
    for n in names:
        assert n in exported, n
        assert hasattr(B.lib(), n)


def test_header_is_c_and_layout_matches(B, tmp_path):
    src = tmp_path / "layout.c"
    src.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "moe_route.h"\n'
        "int main(void){printf(\"%zu %zu %zu %zu\\n\", sizeof(moe_plan_t),"
        " offsetof(moe_plan_t, workspace_bytes), offsetof(moe_plan_t, off_y),"
        " offsetof(moe_plan_t, tile_n)); return 0;}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.dirname(HEADER),
                    str(src), "-o", str(exe)], check=True)
    vals = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True,
                                           check=True).stdout.split()]
    P = B.MoePlan
    assert vals == [ctypes.sizeof(P), P.workspace_bytes.offset, P.off_y.offset,
                    P.tile_n.offset]


def test_plan_estimate_worked_example(B):
    # 288 tokens x top-6 over 400 experts: 4.32 rows per expert -> 5
    p = B.moe_plan(288, 2048, 768, 400, 6, B.MOE_DTYPE_BF16)
    assert p.est == 5 and p.tile_n == 16
    old = B.moe_plan(288, 2048, 768, 400, 6, B.MOE_DTYPE_BF16, force_est=288)
    assert old.est == 288 and old.tile_n == 128
    # capacity is fixed before the estimate: identical workspace either way
    assert old.workspace_bytes == p.workspace_bytes
    assert old.max_tiles == p.max_tiles


@pytest.mark.parametrize("T,est,tile", [(1, 1, 16), (2, 1, 16), (4, 1, 16), (16, 1, 16),
                                        (64, 4, 16), (128, 8, 16), (256, 16, 16),
                                        (1024, 64, 64), (4096, 256, 64), (512, 32, 32)])
def test_plan_tile_table(B, T, est, tile):
    p = B.moe_plan(T, 2048, 768, 128, 8, B.MOE_DTYPE_FP8_BLOCK128)
    assert p.est == est and p.tile_n == tile
    pb = B.moe_plan(T, 2048, 768, 128, 8, B.MOE_DTYPE_BF16)  # bf16: no 64 cap
    assert pb.tile_n == (128 if est > 64 else tile)
    assert p.g1_mblocks == 6 and p.g2_mblocks == 16
    assert p.max_tiles >= -(-T * 8 // 16) + min(128, T * 8)


def test_plan_workspace_layout(B):
    p = B.moe_plan(128, 2048, 768, 128, 8, B.MOE_DTYPE_BF16)
    offs = [p.off_err, p.off_ids, p.off_w, p.off_chunk_counts, p.off_lrank, p.off_counts,
            p.off_offsets, p.off_chunk_base, p.off_src, p.off_pos, p.off_tiles, p.off_ntiles,
            p.off_xq, p.off_xs, p.off_act, p.off_as, p.off_y]
    assert all(o % 256 == 0 for o in offs)
    assert offs == sorted(offs)
    R = 128 * 8
    assert p.off_act - p.off_xq >= R * 2048 * 2
    assert p.workspace_bytes - p.off_y >= 128 * 2048 * 4
    assert "est=8" in p.describe() and "tile_n=16" in p.describe()


@pytest.mark.parametrize("args,code", [
    ((16, 128, 64, 8, 0, 1), -1),      # k = 0
    ((16, 128, 64, 8, 9, 1), -1),      # k > E
    ((16, 128, 64, 2000, 8, 1), -1),   # E > 1024
    ((-1, 128, 64, 8, 2, 1), -1),      # T < 0
    ((16, 128, 64, 8, 2, 7), -1),      # bad dtype
    ((16, 96, 64, 8, 2, 1), -2),       # H not a multiple of 64 for bf16
    ((16, 128, 64, 8, 2, 2), -2),      # I not a multiple of 128 for fp8
    ((16, 100, 64, 8, 2, 0), -2),      # H not a multiple of 32 for f32
])
def test_plan_rejects(B, args, code):
    p = B.MoePlan()
    rc = B.lib().moe_plan(*args, 0, 1, 0, ctypes.byref(p))
    assert rc == code
    assert B.strerror(rc)


def test_forward_validates_before_launch(B):
    p = B.moe_plan(16, 128, 64, 8, 2, B.MOE_DTYPE_BF16)
    # null pointers and short workspace are rejected on the host: no launch
    assert B.moe_forward(p, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0) == B.MOE_ERR_INVALID_ARG
    fake = 1 << 20  # never dereferenced: validation fails first
    assert B.moe_forward(p, fake, fake, fake, 0, fake, 0, fake, fake, 16, 0) == \
        B.MOE_ERR_WORKSPACE
    assert B.moe_forward(p, fake + 4, fake, fake, 0, fake, 0, fake, fake,
                         p.workspace_bytes, 0) == B.MOE_ERR_INVALID_ARG
    assert B.moe_forward(p, fake, fake, fake, fake, fake, 0, fake, fake, p.workspace_bytes,
                         0) == B.MOE_ERR_INVALID_ARG  # scales given to a bf16 layer
    assert B.moe_route_topk(fake, 1, 4, 8, 9, 0, 1, fake, fake, 0) == B.MOE_ERR_INVALID_ARG


def test_expert_parallel_plan(B):
    with pytest.raises(B.MoeError):
        B.moe_plan_ep(16, 256, 128, 10, 2, B.MOE_DTYPE_BF16, ep_size=4)   # 10 % 4 != 0
    with pytest.raises(B.MoeError):
        B.moe_plan_ep(16, 256, 128, 16, 2, B.MOE_DTYPE_BF16, ep_size=4, ep_rank=4)
    # the H20 article's setting: 400 slots on 8 ranks -> 50 local experts; the
    # estimate still divides by all 400 slots
    p = B.moe_plan_ep(288, 2048, 768, 400, 6, B.MOE_DTYPE_BF16, ep_size=8, ep_rank=3)
    assert (p.ep_size, p.ep_rank, p.e_local, p.est) == (8, 3, 50, 5)
    full = B.moe_plan(288, 2048, 768, 400, 6, B.MOE_DTYPE_BF16)
    assert p.workspace_bytes < full.workspace_bytes


def test_group_limited_plan(B):
    p = B.moe_plan(128, 2048, 768, 128, 8, B.MOE_DTYPE_BF16)
    assert (p.n_group, p.topk_group) == (1, 1)
    for ng, tg in [(0, 1), (3, 1), (8, 0), (8, 9), (64, 4), (8, 1)]:
        # 0 groups; 128 % 3; no kept group; more kept than groups; >32 groups;
        # one kept group of 16 holds k = 8 experts, so (8, 1) is valid
        if (ng, tg) == (8, 1):
            B.moe_plan_set_groups(p, ng, tg)
            continue
        with pytest.raises(B.MoeError):
            B.moe_plan_set_groups(p, ng, tg)
    q = B.moe_plan(16, 256, 128, 16, 8, B.MOE_DTYPE_BF16)
    with pytest.raises(B.MoeError):   # 1 kept group of 2 experts cannot hold k = 8
        B.moe_plan_set_groups(q, 8, 1)
    B.moe_plan_set_groups(q, 8, 4)
    assert (q.n_group, q.topk_group) == (8, 4)
    fake = 256
    assert B.moe_route_grouped_topk(fake, 0, 4, 16, 8, 8, 1, 0, 1, fake, fake, 0) == \
        B.MOE_ERR_INVALID_ARG
    assert B.moe_route_grouped_topk(None, 0, 0, 16, 8, 8, 4, 0, 1, None, None, 0) == B.MOE_OK


def test_plan_gemm_pair_choice(B):
    # CTA-pair GEMMs for BF16/F32 plans whose experts average more than 32 rows
    assert B.moe_plan(4096, 2048, 768, 128, 8, B.MOE_DTYPE_BF16).gemm_pair == 1   # est 256
    assert B.moe_plan(512, 2048, 768, 128, 8, B.MOE_DTYPE_BF16).gemm_pair == 0    # est 32
    assert B.moe_plan(528, 2048, 768, 128, 8, B.MOE_DTYPE_BF16).gemm_pair == 1    # est 33
    assert B.moe_plan(4096, 2048, 768, 128, 8, B.MOE_DTYPE_FP8_BLOCK128).gemm_pair == 0
    assert B.moe_plan(300, 160, 96, 8, 2, B.MOE_DTYPE_F32).gemm_pair == 1
    assert B.moe_plan(288, 2048, 768, 400, 6, B.MOE_DTYPE_BF16, force_est=288).gemm_pair == 1


def test_plan_gemm_tm_choice(B):
    # token-major FP8 GEMMs once experts average 32 rows or more
    fp8 = B.MOE_DTYPE_FP8_BLOCK128
    assert B.moe_plan(512, 2048, 768, 128, 8, fp8).gemm_tm == 1    # est 32
    assert B.moe_plan(4096, 2048, 768, 128, 8, fp8).gemm_tm == 1   # est 256
    assert B.moe_plan(496, 2048, 768, 128, 8, fp8).gemm_tm == 0    # est 31
    assert B.moe_plan(256, 2048, 768, 128, 8, fp8).gemm_tm == 0    # est 16
    assert B.moe_plan(1, 2048, 768, 128, 8, fp8).gemm_tm == 0
    assert B.moe_plan(4096, 2048, 768, 128, 8, B.MOE_DTYPE_BF16).gemm_tm == 0
    assert "token-major" in B.moe_plan(4096, 2048, 768, 128, 8, fp8).describe()
    assert "cta-pair" in B.moe_plan(4096, 2048, 768, 128, 8, B.MOE_DTYPE_BF16).describe()


def test_plan_gemm_dyn_choice(B):
    # the device picks the GEMM kernel family for one-CTA-per-tile BF16/F32
    # plans whose batch can give one expert a whole 256-row tile
    bf16, f32, fp8 = B.MOE_DTYPE_BF16, B.MOE_DTYPE_F32, B.MOE_DTYPE_FP8_BLOCK128
    assert B.moe_plan(288, 2048, 768, 400, 6, bf16).gemm_dyn == 1     # est 5
    assert B.moe_plan(256, 256, 256, 128, 8, f32).gemm_dyn == 1       # est 16
    assert B.moe_plan(255, 2048, 768, 400, 6, bf16).gemm_dyn == 0     # T < 256
    assert B.moe_plan(128, 2048, 768, 128, 8, bf16).gemm_dyn == 0     # decode
    p = B.moe_plan(4096, 2048, 768, 128, 8, bf16)                     # est 256: CTA pairs
    assert p.gemm_pair == 1 and p.gemm_dyn == 0
    assert B.moe_plan(288, 2048, 768, 400, 6, fp8).gemm_dyn == 0
    assert "per call" in B.moe_plan(288, 2048, 768, 400, 6, bf16).describe()
    assert "per call" not in B.moe_plan(128, 2048, 768, 128, 8, bf16).describe()
