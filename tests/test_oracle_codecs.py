"""Pins for the oracle's number codecs (bf16, OCP e4m3) and its FP8 group
quantisation, against torch's own dtype conversions and the format's
definition.  CPU only."""
import math

import numpy as np
import pytest
import torch


def test_bf16_rne_hand_values(oracle):
    # 1.0 exactly; a tie that rounds down to even; a tie that rounds up to even
    assert oracle.f32_to_bf16(1.0) == 0x3F80
    tie_down = np.array([0x3F808000], np.uint32).view(np.float32)[0]
    tie_up = np.array([0x3F818000], np.uint32).view(np.float32)[0]
    assert oracle.f32_to_bf16(float(tie_down)) == 0x3F80
    assert oracle.f32_to_bf16(float(tie_up)) == 0x3F82
    assert oracle.f32_to_bf16(-2.0) == 0xC000
    assert oracle.bf16_to_f32(0x3F80) == 1.0


def test_bf16_matches_torch(oracle):
    g = torch.Generator().manual_seed(3)
    v = torch.randn(4000, generator=g) * torch.logspace(-20, 20, 4000)
    bits = v.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    for val, b in zip(v.tolist(), bits.tolist()):
        assert oracle.f32_to_bf16(val) == b
    back = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).float().tolist()
    for b, r in zip(bits.tolist(), back):
        assert oracle.bf16_to_f32(b) == r


def test_e4m3_decode_all_codes(oracle):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).float().tolist()
    for c in range(256):
        got = oracle.e4m3_decode(c)
        if math.isnan(ref[c]):
            assert math.isnan(got), c
            assert c in (0x7F, 0xFF)
        else:
            assert got == ref[c], (c, got, ref[c])
    # format landmarks: largest finite, smallest subnormal, smallest normal
    assert oracle.e4m3_decode(0x7E) == 448.0
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9
    assert oracle.e4m3_decode(0x08) == 2.0 ** -6


def test_e4m3_encode_in_range_matches_torch(oracle):
    g = torch.Generator().manual_seed(5)
    v = (torch.randn(3000, generator=g) * torch.logspace(-4, 2.6, 3000)).clamp(-447.0, 447.0)
    ref = v.to(torch.float8_e4m3fn).view(torch.uint8).tolist()
    for val, r in zip(v.tolist(), ref):
        assert oracle.e4m3_encode(val) == r, (val, r)


def test_e4m3_encode_ties_to_even_and_saturation(oracle):
    # every midpoint between adjacent positive codes goes to the even code
    for c in range(0, 0x7E):
        lo, hi = oracle.e4m3_decode(c), oracle.e4m3_decode(c + 1)
        mid = (lo + hi) / 2
        want = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode(mid) == want, (c, mid)
        assert oracle.e4m3_encode(-mid) == 0x80 | want
    assert oracle.e4m3_encode(448.0) == 0x7E
    assert oracle.e4m3_encode(500.0) == 0x7E
    assert oracle.e4m3_encode(-1e30) == 0xFE
    assert oracle.e4m3_encode(float("inf")) == 0x7E


def test_group128_quant_properties(oracle):
    g = np.random.default_rng(11)
    v = g.standard_normal(384).astype(np.float32) * np.float32(3.0)
    v[130] = np.nan  # NaN clamps to +448 (fminf first, then fmaxf)
    v[256:384] = 0.0  # an all-zero group
    codes, scales = oracle.quant_group128(v)
    assert scales.shape == (3,)
    for gi in range(2):
        grp = v[gi * 128:(gi + 1) * 128]
        amax = np.float32(np.nanmax(np.abs(grp)))
        assert scales[gi] == np.float32(amax / np.float32(448.0))
        # the element that sets amax lands exactly on +-448
        i = int(np.nanargmax(np.abs(grp)))
        assert codes[gi * 128 + i] in (0x7E, 0xFE)
    assert codes[130] == 0x7E
    assert scales[2] == np.float32(np.float32(1e-10) / np.float32(448.0))
    assert np.all(codes[256:] == 0)
    # dequantised error within half a code step of the element's binade
    deq = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    for i in range(256):
        if i == 130:
            continue
        s = scales[i // 128]
        q = v[i] / s
        step = 2.0 ** (max(math.floor(math.log2(max(abs(q), 2 ** -6))), -6) - 3)
        assert abs(deq[i] - q) <= step / 2 + 1e-6
