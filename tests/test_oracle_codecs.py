"""Pins of the oracle's number formats and NVFP4 quantiser against things other
than itself: torch's float8_e4m3fn (a library routine), the published E2M1
table, hand-derived round-to-nearest-even cases, and brute-force properties.

Format sources: "DeepSeek-V4.1-Flash-NVFP4" §3.2 (NVFP4 = E2M1 values, one E4M3
scale per 16 elements) and §3.1 (FP8 window).
"""
import math

import numpy as np
import pytest
import torch

from conftest import read_golden
from oracle import oracle as orc

E2M1_GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def torch_e4m3_value(codes):
    return torch.tensor(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn).double().numpy()


def torch_e4m3_encode(x):
    return torch.tensor(np.asarray(x, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e2m1_decode_matches_published_table():
    for code, value in read_golden("e2m1.txt"):
        c, v = int(code, 16), float(value)
        got = orc.e2m1_value(c)
        assert got == v and math.copysign(1, got) == math.copysign(1, v), (code, got, v)


def test_e4m3_decode_all_codes_match_torch():
    ref = torch_e4m3_value(np.arange(256))
    for c in range(256):
        got = orc.e4m3_value(c)
        if np.isnan(ref[c]):
            assert math.isnan(got), c
        else:
            assert got == ref[c], (c, got, ref[c])
    assert orc.e4m3_value(0x7E) == 448.0 and orc.e4m3_value(0x01) == 2.0 ** -9


def test_e4m3_encode_matches_torch_rne_within_range():
    rng = np.random.default_rng(7)
    xs = np.concatenate([
        rng.uniform(-448, 448, 4000), rng.standard_normal(4000),
        rng.uniform(-2e-2, 2e-2, 4000),
        # every midpoint between adjacent finite codes and one ulp either side
        *[(lambda m: np.array([m, np.nextafter(np.float32(m), np.float32(0)),
                               np.nextafter(np.float32(m), np.float32(1e9))]))(
            (orc.e4m3_value(c) + orc.e4m3_value(c + 1)) / 2) for c in range(0, 126)],
    ]).astype(np.float32)
    ref = torch_e4m3_encode(xs)
    got = np.array([orc.e4m3_encode(float(x)) for x in xs], np.uint8)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(xs[i]), int(got[i]), int(ref[i])) for i in bad[:5]]


def test_e4m3_encode_saturates():
    for x in (448.0, 449.0, 463.9, 464.0, 1e6, 3.0e38):
        assert orc.e4m3_encode(x) == 0x7E
        assert orc.e4m3_encode(-x) == 0xFE


def test_e2m1_encode_rne_golden_cases():
    for x, code in read_golden("e2m1_rne.txt"):
        assert orc.e2m1_encode(float(np.float32(x))) == int(code, 16), (x, code)


def test_e2m1_encode_is_nearest_by_brute_force():
    rng = np.random.default_rng(3)
    xs = np.concatenate([rng.uniform(-8, 8, 3000), rng.uniform(-0.6, 0.6, 1000)]).astype(np.float32)
    for x in xs:
        c = orc.e2m1_encode(float(x))
        a = min(abs(float(x)), 6.0)
        d = [abs(a - g) for g in E2M1_GRID]
        best = min(d)
        assert d[c & 7] == best
        ties = [i for i in range(8) if d[i] == best]
        if len(ties) > 1:
            assert (c & 7) % 2 == 0
        assert bool(c & 8) == (np.signbit(x))


def _decode_nibbles(vals):
    v = np.asarray(vals, np.uint8)
    out = np.empty(v.shape[:-1] + (v.shape[-1] * 2,), np.uint8)
    out[..., 0::2] = v & 15
    out[..., 1::2] = v >> 4
    return out


def test_nvfp4_exact_round_trip_of_representable_groups():
    rng = np.random.default_rng(11)
    grid = np.array(E2M1_GRID[1:], np.float64)
    for _ in range(300):
        S_code = int(rng.integers(1, 0x7E))
        S = orc.e4m3_value(S_code)
        if S * 6 > 3e38 or S * 6 != np.float32(S * 6):
            continue
        mags = rng.choice(np.concatenate([[0.0], grid]), 16)
        mags[rng.integers(16)] = 6.0  # amax = 6 S, so amax/6 = S exactly
        signs = rng.choice([-1.0, 1.0], 16)
        x = (signs * mags * S).astype(np.float32)
        assert np.all(x.astype(np.float64) == signs * mags * S)
        vals, scales = orc.nvfp4_quantize(x)
        assert scales[0] == S_code
        codes = _decode_nibbles(vals)
        back = np.array([orc.e2m1_value(int(c)) for c in codes]) * S
        assert np.array_equal(back, x.astype(np.float64))


def test_nvfp4_scale_and_codes_by_brute_force():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((200, 16)) * rng.choice([1e-3, 1.0, 30.0], (200, 1))).astype(np.float32)
    vals, scales = orc.nvfp4_quantize(x)
    codes = _decode_nibbles(vals)
    for g in range(x.shape[0]):
        amax = np.max(np.abs(x[g]))
        s32 = np.float32(amax) / np.float32(6.0)  # numpy fp32 division is IEEE RN
        assert scales[g, 0] == torch_e4m3_encode([s32])[0]  # S = E4M3(fl32(amax/6))
        S = torch_e4m3_value([scales[g, 0]])[0]
        if S == 0:
            assert not codes[g].any()
            continue
        for i in range(16):
            y = np.float32(x[g, i]) / np.float32(S)
            a = min(abs(float(y)), 6.0)
            d = [abs(a - v) for v in E2M1_GRID]
            assert d[codes[g, i] & 7] == min(d)


def test_nvfp4_zero_group_and_saturation_and_nibble_order():
    v, s = orc.nvfp4_quantize(np.zeros(16, np.float32))
    assert s[0] == 0 and not v.any()
    v, s = orc.nvfp4_quantize(np.full(16, 1e9, np.float32))
    assert s[0] == 0x7E and np.all(v == 0x77)
    x = np.zeros(16, np.float32)
    x[0], x[1] = 6.0, 0.5  # S = 1.0: element 0 -> low nibble 0x7, element 1 -> high nibble 0x1
    x[2], x[3] = -1.0, 3.0
    v, s = orc.nvfp4_quantize(x)
    assert s[0] == 0x38 and v[0] == 0x17 and v[1] == 0x5A


def test_nvfp4_value_reads_group_scales():
    x = np.concatenate([np.full(16, 6.0), np.full(16, 0.75)]).astype(np.float32)
    v, s = orc.nvfp4_quantize(x)
    assert list(s) == [0x38, torch_e4m3_encode([0.125])[0]]
    deq = orc.nvfp4_dequant(v, s)
    assert np.all(deq[:16] == 6.0) and np.all(deq[16:] == 0.75)
